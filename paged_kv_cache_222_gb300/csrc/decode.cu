// Single-token paged decode attention: split-KV (flash-decoding) kernel and the
// log-sum-exp combine kernel.
//
// What it computes: out[b, hq, :] = softmax(scale * q[b, hq] . K_b^T) V_b, where
// K_b / V_b are the first ctx_b tokens of sequence b gathered through its block
// table, and query head hq reads KV head hq / G.  Sources: [SC] "LLM
// inference: prefill, decode, KV cache" ("Why We Need the Key-Value (KV)
// Cache"; "PagedAttention & Memory Management (vLLM)"; "Attention
// Architectures: MHA vs. MQA vs. GQA"); [UI] "Architecting Multi-Tier
// Disaggregated KV-Cache Hierarchies...", "High-Throughput Paged Attention
// Kernel Integration" (cache layout [blocks, H_kv, block_size, D], masking of
// the ragged last block, running max / running sum / rescaled accumulator of
// the online softmax, final division by the sum).
//
// Design (GB300):
//  * One CTA per (split, KV head, sequence); a split is `split_tokens`
//    consecutive tokens.  The CTA's 4 warps take 16-token tiles round robin.
//  * Each warp runs its own ring of NS stages.  Lane 0 issues 4-D tiled TMA
//    loads (cp.async.bulk.tensor) of the tile's K and V rows straight from the
//    cache, addressed as (d, token-in-block, kv-head, physical block), into
//    128B-swizzled shared memory, completing on a per-stage mbarrier.  The
//    block table is read 32 tiles at a time by one coalesced warp load.
//  * GQA packing: the G query heads of the KV head share every K/V byte read.
//    S^T[16 tokens x 8 heads] = K_tile . Q^T and O^T[D x 8 heads] += V^T . P^T
//    are mma.sync m16n8k16 tiles (fp32 accumulate); K/V fragments come from
//    ldmatrix (V transposed on load), P^T from the S^T accumulator through
//    movmatrix.  P is fed as a bf16 (or f16) hi + lo pair so that its rounding
//    does not reach the output at the 1e-3 level.
//  * FP8 E4M3 K/V are widened to f16 in registers (exact); the per-(sequence,
//    head) K scale is folded into the logit multiplier, the V scale into the
//    output.
//  * Online softmax in the log2 domain, fp32, warp-shuffle max / sum.  Warps
//    merge through shared memory; a sequence with one split writes `out`
//    directly, otherwise (acc, m, l) partials go to the workspace and the
//    combine kernel merges them.

#include <math_constants.h>

#include <utility>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

template <int D, bool FP8, int NT>
struct Smem {
  using L = Layout<D, FP8>;
  static constexpr int GP = 8 * NT;
  static constexpr int DP = D + 4;                        // padded row of the merge buffer
  static constexpr int MERGE_BYTES = kDecodeWarps * GP * DP * 4;
  static constexpr int MAIN = L::PIPE_BYTES > MERGE_BYTES ? L::PIPE_BYTES : MERGE_BYTES;
  static constexpr int BARS = MAIN;                                   // mbarriers
  static constexpr int ML = BARS + kDecodeWarps * L::NS * 8;          // per-warp m, l
  static constexpr int END = ML + kDecodeWarps * GP * 2 * 4;
  static constexpr int TOTAL = END + 1024;                            // + alignment slack
};

// ----------------------------------------------------------------------------
// One 16-token tile: scores, online-softmax update, P.V accumulation.
// ----------------------------------------------------------------------------
template <int D, bool FP8, int NT>
__device__ __forceinline__ void process_tile(uint32_t stage, int valid, float qk_mult,
                                             const uint32_t (&qb)[D / 16][NT][2],
                                             float (&m_run)[NT][2], float (&l_run)[NT][2],
                                             float (&o)[D / 16][NT][4]) {
  using L = Layout<D, FP8>;
  constexpr int KS = D / 16;
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2;
  // ldmatrix row addresses: matrices (tokens 0-7, c) (tokens 8-15, c)
  // (tokens 0-7, c+1) (tokens 8-15, c+1) for K and for FP8 V.
  const int tok_a = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int chunk_a = lane >> 4;

  // ---- S^T = K . Q^T  (rows: tokens, cols: the group's query heads), with
  // even and odd k-steps in two accumulators to halve the dependent MMA chain
  float s[NT][4], s2[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
  }

  if constexpr (!FP8) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      ldsm_x4(stage + L::off(tok_a, 2 * ks + chunk_a), a);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (ks & 1)
          mma_bf16_16816(s2[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
        else
          mma_bf16_16816(s[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
      }
    }
  } else {
#pragma unroll
    for (int pk = 0; pk < KS / 2; ++pk) {
      uint32_t R[4];
      ldsm_x4(stage + L::off(tok_a, 2 * pk + chunk_a), R);
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        const uint32_t lo = R[2 * q2], hi = R[2 * q2 + 1];   // rows r and r+8
        uint32_t a[4];
        a[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(lo & 0xFFFFu));
        a[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(hi & 0xFFFFu));
        a[2] = e4m3x2_to_f16x2(static_cast<uint16_t>(lo >> 16));
        a[3] = e4m3x2_to_f16x2(static_cast<uint16_t>(hi >> 16));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (q2)
            mma_f16_16816(s2[nt], a, qb[2 * pk + q2][nt][0], qb[2 * pk + q2][nt][1]);
          else
            mma_f16_16816(s[nt], a, qb[2 * pk + q2][nt][0], qb[2 * pk + q2][nt][1]);
        }
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s[nt][0] += s2[nt][0];
    s[nt][1] += s2[nt][1];
    s[nt][2] += s2[nt][2];
    s[nt][3] += s2[nt][3];
  }

  // ---- online softmax (log2 domain); lane holds tokens r, r+8 x heads 2j, 2j+1
  uint32_t pb_hi[NT][2], pb_lo[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // packed f32x2 arithmetic (the same IEEE operations, half the instructions)
    const float2 qm = make_float2(qk_mult, qk_mult);
    const float2 xa = __fmul2_rn(make_float2(s[nt][0], s[nt][1]), qm);
    const float2 xb = __fmul2_rn(make_float2(s[nt][2], s[nt][3]), qm);
    float x0 = xa.x, x1 = xa.y, x2 = xb.x, x3 = xb.y;
    if (valid < kTileTokens) {
      if (r >= valid) x0 = x1 = -CUDART_INF_F;
      if (r + 8 >= valid) x2 = x3 = -CUDART_INF_F;
    }
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, sh));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, sh));
    }
    const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
    const float mu0 = (mn0 == -CUDART_INF_F) ? 0.f : mn0;
    const float mu1 = (mn1 == -CUDART_INF_F) ? 0.f : mn1;
    const float al0 = fast_exp2(m_run[nt][0] - mu0), al1 = fast_exp2(m_run[nt][1] - mu1);
    m_run[nt][0] = mn0;
    m_run[nt][1] = mn1;
    const float2 nmu = make_float2(-mu0, -mu1);
    const float2 ea = __fadd2_rn(make_float2(x0, x1), nmu);
    const float2 eb = __fadd2_rn(make_float2(x2, x3), nmu);
    const float p0 = fast_exp2(ea.x), p1 = fast_exp2(ea.y);
    const float p2 = fast_exp2(eb.x), p3 = fast_exp2(eb.y);
    l_run[nt][0] = l_run[nt][0] * al0 + (p0 + p2);
    l_run[nt][1] = l_run[nt][1] * al1 + (p1 + p3);
    const float2 al = make_float2(al0, al1);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const float2 u = __fmul2_rn(make_float2(o[mt][nt][0], o[mt][nt][1]), al);
      const float2 w = __fmul2_rn(make_float2(o[mt][nt][2], o[mt][nt][3]), al);
      o[mt][nt][0] = u.x;
      o[mt][nt][1] = u.y;
      o[mt][nt][2] = w.x;
      o[mt][nt][3] = w.y;
    }
    // P rows (token r | token r+8) x (heads 2j, 2j+1) as 16-bit pairs,
    // transposed in registers into the B fragment of the P.V product.  With
    // bf16 V, P is a bf16 hi + lo pair (bf16 alone would round each p to 8
    // bits: up to 2^-9 max|v| in the output, above the 2e-3 budget for
    // |v| ~ 4).  With E4M3 V, P is one f16 term: its rounding, at most
    // 2^-11 of the largest |v|, is far below the E4M3 codes' own 2^-4 (the
    // FP8 workload's error moved from 5e-7 to 3e-5 against its 5e-3 budget)
    // and halves the P.V products.
    if constexpr (!FP8) {
      const uint32_t h0 = pack_bf16x2(p0, p1);
      const uint32_t h1 = pack_bf16x2(p2, p3);
      const uint32_t l0 = pack_bf16x2(p0 - bf16lo_to_f32(h0), p1 - bf16hi_to_f32(h0));
      const uint32_t l1 = pack_bf16x2(p2 - bf16lo_to_f32(h1), p3 - bf16hi_to_f32(h1));
      pb_hi[nt][0] = movmatrix_trans(h0);
      pb_hi[nt][1] = movmatrix_trans(h1);
      pb_lo[nt][0] = movmatrix_trans(l0);
      pb_lo[nt][1] = movmatrix_trans(l1);
    } else {
      pb_hi[nt][0] = movmatrix_trans(pack_f16x2(p0, p1));
      pb_hi[nt][1] = movmatrix_trans(pack_f16x2(p2, p3));
    }
  }

  // ---- O^T += V^T . P^T
  const uint32_t vtile = stage + L::TILEB;
  if constexpr (!FP8) {
    // matrices (tokens 0-7, c) (tokens 0-7, c+1) (tokens 8-15, c) (tokens 8-15, c+1)
    const int tok_v = (lane & 7) + ((lane >> 4) & 1) * 8;
    const int chunk_v = (lane >> 3) & 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a[4];
      ldsm_x4_trans(vtile + L::off(tok_v, 2 * mt + chunk_v), a);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16_16816(o[mt][nt], a, pb_hi[nt][0], pb_hi[nt][1]);
        mma_bf16_16816(o[mt][nt], a, pb_lo[nt][0], pb_lo[nt][1]);
      }
    }
  } else {
#pragma unroll
    for (int pk = 0; pk < KS / 2; ++pk) {
      uint32_t R[4];
      ldsm_x4_trans(vtile + L::off(tok_a, 2 * pk + chunk_a), R);
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        // bytes of R: V[2j][2r'] V[2j][2r'+1] V[2j+1][2r'] V[2j+1][2r'+1];
        // regroup to (even d: tokens 2j, 2j+1 | odd d: tokens 2j, 2j+1)
        const uint32_t e0 = prmt(R[2 * q2], 0u, 0x3120u);       // tokens 0-7
        const uint32_t e1 = prmt(R[2 * q2 + 1], 0u, 0x3120u);   // tokens 8-15
        uint32_t a[4];
        a[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(e0 & 0xFFFFu));
        a[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(e0 >> 16));
        a[2] = e4m3x2_to_f16x2(static_cast<uint16_t>(e1 & 0xFFFFu));
        a[3] = e4m3x2_to_f16x2(static_cast<uint16_t>(e1 >> 16));
        const int mt = 2 * pk + q2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16_16816(o[mt][nt], a, pb_hi[nt][0], pb_hi[nt][1]);
      }
    }
  }
}

// ----------------------------------------------------------------------------
// Pieces shared by the two decode kernels.
// ----------------------------------------------------------------------------

// Warps the stream-K split uses for T flat tiles: at most the grid's warps,
// and never fewer than kMinTilesPerWorker tiles per warp, so no range is empty.
constexpr int kMinTilesPerWorker = 8;
__host__ __device__ __forceinline__ int64_t streamk_workers_used(int64_t T, int64_t grid_workers) {
  const int64_t by_work = T / kMinTilesPerWorker;
  const int64_t w = by_work < grid_workers ? by_work : grid_workers;
  return w < 1 ? 1 : w;
}

// Query fragments (B operand of S^T = K . Q^T) of heads 8nt + r of the group
// whose first row is `qrow`; zero past G.  FP8 caches take f16 fragments in the
// d-order of the widened E4M3 A fragments.
template <int D, bool FP8, int NT>
__device__ __forceinline__ void load_q_frags(const uint16_t* qrow, int G,
                                             uint32_t (&qb)[D / 16][NT][2]) {
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, j = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = 8 * nt + r;
    const uint16_t* qg = qrow + static_cast<int64_t>(g) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      if (g >= G) {
        qb[ks][nt][0] = qb[ks][nt][1] = 0u;
      } else if constexpr (!FP8) {
        const int d0 = 16 * ks + 2 * j;
        qb[ks][nt][0] = *reinterpret_cast<const uint32_t*>(qg + d0);
        qb[ks][nt][1] = *reinterpret_cast<const uint32_t*>(qg + d0 + 8);
      } else {
        const int d0 = 16 * ks + 4 * j;
        const uint2 w = *reinterpret_cast<const uint2*>(qg + d0);
        qb[ks][nt][0] = pack_f16x2(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x));
        qb[ks][nt][1] = pack_f16x2(bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
      }
    }
  }
}

template <int D, int NT>
__device__ __forceinline__ void reset_state(float (&m_run)[NT][2], float (&l_run)[NT][2],
                                            float (&o)[D / 16][NT][4]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
  }
}

// Sum each lane's partial row sums over the 8 lanes that share its heads.
template <int NT>
__device__ __forceinline__ void reduce_l(float (&l_run)[NT][2]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = l_run[nt][e];
      l += __shfl_xor_sync(kFull, l, 4);
      l += __shfl_xor_sync(kFull, l, 8);
      l += __shfl_xor_sync(kFull, l, 16);
      l_run[nt][e] = l;
    }
  }
}

// Issue the TMA loads of one 16-token K/V tile into a stage (lane 0 only).
template <class L>
__device__ __forceinline__ void issue_tile(uint32_t dst, uint32_t bar, const CUtensorMap* tk,
                                           const CUtensorMap* tv, int tok0, int h, int phys) {
  fence_proxy_async_smem();
  mbar_arrive_expect_tx(bar, L::STAGEB);
#pragma unroll
  for (int bx = 0; bx < L::NBOX; ++bx)
    tma_load_4d(dst + bx * L::BOX_BYTES, tk, bar, bx * L::BOX_ELEMS, tok0, h, phys);
#pragma unroll
  for (int bx = 0; bx < L::NBOX; ++bx)
    tma_load_4d(dst + L::TILEB + bx * L::BOX_BYTES, tv, bar, bx * L::BOX_ELEMS, tok0, h, phys);
}

// Rows past the end of the sequence may hold anything (NaN included): zero
// them in the V tile so that P = 0 times V stays 0 in the MMA.
template <class L>
__device__ __forceinline__ void zero_v_tail(uint8_t* vtile, int valid) {
  const int lane = threadIdx.x & 31;
  const int nchunks = (kTileTokens - valid) * (L::ROWB / 16);
  for (int c = lane; c < nchunks; c += 32) {
    const int tr = valid + c / (L::ROWB / 16);
    const int cc = c % (L::ROWB / 16);
    *reinterpret_cast<uint4*>(vtile + L::off(tr, cc)) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// Head g and dims (d_a, d_b) held by this lane for accumulator element pairs.
template <bool FP8>
__device__ __forceinline__ void frag_dims(int mt, int& d_a, int& d_b) {
  const int r = (threadIdx.x & 31) >> 2;
  if constexpr (!FP8) {
    d_a = 16 * mt + r;
    d_b = d_a + 8;
  } else {
    d_a = 16 * mt + 2 * r;
    d_b = d_a + 1;
  }
}

// ----------------------------------------------------------------------------
// Fixed-split kernel: one CTA per (split, KV head, sequence), a split being
// `split_tokens` consecutive tokens; its 4 warps take 16-token tiles round
// robin and merge through shared memory.  Used when the caller asks for a
// split size, and for batches too large for the stream-K kernel's table.
// ----------------------------------------------------------------------------
template <int D, bool FP8, int NT>
__global__ void __launch_bounds__(kDecodeWarps * 32, 3)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using L = Layout<D, FP8>;
  using S = Smem<D, FP8, NT>;
  constexpr int NW = kDecodeWarps;
  constexpr int NS = L::NS;
  constexpr int KS = D / 16;

  wait_prior_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, j = lane & 3;
  const int G = p.group;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;

  const int ctx_raw = p.context_lens[b];
  const int ctx = clamp_ctx(p, ctx_raw);
  // a cascade call's sequences must hold the whole shared prefix
  // (token_offset); the prefix kernel attends it for every row
  if ((ctx != ctx_raw || ctx_raw < p.token_offset) && split == 0 && h == 0 && threadIdx.x == 0)
    record_error(p.err, kDevErrContextLen);
  const int64_t row0 = static_cast<int64_t>(b) * p.num_q_heads + static_cast<int64_t>(h) * G;

  // tokens [token_offset, ctx) are split; token_offset > 0 leaves a shared
  // prefix to the cascade prefix kernel
  const int t_begin = p.token_offset + split * p.split_tokens;
  if (t_begin >= ctx) {
    if (ctx == 0 && split == 0 && !p.force_partial) {
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) p.out[row0 * D + i] = 0.f;
    }
    return;
  }
  const int t_end = min(ctx, t_begin + p.split_tokens);
  const int n_tiles = (t_end - t_begin + kTileTokens - 1) / kTileTokens;
  const int nsplit = (ctx - p.token_offset + p.split_tokens - 1) / p.split_tokens;

  // Fused append: the CTA that attends the sequence's newest token (position
  // ctx - 1, in its last split) writes that token's K / V rows of head h into
  // their slot, encoded as the append kernel does, so the step needs no
  // separate append launch.  No other CTA reads the slot.  The warp whose
  // tile holds the token writes it (after its first loads are in flight,
  // unless that tile is one of them) and orders the writes before its own
  // load of the tile with a proxy fence: no other warp waits.
  const bool fuse_new = p.new_src != 0 && t_end == ctx && ctx == ctx_raw;
  const int w_new = (n_tiles - 1) % NW, k_tok = (n_tiles - 1) / NW;  // owner warp, its tile index
  auto write_new = [&]() {
    constexpr int PER_ROW = D / 8;                  // lanes per row, eight elements each
    if (lane < 2 * PER_ROW) {
      const int pos = ctx - 1;
      const int phys = p.block_tables[static_cast<int64_t>(b) * p.max_blocks + pos / p.block_size];
      if (phys >= 0 && phys < p.num_blocks) {
        const bool is_v = lane >= PER_ROW;
        const int part = lane - (is_v ? PER_ROW : 0);
        const int64_t src = (static_cast<int64_t>(b) * p.num_kv_heads + h) * D + part * 8;
        const int64_t dst =
            ((static_cast<int64_t>(phys) * p.num_kv_heads + h) * p.block_size + pos % p.block_size) * D + part * 8;
        float sc = 1.f;
        if constexpr (FP8) sc = (is_v ? p.v_scale : p.k_scale)[static_cast<int64_t>(b) * p.scale_stride + h];
        constexpr int DST = FP8 ? kEncE4M3 : kEncBF16;
        float x[8];
        uint4 raw;
        if (p.new_src == kEncBF16 + 1) {
          enc_load8<kEncBF16>(is_v ? p.v_new : p.k_new, src, x, raw);
          enc_store8<kEncBF16, DST>(is_v ? p.v_cache : p.k_cache, dst, x, raw, sc);
        } else {
          enc_load8<kEncF32>(is_v ? p.v_new : p.k_new, src, x, raw);
          enc_store8<kEncF32, DST>(is_v ? p.v_cache : p.k_cache, dst, x, raw, sc);
        }
      } else if (lane == 0) {
        record_error(p.err, kDevErrBlockId);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncwarp();
  };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BARS);
  float* s_ml = reinterpret_cast<float*>(smem + S::ML);

  const uint32_t wstage0 = smem_u32(smem) + warp * NS * L::STAGEB;
  const uint32_t wbar0 = smem_u32(bars + warp * NS);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(wbar0 + 8 * s, 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  __syncwarp();

  float qk_mult = p.qk_log2_scale;
  float v_mult = 1.f;
  if constexpr (FP8) {
    qk_mult *= p.k_scale[static_cast<int64_t>(b) * p.scale_stride + h];
    v_mult = p.v_scale[static_cast<int64_t>(b) * p.scale_stride + h];
  }
  uint32_t qb[KS][NT][2];
  load_q_frags<D, FP8, NT>(static_cast<const uint16_t*>(p.q) + row0 * D, G, qb);

  // this warp's tiles: the k-th covers tokens t_begin + 16 (warp + k NW)
  const int nk = n_tiles > warp ? (n_tiles - warp + NW - 1) / NW : 0;
  const int32_t* tbl = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
  auto load_phys = [&](int kbase) -> int {
    const int k = kbase + lane;
    int phys = -1;
    if (k < nk) {
      const int t = t_begin + kTileTokens * (warp + k * NW);
      phys = tbl[t / p.block_size];
      if (phys < 0 || phys >= p.num_blocks) {
        record_error(p.err, kDevErrBlockId);
        phys = -1;  // fully outside the tensor: the TMA unit fills zeros
      }
    }
    return phys;
  };
  auto issue = [&](int k, int phys) {
    const int s = k % NS;
    const int t = t_begin + kTileTokens * (warp + k * NW);
    // token within its block: the block size is 16 or 32 (a power of two), so a
    // mask instead of a run-time remainder (2 % on the issue-heavy E4M3 path)
    issue_tile<L>(wstage0 + s * L::STAGEB, wbar0 + 8 * s, &tmap_k, &tmap_v, t & (p.block_size - 1), h, phys);
  };

  const bool writer = fuse_new && warp == w_new;
  if (writer && k_tok < NS) write_new();   // the token's tile is one of the first loads
  int phys_reg = load_phys(0);
  const int npro = nk < NS ? nk : NS;
  for (int k = 0; k < npro; ++k) {
    const int ph = __shfl_sync(kFull, phys_reg, k);
    if (lane == 0) issue(k, ph);
  }
  if (writer && k_tok >= NS) write_new();  // its load comes later in the loop below

  float m_run[NT][2], l_run[NT][2], o[KS][NT][4];
  reset_state<D, NT>(m_run, l_run, o);

  bool healthy = true;
  for (int k = 0; k < nk; ++k) {
    const int s = k % NS;
    const uint32_t stage = wstage0 + s * L::STAGEB;
    // the whole warp takes the same branch below (ldmatrix / mma / shfl)
    const bool arrived = mbar_wait(wbar0 + 8 * s, static_cast<uint32_t>((k / NS) & 1), p.err);
    if (!__all_sync(kFull, arrived)) healthy = false;
    if (healthy) {
      const int t = t_begin + kTileTokens * (warp + k * NW);
      const int valid = min(kTileTokens, ctx - t);
      if (valid < kTileTokens) zero_v_tail<L>(smem + (stage - smem_u32(smem)) + L::TILEB, valid);
      process_tile<D, FP8, NT>(stage, valid, qk_mult, qb, m_run, l_run, o);
    }
    __syncwarp();
    const int kn = k + NS;
    if (kn < nk && healthy) {
      if ((kn & 31) == 0) phys_reg = load_phys(kn);
      const int ph = __shfl_sync(kFull, phys_reg, kn & 31);
      if (lane == 0) issue(kn, ph);
    }
  }
  if (!healthy) {
    // a copy may still be landing: give each stage one more bounded wait on
    // its last phase before the shared memory is reused or released
    for (int s = 0; s < NS && s < nk; ++s) {
      const int klast = s + ((nk - 1 - s) / NS) * NS;
      mbar_wait(wbar0 + 8 * s, static_cast<uint32_t>((klast / NS) & 1), nullptr);
    }
  }
  allow_next_grid();

  // ---- finish the per-lane sums, merge the warps through shared memory
  reduce_l<NT>(l_run);
  __syncthreads();  // every warp is done with the pipeline buffers
  float* s_o = reinterpret_cast<float*>(smem);  // [NW][GP][DP]
  {
    float* wo = s_o + warp * S::GP * S::DP;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int g0 = 8 * nt + 2 * j;
        int d_a, d_b;
        frag_dims<FP8>(mt, d_a, d_b);
        wo[g0 * S::DP + d_a] = o[mt][nt][0];
        wo[(g0 + 1) * S::DP + d_a] = o[mt][nt][1];
        wo[g0 * S::DP + d_b] = o[mt][nt][2];
        wo[(g0 + 1) * S::DP + d_b] = o[mt][nt][3];
      }
    }
    if (r == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int g0 = 8 * nt + 2 * j;
        float* ml = s_ml + (warp * S::GP + g0) * 2;
        ml[0] = m_run[nt][0];
        ml[1] = l_run[nt][0];
        ml[2] = m_run[nt][1];
        ml[3] = l_run[nt][1];
      }
    }
  }
  __syncthreads();

  const bool direct = (nsplit == 1) && !p.force_partial;
  const int64_t S_max = p.slots_per_row;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, d = idx - (idx / D) * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_ml[(w * S::GP + g) * 2]);
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = s_ml[(w * S::GP + g) * 2];
      const float wt = (mw == -CUDART_INF_F) ? 0.f : fast_exp2(mw - M);
      acc += wt * s_o[(w * S::GP + g) * S::DP + d];
      lsum += wt * s_ml[(w * S::GP + g) * 2 + 1];
    }
    const int64_t row = row0 + g;
    if (direct) {
      p.out[row * D + d] = acc * v_mult / lsum;
    } else {
      const int64_t slot = row * S_max + split;
      p.ws_o[slot * D + d] = acc * v_mult;
      if (d == 0) {
        p.ws_ml[slot * 2] = M;
        p.ws_ml[slot * 2 + 1] = lsum;
      }
    }
  }
}

// ----------------------------------------------------------------------------
// LSE combine for few splits (<= 8): one warp per (sequence, query head), all
// of the row's loads issued at once; each lane owns D/32 consecutive dims.
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) combine_rows_kernel(const DecodeParams p) {
  constexpr int V = D / 32;
  constexpr int R = 8;
  wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(p.batch) * p.num_q_heads) return;
  const int b = static_cast<int>(row / p.num_q_heads);
  const int ctx = clamp_ctx(p, p.context_lens[b]);
  const int cs = ctx > p.token_offset ? ctx - p.token_offset : 0;
  const int nsplit = (cs + p.split_tokens - 1) / p.split_tokens;
  if (!p.force_partial && nsplit <= 1) return;  // written by the split kernel
  const int ntot = nsplit + p.extra_count;      // + shared-prefix pieces
  const int64_t S_max = p.slots_per_row;
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml + row * S_max * 2);
  const float* wo = p.ws_o + row * S_max * D + lane * V;
  float2 mlr[R];
  float x[R][V];
#pragma unroll
  for (int u = 0; u < R; ++u) {
    mlr[u] = make_float2(-CUDART_INF_F, 0.f);
#pragma unroll
    for (int v = 0; v < V; ++v) x[u][v] = 0.f;
    if (u < ntot) {
      const int slot = u < nsplit ? u : p.extra_slot + (u - nsplit);
      mlr[u] = ml[slot];
      if constexpr (V == 4) {
        const float4 t = *reinterpret_cast<const float4*>(wo + static_cast<int64_t>(slot) * D);
        x[u][0] = t.x; x[u][1] = t.y; x[u][2] = t.z; x[u][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(wo + static_cast<int64_t>(slot) * D);
        x[u][0] = t.x; x[u][1] = t.y;
      }
    }
  }
  float M = -CUDART_INF_F;
#pragma unroll
  for (int u = 0; u < R; ++u) M = fmaxf(M, mlr[u].x);
  float L = 0.f, acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
#pragma unroll
  for (int u = 0; u < R; ++u) {
    const float w = (mlr[u].x == -CUDART_INF_F) ? 0.f : fast_exp2(mlr[u].x - M);
    L += w * mlr[u].y;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] += w * x[u][v];
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;  // a row with nothing to attend gives zeros
  float* dst = p.out + row * D + lane * V;
  if constexpr (V == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
  }
}

// ----------------------------------------------------------------------------
// LSE combine of a cascade call (at most R = 4 or 8 slots per row: the row's
// suffix splits, then the shared-prefix pieces).  Every slot is written but
// suffix splits past a row's own count, so the loads go out before the
// context length arrives and the unwritten slots (which may hold anything)
// are dropped by selection afterwards.  One warp per (sequence, query head);
// each lane owns D/32 consecutive dims; with 4 slots sixteen CTAs fit an SM.
// ----------------------------------------------------------------------------
template <int D, int R>
__global__ void __launch_bounds__(128, R <= 4 ? 16 : 1) combine_cascade_kernel(const DecodeParams p) {
  constexpr int V = D / 32;
  wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(p.batch) * p.num_q_heads) return;
  const int b = static_cast<int>(row / p.num_q_heads);
  const int S_max = p.slots_per_row;
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml + row * S_max * 2);
  const float* wo = p.ws_o + row * S_max * D + lane * V;
  float2 mlr[R];
  float x[R][V];
#pragma unroll
  for (int s = 0; s < R; ++s) {
    mlr[s] = make_float2(-CUDART_INF_F, 0.f);
#pragma unroll
    for (int v = 0; v < V; ++v) x[s][v] = 0.f;
    if (s < S_max) {
      mlr[s] = ml[s];
      if constexpr (V == 4) {
        const float4 t = *reinterpret_cast<const float4*>(wo + static_cast<int64_t>(s) * D);
        x[s][0] = t.x; x[s][1] = t.y; x[s][2] = t.z; x[s][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(wo + static_cast<int64_t>(s) * D);
        x[s][0] = t.x; x[s][1] = t.y;
      }
    }
  }
  const int ctx = clamp_ctx(p, p.context_lens[b]);
  const int cs = ctx > p.token_offset ? ctx - p.token_offset : 0;
  const int nsplit = (cs + p.split_tokens - 1) / p.split_tokens;
  float M = -CUDART_INF_F;
#pragma unroll
  for (int s = 0; s < R; ++s) {
    // a split of the row, or a shared-prefix piece
    const bool holds = s < nsplit || (s >= p.extra_slot && s < p.extra_slot + p.extra_count);
    if (!holds) {
      mlr[s] = make_float2(-CUDART_INF_F, 0.f);
#pragma unroll
      for (int v = 0; v < V; ++v) x[s][v] = 0.f;
    }
    M = fmaxf(M, mlr[s].x);
  }
  float L = 0.f, acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
#pragma unroll
  for (int s = 0; s < R; ++s) {
    const float w = (mlr[s].x == -CUDART_INF_F) ? 0.f : fast_exp2(mlr[s].x - M);
    L += w * mlr[s].y;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] += w * x[s][v];
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;  // a row with nothing to attend gives zeros
  float* dst = p.out + row * D + lane * V;
  if constexpr (V == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
  }
}

// ----------------------------------------------------------------------------
// LSE combine of the fixed-split kernel's partials:
//   out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
// One CTA (4 warps) per (sequence, query head).  Warp w takes splits w, w+4,
// ..., 8 of them per round with every load of the round issued before any is
// used, keeping a running (M, L, acc) that is rescaled between rounds; the
// warps then merge through shared memory.  Each lane owns D/32 dims.
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p) {
  constexpr int V = D / 32;
  constexpr int R = 8;
  __shared__ float s_acc[4][D];
  __shared__ float s_ml[4][2];
  wait_prior_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  const int b = static_cast<int>(row / p.num_q_heads);
  const int ctx = clamp_ctx(p, p.context_lens[b]);
  const int cs = ctx > p.token_offset ? ctx - p.token_offset : 0;
  const int nsplit = (cs + p.split_tokens - 1) / p.split_tokens;
  if (!p.force_partial && nsplit <= 1) return;  // written by the split kernel
  const int ntot = nsplit + p.extra_count;      // + shared-prefix pieces
  const int64_t S_max = p.slots_per_row;
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml + row * S_max * 2);
  const float* wo = p.ws_o + row * S_max * D + lane * V;
  float M = -CUDART_INF_F, L = 0.f, acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int i0 = warp; i0 < ntot; i0 += 4 * R) {
    float2 mlr[R];
    float x[R][V];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int i = i0 + 4 * u;
      mlr[u] = make_float2(-CUDART_INF_F, 0.f);
#pragma unroll
      for (int v = 0; v < V; ++v) x[u][v] = 0.f;
      if (i < ntot) {
        const int slot = i < nsplit ? i : p.extra_slot + (i - nsplit);
        mlr[u] = ml[slot];
        if constexpr (V == 4) {
          const float4 t = *reinterpret_cast<const float4*>(wo + static_cast<int64_t>(slot) * D);
          x[u][0] = t.x; x[u][1] = t.y; x[u][2] = t.z; x[u][3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(wo + static_cast<int64_t>(slot) * D);
          x[u][0] = t.x; x[u][1] = t.y;
        }
      }
    }
    float Mn = M;
#pragma unroll
    for (int u = 0; u < R; ++u) Mn = fmaxf(Mn, mlr[u].x);
    const float keep = (M == -CUDART_INF_F) ? 0.f : fast_exp2(M - Mn);
    L *= keep;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] *= keep;
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const float w = (mlr[u].x == -CUDART_INF_F) ? 0.f : fast_exp2(mlr[u].x - Mn);
      L += w * mlr[u].y;
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] += w * x[u][v];
    }
    M = Mn;
  }
#pragma unroll
  for (int v = 0; v < V; ++v) s_acc[warp][lane * V + v] = acc[v];
  if (lane == 0) {
    s_ml[warp][0] = M;
    s_ml[warp][1] = L;
  }
  __syncthreads();
  float Mt = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < 4; ++w) Mt = fmaxf(Mt, s_ml[w][0]);
  float wt[4], Lt = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    wt[w] = (s_ml[w][0] == -CUDART_INF_F) ? 0.f : fast_exp2(s_ml[w][0] - Mt);
    Lt += wt[w] * s_ml[w][1];
  }
  const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x)
    p.out[row * D + d] =
        (wt[0] * s_acc[0][d] + wt[1] * s_acc[1][d] + wt[2] * s_acc[2][d] + wt[3] * s_acc[3][d]) * inv;
}

// ----------------------------------------------------------------------------
// Stream-K kernel.  The (sequence, KV head, 16-token tile) space is flattened:
// unit (b, h) holds tiles_b = ceil(ctx_b / 16) tiles and its tile lt has flat
// index H_kv * Q[b] + h * tiles_b + lt, Q[b] = sum of tiles_b' over b' < b.
// Warp w of the persistent grid (W warps in all) owns flat tiles
// [floor(w T / W), floor((w+1) T / W)): every warp streams the same number of
// tiles (+-1), and its TMA ring keeps running across unit boundaries.  A unit
// that lies wholly inside one warp's range is written to `out` directly; the
// pieces of a unit cut by range boundaries go to the workspace as (acc, m, l)
// and the fix-up kernel merges them.
// ----------------------------------------------------------------------------
template <int D, bool FP8, int NT, int NW, int NS, int MINB>
__global__ void __launch_bounds__(NW * 32, MINB)
    decode_streamk_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using L = Layout<D, FP8>;
  constexpr int KS = D / 16;
  constexpr int GP = 8 * NT;
  static_assert(L::STAGEB * NS * NW <= 160 * 1024, "pipeline too large");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, j = lane & 3;
  const int B = p.batch, Hkv = p.num_kv_heads, G = p.group;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * NS * L::STAGEB);
  int* sQ = reinterpret_cast<int*>(bars + NW * NS);  // [B + 1] tile prefix

  const uint32_t wstage0 = smem_u32(smem) + warp * NS * L::STAGEB;
  const uint32_t wbar0 = smem_u32(bars + warp * NS);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(wbar0 + 8 * s, 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  wait_prior_grid();

  // ---- tile prefix Q over sequences (every CTA; CTA 0 also stores it)
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    const int raw = p.context_lens[i];
    const int c = clamp_ctx(p, raw);
    if (c != raw && blockIdx.x == 0) record_error(p.err, kDevErrContextLen);
    sQ[i + 1] = (c + kTileTokens - 1) / kTileTokens;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (B + 31) / 32;
    const int lo = lane * per, hi = min(B, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += sQ[i + 1];
    int incl = sum;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, sh);
      if (lane >= sh) incl += v;
    }
    int run = incl - sum;
    for (int i = lo; i < hi; ++i) {
      run += sQ[i + 1];
      sQ[i + 1] = run;
    }
    if (lane == 0) sQ[0] = 0;
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i <= B; i += blockDim.x) p.ws_q[i] = sQ[i];

  const int64_t T = static_cast<int64_t>(Hkv) * sQ[B];
  const int64_t Wt = streamk_workers_used(T, p.workers);
  const int w = blockIdx.x * NW + warp;
  const int64_t f_begin = w < Wt ? static_cast<int64_t>(w) * T / Wt : T;
  const int nk = w < Wt ? static_cast<int>(static_cast<int64_t>(w + 1) * T / Wt - f_begin) : 0;

  // flat tile -> (sequence, head, tile in unit)
  auto locate = [&](int64_t f, int& b, int& h, int& lt) {
    int lo = 0, hi = B;  // first i with Hkv * Q[i] > f is in (lo, hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<int64_t>(Hkv) * sQ[mid] > f) hi = mid; else lo = mid;
    }
    b = lo;
    const int tb = sQ[b + 1] - sQ[b];
    const int rr = static_cast<int>(f - static_cast<int64_t>(Hkv) * sQ[b]);
    h = rr / tb;
    lt = rr - h * tb;
  };
  // lane i: physical block and (head, token offset) of tile kbase + i
  auto fetch = [&](int kbase, int& phys, int& hinfo) {
    const int k = kbase + lane;
    phys = -1;
    hinfo = 0;
    if (k < nk) {
      int b, h, lt;
      locate(f_begin + k, b, h, lt);
      const int t = lt * kTileTokens;
      phys = p.block_tables[static_cast<int64_t>(b) * p.max_blocks + t / p.block_size];
      if (phys < 0 || phys >= p.num_blocks) {
        record_error(p.err, kDevErrBlockId);
        phys = -1;  // fully outside the tensor: the TMA unit fills zeros
      }
      hinfo = (h << 6) | (t % p.block_size);
    }
  };
  int phys_reg, hinfo_reg;
  auto issue = [&](int k) {
    const int ph = __shfl_sync(kFull, phys_reg, k & 31);
    const int hi = __shfl_sync(kFull, hinfo_reg, k & 31);
    if (lane == 0) {
      const int s = k % NS;
      issue_tile<L>(wstage0 + s * L::STAGEB, wbar0 + 8 * s, &tmap_k, &tmap_v, hi & 63, hi >> 6, ph);
    }
  };

  if (nk > 0) {
    fetch(0, phys_reg, hinfo_reg);
    const int npro = nk < NS ? nk : NS;
    for (int k = 0; k < npro; ++k) issue(k);
  }

  // ---- compute cursor
  int cb = 0, ch = 0, clt = 0;
  if (nk > 0) locate(f_begin, cb, ch, clt);
  int ctiles = nk > 0 ? sQ[cb + 1] - sQ[cb] : 0;
  int cctx = 0, seg_lt0 = clt, seg_slot = 0;
  uint32_t qb[KS][NT][2];
  float m_run[NT][2], l_run[NT][2], o[KS][NT][4];
  float qk_mult = 0.f, v_mult = 1.f;
  auto begin_unit = [&]() {
    cctx = clamp_ctx(p, p.context_lens[cb]);
    const int64_t row0 = static_cast<int64_t>(cb) * p.num_q_heads + static_cast<int64_t>(ch) * G;
    load_q_frags<D, FP8, NT>(static_cast<const uint16_t*>(p.q) + row0 * D, G, qb);
    qk_mult = p.qk_log2_scale;
    v_mult = 1.f;
    if constexpr (FP8) {
      qk_mult *= p.k_scale[static_cast<int64_t>(cb) * p.scale_stride + ch];
      v_mult = p.v_scale[static_cast<int64_t>(cb) * p.scale_stride + ch];
    }
    reset_state<D, NT>(m_run, l_run, o);
  };
  if (nk > 0) begin_unit();

  bool healthy = true;
  for (int k = 0; k < nk; ++k) {
    const int s = k % NS;
    const uint32_t stage = wstage0 + s * L::STAGEB;
    const bool arrived = mbar_wait(wbar0 + 8 * s, static_cast<uint32_t>((k / NS) & 1), p.err);
    if (!__all_sync(kFull, arrived)) healthy = false;
    if (healthy) {
      const int valid = min(kTileTokens, cctx - clt * kTileTokens);
      if (valid < kTileTokens) zero_v_tail<L>(smem + (stage - smem_u32(smem)) + L::TILEB, valid);
      process_tile<D, FP8, NT>(stage, valid, qk_mult, qb, m_run, l_run, o);
    }
    __syncwarp();
    const int kn = k + NS;
    if (kn < nk && healthy) {
      if ((kn & 31) == 0) fetch(kn, phys_reg, hinfo_reg);
      issue(kn);
    }
    // ---- advance; close the segment at a unit end or at the end of the range
    ++clt;
    const bool unit_end = (clt == ctiles);
    if (unit_end || k == nk - 1) {
      reduce_l<NT>(l_run);
      const int64_t row0 = static_cast<int64_t>(cb) * p.num_q_heads + static_cast<int64_t>(ch) * G;
      if (seg_lt0 == 0 && unit_end) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int g0 = 8 * nt + 2 * j;
          const float s0 = v_mult / l_run[nt][0], s1 = v_mult / l_run[nt][1];
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            int d_a, d_b;
            frag_dims<FP8>(mt, d_a, d_b);
            if (g0 < G) {
              float* dst = p.out + (row0 + g0) * D;
              dst[d_a] = o[mt][nt][0] * s0;
              dst[d_b] = o[mt][nt][2] * s0;
            }
            if (g0 + 1 < G) {
              float* dst = p.out + (row0 + g0 + 1) * D;
              dst[d_a] = o[mt][nt][1] * s1;
              dst[d_b] = o[mt][nt][3] * s1;
            }
          }
        }
      } else {
        const int64_t pw = static_cast<int64_t>(w) * 2 + seg_slot;
        float* wo = p.ws_o + pw * GP * D;
        float* wml = p.ws_ml + pw * GP * 2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int g0 = 8 * nt + 2 * j;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            int d_a, d_b;
            frag_dims<FP8>(mt, d_a, d_b);
            wo[g0 * D + d_a] = o[mt][nt][0] * v_mult;
            wo[g0 * D + d_b] = o[mt][nt][2] * v_mult;
            wo[(g0 + 1) * D + d_a] = o[mt][nt][1] * v_mult;
            wo[(g0 + 1) * D + d_b] = o[mt][nt][3] * v_mult;
          }
          if (r == 0) {
            wml[g0 * 2] = m_run[nt][0];
            wml[g0 * 2 + 1] = l_run[nt][0];
            wml[(g0 + 1) * 2] = m_run[nt][1];
            wml[(g0 + 1) * 2 + 1] = l_run[nt][1];
          }
        }
      }
      if (k != nk - 1) {
        // next unit: next head of this sequence, or the next non-empty sequence
        if (++ch == Hkv) {
          ch = 0;
          do { ++cb; } while (sQ[cb + 1] == sQ[cb]);
        }
        clt = 0;
        ctiles = sQ[cb + 1] - sQ[cb];
        seg_lt0 = 0;
        seg_slot = 1;
        begin_unit();
      }
    }
  }
  if (!healthy) {
    for (int s = 0; s < NS && s < nk; ++s) {
      const int klast = s + ((nk - 1 - s) / NS) * NS;
      mbar_wait(wbar0 + 8 * s, static_cast<uint32_t>((klast / NS) & 1), nullptr);
    }
  }
  allow_next_grid();
}

// ----------------------------------------------------------------------------
// Stream-K fix-up: merge the pieces of every unit that range boundaries cut,
// and write zeros for empty sequences.  One CTA (4 warps) per (sequence, KV
// head); the pieces are split among the warps, each lane owning float4 columns
// of the [heads x D] accumulator, and the warps are summed in shared memory.
// ----------------------------------------------------------------------------
template <int D, int NT>
__global__ void __launch_bounds__(128) streamk_fixup_kernel(const DecodeParams p) {
  constexpr int GP = 8 * NT;
  constexpr int K4 = GP * D / 128;        // float4 columns per lane
  __shared__ float s_red[4][GP];
  __shared__ float s_M[GP], s_L[GP];
  __shared__ __align__(16) float s_acc[4][GP * D];
  wait_prior_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;
  const int b = u / p.num_kv_heads, h = u - b * p.num_kv_heads;
  const int G = p.group;
  const int Qb = p.ws_q[b], tb = p.ws_q[b + 1] - Qb;
  const int64_t row0 = static_cast<int64_t>(b) * p.num_q_heads + static_cast<int64_t>(h) * G;
  if (tb == 0) {
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) p.out[row0 * D + i] = 0.f;
    return;
  }
  const int64_t T = static_cast<int64_t>(p.num_kv_heads) * p.ws_q[p.batch];
  const int64_t W = streamk_workers_used(T, p.workers);
  const int64_t a = static_cast<int64_t>(p.num_kv_heads) * Qb + static_cast<int64_t>(h) * tb;
  const int64_t e = a + tb;
  const int64_t wa = ((a + 1) * W - 1) / T, wb = (e * W - 1) / T;
  if (wa == wb) return;  // one warp held the whole unit and wrote it
  const int n = static_cast<int>(wb - wa + 1);
  const bool first_is_second_piece = (wa * T / W) < a;   // unit starts inside wa's range
  auto piece = [&](int i) -> int64_t {
    return (wa + i) * 2 + ((i == 0 && first_is_second_piece) ? 1 : 0);
  };

  // per head: M = max m over pieces, then L = sum 2^(m - M) l
  float red[GP];
#pragma unroll
  for (int g = 0; g < GP; ++g) red[g] = -CUDART_INF_F;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float* ml = p.ws_ml + piece(i) * GP * 2;
#pragma unroll
    for (int g = 0; g < GP; ++g) red[g] = fmaxf(red[g], ml[2 * g]);
  }
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    float v = red[g];
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, sh));
    if (lane == 0) s_red[warp][g] = v;
  }
  __syncthreads();
  if (threadIdx.x < GP)
    s_M[threadIdx.x] = fmaxf(fmaxf(s_red[0][threadIdx.x], s_red[1][threadIdx.x]),
                             fmaxf(s_red[2][threadIdx.x], s_red[3][threadIdx.x]));
  __syncthreads();
#pragma unroll
  for (int g = 0; g < GP; ++g) red[g] = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float* ml = p.ws_ml + piece(i) * GP * 2;
#pragma unroll
    for (int g = 0; g < GP; ++g) red[g] += fast_exp2(ml[2 * g] - s_M[g]) * ml[2 * g + 1];
  }
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    float v = red[g];
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) v += __shfl_xor_sync(kFull, v, sh);
    if (lane == 0) s_red[warp][g] = v;
  }
  __syncthreads();
  if (threadIdx.x < GP)
    s_L[threadIdx.x] = s_red[0][threadIdx.x] + s_red[1][threadIdx.x] + s_red[2][threadIdx.x] +
                       s_red[3][threadIdx.x];
  __syncthreads();

  // weighted sum of the accumulators: warp w takes pieces w, w+4, ...
  float4 acc[K4];
#pragma unroll
  for (int k = 0; k < K4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = warp; i < n; i += 4) {
    const int64_t pc = piece(i);
    const float* ml = p.ws_ml + pc * GP * 2;
    const float4* src = reinterpret_cast<const float4*>(p.ws_o + pc * GP * D);
#pragma unroll
    for (int k = 0; k < K4; ++k) {
      const int c = lane + 32 * k;        // float4 column: floats 4c..4c+3
      const int g = (4 * c) / D;
      const float wt = fast_exp2(ml[2 * g] - s_M[g]);
      const float4 x = src[c];
      acc[k].x += wt * x.x;
      acc[k].y += wt * x.y;
      acc[k].z += wt * x.z;
      acc[k].w += wt * x.w;
    }
  }
#pragma unroll
  for (int k = 0; k < K4; ++k)
    reinterpret_cast<float4*>(s_acc[warp])[lane + 32 * k] = acc[k];
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D;
    const float v = s_acc[0][idx] + s_acc[1][idx] + s_acc[2][idx] + s_acc[3][idx];
    p.out[row0 * D + idx] = v / s_L[g];
  }
}

// Persistent-grid shape of the stream-K kernel per (D, dtype): warps per CTA,
// pipeline stages per warp, CTAs per SM.
template <int D, bool FP8>
struct StreamKShape {
  static constexpr int NW = 4;
  static constexpr int NS = (24576 / Layout<D, FP8>::STAGEB) > 8 ? 8 : (24576 / Layout<D, FP8>::STAGEB);
  static constexpr int MINB = 2;
  static int workers(int sms) { return MINB * sms * NW; }
};

template <int D, bool FP8>
int streamk_smem_bytes_t(int batch) {
  using L = Layout<D, FP8>;
  using Shape = StreamKShape<D, FP8>;
  return Shape::NW * Shape::NS * L::STAGEB + Shape::NW * Shape::NS * 8 + 4 * (batch + 1) + 1024;
}

template <int D, bool FP8, int NT>
cudaError_t launch_split_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           cudaStream_t stream) {
  auto kern = decode_split_kernel<D, FP8, NT>;
  constexpr int smem = Smem<D, FP8, NT>::TOTAL;
  static int configured[64] = {};
  cudaError_t e = set_smem_once(kern, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.max_splits, p.num_kv_heads, p.batch), dim3(kDecodeWarps * 32),
                    smem, stream, tk, tv, p);
}

template <int D, bool FP8, int NT>
cudaError_t launch_streamk_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             cudaStream_t stream) {
  using Shape = StreamKShape<D, FP8>;
  auto kern = decode_streamk_kernel<D, FP8, NT, Shape::NW, Shape::NS, Shape::MINB>;
  const int smem = streamk_smem_bytes_t<D, FP8>(p.batch);
  static int configured[64] = {};
  cudaError_t e = set_smem_once(kern, streamk_smem_bytes_t<D, FP8>(kMaxStreamKBatch), configured);
  if (e != cudaSuccess) return e;
  const int ctas = p.workers / Shape::NW;
  return launch_pdl(kern, dim3(ctas), dim3(Shape::NW * 32), smem, stream, tk, tv, p);
}

}  // namespace

int decode_smem_bytes(int head_dim, int cache_dtype, int n_tiles8) {
  const bool fp8 = cache_dtype == kE4M3;
  if (head_dim == 128) {
    if (fp8) return n_tiles8 == 1 ? Smem<128, true, 1>::TOTAL : Smem<128, true, 2>::TOTAL;
    return n_tiles8 == 1 ? Smem<128, false, 1>::TOTAL : Smem<128, false, 2>::TOTAL;
  }
  if (fp8) return n_tiles8 == 1 ? Smem<64, true, 1>::TOTAL : Smem<64, true, 2>::TOTAL;
  return n_tiles8 == 1 ? Smem<64, false, 1>::TOTAL : Smem<64, false, 2>::TOTAL;
}

int streamk_grid_workers(int head_dim, int cache_dtype, int sms) {
  const bool fp8 = cache_dtype == kE4M3;
  if (head_dim == 128)
    return fp8 ? StreamKShape<128, true>::workers(sms) : StreamKShape<128, false>::workers(sms);
  return fp8 ? StreamKShape<64, true>::workers(sms) : StreamKShape<64, false>::workers(sms);
}

cudaError_t launch_decode_split(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t stream) {
  const bool fp8 = p.cache_dtype == kE4M3;
  const int nt = p.group > 8 ? 2 : 1;
  if (p.mode == kModeStreamK) {
    if (p.head_dim == 128) {
      if (fp8) return nt == 1 ? launch_streamk_t<128, true, 1>(p, tk, tv, stream)
                              : launch_streamk_t<128, true, 2>(p, tk, tv, stream);
      return nt == 1 ? launch_streamk_t<128, false, 1>(p, tk, tv, stream)
                     : launch_streamk_t<128, false, 2>(p, tk, tv, stream);
    }
    if (fp8) return nt == 1 ? launch_streamk_t<64, true, 1>(p, tk, tv, stream)
                            : launch_streamk_t<64, true, 2>(p, tk, tv, stream);
    return nt == 1 ? launch_streamk_t<64, false, 1>(p, tk, tv, stream)
                   : launch_streamk_t<64, false, 2>(p, tk, tv, stream);
  }
  if (p.head_dim == 128) {
    if (fp8) return nt == 1 ? launch_split_t<128, true, 1>(p, tk, tv, stream)
                            : launch_split_t<128, true, 2>(p, tk, tv, stream);
    return nt == 1 ? launch_split_t<128, false, 1>(p, tk, tv, stream)
                   : launch_split_t<128, false, 2>(p, tk, tv, stream);
  }
  if (fp8) return nt == 1 ? launch_split_t<64, true, 1>(p, tk, tv, stream)
                          : launch_split_t<64, true, 2>(p, tk, tv, stream);
  return nt == 1 ? launch_split_t<64, false, 1>(p, tk, tv, stream)
                 : launch_split_t<64, false, 2>(p, tk, tv, stream);
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.batch) * p.num_q_heads;
  if (rows == 0) return cudaSuccess;
  if (p.mode == kModeStreamK) {
    const int units = p.batch * p.num_kv_heads;
    const bool nt2 = p.group > 8;
    if (p.head_dim == 128)
      return nt2 ? launch_pdl(streamk_fixup_kernel<128, 2>, dim3(units), dim3(128), 0, stream, p)
                 : launch_pdl(streamk_fixup_kernel<128, 1>, dim3(units), dim3(128), 0, stream, p);
    return nt2 ? launch_pdl(streamk_fixup_kernel<64, 2>, dim3(units), dim3(128), 0, stream, p)
               : launch_pdl(streamk_fixup_kernel<64, 1>, dim3(units), dim3(128), 0, stream, p);
  }
  if (p.max_splits + p.extra_count <= 1 && !p.force_partial) return cudaSuccess;
  if (p.force_partial && p.slots_per_row <= 8) {
    // a cascade call: every slot written but suffix splits past a row's count
    const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
    const bool d128 = p.head_dim == 128;
    if (p.slots_per_row <= 4)
      return d128 ? launch_pdl(combine_cascade_kernel<128, 4>, dim3(blocks), dim3(128), 0, stream, p)
                  : launch_pdl(combine_cascade_kernel<64, 4>, dim3(blocks), dim3(128), 0, stream, p);
    return d128 ? launch_pdl(combine_cascade_kernel<128, 8>, dim3(blocks), dim3(128), 0, stream, p)
                : launch_pdl(combine_cascade_kernel<64, 8>, dim3(blocks), dim3(128), 0, stream, p);
  }
  if (p.max_splits + p.extra_count <= 8) {
    const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
    if (p.head_dim == 128) return launch_pdl(combine_rows_kernel<128>, dim3(blocks), dim3(128), 0, stream, p);
    return launch_pdl(combine_rows_kernel<64>, dim3(blocks), dim3(128), 0, stream, p);
  }
  const unsigned blocks = static_cast<unsigned>(rows);
  if (p.head_dim == 128) return launch_pdl(combine_kernel<128>, dim3(blocks), dim3(128), 0, stream, p);
  return launch_pdl(combine_kernel<64>, dim3(blocks), dim3(128), 0, stream, p);
}

}  // namespace pkv
