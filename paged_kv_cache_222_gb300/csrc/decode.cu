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

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kE4M3 = 2;

template <int D, bool FP8>
struct Layout {
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int ROWB = D * ESZ;                    // bytes of one token row
  static constexpr int BOXB = ROWB < 128 ? ROWB : 128;    // row bytes per TMA box
  static constexpr int NBOX = ROWB / BOXB;                // boxes per tile
  static constexpr int BOX_ELEMS = BOXB / ESZ;
  static constexpr int CPB = BOXB / 16;                   // 16-byte chunks per box row
  static constexpr int BOX_BYTES = kTileTokens * BOXB;
  static constexpr int TILEB = kTileTokens * ROWB;        // K (or V) bytes of one tile
  static constexpr int STAGEB = 2 * TILEB;                // K + V
  static constexpr int NS = (24576 / STAGEB) > 8 ? 8 : (24576 / STAGEB);
  static constexpr int PIPE_BYTES = kDecodeWarps * NS * STAGEB;

  // Byte offset, inside a tile, of 16-byte chunk c of token row t as the TMA
  // unit stores it: 128-byte rows swizzled by XOR of the chunk with (t mod 8),
  // 64-byte rows by XOR with ((t / 2) mod 4).
  __device__ static __forceinline__ uint32_t off(int t, int c) {
    const int box = c / CPB;
    const int cc = c % CPB;
    const int sw = (BOXB == 128) ? (t & 7) : ((t >> 1) & 3);
    return static_cast<uint32_t>(box * BOX_BYTES + t * BOXB + ((cc ^ sw) << 4));
  }
};

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

  // ---- S^T = K . Q^T  (rows: tokens, cols: the group's query heads)
  float s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;

  if constexpr (!FP8) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      ldsm_x4(stage + L::off(tok_a, 2 * ks + chunk_a), a);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(s[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
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
        for (int nt = 0; nt < NT; ++nt)
          mma_f16_16816(s[nt], a, qb[2 * pk + q2][nt][0], qb[2 * pk + q2][nt][1]);
      }
    }
  }

  // ---- online softmax (log2 domain); lane holds tokens r, r+8 x heads 2j, 2j+1
  uint32_t pb_hi[NT][2], pb_lo[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float x0 = s[nt][0] * qk_mult, x1 = s[nt][1] * qk_mult;
    float x2 = s[nt][2] * qk_mult, x3 = s[nt][3] * qk_mult;
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
    const float p0 = fast_exp2(x0 - mu0), p1 = fast_exp2(x1 - mu1);
    const float p2 = fast_exp2(x2 - mu0), p3 = fast_exp2(x3 - mu1);
    l_run[nt][0] = l_run[nt][0] * al0 + (p0 + p2);
    l_run[nt][1] = l_run[nt][1] * al1 + (p1 + p3);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      o[mt][nt][0] *= al0;
      o[mt][nt][1] *= al1;
      o[mt][nt][2] *= al0;
      o[mt][nt][3] *= al1;
    }
    // P rows (token r | token r+8) x (heads 2j, 2j+1) as hi + lo 16-bit pairs,
    // transposed in registers into the B fragment of the P.V product.
    uint32_t h0, h1, l0, l1;
    if constexpr (!FP8) {
      h0 = pack_bf16x2(p0, p1);
      h1 = pack_bf16x2(p2, p3);
      l0 = pack_bf16x2(p0 - bf16lo_to_f32(h0), p1 - bf16hi_to_f32(h0));
      l1 = pack_bf16x2(p2 - bf16lo_to_f32(h1), p3 - bf16hi_to_f32(h1));
    } else {
      h0 = pack_f16x2(p0, p1);
      h1 = pack_f16x2(p2, p3);
      l0 = pack_f16x2(p0 - f16lo_to_f32(h0), p1 - f16hi_to_f32(h0));
      l1 = pack_f16x2(p2 - f16lo_to_f32(h1), p3 - f16hi_to_f32(h1));
    }
    pb_hi[nt][0] = movmatrix_trans(h0);
    pb_hi[nt][1] = movmatrix_trans(h1);
    pb_lo[nt][0] = movmatrix_trans(l0);
    pb_lo[nt][1] = movmatrix_trans(l1);
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
        for (int nt = 0; nt < NT; ++nt) {
          mma_f16_16816(o[mt][nt], a, pb_hi[nt][0], pb_hi[nt][1]);
          mma_f16_16816(o[mt][nt], a, pb_lo[nt][0], pb_lo[nt][1]);
        }
      }
    }
  }
}

// ----------------------------------------------------------------------------
// Context length as both kernels see it (clamped to what the grid and the table
// can hold; the violation itself is recorded by the split kernel).
// ----------------------------------------------------------------------------
__device__ __forceinline__ int clamp_ctx(const DecodeParams& p, int ctx) {
  const int64_t table_cap = static_cast<int64_t>(p.max_blocks) * p.block_size;
  const int lim = static_cast<int>(table_cap < p.max_ctx ? table_cap : p.max_ctx);
  return ctx < 0 ? 0 : (ctx > lim ? lim : ctx);
}

template <int D, bool FP8, int NT>
__global__ void __launch_bounds__(kDecodeWarps * 32, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using L = Layout<D, FP8>;
  using S = Smem<D, FP8, NT>;
  constexpr int NW = kDecodeWarps;
  constexpr int NS = L::NS;
  constexpr int KS = D / 16;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, j = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = p.group;

  const int ctx_raw = p.context_lens[b];
  const int ctx = clamp_ctx(p, ctx_raw);
  if (ctx != ctx_raw && split == 0 && h == 0 && threadIdx.x == 0)
    record_error(p.err, kDevErrContextLen);
  const int64_t row0 = static_cast<int64_t>(b) * p.num_q_heads + static_cast<int64_t>(h) * G;

  const int t_begin = split * p.split_tokens;
  if (t_begin >= ctx) {
    if (ctx == 0 && split == 0) {
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) p.out[row0 * D + i] = 0.f;
    }
    return;
  }
  const int t_end = min(ctx, t_begin + p.split_tokens);
  const int n_tiles = (t_end - t_begin + kTileTokens - 1) / kTileTokens;
  const int nsplit = (ctx + p.split_tokens - 1) / p.split_tokens;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
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

  // ---- query fragments (B operand of S^T = K . Q^T): heads 8nt + r, zero past G
  uint32_t qb[KS][NT][2];
  {
    const uint16_t* qbase = static_cast<const uint16_t*>(p.q) + row0 * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = 8 * nt + r;
      const uint16_t* qg = qbase + static_cast<int64_t>(g) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
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

  // ---- this warp's tiles: k-th tile covers tokens t_begin + 16 (warp + k NW)
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
    const uint32_t dst = wstage0 + s * L::STAGEB;
    const uint32_t bar = wbar0 + 8 * s;
    const int t = t_begin + kTileTokens * (warp + k * NW);
    const int tok0 = t % p.block_size;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, L::STAGEB);
#pragma unroll
    for (int bx = 0; bx < L::NBOX; ++bx)
      tma_load_4d(dst + bx * L::BOX_BYTES, &tmap_k, bar, bx * L::BOX_ELEMS, tok0, h, phys);
#pragma unroll
    for (int bx = 0; bx < L::NBOX; ++bx)
      tma_load_4d(dst + L::TILEB + bx * L::BOX_BYTES, &tmap_v, bar, bx * L::BOX_ELEMS, tok0, h,
                  phys);
  };

  int phys_reg = load_phys(0);
  const int npro = nk < NS ? nk : NS;
  for (int k = 0; k < npro; ++k) {
    const int ph = __shfl_sync(kFull, phys_reg, k);
    if (lane == 0) issue(k, ph);
  }

  float m_run[NT][2], l_run[NT][2], o[KS][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
  }

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
      if (valid < kTileTokens) {
        // rows past the end of the sequence may hold anything (NaN included):
        // zero them in V so that P = 0 times V stays 0 in the MMA
        uint8_t* vt = smem + (stage - smem_u32(smem)) + L::TILEB;
        const int nchunks = (kTileTokens - valid) * (L::ROWB / 16);
        for (int c = lane; c < nchunks; c += 32) {
          const int tr = valid + c / (L::ROWB / 16);
          const int cc = c % (L::ROWB / 16);
          *reinterpret_cast<uint4*>(vt + L::off(tr, cc)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
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

  // ---- finish the per-lane sums, merge the warps through shared memory
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
        if constexpr (!FP8) {
          d_a = 16 * mt + r;
          d_b = d_a + 8;
        } else {
          d_a = 16 * mt + 2 * r;
          d_b = d_a + 1;
        }
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

  const bool direct = (nsplit == 1);
  const int64_t S_max = p.max_splits;
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
// LSE combine: out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
// One warp per (sequence, query head); each lane owns D/32 consecutive dims.
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p) {
  constexpr int V = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(p.batch) * p.num_q_heads) return;
  const int b = static_cast<int>(row / p.num_q_heads);
  const int ctx = clamp_ctx(p, p.context_lens[b]);
  const int nsplit = (ctx + p.split_tokens - 1) / p.split_tokens;
  if (nsplit <= 1) return;  // written by the split kernel
  const int64_t S_max = p.max_splits;
  const float* ml = p.ws_ml + row * S_max * 2;
  const float* wo = p.ws_o + row * S_max * D;
  float M = -CUDART_INF_F;
  for (int i = lane; i < nsplit; i += 32) M = fmaxf(M, ml[2 * i]);
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, sh));
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  float lsum = 0.f;
  for (int i = 0; i < nsplit; ++i) {
    const float w = fast_exp2(ml[2 * i] - M);
    lsum += w * ml[2 * i + 1];
    const float* src = wo + static_cast<int64_t>(i) * D + lane * V;
    if constexpr (V == 4) {
      const float4 x = *reinterpret_cast<const float4*>(src);
      acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(src);
      acc[0] += w * x.x; acc[1] += w * x.y;
    }
  }
  const float inv = 1.f / lsum;
  float* dst = p.out + row * D + lane * V;
  if constexpr (V == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
  }
}

template <int D, bool FP8, int NT>
cudaError_t launch_split_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           cudaStream_t stream) {
  auto kern = decode_split_kernel<D, FP8, NT>;
  constexpr int smem = Smem<D, FP8, NT>::TOTAL;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  dim3 grid(p.max_splits, p.num_kv_heads, p.batch);
  kern<<<grid, kDecodeWarps * 32, smem, stream>>>(tk, tv, p);
  return cudaGetLastError();
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

cudaError_t launch_decode_split(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t stream) {
  const bool fp8 = p.cache_dtype == kE4M3;
  const int nt = p.group > 8 ? 2 : 1;
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
  if (rows == 0 || p.max_splits <= 1) return cudaSuccess;
  const int blocks = static_cast<int>((rows + 3) / 4);
  if (p.head_dim == 128)
    combine_kernel<128><<<blocks, 128, 0, stream>>>(p);
  else
    combine_kernel<64><<<blocks, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
