// Multi-token query paged attention: q_len new tokens per sequence (a chunk of
// a chunked prefill run beside decode steps, [SC] "LLM inference: prefill,
// decode, KV cache", "9. Failure modes and limitations", item 3; or the tokens
// a draft model proposed, checked in one pass, [SC] "7. Practical
// applications", item 3), each attending the sequence's cached tokens and the
// new tokens up to itself.  Query i of sequence b sits at position
// ctx_b - q_len + i (context_lens counts the new tokens, which are already
// appended) and attends tokens [0, ctx_b - q_len + i].
//
// Design (GB300):
//  * Rows are (query token i, head g) pairs of one KV head: R = q_len * G of
//    them share every K/V byte.  A CTA takes up to 16 rows of one (sequence,
//    KV head) (more go to the persistent tcgen05 kernel of cascade.cu) over
//    one split of `split_tokens` tokens, streamed in 64-token tiles, block
//    ids of the split staged in shared memory.
//  * All four warps hold the same 16 rows; warp w takes tokens 16w..16w+15
//    of every tile, loading them itself (one 16-token TMA box per lane, K
//    and V, 128B-swizzled, into its part of a two-stage ring, on barriers of
//    its own) and refilling its slot as soon as it has read it, so no warp
//    waits for another.  The warps merge (m, l, acc) through shared memory
//    at the end.  (The row-group x token-lane shapes for 17-64 rows are in
//    the template but not instantiated.)
//  * S = Q K^T and O += P V are mma.sync m16n8k16 tiles (bf16, fp32
//    accumulate); P is fed as a bf16 hi + lo pair.  The causal limit is per
//    row; V rows past the end of the sequence are zeroed in registers.
//  * Splits write (acc, m, l) partials that the decode combine kernel merges
//    (rows (b, i, hq) flatten to b * (q_len * H_q) + i * H_q + hq).

#include "decode_common.cuh"

namespace pkv {
namespace {

// Shared-memory stages per CTA and CTAs per SM: with two or four token lanes
// (R <= 32 rows) a CTA is light enough on registers that two stages let three
// CTAs share an SM.
template <int TL>
struct MqShape {
  static constexpr int NS = TL >= 2 ? 2 : 3;
  static constexpr int MINB = TL >= 2 ? 3 : 2;
};

template <int D, int TL>
__global__ void __launch_bounds__(128, MqShape<TL>::MINB)
    multi_query_kernel(const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using L = Layout<D, false>;
  constexpr int KS = D / 16;
  constexpr int NSUB = kMultiQueryTile / kTileTokens;  // sub-tiles per tile
  static_assert(2 * NSUB * L::NBOX <= 32, "one TMA box per lane");
  constexpr int NSW = NSUB / TL;                       // sub-tiles per warp per tile
  constexpr int RG = 4 / TL;                           // row groups
  constexpr int RPC = 16 * RG;                         // rows per CTA
  constexpr int STAGE = NSUB * L::STAGEB;
  constexpr int NS = MqShape<TL>::NS;
  constexpr int DP = D + 4;
  static_assert(4 * 16 * DP * 4 + 4 * 16 * 2 * 4 <= NS * STAGE, "merge buffer fits the stages");
  static_assert(TL == 4, "each warp loads and reads its own 16-token sub-tile of every tile");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, j = lane & 3;
  const int rg = warp / TL, tl = warp % TL;
  const int G = p.group, QL = p.q_len;
  const int R = QL * G;
  const int nrb = (R + RPC - 1) / RPC;
  const int h = blockIdx.y / nrb, rblk = blockIdx.y - (blockIdx.y / nrb) * nrb;
  const int b = blockIdx.z, split = blockIdx.x;
  const int H_q = p.num_q_heads;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * STAGE);  // [NS][4]: per stage and warp
  int* s_blk = reinterpret_cast<int*>(full + 4 * NS);
  const uint32_t stage0 = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 4 * NS; ++s) mbar_init(smem_u32(full + s), 1);
    fence_mbar_init();
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  wait_prior_grid();

  const int ctx_raw = p.context_lens[b];
  const int ctx = clamp_ctx(p, ctx_raw);
  if (ctx != ctx_raw && split == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    record_error(p.err, kDevErrContextLen);
  const int row0 = rblk * RPC;
  const int row_end = min(R, row0 + RPC);
  const int64_t b_rows = static_cast<int64_t>(b) * QL;  // first (b, i) row of the sequence
  const int t_begin = split * p.split_tokens;
  if (t_begin >= ctx) {
    if (ctx == 0 && split == 0) {  // empty sequence: zeros, nothing to combine
      for (int idx = threadIdx.x; idx < (row_end - row0) * D; idx += blockDim.x) {
        const int row = row0 + idx / D;
        const int64_t orow = (b_rows + row / G) * H_q + h * G + row % G;
        p.out[orow * D + idx % D] = 0.f;
      }
    }
    return;
  }
  const int nsplit = (ctx + p.split_tokens - 1) / p.split_tokens;
  // query row -> tokens it may attend: [0, lim)
  auto lim_of = [&](int row) { return min(ctx, ctx - QL + row / G + 1); };
  const int t_stop = min(min(ctx, t_begin + p.split_tokens), lim_of(row_end - 1));
  const int ntile = t_stop > t_begin ? (t_stop - t_begin + kMultiQueryTile - 1) / kMultiQueryTile : 0;
  const int nblk = ntile > 0 ? (t_stop - t_begin + p.block_size - 1) / p.block_size : 0;
  const int32_t* tbl = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
  for (int i = threadIdx.x; i < nblk && i < kMultiQueryMaxSplitBlocks; i += blockDim.x) {
    int phys = tbl[t_begin / p.block_size + i];
    if (phys < 0 || phys >= p.num_blocks) {
      record_error(p.err, kDevErrBlockId);
      phys = -1;  // outside the tensor map: the TMA unit fills zeros
    }
    s_blk[i] = phys;
  }
  __syncthreads();

  // Each warp loads its own 16-token sub-tile (warp w: tokens 16w..16w+15
  // of every 64-token tile) into its part of the stage, on a barrier of its
  // own, one TMA box per lane (K and V, per 128-byte column band), and
  // refills the slot as soon as it has read it: no warp waits for another,
  // and a tile's boxes are issued by four warps at once (one warp issuing
  // all of a tile's boxes held an SM to about 12-19 bytes per cycle).
  auto issue = [&](int k) {
    const int s = k % NS;
    const uint32_t dst = stage0 + s * STAGE + warp * L::STAGEB;
    const uint32_t bar = smem_u32(full + 4 * s + warp);
    if (lane == 0) {
      fence_proxy_async_smem();  // this warp's reads of the slot come before the copy
      mbar_arrive_expect_tx(bar, L::STAGEB);
    }
    __syncwarp();
    if (lane < 2 * L::NBOX) {
      const int v = lane / L::NBOX;
      const int bx = lane % L::NBOX;
      const int t = t_begin + k * kMultiQueryTile + warp * kTileTokens;
      // block of the split and token within it: the block size is 16 or 32,
      // so a shift and a mask instead of a run-time division per box
      const int bi = (t - t_begin) >> (p.block_size == 16 ? 4 : 5);
      const int phys = (t < t_stop && bi < kMultiQueryMaxSplitBlocks) ? s_blk[bi] : -1;
      tma_load_4d(dst + v * L::TILEB + bx * L::BOX_BYTES, v ? &tmap_v : &tmap_k, bar, bx * L::BOX_ELEMS,
                  t & (p.block_size - 1), h, phys);
    }
  };
  int issued = 0;
  for (; issued < ntile && issued < NS; ++issued) issue(issued);

  // query fragments (A operand of S = Q K^T): rows ra and rb = ra + 8
  const int ra = row0 + rg * 16 + r, rb = ra + 8;
  uint32_t qa[KS][4];
  {
    const uint16_t* q = static_cast<const uint16_t*>(p.q);
    const uint16_t* qra = ra < R ? q + ((b_rows + ra / G) * H_q + h * G + ra % G) * D : nullptr;
    const uint16_t* qrb = rb < R ? q + ((b_rows + rb / G) * H_q + h * G + rb % G) * D : nullptr;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = 16 * ks + 2 * j;
      qa[ks][0] = qra ? *reinterpret_cast<const uint32_t*>(qra + d0) : 0u;
      qa[ks][1] = qrb ? *reinterpret_cast<const uint32_t*>(qrb + d0) : 0u;
      qa[ks][2] = qra ? *reinterpret_cast<const uint32_t*>(qra + d0 + 8) : 0u;
      qa[ks][3] = qrb ? *reinterpret_cast<const uint32_t*>(qrb + d0 + 8) : 0u;
    }
  }
  const int lim_a = ra < R ? lim_of(ra) : 0;
  const int lim_b = rb < R ? lim_of(rb) : 0;

  const float qk_mult = p.qk_log2_scale;
  float m_a = -CUDART_INF_F, m_b = -CUDART_INF_F, l_a = 0.f, l_b = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  // ldmatrix lanes: K (tok 0-7,c)(tok 0-7,c+1)(tok 8-15,c)(tok 8-15,c+1);
  //                 V (tok 0-7,c)(tok 8-15,c)(tok 0-7,c+1)(tok 8-15,c+1)
  const int mq = lane >> 3;
  const int tok_k = (lane & 7) + (mq >> 1) * 8, ch_k = mq & 1;
  const int tok_v = (lane & 7) + (mq & 1) * 8, ch_v = mq >> 1;

  bool healthy = true;
  for (int k = 0; k < ntile; ++k) {
    const int s = k % NS;
    const uint32_t par = static_cast<uint32_t>((k / NS) & 1);
    const bool arrived = mbar_wait(smem_u32(full + 4 * s + warp), par, p.err);
    if (!__all_sync(kFull, arrived)) healthy = false;
    const uint32_t base = stage0 + s * STAGE;
    const int tile_t0 = t_begin + k * kMultiQueryTile;
    if (healthy) {
      // ---- S = Q K^T over this warp's sub-tiles: two 8-token n-tiles each
      float sc[2 * NSW][4];
#pragma unroll
      for (int nt = 0; nt < 2 * NSW; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int u = 0; u < NSW; ++u) {
        const int sub = tl + u * TL;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t Rk[4];
          ldsm_x4(base + sub * L::STAGEB + L::off(tok_k, 2 * ks + ch_k), Rk);
          mma_bf16_16816(sc[2 * u], qa[ks], Rk[0], Rk[1]);
          mma_bf16_16816(sc[2 * u + 1], qa[ks], Rk[2], Rk[3]);
        }
      }
      // ---- causal mask per row, online softmax (rows a: e = 0, 1; b: e = 2, 3)
      float mx_a = -CUDART_INF_F, mx_b = -CUDART_INF_F;
#pragma unroll
      for (int nt = 0; nt < 2 * NSW; ++nt) {
        const int tok = tile_t0 + 16 * (tl + (nt >> 1) * TL) + 8 * (nt & 1) + 2 * j;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int lim = e < 2 ? lim_a : lim_b;
          sc[nt][e] = (tok + (e & 1) < lim) ? sc[nt][e] * qk_mult : -CUDART_INF_F;
        }
        mx_a = fmaxf(mx_a, fmaxf(sc[nt][0], sc[nt][1]));
        mx_b = fmaxf(mx_b, fmaxf(sc[nt][2], sc[nt][3]));
      }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(kFull, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(kFull, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(kFull, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(kFull, mx_b, 2));
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float mu_a = (mn_a == -CUDART_INF_F) ? 0.f : mn_a;
      const float mu_b = (mn_b == -CUDART_INF_F) ? 0.f : mn_b;
      const float al_a = fast_exp2(m_a - mu_a), al_b = fast_exp2(m_b - mu_b);
      m_a = mn_a;
      m_b = mn_b;
      float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2 * NSW; ++nt) {  // packed f32x2 subtractions and multiplies below
        const float2 ea = __fadd2_rn(make_float2(sc[nt][0], sc[nt][1]), make_float2(-mu_a, -mu_a));
        const float2 eb = __fadd2_rn(make_float2(sc[nt][2], sc[nt][3]), make_float2(-mu_b, -mu_b));
        sc[nt][0] = fast_exp2(ea.x);
        sc[nt][1] = fast_exp2(ea.y);
        sc[nt][2] = fast_exp2(eb.x);
        sc[nt][3] = fast_exp2(eb.y);
        sum_a += sc[nt][0] + sc[nt][1];
        sum_b += sc[nt][2] + sc[nt][3];
      }
      l_a = l_a * al_a + sum_a;
      l_b = l_b * al_b + sum_b;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        const float2 u = __fmul2_rn(make_float2(o[nt][0], o[nt][1]), make_float2(al_a, al_a));
        const float2 w = __fmul2_rn(make_float2(o[nt][2], o[nt][3]), make_float2(al_b, al_b));
        o[nt][0] = u.x;
        o[nt][1] = u.y;
        o[nt][2] = w.x;
        o[nt][3] = w.y;
      }
      // ---- O += P V, one 16-token k-step per sub-tile
#pragma unroll
      for (int u = 0; u < NSW; ++u) {
        const int sub = tl + u * TL;
        uint32_t ph[4], pl[4];
        const float* c0 = sc[2 * u];
        const float* c1 = sc[2 * u + 1];
        ph[0] = pack_bf16x2(c0[0], c0[1]);
        ph[1] = pack_bf16x2(c0[2], c0[3]);
        ph[2] = pack_bf16x2(c1[0], c1[1]);
        ph[3] = pack_bf16x2(c1[2], c1[3]);
        pl[0] = pack_bf16x2(c0[0] - bf16lo_to_f32(ph[0]), c0[1] - bf16hi_to_f32(ph[0]));
        pl[1] = pack_bf16x2(c0[2] - bf16lo_to_f32(ph[1]), c0[3] - bf16hi_to_f32(ph[1]));
        pl[2] = pack_bf16x2(c1[0] - bf16lo_to_f32(ph[2]), c1[1] - bf16hi_to_f32(ph[2]));
        pl[3] = pack_bf16x2(c1[2] - bf16lo_to_f32(ph[3]), c1[3] - bf16hi_to_f32(ph[3]));
        // V rows at or past the end of the sequence may hold anything (NaN
        // included): zero them in the fragments, P is already 0 there.
        const int vvalid = ctx - (tile_t0 + 16 * sub);
        const uint32_t keep_lo0 = (2 * j < vvalid) ? 0x0000FFFFu : 0u;
        const uint32_t keep_hi0 = (2 * j + 1 < vvalid) ? 0xFFFF0000u : 0u;
        const uint32_t keep_lo1 = (2 * j + 8 < vvalid) ? 0x0000FFFFu : 0u;
        const uint32_t keep_hi1 = (2 * j + 9 < vvalid) ? 0xFFFF0000u : 0u;
        const uint32_t keep0 = keep_lo0 | keep_hi0, keep1 = keep_lo1 | keep_hi1;
        const uint32_t vt = base + sub * L::STAGEB + L::TILEB;
#pragma unroll
        for (int dp = 0; dp < KS; ++dp) {
          uint32_t Rv[4];
          ldsm_x4_trans(vt + L::off(tok_v, 2 * dp + ch_v), Rv);
          Rv[0] &= keep0;
          Rv[1] &= keep1;
          Rv[2] &= keep0;
          Rv[3] &= keep1;
          mma_bf16_16816(o[2 * dp], ph, Rv[0], Rv[1]);
          mma_bf16_16816(o[2 * dp], pl, Rv[0], Rv[1]);
          mma_bf16_16816(o[2 * dp + 1], ph, Rv[2], Rv[3]);
          mma_bf16_16816(o[2 * dp + 1], pl, Rv[2], Rv[3]);
        }
      }
    }
    // ---- this warp has read its part of the slot: refill it
    __syncwarp();
    if (healthy && k + NS < ntile) issue(issued++);
  }
  if (!healthy && lane == 0) {
    // a copy of this warp's may still be landing: one more bounded wait each
    for (int kk = issued > NS ? issued - NS : 0; kk < issued; ++kk)
      mbar_wait(smem_u32(full + 4 * (kk % NS) + warp), static_cast<uint32_t>((kk / NS) & 1), nullptr);
  }
  allow_next_grid();

  // ---- row sums over the quad; stage per-warp results for the lane merge
  l_a += __shfl_xor_sync(kFull, l_a, 1);
  l_a += __shfl_xor_sync(kFull, l_a, 2);
  l_b += __shfl_xor_sync(kFull, l_b, 1);
  l_b += __shfl_xor_sync(kFull, l_b, 2);
  __syncthreads();  // every warp is done with the stages
  float* s_o = reinterpret_cast<float*>(smem);          // [4 warps][16][DP]
  float* s_ml = s_o + 4 * 16 * DP;                      // [4 warps][16][2]
  {
    float* wo = s_o + warp * 16 * DP;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      *reinterpret_cast<float2*>(wo + r * DP + 8 * nt + 2 * j) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(wo + (r + 8) * DP + 8 * nt + 2 * j) = make_float2(o[nt][2], o[nt][3]);
    }
    if (j == 0) {
      float* ml = s_ml + warp * 32;
      ml[2 * r] = m_a;
      ml[2 * r + 1] = l_a;
      ml[2 * (r + 8)] = m_b;
      ml[2 * (r + 8) + 1] = l_b;
    }
  }
  __syncthreads();

  const bool direct = nsplit == 1;
  const int64_t S_max = p.slots_per_row;
  for (int idx = threadIdx.x; idx < RPC * D; idx += blockDim.x) {
    const int lr = idx / D, d = idx - (idx / D) * D;
    const int row = row0 + lr;
    if (row >= R) break;
    const int g0 = lr >> 4, loc = lr & 15;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int t = 0; t < TL; ++t) M = fmaxf(M, s_ml[(g0 * TL + t) * 32 + 2 * loc]);
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int t = 0; t < TL; ++t) {
      const int w = g0 * TL + t;
      const float mw = s_ml[w * 32 + 2 * loc];
      const float wt = (mw == -CUDART_INF_F) ? 0.f : fast_exp2(mw - M);
      acc += wt * s_o[(w * 16 + loc) * DP + d];
      lsum += wt * s_ml[w * 32 + 2 * loc + 1];
    }
    const int64_t orow = (b_rows + row / G) * H_q + h * G + row % G;
    if (direct) {
      p.out[orow * D + d] = lsum > 0.f ? acc / lsum : 0.f;
    } else {
      const int64_t slot = orow * S_max + split;
      p.ws_o[slot * D + d] = acc;
      if (d == 0) {
        p.ws_ml[slot * 2] = M;
        p.ws_ml[slot * 2 + 1] = lsum;
      }
    }
  }
}

template <int D, int TL>
cudaError_t launch_mq_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                        cudaStream_t stream) {
  auto kern = multi_query_kernel<D, TL>;
  const int stage = (kMultiQueryTile / kTileTokens) * 2 * kTileTokens * D * 2;
  const int smem = MqShape<TL>::NS * stage + 4 * MqShape<TL>::NS * 8 + kMultiQueryMaxSplitBlocks * 4 + 1024;
  static int configured[64] = {};
  cudaError_t e = set_smem_once(kern, smem, configured);
  if (e != cudaSuccess) return e;
  const int rows = p.q_len * p.group;
  const int nrb = (rows + 16 * (4 / TL) - 1) / (16 * (4 / TL));
  return launch_pdl(kern, dim3(p.max_splits, p.num_kv_heads * nrb, p.batch), dim3(128), smem, stream,
                    tk, tv, p);
}

}  // namespace

cudaError_t launch_multi_query(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream) {
  // the library sends this kernel up to 16 rows (kMultiQueryTcRows): four
  // token lanes; the two- and one-lane shapes are not instantiated
  if (multi_query_lanes(p.q_len * p.group) != 4) return cudaErrorInvalidValue;
  if (p.head_dim == 128) return launch_mq_t<128, 4>(p, tk, tv, stream);
  return launch_mq_t<64, 4>(p, tk, tv, stream);
}

}  // namespace pkv
