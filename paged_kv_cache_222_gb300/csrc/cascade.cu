// Cascade (shared-prefix) decode: the prefix kernel.  When every sequence of
// the batch starts with the same `prefix_len` tokens held in the same physical
// blocks (shared by reference: [FN] "Sub-Millisecond Token Scheduling...",
// "Paged KV-Cache with Radix Tree Prefix Cache", copy-on-write prefix blocks),
// the prefix part of decode attention is one dense product per KV head,
//   S = Q_h K_prefix^T,  Q_h = the B*G query rows (b, g) of KV head h,
// followed by the online softmax and P V_prefix.  Each CTA takes 128 query
// rows of one KV head over one range of prefix tokens and writes (acc, m, l)
// per row into the workspace slot reserved for its range; the combine kernel
// of decode.cu merges those with the private-suffix splits.

#include "decode_common.cuh"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

// ----------------------------------------------------------------------------
// Cascade prefix kernel on the 5th-generation tensor cores (tcgen05 + TMEM).
// 128 query rows per CTA, one row per thread (= one TMEM lane):
//   TMEM columns   [0, D/2)   Q rows, bf16 pairs (A operand of S = Q K^T)
//                  [64, 128)  S (fp32), then P = 2^(s - m) as bf16 hi | lo
//                             (A operand of O += P V; P aliases S)
//                  [128, 128 + D)  O (fp32 accumulator)
//   shared memory  3 stages of 64-token K and V tiles, TMA-loaded with the
//                  128-byte swizzle: K read as a K-major B operand, V as an
//                  MN-major B operand, through sm_100 matrix descriptors.
// Thread 0 issues the MMAs and commits them to mbarriers; every thread reads
// its S row, keeps a lazy running max (O in TMEM is rescaled only when the
// max grows by more than 2^8, so P stays <= 256) and writes its P row back.
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128, 2)
    cascade_prefix_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using L = Layout<D, false>;
  constexpr int M = 128;
  constexpr int NKEY = kCascadeTile;
  constexpr int NSUB = NKEY / kTileTokens;
  constexpr int HALVES = D / 64;                 // 128-byte d-halves of a row
  constexpr int HALF_BYTES = NKEY * 128;         // one d-half of a 64-key tile
  constexpr int KREG = HALVES * HALF_BYTES;      // K (or V) tile
  constexpr int STAGE = 2 * KREG;
  constexpr int NS = 3;
  constexpr int kMaxPrefixBlocks = 1024;
  constexpr uint32_t TCOLS = 256;
  constexpr uint32_t COL_Q = 0, COL_S = 64, COL_PHI = 64, COL_PLO = 96, COL_O = 128;
  constexpr uint32_t IDESC_S = idesc_bf16(M, NKEY, false);
  constexpr uint32_t IDESC_PV = idesc_bf16(M, D, true);
  static_assert(D == 64 || D == 128, "head_dim");

  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.y, ps = blockIdx.z;
  const int G = p.group;
  const int rows = p.batch * G;
  const int row = blockIdx.x * M + threadIdx.x;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * STAGE);
  uint64_t* bar_s = full + NS;
  uint64_t* bar_pv = bar_s + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_pv + 1);
  int* s_blk = reinterpret_cast<int*>(s_tmem + 2);
  const uint32_t stage0 = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(smem_u32(full + s), 1);
    mbar_init(smem_u32(bar_s), 1);
    mbar_init(smem_u32(bar_pv), 1);
    fence_mbar_init();
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_tmem;
  const uint32_t tlane = tbase + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's lanes

  wait_prior_grid();
  const int t0 = ps * p.prefix_split_tokens;
  const int t1 = min(p.prefix_len, t0 + p.prefix_split_tokens);
  const int nblk = (t1 - t0 + p.block_size - 1) / p.block_size;
  for (int i = threadIdx.x; i < nblk && i < kMaxPrefixBlocks; i += blockDim.x) {
    int phys = p.prefix_blocks[t0 / p.block_size + i];
    if (phys < 0 || phys >= p.num_blocks) {
      record_error(p.err, kDevErrBlockId);
      phys = -1;
    }
    s_blk[i] = phys;
  }
  __syncthreads();
  const int ntile = (t1 - t0 + NKEY - 1) / NKEY;

  auto issue = [&](int k) {  // thread 0: tile k -> stage k % NS, laid out [K|V][d-half][key][128 B]
    const int s = k % NS;
    const uint32_t dst = stage0 + s * STAGE;
    const uint32_t bar = smem_u32(full + s);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
    for (int i = 0; i < NSUB; ++i) {
      const int t = t0 + k * NKEY + i * kTileTokens;
      const int phys = t < t1 ? s_blk[(t - t0) / p.block_size] : -1;   // past the end: zeros
      const int tok0 = t % p.block_size;
#pragma unroll
      for (int bx = 0; bx < HALVES; ++bx) {
        const uint32_t off = bx * HALF_BYTES + i * kTileTokens * 128;
        tma_load_4d(dst + off, &tmap_k, bar, bx * L::BOX_ELEMS, tok0, h, phys);
        tma_load_4d(dst + KREG + off, &tmap_v, bar, bx * L::BOX_ELEMS, tok0, h, phys);
      }
    }
  };
  if (threadIdx.x == 0)
    for (int k = 0; k < ntile && k < NS; ++k) issue(k);

  // ---- this thread's query row into TMEM (zeros for padding rows)
  {
    const uint16_t* q = static_cast<const uint16_t*>(p.q);
    const uint16_t* qr = row < rows ? q + (static_cast<int64_t>(row / G) * p.num_q_heads + h * G + row % G) * D
                                    : nullptr;
#pragma unroll
    for (int c0 = 0; c0 < D / 2; c0 += 16) {
      uint32_t v[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 w = qr ? *reinterpret_cast<const uint4*>(qr + 2 * c0 + 8 * i) : make_uint4(0u, 0u, 0u, 0u);
        v[4 * i] = w.x;
        v[4 * i + 1] = w.y;
        v[4 * i + 2] = w.z;
        v[4 * i + 3] = w.w;
      }
      tmem_st16(tlane + COL_Q + c0, v);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();

  const float qk_mult = p.qk_log2_scale;
  float m_used = -CUDART_INF_F, lsum = 0.f;
  bool healthy = true;
  int k = 0;
  for (; k < ntile; ++k) {
    const int s = k % NS;
    const uint32_t kbase = stage0 + s * STAGE, vbase = kbase + KREG;
    // ---- S = Q K^T, issued by thread 0 once the tile has landed and the
    // previous tile's P.V has completed: S shares TMEM columns with the P that
    // P.V reads, and tcgen05 orders MMAs only on the same accumulator.  When
    // bar_s flips, O is stable, P may be overwritten and the previous stage
    // is free.
    bool ok = true;
    if (threadIdx.x == 0) {
      ok = mbar_wait(smem_u32(full + s), static_cast<uint32_t>((k / NS) & 1), p.err);
      if (ok && k > 0) ok = mbar_wait(smem_u32(bar_pv), static_cast<uint32_t>((k - 1) & 1), p.err);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t kd = smem_desc_sw128(kbase + (ks / 4) * HALF_BYTES + (ks % 4) * 32, 0, 1024);
          tc_mma_ts(tbase + COL_S, tbase + COL_Q + ks * 8, kd, IDESC_S, ks > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(bar_s));
      }
    }
    if (!__syncthreads_and(ok)) {
      healthy = false;
      break;
    }
    if (!mbar_wait(smem_u32(bar_s), static_cast<uint32_t>(k & 1), p.err)) ok = false;
    tc_fence_after();
    if (threadIdx.x == 0 && ok && k > 0 && k - 1 + NS < ntile) issue(k - 1 + NS);
    float x[NKEY];
    {
      uint32_t v[NKEY / 16][16];
#pragma unroll
      for (int c = 0; c < NKEY / 16; ++c) tmem_ld16(tlane + COL_S + 16 * c, v[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < NKEY / 16; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) x[16 * c + i] = __uint_as_float(v[c][i]);
    }
    const int valid = t1 - (t0 + k * NKEY);
    float mt = -CUDART_INF_F;
#pragma unroll
    for (int i = 0; i < NKEY; ++i) {
      x[i] = i < valid ? x[i] * qk_mult : -CUDART_INF_F;
      mt = fmaxf(mt, x[i]);
    }
    float alpha = 1.f;
    bool resc = false;
    if (k == 0) {
      m_used = mt;
    } else if (mt > m_used + 8.f) {
      alpha = fast_exp2(m_used - mt);
      m_used = mt;
      resc = true;
    }
    if (__any_sync(kFull, resc)) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[2][16];
        tmem_ld16(tlane + COL_O + c0, v[0]);
        tmem_ld16(tlane + COL_O + c0 + 16, v[1]);
        tmem_wait_ld();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int i = 0; i < 16; ++i) v[hh][i] = __float_as_uint(__uint_as_float(v[hh][i]) * alpha);
        tmem_st16(tlane + COL_O + c0, v[0]);
        tmem_st16(tlane + COL_O + c0 + 16, v[1]);
      }
    }
    lsum *= alpha;
#pragma unroll
    for (int c0 = 0; c0 < NKEY / 2; c0 += 16) {
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = fast_exp2(x[2 * (c0 + i)] - m_used);
        const float p1 = fast_exp2(x[2 * (c0 + i) + 1] - m_used);
        lsum += p0 + p1;
        hi[i] = pack_bf16x2(p0, p1);
        lo[i] = pack_bf16x2(p0 - bf16lo_to_f32(hi[i]), p1 - bf16hi_to_f32(hi[i]));
      }
      tmem_st16(tlane + COL_PHI + c0, hi);
      tmem_st16(tlane + COL_PLO + c0, lo);
    }
    tmem_wait_st();
    tc_fence_before();
    if (!__syncthreads_and(ok)) {
      healthy = false;
      break;
    }
    if (threadIdx.x == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < NKEY / 16; ++kk) {
        // MN-major V: 8-key groups 1024 B apart, the two 64-wide d-halves
        // HALF_BYTES apart (a single half for D = 64)
        const uint64_t vd = smem_desc_sw128(vbase + kk * 2048, HALVES > 1 ? HALF_BYTES : 0, 1024);
        tc_mma_ts(tbase + COL_O, tbase + COL_PHI + kk * 8, vd, IDESC_PV, (k > 0 || kk > 0) ? 1u : 0u);
        tc_mma_ts(tbase + COL_O, tbase + COL_PLO + kk * 8, vd, IDESC_PV, 1u);
      }
      tc_commit(smem_u32(bar_pv));
    }
  }
  if (healthy && ntile > 0) {
    const bool pv_done = mbar_wait(smem_u32(bar_pv), static_cast<uint32_t>((ntile - 1) & 1), p.err);
    healthy = __syncthreads_and(pv_done);
  }
  if (healthy && ntile > 0) {
    tc_fence_after();
    const int64_t S_row = p.slots_per_row;
    const int64_t piece = (row < rows ? (static_cast<int64_t>(row / G) * p.num_q_heads + h * G + row % G) : 0) *
                              S_row + p.extra_slot + ps;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t v[2][16];
      tmem_ld16(tlane + COL_O + c0, v[0]);
      tmem_ld16(tlane + COL_O + c0 + 16, v[1]);
      tmem_wait_ld();
      if (row < rows) {
        float4* dst = reinterpret_cast<float4*>(p.ws_o + piece * D + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(v[i / 4][4 * (i % 4)]), __uint_as_float(v[i / 4][4 * (i % 4) + 1]),
                               __uint_as_float(v[i / 4][4 * (i % 4) + 2]), __uint_as_float(v[i / 4][4 * (i % 4) + 3]));
      }
    }
    if (row < rows) {
      p.ws_ml[piece * 2] = m_used;
      p.ws_ml[piece * 2 + 1] = lsum;
    }
  } else if (!healthy && threadIdx.x == 0) {
    // let whatever is still in flight land before the memory is released
    for (int s = 0; s < NS && s < ntile; ++s) mbar_wait(smem_u32(full + s), static_cast<uint32_t>((k / NS) & 1), nullptr);
    mbar_wait(smem_u32(bar_s), static_cast<uint32_t>(k & 1), nullptr);
    if (k > 0) mbar_wait(smem_u32(bar_pv), static_cast<uint32_t>((k - 1) & 1), nullptr);
  }
  allow_next_grid();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, TCOLS);
  }
}

}  // namespace

int cascade_smem_bytes(int head_dim) {
  const int stage = (kCascadeTile / kTileTokens) * 2 * kTileTokens * head_dim * 2;
  return 3 * stage + 6 * 8 + 1024 * 4 + 1024;
}

namespace {
template <int D>
cudaError_t launch_cascade_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             cudaStream_t stream) {
  auto kern = cascade_prefix_tc_kernel<D>;
  const int smem = cascade_smem_bytes(D);
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
  const int rows = p.batch * p.group;
  const int nps = (p.prefix_len + p.prefix_split_tokens - 1) / p.prefix_split_tokens;
  const dim3 grid((rows + kCascadeRowsTc - 1) / kCascadeRowsTc, p.num_kv_heads, nps);
  return launch_pdl(kern, grid, dim3(128), smem, stream, tk, tv, p);
}

}  // namespace

cudaError_t launch_cascade_prefix(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream) {
  if (p.head_dim == 128) return launch_cascade_t<128>(p, tk, tv, stream);
  return launch_cascade_t<64>(p, tk, tv, stream);
}

}  // namespace pkv
