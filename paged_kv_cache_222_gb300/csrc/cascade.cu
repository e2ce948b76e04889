// Tensor-core (tcgen05) paged attention for many query rows per KV head.
//
// Cascade (shared-prefix) decode, the prefix part: when every sequence of the
// batch starts with the same `prefix_len` tokens held in the same physical
// blocks (shared by reference: [FN] "Sub-Millisecond Token Scheduling...",
// "Paged KV-Cache with Radix Tree Prefix Cache", copy-on-write prefix blocks),
// the prefix part of decode attention is one dense product per KV head,
//   S = Q_h K_prefix^T,  Q_h = the B*G query rows (b, g) of KV head h,
// followed by the online softmax and P V_prefix.  Each CTA takes 256 query
// rows of one KV head over one range of prefix tokens and writes (acc, m, l)
// per row into the workspace slot reserved for its range; the combine kernel
// of decode.cu merges those with the private-suffix splits.
//
// Multi-token queries ([SC] "LLM inference: prefill, decode, KV cache", "7.
// Practical applications", item 3, and "9. Failure modes and limitations",
// item 3) with more than 16 rows (q_len * G) per (sequence, KV head): a
// persistent kernel whose CTAs take (split, sequence, KV head, 128-row block)
// units, longest first, with a causal limit per row.

#include "decode_common.cuh"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

// ----------------------------------------------------------------------------
// Paged attention of many query rows on the 5th-generation tensor cores
// (tcgen05 + TMEM), pipelined, one CTA per SM with all 512 TMEM columns.  Its
// warps have fixed roles:
//   softmax warps (4 per 128-row group): thread t of a group is its query row
//              t (= TMEM lane t, in the group's columns)
//   two TMA producer warps: 64-token K and V tiles into a ring of stages of
//              128B-swizzled shared memory, one box (a block's rows of one
//              128-byte d-half) per lane
//   MMA issuers (one lane issues): S(k) = Q K(k)^T and O += P(k) V(k)
// K is a K-major and V an MN-major B operand; P (as bf16 hi | lo pairs, so
// that P.V keeps fp32-like accuracy) comes from TMEM.  While a group's
// softmax turns S(k) into P(k), the tensor core works on S(k+1) and O +=
// P(k-1) V.  Hand-offs are mbarriers: full / empty per stage (TMA bytes; an
// MMA commit after the stage's P.V), and per buffer sfull / pfree (MMA
// commits) and pfull (one arrive per softmax warp).  The softmax keeps a lazy
// running max: O in TMEM is rescaled only when the max grows by more than
// 2^8 (then after the previous P.V has completed), so P stays <= 256.  Every
// wait is bounded; a time-out records the error, raises a shared abort flag
// that ends every role's loop, and the CTA drains its copies and MMAs before
// it frees TMEM.
//
// The cascade prefix kernel has two groups sharing each tile, Q in shared
// memory and P over S; its CTAs of one KV head each start at a different
// tile of their range (the online softmax takes tiles in any order) so that
// they do not all ask L2 for the same lines at once.  The multi-token kernel
// has one group, Q in TMEM (A operand of S), P in buffers of its own (so S
// never waits for a P.V), S and P.V issued by two warps, and six stages.
// ----------------------------------------------------------------------------

// Wait for a barrier phase; false once the CTA aborts (or on time-out, which
// records the error and raises the abort flag).
// max(a, b, c) in one instruction (three-input max.f32).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, int* err, volatile int* abort,
                                              uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (n % 16 == 0 && *abort) return false;
    if (n % kWaitTriesPerClockRead == 0) {
      const uint64_t t = global_timer_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > limit_ns) {
        record_error(err, kDevErrWaitTimeout);
        *abort = 1;
        return false;
      }
    }
  }
}

// Tile geometry of the tensor-core kernels: 128 query rows per group, 64-key
// K and V tiles stored as 128-byte rows (one d-half after the other),
// 128B-swizzled.
template <int D, int NK = kCascadeTile>
struct TcTile {
  static constexpr int M = 128;                       // query rows per group
  static constexpr int NKEY = NK;                     // keys per tile
  static constexpr int HALVES = D / 64;               // 128-byte d-halves of a row
  static constexpr int QHALF = M * 128;               // one d-half of one group's Q
  static constexpr int HALF_BYTES = NKEY * 128;       // one d-half of a K (or V) tile
  static constexpr int KREG = HALVES * HALF_BYTES;    // K (or V) tile
  static constexpr int STAGE = 2 * KREG;
};

// Cascade prefix CTA: two 128-row groups (their rows all read the same
// prefix tiles), Q of both in shared memory, five K/V stages, and threads:
// 4 softmax warps per group, two TMA producer warps, an S issuer and a P.V
// issuer.  One CTA per SM with all 512 TMEM columns, 256 per group: O, S and
// P in columns of their own, so that S(k+1) waits only for the softmax to
// have read S(k), and P(k).V for the softmax to have written P(k).
template <int D>
struct CascadeShape : TcTile<D> {
  using T = TcTile<D>;
  static constexpr int GROUPS = 2;
  static constexpr int QBYTES = GROUPS * T::HALVES * T::QHALF;
  // the tiles come from L2, about 5000 cycles from issue to arrival while the
  // suffix decode streams from HBM beside this kernel: five stages (the most
  // that fit beside Q) keep four in flight while one is computed on
  static constexpr int NS = 5;
  // full, empty; sfull, sfree, pfull, pfree per group; done per issuer
  static constexpr int NBARS = 2 * NS + 4 * GROUPS + 2;
  static constexpr int BYTES = QBYTES + NS * T::STAGE + NBARS * 8 + 16 + kCascadeMaxRangeBlocks * 4 + 1024;
  static_assert(BYTES <= 232448, "shared memory per CTA");
  // two producer warps issue a tile's boxes in parallel (one warp issuing a
  // tile's boxes was measured to hold an SM to about 12-19 bytes per cycle)
  static constexpr int NPROD = 2;
  static constexpr int THREADS = 32 * (4 * GROUPS + NPROD + 2);
};

// Rows (b, g) of KV head blockIdx.y, 256 per CTA (blockIdx.x), over prefix
// range blockIdx.z; (acc, m, l) pieces go to workspace slot extra_slot +
// range.
template <int D>
__global__ void __launch_bounds__(CascadeShape<D>::THREADS, 1)
    cascade_prefix_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                          const DecodeParams p) {
  using L = Layout<D, false>;
  using C = CascadeShape<D>;
  constexpr int M = C::M, NKEY = C::NKEY, NS = C::NS, GROUPS = C::GROUPS;
  constexpr int kMaxBlocks = kCascadeMaxRangeBlocks;  // block ids of one range, in shared memory
  constexpr uint32_t GCOLS = 512 / GROUPS;            // TMEM columns of one group
  // within a group's columns: O, S (fp32, one column per key), P (bf16 hi
  // then lo pairs, half a column per key each)
  constexpr uint32_t COL_O = 0, COL_S = D, COL_P = D + NKEY;
  constexpr uint32_t IDESC_S = idesc_bf16(M, NKEY, false);
  constexpr uint32_t IDESC_PV = idesc_bf16(M, D, true);
  constexpr int PRODUCER = 4 * GROUPS;                // first producer warp
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(COL_P + NKEY <= GCOLS, "TMEM columns");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  const int H_q = p.num_q_heads;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_sm = smem;                                // group g at g * HALVES * QHALF
  const uint32_t stage0 = smem_u32(smem + C::QBYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::QBYTES + NS * C::STAGE);
  uint64_t* full = bars;
  uint64_t* empty = full + NS;
  uint64_t* sfull = empty + NS;       // [GROUPS]: S(k) is in TMEM
  uint64_t* sfree = sfull + GROUPS;   // [GROUPS]: the softmax has read S(k)
  uint64_t* pfull = sfree + GROUPS;   // [GROUPS]: P(k) is in TMEM
  uint64_t* pfree = pfull + GROUPS;   // [GROUPS]: P(k).V has completed
  uint64_t* done = pfree + GROUPS;    // [2]: the S and the P.V issuer's last MMAs
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 2);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_blk = reinterpret_cast<int*>(s_tmem + 4);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(full + s), C::NPROD);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int i = 0; i < GROUPS; ++i) {
      mbar_init(smem_u32(sfull + i), 1);
      mbar_init(smem_u32(sfree + i), 4);
      mbar_init(smem_u32(pfull + i), 4);
      mbar_init(smem_u32(pfree + i), 1);
    }
    mbar_init(smem_u32(done), 1);
    mbar_init(smem_u32(done + 1), 1);
    *s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  wait_prior_grid();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_tmem;

  // ---- the CTA's rows, token range [t0, t1) and tiles
  const int h = blockIdx.y;
  const int rows = p.batch * G;
  const int row0 = blockIdx.x * (GROUPS * M);
  const int t0 = blockIdx.z * p.prefix_split_tokens;
  const int t1 = min(p.prefix_len, t0 + p.prefix_split_tokens);
  const int32_t* blocks = p.prefix_blocks;
  const int nblk = (t1 - t0 + p.block_size - 1) / p.block_size;
  const int ntile = (t1 - t0 + NKEY - 1) / NKEY;
  // k-th tile processed = tile (k + first) % ntile of the range: the CTAs of
  // one head start at different tiles (they all read the same prefix)
  const int first = ntile > 0 ? static_cast<int>((static_cast<int64_t>(blockIdx.x) * ntile) / gridDim.x) : 0;

  const int grp = warp / 4;                            // softmax warps only
  const int r_in = (warp % 4) * 32 + lane;             // row within the group
  const int row = row0 + grp * M + r_in;
  const bool row_ok = warp < PRODUCER && row < rows;
  const int64_t orow = static_cast<int64_t>(row / G) * H_q + h * G + row % G;  // output row (b, hq)
  // The producers start loading tiles at once; the softmax warps put Q into
  // shared memory meanwhile and hand it to the S issuer at named barrier 2.
  constexpr uint32_t kQBar = 2, kQThreads = 32 * (4 * GROUPS + 1);
  if (warp >= PRODUCER && warp < PRODUCER + C::NPROD) {
    // ------------------------------------------------------------ producers
    // A tile's TMA boxes (K then V; d-half; block) are split evenly over the
    // producer warps, one box per lane.
    const int pw = warp - PRODUCER;
    for (int i = pw * 32 + lane; i < nblk && i < kMaxBlocks; i += 32 * C::NPROD) {
      int phys = blocks[t0 / p.block_size + i];
      if (phys < 0 || phys >= p.num_blocks) {
        record_error(p.err, kDevErrBlockId);
        phys = -1;
      }
      s_blk[i] = phys;
    }
    named_bar_sync(1, 32 * C::NPROD);
    const int box = p.block_size < NKEY ? p.block_size : NKEY;  // token rows per TMA box
    const int per_half = NKEY / box;
    const int nbox = 2 * C::HALVES * per_half / C::NPROD;        // boxes of a tile per warp (<= 32)
    // This lane's box of every tile, set up once.  Ranges start at multiples
    // of 64 tokens and the block size (16 or 32) divides 64, so each box is a
    // whole block: box i of tile kt is block kt * per_half + i of the range.
    const int gi = pw * nbox + lane;                             // box of the tile
    const int bv = gi / (C::HALVES * per_half);                  // 0: K, 1: V
    const int bx = (gi / per_half) % C::HALVES;                  // d-half
    const int bi = gi % per_half;                                // block within the half
    const uint32_t off = bv * C::KREG + bx * C::HALF_BYTES + bi * box * 128;
    const CUtensorMap* tmap = bv ? &tmap_v : &tmap_k;
    const int c0 = bx * L::BOX_ELEMS;
    int kt = first;                                              // tile of the range at step k
    int issued = 0;
    for (int k = 0; k < ntile; ++k) {
      const int s = k % NS;
      bool go = true;
      if (lane == 0 && k >= NS)
        go = wait_or_abort(smem_u32(empty + s), static_cast<uint32_t>((k / NS - 1) & 1), p.err, s_abort);
      if (!__shfl_sync(kFull, go ? 1 : 0, 0)) break;
      const uint32_t dst = stage0 + s * C::STAGE;
      const uint32_t bar = smem_u32(full + s);
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, C::STAGE / C::NPROD);
      }
      __syncwarp();
      if (lane < nbox) {
        const int j = kt * per_half + bi;
        const int phys = j < nblk ? s_blk[j] : -1;  // past the range: zeros
        tma_load_4d(dst + off, tmap, bar, c0, 0, h, phys);
      }
      if (++kt == ntile) kt = 0;
      issued = k + 1;
    }
    if (lane == 0 && *s_abort) {  // the copies in flight land before the stages are released
      for (int k = issued > NS ? issued - NS : 0; k < issued; ++k)
        mbar_wait(smem_u32(full + k % NS), static_cast<uint32_t>((k / NS) & 1), nullptr);
    }
  } else if (warp == PRODUCER + C::NPROD) {
    // ------------------------------------------------------------ S issuer
    // S_g(k) = Q_g K(k)^T for both groups, once the tile has arrived and the
    // group's softmax has read S_g(k-1)
    named_bar_sync(kQBar, kQThreads);                  // Q is in shared memory
    for (int k = 0; k < ntile; ++k) {
      const int s = k % NS;
      bool ok = true;
      if (lane == 0) ok = wait_or_abort(smem_u32(full + s), static_cast<uint32_t>((k / NS) & 1), p.err, s_abort);
#pragma unroll
      for (int g = 0; g < GROUPS; ++g) {
        if (lane == 0 && ok && k >= 1)
          ok = wait_or_abort(smem_u32(sfree + g), static_cast<uint32_t>((k - 1) & 1), p.err, s_abort);
        if (lane == 0 && ok) {
          tc_fence_after();
          const uint32_t qa = smem_u32(q_sm + g * C::HALVES * C::QHALF);
          const uint32_t kst = stage0 + s * C::STAGE;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(qa + (kk / 4) * C::QHALF + (kk % 4) * 32, 0, 1024);
            const uint64_t bd = smem_desc_sw128(kst + (kk / 4) * C::HALF_BYTES + (kk % 4) * 32, 0, 1024);
            tc_mma_ss(tbase + g * GCOLS + COL_S, ad, bd, IDESC_S, kk > 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(sfull + g));
        }
      }
      if (!__shfl_sync(kFull, ok ? 1 : 0, 0)) break;
    }
    if (lane == 0) {  // nothing of this thread's may still be running when TMEM is freed
      tc_commit(smem_u32(done));
      mbar_wait(smem_u32(done), 0u, nullptr);
    }
  } else if (warp == PRODUCER + C::NPROD + 1) {
    // ------------------------------------------------------------ P.V issuer
    // O_g += P_g(j) V(j) for both groups as each group's softmax hands over
    // P_g(j); then the stage goes back to the producers.  Separate from the S
    // issuer, so that a ready P.V never waits behind the next tile's arrival.
    for (int j = 0; j < ntile; ++j) {
      const int sj = j % NS;
      bool ok = true;
      if (lane == 0) ok = wait_or_abort(smem_u32(full + sj), static_cast<uint32_t>((j / NS) & 1), p.err, s_abort);
#pragma unroll
      for (int g = 0; g < GROUPS; ++g) {
        if (lane == 0 && ok) ok = wait_or_abort(smem_u32(pfull + g), static_cast<uint32_t>(j & 1), p.err, s_abort);
        if (lane == 0 && ok) {
          tc_fence_after();
          const uint32_t tg = tbase + g * GCOLS;
          const uint32_t vst = stage0 + sj * C::STAGE + C::KREG;
          const uint32_t pa = tg + COL_P;
#pragma unroll
          for (int kk = 0; kk < NKEY / 16; ++kk) {
            // MN-major V: 8-key groups 1024 B apart, d-halves HALF_BYTES apart
            const uint64_t vd = smem_desc_sw128(vst + kk * 2048, C::HALVES > 1 ? C::HALF_BYTES : 0, 1024);
            tc_mma_ts(tg + COL_O, pa + kk * 8, vd, IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
            tc_mma_ts(tg + COL_O, pa + NKEY / 2 + kk * 8, vd, IDESC_PV, 1u);
          }
          tc_commit(smem_u32(pfree + g));
        }
      }
      if (lane == 0 && ok) tc_commit(smem_u32(empty + sj));
      if (!__shfl_sync(kFull, ok ? 1 : 0, 0)) break;
    }
    if (lane == 0) {
      tc_commit(smem_u32(done + 1));
      mbar_wait(smem_u32(done + 1), 0u, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    {
      // Q rows into shared memory: group g, row r, 16-byte chunk c of d-half
      // hf at g * HALVES * QHALF + hf * QHALF + r * 128 + ((c ^ (r % 8)) * 16)
      // (the 128-byte swizzle)
      const uint16_t* qr = row_ok ? static_cast<const uint16_t*>(p.q) + orow * D : nullptr;
      uint8_t* qg = q_sm + grp * C::HALVES * C::QHALF;
      // a negative scale enters as negated Q (exact in bf16): the softmax
      // below applies a positive multiplier to the raw products
      const uint32_t q_sign = p.qk_log2_scale < 0.f ? 0x80008000u : 0u;
      uint4 w[D / 8];  // every load issued before the first store
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        w[c] = qr ? *reinterpret_cast<const uint4*>(qr + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        w[c].x ^= q_sign;
        w[c].y ^= q_sign;
        w[c].z ^= q_sign;
        w[c].w ^= q_sign;
        const int hf = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(qg + hf * C::QHALF + r_in * 128 + ((cc ^ (r_in & 7)) << 4)) = w[c];
      }
      fence_proxy_async_smem();  // the tensor core reads Q through the async proxy
      named_bar_sync(kQBar, kQThreads);
    }
    const uint32_t tl = tbase + grp * GCOLS + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const uint32_t g_sfull = smem_u32(sfull + grp), g_sfree = smem_u32(sfree + grp);
    const uint32_t g_pfull = smem_u32(pfull + grp), g_pfree = smem_u32(pfree + grp);
    // the logit multiplier (scale x log2 e, made positive above) is applied
    // inside the exponent's FMA; a zero scale takes the smallest normal one
    const float qk_mult = fmaxf(fabsf(p.qk_log2_scale), 1.17549435e-38f);
    float m_used = -CUDART_INF_F, lsum = 0.f;
    bool ok = true;
    for (int k = 0; k < ntile && ok; ++k) {
      ok = __all_sync(kFull, wait_or_abort(g_sfull, static_cast<uint32_t>(k & 1), p.err, s_abort));
      if (!ok) break;
      tc_fence_after();
      float x[NKEY];
      {
        uint32_t v[NKEY / 16][16];
#pragma unroll
        for (int c = 0; c < NKEY / 16; ++c) tmem_ld16(tl + COL_S + 16 * c, v[c]);
        tmem_wait_ld();
        tc_fence_before();  // S may be overwritten by S(k+1)
        __syncwarp();
        if (lane == 0) mbar_arrive(g_sfree);
#pragma unroll
        for (int c = 0; c < NKEY / 16; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) x[16 * c + i] = __uint_as_float(v[c][i]);
      }
      const int valid = t1 - (t0 + ((k + first) % ntile) * NKEY);  // the prefix has no causal limit
      if (__any_sync(kFull, valid < NKEY)) {
#pragma unroll
        for (int i = 0; i < NKEY; ++i)
          if (i >= valid) x[i] = -CUDART_INF_F;
      }
      float mt;
      {  // eight chains of three-input maxima, then their maximum (in log2 units)
        static_assert(NKEY == 64, "eight chains of eight keys");
        float mp[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          mp[j] = max3f(x[j], x[8 + j], x[16 + j]);
          mp[j] = max3f(mp[j], x[24 + j], x[32 + j]);
          mp[j] = max3f(mp[j], x[40 + j], x[48 + j]);
          mp[j] = fmaxf(mp[j], x[56 + j]);
        }
        mt = max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])) * qk_mult;
      }
      float alpha = 1.f;
      bool resc = false;
      if (m_used == -CUDART_INF_F) {
        m_used = mt;  // nothing accumulated yet for this row
      } else if (mt > m_used + 8.f) {
        alpha = fast_exp2(m_used - mt);
        m_used = mt;
        resc = true;
      }
      // P(k-1).V must have completed before O is rescaled (O then holds
      // tiles 0..k-1) and before P(k) is written over P(k-1); the wait comes
      // as late as possible, so that it overlaps this tile's exponentials
      bool pv_done = k == 0;
      if (__any_sync(kFull, resc)) {
        ok = __all_sync(kFull, wait_or_abort(g_pfree, static_cast<uint32_t>((k - 1) & 1), p.err, s_abort));
        if (!ok) break;
        tc_fence_after();
        pv_done = true;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[2][16];
          tmem_ld16(tl + COL_O + c0, v[0]);
          tmem_ld16(tl + COL_O + c0 + 16, v[1]);
          tmem_wait_ld();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int i = 0; i < 16; ++i) v[hh][i] = __float_as_uint(__uint_as_float(v[hh][i]) * alpha);
          tmem_st16(tl + COL_O + c0, v[0]);
          tmem_st16(tl + COL_O + c0 + 16, v[1]);
        }
        tmem_wait_st();
      }
      lsum *= alpha;
      const float mu = m_used == -CUDART_INF_F ? 0.f : m_used;
      const float2 neg_mu = make_float2(-mu, -mu);
      const float2 mult2 = make_float2(qk_mult, qk_mult);
      float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t hi[NKEY / 32][16], lo[NKEY / 32][16];
#pragma unroll
      for (int c = 0; c < NKEY / 32; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = 16 * c + i;                      // key pair j: keys 2j, 2j + 1
          const float2 e = __ffma2_rn(make_float2(x[2 * j], x[2 * j + 1]), mult2, neg_mu);
          const float2 pp = make_float2(fast_exp2(e.x), fast_exp2(e.y));
          ls[i & 1] = __fadd2_rn(ls[i & 1], pp);
          hi[c][i] = pack_bf16x2(pp.x, pp.y);
          const float2 r = __fadd2_rn(pp, make_float2(-bf16lo_to_f32(hi[c][i]), -bf16hi_to_f32(hi[c][i])));
          lo[c][i] = pack_bf16x2(r.x, r.y);
        }
      lsum += (ls[0].x + ls[1].x) + (ls[0].y + ls[1].y);
      if (!__all_sync(kFull, pv_done)) {
        ok = __all_sync(kFull, wait_or_abort(g_pfree, static_cast<uint32_t>((k - 1) & 1), p.err, s_abort));
        if (!ok) break;
        tc_fence_after();
      }
#pragma unroll
      for (int c = 0; c < NKEY / 32; ++c) {
        tmem_st16(tl + COL_P + 16 * c, hi[c]);
        tmem_st16(tl + COL_P + NKEY / 2 + 16 * c, lo[c]);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(g_pfull);   // P(k) is in TMEM
    }
    if (ok && ntile > 0)
      ok = __all_sync(kFull, wait_or_abort(g_pfree, static_cast<uint32_t>((ntile - 1) & 1), p.err, s_abort));
    // ---- this row's (acc, m, l) piece of the prefix range.  O leaves through
    // shared memory, the group's Q region (every S of the group has
    // completed), one bulk copy per row and pass: 16-byte stores straight
    // from the TMEM rows would scatter each warp instruction over 32 rows.
    const int64_t piece = orow * p.slots_per_row + p.extra_slot + blockIdx.z;
    if (ok && ntile > 0) {
      tc_fence_after();
      constexpr int CP = C::HALVES * 32;                 // columns per pass (half a row)
      uint8_t* srow = q_sm + grp * C::HALVES * C::QHALF + r_in * (CP * 4);
      float* dst_row = p.ws_o + piece * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += CP) {
        if (c0 > 0) bulk_wait_read_all();                // the previous pass has left srow
        uint32_t v[CP / 16][16];
#pragma unroll
        for (int c = 0; c < CP / 16; ++c) tmem_ld16(tl + COL_O + c0 + 16 * c, v[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < CP / 16; ++c)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(srow + (16 * c + 4 * i) * 4) =
                make_uint4(v[c][4 * i], v[c][4 * i + 1], v[c][4 * i + 2], v[c][4 * i + 3]);
        fence_proxy_async_smem();
        if (row_ok) {
          bulk_store_s2g(dst_row + c0, smem_u32(srow), CP * 4);
          bulk_commit();
        }
      }
      if (row_ok) {
        p.ws_ml[piece * 2] = m_used;
        p.ws_ml[piece * 2 + 1] = lsum;
      }
      bulk_wait_read_all();  // the writes complete with the grid
    }
  }
  allow_next_grid();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// Self-test of the bounded waits and of the abort path of the tensor-core
// kernels: barriers that nothing ever arrives on.
//   which 0: one thread waits with mbar_wait until the limit, records the
//            time-out, returns.
//   which 1: as a tensor-core CTA: warp 0 holds all TMEM; thread 32 waits
//            with wait_or_abort until the limit (recording the time-out and
//            raising the abort flag); the threads of warps 2-3 wait on another
//            such barrier and leave when they see the flag; then the CTA
//            frees TMEM as the attention kernels do.
__global__ void __launch_bounds__(128) wait_selftest_kernel(int which, uint64_t limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (which == 1 && warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (which == 0) {
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bars[0]), 0u, err, limit_ns);
    return;
  }
  volatile int* abort = &s_abort;
  if (threadIdx.x == 32) {
    wait_or_abort(smem_u32(&bars[0]), 0u, err, abort, limit_ns);
  } else if (warp >= 2) {
    // leaves when the abort flag rises, or after four limits of its own
    wait_or_abort(smem_u32(&bars[1]), 0u, err, abort, 4 * limit_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(s_tmem, 512);
  }
}

// ----------------------------------------------------------------------------
// Multi-token queries on the tensor cores, persistent.  One CTA per SM takes
// work units (split, sequence, KV head, 128-row block) from a counter in the
// caller's workspace, in split-major order (the first, longest splits of all
// sequences first), until none are left; the producers run ahead into the
// next unit while the softmax warps finish the current one, so a unit costs
// no pipeline fill and no setup.  Warps:
//   0-3  softmax: thread t is query row t of the unit (TMEM lane t); at the
//        end of a unit they put the next unit's Q into TMEM (one buffer: all
//        S of the unit have completed by then), then read O of the unit
//        and write its output row or (acc, m, l) piece
//   4-5  TMA producers: half of each tile's boxes each; warp 4 takes units
//        from the counter and publishes them in a ring of shared slots
//   6    S issuer: S(g) = Q K(g)^T (A from TMEM)
//   7    P.V issuer: O += P(g) V(g) (P from TMEM as bf16 hi | lo pairs)
// g counts tiles over all of the CTA's units, so ring slots and TMEM
// buffers keep their phases across units.  Every wait is bounded; a time-out
// records the error and raises the CTA's abort flag, which ends every loop.
// ----------------------------------------------------------------------------
// Keys per tile and the depths of the persistent kernel's K and V rings: its
// tiles come from HBM, where the bytes in flight set the speed, and Q in TMEM
// leaves it the shared memory (192 KB of K and V tiles).  A K tile goes back
// to its producer as soon as S has read it, a V tile after P.V; with rings
// of their own the K tiles of later tiles arrive earlier and S is ready when
// the softmax wants it (q_len 4: 4.69 -> 4.81 TB/s against one ring of six
// K+V stages).  Measured on the GQA workload: 6 + 6 slots beat 4 + 8 and
// 8 + 4 (-6 %), every other split of 12 or 13 slots (-11 %).  Twelve stages
// of 32-key tiles measured 38 % slower than six of 64 (per-tile costs
// double).
constexpr int kMqTile = 64;
// Bytes of the barrier / unit-ring block after the block ids, and the stride
// of one row of the output staging after it: 32 floats (128 B) and 16 B of
// padding, so that the 16-byte stores of a quarter warp hit distinct banks.
constexpr int kMqBarBytes = 1024;
constexpr int kMqStageRow = 144;
constexpr int kMqKStages = 6;
constexpr int kMqVStages = 6;

struct MqUnit {
  int b, h, row0, t0, t1, ctx, nsplit, split, ntile;
};

// Work unit u (split-major: split, then sequence, then KV head and row block).
__device__ __forceinline__ MqUnit mq_unit(const DecodeParams& p, int u, int nrb, bool note) {
  MqUnit w;
  const int rows = p.q_len * p.group;
  const int hn_all = p.num_kv_heads * nrb;
  w.split = u / (p.batch * hn_all);
  const int r = u - w.split * (p.batch * hn_all);
  w.b = r / hn_all;
  const int hn = r - w.b * hn_all;
  w.h = hn / nrb;
  w.row0 = (hn - w.h * nrb) * 128;
  const int ctx_raw = p.context_lens[w.b];
  w.ctx = clamp_ctx(p, ctx_raw);
  if (note && w.ctx != ctx_raw && w.split == 0 && hn == 0) record_error(p.err, kDevErrContextLen);
  w.nsplit = (w.ctx + p.split_tokens - 1) / p.split_tokens;
  w.t0 = w.split * p.split_tokens;
  const int row_last = min(rows, w.row0 + 128) - 1;
  const int lim_last = min(w.ctx, w.ctx - p.q_len + row_last / p.group + 1);  // rows attend monotonically more
  w.t1 = w.t0 < w.ctx ? min(min(w.ctx, w.t0 + p.split_tokens), lim_last) : w.t0;
  if (w.t1 < w.t0) w.t1 = w.t0;
  w.ntile = (w.t1 - w.t0 + kMqTile - 1) / kMqTile;
  return w;
}

// Work units in order of decreasing tile count (longest first, so that the
// last units any CTA takes are short): a counting sort over the tile counts
// into `perm`, by one CTA.  Also zeroes the unit counter and prefetches the
// units' block-table rows into L2.
__global__ void __launch_bounds__(1024) mq_order_kernel(const DecodeParams p, int* perm) {
  __shared__ int cnt[kMultiQueryMaxSplitBlocks + 1];
  const int rows = p.q_len * p.group, nrb = (rows + 127) / 128;
  const int U = p.max_splits * p.batch * p.num_kv_heads * nrb;
  const int nb = p.split_tokens / kMqTile + 1;      // tile counts 0 .. split_tokens / kMqTile
  for (int i = threadIdx.x; i < nb; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  for (int u = threadIdx.x; u < U; u += blockDim.x) atomicAdd(&cnt[mq_unit(p, u, nrb, false).ntile], 1);
  __syncthreads();
  if (threadIdx.x == 0) {  // start of each count's run, largest count first
    int run = 0;
    for (int i = nb - 1; i >= 0; --i) {
      const int c = cnt[i];
      cnt[i] = run;
      run += c;
    }
    p.ws_q[0] = 0;
  }
  __syncthreads();
  for (int u = threadIdx.x; u < U; u += blockDim.x) perm[atomicAdd(&cnt[mq_unit(p, u, nrb, false).ntile], 1)] = u;
  // The producers read a unit's block ids with one dependent load per lane
  // per 32 ids before its first tile: bring every unit's table row into L2
  // now (+0.7-0.8 % at q_len 4-16 on the GQA batch).
  for (int u = threadIdx.x; u < U; u += blockDim.x) {
    const MqUnit w = mq_unit(p, u, nrb, false);
    const int nblk = (w.t1 - w.t0 + p.block_size - 1) / p.block_size;
    const char* row = reinterpret_cast<const char*>(p.block_tables + static_cast<int64_t>(w.b) * p.max_blocks +
                                                     w.t0 / p.block_size);
    for (int off = 0; off < nblk * 4; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
  }
}

// Unit number n of this CTA from the ring (readers: one call per warp, lane
// 0 waits); -1 when none is left or the CTA aborts.
__device__ __forceinline__ int mq_read_unit(uint64_t* ufull, uint64_t* uempty, const int* s_unit, int n,
                                            int* err, volatile int* abort) {
  constexpr int R = 8;
  int u = -1;
  if ((threadIdx.x & 31) == 0) {
    const int slot = n % R;
    if (wait_or_abort(smem_u32(ufull + slot), static_cast<uint32_t>((n / R) & 1), err, abort)) {
      u = *reinterpret_cast<const volatile int*>(s_unit + slot);
      mbar_arrive(smem_u32(uempty + slot));
    }
  }
  return __shfl_sync(kFull, u, 0);
}

// IDLE: some row block leaves a softmax warp without a query row (q_len x G
// not a multiple of 128 and its last block at most 96 rows).  Row counts
// that fill every warp take the instance without the idle-warp path: on 8
// sequences of 131k tokens at q_len 16 its mere presence cost 3.6 %.
template <int D, bool IDLE>
__global__ void __launch_bounds__(256, 1)
    mq_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const DecodeParams p) {
  using L = Layout<D, false>;
  using C = TcTile<D, kMqTile>;
  constexpr int M = 128, NKEY = C::NKEY, NK = kMqKStages, NV = kMqVStages;
  constexpr int R = 8;                                // unit ring slots
  constexpr int READERS = 7;                          // warps 0-3, 5, 6, 7
  constexpr uint32_t COL_O = 0, COL_S = D, COL_P = D + 2 * NKEY, COL_Q = COL_P + 2 * NKEY;
  constexpr uint32_t IDESC_S = idesc_bf16(M, NKEY, false);
  constexpr uint32_t IDESC_PV = idesc_bf16(M, D, true);
  static_assert(COL_Q + D / 2 <= 512, "TMEM columns");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group, QL = p.q_len, H_q = p.num_q_heads;
  const int rows = QL * G, nrb = (rows + M - 1) / M;
  const int U = p.max_splits * p.batch * p.num_kv_heads * nrb;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t kring = smem_u32(smem);             // [NK] K tiles
  const uint32_t vring = kring + NK * C::KREG;        // [NV] V tiles
  int* s_ids = reinterpret_cast<int*>(smem + (NK + NV) * C::KREG);  // [2][1024] each producer's block ids
  uint64_t* kfull = reinterpret_cast<uint64_t*>(s_ids + 2 * kMultiQueryMaxSplitBlocks);  // [NK]
  uint64_t* kempty = kfull + NK;                      // [NK]
  uint64_t* vfull = kempty + NK;                      // [NV]
  uint64_t* vempty = vfull + NV;                      // [NV]
  uint64_t* sfull = vempty + NV;                      // [2]
  uint64_t* sfree = sfull + 2;                        // [2]
  uint64_t* pfull = sfree + 2;                        // [2]
  uint64_t* pfree = pfull + 2;                        // [2]
  uint64_t* qready = pfree + 2;                       // [1]
  uint64_t* ufull = qready + 1;                       // [R]
  uint64_t* uempty = ufull + R;                       // [R]
  uint64_t* done = uempty + R;                        // [2]
  int* s_unit = reinterpret_cast<int*>(done + 2);     // [R]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_unit + R);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  static_assert((2 * NK + 2 * NV + 8 + 1 + 2 * R + 2) * 8 + R * 4 + 8 <= kMqBarBytes, "barrier block");
  // [128][kMqStageRow] the softmax rows' output staging
  uint8_t* s_stage = smem + (NK + NV) * C::KREG + 2 * kMultiQueryMaxSplitBlocks * 4 + kMqBarBytes;

  if (tid == 0) {
    for (int s = 0; s < NK; ++s) {
      mbar_init(smem_u32(kfull + s), 1);
      mbar_init(smem_u32(kempty + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(smem_u32(vfull + s), 1);
      mbar_init(smem_u32(vempty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(sfull + i), 1);
      mbar_init(smem_u32(sfree + i), 4);
      mbar_init(smem_u32(pfull + i), 4);
      mbar_init(smem_u32(pfree + i), 1);
      mbar_init(smem_u32(done + i), 1);
    }
    mbar_init(smem_u32(qready), 4);
    for (int i = 0; i < R; ++i) {
      mbar_init(smem_u32(ufull + i), 1);
      mbar_init(smem_u32(uempty + i), READERS);
    }
    *s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  wait_prior_grid();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_tmem;

  if (warp == 4 || warp == 5) {
    // ------------------------------------------------------------ producers
    const int pw = warp - 4;
    const int box = p.block_size < NKEY ? p.block_size : NKEY;  // token rows per TMA box
    const int per_half = NKEY / box;
    const int nbox = C::HALVES * per_half;                       // boxes of a K (or V) tile
    int g = 0;
    for (int n = 0;; ++n) {
      int u;
      if (pw == 0) {
        u = -1;
        if (lane == 0) {
          const int slot = n % R;
          if (n < R || wait_or_abort(smem_u32(uempty + slot), static_cast<uint32_t>((n / R - 1) & 1), p.err,
                                     s_abort)) {
            u = *s_abort ? -1 : atomicAdd(p.ws_q, 1);
            u = u < U ? p.ws_q[64 + u] : -1;  // the order of mq_order_kernel
          }
          s_unit[slot] = u;
          mbar_arrive(smem_u32(ufull + slot));  // releases the slot's value to the readers
        }
        u = __shfl_sync(kFull, u, 0);
      } else {
        u = mq_read_unit(ufull, uempty, s_unit, n, p.err, s_abort);
      }
      if (u < 0) break;
      const MqUnit w = mq_unit(p, u, nrb, pw == 0 && lane == 0);
      // the unit's block ids into this warp's shared array (it has issued
      // every box of the previous unit)
      const int32_t* blocks = p.block_tables + static_cast<int64_t>(w.b) * p.max_blocks + w.t0 / p.block_size;
      int* ids = s_ids + pw * kMultiQueryMaxSplitBlocks;
      const int nblk = (w.t1 - w.t0 + p.block_size - 1) / p.block_size;
      // eight independent loads per lane in flight at a time (the table row
      // is in L2: the unit-order kernel prefetched it)
      for (int j0 = lane; j0 < nblk; j0 += 32 * 8) {
        int ph[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) ph[q] = j0 + 32 * q < nblk ? __ldg(blocks + j0 + 32 * q) : 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = j0 + 32 * q;
          if (j < nblk) {
            int phys = ph[q];
            if (phys < 0 || phys >= p.num_blocks) {
              if (pw == 0) record_error(p.err, kDevErrBlockId);
              phys = -1;  // fully outside the tensor: the TMA unit fills zeros
            }
            ids[j] = phys;
          }
        }
      }
      __syncwarp();
      // this lane's box of each tile: d-half, block within the tile (warp 4
      // loads the K ring, warp 5 the V ring).  A unit starts at a multiple of
      // 64 tokens and the block size (16 or 32) divides 64, so every box is a
      // whole block: box i of tile k is block k * per_half + i of the unit,
      // from its first row.  The operands are set up once per unit: the issue
      // loop shares its sub-partition with a softmax warp, and every
      // instruction in it delays the next box.
      const int bx = lane / per_half;
      const int i = lane % per_half;
      const int nring = pw == 0 ? NK : NV;
      const uint32_t ring = pw == 0 ? kring : vring;
      uint64_t* rfull = pw == 0 ? kfull : vfull;
      uint64_t* rempty = pw == 0 ? kempty : vempty;
      const CUtensorMap* tmap = pw ? &tmap_v : &tmap_k;
      const uint32_t off = bx * C::HALF_BYTES + i * box * 128;
      const int c0 = bx * L::BOX_ELEMS;
      bool ok = true;
      for (int k = 0; k < w.ntile; ++k, ++g) {
        const int s = g % nring;
        bool go = true;
        if (lane == 0 && g >= nring)
          go = wait_or_abort(smem_u32(rempty + s), static_cast<uint32_t>((g / nring - 1) & 1), p.err, s_abort);
        if (!__shfl_sync(kFull, go ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        const uint32_t dst = ring + s * C::KREG;
        const uint32_t bar = smem_u32(rfull + s);
        if (lane == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bar, C::KREG);
        }
        __syncwarp();
        if (lane < nbox) {
          const int j = k * per_half + i;
          const int phys = j < nblk ? ids[j] : -1;  // past the range: zeros
          tma_load_4d(dst + off, tmap, bar, c0, 0, w.h, phys);
        }
      }
      if (!ok) break;
    }
    if (lane == 0 && *s_abort) {  // the copies in flight land before the stages are released
      const int nring = pw == 0 ? NK : NV;
      uint64_t* rfull = pw == 0 ? kfull : vfull;
      for (int k = g > nring ? g - nring : 0; k < g; ++k)
        mbar_wait(smem_u32(rfull + k % nring), static_cast<uint32_t>((k / nring) & 1), nullptr);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ S issuer
    int g = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int u = mq_read_unit(ufull, uempty, s_unit, n, p.err, s_abort);
      if (u < 0) break;
      const MqUnit w = mq_unit(p, u, nrb, false);
      if (lane == 0) ok = wait_or_abort(smem_u32(qready), static_cast<uint32_t>(n & 1), p.err, s_abort);
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      for (int k = 0; k < w.ntile && ok; ++k, ++g) {
        const int s = g % NK, b = g & 1;
        bool ok2 = true;
        if (lane == 0) {
          ok2 = wait_or_abort(smem_u32(kfull + s), static_cast<uint32_t>((g / NK) & 1), p.err, s_abort);
          if (ok2 && g >= 2)  // the softmax has read S(g-2) out of buffer b
            ok2 = wait_or_abort(smem_u32(sfree + b), static_cast<uint32_t>(((g - 2) >> 1) & 1), p.err, s_abort);
        }
        ok = __shfl_sync(kFull, ok2 ? 1 : 0, 0) != 0;
        if (ok && lane == 0) {
          tc_fence_after();
          const uint32_t kst = kring + s * C::KREG;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(kst + (kk / 4) * C::HALF_BYTES + (kk % 4) * 32, 0, 1024);
            tc_mma_ts(tbase + COL_S + b * NKEY, tbase + COL_Q + kk * 8, bd, IDESC_S, kk > 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(sfull + b));
          tc_commit(smem_u32(kempty + s));  // S(g) has read the K tile
        }
      }
    }
    if (lane == 0) {  // nothing of this thread's may still be running when TMEM is freed
      tc_commit(smem_u32(done));
      mbar_wait(smem_u32(done), 0u, nullptr);
    }
  } else if (warp == 7) {
    // ------------------------------------------------------------ P.V issuer
    int g = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int u = mq_read_unit(ufull, uempty, s_unit, n, p.err, s_abort);
      if (u < 0) break;
      const MqUnit w = mq_unit(p, u, nrb, false);
      for (int k = 0; k < w.ntile && ok; ++k, ++g) {
        const int s = g % NV, b = g & 1;
        bool ok2 = true;
        if (lane == 0) {
          ok2 = wait_or_abort(smem_u32(pfull + b), static_cast<uint32_t>((g >> 1) & 1), p.err, s_abort);
          if (ok2)  // the V tile has arrived (also orders its bytes before the zeroing below)
            ok2 = wait_or_abort(smem_u32(vfull + s), static_cast<uint32_t>((g / NV) & 1), p.err, s_abort);
        }
        ok = __shfl_sync(kFull, ok2 ? 1 : 0, 0) != 0;
        if (!ok) break;
        const uint32_t vst = vring + s * C::KREG;
        // rows of the last block past the sequence end may hold anything (NaN
        // included): zero them in the V tile, P is 0 there
        const int vr0 = w.ctx - (w.t0 + k * NKEY);
        if (vr0 < NKEY) {
          uint8_t* vt = smem + (vst - kring);
          const int first_row = vr0 > 0 ? vr0 : 0;
          const int chunks = (NKEY - first_row) * 8;   // 16-byte chunks per d-half
          for (int c = lane; c < C::HALVES * chunks; c += 32) {
            const int hf = c / chunks, cc = c - hf * chunks;
            *reinterpret_cast<uint4*>(vt + hf * C::HALF_BYTES + first_row * 128 + cc * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t pa = tbase + COL_P + b * NKEY;
#pragma unroll
          for (int kk = 0; kk < NKEY / 16; ++kk) {
            // MN-major V: 8-key groups 1024 B apart, d-halves HALF_BYTES apart
            const uint64_t vd = smem_desc_sw128(vst + kk * 2048, C::HALVES > 1 ? C::HALF_BYTES : 0, 1024);
            tc_mma_ts(tbase + COL_O, pa + kk * 8, vd, IDESC_PV, (k > 0 || kk > 0) ? 1u : 0u);
            tc_mma_ts(tbase + COL_O, pa + NKEY / 2 + kk * 8, vd, IDESC_PV, 1u);
          }
          tc_commit(smem_u32(pfree + b));
          tc_commit(smem_u32(vempty + s));
        }
      }
    }
    if (lane == 0) {
      tc_commit(smem_u32(done + 1));
      mbar_wait(smem_u32(done + 1), 0u, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r_in = warp * 32 + lane;                 // row within the unit's row block
    const uint32_t tl = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    // The softmax works on the raw products S = Q K^T and applies the logit
    // multiplier (scale x log2 e) inside the exponent's FMA; a negative scale
    // enters as negated Q (exact in bf16), so that the multiplier is positive
    // and the row maximum of S maps to the maximum logit.  A zero scale takes
    // the smallest normal multiplier: every logit rounds to 0 all the same.
    const float qk_mult = fmaxf(fabsf(p.qk_log2_scale), 1.17549435e-38f);
    const uint32_t q_sign = p.qk_log2_scale < 0.f ? 0x80008000u : 0u;
    uint4 qw[D / 8];                                   // the next unit's Q row
    // load this thread's Q row of unit w (zeros past the rows)
    auto load_q = [&](const MqUnit& w) {
      const int row = w.row0 + r_in;
      const int64_t orow = (static_cast<int64_t>(w.b) * QL + row / G) * H_q + w.h * G + row % G;
      const uint16_t* qr = row < rows ? static_cast<const uint16_t*>(p.q) + orow * D : nullptr;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        qw[c] = qr ? *reinterpret_cast<const uint4*>(qr + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
        qw[c].x ^= q_sign;
        qw[c].y ^= q_sign;
        qw[c].z ^= q_sign;
        qw[c].w ^= q_sign;
      }
    };
    // row r of Q into TMEM lane r as bf16 pairs (element 2j in the low half
    // of column j, the memory order of the loaded words), then tell the S issuer
    auto store_q = [&]() {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[4 * j] = qw[4 * c + j].x;
          v[4 * j + 1] = qw[4 * c + j].y;
          v[4 * j + 2] = qw[4 * c + j].z;
          v[4 * j + 3] = qw[4 * c + j].w;
        }
        tmem_st16(tl + COL_Q + 16 * c, v);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(qready));
    };
    int g = 0;
    bool ok = true;
    int u = mq_read_unit(ufull, uempty, s_unit, 0, p.err, s_abort);
    MqUnit w;
    if (u >= 0) {
      w = mq_unit(p, u, nrb, false);
      load_q(w);
      store_q();
    }
    for (int n = 0; u >= 0 && ok; ++n) {
      const int row = w.row0 + r_in;
      const bool row_ok = row < rows;
      const int64_t orow = (static_cast<int64_t>(w.b) * QL + row / G) * H_q + w.h * G + row % G;
      // tokens this row may attend: [0, lim).  A padding row (past the
      // unit's q_len x G rows) takes no mask: its P feeds only O rows that
      // are never written, and a mask there would run the masking loop of
      // its whole warp on every tile.
      const int lim = row_ok ? min(w.t1, w.ctx - QL + row / G + 1) : w.t1 + NKEY;
      // a warp past the unit's last query row (q_len x G rows fill only part
      // of the 128-row block) keeps the barrier phases and computes nothing:
      // its P rows feed only O rows that are never written
      const bool idle = IDLE && w.row0 + warp * 32 >= rows;
      float m_used = -CUDART_INF_F, lsum = 0.f;
      if (idle) {
        for (int k = 0; k < w.ntile; ++k, ++g) {
          const int b = g & 1;
          ok = __all_sync(kFull, wait_or_abort(smem_u32(sfull + b), static_cast<uint32_t>((g >> 1) & 1), p.err,
                                               s_abort));
          if (!ok) break;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(sfree + b));
          if (g >= 2) {  // the phase order of P[b]: P(g-2).V has been issued and read it
            ok = __all_sync(kFull, wait_or_abort(smem_u32(pfree + b), static_cast<uint32_t>(((g - 2) >> 1) & 1),
                                                 p.err, s_abort));
            if (!ok) break;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(pfull + b));
        }
      } else
      for (int k = 0; k < w.ntile; ++k, ++g) {
        const int b = g & 1;
        ok = __all_sync(kFull, wait_or_abort(smem_u32(sfull + b), static_cast<uint32_t>((g >> 1) & 1), p.err,
                                             s_abort));
        if (!ok) break;
        tc_fence_after();
        float x[NKEY];
        {
          uint32_t v[NKEY / 16][16];
#pragma unroll
          for (int c = 0; c < NKEY / 16; ++c) tmem_ld16(tl + COL_S + b * NKEY + 16 * c, v[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < NKEY / 16; ++c)
#pragma unroll
            for (int i = 0; i < 16; ++i) x[16 * c + i] = __uint_as_float(v[c][i]);
        }
        tc_fence_before();  // S[b] may be overwritten
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sfree + b));
        const int valid = lim - (w.t0 + k * NKEY);
        if (__any_sync(kFull, valid < NKEY)) {
#pragma unroll
          for (int i = 0; i < NKEY; ++i)
            if (i >= valid) x[i] = -CUDART_INF_F;
        }
        float mt;
        {  // eight chains of three-input maxima, then their maximum (in log2 units)
          static_assert(NKEY == 64, "eight chains of eight keys");
          float mp[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            mp[j] = max3f(x[j], x[8 + j], x[16 + j]);
            mp[j] = max3f(mp[j], x[24 + j], x[32 + j]);
            mp[j] = max3f(mp[j], x[40 + j], x[48 + j]);
            mp[j] = fmaxf(mp[j], x[56 + j]);
          }
          mt = max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])) * qk_mult;
        }
        float alpha = 1.f;
        bool resc = false;
        if (m_used == -CUDART_INF_F) {
          m_used = mt;  // nothing accumulated yet for this row
        } else if (mt > m_used + 8.f) {
          alpha = fast_exp2(m_used - mt);
          m_used = mt;
          resc = true;
        }
        if (__any_sync(kFull, resc)) {
          // O holds tiles 0..k-1 of the unit once P(g-1).V has completed
          ok = __all_sync(kFull, wait_or_abort(smem_u32(pfree + ((g - 1) & 1)),
                                               static_cast<uint32_t>(((g - 1) >> 1) & 1), p.err, s_abort));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[2][16];
            tmem_ld16(tl + COL_O + c0, v[0]);
            tmem_ld16(tl + COL_O + c0 + 16, v[1]);
            tmem_wait_ld();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
              for (int i = 0; i < 16; ++i) v[hh][i] = __float_as_uint(__uint_as_float(v[hh][i]) * alpha);
            tmem_st16(tl + COL_O + c0, v[0]);
            tmem_st16(tl + COL_O + c0 + 16, v[1]);
          }
          tmem_wait_st();
        }
        lsum *= alpha;
        if (g >= 2) {  // P(g-2).V has read P[b]
          ok = __all_sync(kFull, wait_or_abort(smem_u32(pfree + b), static_cast<uint32_t>(((g - 2) >> 1) & 1),
                                               p.err, s_abort));
          if (!ok) break;
          tc_fence_after();
        }
        const float mu = m_used == -CUDART_INF_F ? 0.f : m_used;
        const float2 neg_mu = make_float2(-mu, -mu);
        const float2 mult2 = make_float2(qk_mult, qk_mult);
        float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c0 = 0; c0 < NKEY / 2; c0 += 16) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 e = __ffma2_rn(make_float2(x[2 * (c0 + i)], x[2 * (c0 + i) + 1]), mult2, neg_mu);
            const float2 pp = make_float2(fast_exp2(e.x), fast_exp2(e.y));
            ls[i & 1] = __fadd2_rn(ls[i & 1], pp);
            hi[i] = pack_bf16x2(pp.x, pp.y);
            const float2 rr = __fadd2_rn(pp, make_float2(-bf16lo_to_f32(hi[i]), -bf16hi_to_f32(hi[i])));
            lo[i] = pack_bf16x2(rr.x, rr.y);
          }
          tmem_st16(tl + COL_P + b * NKEY + c0, hi);
          tmem_st16(tl + COL_P + b * NKEY + NKEY / 2 + c0, lo);
        }
        lsum += (ls[0].x + ls[1].x) + (ls[0].y + ls[1].y);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(pfull + b));   // P(g) is in TMEM
      }
      if (!ok) break;
      // the next unit: its Q rows are loaded now and go into TMEM once this
      // unit's last P.V has completed (every S of this unit has completed
      // too: the loop above saw each one's sfull)
      const int u_next = mq_read_unit(ufull, uempty, s_unit, n + 1, p.err, s_abort);
      MqUnit w_next;
      if (u_next >= 0) {
        w_next = mq_unit(p, u_next, nrb, false);
        load_q(w_next);
      }
      // ---- this unit's result: a workspace piece, or (one split) the output row
      if (w.ntile > 0)
        ok = __all_sync(kFull, wait_or_abort(smem_u32(pfree + ((g - 1) & 1)),
                                             static_cast<uint32_t>(((g - 1) >> 1) & 1), p.err, s_abort));
      if (!ok) break;
      // The next unit's Q goes in first, so that its first S runs beside this
      // epilogue.  Its first P.V, which overwrites O, waits for P from these
      // warps, which they write only after reading O below.
      if (u_next >= 0) store_q();
      const bool writes = w.t0 < w.ctx || (w.ctx == 0 && w.split == 0);
      const bool direct = w.nsplit <= 1;
      const int64_t piece = orow * p.slots_per_row + w.split;
      if (writes && !idle) {
        if (w.ntile > 0) tc_fence_after();
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const float sc = direct ? inv : 1.f;
        float* dst_row = direct ? p.out + orow * D : p.ws_o + piece * D;
        // O leaves through shared memory, 32 columns of the warp's 32 rows per
        // pass: each thread stages its row piece, then every store
        // instruction writes four whole 128-byte row pieces (16-byte stores
        // straight from the TMEM rows would scatter each one over 32 rows).
        // Lane l stores chunk l % 8 of rows l / 8 + 4 j; rd[j] is that row's
        // destination (0: no such row).
        uint8_t* swarp = s_stage + warp * 32 * kMqStageRow;
        uint8_t* srow = swarp + lane * kMqStageRow;
        const uint64_t my_dst = row_ok ? reinterpret_cast<uint64_t>(dst_row) : 0ull;
        uint64_t rd[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) rd[j] = __shfl_sync(kFull, my_dst, (lane >> 3) + 4 * j);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[2][16];
          if (w.ntile > 0) {
            tmem_ld16(tl + COL_O + c0, v[0]);
            tmem_ld16(tl + COL_O + c0 + 16, v[1]);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[0][i] = v[1][i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(srow + 16 * i) =
                make_float4(__uint_as_float(v[i / 4][4 * (i % 4)]) * sc, __uint_as_float(v[i / 4][4 * (i % 4) + 1]) * sc,
                            __uint_as_float(v[i / 4][4 * (i % 4) + 2]) * sc,
                            __uint_as_float(v[i / 4][4 * (i % 4) + 3]) * sc);
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 val =
                *reinterpret_cast<const float4*>(swarp + ((lane >> 3) + 4 * j) * kMqStageRow + (lane & 7) * 16);
            if (rd[j] != 0ull) reinterpret_cast<float4*>(rd[j])[c0 / 4 + (lane & 7)] = val;
          }
          __syncwarp();  // the warp has read the staging before the next pass
        }
        if (row_ok && !direct) {
          p.ws_ml[piece * 2] = m_used;
          p.ws_ml[piece * 2 + 1] = lsum;
        }
      }
      u = u_next;
      w = w_next;
    }
  }
  allow_next_grid();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D>
int mq_tc_smem_bytes() {
  // at least 120 KB: one CTA per SM (it holds all 512 TMEM columns)
  const int need = (kMqKStages + kMqVStages) * TcTile<D, kMqTile>::KREG + 2 * kMultiQueryMaxSplitBlocks * 4 +
                   kMqBarBytes + 128 * kMqStageRow + 1024;
  return need > 120 * 1024 ? need : 120 * 1024;
}

template <int D, bool IDLE>
cudaError_t launch_mq_tc_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           cudaStream_t stream) {
  auto kern = mq_tc_kernel<D, IDLE>;
  const int smem = mq_tc_smem_bytes<D>();
  static int configured[64] = {};
  cudaError_t e = set_smem_once(kern, smem, configured);
  if (e != cudaSuccess) return e;
  // plain launches: the order kernel writes the unit order and zeroes the
  // counter just before the persistent grid starts
  mq_order_kernel<<<1, 1024, 0, stream>>>(p, p.ws_q + 64);
  kern<<<dim3(p.workers), dim3(256), smem, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_cascade_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                             cudaStream_t stream) {
  auto kern = cascade_prefix_kernel<D>;
  // at least 120 KB: one CTA per SM (it holds all 512 TMEM columns)
  const int smem = CascadeShape<D>::BYTES > 120 * 1024 ? CascadeShape<D>::BYTES : 120 * 1024;
  static int configured[64] = {};
  cudaError_t e = set_smem_once(kern, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(CascadeShape<D>::THREADS), smem, stream, tk, tv, p);
}

}  // namespace

cudaError_t launch_cascade_prefix(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream) {
  const int rows = p.batch * p.group;
  const int nps = (p.prefix_len + p.prefix_split_tokens - 1) / p.prefix_split_tokens;
  const dim3 grid((rows + kCascadeRowsTc - 1) / kCascadeRowsTc, p.num_kv_heads, nps);
  if (p.head_dim == 128) return launch_cascade_t<128>(p, tk, tv, grid, stream);
  return launch_cascade_t<64>(p, tk, tv, grid, stream);
}

cudaError_t launch_wait_selftest(int which, uint64_t limit_ns, int* err, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 128, 0, stream>>>(which, limit_ns, err);
  return cudaGetLastError();
}

cudaError_t launch_multi_query_tc(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream) {
  const int last_rows = (p.q_len * p.group) % 128;        // rows of the last 128-row block (0: full)
  const bool idle = last_rows != 0 && last_rows <= 96;   // a warp of that block has no query row
  if (p.head_dim == 128)
    return idle ? launch_mq_tc_t<128, true>(p, tk, tv, stream) : launch_mq_tc_t<128, false>(p, tk, tv, stream);
  return idle ? launch_mq_tc_t<64, true>(p, tk, tv, stream) : launch_mq_tc_t<64, false>(p, tk, tv, stream);
}

}  // namespace pkv
