// Device-side building blocks for the sm_103a kernels: shared-memory address
// conversion, mbarrier + TMA (cp.async.bulk.tensor) staging with time-bounded
// waits, ldmatrix / movmatrix / mma.sync fragments, and the FP8 E4M3 / bf16 /
// f16 conversions.  Everything is inline PTX written for this library.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pkv_internal.h"

namespace pkv {

// Give up on a pipeline wait after this long (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // one second

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// First error recorded wins; later ones are dropped.
__device__ __forceinline__ void record_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Try-waits between two reads of the global timer: the timer read is slow,
// and a phase that completes while the thread reads it would be noticed late.
constexpr uint32_t kWaitTriesPerClockRead = 256;

// Wait for phase `parity` of the barrier, at most about `limit_ns` (one
// second unless a self-test asks for less).  On time-out the error word gets
// PKV_DEVERR_WAIT_TIMEOUT and false is returned.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (n % kWaitTriesPerClockRead == 0) {
      const uint64_t t = global_timer_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > limit_ns) {
        record_error(err, kDevErrWaitTimeout);
        return false;
      }
    }
  }
}

// 4-D tiled TMA load global -> shared, completing on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Barrier `id` (1..15; 0 is __syncthreads) over the first `threads` threads
// that reach it (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Bulk copy shared -> global of `bytes` (a multiple of 16; both addresses
// 16-byte aligned), in this thread's bulk group.
__device__ __forceinline__ void bulk_store_s2g(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk copies have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until this thread's bulk copies have completed (their writes done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- fragments

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Transpose of an 8x8 b16 matrix held one row pair per lane (ldmatrix layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// D += A(16x16, row) * B(16x8, col); fp32 accumulate.  Volatile so that the
// MMAs reading ldmatrix results stay ahead of the next TMA write into the
// same stage in program order.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- conversions

// Two floats -> packed bf16x2, round to nearest even; `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two floats -> packed f16x2, round to nearest even; `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two E4M3 codes (low byte first) -> f16x2 (exact: E4M3 is a subset of f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(codes));
  return d;
}

// Two floats -> two E4M3 codes, RNE with saturation to +-448; `lo` -> low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Byte permute: picks bytes of {b:a} by the 4 selector nibbles.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ float f16lo_to_f32(uint32_t x) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(x & 0xFFFFu)));
}
__device__ __forceinline__ float f16hi_to_f32(uint32_t x) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(x >> 16)));
}

// ---------------------------------------------------------------- KV rows
// Encoding of new K / V rows into the cache, shared by the append kernel and
// the decode kernel's fused append: sources bf16 or f32, caches bf16 (bf16
// sources copied bit for bit, f32 sources rounded to nearest even) or E4M3
// (RNE-satfinite of x / scale, x / scale an IEEE binary32 quotient).  The
// element types are kEncBF16 / kEncF32 / kEncE4M3 (pkv_internal.h).

// Eight source elements as floats (bf16 widening is exact); `raw` keeps the
// bf16 bits for the bit copy.
template <int SRC>
__device__ __forceinline__ void enc_load8(const void* base, int64_t elem, float (&x)[8], uint4& raw) {
  if constexpr (SRC == kEncBF16) {
    raw = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16lo_to_f32(w[i]);
      x[2 * i + 1] = bf16hi_to_f32(w[i]);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// Eight elements into the cache at element `elem` (DST kEncBF16 or kEncE4M3).
template <int SRC, int DST>
__device__ __forceinline__ void enc_store8(void* cache, int64_t elem, const float (&x)[8], const uint4& raw,
                                           float scale) {
  if constexpr (DST == kEncBF16) {
    uint4 o;
    if constexpr (SRC == kEncBF16) {
      o = raw;  // bit copy
    } else {
      o.x = pack_bf16x2(x[0], x[1]);
      o.y = pack_bf16x2(x[2], x[3]);
      o.z = pack_bf16x2(x[4], x[5]);
      o.w = pack_bf16x2(x[6], x[7]);
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(cache) + elem) = o;
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __fdiv_rn(x[2 * i], scale);
      const float hi = __fdiv_rn(x[2 * i + 1], scale);
      w[i] = f32x2_to_e4m3x2(lo, hi);
    }
    uint2 o;
    o.x = w[0] | (w[1] << 16);
    o.y = w[2] | (w[3] << 16);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + elem) = o;
  }
}

// 2^x on the special-function unit.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


}  // namespace pkv
