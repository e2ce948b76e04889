// Whole-block copies of the paged K/V caches: the device half of
// copy-on-write (a shared block duplicated before its first private write,
// [FN] "Sub-Millisecond Token Scheduling...", "Paged KV-Cache with Radix Tree
// Prefix Cache": copy-on-write pointers) and of tiering (blocks moved between
// the HBM pool and a pool in host memory that the GPU addresses directly,
// [UI] "Architecting Multi-Tier Disaggregated KV-Cache Hierarchies...",
// "C++ Block Scheduler and Asynchronous Fetch Kernel": promote / demote a
// block between Tier-1 HBM and Tier-2 host memory).
//
// A block of one cache is num_kv_heads * block_size * head_dim elements,
// contiguous.  The kernel walks the flat space of 16-byte words of all pairs
// (K words, then V words, pair after pair) with a grid-stride loop over one
// wave of resident CTAs; each thread issues four independent 16-byte loads
// before its four stores, so a warp keeps 2 KB in flight.  Source and destination ids are range-checked;
// a bad pair is skipped and recorded in the device error word.

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p) {
  // Start the next kernel's launch now (it waits for this grid before it
  // reads), then wait for the previous kernel: it may still read a source or
  // write a destination block.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t per_pair = 2 * p.block_vec;
  const int64_t total = p.n_pairs * per_pair;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < total;
       base += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
    uint4* dst[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      dst[u] = nullptr;
      const int64_t idx = base + u * stride;
      if (idx >= total) continue;
      const int64_t pair = idx / per_pair;
      const int64_t r = idx - pair * per_pair;
      const bool is_v = r >= p.block_vec;
      const int64_t w = is_v ? r - p.block_vec : r;
      const int64_t s = p.src[pair], d = p.dst[pair];
      if (s < 0 || s >= p.src_blocks || d < 0 || d >= p.dst_blocks) {
        if (w == 0 && !is_v) record_error(p.err, kDevErrBlockId);
        continue;
      }
      const uint4* src = static_cast<const uint4*>(is_v ? p.v_src : p.k_src) + s * p.block_vec + w;
      v[u] = *src;
      dst[u] = static_cast<uint4*>(is_v ? p.v_dst : p.k_dst) + d * p.block_vec + w;
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (dst[u] != nullptr) *dst[u] = v[u];
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream) {
  const int64_t words = p.n_pairs * 2 * p.block_vec;
  if (words == 0) return cudaSuccess;
  // one full wave of resident CTAs (a partial second wave leaves SMs idle at
  // the end), fewer when the copy is small or the caller bounds it
  static int resident[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (resident[dev] == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, copy_blocks_kernel, kCopyThreads, 0);
    if (e != cudaSuccess) return e;
    resident[dev] = sms * (per_sm > 0 ? per_sm : 1);
  }
  const int64_t want = (words + kCopyThreads * kCopyUnroll - 1) / (kCopyThreads * kCopyUnroll);
  int64_t cap = resident[dev];
  if (p.max_ctas > 0 && p.max_ctas < cap) cap = p.max_ctas;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, p);
}

}  // namespace pkv
