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
// contiguous.  The work is cut into chunks of 32 KB of one block (the K block
// of a pair, then its V block, pair after pair), which one wave of resident
// CTAs takes in a grid-stride loop: a CTA step reads the pair's ids once (the
// next step's ids are loaded while this one copies), then each thread issues
// eight independent 16-byte loads before its eight stores, so a warp keeps
// 4 KB in flight.  Source and destination ids are range-checked; a bad pair
// is skipped and recorded in the device error word.

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;
constexpr int64_t kChunkWords = kCopyThreads * kCopyUnroll;  // 16-byte words per CTA step (32 KB)

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p) {
  // Start the next kernel's launch now (it waits for this grid before it
  // reads), then wait for the previous kernel: it may still read a source or
  // write a destination block.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t per_block = (p.block_vec + kChunkWords - 1) / kChunkWords;  // chunks of one block
  const int64_t total = p.n_pairs * 2 * per_block;
  // ids of chunk c's pair
  auto ids = [&](int64_t c, int64_t& s, int64_t& d) {
    const int64_t pair = c / (2 * per_block);
    s = p.src[pair];
    d = p.dst[pair];
  };
  int64_t c = blockIdx.x;
  int64_t s = 0, d = 0;
  if (c < total) ids(c, s, d);
  while (c < total) {
    const int64_t c_next = c + gridDim.x;
    int64_t s_next = 0, d_next = 0;
    if (c_next < total) ids(c_next, s_next, d_next);  // in flight while this chunk copies
    const int64_t pb = c / per_block;                 // (pair, cache): K of pair pb/2, or its V
    const bool is_v = (pb & 1) != 0;
    const int64_t w0 = (c - pb * per_block) * kChunkWords;
    if (s < 0 || s >= p.src_blocks || d < 0 || d >= p.dst_blocks) {
      if (w0 == 0 && !is_v && threadIdx.x == 0) record_error(p.err, kDevErrBlockId);
    } else {
      const uint4* src = static_cast<const uint4*>(is_v ? p.v_src : p.k_src) + s * p.block_vec + w0;
      uint4* dst = static_cast<uint4*>(is_v ? p.v_dst : p.k_dst) + d * p.block_vec + w0;
      const int64_t n = p.block_vec - w0 < kChunkWords ? p.block_vec - w0 : kChunkWords;
      uint4 v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int i = threadIdx.x + u * kCopyThreads;
        if (i < n) v[u] = src[i];
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int i = threadIdx.x + u * kCopyThreads;
        if (i < n) dst[i] = v[u];
      }
    }
    c = c_next;
    s = s_next;
    d = d_next;
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
  const int64_t want = p.n_pairs * 2 * ((p.block_vec + kChunkWords - 1) / kChunkWords);  // chunks
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
