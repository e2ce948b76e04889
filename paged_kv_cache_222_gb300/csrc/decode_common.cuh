// Pieces shared by the attention kernels (decode.cu, cascade.cu,
// multi_query.cu): the shared-memory layout of TMA-staged K/V tiles, context
// clamping, programmatic-dependent-launch hooks and the launch helper.
#pragma once

#include <math_constants.h>

#include <utility>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

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
  // 16 KB of stages per warp: 64 KB per 4-warp CTA, three CTAs per SM, so one
  // CTA's ramp-up and merge overlap the other two CTAs' streaming
  static constexpr int NS = (16384 / STAGEB) > 8 ? 8 : (16384 / STAGEB);
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

// Context length as every kernel sees it: clamped to what the grid, the
// workspace and the block table can hold (the violation is recorded once).
__device__ __forceinline__ int clamp_ctx(const DecodeParams& p, int ctx) {
  const int64_t table_cap = static_cast<int64_t>(p.max_blocks) * p.block_size;
  const int lim = static_cast<int>(table_cap < p.max_ctx ? table_cap : p.max_ctx);
  return ctx < 0 ? 0 : (ctx > lim ? lim : ctx);
}

// Wait for the kernel that precedes this one in the stream (programmatic
// dependent launch); a no-op when launched without that attribute.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while its predecessor in the stream drains; it waits for the
// predecessor's completion (griddepcontrol.wait) before touching its data.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, int smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared-memory limit once per device (again after
// pkv_shutdown, which starts a new configuration epoch: a caller may reset the
// device after it, and a reset drops the limits set in the old context).
template <class K>
cudaError_t set_smem_once(K kern, int smem, int (&configured)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int epoch = config_epoch();
  if (configured[dev] != epoch) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = epoch;
  }
  return cudaSuccess;
}

}  // namespace pkv
