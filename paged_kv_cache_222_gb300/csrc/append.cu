// KV append: scatter each new token's K/V rows into their cache slots, copying
// bf16 or quantising to FP8 E4M3 with a per-row, per-KV-head scale.
//
// What it computes: [SC] "LLM inference: prefill, decode, KV cache", section
// "4. Internal workings", step 5 (the new token's K/V are appended to the
// cache); FP8 E4M3 with per-head scales: [FN] "Sub-Millisecond Token
// Scheduling...", FAQ "How much HBM memory does FP8 KV-cache quantization
// save?".  Slot = physical_block * block_size + offset, negative = skip.
//
// Mapping: one thread per 8 consecutive elements of one (token, head) row, so a
// warp moves 2 (D=128) or 4 (D=64) whole rows with 16-byte (bf16) or 8-byte
// (E4M3) stores; loads are 16-byte (bf16 source) or 2x16-byte (f32 source).
// Grid-stride, so any number of rows fits a bounded grid.
//
// The slot-mapping kernel turns (sequence, logical position) pairs into those
// flat slots through the block tables ([SC] "PagedAttention & Memory
// Management (vLLM)": logical block j of a sequence lives in the physical
// block its table names).

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kBF16 = kEncBF16, kF32 = kEncF32, kE4M3 = kEncE4M3;

template <int SRC, int DST>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  // Let the next kernel in the stream start launching now (it waits for this
  // grid to finish before it reads anything), then wait for the previous one:
  // a slot written here may be one it still reads.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int D = p.head_dim;
  const int H = p.num_kv_heads;
  const int per_row = D / 8;
  const int64_t total = p.n_tokens * H * per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int64_t row = idx / per_row;  // token * H + head
    const int part = static_cast<int>(idx - row * per_row);
    const int64_t tok = row / H;
    const int h = static_cast<int>(row - tok * H);
    const int64_t slot = p.slots[tok];
    if (slot < 0) continue;
    if (slot >= p.num_slots) {
      if (part == 0 && h == 0) record_error(p.err, kDevErrSlot);
      continue;
    }
    const int64_t blk = slot / p.block_size;
    const int64_t off = slot - blk * p.block_size;
    const int64_t src_elem = row * D + part * 8;
    const int64_t dst_elem = ((blk * H + h) * p.block_size + off) * D + part * 8;
    float ks = 1.f, vs = 1.f;
    if constexpr (DST == kE4M3) {
      ks = p.k_scale[tok * p.scale_stride + h];
      vs = p.v_scale[tok * p.scale_stride + h];
    }
    float x[8];
    uint4 raw;
    enc_load8<SRC>(p.k_new, src_elem, x, raw);
    enc_store8<SRC, DST>(p.k_cache, dst_elem, x, raw, ks);
    enc_load8<SRC>(p.v_new, src_elem, x, raw);
    enc_store8<SRC, DST>(p.v_cache, dst_elem, x, raw, vs);
  }
}

// Slot of each new token: the block table's entry for the token's logical
// block, times the block size, plus its offset in the block.  One thread per
// token; a negative position is padding (slot -1, nothing recorded).
__global__ void __launch_bounds__(256) slot_mapping_kernel(SlotParams p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t cap = static_cast<int64_t>(p.max_blocks) * p.block_size;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.n; i += stride) {
    const int64_t pos = p.positions[i];
    int64_t slot = -1;
    if (pos >= 0) {
      const int64_t seq = p.seq_index != nullptr ? p.seq_index[i] : i;
      if (seq < 0 || seq >= p.num_seqs || pos >= cap) {
        record_error(p.err, kDevErrContextLen);
      } else {
        const int64_t j = pos / p.block_size;
        const int32_t blk = p.block_tables[seq * p.max_blocks + j];
        if (blk < 0 || blk >= p.num_blocks)
          record_error(p.err, kDevErrBlockId);
        else
          slot = static_cast<int64_t>(blk) * p.block_size + (pos - j * p.block_size);
      }
    }
    p.slots[i] = slot;
  }
}

}  // namespace

cudaError_t launch_slot_mapping(const SlotParams& p, cudaStream_t stream) {
  if (p.n == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (p.n + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 152 * 8 ? want : 152 * 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, slot_mapping_kernel, p);
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const int64_t work = p.n_tokens * p.num_kv_heads * (p.head_dim / 8);
  if (work == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (work + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 152 * 32 ? want : 152 * 32);
  void (*kern)(AppendParams);
  if (p.cache_dtype == kBF16)
    kern = p.src_dtype == kBF16 ? append_kernel<kBF16, kBF16> : append_kernel<kF32, kBF16>;
  else
    kern = p.src_dtype == kBF16 ? append_kernel<kBF16, kE4M3> : append_kernel<kF32, kE4M3>;
  // programmatic dependent launch: may be scheduled while the previous kernel
  // drains; the kernel itself waits for it before touching memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace pkv
