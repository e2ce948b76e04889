// Internal interface between the C ABI (api.cu) and the kernel translation
// units (append.cu, decode.cu).  Not installed; no stability promise.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pkv {

// Mirrors PKV_DEVERR_* of pkv.h (kept separate so device code needs no C ABI).
constexpr int kDevErrWaitTimeout = 1;
constexpr int kDevErrBlockId = 2;
constexpr int kDevErrContextLen = 3;
constexpr int kDevErrSlot = 4;

// Tokens per pipeline tile: one mma M dimension of keys.
constexpr int kTileTokens = 16;
// Consumer warps per decode CTA.
constexpr int kDecodeWarps = 4;

enum KernelKind {
  kKindAppend = 0,
  kKindDecodeSplit = 1,
  kKindCombine = 2,
  kKindCascadePrefix = 3,
  kKindBlockCopy = 4,
  kKindMultiQuery = 5,
  kKindSlotMapping = 6,
  kNumKernelKinds = 8  // room for later kinds; the trace aggregates by kind
};

// Decode work split: balanced stream-K ranges over the flattened
// (sequence, head, tile) space, or fixed `split_tokens` chunks per sequence.
constexpr int kModeStreamK = 0;
constexpr int kModeFixedSplit = 1;
// Largest batch the stream-K kernel takes (its tile prefix lives in shared
// memory); larger batches use fixed splits.
constexpr int kMaxStreamKBatch = 2048;

struct AppendParams {
  const void* k_new;
  const void* v_new;
  const int64_t* slots;
  void* k_cache;
  void* v_cache;
  const float* k_scale;
  const float* v_scale;
  int64_t scale_stride;
  int64_t n_tokens;
  int64_t num_slots;  // num_blocks * block_size
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t src_dtype;    // PKV_BF16 / PKV_F32
  int32_t cache_dtype;  // PKV_BF16 / PKV_E4M3
  int* err;
};

// Flat cache slots of new tokens from the block tables.
struct SlotParams {
  const int32_t* block_tables;  // [num_seqs, max_blocks]
  const int64_t* seq_index;     // [n] sequence of token i, or NULL: token i is sequence i
  const int64_t* positions;     // [n] logical position of token i (< 0: padding)
  int64_t* slots;               // [n] out: block * block_size + offset, -1 for padding
  int64_t n;
  int64_t num_blocks;
  int32_t num_seqs;
  int32_t max_blocks;
  int32_t block_size;
  int* err;
};

// Element types of K / V rows being encoded into the cache: the sources of
// an append (bf16, f32) and the cache's own (bf16, E4M3).
constexpr int kEncBF16 = 0, kEncF32 = 1, kEncE4M3 = 2;

struct DecodeParams {
  const void* q;              // bf16 [B, H_q, D]
  const int32_t* block_tables;  // [B, MB]
  const int32_t* context_lens;  // [B]
  float* out;                 // [B, H_q, D]
  float* ws_o;                // fixed split: [B, H_q, S, D]; stream-K: [2W, GP, D]
  float* ws_ml;               // fixed split: [B, H_q, S, 2]; stream-K: [2W, GP, 2]
  int* ws_q;                  // stream-K: tile prefix over sequences [B + 1];
                              // tcgen05 multi-token: the work-unit counter
  const float* k_scale;
  const float* v_scale;
  int64_t scale_stride;
  int64_t num_blocks;
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;              // G = H_q / H_kv
  int32_t head_dim;
  int32_t block_size;
  int32_t max_blocks;         // MB
  int32_t max_ctx;
  int32_t split_tokens;
  int32_t max_splits;
  float qk_log2_scale;        // softmax scale * log2(e)
  int32_t cache_dtype;
  int32_t mode;               // kModeStreamK / kModeFixedSplit
  int32_t workers;            // stream-K: warps of the persistent grid (W);
                              // tcgen05 multi-token: CTAs of the persistent grid
  // cascade (shared-prefix) decode; zero / -1 / NULL otherwise
  int32_t token_offset;       // fixed split: attend tokens [token_offset, ctx)
  int32_t force_partial;      // fixed split: always write partials, never `out`
  int32_t extra_slot;         // combine: first workspace slot of the prefix pieces (-1: none)
  int32_t extra_count;        // combine: number of prefix pieces per row
  int32_t slots_per_row;      // fixed split / cascade: workspace slots per (b, hq) row
  const int32_t* prefix_blocks;  // [prefix_len / block_size] physical blocks
  int32_t prefix_len;
  int32_t prefix_split_tokens;   // prefix tokens per prefix CTA (multiple of 64)
  // multi-token queries: q_len new tokens per sequence (1 for decode)
  int32_t q_len;
  // fixed split, fused append: each sequence's newest token (position
  // context_lens[b] - 1) is written from k_new / v_new [B, H_kv, D] into its
  // slot by the CTA that attends it, before that CTA's first load
  int32_t new_src;            // 0: no append; else kEncBF16 + 1 or kEncF32 + 1
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  int* err;
};

// Whole-block copies between (or within) block pools: pair i copies block
// src[i] of the K and V caches to block dst[i].
struct CopyParams {
  const void* k_src;      // K cache the sources live in
  const void* v_src;
  void* k_dst;            // K cache the destinations live in
  void* v_dst;
  const int32_t* src;     // [n_pairs] source block ids
  const int32_t* dst;     // [n_pairs] destination block ids
  int64_t n_pairs;
  int64_t block_vec;      // 16-byte words per block of one cache
  int64_t src_blocks;     // valid source ids: [0, src_blocks)
  int64_t dst_blocks;     // valid destination ids: [0, dst_blocks)
  int32_t max_ctas;       // grid bound (0: as many as the copy can use)
  int* err;
};

// Message returned by pkv_last_error() on this host thread.
void set_last_error(const char* msg);

// Configuration epoch (>= 1): pkv_shutdown starts a new one, after which every
// per-device set-up the launchers cached (shared-memory limits) is made again.
int config_epoch();

// Launchers (return the launch's cudaError_t; nothing is synchronised).
cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream);
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_slot_mapping(const SlotParams& p, cudaStream_t stream);
cudaError_t launch_decode_split(const DecodeParams& p, const CUtensorMap& tmap_k,
                                const CUtensorMap& tmap_v, cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_cascade_prefix(const DecodeParams& p, const CUtensorMap& tmap_k,
                                  const CUtensorMap& tmap_v, cudaStream_t stream);
cudaError_t launch_multi_query(const DecodeParams& p, const CUtensorMap& tmap_k,
                               const CUtensorMap& tmap_v, cudaStream_t stream);
// Multi-token queries of 64 or more rows per (sequence, KV head) on tcgen05
// (the cascade kernel's pipeline, one 128-row group per CTA).
cudaError_t launch_multi_query_tc(const DecodeParams& p, const CUtensorMap& tmap_k,
                                  const CUtensorMap& tmap_v, cudaStream_t stream);
// Self-test of the bounded waits (0: mbarrier wait; 1: tensor-core CTA abort
// path); records PKV_DEVERR_WAIT_TIMEOUT after about limit_ns.
cudaError_t launch_wait_selftest(int which, uint64_t limit_ns, int* err, cudaStream_t stream);
// Rows (q_len * G) from which multi-token queries take the tcgen05 kernel.
// Its speed hardly depends on the rows (0.68-0.70 of HBM from 8 to 128 rows
// on the 70B-class GQA batch); the mma.sync kernel measured 0.82 at 16 rows,
// 0.65 at 24, 0.63 at 32 and 0.41 at 40.
constexpr int kMultiQueryTcRows = 17;

// Multi-token query kernel: 64-token tiles, rows of (query token, head) pairs
// in 16-row warp groups; the block ids of one split staged in shared memory.
constexpr int kMultiQueryTile = 64;
constexpr int kMultiQueryMaxSplitBlocks = 1024;
// Token lanes (warps sharing the same 16 rows) for R rows per (sequence, head).
inline int multi_query_lanes(int rows) { return rows <= 16 ? 4 : (rows <= 32 ? 2 : 1); }

// Rows of query heads one cascade prefix CTA covers: two groups of 128 TMEM
// lanes.
constexpr int kCascadeRowsTc = 256;
// Keys per cascade prefix tile (4 sub-tiles of kTileTokens).
constexpr int kCascadeTile = 64;
// Blocks of one cascade prefix range (their ids are staged in shared memory):
// a range holds at most this many times the block size of tokens.
constexpr int kCascadeMaxRangeBlocks = 256;

// Dynamic shared memory the split kernel needs for (head_dim, dtype, groups).
int decode_smem_bytes(int head_dim, int cache_dtype, int n_tiles8);

// Warps in the stream-K kernel's persistent grid on a GPU with `sms` SMs.
int streamk_grid_workers(int head_dim, int cache_dtype, int sms);

}  // namespace pkv
