/*
 * pkv.h — C ABI of the GB300 (sm_103a) paged-KV decode-attention library.
 *
 * Two calls make up one decode step of one attention layer:
 *
 *   pkv_append            write each new token's K/V rows into their cache slots
 *                         (bf16 copy, or FP8 E4M3 quantisation with scales);
 *   pkv_decode_attention  single-token attention of every sequence over its
 *                         paged K/V (GQA, split-KV flash-decoding + LSE combine).
 *
 * pkv_decode_attention_append does both in one launch when each sequence
 * appends one token.
 *
 * Sources for what is computed (web pages, cited by title and section):
 *   [FN] FactNode, "Sub-Millisecond Token Scheduling: Inside Disaggregated
 *        KV-Cache Paging for Frontier LLMs".
 *   [SC] systemcraft.online lesson "LLM inference: prefill, decode, KV cache".
 *   [UI] ultrainstinct.tech, "Architecting Multi-Tier Disaggregated KV-Cache
 *        Hierarchies for Terabyte-Scale LLM Inference".
 *
 * Conventions for every call:
 *   - Pointers named *_cache, q, out, k_new, v_new, slot_mapping, block_tables,
 *     context_lens, k_scale, v_scale and workspace are DEVICE pointers owned by
 *     the caller; the library never frees them and keeps no reference after the
 *     call returns.  Descriptor structs are host memory, read during the call.
 *   - Tensors are dense, row-major (last index fastest), with the shapes given.
 *   - Work is enqueued on `stream` and the call returns without synchronising.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns PKV_ERR_INVALID_ARG (or PKV_ERR_UNSUPPORTED for a
 *     shape the library has no kernel for) and enqueues nothing.  A CUDA
 *     runtime failure returns PKV_ERR_CUDA.  pkv_last_error() gives a message.
 *   - Values that only the device can see (block ids, slots, lengths) are
 *     checked in the kernels: an out-of-range value is skipped (reads as zero,
 *     writes are dropped) and its code is recorded in a per-device error word
 *     read by pkv_get_device_error().  Kernels never trap.
 *   - Thread safety: calls may come from several host threads; the library's
 *     shared state (per-device workspace pool, trace buffer) is locked.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* a pointer, size, dtype or stride is not acceptable */
  PKV_ERR_UNSUPPORTED = 2,  /* valid in principle, no kernel built for it          */
  PKV_ERR_CUDA = 3,         /* the CUDA runtime reported an error                  */
  PKV_ERR_WORKSPACE = 4,    /* caller workspace smaller than required              */
  PKV_ERR_OUT_OF_BLOCKS = 5 /* block manager: free pool exhausted (preempt, retry) */
} pkv_status;

typedef enum {
  PKV_BF16 = 0,  /* bfloat16 (2 bytes)                                   */
  PKV_F32 = 1,   /* IEEE binary32 (4 bytes); append sources only         */
  PKV_E4M3 = 2   /* OCP FP8 E4M3 (1 byte), no infinities, max 448        */
} pkv_dtype;

/*
 * One layer's paged cache.  K and V are separate tensors of identical shape
 *   [num_blocks, num_kv_heads, block_size, head_dim]
 * ([UI] "High-Throughput Paged Attention Kernel Integration": the decode
 * kernel's K_Buffer / V_Buffer arguments).  Token t of a sequence whose block
 * table row is tbl lives at cache[tbl[t / block_size], h, t % block_size, :]
 * ([SC] "PagedAttention & Memory Management (vLLM)").
 *   block_size    16 or 32 tokens ([FN] "Paged KV-Cache with Radix Tree
 *                 Prefix Cache": fixed blocks of typically 16 or 32 tokens)
 *   head_dim      64 or 128
 *   num_kv_heads  >= 1
 *   dtype         PKV_BF16 or PKV_E4M3
 * Both cache pointers must be 16-byte aligned.
 */
typedef struct {
  int64_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t dtype;
} pkv_cache_desc;

/*
 * pkv_append — KV append ([SC] "4. Internal workings", step 5 "Autoregressive
 * Cache Append & Loopback": the new token's K/V vectors are appended to the
 * cache before it attends; FP8 E4M3 with per-head scaling factors: [FN] FAQ
 * "How much HBM memory does FP8 KV-cache quantization save?").
 *
 *   k_new, v_new   [n_tokens, num_kv_heads, head_dim] of src_dtype
 *                  (PKV_BF16 or PKV_F32), 16-byte aligned.
 *   slot_mapping   int64 [n_tokens]: row i goes to flat slot
 *                  s = physical_block * block_size + offset; s < 0 skips the
 *                  row (padding).  s >= num_blocks * block_size is recorded in
 *                  the device error word and skipped.  Two rows with the same
 *                  slot in one call: which one lands is unspecified.
 *   k_cache, v_cache  written in place (only the addressed slots change).
 *   k_scale, v_scale  E4M3 caches only (NULL otherwise): float32, row i and
 *                  KV head h use element [i * scale_row_stride + h];
 *                  scale_row_stride 0 gives one scale per KV head.  The code is
 *                  RNE-satfinite(x / scale) with x / scale an IEEE binary32
 *                  division.  bf16 caches: bf16 sources are copied bit for bit,
 *                  f32 sources are rounded to nearest even.
 *   n_tokens == 0 is a no-op.
 */
pkv_status pkv_append(const void* k_new, const void* v_new, int32_t src_dtype,
                      int64_t n_tokens, const int64_t* slot_mapping,
                      void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                      const float* k_scale, const float* v_scale,
                      int64_t scale_row_stride, pkv_stream_t stream);

/*
 * pkv_slot_mapping — the flat cache slot of each new token, from the block
 * tables: token i of sequence s at logical position pos goes to
 *   block_tables[s, pos / block_size] * block_size + pos % block_size
 * ([SC] "PagedAttention & Memory Management (vLLM)": logical block j of a
 * sequence lives in the physical block its table names; [FN] "Paged KV-Cache
 * with Radix Tree Prefix Cache": fixed-size blocks reached through a
 * per-sequence table).  The result is pkv_append's slot_mapping.
 *
 *   block_tables   int32 [num_seqs, max_blocks_per_seq] (device).
 *   seq_index      int64 [n_tokens] (device): the sequence of token i, or NULL
 *                  when token i belongs to sequence i (one new token per
 *                  sequence; then n_tokens <= num_seqs).
 *   positions      int64 [n_tokens] (device): logical position of token i; a
 *                  negative position is padding and gives slot -1.
 *   cache          the cache the slots address (block size; num_blocks bounds
 *                  the table entries).
 *   slot_mapping   int64 [n_tokens] (device), written.
 * A sequence index outside [0, num_seqs) or a position at or beyond
 * max_blocks_per_seq * block_size records PKV_DEVERR_CONTEXT_LEN; a table
 * entry outside [0, num_blocks) records PKV_DEVERR_BLOCK_ID; either gives
 * slot -1 (which pkv_append skips).  n_tokens == 0 is a no-op.
 */
pkv_status pkv_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                            const int64_t* seq_index, const int64_t* positions, int64_t n_tokens,
                            const pkv_cache_desc* cache, int64_t* slot_mapping, pkv_stream_t stream);

/*
 * pkv_decode_attention — single-token decode attention over a paged cache
 * ([SC] "Why We Need the Key-Value (KV) Cache" and step 4 "Decode Phase";
 * [UI] "High-Throughput Paged Attention Kernel Integration" for the argument
 * list; softmax(q K^T * scale) V as in [UI] "Mathematical Formulation of Block
 * Salience", definition of A).
 *
 *   batch          0..65535 sequences (the split kernel puts the sequence on
 *                  the grid's z axis); more is rejected with PKV_ERR_INVALID_ARG.
 *   q              bf16 [batch, num_q_heads, head_dim], 16-byte aligned.
 *                  num_q_heads = G * num_kv_heads with 1 <= G <= 16; query
 *                  head hq reads KV head hq / G ([SC] "Attention Architectures:
 *                  MHA vs. MQA vs. GQA").
 *   block_tables   int32 [batch, max_blocks_per_seq].  Entries at index
 *                  >= ceil(context_lens[b] / block_size) are never read.
 *   context_lens   int32 [batch]: tokens attended by sequence b, the token
 *                  appended in this step included.  0 gives an all-zero row.
 *                  A length above max_blocks_per_seq * block_size or above
 *                  max_context_len is recorded in the error word and clamped.
 *   max_context_len  host-side upper bound on context_lens (it sizes the
 *                  split-KV grid without reading device memory).
 *   scale          softmax scale (typically 1 / sqrt(head_dim)).
 *   out            float32 [batch, num_q_heads, head_dim], 16-byte aligned.
 *   k_scale, v_scale  E4M3 caches only (NULL otherwise): float32, sequence b
 *                  and KV head h use [b * scale_row_stride + h]; stride 0 gives
 *                  one scale per KV head.
 *
 * The split-KV partial results need scratch memory; this call takes it from a
 * library-owned stream-ordered pool on the current device (released by
 * pkv_shutdown).  pkv_decode_attention_ex takes caller memory instead.
 */
pkv_status pkv_decode_attention(const void* q, int32_t batch, int32_t num_q_heads,
                                const void* k_cache, const void* v_cache,
                                const pkv_cache_desc* cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t max_context_len,
                                float scale, float* out,
                                const float* k_scale, const float* v_scale,
                                int64_t scale_row_stride, pkv_stream_t stream);

/*
 * Split-KV plan (host only, no CUDA call): how a decode call with
 * `split_tokens` divides the work, and the scratch it needs.
 *   mode          1 = fixed splits of `split_tokens` tokens per sequence (the
 *                 default; split_tokens 0 picks the size), one CTA each, which
 *                 the hardware scheduler balances across SMs.  The automatic
 *                 size: one split per (sequence, KV head) when those alone
 *                 give four waves of three CTAs per SM; else the fewest
 *                 splits of max_context_len giving at least three waves with
 *                 a last wave 40-70 % full, when such a count lies below the
 *                 count of a six-wave power-of-two split; else that split.
 *                 0 = balanced ("stream-K"), on request with split_tokens -1
 *                 and batch <= 2048: the (sequence, KV head, 16-token tile)
 *                 space is cut into equal contiguous ranges, one per warp of a
 *                 persistent grid (`workers` warps).
 *   split_tokens  tokens per split (mode 1), 0 in mode 0
 *   max_splits    ceil(max_context_len / split_tokens) (mode 1), 0 in mode 0
 *   workers       warps of the persistent grid (mode 0), 0 in mode 1
 *   workspace_bytes  scratch needed (0 when mode 1 has one split)
 * `num_sms` is the GPU's SM count (152 on GB300); <= 0 means 152.
 */
typedef struct {
  int32_t split_tokens;
  int32_t max_splits;
  int64_t workspace_bytes;
  int32_t mode;
  int32_t workers;
  int32_t prefix_split_tokens;   /* cascade plans only (mode 2) */
  int32_t reserved;
} pkv_decode_plan_t;

pkv_status pkv_decode_plan(int32_t batch, int32_t num_q_heads, const pkv_cache_desc* cache,
                           int32_t max_context_len, int32_t split_tokens, int32_t num_sms,
                           pkv_decode_plan_t* plan);

/*
 * pkv_decode_attention_ex — as pkv_decode_attention, with caller scratch.
 *   workspace        device memory of at least plan.workspace_bytes for the
 *                    same (batch, num_q_heads, cache, max_context_len,
 *                    split_tokens), 256-byte aligned; may be NULL when that is
 *                    0.  Overlapping calls must not share a workspace.
 *   split_tokens     0 = automatic, -1 = balanced ranges, else tokens per
 *                    split (a multiple of 64); see pkv_decode_plan.
 */
pkv_status pkv_decode_attention_ex(const void* q, int32_t batch, int32_t num_q_heads,
                                   const void* k_cache, const void* v_cache,
                                   const pkv_cache_desc* cache,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t max_context_len,
                                   float scale, float* out,
                                   const float* k_scale, const float* v_scale,
                                   int64_t scale_row_stride,
                                   void* workspace, size_t workspace_bytes,
                                   int32_t split_tokens, pkv_stream_t stream);

/*
 * pkv_decode_attention_append — one decode step: append each sequence's new
 * token and attend, in one launch ([SC] "LLM inference: prefill, decode, KV
 * cache", section 4, step 5: the new token's K/V join the cache, then the
 * token attends the whole cache).  The result equals pkv_append of the new
 * rows into the slots of positions context_lens[b] - 1 followed by
 * pkv_decode_attention_ex, bit for bit in the cache and in `out`.
 *
 *   k_cache, v_cache  written: the new rows go into their slots.
 *   k_new, v_new   [batch, num_kv_heads, head_dim] of type new_dtype
 *                  (PKV_BF16 or PKV_F32), 16-byte aligned: the new token of
 *                  sequence b, encoded as pkv_append encodes a row (bf16:
 *                  bf16 copied, f32 rounded to nearest even; E4M3:
 *                  RNE-satfinite(x / scale) with the scales below).
 *   context_lens   as for decode: the new token included; the row of
 *                  sequence b goes to position context_lens[b] - 1 through
 *                  its block table.  A sequence with context_lens[b] == 0
 *                  appends nothing (its output row is zeros); a length that
 *                  is clamped (see pkv_decode_attention) appends nothing and
 *                  is recorded.  A table entry outside [0, num_blocks) at the
 *                  new position records PKV_DEVERR_BLOCK_ID and writes
 *                  nothing.
 *   k_scale, v_scale  E4M3: row b, KV head h use [b * scale_row_stride + h]
 *                  for both the append and the attention.
 *   split_tokens   0 (automatic) or a multiple of 64; the balanced mode (-1)
 *                  is PKV_ERR_INVALID_ARG here.
 * Other arguments and the workspace as pkv_decode_attention_ex.  The new
 * token's slot is written by the warp whose tile holds it, before that warp
 * loads the tile; nothing else reads it during the call.
 */
pkv_status pkv_decode_attention_append(const void* q, int32_t batch, int32_t num_q_heads,
                                       void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                       const void* k_new, const void* v_new, int32_t new_dtype,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t max_context_len,
                                       float scale, float* out,
                                       const float* k_scale, const float* v_scale,
                                       int64_t scale_row_stride,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t split_tokens, pkv_stream_t stream);

/*
 * pkv_decode_attention_noalloc — pkv_decode_attention without any allocation.
 * The source pages have no counterpart to this call; it exists for callers
 * that must not allocate device memory when they run attention (a serving
 * loop that reserved all memory at start-up, a runtime whose memory belongs
 * to another allocator, code that must not wait on an allocator's locks).
 *
 * Same arguments, layouts and checks as pkv_decode_attention.  The split-KV
 * partials go to a fixed 32 MiB array of device memory owned by the library
 * (every GPU that loads the library holds it until the process exits).  A call
 * whose plan needs more scratch than that (see pkv_decode_plan with
 * split_tokens 0) returns PKV_ERR_WORKSPACE without launching anything.  The
 * call makes no cudaMalloc, cudaFree or other allocating call.  (With the
 * kernel timing trace switched on by pkv_trace_enable, which is off by
 * default, every library launch also records two CUDA events taken from a
 * host-side event pool; no device memory is allocated for them either.)
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls on a device share the one array and it keeps the last
 * call's contents (nothing in it needs to start at zero): calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race on
 * it and give wrong results.  Serialise them, or use pkv_decode_attention_ex.
 * A caller that resets the device (cudaDeviceReset) calls pkv_shutdown first;
 * the next call then looks the array's address up again.
 */
pkv_status pkv_decode_attention_noalloc(const void* q, int32_t batch, int32_t num_q_heads,
                                        const void* k_cache, const void* v_cache,
                                        const pkv_cache_desc* cache,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t max_context_len,
                                        float scale, float* out,
                                        const float* k_scale, const float* v_scale,
                                        int64_t scale_row_stride, pkv_stream_t stream);

/*
 * Cascade (shared-prefix) decode — decode attention for a batch whose
 * sequences all begin with the same `prefix_len` tokens held in the same
 * physical blocks (shared by reference: [FN] "Paged KV-Cache with Radix Tree
 * Prefix Cache", copy-on-write prefix blocks; [SC] "7. Practical
 * applications", prompt caching of identical prefixes).  The result equals
 * pkv_decode_attention's; the prefix is attended once for all B x G query rows
 * of each KV head (a dense Q.K^T / P.V product on the tensor cores) instead
 * of once per sequence, and merged with each private suffix by the same
 * log-sum-exp combine.
 *
 *   batch          0..65535 sequences (0: nothing to do; pkv_cascade_plan
 *                  takes 1..65535); more is rejected with PKV_ERR_INVALID_ARG.
 *   prefix_blocks  int32 [prefix_len / block_size]: the prefix's physical
 *                  blocks.  For every sequence b the first prefix_len /
 *                  block_size entries of block_tables[b] must equal them
 *                  (they are not read), and context_lens[b] >= prefix_len.
 *   prefix_len     > 0, a multiple of block_size, <= max_context_len.
 *   Other arguments as pkv_decode_attention_ex; bf16 caches only (E4M3:
 *   PKV_ERR_UNSUPPORTED).  Scratch: at least plan.workspace_bytes from
 *   pkv_cascade_plan, 256-byte aligned.
 *
 * The prefix product runs on `stream`; the suffix decode runs beside it on a
 * stream the library owns (one per device, made on first use, destroyed by
 * pkv_shutdown), forked from `stream` and joined back to it by events before
 * the combine; the call stays asynchronous and ordered on `stream` (also
 * under stream capture).
 *
 * pkv_cascade_plan (host only): mode 2; split_tokens / max_splits describe the
 * suffix splits, workers the number of prefix ranges and prefix_split_tokens
 * their length.  The ranges are chosen to balance the prefix CTAs (one per
 * SM) against the suffix decode beside them; the suffix splits are then sized
 * for the SMs the prefix leaves free (about two waves of three CTAs per SM),
 * so they are longer than a plain decode of the same batch would take.  The
 * call plans again with the device's SM count and refuses a smaller
 * workspace (PKV_ERR_WORKSPACE): plan with that count (num_sms), or 0 for 152.
 */
pkv_status pkv_cascade_plan(int32_t batch, int32_t num_q_heads, const pkv_cache_desc* cache,
                            int32_t prefix_len, int32_t max_context_len, int32_t num_sms,
                            pkv_decode_plan_t* plan);

pkv_status pkv_cascade_decode_attention(const void* q, int32_t batch, int32_t num_q_heads,
                                        const void* k_cache, const void* v_cache,
                                        const pkv_cache_desc* cache,
                                        const int32_t* prefix_blocks, int32_t prefix_len,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t max_context_len,
                                        float scale, float* out,
                                        void* workspace, size_t workspace_bytes,
                                        pkv_stream_t stream);

/*
 * Multi-token query attention — q_len new tokens per sequence attend the
 * sequence's paged K/V causally: the chunk of a chunked prefill that runs
 * next to decode steps ([SC] "9. Failure modes and limitations", item 3,
 * Chunked Prefill) or the tokens a draft model proposed, verified in one
 * parallel pass ([SC] "7. Practical applications", item 3, Speculative
 * Decoding).
 *
 *   batch          0..65535 sequences; more is rejected with
 *                  PKV_ERR_INVALID_ARG.
 *   q              bf16 [batch, q_len, num_q_heads, head_dim], 16-byte aligned;
 *                  1 <= q_len <= 16.
 *   context_lens   int32 [batch]: tokens of sequence b, its q_len new tokens
 *                  included (they must already be appended).  Query i sits at
 *                  position context_lens[b] - q_len + i and attends tokens
 *                  0 .. that position; a query before position 0 (a context
 *                  shorter than q_len) gives zeros.
 *   out            float32 [batch, q_len, num_q_heads, head_dim].
 *   split_tokens   0 = automatic, else tokens per split: a multiple of 64, at
 *                  most 1024 * block_size.
 *   workspace      device scratch of at least plan.workspace_bytes from
 *                  pkv_multi_query_plan with the same arguments (256-byte
 *                  aligned; may be NULL when that is 0).
 *   Other arguments as pkv_decode_attention; bf16 caches only (E4M3:
 *   PKV_ERR_UNSUPPORTED).  q_len = 1 computes decode attention.
 *
 * Up to 16 query rows (q_len * G) per (sequence, KV head) run on an mma.sync
 * kernel whose warps split the tokens; more run on a persistent tcgen05
 * kernel (one CTA per SM taking (split, sequence, KV head, 128-row block)
 * units longest first; operands staged by TMA, accumulators in tensor
 * memory), which keeps a work-unit counter and the unit order in the last
 * part of the workspace (so a workspace is always needed there).
 *
 * pkv_multi_query_plan (host only): mode 3; split_tokens / max_splits as for
 * decode; workers = warps per CTA that share each 16 query rows (4)
 * on the mma.sync kernel, 0 when the tcgen05 kernel runs.
 */
pkv_status pkv_multi_query_plan(int32_t batch, int32_t q_len, int32_t num_q_heads,
                                const pkv_cache_desc* cache, int32_t max_context_len,
                                int32_t split_tokens, int32_t num_sms, pkv_decode_plan_t* plan);

pkv_status pkv_multi_query_attention(const void* q, int32_t batch, int32_t q_len,
                                     int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                     const pkv_cache_desc* cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t max_context_len,
                                     float scale, float* out,
                                     void* workspace, size_t workspace_bytes,
                                     int32_t split_tokens, pkv_stream_t stream);

/* Device error codes (first one recorded wins). */
enum {
  PKV_DEVERR_NONE = 0,
  PKV_DEVERR_WAIT_TIMEOUT = 1,    /* a pipeline wait gave up (bounded spin)     */
  PKV_DEVERR_BLOCK_ID = 2,        /* block table entry outside [0, num_blocks)  */
  PKV_DEVERR_CONTEXT_LEN = 3,     /* context length beyond the table or bound   */
  PKV_DEVERR_SLOT = 4             /* append slot beyond the cache               */
};

/*
 * Reads and clears the current device's error word.  Synchronises `stream`
 * first (the only call that waits for the GPU).  Returns the code, or -1 if
 * the read itself failed.
 */
int32_t pkv_get_device_error(pkv_stream_t stream);

/*
 * Self-test of the device-side failure detection: launches one CTA that
 * waits on a barrier nothing ever arrives on, with a limit of `limit_us`
 * microseconds (1..1000000) instead of the kernels' one second.
 *   which 0: a plain bounded mbarrier wait;
 *   which 1: the abort path of the tensor-core attention kernels (tensor
 *            memory held, one wait times out and raises the CTA's abort flag,
 *            the other waits leave on it, tensor memory is freed).
 * The kernel returns normally; afterwards pkv_get_device_error reads
 * PKV_DEVERR_WAIT_TIMEOUT and the context stays usable.
 */
pkv_status pkv_selftest_wait_timeout(int32_t which, int32_t limit_us, pkv_stream_t stream);

/* Human-readable name of a status. */
const char* pkv_status_string(int32_t status);

/* Message describing the last non-OK status returned on this host thread. */
const char* pkv_last_error(void);

/* ABI version of this library (major * 100 + minor). */
int32_t pkv_abi_version(void);

/*
 * Kernel timing trace.  While enabled, every kernel the library launches is
 * bracketed by CUDA events recorded on the stream it runs on.
 * pkv_trace_read synchronises those events and returns, per kernel kind,
 * the number of launches and their summed device time; it then clears the
 * buffer.  Kinds: 0 append, 1 decode split, 2 combine, 3 cascade prefix,
 * 4 block copy, 5 multi-token query, 6 slot mapping.
 */
typedef struct {
  int32_t kind;
  int32_t launches;
  double total_ms;
} pkv_trace_entry;

pkv_status pkv_trace_enable(int32_t on);
int32_t pkv_trace_read(pkv_trace_entry* entries, int32_t capacity);

/*
 * Frees library-owned device memory and objects (workspace pools, the side
 * streams of the cascade call, trace events) and forgets every per-device
 * address and launch limit looked up so far, so that the next call sets them
 * up again.  Call it before a cudaDeviceReset if the library is used after
 * the reset.  No call of the library may run concurrently with it.
 */
pkv_status pkv_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
