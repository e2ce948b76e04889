// C ABI of the paged-KV library: argument checks, split-KV planning, TMA
// descriptors, scratch memory, launches, the device error word and the kernel
// timing trace.  Every check that can be made on the host is made before any
// CUDA runtime call, so a rejected call touches no GPU state.

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "pkv.h"
#include "pkv_blocks.h"
#include "pkv_internal.h"

namespace {

using pkv::AppendParams;
using pkv::DecodeParams;

constexpr int kMaxDevices = 64;
constexpr int kDefaultSms = 152;
// Thread blocks of a block copy that crosses the host link (it reaches the
// link's bandwidth with about 32 on GB300).
constexpr int kHostLinkCopyCtas = 64;

thread_local std::string t_last_error;

}  // namespace

void pkv::set_last_error(const char* msg) { t_last_error = msg; }

namespace {
std::atomic<int> g_config_epoch{1};
}  // namespace

int pkv::config_epoch() { return g_config_epoch.load(std::memory_order_relaxed); }

namespace {

pkv_status fail(pkv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ device state

__device__ int g_device_error;  // one word per device: first bad value seen

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int* err = nullptr;
  cudaMemPool_t pool = nullptr;
  // a stream of the library's own with a fork and a join event: the
  // cascade's suffix decode runs there beside the prefix
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
// Device address of the no-allocation entry point's scratch array, looked up
// once per device (under g_mu); cleared by pkv_shutdown.
void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_fork_mu;  // one fork / join on the side streams at a time

// The device's side stream and events, made on first use.
pkv_status side_stream(DeviceState* st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (st->side != nullptr) return PKV_OK;
  cudaError_t e = cudaStreamCreateWithFlags(&st->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st->fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st->join, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e, "side stream");
  return PKV_OK;
}

pkv_status current_device(int* dev, DeviceState** st) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device index %d", *dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[*dev];
  if (!s.ready) {
    e = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, *dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err), g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    s.ready = true;
  }
  *st = &s;
  return PKV_OK;
}

// ------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D view (d, token-in-block, kv-head, block) of one cache tensor; a box is
// `box_tokens` token rows (16 by default: one decode tile) of up to 128 bytes,
// 128B- or 64B-swizzled.
pkv_status make_cache_tmap(CUtensorMap* tm, const void* base, const pkv_cache_desc& c,
                           int box_tokens = pkv::kTileTokens) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const uint64_t esz = c.dtype == PKV_E4M3 ? 1 : 2;
  const uint64_t row = static_cast<uint64_t>(c.head_dim) * esz;
  const uint64_t boxb = row < 128 ? row : 128;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(c.head_dim), static_cast<cuuint64_t>(c.block_size),
                        static_cast<cuuint64_t>(c.num_kv_heads),
                        static_cast<cuuint64_t>(c.num_blocks)};
  cuuint64_t strides[3] = {row, row * c.block_size, row * c.block_size * c.num_kv_heads};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(boxb / esz), static_cast<cuuint32_t>(box_tokens), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(tm, c.dtype == PKV_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  boxb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return PKV_OK;
}

// ------------------------------------------------------------ trace

struct TraceRec {
  int kind;
  int dev;
  cudaEvent_t a, b;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<std::pair<int, cudaEvent_t>> g_event_pool;

cudaEvent_t take_event(int dev) {
  for (size_t i = 0; i < g_event_pool.size(); ++i) {
    if (g_event_pool[i].first == dev) {
      cudaEvent_t e = g_event_pool[i].second;
      g_event_pool.erase(g_event_pool.begin() + i);
      return e;
    }
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

template <class F>
cudaError_t traced(int kind, cudaStream_t stream, F&& launch) {
  bool on;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    on = g_trace_on;
  }
  if (!on) return launch();
  int dev = 0;
  cudaGetDevice(&dev);
  cudaEvent_t a, b;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    a = take_event(dev);
    b = take_event(dev);
  }
  if (a == nullptr || b == nullptr) return launch();
  cudaEventRecord(a, stream);
  cudaError_t e = launch();
  cudaEventRecord(b, stream);
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace.push_back({kind, dev, a, b});
  return e;
}

// ------------------------------------------------------------ checks

pkv_status check_cache(const pkv_cache_desc* c) {
  if (c == nullptr) return fail(PKV_ERR_INVALID_ARG, "cache descriptor is NULL");
  if (c->dtype != PKV_BF16 && c->dtype != PKV_E4M3)
    return fail(PKV_ERR_INVALID_ARG, "cache dtype %d (want PKV_BF16 or PKV_E4M3)", c->dtype);
  if (c->block_size != 16 && c->block_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (16 or 32)", c->block_size);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (64 or 128)", c->head_dim);
  if (c->num_kv_heads < 1 || c->num_kv_heads > 65535)
    return fail(PKV_ERR_INVALID_ARG, "num_kv_heads %d", c->num_kv_heads);
  if (c->num_blocks < 1 || c->num_blocks > 0x7FFFFFFFll)
    return fail(PKV_ERR_INVALID_ARG, "num_blocks %lld", static_cast<long long>(c->num_blocks));
  return PKV_OK;
}

int32_t auto_split_tokens(int32_t batch, int32_t num_kv_heads, int32_t max_ctx, int32_t sms, int32_t waves = 6) {
  // Largest power-of-two chunk (256..4096 tokens) that still gives about
  // `waves` waves of three CTAs per SM when every sequence is as long as the
  // bound.
  const int64_t units = static_cast<int64_t>(batch) * num_kv_heads;
  const int64_t want = static_cast<int64_t>(sms) * 3 * waves;
  int32_t st = 4096;
  while (st > 256 && units * ceil_div(max_ctx, st) < want) st /= 2;
  return st;
}

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

// Tokens per split of a plain decode call.  One split per (sequence, KV head)
// when those alone give four waves of three CTAs per SM: every CTA then writes
// its output rows directly and no combine runs (the FP8 workload, 2048 units:
// the split kernel takes 248 us either way and the step goes from 259.6 to
// 252.8 us).  Otherwise the six-wave power-of-two rule of auto_split_tokens,
// with a last split shorter than an eighth of the others folded into them
// (8193 tokens: eight splits of 1088 rather than eight of 1024 and one of 1).
// Split length for grids of three CTAs per SM, given the six-wave rule's
// `st` (which cuts the longest context `max_ctx` into n pieces): when n is
// above `min_splits`, the fewest splits that give at least three waves with
// a last wave 40-70 % full.  The SMs of a GB300 do not all stream at the same
// rate, so a grid's tail is set by how full its last wave is: on 8 sequences
// of 131k tokens the decode kernel ran at 7.15 TB/s with the six-wave rule's
// 63 splits (8.8 waves), in troughs of 7.01-7.09 wherever the last wave was
// nearly full (28, 35, 42 splits) and at 7.25-7.32 where it was about half
// full (25, 32, 38 splits); the multi-token mma.sync kernel (q_len 2) showed
// the same period.  The shared-prefix batch (128 sequences of 4.2-5.1k
// tokens) took 2 splits instead of 3 (+2.6 %); the GQA batch 4 instead of 8
// (no change).
int32_t half_wave_split(int64_t units, int32_t max_ctx, int32_t sms, int32_t st, int64_t min_splits) {
  const int64_t n = ceil_div(max_ctx, st);
  if (n <= min_splits) return st;
  const int64_t slots = static_cast<int64_t>(3) * sms;
  for (int64_t s = 2; s < n; ++s) {
    const int64_t waves100 = units * s * 100 / slots;  // waves of the grid x 100
    const int64_t frac = waves100 % 100;
    if (waves100 >= 300 && frac >= 40 && frac <= 70) return static_cast<int32_t>(ceil_div(ceil_div(max_ctx, s), 64) * 64);
  }
  return st;
}

int32_t decode_split_tokens(int32_t batch, int32_t num_kv_heads, int32_t max_ctx, int32_t sms) {
  const int64_t units = static_cast<int64_t>(batch) * num_kv_heads;
  if (units >= static_cast<int64_t>(4) * 3 * sms)
    return static_cast<int32_t>(max_ctx > 64 ? ceil_div(max_ctx, 64) * 64 : 64);
  int32_t st = auto_split_tokens(batch, num_kv_heads, max_ctx, sms);
  const int64_t n = ceil_div(max_ctx, st);
  if (n >= 2 && max_ctx - (n - 1) * st < st / 8)
    st = static_cast<int32_t>(ceil_div(ceil_div(max_ctx, n - 1), 64) * 64);
  return half_wave_split(static_cast<int64_t>(batch) * num_kv_heads, max_ctx, sms, st, 1);
}

pkv_status plan(int32_t batch, int32_t num_q_heads, const pkv_cache_desc* c, int32_t max_ctx,
                int32_t split_tokens, int32_t sms, pkv_decode_plan_t* out) {
  pkv_status s = check_cache(c);
  if (s != PKV_OK) return s;
  if (batch < 0 || batch > 65535) return fail(PKV_ERR_INVALID_ARG, "batch %d", batch);
  if (num_q_heads < 1 || num_q_heads % c->num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d",
                num_q_heads, c->num_kv_heads);
  if (num_q_heads / c->num_kv_heads > 16)
    return fail(PKV_ERR_UNSUPPORTED, "group size %d > 16", num_q_heads / c->num_kv_heads);
  if (max_ctx < 0) return fail(PKV_ERR_INVALID_ARG, "max_context_len %d", max_ctx);
  if (split_tokens < -1 || (split_tokens > 0 && split_tokens % 64 != 0))
    return fail(PKV_ERR_INVALID_ARG, "split_tokens %d (-1, 0 or a multiple of 64)", split_tokens);
  if (sms <= 0) sms = kDefaultSms;
  const int64_t gp = num_q_heads / c->num_kv_heads > 8 ? 16 : 8;
  const int64_t tiles_bound =
      static_cast<int64_t>(batch) * c->num_kv_heads * ceil_div(max_ctx, pkv::kTileTokens);
  *out = pkv_decode_plan_t{};
  // Fixed splits by default: many CTAs that the hardware scheduler balances
  // across SMs (whose share of HBM bandwidth differs); balanced static ranges
  // on request.
  const bool want_balanced = split_tokens == -1;
  if (want_balanced && batch <= pkv::kMaxStreamKBatch && tiles_bound < 0x7FFFFFFFll) {
    const int64_t w = pkv::streamk_grid_workers(c->head_dim, c->dtype, sms);
    out->mode = pkv::kModeStreamK;
    out->workers = static_cast<int32_t>(w);
    out->workspace_bytes = align256(2 * w * gp * c->head_dim * 4) + align256(2 * w * gp * 2 * 4) +
                           align256((static_cast<int64_t>(batch) + 1) * 4);
    return PKV_OK;
  }
  const int32_t st =
      split_tokens > 0 ? split_tokens : decode_split_tokens(batch, c->num_kv_heads, max_ctx, sms);
  const int64_t splits = max_ctx > 0 ? ceil_div(max_ctx, st) : 1;
  if (splits > 0x7FFFFFFFll) return fail(PKV_ERR_INVALID_ARG, "too many splits");
  out->mode = pkv::kModeFixedSplit;
  out->split_tokens = st;
  out->max_splits = static_cast<int32_t>(splits);
  if (splits > 1) {
    const int64_t rows = static_cast<int64_t>(batch) * num_q_heads * splits;
    out->workspace_bytes = align256(rows * c->head_dim * 4) + rows * 2 * 4;
  }
  return PKV_OK;
}

struct DecodeArgs {
  const void* q;
  int32_t batch, num_q_heads;
  const void* k_cache;
  const void* v_cache;
  const pkv_cache_desc* cache;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* context_lens;
  int32_t max_ctx;
  float scale;
  float* out;
  const float* k_scale;
  const float* v_scale;
  int64_t scale_stride;
  // fused append (pkv_decode_attention_append): one new token per sequence
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  int32_t new_dtype = -1;
};

pkv_status check_decode(const DecodeArgs& a) {
  pkv_status s = check_cache(a.cache);
  if (s != PKV_OK) return s;
  const pkv_cache_desc& c = *a.cache;
  if (a.batch < 0 || a.batch > 65535) return fail(PKV_ERR_INVALID_ARG, "batch %d", a.batch);
  if (a.num_q_heads < 1 || a.num_q_heads % c.num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d",
                a.num_q_heads, c.num_kv_heads);
  if (a.num_q_heads / c.num_kv_heads > 16)
    return fail(PKV_ERR_UNSUPPORTED, "group size %d > 16", a.num_q_heads / c.num_kv_heads);
  if (!std::isfinite(a.scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (a.max_blocks < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d", a.max_blocks);
  if (a.max_ctx < 0 || static_cast<int64_t>(a.max_ctx) > static_cast<int64_t>(a.max_blocks) * c.block_size)
    return fail(PKV_ERR_INVALID_ARG, "max_context_len %d outside [0, max_blocks_per_seq * block_size]",
                a.max_ctx);
  const bool fp8 = c.dtype == PKV_E4M3;
  if (fp8 && (a.k_scale == nullptr || a.v_scale == nullptr))
    return fail(PKV_ERR_INVALID_ARG, "E4M3 cache needs k_scale and v_scale");
  if (!fp8 && (a.k_scale != nullptr || a.v_scale != nullptr))
    return fail(PKV_ERR_INVALID_ARG, "scales given for a bf16 cache");
  if (a.scale_stride < 0) return fail(PKV_ERR_INVALID_ARG, "scale_row_stride < 0");
  if (a.batch == 0) return PKV_OK;
  if (a.q == nullptr || a.k_cache == nullptr || a.v_cache == nullptr || a.out == nullptr ||
      a.block_tables == nullptr || a.context_lens == nullptr)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned(a.q, 16) || !aligned(a.k_cache, 16) || !aligned(a.v_cache, 16) || !aligned(a.out, 16))
    return fail(PKV_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned");
  if (!aligned(a.block_tables, 4) || !aligned(a.context_lens, 4))
    return fail(PKV_ERR_INVALID_ARG, "block_tables / context_lens must be 4-byte aligned");
  if (fp8 && (!aligned(a.k_scale, 4) || !aligned(a.v_scale, 4)))
    return fail(PKV_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  if (a.new_dtype != -1) {
    if (a.new_dtype != PKV_BF16 && a.new_dtype != PKV_F32)
      return fail(PKV_ERR_INVALID_ARG, "new_dtype %d (want PKV_BF16 or PKV_F32)", a.new_dtype);
    if (a.k_new == nullptr || a.v_new == nullptr) return fail(PKV_ERR_INVALID_ARG, "NULL k_new / v_new");
    if (!aligned(a.k_new, 16) || !aligned(a.v_new, 16))
      return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  }
  return PKV_OK;
}

pkv_status run_decode(const DecodeArgs& a, void* ws, size_t ws_bytes, int32_t split_tokens,
                      cudaStream_t stream, bool own_workspace) {
  int dev;
  DeviceState* st;
  pkv_status s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  pkv_decode_plan_t pl;
  s = plan(a.batch, a.num_q_heads, a.cache, a.max_ctx, split_tokens, st->sms, &pl);
  if (s != PKV_OK) return s;
  if (a.new_dtype != -1 && pl.mode != pkv::kModeFixedSplit)
    return fail(PKV_ERR_UNSUPPORTED, "the fused append takes fixed splits (split_tokens >= 0)");
  if (!own_workspace && pl.workspace_bytes > 0) {
    if (ws == nullptr || ws_bytes < static_cast<size_t>(pl.workspace_bytes))
      return fail(PKV_ERR_WORKSPACE, "workspace %zu bytes, need %lld", ws_bytes,
                  static_cast<long long>(pl.workspace_bytes));
    if (!aligned(ws, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  const pkv_cache_desc& c = *a.cache;
  CUtensorMap tk, tv;
  s = make_cache_tmap(&tk, a.k_cache, c);
  if (s != PKV_OK) return s;
  s = make_cache_tmap(&tv, a.v_cache, c);
  if (s != PKV_OK) return s;

  cudaError_t e;
  if (own_workspace && pl.workspace_bytes > 0) {
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if (st->pool == nullptr) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        e = cudaMemPoolCreate(&st->pool, &props);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
        uint64_t keep = ~0ull;
        cudaMemPoolSetAttribute(st->pool, cudaMemPoolAttrReleaseThreshold, &keep);
      }
    }
    e = cudaMallocFromPoolAsync(&ws, static_cast<size_t>(pl.workspace_bytes), st->pool, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync(workspace)");
  }

  DecodeParams p = {};
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = a.out;
  if (pl.mode == pkv::kModeStreamK) {
    const int64_t gp = a.num_q_heads / c.num_kv_heads > 8 ? 16 : 8;
    const int64_t o_bytes = align256(2 * static_cast<int64_t>(pl.workers) * gp * c.head_dim * 4);
    const int64_t ml_bytes = align256(2 * static_cast<int64_t>(pl.workers) * gp * 2 * 4);
    p.ws_o = static_cast<float*>(ws);
    p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + o_bytes);
    p.ws_q = reinterpret_cast<int*>(static_cast<char*>(ws) + o_bytes + ml_bytes);
  } else if (pl.workspace_bytes > 0) {
    const int64_t rows = static_cast<int64_t>(a.batch) * a.num_q_heads * pl.max_splits;
    p.ws_o = static_cast<float*>(ws);
    p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(rows * c.head_dim * 4));
  }
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.scale_stride = a.scale_stride;
  p.num_blocks = c.num_blocks;
  p.batch = a.batch;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.group = a.num_q_heads / c.num_kv_heads;
  p.head_dim = c.head_dim;
  p.block_size = c.block_size;
  p.max_blocks = a.max_blocks;
  p.max_ctx = a.max_ctx;
  p.split_tokens = pl.split_tokens;
  p.max_splits = pl.max_splits;
  p.qk_log2_scale = a.scale * 1.4426950408889634f;
  p.cache_dtype = c.dtype;
  p.mode = pl.mode;
  p.workers = pl.workers;
  p.extra_slot = -1;
  p.slots_per_row = pl.max_splits;
  if (a.new_dtype != -1) {
    p.new_src = (a.new_dtype == PKV_BF16 ? pkv::kEncBF16 : pkv::kEncF32) + 1;
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.k_cache = const_cast<void*>(a.k_cache);
    p.v_cache = const_cast<void*>(a.v_cache);
  }
  p.err = st->err;

  e = traced(pkv::kKindDecodeSplit, stream,
             [&] { return pkv::launch_decode_split(p, tk, tv, stream); });
  if (e == cudaSuccess && (pl.mode == pkv::kModeStreamK || pl.max_splits > 1))
    e = traced(pkv::kKindCombine, stream, [&] { return pkv::launch_decode_combine(p, stream); });
  if (own_workspace && pl.workspace_bytes > 0) {
    cudaError_t e2 = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = e2;
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_append(const void* k_new, const void* v_new, int32_t src_dtype, int64_t n_tokens,
                      const int64_t* slot_mapping, void* k_cache, void* v_cache,
                      const pkv_cache_desc* cache, const float* k_scale, const float* v_scale,
                      int64_t scale_row_stride, pkv_stream_t stream) {
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  if (src_dtype != PKV_BF16 && src_dtype != PKV_F32)
    return fail(PKV_ERR_INVALID_ARG, "source dtype %d (PKV_BF16 or PKV_F32)", src_dtype);
  if (n_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "n_tokens %lld", static_cast<long long>(n_tokens));
  const bool fp8 = cache->dtype == PKV_E4M3;
  if (fp8 && (k_scale == nullptr || v_scale == nullptr))
    return fail(PKV_ERR_INVALID_ARG, "E4M3 cache needs k_scale and v_scale");
  if (!fp8 && (k_scale != nullptr || v_scale != nullptr))
    return fail(PKV_ERR_INVALID_ARG, "scales given for a bf16 cache");
  if (scale_row_stride < 0) return fail(PKV_ERR_INVALID_ARG, "scale_row_stride < 0");
  if (n_tokens == 0) return PKV_OK;
  if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr || k_cache == nullptr ||
      v_cache == nullptr)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PKV_ERR_INVALID_ARG, "k_new, v_new and caches must be 16-byte aligned");
  if (!aligned(slot_mapping, 8)) return fail(PKV_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
  if (fp8 && (!aligned(k_scale, 4) || !aligned(v_scale, 4)))
    return fail(PKV_ERR_INVALID_ARG, "scales must be 4-byte aligned");

  int dev;
  DeviceState* st;
  s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  AppendParams p = {};
  p.k_new = k_new;
  p.v_new = v_new;
  p.slots = slot_mapping;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.scale_stride = scale_row_stride;
  p.n_tokens = n_tokens;
  p.num_slots = cache->num_blocks * cache->block_size;
  p.block_size = cache->block_size;
  p.num_kv_heads = cache->num_kv_heads;
  p.head_dim = cache->head_dim;
  p.src_dtype = src_dtype;
  p.cache_dtype = cache->dtype;
  p.err = st->err;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = traced(pkv::kKindAppend, cs, [&] { return pkv::launch_append(p, cs); });
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return PKV_OK;
}

pkv_status pkv_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                            const int64_t* seq_index, const int64_t* positions, int64_t n_tokens,
                            const pkv_cache_desc* cache, int64_t* slot_mapping, pkv_stream_t stream) {
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  if (n_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "n_tokens %lld", static_cast<long long>(n_tokens));
  if (num_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "num_seqs %d", num_seqs);
  if (max_blocks_per_seq < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d", max_blocks_per_seq);
  if (n_tokens == 0) return PKV_OK;
  if (positions == nullptr || slot_mapping == nullptr || (num_seqs > 0 && block_tables == nullptr))
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (seq_index == nullptr && n_tokens > num_seqs)
    return fail(PKV_ERR_INVALID_ARG, "without seq_index token i is sequence i: n_tokens %lld > num_seqs %d",
                static_cast<long long>(n_tokens), num_seqs);
  if (!aligned(positions, 8) || !aligned(slot_mapping, 8) || (seq_index != nullptr && !aligned(seq_index, 8)) ||
      !aligned(block_tables, 4))
    return fail(PKV_ERR_INVALID_ARG, "positions, seq_index, slot_mapping must be 8-byte aligned, tables 4");
  int dev;
  DeviceState* st;
  s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  pkv::SlotParams p = {};
  p.block_tables = block_tables;
  p.seq_index = seq_index;
  p.positions = positions;
  p.slots = slot_mapping;
  p.n = n_tokens;
  p.num_blocks = cache->num_blocks;
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = cache->block_size;
  p.err = st->err;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = traced(pkv::kKindSlotMapping, cs, [&] { return pkv::launch_slot_mapping(p, cs); });
  if (e != cudaSuccess) return cuda_fail(e, "slot mapping launch");
  return PKV_OK;
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                           const int32_t* src_blocks, const int32_t* dst_blocks, int32_t n_pairs,
                           pkv_stream_t stream) {
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  if (n_pairs < 0) return fail(PKV_ERR_INVALID_ARG, "n_pairs %d", n_pairs);
  if (n_pairs == 0) return PKV_OK;
  if (k_cache == nullptr || v_cache == nullptr || src_blocks == nullptr || dst_blocks == nullptr)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PKV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  if (!aligned(src_blocks, 4) || !aligned(dst_blocks, 4))
    return fail(PKV_ERR_INVALID_ARG, "block id arrays must be 4-byte aligned");
  int dev;
  DeviceState* st;
  s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  const int64_t esz = cache->dtype == PKV_E4M3 ? 1 : 2;
  pkv::CopyParams p = {};
  p.k_src = k_cache;
  p.v_src = v_cache;
  p.k_dst = k_cache;
  p.v_dst = v_cache;
  p.src = src_blocks;
  p.dst = dst_blocks;
  p.n_pairs = n_pairs;
  p.block_vec = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size * cache->head_dim * esz / 16;
  p.src_blocks = cache->num_blocks;
  p.dst_blocks = cache->num_blocks;
  p.err = st->err;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = traced(pkv::kKindBlockCopy, cs, [&] { return pkv::launch_copy_blocks(p, cs); });
  if (e != cudaSuccess) return cuda_fail(e, "block copy launch");
  return PKV_OK;
}

pkv_status pkv_copy_blocks_between(const void* src_k, const void* src_v, int64_t src_num_blocks,
                                   void* dst_k, void* dst_v, int64_t dst_num_blocks,
                                   const pkv_cache_desc* cache, const int32_t* src_blocks,
                                   const int32_t* dst_blocks, int32_t n_pairs, int32_t max_ctas,
                                   pkv_stream_t stream) {
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  if (n_pairs < 0) return fail(PKV_ERR_INVALID_ARG, "n_pairs %d", n_pairs);
  if (max_ctas < 0) return fail(PKV_ERR_INVALID_ARG, "max_ctas %d", max_ctas);
  if (src_num_blocks < 1 || dst_num_blocks < 1)
    return fail(PKV_ERR_INVALID_ARG, "pool sizes %lld, %lld", static_cast<long long>(src_num_blocks),
                static_cast<long long>(dst_num_blocks));
  if (n_pairs == 0) return PKV_OK;
  if (src_k == nullptr || src_v == nullptr || dst_k == nullptr || dst_v == nullptr || src_blocks == nullptr ||
      dst_blocks == nullptr)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(src_k, 16) || !aligned(src_v, 16) || !aligned(dst_k, 16) || !aligned(dst_v, 16))
    return fail(PKV_ERR_INVALID_ARG, "pools must be 16-byte aligned");
  if (!aligned(src_blocks, 4) || !aligned(dst_blocks, 4))
    return fail(PKV_ERR_INVALID_ARG, "block id arrays must be 4-byte aligned");
  int dev;
  DeviceState* st;
  s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  const int64_t esz = cache->dtype == PKV_E4M3 ? 1 : 2;
  pkv::CopyParams p = {};
  p.k_src = src_k;
  p.v_src = src_v;
  p.k_dst = dst_k;
  p.v_dst = dst_v;
  p.src = src_blocks;
  p.dst = dst_blocks;
  p.n_pairs = n_pairs;
  p.block_vec = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size * cache->head_dim * esz / 16;
  p.src_blocks = src_num_blocks;
  p.dst_blocks = dst_num_blocks;
  if (max_ctas == 0) {
    // a copy across the host link saturates it with a few dozen CTAs; keep
    // the other SMs free for attention running beside it
    bool host_side = false;
    const void* pools[2] = {src_k, dst_k};
    for (const void* ptr : pools) {
      cudaPointerAttributes attr;
      if (cudaPointerGetAttributes(&attr, ptr) == cudaSuccess && attr.type == cudaMemoryTypeHost) host_side = true;
    }
    cudaGetLastError();  // a pointer the runtime does not know is not an error here
    max_ctas = host_side ? kHostLinkCopyCtas : 0;
  }
  p.max_ctas = max_ctas;
  p.err = st->err;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = traced(pkv::kKindBlockCopy, cs, [&] { return pkv::launch_copy_blocks(p, cs); });
  if (e != cudaSuccess) return cuda_fail(e, "block copy launch");
  return PKV_OK;
}

pkv_status pkv_selftest_wait_timeout(int32_t which, int32_t limit_us, pkv_stream_t stream) {
  if (which != 0 && which != 1) return fail(PKV_ERR_INVALID_ARG, "which %d (0 or 1)", which);
  if (limit_us < 1 || limit_us > 1000000) return fail(PKV_ERR_INVALID_ARG, "limit_us %d (1..1000000)", limit_us);
  int dev;
  DeviceState* st;
  pkv_status s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  cudaError_t e = pkv::launch_wait_selftest(which, static_cast<uint64_t>(limit_us) * 1000ull, st->err,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return PKV_OK;
}

pkv_status pkv_host_alloc(size_t bytes, void** ptr) {
  if (ptr == nullptr) return fail(PKV_ERR_INVALID_ARG, "ptr is NULL");
  *ptr = nullptr;
  if (bytes == 0) return fail(PKV_ERR_INVALID_ARG, "zero bytes");
  cudaError_t e = cudaHostAlloc(ptr, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc");
  return PKV_OK;
}

pkv_status pkv_host_free(void* ptr) {
  if (ptr == nullptr) return PKV_OK;
  cudaError_t e = cudaFreeHost(ptr);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeHost");
  return PKV_OK;
}

pkv_status pkv_decode_plan(int32_t batch, int32_t num_q_heads, const pkv_cache_desc* cache,
                           int32_t max_context_len, int32_t split_tokens, int32_t num_sms,
                           pkv_decode_plan_t* out) {
  if (out == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan output is NULL");
  return plan(batch, num_q_heads, cache, max_context_len, split_tokens, num_sms, out);
}

pkv_status pkv_decode_attention_ex(const void* q, int32_t batch, int32_t num_q_heads,
                                   const void* k_cache, const void* v_cache,
                                   const pkv_cache_desc* cache, const int32_t* block_tables,
                                   int32_t max_blocks_per_seq, const int32_t* context_lens,
                                   int32_t max_context_len, float scale, float* out,
                                   const float* k_scale, const float* v_scale,
                                   int64_t scale_row_stride, void* workspace,
                                   size_t workspace_bytes, int32_t split_tokens,
                                   pkv_stream_t stream) {
  DecodeArgs a = {q, batch, num_q_heads, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                  context_lens, max_context_len, scale, out, k_scale, v_scale, scale_row_stride};
  pkv_status s = check_decode(a);
  if (s != PKV_OK) return s;
  if (split_tokens < -1 || (split_tokens > 0 && split_tokens % 64 != 0))
    return fail(PKV_ERR_INVALID_ARG, "split_tokens %d (-1, 0 or a multiple of 64)", split_tokens);
  if (batch == 0) return PKV_OK;
  return run_decode(a, workspace, workspace_bytes, split_tokens,
                    reinterpret_cast<cudaStream_t>(stream), false);
}

pkv_status pkv_decode_attention_append(const void* q, int32_t batch, int32_t num_q_heads, void* k_cache,
                                       void* v_cache, const pkv_cache_desc* cache, const void* k_new,
                                       const void* v_new, int32_t new_dtype, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t max_context_len, float scale, float* out,
                                       const float* k_scale, const float* v_scale,
                                       int64_t scale_row_stride, void* workspace,
                                       size_t workspace_bytes, int32_t split_tokens,
                                       pkv_stream_t stream) {
  DecodeArgs a = {q, batch, num_q_heads, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                  context_lens, max_context_len, scale, out, k_scale, v_scale, scale_row_stride,
                  k_new, v_new, new_dtype};
  if (new_dtype == -1) return fail(PKV_ERR_INVALID_ARG, "new_dtype -1");
  pkv_status s = check_decode(a);
  if (s != PKV_OK) return s;
  if (split_tokens < 0 || split_tokens % 64 != 0)
    return fail(PKV_ERR_INVALID_ARG, "split_tokens %d (0 or a multiple of 64)", split_tokens);
  if (batch == 0) return PKV_OK;
  return run_decode(a, workspace, workspace_bytes, split_tokens,
                    reinterpret_cast<cudaStream_t>(stream), false);
}

pkv_status pkv_decode_attention(const void* q, int32_t batch, int32_t num_q_heads,
                                const void* k_cache, const void* v_cache,
                                const pkv_cache_desc* cache, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* context_lens,
                                int32_t max_context_len, float scale, float* out,
                                const float* k_scale, const float* v_scale,
                                int64_t scale_row_stride, pkv_stream_t stream) {
  DecodeArgs a = {q, batch, num_q_heads, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                  context_lens, max_context_len, scale, out, k_scale, v_scale, scale_row_stride};
  pkv_status s = check_decode(a);
  if (s != PKV_OK) return s;
  if (batch == 0) return PKV_OK;
  return run_decode(a, nullptr, 0, 0, reinterpret_cast<cudaStream_t>(stream), true);
}

int32_t pkv_get_device_error(pkv_stream_t stream) {
  int dev;
  DeviceState* st;
  if (current_device(&dev, &st) != PKV_OK) return -1;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return -1;
  int v = 0;
  if (cudaMemcpy(&v, st->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  const int zero = 0;
  if (cudaMemcpy(st->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return -1;
  return v;
}

const char* pkv_status_string(int32_t status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
    default: return "PKV_ERR_UNKNOWN";
  }
}

const char* pkv_last_error(void) { return t_last_error.c_str(); }

int32_t pkv_abi_version(void) { return 102; }

pkv_status pkv_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = on != 0;
  return PKV_OK;
}

int32_t pkv_trace_read(pkv_trace_entry* entries, int32_t capacity) {
  std::vector<TraceRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    recs.swap(g_trace);
  }
  pkv_trace_entry agg[pkv::kNumKernelKinds];
  for (int k = 0; k < pkv::kNumKernelKinds; ++k) agg[k] = {k, 0, 0.0};
  int bad = 0;
  for (const TraceRec& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      agg[r.kind].launches += 1;
      agg[r.kind].total_ms += ms;
    } else {
      ++bad;
    }
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_event_pool.push_back({r.dev, r.a});
    g_event_pool.push_back({r.dev, r.b});
  }
  if (bad) return -1;
  int n = 0;
  for (int k = 0; k < pkv::kNumKernelKinds && n < capacity; ++k) {
    if (agg[k].launches > 0 && entries != nullptr) entries[n++] = agg[k];
  }
  return n;
}

pkv_status pkv_shutdown(void) {
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    for (auto& pe : g_event_pool) cudaEventDestroy(pe.second);
    g_event_pool.clear();
    for (auto& r : g_trace) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
    g_trace.clear();
  }
  std::lock_guard<std::mutex> lk(g_mu);
  // Addresses and limits looked up in the current context are forgotten, so
  // that a device reset after this call leaves nothing stale: the next call
  // looks up the error word and the scratch array again and sets the kernels'
  // shared-memory limits again.
  g_config_epoch.fetch_add(1, std::memory_order_relaxed);
  for (auto& p : g_noalloc_ptr) p = nullptr;
  for (auto& s : g_dev) {
    s.ready = false;
    s.err = nullptr;
    if (s.pool != nullptr) {
      cudaMemPoolDestroy(s.pool);
      s.pool = nullptr;
    }
    if (s.side != nullptr) {
      cudaStreamDestroy(s.side);
      cudaEventDestroy(s.fork);
      cudaEventDestroy(s.join);
      s.side = nullptr;
      s.fork = s.join = nullptr;
    }
  }
  return PKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Cascade (shared-prefix) decode.
// ---------------------------------------------------------------------------

namespace {

pkv_status cascade_plan(int32_t batch, int32_t num_q_heads, const pkv_cache_desc* c, int32_t prefix_len,
                        int32_t max_ctx, int32_t sms, pkv_decode_plan_t* out) {
  pkv_status s = check_cache(c);
  if (s != PKV_OK) return s;
  if (c->dtype != PKV_BF16) return fail(PKV_ERR_UNSUPPORTED, "cascade decode takes bf16 caches");
  if (batch < 1 || batch > 65535) return fail(PKV_ERR_INVALID_ARG, "batch %d", batch);
  if (num_q_heads < 1 || num_q_heads % c->num_kv_heads != 0 || num_q_heads / c->num_kv_heads > 16)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d for %d KV heads", num_q_heads, c->num_kv_heads);
  if (prefix_len <= 0 || prefix_len % c->block_size != 0)
    return fail(PKV_ERR_INVALID_ARG, "prefix_len %d (a positive multiple of block_size %d)", prefix_len,
                c->block_size);
  if (max_ctx < prefix_len) return fail(PKV_ERR_INVALID_ARG, "max_context_len %d < prefix_len %d", max_ctx, prefix_len);
  if (sms <= 0) sms = kDefaultSms;
  const int32_t suffix = max_ctx - prefix_len;
  // Prefix ranges.  The prefix kernel runs one CTA (256 rows x one range)
  // per SM and the suffix decode runs beside it on the other SMs, so the
  // number of ranges n is the one that minimises the longer of (a) the
  // prefix CTAs' own time, waves x (tiles per range + two tiles of per-CTA
  // cost), and (b) prefix and suffix work spread over every SM.  Work is in
  // prefix-tile units: on GB300 a 64-key tile of a 256-row CTA took about as
  // long as one SM streams 92 KB of suffix K/V (2.2 us at 42 KB/us).  Fewer
  // ranges on ties (fewer pieces to combine).  On the 128-sequence workload
  // this picks 2 ranges (with 256-token suffix splits the call took 83.6 us,
  // against 93.1 with 4 ranges).
  const int64_t rows = static_cast<int64_t>(batch) * (num_q_heads / c->num_kv_heads);
  const int64_t row_blocks = ceil_div(rows, pkv::kCascadeRowsTc) * c->num_kv_heads;
  const int64_t tiles = ceil_div(prefix_len, pkv::kCascadeTile);
  const double suffix_work = static_cast<double>(batch) * c->num_kv_heads * (suffix > 0 ? suffix : 0) * 2.0 *
                             c->head_dim * 2.0 / (92.0 * 1024.0);
  int64_t nps = 1;
  double best = -1.0;
  for (int64_t n = 1; n <= tiles && n <= 64; ++n) {
    const int64_t per_cta = ceil_div(tiles, n) + 2;
    const double own = static_cast<double>(ceil_div(row_blocks * n, sms) * per_cta);
    const double spread = (static_cast<double>(row_blocks * n * per_cta) + suffix_work) / sms;
    const double est = own > spread ? own : spread;
    if (best < 0 || est < best) {
      best = est;
      nps = n;
    }
  }
  int64_t pst = ceil_div(ceil_div(prefix_len, nps), pkv::kCascadeTile) * pkv::kCascadeTile;
  const int64_t max_pst =
      static_cast<int64_t>(pkv::kCascadeMaxRangeBlocks) * c->block_size / pkv::kCascadeTile * pkv::kCascadeTile;
  if (pst > max_pst) pst = max_pst;
  nps = ceil_div(prefix_len, pst);
  // Suffix splits, sized for the SMs the prefix CTAs leave free and for two
  // waves of three CTAs per SM there rather than six: the suffix decode
  // streams beside the prefix, which covers its tail, and on short suffixes
  // each CTA's fixed cost (setup, pipeline fill, partial write) weighs on
  // every split.  On the 128-sequence workload (suffixes up to 1024 tokens)
  // this leaves each suffix whole: call 73.4 us, against 76.0 with 512-token
  // splits and 83.6 with the 256 of the six-wave rule over all SMs.
  const int64_t prefix_ctas = row_blocks * nps;
  const int32_t free_sms = static_cast<int32_t>(
      prefix_ctas < sms - sms / 4 ? sms - prefix_ctas : sms / 4 > 0 ? sms / 4 : 1);
  const int32_t st = auto_split_tokens(batch, c->num_kv_heads, suffix > 0 ? suffix : 1, free_sms, 2);
  const int64_t splits = suffix > 0 ? ceil_div(suffix, st) : 1;
  *out = pkv_decode_plan_t{};
  out->mode = 2;
  out->split_tokens = st;
  out->max_splits = static_cast<int32_t>(splits);
  out->workers = static_cast<int32_t>(nps);
  const int64_t slots = static_cast<int64_t>(batch) * num_q_heads * (splits + nps);
  out->workspace_bytes = align256(slots * c->head_dim * 4) + slots * 2 * 4;
  out->prefix_split_tokens = static_cast<int32_t>(pst);
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_cascade_plan(int32_t batch, int32_t num_q_heads, const pkv_cache_desc* cache,
                                       int32_t prefix_len, int32_t max_context_len, int32_t num_sms,
                                       pkv_decode_plan_t* plan) {
  if (plan == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan output is NULL");
  return cascade_plan(batch, num_q_heads, cache, prefix_len, max_context_len, num_sms, plan);
}

extern "C" pkv_status pkv_cascade_decode_attention(
    const void* q, int32_t batch, int32_t num_q_heads, const void* k_cache, const void* v_cache,
    const pkv_cache_desc* cache, const int32_t* prefix_blocks, int32_t prefix_len,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, float scale, float* out, void* workspace, size_t workspace_bytes,
    pkv_stream_t stream) {
  DecodeArgs a = {q, batch, num_q_heads, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                  context_lens, max_context_len, scale, out, nullptr, nullptr, 0};
  pkv_status s = check_decode(a);
  if (s != PKV_OK) return s;
  if (batch == 0) return PKV_OK;
  if (prefix_blocks == nullptr || !aligned(prefix_blocks, 4))
    return fail(PKV_ERR_INVALID_ARG, "prefix_blocks must be a 4-byte aligned device pointer");
  int dev;
  DeviceState* st;
  s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  pkv_decode_plan_t pl;
  s = cascade_plan(batch, num_q_heads, cache, prefix_len, max_context_len, st->sms, &pl);
  if (s != PKV_OK) return s;
  if (workspace == nullptr || workspace_bytes < static_cast<size_t>(pl.workspace_bytes))
    return fail(PKV_ERR_WORKSPACE, "workspace %zu bytes, need %lld", workspace_bytes,
                static_cast<long long>(pl.workspace_bytes));
  if (!aligned(workspace, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const pkv_cache_desc& c = *cache;
  CUtensorMap tk, tv;
  s = make_cache_tmap(&tk, k_cache, c);
  if (s != PKV_OK) return s;
  s = make_cache_tmap(&tv, v_cache, c);
  if (s != PKV_OK) return s;
  // the prefix kernel reads whole blocks (up to 64 tokens) per TMA box
  const int box = c.block_size < pkv::kCascadeTile ? c.block_size : pkv::kCascadeTile;
  CUtensorMap tkb, tvb;
  s = make_cache_tmap(&tkb, k_cache, c, box);
  if (s != PKV_OK) return s;
  s = make_cache_tmap(&tvb, v_cache, c, box);
  if (s != PKV_OK) return s;

  const int64_t slots = pl.max_splits + pl.workers;
  const int64_t rows = static_cast<int64_t>(batch) * num_q_heads * slots;
  DecodeParams p = {};
  p.q = q;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * c.head_dim * 4));
  p.num_blocks = c.num_blocks;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.group = num_q_heads / c.num_kv_heads;
  p.head_dim = c.head_dim;
  p.block_size = c.block_size;
  p.max_blocks = max_blocks_per_seq;
  p.max_ctx = max_context_len;
  p.split_tokens = pl.split_tokens;
  p.max_splits = pl.max_splits;
  p.qk_log2_scale = scale * 1.4426950408889634f;
  p.cache_dtype = c.dtype;
  p.mode = pkv::kModeFixedSplit;
  p.token_offset = prefix_len;
  p.force_partial = 1;
  p.extra_slot = pl.max_splits;
  p.extra_count = pl.workers;
  p.slots_per_row = static_cast<int32_t>(slots);
  p.prefix_blocks = prefix_blocks;
  p.prefix_len = prefix_len;
  p.prefix_split_tokens = pl.prefix_split_tokens;
  p.err = st->err;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // The prefix (tensor-core bound, from L2) and the suffix (HBM bound) do not
  // depend on each other.  The prefix is launched first, on the caller's
  // stream, so that its CTAs (one per SM) take their SMs before the suffix
  // decode, forked onto the library's side stream, fills the rest; the
  // combine waits for both.
  s = side_stream(st);
  if (s != PKV_OK) return s;
  std::lock_guard<std::mutex> fj(g_fork_mu);
  cudaError_t e = cudaEventRecord(st->fork, cs);
  if (e == cudaSuccess)
    e = traced(pkv::kKindCascadePrefix, cs, [&] { return pkv::launch_cascade_prefix(p, tkb, tvb, cs); });
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st->side, st->fork, 0);
  if (e == cudaSuccess)
    e = traced(pkv::kKindDecodeSplit, st->side, [&] { return pkv::launch_decode_split(p, tk, tv, st->side); });
  if (e == cudaSuccess) e = cudaEventRecord(st->join, st->side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, st->join, 0);
  if (e == cudaSuccess)
    e = traced(pkv::kKindCombine, cs, [&] { return pkv::launch_decode_combine(p, cs); });
  if (e != cudaSuccess) return cuda_fail(e, "cascade decode launch");
  return PKV_OK;
}

// ---------------------------------------------------------------------------
// Multi-token query attention (q_len new tokens per sequence, causal).
// ---------------------------------------------------------------------------

namespace {

// Work units of the tcgen05 multi-token kernel: (split, sequence, KV head,
// 128-row block).
int64_t tc_units(const pkv_decode_plan_t& pl, int32_t batch, int32_t q_len, int32_t num_q_heads,
                 const pkv_cache_desc& c) {
  const int64_t rows = static_cast<int64_t>(q_len) * (num_q_heads / c.num_kv_heads);
  return static_cast<int64_t>(pl.max_splits) * batch * c.num_kv_heads * ((rows + 127) / 128);
}

pkv_status mq_plan(int32_t batch, int32_t q_len, int32_t num_q_heads, const pkv_cache_desc* c,
                   int32_t max_ctx, int32_t split_tokens, int32_t sms, pkv_decode_plan_t* out) {
  pkv_status s = check_cache(c);
  if (s != PKV_OK) return s;
  if (c->dtype != PKV_BF16) return fail(PKV_ERR_UNSUPPORTED, "multi-token attention takes bf16 caches");
  if (batch < 0 || batch > 65535) return fail(PKV_ERR_INVALID_ARG, "batch %d", batch);
  if (q_len < 1 || q_len > 16) return fail(PKV_ERR_UNSUPPORTED, "q_len %d (1..16)", q_len);
  if (num_q_heads < 1 || num_q_heads % c->num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads,
                c->num_kv_heads);
  if (num_q_heads / c->num_kv_heads > 16)
    return fail(PKV_ERR_UNSUPPORTED, "group size %d > 16", num_q_heads / c->num_kv_heads);
  if (max_ctx < 0) return fail(PKV_ERR_INVALID_ARG, "max_context_len %d", max_ctx);
  const int64_t max_st = static_cast<int64_t>(pkv::kMultiQueryMaxSplitBlocks) * c->block_size;
  if (split_tokens < 0 || (split_tokens > 0 && (split_tokens % pkv::kMultiQueryTile != 0 || split_tokens > max_st)))
    return fail(PKV_ERR_INVALID_ARG, "split_tokens %d (0, or a multiple of 64 up to %lld)", split_tokens,
                static_cast<long long>(max_st));
  if (sms <= 0) sms = kDefaultSms;
  const int32_t rows = q_len * (num_q_heads / c->num_kv_heads);
  const int32_t lanes = pkv::multi_query_lanes(rows);
  const bool tc = rows >= pkv::kMultiQueryTcRows;
  const int64_t nrb = tc ? ceil_div(rows, 128) : ceil_div(rows, 16 * (4 / lanes));
  const int64_t units = static_cast<int64_t>(batch) * c->num_kv_heads * nrb;
  int32_t st = split_tokens;
  if (st == 0) {
    // mma.sync: as for decode, the largest power of two (256..4096) that
    // still gives about six waves of three CTAs per SM when every sequence is
    // as long as the bound (q_len 1 / 2 on the GQA workload: 1024-token
    // splits, 0.92 / 0.89 of HBM, against 0.90 / 0.87 at 2048).  tcgen05
    // (persistent, longest units first): the largest power of two up to the
    // longest split (1024 blocks) that still gives three units per SM (larger
    // units cost less per token: one setup, fewer partials)
    const int64_t want = static_cast<int64_t>(sms) * (tc ? 3 : 18);
    st = tc ? static_cast<int32_t>(max_st) : 4096;
    while (st > 256 && units * ceil_div(max_ctx, st) < want) st /= 2;
    // long contexts (more than 16 splits) on the mma.sync kernel (three CTAs
    // per SM): as for decode (q_len 2 on 8 sequences of 131k tokens: 6.94 TB/s
    // at 25 splits, 6.75 at the six-wave rule's 65); on the GQA batch the
    // half-wave choice measured 1-1.5 % slower, so shorter contexts keep the
    // six-wave rule
    if (!tc) {
      const int64_t lc = half_wave_split(units, max_ctx, sms, st, 16);
      st = static_cast<int32_t>(lc < max_st ? lc : max_st);
    }
  }
  const int64_t splits = max_ctx > 0 ? ceil_div(max_ctx, st) : 1;
  if (splits > 0x7FFFFFFFll) return fail(PKV_ERR_INVALID_ARG, "too many splits");
  if (static_cast<int64_t>(c->num_kv_heads) * nrb > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads x row blocks beyond the grid");
  *out = pkv_decode_plan_t{};
  out->mode = 3;
  out->split_tokens = st;
  out->max_splits = static_cast<int32_t>(splits);
  out->workers = rows >= pkv::kMultiQueryTcRows ? 0 : lanes;  // 0: the tcgen05 kernel
  if (splits > 1) {
    const int64_t n = static_cast<int64_t>(batch) * q_len * num_q_heads * splits;
    out->workspace_bytes = align256(n * c->head_dim * 4) + n * 2 * 4;
  }
  // the tcgen05 kernel's work-unit counter and unit order, after the partials
  if (tc) {
    const int64_t units = tc_units(*out, batch, q_len, num_q_heads, *c);
    if (units > (1ll << 28)) return fail(PKV_ERR_UNSUPPORTED, "%lld work units", static_cast<long long>(units));
    out->workspace_bytes = align256(out->workspace_bytes) + 256 + align256(units * 4);
  }
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_multi_query_plan(int32_t batch, int32_t q_len, int32_t num_q_heads,
                                           const pkv_cache_desc* cache, int32_t max_context_len,
                                           int32_t split_tokens, int32_t num_sms, pkv_decode_plan_t* plan) {
  if (plan == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan output is NULL");
  return mq_plan(batch, q_len, num_q_heads, cache, max_context_len, split_tokens, num_sms, plan);
}

extern "C" pkv_status pkv_multi_query_attention(
    const void* q, int32_t batch, int32_t q_len, int32_t num_q_heads, const void* k_cache,
    const void* v_cache, const pkv_cache_desc* cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len, float scale,
    float* out, void* workspace, size_t workspace_bytes, int32_t split_tokens, pkv_stream_t stream) {
  DecodeArgs a = {q, batch, num_q_heads, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                  context_lens, max_context_len, scale, out, nullptr, nullptr, 0};
  pkv_status s = check_decode(a);
  if (s != PKV_OK) return s;
  pkv_decode_plan_t pl;
  s = mq_plan(batch, q_len, num_q_heads, cache, max_context_len, split_tokens, kDefaultSms, &pl);
  if (s != PKV_OK) return s;
  if (batch == 0) return PKV_OK;
  int dev;
  DeviceState* st;
  s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  if (split_tokens == 0) {
    s = mq_plan(batch, q_len, num_q_heads, cache, max_context_len, 0, st->sms, &pl);
    if (s != PKV_OK) return s;
  }
  if (pl.workspace_bytes > 0) {
    if (workspace == nullptr || workspace_bytes < static_cast<size_t>(pl.workspace_bytes))
      return fail(PKV_ERR_WORKSPACE, "workspace %zu bytes, need %lld", workspace_bytes,
                  static_cast<long long>(pl.workspace_bytes));
    if (!aligned(workspace, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  const pkv_cache_desc& c = *cache;
  // q_len * G >= 64 rows: the tcgen05 kernel, which reads whole blocks per TMA box
  const bool tc = pl.workers == 0;
  const int box = tc ? (c.block_size < pkv::kCascadeTile ? c.block_size : pkv::kCascadeTile) : pkv::kTileTokens;
  CUtensorMap tk, tv;
  s = make_cache_tmap(&tk, k_cache, c, box);
  if (s != PKV_OK) return s;
  s = make_cache_tmap(&tv, v_cache, c, box);
  if (s != PKV_OK) return s;
  const int64_t n = static_cast<int64_t>(batch) * q_len * num_q_heads * pl.max_splits;
  DecodeParams p = {};
  p.q = q;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.ws_o = pl.max_splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.ws_ml = pl.max_splits > 1
                ? reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(n * c.head_dim * 4))
                : nullptr;
  p.num_blocks = c.num_blocks;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.group = num_q_heads / c.num_kv_heads;
  p.head_dim = c.head_dim;
  p.block_size = c.block_size;
  p.max_blocks = max_blocks_per_seq;
  p.max_ctx = max_context_len;
  p.split_tokens = pl.split_tokens;
  p.max_splits = pl.max_splits;
  p.qk_log2_scale = scale * 1.4426950408889634f;
  p.cache_dtype = c.dtype;
  p.mode = pkv::kModeFixedSplit;
  p.extra_slot = -1;
  p.slots_per_row = pl.max_splits;
  p.q_len = q_len;
  p.err = st->err;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (tc) {
    // persistent grid (one CTA per SM) over work units taken, longest first,
    // from a counter after the partials in the workspace (the unit order
    // follows it)
    const int64_t units = tc_units(pl, batch, q_len, num_q_heads, c);
    p.workers = static_cast<int32_t>(units < st->sms ? (units > 0 ? units : 1) : st->sms);
    const int64_t part = pl.max_splits > 1 ? align256(align256(n * c.head_dim * 4) + n * 2 * 4) : 0;
    p.ws_q = reinterpret_cast<int*>(static_cast<char*>(workspace) + part);
  }
  if (e == cudaSuccess)
    e = traced(pkv::kKindMultiQuery, cs, [&] {
      return tc ? pkv::launch_multi_query_tc(p, tk, tv, cs) : pkv::launch_multi_query(p, tk, tv, cs);
    });
  if (e == cudaSuccess && pl.max_splits > 1) {
    DecodeParams pc = p;            // rows (b, i, hq) flatten to b * (q_len * H_q) + i * H_q + hq
    pc.num_q_heads = q_len * num_q_heads;
    e = traced(pkv::kKindCombine, cs, [&] { return pkv::launch_decode_combine(pc, cs); });
  }
  if (e != cudaSuccess) return cuda_fail(e, "multi-token attention launch");
  return PKV_OK;
}

// ---------------------------------------------------------------------------
// Decode attention that allocates nothing.
//
// The split-KV partials live in a fixed array in device memory that belongs to
// this library, instead of memory the caller or a pool hands over.  This is
// for callers that are not allowed to call cudaMalloc (or any allocator) at
// the point where they run attention: serving loops that reserve all device
// memory up front and forbid allocation afterwards, runtimes whose memory is
// owned by a different allocator, and code that must not block on the
// allocator's locks.  Host code only ever uses the array through the address
// returned by cudaGetSymbolAddress; the array's name itself is a host-side
// stand-in and must never be passed to a kernel.
// ---------------------------------------------------------------------------

static constexpr size_t kNoAllocScratchBytes = 32ull << 20;  // 32 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Once per device, with that device current: the device address of the array.
pkv_status noalloc_scratch(int dev, void** ptr) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_decode_attention_noalloc(
    const void* q, int32_t batch, int32_t num_q_heads, const void* k_cache, const void* v_cache,
    const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, float scale, float* out,
    const float* k_scale, const float* v_scale, int64_t scale_row_stride, pkv_stream_t stream) {
  DecodeArgs a = {q, batch, num_q_heads, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                  context_lens, max_context_len, scale, out, k_scale, v_scale, scale_row_stride};
  pkv_status s = check_decode(a);
  if (s != PKV_OK) return s;
  if (batch == 0) return PKV_OK;
  int dev;
  DeviceState* st;
  s = current_device(&dev, &st);
  if (s != PKV_OK) return s;
  pkv_decode_plan_t pl;
  s = plan(batch, num_q_heads, cache, max_context_len, 0, st->sms, &pl);
  if (s != PKV_OK) return s;
  if (static_cast<size_t>(pl.workspace_bytes) > kNoAllocScratchBytes)
    return fail(PKV_ERR_WORKSPACE,
                "this decode needs %lld bytes of split-KV scratch but the no-allocation entry "
                "point has %zu; use pkv_decode_attention_ex with caller memory",
                static_cast<long long>(pl.workspace_bytes), kNoAllocScratchBytes);
  void* ws = nullptr;
  s = noalloc_scratch(dev, &ws);
  if (s != PKV_OK) return s;
  return run_decode(a, ws, kNoAllocScratchBytes, 0, reinterpret_cast<cudaStream_t>(stream), false);
}
