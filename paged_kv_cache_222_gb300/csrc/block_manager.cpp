// Host block manager of the paged KV cache: free pool (a stack), reference
// counts, per-sequence block tables, copy-on-write and all-or-nothing appends.
//
// What it does: [FN] "Sub-Millisecond Token Scheduling...", section "Paged
// KV-Cache with Radix Tree Prefix Cache" (blocks with reference counts, a free
// pool, tables grown one block at a time, exhaustion reported so that the
// scheduler preempts, shared prompts referencing the same blocks through
// copy-on-write pointers); [SC] "LLM inference: prefill, decode, KV cache",
// "PagedAttention & Memory Management (vLLM)" and "9. Failure modes and
// limitations", item 2.  The policy choices (stack order, copy-on-write on the
// first write into a shared last block, all-or-nothing batches) are stated in
// pkv_blocks.h.
//
// Every operation is O(blocks touched): an append of n tokens costs
// O(n / block_size) pool operations plus O(n) slot writes, with one hash
// lookup per sequence.

#include <cstdarg>
#include <algorithm>
#include <cstdio>
#include <limits>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_blocks.h"
#include "pkv_internal.h"

struct pkv_block_manager {
  struct Seq {
    std::vector<int32_t> blocks;  // device id, or host id where on_host[j]
    std::vector<uint8_t> on_host;
    int64_t len = 0;
    int64_t host_entries = 0;
  };
  std::mutex mu;
  int32_t block_size = 0;
  std::vector<int32_t> ref;
  std::vector<int32_t> free_stack;  // top = back()
  bool host_tier = false;
  std::vector<int32_t> host_free;   // host pool, same stack rule
  std::unordered_map<int64_t, Seq> seqs;
};

namespace {

pkv_status fail(pkv_status s, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  pkv::set_last_error(buf);
  return s;
}

using Manager = pkv_block_manager;

// Blocks of the pool that appending n tokens to `q` takes, with the pending
// reference drops of earlier sequences of the same call in `dropped`.
struct Need {
  int64_t fresh = 0;  // positions that start a block
  bool cow = false;   // first write lands in a shared last block
};

Need need_of(const Manager& m, const Manager::Seq& q, int64_t n,
             std::unordered_map<int32_t, int32_t>& dropped) {
  Need r;
  if (n <= 0) return r;
  const int64_t bs = m.block_size;
  const int64_t have = (q.len + bs - 1) / bs;
  const int64_t want = (q.len + n + bs - 1) / bs;
  r.fresh = want - have;
  if (q.len % bs != 0) {
    const int32_t last = q.blocks[static_cast<size_t>(q.len / bs)];
    auto it = dropped.find(last);
    const int32_t refs = m.ref[static_cast<size_t>(last)] - (it == dropped.end() ? 0 : it->second);
    if (refs > 1) {
      r.cow = true;
      dropped[last] += 1;
    }
  }
  return r;
}

pkv_status check_batch(Manager* m, int32_t n_seqs, const int64_t* ids, const int32_t* n_new,
                       std::vector<Manager::Seq*>& out) {
  if (n_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "n_seqs %d", n_seqs);
  if (n_seqs > 0 && (ids == nullptr || n_new == nullptr))
    return fail(PKV_ERR_INVALID_ARG, "NULL seq_ids / n_new");
  out.resize(static_cast<size_t>(n_seqs));
  std::unordered_map<int64_t, int32_t> seen;
  seen.reserve(static_cast<size_t>(n_seqs) * 2);
  for (int32_t i = 0; i < n_seqs; ++i) {
    if (n_new[i] < 0) return fail(PKV_ERR_INVALID_ARG, "n_new[%d] = %d", i, n_new[i]);
    auto it = m->seqs.find(ids[i]);
    if (it == m->seqs.end())
      return fail(PKV_ERR_INVALID_ARG, "unknown sequence %lld", static_cast<long long>(ids[i]));
    if (!seen.emplace(ids[i], i).second)
      return fail(PKV_ERR_INVALID_ARG, "sequence %lld appears twice", static_cast<long long>(ids[i]));
    if (it->second.host_entries != 0)
      return fail(PKV_ERR_INVALID_ARG, "sequence %lld has blocks on the host", static_cast<long long>(ids[i]));
    out[static_cast<size_t>(i)] = &it->second;
  }
  return PKV_OK;
}

int32_t take(Manager& m) {
  const int32_t b = m.free_stack.back();
  m.free_stack.pop_back();
  m.ref[static_cast<size_t>(b)] += 1;
  return b;
}

}  // namespace

extern "C" {

pkv_status pkv_bm_create(int64_t num_blocks, int32_t block_size, pkv_block_manager** out) {
  if (out == nullptr) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_blocks < 1 || num_blocks > std::numeric_limits<int32_t>::max())
    return fail(PKV_ERR_INVALID_ARG, "num_blocks %lld", static_cast<long long>(num_blocks));
  if (block_size < 1) return fail(PKV_ERR_INVALID_ARG, "block_size %d", block_size);
  Manager* m = new (std::nothrow) Manager();
  if (m == nullptr) return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  m->block_size = block_size;
  m->ref.assign(static_cast<size_t>(num_blocks), 0);
  m->free_stack.resize(static_cast<size_t>(num_blocks));
  for (int64_t i = 0; i < num_blocks; ++i) m->free_stack[static_cast<size_t>(i)] = static_cast<int32_t>(i);
  *out = m;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int64_t pkv_bm_num_free(pkv_block_manager* bm) {
  if (bm == nullptr) return -1;
  std::lock_guard<std::mutex> lk(bm->mu);
  return static_cast<int64_t>(bm->free_stack.size());
}

int32_t pkv_bm_ref_count(pkv_block_manager* bm, int64_t block) {
  if (bm == nullptr) return -1;
  std::lock_guard<std::mutex> lk(bm->mu);
  if (block < 0 || block >= static_cast<int64_t>(bm->ref.size())) return -1;
  return bm->ref[static_cast<size_t>(block)];
}

int64_t pkv_bm_seq_len(pkv_block_manager* bm, int64_t seq_id) {
  if (bm == nullptr) return -1;
  std::lock_guard<std::mutex> lk(bm->mu);
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : it->second.len;
}

int64_t pkv_bm_num_sequences(pkv_block_manager* bm) {
  if (bm == nullptr) return -1;
  std::lock_guard<std::mutex> lk(bm->mu);
  return static_cast<int64_t>(bm->seqs.size());
}

pkv_status pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id) {
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARG, "manager is NULL");
  std::lock_guard<std::mutex> lk(bm->mu);
  if (!bm->seqs.emplace(seq_id, Manager::Seq()).second)
    return fail(PKV_ERR_INVALID_ARG, "sequence %lld exists", static_cast<long long>(seq_id));
  return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id) {
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARG, "manager is NULL");
  std::lock_guard<std::mutex> lk(bm->mu);
  auto p = bm->seqs.find(parent_id);
  if (p == bm->seqs.end())
    return fail(PKV_ERR_INVALID_ARG, "unknown parent %lld", static_cast<long long>(parent_id));
  if (bm->seqs.count(child_id) != 0)
    return fail(PKV_ERR_INVALID_ARG, "sequence %lld exists", static_cast<long long>(child_id));
  if (p->second.host_entries != 0)
    return fail(PKV_ERR_INVALID_ARG, "parent %lld has blocks on the host", static_cast<long long>(parent_id));
  Manager::Seq child = p->second;  // copy before the map may rehash
  for (int32_t b : child.blocks) bm->ref[static_cast<size_t>(b)] += 1;
  bm->seqs.emplace(child_id, std::move(child));
  return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id) {
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARG, "manager is NULL");
  std::lock_guard<std::mutex> lk(bm->mu);
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end())
    return fail(PKV_ERR_INVALID_ARG, "unknown sequence %lld", static_cast<long long>(seq_id));
  const Manager::Seq& sq = it->second;
  for (size_t j = 0; j < sq.blocks.size(); ++j) {
    const int32_t b = sq.blocks[j];
    if (sq.on_host[j]) {
      bm->host_free.push_back(b);
      continue;
    }
    int32_t& r = bm->ref[static_cast<size_t>(b)];
    r -= 1;
    if (r == 0) bm->free_stack.push_back(b);
  }
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_blocks_needed(pkv_block_manager* bm, int32_t n_seqs, const int64_t* seq_ids,
                                const int32_t* n_new, int64_t* blocks_needed) {
  if (bm == nullptr || blocks_needed == nullptr) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  std::lock_guard<std::mutex> lk(bm->mu);
  std::vector<Manager::Seq*> q;
  pkv_status s = check_batch(bm, n_seqs, seq_ids, n_new, q);
  if (s != PKV_OK) return s;
  std::unordered_map<int32_t, int32_t> dropped;
  int64_t total = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    const Need nd = need_of(*bm, *q[static_cast<size_t>(i)], n_new[i], dropped);
    total += nd.fresh + (nd.cow ? 1 : 0);
  }
  *blocks_needed = total;
  return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager* bm, int32_t n_seqs, const int64_t* seq_ids,
                         const int32_t* n_new, int64_t* slots, int32_t* cow_src,
                         int32_t* cow_dst, int32_t cow_capacity, int32_t* n_cow) {
  if (bm == nullptr || n_cow == nullptr) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  std::lock_guard<std::mutex> lk(bm->mu);
  std::vector<Manager::Seq*> q;
  pkv_status s = check_batch(bm, n_seqs, seq_ids, n_new, q);
  if (s != PKV_OK) return s;
  // phase 1: what the whole call takes, nothing changed yet
  std::unordered_map<int32_t, int32_t> dropped;
  int64_t fresh = 0, cows = 0, tokens = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    const Need nd = need_of(*bm, *q[static_cast<size_t>(i)], n_new[i], dropped);
    fresh += nd.fresh;
    cows += nd.cow ? 1 : 0;
    tokens += n_new[i];
  }
  if (tokens > 0 && slots == nullptr) return fail(PKV_ERR_INVALID_ARG, "slots is NULL");
  if (cows > cow_capacity || (cows > 0 && (cow_src == nullptr || cow_dst == nullptr)))
    return fail(PKV_ERR_INVALID_ARG, "%lld copy-on-write pairs, capacity %d", static_cast<long long>(cows),
                cow_capacity);
  if (fresh + cows > static_cast<int64_t>(bm->free_stack.size()))
    return fail(PKV_ERR_OUT_OF_BLOCKS, "append needs %lld blocks, %zu free",
                static_cast<long long>(fresh + cows), bm->free_stack.size());
  // phase 2: apply, in the order the policy fixes
  const int64_t bs = bm->block_size;
  int64_t k = 0;
  int32_t nc = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    Manager::Seq& sq = *q[static_cast<size_t>(i)];
    for (int32_t j = 0; j < n_new[i]; ++j) {
      const int64_t pos = sq.len + j;
      const size_t lb = static_cast<size_t>(pos / bs);
      if (pos % bs == 0) {
        sq.blocks.push_back(take(*bm));
        sq.on_host.push_back(0);
      } else {
        const int32_t last = sq.blocks[lb];
        if (bm->ref[static_cast<size_t>(last)] > 1) {
          const int32_t nb = take(*bm);
          cow_src[nc] = last;
          cow_dst[nc] = nb;
          ++nc;
          bm->ref[static_cast<size_t>(last)] -= 1;
          sq.blocks[lb] = nb;
        }
      }
      slots[k++] = static_cast<int64_t>(sq.blocks[lb]) * bs + pos % bs;
    }
    sq.len += n_new[i];
  }
  *n_cow = nc;
  return PKV_OK;
}

pkv_status pkv_bm_block_tables(pkv_block_manager* bm, int32_t n_seqs, const int64_t* seq_ids,
                                int32_t max_blocks_per_seq, int32_t* block_tables,
                                int32_t* context_lens) {
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARG, "manager is NULL");
  if (n_seqs < 0 || max_blocks_per_seq < 1)
    return fail(PKV_ERR_INVALID_ARG, "n_seqs %d, max_blocks_per_seq %d", n_seqs, max_blocks_per_seq);
  if (n_seqs > 0 && (seq_ids == nullptr || block_tables == nullptr))
    return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  std::lock_guard<std::mutex> lk(bm->mu);
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end())
      return fail(PKV_ERR_INVALID_ARG, "unknown sequence %lld", static_cast<long long>(seq_ids[i]));
    if (it->second.blocks.size() > static_cast<size_t>(max_blocks_per_seq))
      return fail(PKV_ERR_INVALID_ARG, "sequence %lld holds %zu blocks > %d",
                  static_cast<long long>(seq_ids[i]), it->second.blocks.size(), max_blocks_per_seq);
    if (it->second.len > std::numeric_limits<int32_t>::max())
      return fail(PKV_ERR_INVALID_ARG, "sequence length beyond int32");
    if (it->second.host_entries != 0)
      return fail(PKV_ERR_INVALID_ARG, "sequence %lld has blocks on the host",
                  static_cast<long long>(seq_ids[i]));
  }
  for (int32_t i = 0; i < n_seqs; ++i) {
    const Manager::Seq& sq = bm->seqs.find(seq_ids[i])->second;
    int32_t* row = block_tables + static_cast<int64_t>(i) * max_blocks_per_seq;
    const size_t n = sq.blocks.size();
    for (size_t j = 0; j < static_cast<size_t>(max_blocks_per_seq); ++j)
      row[j] = j < n ? sq.blocks[j] : -1;
    if (context_lens != nullptr) context_lens[i] = static_cast<int32_t>(sq.len);
  }
  return PKV_OK;
}

// ------------------------------------------------------------ host tier

namespace {

// Logical indices of one call: distinct and inside the table.
pkv_status check_logical(const Manager::Seq& sq, int32_t n, const int32_t* logical) {
  if (n < 0 || (n > 0 && logical == nullptr)) return fail(PKV_ERR_INVALID_ARG, "bad logical list");
  std::vector<uint8_t> seen(sq.blocks.size(), 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t j = logical[i];
    if (j < 0 || static_cast<size_t>(j) >= sq.blocks.size())
      return fail(PKV_ERR_INVALID_ARG, "logical block %d outside the table (%zu)", j, sq.blocks.size());
    if (seen[static_cast<size_t>(j)]) return fail(PKV_ERR_INVALID_ARG, "logical block %d repeated", j);
    seen[static_cast<size_t>(j)] = 1;
  }
  return PKV_OK;
}

pkv_status find_seq(Manager* bm, int64_t seq_id, Manager::Seq** out) {
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID_ARG, "unknown sequence %lld", static_cast<long long>(seq_id));
  *out = &it->second;
  return PKV_OK;
}

// Demote (to_host) or promote entries; pairs are (from id, to id).
pkv_status move_entries(Manager* bm, Manager::Seq& sq, int32_t n, const int32_t* logical, bool to_host,
                        int32_t* from, int32_t* to, int32_t* n_pairs) {
  if (!bm->host_tier) return fail(PKV_ERR_INVALID_ARG, "no host tier (pkv_bm_set_host_blocks)");
  if (n_pairs == nullptr) return fail(PKV_ERR_INVALID_ARG, "n_pairs is NULL");
  pkv_status s = check_logical(sq, n, logical);
  if (s != PKV_OK) return s;
  int64_t todo = 0;
  for (int32_t i = 0; i < n; ++i) todo += (sq.on_host[static_cast<size_t>(logical[i])] != 0) != to_host;
  if (todo > 0 && (from == nullptr || to == nullptr)) return fail(PKV_ERR_INVALID_ARG, "NULL pair arrays");
  const size_t avail = to_host ? bm->host_free.size() : bm->free_stack.size();
  if (todo > static_cast<int64_t>(avail))
    return fail(PKV_ERR_OUT_OF_BLOCKS, "%s pool: %lld blocks needed, %zu free", to_host ? "host" : "device",
                static_cast<long long>(todo), avail);
  int32_t k = 0;
  for (int32_t i = 0; i < n; ++i) {
    const size_t j = static_cast<size_t>(logical[i]);
    if ((sq.on_host[j] != 0) == to_host) continue;  // already in the target tier
    const int32_t old = sq.blocks[j];
    int32_t nb;
    if (to_host) {
      nb = bm->host_free.back();
      bm->host_free.pop_back();
      int32_t& r = bm->ref[static_cast<size_t>(old)];
      r -= 1;
      if (r == 0) bm->free_stack.push_back(old);
      sq.host_entries += 1;
    } else {
      nb = take(*bm);
      bm->host_free.push_back(old);
      sq.host_entries -= 1;
    }
    from[k] = old;
    to[k] = nb;
    ++k;
    sq.blocks[j] = nb;
    sq.on_host[j] = to_host ? 1 : 0;
  }
  *n_pairs = k;
  return PKV_OK;
}

}  // namespace

pkv_status pkv_bm_set_host_blocks(pkv_block_manager* bm, int64_t num_host_blocks) {
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARG, "manager is NULL");
  if (num_host_blocks < 1 || num_host_blocks > std::numeric_limits<int32_t>::max())
    return fail(PKV_ERR_INVALID_ARG, "num_host_blocks %lld", static_cast<long long>(num_host_blocks));
  std::lock_guard<std::mutex> lk(bm->mu);
  if (bm->host_tier) return fail(PKV_ERR_INVALID_ARG, "host tier already set");
  bm->host_free.resize(static_cast<size_t>(num_host_blocks));
  for (int64_t i = 0; i < num_host_blocks; ++i) bm->host_free[static_cast<size_t>(i)] = static_cast<int32_t>(i);
  bm->host_tier = true;
  return PKV_OK;
}

int64_t pkv_bm_num_free_host(pkv_block_manager* bm) {
  if (bm == nullptr) return -1;
  std::lock_guard<std::mutex> lk(bm->mu);
  return static_cast<int64_t>(bm->host_free.size());
}

int64_t pkv_bm_host_entries(pkv_block_manager* bm, int64_t seq_id) {
  if (bm == nullptr) return -1;
  std::lock_guard<std::mutex> lk(bm->mu);
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : it->second.host_entries;
}

pkv_status pkv_bm_evict(pkv_block_manager* bm, int64_t seq_id, int32_t n, const int32_t* logical,
                        int32_t* dev_src, int32_t* host_dst, int32_t* n_pairs) {
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARG, "manager is NULL");
  std::lock_guard<std::mutex> lk(bm->mu);
  Manager::Seq* sq;
  pkv_status s = find_seq(bm, seq_id, &sq);
  if (s != PKV_OK) return s;
  return move_entries(bm, *sq, n, logical, true, dev_src, host_dst, n_pairs);
}

pkv_status pkv_bm_stage(pkv_block_manager* bm, int64_t seq_id, int32_t n, const int32_t* logical,
                        int32_t* host_src, int32_t* dev_dst, int32_t* n_pairs) {
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARG, "manager is NULL");
  std::lock_guard<std::mutex> lk(bm->mu);
  Manager::Seq* sq;
  pkv_status s = find_seq(bm, seq_id, &sq);
  if (s != PKV_OK) return s;
  return move_entries(bm, *sq, n, logical, false, host_src, dev_dst, n_pairs);
}

pkv_status pkv_bm_table_entries(pkv_block_manager* bm, int64_t seq_id, int32_t capacity, int32_t* ids,
                                int32_t* on_host, int32_t* n_entries) {
  if (bm == nullptr || n_entries == nullptr) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  std::lock_guard<std::mutex> lk(bm->mu);
  Manager::Seq* sq;
  pkv_status s = find_seq(bm, seq_id, &sq);
  if (s != PKV_OK) return s;
  const size_t n = sq->blocks.size();
  if (static_cast<int64_t>(n) > capacity || (n > 0 && (ids == nullptr || on_host == nullptr)))
    return fail(PKV_ERR_INVALID_ARG, "table of %zu entries, capacity %d", n, capacity);
  for (size_t j = 0; j < n; ++j) {
    ids[j] = sq->blocks[j];
    on_host[j] = sq->on_host[j];
  }
  *n_entries = static_cast<int32_t>(n);
  return PKV_OK;
}

pkv_status pkv_bm_prefetch_candidates(pkv_block_manager* bm, int64_t seq_id, const float* activation,
                                      float threshold, int32_t capacity, int32_t* logical, int32_t* n_out) {
  if (bm == nullptr || n_out == nullptr) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  if (capacity < 0) return fail(PKV_ERR_INVALID_ARG, "capacity %d", capacity);
  std::lock_guard<std::mutex> lk(bm->mu);
  Manager::Seq* sq;
  pkv_status s = find_seq(bm, seq_id, &sq);
  if (s != PKV_OK) return s;
  const int64_t n = static_cast<int64_t>(sq->blocks.size());
  if (n > 0 && activation == nullptr) return fail(PKV_ERR_INVALID_ARG, "activation is NULL");
  std::vector<int32_t> c;
  for (int64_t j = 0; j < n; ++j)
    if (sq->on_host[static_cast<size_t>(j)] && activation[j] > threshold) c.push_back(static_cast<int32_t>(j));
  std::stable_sort(c.begin(), c.end(), [&](int32_t a, int32_t b) { return activation[a] > activation[b]; });
  size_t keep = c.size();
  if (keep > static_cast<size_t>(capacity)) keep = static_cast<size_t>(capacity);
  if (keep > bm->free_stack.size()) keep = bm->free_stack.size();
  if (keep > 0 && logical == nullptr) return fail(PKV_ERR_INVALID_ARG, "logical is NULL");
  for (size_t i = 0; i < keep; ++i) logical[i] = c[i];
  *n_out = static_cast<int32_t>(keep);
  return PKV_OK;
}

}  // extern "C"
