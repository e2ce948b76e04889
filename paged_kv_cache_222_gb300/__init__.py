"""GB300-native paged-KV decode attention: Python binding of libpkv.so.

Every function here only checks tensor shapes / dtypes and hands raw device
pointers plus the current CUDA stream to the C ABI (include/pkv.h); all of the
computation runs in the library's sm_103a kernels.  PyTorch supplies device
memory and streams.

    append(k_new, v_new, slot_mapping, k_cache, v_cache[, k_scale, v_scale])
    decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale
                     [, k_scale, v_scale]) -> out (float32)

Cache tensors are [num_blocks, H_kv, block_size, head_dim], bf16 or E4M3
(torch.uint8 or torch.float8_e4m3fn storage).
"""

import ctypes

import numpy as np
import torch

from . import _lib
from ._lib import (PKV_BF16, PKV_E4M3, PKV_F32, CacheDesc, DecodePlan, PkvError,  # noqa: F401
                   TraceEntry)

__all__ = ["append", "decode_attention", "decode_plan", "cache_desc", "slot_mapping",
           "cascade_plan", "cascade_decode_attention", "multi_query_plan", "multi_query_attention",
           "BlockManager", "OutOfBlocks", "copy_blocks",
           "host_pool_like", "copy_blocks_between",
           "device_error", "trace_enable", "trace_read", "library", "PkvError"]

KERNEL_KINDS = {0: "append", 1: "decode_split", 2: "combine", 3: "cascade_prefix", 4: "block_copy",
                5: "multi_query", 6: "slot_mapping"}


def library():
    """The loaded ctypes library (raises if libpkv.so is not built)."""
    return _lib.load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cache_dtype(t):
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return PKV_E4M3
    raise TypeError(f"cache dtype {t.dtype}: expected bfloat16 or uint8/float8_e4m3fn")


def cache_desc(k_cache):
    """C descriptor of a [num_blocks, H_kv, block_size, head_dim] cache tensor."""
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d, _cache_dtype(k_cache))


def _check_pair(k_cache, v_cache):
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must have the same shape and dtype")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    if k_cache.device != v_cache.device or k_cache.device.type != "cuda":
        raise ValueError("caches must be CUDA tensors on one device")


def _contig(t, dtype, name, device):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def append(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None,
           scale_row_stride=None):
    """Write rows k_new[i] / v_new[i] ([N, H_kv, D], bf16 or fp32) into flat slots
    slot_mapping[i] (int64; phys * block_size + offset; < 0 skips).

    E4M3 caches need k_scale / v_scale (float32): [N, H_kv] per-row scales, or
    [H_kv] per-head scales (then scale_row_stride defaults to 0).
    """
    lib = library()
    _check_pair(k_cache, v_cache)
    dev = k_cache.device
    desc = cache_desc(k_cache)
    if k_new.shape != v_new.shape or k_new.dim() != 3:
        raise ValueError("k_new / v_new must both be [N, H_kv, D]")
    n, hkv, d = k_new.shape
    if hkv != desc.num_kv_heads or d != desc.head_dim:
        raise ValueError("k_new heads / head_dim do not match the cache")
    if k_new.dtype == torch.bfloat16:
        src = PKV_BF16
    elif k_new.dtype == torch.float32:
        src = PKV_F32
    else:
        raise TypeError(f"k_new dtype {k_new.dtype}: expected bfloat16 or float32")
    _contig(k_new, k_new.dtype, "k_new", dev)
    _contig(v_new, k_new.dtype, "v_new", dev)
    _contig(slot_mapping, torch.int64, "slot_mapping", dev)
    if slot_mapping.numel() != n:
        raise ValueError("slot_mapping must have one entry per row")
    if desc.dtype == PKV_E4M3:
        if k_scale is None or v_scale is None:
            raise ValueError("E4M3 cache needs k_scale and v_scale")
        _contig(k_scale, torch.float32, "k_scale", dev)
        _contig(v_scale, torch.float32, "v_scale", dev)
        if scale_row_stride is None:
            scale_row_stride = hkv if k_scale.dim() == 2 else 0
    else:
        scale_row_stride = 0
    st = lib.pkv_append(_ptr(k_new), _ptr(v_new), src, n, _ptr(slot_mapping), _ptr(k_cache),
                        _ptr(v_cache), ctypes.byref(desc), _ptr(k_scale), _ptr(v_scale),
                        int(scale_row_stride), _stream(dev))
    _lib.check(st, "pkv_append")


def decode_plan(batch, num_q_heads, k_cache_or_desc, max_context_len, split_tokens=0, num_sms=0):
    """Split-KV plan (host only): tokens per split, splits, workspace bytes."""
    lib = library()
    desc = k_cache_or_desc if isinstance(k_cache_or_desc, CacheDesc) else cache_desc(k_cache_or_desc)
    plan = DecodePlan()
    st = lib.pkv_decode_plan(int(batch), int(num_q_heads), ctypes.byref(desc), int(max_context_len),
                             int(split_tokens), int(num_sms), ctypes.byref(plan))
    _lib.check(st, "pkv_decode_plan")
    return plan


def decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale=None,
                     v_scale=None, max_context_len=None, out=None, split_tokens=0,
                     workspace=None, scale_row_stride=None, k_new=None, v_new=None):
    """Single-token decode attention over the paged cache.

    q [B, H_q, D] bf16; block_tables [B, MB] int32; context_lens [B] int32
    (tokens attended, the appended one included); returns out [B, H_q, D]
    float32.  `max_context_len` is a host bound on context_lens (if None, the
    block tables' capacity MB * block_size, which plans more splits than a
    tighter bound).  E4M3 caches take k_scale /
    v_scale float32 [B, H_kv] (or [H_kv] for one scale per head).

    With k_new / v_new ([B, H_kv, D], bf16 or float32) the step's new tokens
    are appended in the same launch (pkv_decode_attention_append): row b goes
    to position context_lens[b] - 1, encoded as `append` encodes it.
    """
    lib = library()
    _check_pair(k_cache, v_cache)
    dev = k_cache.device
    desc = cache_desc(k_cache)
    _contig(q, torch.bfloat16, "q", dev)
    if q.dim() != 3 or q.shape[2] != desc.head_dim:
        raise ValueError("q must be [B, H_q, head_dim]")
    b, hq, d = q.shape
    _contig(block_tables, torch.int32, "block_tables", dev)
    _contig(context_lens, torch.int32, "context_lens", dev)
    if block_tables.dim() != 2 or block_tables.shape[0] != b or context_lens.shape != (b,):
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    if max_context_len is None:
        max_context_len = block_tables.shape[1] * desc.block_size if b > 0 else 0
    if out is None:
        out = torch.empty((b, hq, d), dtype=torch.float32, device=dev)
    else:
        _contig(out, torch.float32, "out", dev)
        if out.shape != (b, hq, d):
            raise ValueError("out must be [B, H_q, D]")
    stride = 0
    if desc.dtype == PKV_E4M3:
        if k_scale is None or v_scale is None:
            raise ValueError("E4M3 cache needs k_scale and v_scale")
        _contig(k_scale, torch.float32, "k_scale", dev)
        _contig(v_scale, torch.float32, "v_scale", dev)
        stride = scale_row_stride if scale_row_stride is not None else (
            desc.num_kv_heads if k_scale.dim() == 2 else 0)
    mb = block_tables.shape[1] if b > 0 else 1
    # planned for this device's SMs, as the library plans the call itself
    plan = decode_plan(b, hq, desc, max_context_len, split_tokens,
                       torch.cuda.get_device_properties(dev).multi_processor_count)
    ws_bytes = int(plan.workspace_bytes)
    if ws_bytes > 0 and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if k_new is not None or v_new is not None:
        if k_new is None or v_new is None or k_new.shape != v_new.shape:
            raise ValueError("k_new and v_new go together, both [B, H_kv, D]")
        if tuple(k_new.shape) != (b, desc.num_kv_heads, desc.head_dim):
            raise ValueError("k_new / v_new must be [B, H_kv, D]")
        if k_new.dtype == torch.bfloat16:
            src = PKV_BF16
        elif k_new.dtype == torch.float32:
            src = PKV_F32
        else:
            raise TypeError(f"k_new dtype {k_new.dtype}: expected bfloat16 or float32")
        _contig(k_new, k_new.dtype, "k_new", dev)
        _contig(v_new, k_new.dtype, "v_new", dev)
        st = lib.pkv_decode_attention_append(
            _ptr(q), b, hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(k_new), _ptr(v_new), src,
            _ptr(block_tables), mb, _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
            _ptr(k_scale), _ptr(v_scale), int(stride), _ptr(workspace) if ws_bytes > 0 else ctypes.c_void_p(0),
            ws_bytes if ws_bytes > 0 else 0, int(split_tokens), _stream(dev))
        _lib.check(st, "pkv_decode_attention_append")
        return out
    st = lib.pkv_decode_attention_ex(
        _ptr(q), b, hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(block_tables), mb,
        _ptr(context_lens), int(max_context_len), float(scale), _ptr(out), _ptr(k_scale),
        _ptr(v_scale), int(stride), _ptr(workspace) if ws_bytes > 0 else ctypes.c_void_p(0),
        ws_bytes if ws_bytes > 0 else 0, int(split_tokens), _stream(dev))
    _lib.check(st, "pkv_decode_attention_ex")
    return out


def decode_attention_pooled(q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
                            out, k_scale=None, v_scale=None, scale_row_stride=None):
    """The plain C entry point (library-owned scratch pool), same arguments."""
    lib = library()
    desc = cache_desc(k_cache)
    b, hq, _ = q.shape
    stride = 0
    if desc.dtype == PKV_E4M3:
        stride = scale_row_stride if scale_row_stride is not None else (
            desc.num_kv_heads if k_scale.dim() == 2 else 0)
    st = lib.pkv_decode_attention(
        _ptr(q), b, hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
        _ptr(k_scale), _ptr(v_scale), int(stride), _stream(k_cache.device))
    _lib.check(st, "pkv_decode_attention")
    return out


def cascade_plan(batch, num_q_heads, k_cache_or_desc, prefix_len, max_context_len, num_sms=0):
    """Plan of a cascade decode (host only)."""
    lib = library()
    desc = k_cache_or_desc if isinstance(k_cache_or_desc, CacheDesc) else cache_desc(k_cache_or_desc)
    plan = DecodePlan()
    st = lib.pkv_cascade_plan(int(batch), int(num_q_heads), ctypes.byref(desc), int(prefix_len),
                              int(max_context_len), int(num_sms), ctypes.byref(plan))
    _lib.check(st, "pkv_cascade_plan")
    return plan


def cascade_decode_attention(q, k_cache, v_cache, prefix_blocks, prefix_len, block_tables, context_lens,
                             scale, max_context_len, out=None, workspace=None):
    """Decode attention for a batch that shares its first `prefix_len` tokens
    (physical blocks `prefix_blocks`, int32); same result as decode_attention."""
    lib = library()
    _check_pair(k_cache, v_cache)
    dev = k_cache.device
    desc = cache_desc(k_cache)
    _contig(q, torch.bfloat16, "q", dev)
    _contig(prefix_blocks, torch.int32, "prefix_blocks", dev)
    _contig(block_tables, torch.int32, "block_tables", dev)
    _contig(context_lens, torch.int32, "context_lens", dev)
    b, hq, d = q.shape
    if out is None:
        out = torch.empty((b, hq, d), dtype=torch.float32, device=dev)
    # planned for this device's SMs, as the library plans the call itself
    plan = cascade_plan(b, hq, desc, prefix_len, max_context_len,
                        torch.cuda.get_device_properties(dev).multi_processor_count)
    if workspace is None:
        workspace = torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=dev)
    st = lib.pkv_cascade_decode_attention(
        _ptr(q), b, hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(prefix_blocks),
        int(prefix_len), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        int(max_context_len), float(scale), _ptr(out), _ptr(workspace), int(workspace.numel()),
        _stream(dev))
    _lib.check(st, "pkv_cascade_decode_attention")
    return out


def multi_query_plan(batch, q_len, num_q_heads, k_cache_or_desc, max_context_len, split_tokens=0,
                     num_sms=0):
    desc = k_cache_or_desc if isinstance(k_cache_or_desc, CacheDesc) else cache_desc(k_cache_or_desc)
    plan = DecodePlan()
    _lib.check(library().pkv_multi_query_plan(batch, q_len, num_q_heads, ctypes.byref(desc), max_context_len,
                                              split_tokens, num_sms, ctypes.byref(plan)),
               "pkv_multi_query_plan")
    return plan


def multi_query_attention(q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
                          split_tokens=0, out=None, workspace=None):
    """q_len new tokens per sequence attending causally: q [B, q_len, H_q, D]
    bf16, context_lens counting the new tokens; returns out [B, q_len, H_q, D]
    float32."""
    _check_pair(k_cache, v_cache)
    dev = k_cache.device
    if q.dim() != 4:
        raise ValueError("q must be [B, q_len, H_q, D]")
    B, ql, hq, d = q.shape
    _contig(q, torch.bfloat16, "q", dev)
    _contig(block_tables, torch.int32, "block_tables", dev)
    _contig(context_lens, torch.int32, "context_lens", dev)
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    desc = cache_desc(k_cache)
    if out is None:
        out = torch.empty((B, ql, hq, d), dtype=torch.float32, device=dev)
    _contig(out, torch.float32, "out", dev)
    with torch.cuda.device(dev):
        plan = multi_query_plan(B, ql, hq, desc, int(max_context_len), split_tokens,
                                torch.cuda.get_device_properties(dev).multi_processor_count)
        if plan.workspace_bytes > 0 and (workspace is None or workspace.numel() < plan.workspace_bytes):
            workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
        _lib.check(library().pkv_multi_query_attention(
            _ptr(q), B, ql, hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(block_tables),
            block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
            _ptr(workspace), workspace.numel() if workspace is not None else 0, split_tokens,
            _stream(dev)), "pkv_multi_query_attention")
    return out


def slot_mapping(block_tables, positions, k_cache, seq_index=None, out=None):
    """Flat cache slots (int64, on the cache's device) of new tokens at logical
    `positions` (int64; < 0 = padding, slot -1) of sequences `seq_index`
    (int64, or None: token i belongs to sequence i), computed by the library's
    kernel from `block_tables` (int32 [num_seqs, MB]); the slot_mapping that
    `append` takes."""
    dev = k_cache.device
    desc = cache_desc(k_cache)
    _contig(block_tables, torch.int32, "block_tables", dev)
    _contig(positions, torch.int64, "positions", dev)
    if block_tables.dim() != 2 or positions.dim() != 1:
        raise ValueError("block_tables must be [num_seqs, MB] and positions 1-D")
    n = positions.numel()
    if seq_index is not None:
        _contig(seq_index, torch.int64, "seq_index", dev)
        if seq_index.shape != positions.shape:
            raise ValueError("seq_index and positions differ in shape")
    if out is None:
        out = torch.empty(n, dtype=torch.int64, device=dev)
    else:
        _contig(out, torch.int64, "out", dev)
        if out.numel() != n:
            raise ValueError("out must have one entry per position")
    with torch.cuda.device(dev):
        _lib.check(library().pkv_slot_mapping(
            _ptr(block_tables), block_tables.shape[0], max(1, block_tables.shape[1]), _ptr(seq_index),
            _ptr(positions), n, ctypes.byref(desc), _ptr(out), _stream(dev)), "pkv_slot_mapping")
    return out


def device_error(device=None):
    """Read and clear the device error word (synchronises the current stream)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        return library().pkv_get_device_error(_stream(dev))


def selftest_wait_timeout(which, limit_us=20000, device=None):
    """Run the device-side bounded-wait self-test (include/pkv.h); returns the
    device error word read afterwards (1 = PKV_DEVERR_WAIT_TIMEOUT)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _lib.check(library().pkv_selftest_wait_timeout(int(which), int(limit_us), _stream(dev)),
                   "pkv_selftest_wait_timeout")
    return device_error(dev)


def trace_enable(on=True):
    _lib.check(library().pkv_trace_enable(1 if on else 0), "pkv_trace_enable")


def trace_read():
    """{kernel name: (launches, total_ms)} since the last read; clears the trace."""
    buf = (TraceEntry * 8)()
    n = library().pkv_trace_read(buf, 8)
    if n < 0:
        raise RuntimeError("pkv_trace_read failed")
    return {KERNEL_KINDS[buf[i].kind]: (buf[i].launches, buf[i].total_ms) for i in range(n)}


# ---------------------------------------------------------------- block manager

class OutOfBlocks(PkvError):
    """The free pool cannot cover an append (PKV_ERR_OUT_OF_BLOCKS): preempt a
    sequence (free it or swap it out) and retry."""


def _bm_check(status, where):
    if status == _lib.PKV_ERR_OUT_OF_BLOCKS:
        raise OutOfBlocks(status, where)
    _lib.check(status, where)


def _np_ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a.size else ctypes.c_void_p(0)


class BlockManager:
    """Host block manager of one paged pool (include/pkv_blocks.h): free pool,
    reference counts, per-sequence tables, copy-on-write, all-or-nothing
    appends.  Host memory only; pair it with `copy_blocks` and `append`."""

    def __init__(self, num_blocks, block_size):
        h = ctypes.c_void_p()
        _bm_check(library().pkv_bm_create(int(num_blocks), int(block_size), ctypes.byref(h)),
                  "pkv_bm_create")
        self._h = h
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self):
        if self._h:
            library().pkv_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self):
        return library().pkv_bm_num_free(self._h)

    def num_sequences(self):
        return library().pkv_bm_num_sequences(self._h)

    def ref_count(self, block):
        return library().pkv_bm_ref_count(self._h, int(block))

    def seq_len(self, seq_id):
        return library().pkv_bm_seq_len(self._h, int(seq_id))

    def add_sequence(self, seq_id):
        _bm_check(library().pkv_bm_add_sequence(self._h, int(seq_id)), "pkv_bm_add_sequence")

    def fork(self, parent_id, child_id):
        _bm_check(library().pkv_bm_fork(self._h, int(parent_id), int(child_id)), "pkv_bm_fork")

    def free_sequence(self, seq_id):
        _bm_check(library().pkv_bm_free_sequence(self._h, int(seq_id)), "pkv_bm_free_sequence")

    def blocks_needed(self, seq_ids, n_new):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = np.ascontiguousarray(n_new, dtype=np.int32)
        out = ctypes.c_int64()
        _bm_check(library().pkv_bm_blocks_needed(self._h, len(ids), _np_ptr(ids), _np_ptr(n),
                                                 ctypes.byref(out)), "pkv_bm_blocks_needed")
        return out.value

    def append(self, seq_ids, n_new):
        """Reserve slots; returns (slots int64 [sum n_new], cow_pairs int32 [k, 2])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = np.ascontiguousarray(n_new, dtype=np.int32)
        if ids.shape != n.shape:
            raise ValueError("seq_ids and n_new differ in length")
        slots = np.empty(int(np.maximum(n, 0).sum()), dtype=np.int64)
        src = np.empty(max(len(ids), 1), dtype=np.int32)
        dst = np.empty(max(len(ids), 1), dtype=np.int32)
        nc = ctypes.c_int32()
        _bm_check(library().pkv_bm_append(self._h, len(ids), _np_ptr(ids), _np_ptr(n), _np_ptr(slots),
                                          _np_ptr(src), _np_ptr(dst), len(ids), ctypes.byref(nc)),
                  "pkv_bm_append")
        return slots, np.stack([src[:nc.value], dst[:nc.value]], axis=1)

    # ---- host tier
    def set_host_blocks(self, num_host_blocks):
        _bm_check(library().pkv_bm_set_host_blocks(self._h, int(num_host_blocks)), "pkv_bm_set_host_blocks")

    def num_free_host(self):
        return library().pkv_bm_num_free_host(self._h)

    def host_entries(self, seq_id):
        return library().pkv_bm_host_entries(self._h, int(seq_id))

    def table_entries(self, seq_id):
        """(ids int32 [n], on_host int32 [n]) of a sequence's table."""
        cap = max(self.num_blocks, 1) + 1
        ids = np.empty(cap, dtype=np.int32)
        host = np.empty(cap, dtype=np.int32)
        n = ctypes.c_int32()
        _bm_check(library().pkv_bm_table_entries(self._h, int(seq_id), cap, _np_ptr(ids), _np_ptr(host),
                                                 ctypes.byref(n)), "pkv_bm_table_entries")
        return ids[:n.value].copy(), host[:n.value].copy()

    def _move(self, fn, name, seq_id, logical):
        lg = np.ascontiguousarray(logical, dtype=np.int32)
        a = np.empty(max(len(lg), 1), dtype=np.int32)
        b = np.empty(max(len(lg), 1), dtype=np.int32)
        n = ctypes.c_int32()
        _bm_check(fn(self._h, int(seq_id), len(lg), _np_ptr(lg), _np_ptr(a), _np_ptr(b), ctypes.byref(n)), name)
        return np.stack([a[:n.value], b[:n.value]], axis=1)

    def evict(self, seq_id, logical):
        """Demote table entries to the host pool; returns (device, host) pairs [k, 2]."""
        return self._move(library().pkv_bm_evict, "pkv_bm_evict", seq_id, logical)

    def stage(self, seq_id, logical):
        """Promote table entries to the device pool; returns (host, device) pairs [k, 2]."""
        return self._move(library().pkv_bm_stage, "pkv_bm_stage", seq_id, logical)

    def swap_out(self, seq_id):
        return self.evict(seq_id, np.arange(len(self.table_entries(seq_id)[0])))

    def swap_in(self, seq_id):
        return self.stage(seq_id, np.arange(len(self.table_entries(seq_id)[0])))

    def prefetch_candidates(self, seq_id, activation, threshold, capacity=None):
        """Host entries to stage ahead: activation > threshold, most probable
        first, at most `capacity` and the free device blocks."""
        act = np.ascontiguousarray(activation, dtype=np.float32)
        cap = len(act) if capacity is None else int(capacity)
        out = np.empty(max(cap, 1), dtype=np.int32)
        n = ctypes.c_int32()
        _bm_check(library().pkv_bm_prefetch_candidates(self._h, int(seq_id), _np_ptr(act), float(threshold), cap,
                                                       _np_ptr(out), ctypes.byref(n)), "pkv_bm_prefetch_candidates")
        return out[:n.value].copy()

    def block_tables(self, seq_ids, max_blocks_per_seq):
        """(block_tables int32 [n, max_blocks_per_seq] with -1 past each table, lens int32 [n])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tbl = np.empty((len(ids), int(max_blocks_per_seq)), dtype=np.int32)
        lens = np.empty(len(ids), dtype=np.int32)
        _bm_check(library().pkv_bm_block_tables(self._h, len(ids), _np_ptr(ids), int(max_blocks_per_seq),
                                                _np_ptr(tbl), _np_ptr(lens)), "pkv_bm_block_tables")
        return tbl, lens


def copy_blocks(k_cache, v_cache, src_blocks, dst_blocks):
    """Device copy-on-write step: block dst[i] := block src[i] in both caches.
    src/dst: int32 CUDA tensors (or host sequences, copied to the device)."""
    _check_pair(k_cache, v_cache)
    dev = k_cache.device
    src = torch.as_tensor(src_blocks, dtype=torch.int32).to(dev).contiguous()
    dst = torch.as_tensor(dst_blocks, dtype=torch.int32).to(dev).contiguous()
    if src.shape != dst.shape or src.dim() != 1:
        raise ValueError("src_blocks and dst_blocks must be 1-D of equal length")
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        _lib.check(library().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(src),
                                             _ptr(dst), src.numel(), _stream(dev)), "pkv_copy_blocks")


def host_pool_like(k_cache, num_blocks):
    """(k, v) block pools in page-locked host memory with the block geometry
    and dtype of `k_cache`; the GPU addresses them directly."""
    shape = (int(num_blocks),) + tuple(k_cache.shape[1:])
    k = torch.empty(shape, dtype=k_cache.dtype, pin_memory=True)
    v = torch.empty(shape, dtype=k_cache.dtype, pin_memory=True)
    return k, v


def copy_blocks_between(src_k, src_v, dst_k, dst_v, src_blocks, dst_blocks, max_ctas=0,
                        stream_device=None):
    """Block dst_blocks[i] of (dst_k, dst_v) := block src_blocks[i] of (src_k, src_v),
    through one kernel on the current stream; the pools may live in device or
    pinned host memory.  max_ctas bounds the SMs the copy occupies (0: no bound)."""
    if src_k.shape[1:] != dst_k.shape[1:] or src_k.dtype != dst_k.dtype:
        raise ValueError("pools differ in block geometry or dtype")
    for t in (src_k, src_v, dst_k, dst_v):
        if not t.is_contiguous() or (t.device.type == "cpu" and not t.is_pinned()):
            raise ValueError("pools must be contiguous, and pinned when in host memory")
    dev = stream_device or next(t.device for t in (src_k, dst_k) if t.device.type == "cuda")
    src = torch.as_tensor(src_blocks, dtype=torch.int32).to(dev).contiguous()
    dst = torch.as_tensor(dst_blocks, dtype=torch.int32).to(dev).contiguous()
    desc = cache_desc(src_k)
    with torch.cuda.device(dev):
        _lib.check(library().pkv_copy_blocks_between(
            _ptr(src_k), _ptr(src_v), src_k.shape[0], _ptr(dst_k), _ptr(dst_v), dst_k.shape[0],
            ctypes.byref(desc), _ptr(src), _ptr(dst), src.numel(), int(max_ctas), _stream(dev)),
            "pkv_copy_blocks_between")
