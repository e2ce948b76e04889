"""C-ABI library: loads, exports what include/*.h declare, and rejects bad
arguments on the host before touching the GPU (CPU only, no compute calls)."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

from paged_kv_cache_222_gb300 import build as B
from paged_kv_cache_222_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_documented_entry_points():
    names = _declared_functions()
    for n in ["pkv_append", "pkv_decode_attention", "pkv_decode_attention_ex", "pkv_decode_plan",
              "pkv_get_device_error", "pkv_status_string", "pkv_last_error", "pkv_abi_version",
              "pkv_trace_enable", "pkv_trace_read", "pkv_shutdown"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert set(_declared_functions()) <= set(L.SIGNATURES)


def test_status_strings_and_version(lib):
    assert lib.pkv_abi_version() == 102
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(1) == b"PKV_ERR_INVALID_ARG"
    assert lib.pkv_status_string(4) == b"PKV_ERR_WORKSPACE"
    assert lib.pkv_status_string(5) == b"PKV_ERR_OUT_OF_BLOCKS"
    assert lib.pkv_status_string(99) == b"PKV_ERR_UNKNOWN"


def _desc(**kw):
    d = dict(num_blocks=64, block_size=16, num_kv_heads=8, head_dim=128, dtype=L.PKV_BF16)
    d.update(kw)
    return L.CacheDesc(d["num_blocks"], d["block_size"], d["num_kv_heads"], d["head_dim"], d["dtype"])


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
NULL = ctypes.c_void_p(0)


def _decode(lib, desc, **kw):
    a = dict(q=FAKE, batch=2, hq=64, kc=FAKE, vc=FAKE, bt=FAKE, mb=8, cl=FAKE, max_ctx=100,
             scale=0.125, out=FAKE, ks=NULL, vs=NULL, stride=0, ws=NULL, ws_bytes=0, split=0)
    a.update(kw)
    return lib.pkv_decode_attention_ex(a["q"], a["batch"], a["hq"], a["kc"], a["vc"], ctypes.byref(desc),
                                       a["bt"], a["mb"], a["cl"], a["max_ctx"], a["scale"], a["out"],
                                       a["ks"], a["vs"], a["stride"], a["ws"], a["ws_bytes"], a["split"],
                                       NULL)


@pytest.mark.parametrize("kw,desc_kw,code", [
    (dict(hq=60), {}, L.PKV_ERR_INVALID_ARG),                 # not a multiple of H_kv
    (dict(hq=8 * 17), {}, L.PKV_ERR_UNSUPPORTED),             # group of 17
    (dict(batch=-1), {}, L.PKV_ERR_INVALID_ARG),
    (dict(batch=70000), {}, L.PKV_ERR_INVALID_ARG),
    (dict(max_ctx=8 * 16 + 1), {}, L.PKV_ERR_INVALID_ARG),     # beyond the table
    (dict(max_ctx=-5), {}, L.PKV_ERR_INVALID_ARG),
    (dict(mb=0), {}, L.PKV_ERR_INVALID_ARG),
    (dict(scale=float("nan")), {}, L.PKV_ERR_INVALID_ARG),
    (dict(q=NULL), {}, L.PKV_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p(0x10004)), {}, L.PKV_ERR_INVALID_ARG),   # misaligned
    (dict(kc=ctypes.c_void_p(0x10008)), {}, L.PKV_ERR_INVALID_ARG),
    (dict(ks=FAKE, vs=FAKE), {}, L.PKV_ERR_INVALID_ARG),       # scales on a bf16 cache
    (dict(), dict(dtype=L.PKV_E4M3), L.PKV_ERR_INVALID_ARG),    # E4M3 without scales
    (dict(), dict(dtype=L.PKV_F32), L.PKV_ERR_INVALID_ARG),     # f32 is not a cache dtype
    (dict(), dict(head_dim=96), L.PKV_ERR_UNSUPPORTED),
    (dict(), dict(block_size=8), L.PKV_ERR_UNSUPPORTED),
    (dict(), dict(num_blocks=0), L.PKV_ERR_INVALID_ARG),
    (dict(), dict(num_blocks=1 << 31), L.PKV_ERR_INVALID_ARG),
    (dict(split=100), {}, L.PKV_ERR_INVALID_ARG),              # not a multiple of 64
    (dict(split=-2), {}, L.PKV_ERR_INVALID_ARG),
    (dict(stride=-1, ks=FAKE, vs=FAKE), dict(dtype=L.PKV_E4M3), L.PKV_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, desc_kw, code):
    st = _decode(lib, _desc(**desc_kw), **kw)
    assert st == code, lib.pkv_last_error()
    assert lib.pkv_last_error()


def test_decode_with_empty_batch_is_a_noop(lib):
    assert _decode(lib, _desc(), batch=0, q=NULL, out=NULL) == L.PKV_OK


def _decode_append(lib, desc, **kw):
    a = dict(q=FAKE, batch=4, hq=64, kc=FAKE, vc=FAKE, kn=FAKE, vn=FAKE, src=L.PKV_BF16, bt=FAKE, mb=8,
             cl=FAKE, max_ctx=100, scale=0.125, out=FAKE, ks=NULL, vs=NULL, stride=0, ws=FAKE,
             ws_bytes=1 << 20, split=0)
    a.update(kw)
    return lib.pkv_decode_attention_append(a["q"], a["batch"], a["hq"], a["kc"], a["vc"], ctypes.byref(desc),
                                           a["kn"], a["vn"], a["src"], a["bt"], a["mb"], a["cl"],
                                           a["max_ctx"], a["scale"], a["out"], a["ks"], a["vs"], a["stride"],
                                           a["ws"], a["ws_bytes"], a["split"], NULL)


@pytest.mark.parametrize("kw,desc_kw,code", [
    (dict(src=L.PKV_E4M3), {}, L.PKV_ERR_INVALID_ARG),         # sources are bf16 or f32
    (dict(src=-1), {}, L.PKV_ERR_INVALID_ARG),
    (dict(kn=NULL), {}, L.PKV_ERR_INVALID_ARG),
    (dict(vn=ctypes.c_void_p(0x10008)), {}, L.PKV_ERR_INVALID_ARG),   # misaligned
    (dict(split=-1), {}, L.PKV_ERR_INVALID_ARG),              # the balanced mode has no fused append
    (dict(split=100), {}, L.PKV_ERR_INVALID_ARG),
    (dict(hq=60), {}, L.PKV_ERR_INVALID_ARG),                 # the decode checks apply too
    (dict(), dict(dtype=L.PKV_E4M3), L.PKV_ERR_INVALID_ARG),    # E4M3 without scales
])
def test_decode_append_rejects_bad_arguments_on_host(lib, kw, desc_kw, code):
    st = _decode_append(lib, _desc(**desc_kw), **kw)
    assert st == code, lib.pkv_last_error()
    assert lib.pkv_last_error()


def test_decode_append_with_empty_batch_is_a_noop(lib):
    assert _decode_append(lib, _desc(), batch=0, q=NULL, out=NULL) == L.PKV_OK


def _append(lib, desc, **kw):
    a = dict(k=FAKE, v=FAKE, src=L.PKV_BF16, n=4, slots=FAKE, kc=FAKE, vc=FAKE, ks=NULL, vs=NULL,
             stride=0)
    a.update(kw)
    return lib.pkv_append(a["k"], a["v"], a["src"], a["n"], a["slots"], a["kc"], a["vc"],
                          ctypes.byref(desc), a["ks"], a["vs"], a["stride"], NULL)


@pytest.mark.parametrize("kw,desc_kw,code", [
    (dict(src=L.PKV_E4M3), {}, L.PKV_ERR_INVALID_ARG),
    (dict(n=-1), {}, L.PKV_ERR_INVALID_ARG),
    (dict(k=NULL), {}, L.PKV_ERR_INVALID_ARG),
    (dict(slots=ctypes.c_void_p(0x10004)), {}, L.PKV_ERR_INVALID_ARG),
    (dict(v=ctypes.c_void_p(0x10002)), {}, L.PKV_ERR_INVALID_ARG),
    (dict(ks=FAKE, vs=FAKE), {}, L.PKV_ERR_INVALID_ARG),
    (dict(), dict(dtype=L.PKV_E4M3), L.PKV_ERR_INVALID_ARG),
    (dict(ks=FAKE, vs=FAKE, stride=-2), dict(dtype=L.PKV_E4M3), L.PKV_ERR_INVALID_ARG),
    (dict(), dict(head_dim=80), L.PKV_ERR_UNSUPPORTED),
])
def test_append_rejects_bad_arguments_on_host(lib, kw, desc_kw, code):
    assert _append(lib, _desc(**desc_kw), **kw) == code


def test_append_of_nothing_is_a_noop(lib):
    assert _append(lib, _desc(), n=0, k=NULL, v=NULL, slots=NULL, kc=NULL, vc=NULL) == L.PKV_OK


def _plan(lib, desc, batch, hq, max_ctx, split=0, sms=152):
    p = L.DecodePlan()
    st = lib.pkv_decode_plan(batch, hq, ctypes.byref(desc), max_ctx, split, sms, ctypes.byref(p))
    assert st == L.PKV_OK, lib.pkv_last_error()
    return p


def _auto_split(batch, hkv, max_ctx, sms=152):
    """The automatic split length, restated: one split per (sequence, KV head)
    when those give four waves of three CTAs per SM, else the largest power of
    two (256..4096) giving six waves, with a last split shorter than an
    eighth of the others folded into them; then, if that still splits, the
    fewest splits giving at least three waves with the last 40-70 % full."""
    units = batch * hkv
    if units >= 4 * 3 * sms:
        return max(64, -(-max_ctx // 64) * 64)
    st = 4096
    while st > 256 and units * -(-max_ctx // st) < sms * 3 * 6:
        st //= 2
    n = -(-max_ctx // st)
    if n >= 2 and max_ctx - (n - 1) * st < st // 8:
        st = -(-(-(-max_ctx // (n - 1))) // 64) * 64
    n = -(-max_ctx // st)
    if n > 1:           # >= 3 waves, the last 40-70 % full, fewest splits
        for s in range(2, n):
            w100 = units * s * 100 // (3 * sms)
            if w100 >= 300 and 40 <= w100 % 100 <= 70:
                st = -(-(-(-max_ctx // s)) // 64) * 64
                break
    return st


def test_fixed_split_plan_covers_the_context_and_sizes_the_workspace(lib):
    d = _desc()
    for batch, max_ctx, split in [(64, 8193, 1024), (256, 4097, 512), (8, 131104, 2048), (2, 101, 64),
                                  (1, 1, 256), (3000, 4097, 0), (64, 8193, 0), (256, 4097, 0),
                                  (8, 131092, 0), (8, 131104, 0), (3, 4001, 0), (128, 5121, 0)]:
        p = _plan(lib, d, batch, 64, max_ctx, split=split)
        assert p.mode == 1 and p.workers == 0
        assert p.split_tokens % 64 == 0 and p.split_tokens >= 64
        if split:
            assert p.split_tokens == split
        else:
            assert p.split_tokens == _auto_split(batch, 8, max_ctx), (batch, max_ctx, p.split_tokens)
        assert p.max_splits == -(-max_ctx // p.split_tokens)
        assert (p.max_splits - 1) * p.split_tokens < max_ctx <= p.max_splits * p.split_tokens
        rows = batch * 64 * p.max_splits
        if p.max_splits > 1:
            assert p.workspace_bytes >= rows * (128 + 2) * 4
        else:
            assert p.workspace_bytes == 0


def test_balanced_plan_on_request_up_to_2048_sequences(lib):
    for D, G, dtype in [(128, 8, L.PKV_E4M3), (64, 4, L.PKV_E4M3), (128, 16, L.PKV_BF16)]:
        d = _desc(dtype=dtype, head_dim=D, num_kv_heads=2)
        for batch, max_ctx in [(1, 1), (64, 8193), (2048, 4097), (8, 131104), (5, 0)]:
            p = _plan(lib, d, batch, 2 * G, max_ctx, split=-1, sms=152)
            assert p.mode == 0 and p.split_tokens == 0 and p.max_splits == 0
            assert p.workers > 0 and p.workers % 152 == 0
            gp = 16 if G > 8 else 8
            assert p.workspace_bytes >= 2 * p.workers * gp * (D + 2) * 4 + (batch + 1) * 4
        assert _plan(lib, d, 2049, 2 * G, 4097, split=-1).mode == 1     # larger batches: fixed
        assert _plan(lib, d, 64, 2 * G, 8193).mode == 1                  # default: fixed splits
    # the grid follows the SM count
    d8 = _desc(dtype=L.PKV_E4M3)
    assert _plan(lib, d8, 64, 64, 8193, split=-1, sms=100).workers * 152 == \
        _plan(lib, d8, 64, 64, 8193, split=-1, sms=152).workers * 100


def test_fixed_split_auto_size_gives_enough_ctas_for_long_contexts(lib):
    p = _plan(lib, _desc(), 3000, 64, 4097)
    assert p.mode == 1 and 3000 * 8 * p.max_splits >= 152 * 3 * 4
    # enough (sequence, KV head) units alone: one split, no scratch, no combine
    assert p.max_splits == 1 and p.workspace_bytes == 0
    p = _plan(lib, _desc(), 256, 64, 4097)                   # the FP8 workload's shape
    assert p.max_splits == 1 and p.workspace_bytes == 0
    # otherwise the fewest splits giving >= 3 waves with a half-full last wave
    # (the six-wave rule's 8 splits of 1088 tokens before it)
    p = _plan(lib, _desc(), 64, 64, 8193)
    assert p.max_splits == 4 and p.split_tokens == 2112
    p = _plan(lib, _desc(block_size=32), 128, 64, 5121)      # the shared-prefix batch
    assert p.max_splits == 2
    # long contexts: the fewest splits giving >= 3 waves with the last wave 40-70 % full
    for max_ctx in (131092, 131104, 131136):                 # the long-context workload's steps
        p = _plan(lib, _desc(), 8, 64, max_ctx)
        w100 = 8 * 8 * p.max_splits * 100 // (152 * 3)
        assert w100 >= 300 and 40 <= w100 % 100 <= 70, (max_ctx, p.max_splits)
        assert p.max_splits == 25


def test_workspace_too_small_is_reported(lib):
    d = _desc(num_blocks=100000)
    p = _plan(lib, d, 64, 64, 8193)
    assert p.workspace_bytes > 0
    st = _decode(lib, d, batch=64, mb=600, max_ctx=8193, ws=FAKE, ws_bytes=p.workspace_bytes - 1)
    # rejected before any CUDA call: the size check precedes kernel setup only
    # once the device is known, so without a GPU the CUDA query fails first
    assert st in (L.PKV_ERR_WORKSPACE, L.PKV_ERR_CUDA)


def _cplan(lib, desc, batch, hq, prefix, max_ctx, sms=152):
    p = L.DecodePlan()
    st = lib.pkv_cascade_plan(batch, hq, ctypes.byref(desc), prefix, max_ctx, sms, ctypes.byref(p))
    return st, p


def test_cascade_plan_shapes(lib):
    d = _desc(block_size=32)
    st, p = _cplan(lib, d, 128, 64, 4096, 5121)
    assert st == L.PKV_OK, lib.pkv_last_error()
    assert p.mode == 2 and p.workers >= 1 and p.prefix_split_tokens % 64 == 0
    assert p.workers * p.prefix_split_tokens >= 4096 > (p.workers - 1) * p.prefix_split_tokens
    assert p.max_splits == -(-(5121 - 4096) // p.split_tokens)
    slots = 128 * 64 * (p.max_splits + p.workers)
    assert p.workspace_bytes >= slots * (128 + 2) * 4
    # a small batch spreads the prefix over more ranges
    st2, p2 = _cplan(lib, d, 2, 64, 4096, 4200)
    assert st2 == L.PKV_OK and p2.workers > p.workers


def test_cascade_suffix_splits_sized_for_the_free_sms(lib):
    """The suffix decode runs beside the prefix CTAs (one per SM): its split
    length is the largest power of two (256..4096) that still gives two waves
    of three CTAs per SM on the SMs the prefix leaves free, if every suffix
    were as long as the longest."""
    d = _desc(block_size=32)

    def want(batch, max_suffix, free):
        st = 4096
        while st > 256 and batch * 8 * -(-max_suffix // st) < free * 3 * 2:
            st //= 2
        return st

    for batch, max_ctx in [(128, 4096 + 1025), (32, 4096 + 1025), (8, 4096 + 131072), (256, 4096 + 64)]:
        st, p = _cplan(lib, d, batch, 64, 4096, max_ctx)
        assert st == L.PKV_OK, lib.pkv_last_error()
        prefix_ctas = -(-batch * 8 // 256) * 8 * p.workers
        free = 152 - prefix_ctas if prefix_ctas < 152 - 38 else 38
        assert p.split_tokens == want(batch, max_ctx - 4096, free), (batch, p.split_tokens, p.workers)
    # the shared-prefix workload: two prefix ranges, each suffix whole
    st, p = _cplan(lib, d, 128, 64, 4096, 4096 + 1025)
    assert p.workers == 2 and p.max_splits == 1


@pytest.mark.parametrize("desc_kw,prefix,max_ctx,code", [
    (dict(block_size=32), 48, 100, L.PKV_ERR_INVALID_ARG),     # not whole blocks
    (dict(block_size=16), 0, 100, L.PKV_ERR_INVALID_ARG),
    (dict(block_size=16), 128, 100, L.PKV_ERR_INVALID_ARG),    # beyond the longest context
    (dict(dtype=L.PKV_E4M3), 64, 100, L.PKV_ERR_UNSUPPORTED),
])
def test_cascade_plan_rejects(lib, desc_kw, prefix, max_ctx, code):
    st, _ = _cplan(lib, _desc(**desc_kw), 4, 64, prefix, max_ctx)
    assert st == code


@pytest.mark.parametrize("kw,code", [
    (dict(n_pairs=-1), L.PKV_ERR_INVALID_ARG),
    (dict(src=None), L.PKV_ERR_INVALID_ARG),
    (dict(cache_ptr=8), L.PKV_ERR_INVALID_ARG),
    (dict(desc=dict(block_size=8)), L.PKV_ERR_UNSUPPORTED),
])
def test_copy_blocks_rejects_bad_arguments_on_host(lib, kw, code):
    desc = _desc(**kw.get("desc", {}))
    cp = ctypes.c_void_p(kw.get("cache_ptr", 256))
    src = None if "src" in kw else ctypes.c_void_p(1024)
    st = lib.pkv_copy_blocks(cp, cp, ctypes.byref(desc), src, ctypes.c_void_p(2048),
                             kw.get("n_pairs", 4), None)
    assert st == code


def test_copy_of_no_pairs_is_a_noop(lib):
    desc = _desc()
    assert lib.pkv_copy_blocks(None, None, ctypes.byref(desc), None, None, 0, None) == L.PKV_OK


def _mqplan(lib, desc, batch, q_len, hq, max_ctx, st=0, sms=152):
    p = L.DecodePlan()
    r = lib.pkv_multi_query_plan(batch, q_len, hq, ctypes.byref(desc), max_ctx, st, sms, ctypes.byref(p))
    return r, p


def test_multi_query_plan_shapes(lib):
    desc = _desc()
    r, p = _mqplan(lib, desc, 64, 2, 64, 8192)
    assert r == L.PKV_OK and p.mode == 3 and p.workers == 4          # 16 rows: four token lanes
    assert p.split_tokens % 64 == 0 and p.max_splits == -(-8192 // p.split_tokens)
    n = 64 * 2 * 64 * p.max_splits
    assert p.workspace_bytes == -(-n * 128 * 4 // 256) * 256 + n * 8
    r, p = _mqplan(lib, desc, 64, 4, 64, 8192)               # 32 rows: the tcgen05 kernel, whose
    assert r == L.PKV_OK and p.workers == 0                  # splits are the longest (1024 blocks)
    assert p.split_tokens == 16 * 1024 and p.max_splits == 1  # that leave 3 units per SM
    r, p = _mqplan(lib, desc, 1, 16, 64, 131072)
    assert r == L.PKV_OK and p.workers == 0 and 8 * p.max_splits >= 3 * 152 > 8 * (-(-131072 // (2 * p.split_tokens)))
    r, p = _mqplan(lib, desc, 2, 16, 64, 100, st=128)     # 128 rows: the tcgen05 kernel
    assert r == L.PKV_OK and p.workers == 0 and p.max_splits == 1
    assert p.workspace_bytes == 256 + 256                   # work-unit counter, unit order (16 units)
    r, p = _mqplan(lib, desc, 3, 16, 64, 1000, st=128)    # with partials: counter and order after them
    n = 3 * 16 * 64 * p.max_splits
    units = p.max_splits * 3 * 8
    part = -(-(-(-n * 128 * 4 // 256) * 256 + n * 8) // 256) * 256
    assert p.max_splits == 8 and p.workspace_bytes == part + 256 + -(-units * 4 // 256) * 256
    r, p = _mqplan(lib, desc, 2, 8, 64, 100)                # 64 rows: the tcgen05 kernel
    assert r == L.PKV_OK and p.workers == 0
    r, p = _mqplan(lib, desc, 2, 1, 128, 100)               # 16 rows: mma.sync
    assert r == L.PKV_OK and p.workers == 4
    r, p = _mqplan(lib, desc, 2, 2, 72, 100)                # 18 rows: the tcgen05 kernel
    assert r == L.PKV_OK and p.workers == 0
    r, p = _mqplan(lib, desc, 2, 2, 64, 100)
    assert r == L.PKV_OK and p.workers == 4
    # long contexts on the mma.sync kernel: the decode planner's long-context
    # rule (>= 3 waves of three CTAs per SM, the last 40-70 % full)
    r, p = _mqplan(lib, _desc(block_size=32), 8, 2, 64, 131074)
    assert r == L.PKV_OK and p.workers == 4 and p.max_splits == 25
    w100 = 8 * 8 * p.max_splits * 100 // (3 * 152)
    assert w100 >= 300 and 40 <= w100 % 100 <= 70


@pytest.mark.parametrize("kw,code", [
    (dict(q_len=0), L.PKV_ERR_UNSUPPORTED),
    (dict(q_len=17), L.PKV_ERR_UNSUPPORTED),
    (dict(st=100), L.PKV_ERR_INVALID_ARG),
    (dict(st=16 * 1024 + 64), L.PKV_ERR_INVALID_ARG),
    (dict(max_ctx=-1), L.PKV_ERR_INVALID_ARG),
    (dict(desc=dict(dtype=L.PKV_E4M3)), L.PKV_ERR_UNSUPPORTED),
    (dict(hq=60), L.PKV_ERR_INVALID_ARG),
])
def test_multi_query_plan_rejects(lib, kw, code):
    desc = _desc(**kw.get("desc", {}))
    r, _ = _mqplan(lib, desc, 4, kw.get("q_len", 4), kw.get("hq", 64), kw.get("max_ctx", 1000),
                   st=kw.get("st", 0))
    assert r == code


@pytest.mark.parametrize("kw,code", [
    (dict(n_pairs=-1), L.PKV_ERR_INVALID_ARG),
    (dict(max_ctas=-1), L.PKV_ERR_INVALID_ARG),
    (dict(src_nb=0), L.PKV_ERR_INVALID_ARG),
    (dict(dst_ptr=8), L.PKV_ERR_INVALID_ARG),
    (dict(desc=dict(head_dim=96)), L.PKV_ERR_UNSUPPORTED),
])
def test_copy_between_pools_rejects_bad_arguments_on_host(lib, kw, code):
    desc = _desc(**kw.get("desc", {}))
    sp = ctypes.c_void_p(256)
    dp = ctypes.c_void_p(kw.get("dst_ptr", 512))
    st = lib.pkv_copy_blocks_between(sp, sp, kw.get("src_nb", 4), dp, dp, 4, ctypes.byref(desc),
                                     ctypes.c_void_p(1024), ctypes.c_void_p(2048), kw.get("n_pairs", 2),
                                     kw.get("max_ctas", 0), None)
    assert st == code


def test_wait_selftest_rejects_bad_arguments_before_any_launch(lib):
    assert lib.pkv_selftest_wait_timeout(2, 1000, None) == L.PKV_ERR_INVALID_ARG
    assert lib.pkv_selftest_wait_timeout(0, 0, None) == L.PKV_ERR_INVALID_ARG
    assert lib.pkv_selftest_wait_timeout(1, 1000001, None) == L.PKV_ERR_INVALID_ARG
