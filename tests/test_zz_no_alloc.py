"""The allocation-free decode entry point, called through the C ABI.

pkv_decode_attention_noalloc serves callers that must not allocate device
memory while they run attention (for example a serving loop that reserved all
of its memory at start-up, or a runtime whose memory belongs to another
allocator).  It keeps its split-KV scratch in a fixed array owned by the
library.  These tests check that it gives the same result as the entry point
that takes caller memory, on two calls in a row that both use the scratch
(the second must not be disturbed by what the first left there), and that a
call needing more scratch than the array holds is refused before any launch.

This file is collected last on purpose: the tests run after every other test
as well as alone in a fresh process.
"""

import ctypes

import pytest
import torch

import paged_kv_cache_222_gb300 as pkv
import workloads as W
from paged_kv_cache_222_gb300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL_BF16 = 2e-3          # decode tolerance for bf16 KV used across the tests


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_222_gb300 import build
    build.build()
    return pkv.library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, case, bt, lens, max_len, out):
    desc = pkv.cache_desc(case["k_cache"])
    q = case["q"][0]
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return lib.pkv_decode_attention_noalloc(
        _p(q), q.shape[0], q.shape[1], _p(case["k_cache"]), _p(case["v_cache"]), ctypes.byref(desc),
        _p(bt), bt.shape[1], _p(lens), int(max_len), float(case["scale"]), _p(out),
        ctypes.c_void_p(0), ctypes.c_void_p(0), 0, stream)


def test_noalloc_matches_caller_workspace_entry_point_on_two_calls(lib):
    torch.cuda.set_device(DEV)
    for seed, ctx in ((101, (3000, 1200, 4000)), (202, (700, 2900, 64))):
        spec = dict(B=3, H_q=16, H_kv=2, D=128, bs=16, kv="bf16", free_frac=0.1, steps=1,
                    seed=seed, ctx=ctx)
        case = W.make_case(spec, device=DEV)
        bt = case["block_tables"].to(DEV)
        lens = (case["ctx"] + 1).to(DEV)
        max_len = int(lens.max())
        plan = pkv.decode_plan(3, 16, case["k_cache"], max_len)
        assert plan.workspace_bytes > 0                           # the scratch is really used
        ref = pkv.decode_attention(case["q"][0], case["k_cache"], case["v_cache"], bt, lens,
                                   case["scale"], max_context_len=max_len)
        out = torch.full_like(ref, float("nan"))
        torch.cuda.synchronize()
        free_before, _ = torch.cuda.mem_get_info(DEV)
        st = _noalloc(lib, case, bt, lens, max_len, out)
        assert st == L.PKV_OK, lib.pkv_last_error()
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info(DEV)
        assert free_after == free_before                          # the call took no device memory
        assert torch.all(torch.isfinite(out))
        assert float((out - ref).abs().max()) <= TOL_BF16
    assert pkv.device_error(DEV) == 0


def test_noalloc_refuses_more_scratch_than_it_has(lib):
    """A decode whose split-KV plan needs more than the 32 MiB array is
    refused before anything is launched.  The arguments are real device
    buffers that a launch could read safely (a one-block cache, an all-zero
    table, one token per sequence), so that if the refusal ever stopped
    happening the call would still only touch valid memory and the test
    would fail on the status, not on the GPU."""
    torch.cuda.set_device(DEV)
    # 114 x 8 units = two waves of three CTAs on each of 152 SMs, so no split
    # count leaves a half-full last wave and the planner keeps 16 splits
    B, H_q, H_kv, D, bs, mb = 114, 64, 8, 128, 16, 4096
    kc = torch.zeros((1, H_kv, bs, D), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    q = torch.zeros((B, H_q, D), dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros((B, mb), dtype=torch.int32, device=DEV)
    lens = torch.ones(B, dtype=torch.int32, device=DEV)
    out = torch.empty((B, H_q, D), dtype=torch.float32, device=DEV)
    desc = pkv.cache_desc(kc)
    plan = pkv.decode_plan(B, H_q, desc, 65536)            # 16 splits of 4096 tokens
    assert plan.workspace_bytes > (32 << 20)
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    st = lib.pkv_decode_attention_noalloc(_p(q), B, H_q, _p(kc), _p(vc), ctypes.byref(desc), _p(bt), mb,
                                          _p(lens), 65536, 0.088, _p(out), ctypes.c_void_p(0),
                                          ctypes.c_void_p(0), 0, stream)
    assert st == L.PKV_ERR_WORKSPACE
    assert b"no-allocation" in lib.pkv_last_error()
    torch.cuda.synchronize()
    assert pkv.device_error(DEV) == 0


def test_noalloc_after_shutdown_looks_the_array_up_again(lib):
    """pkv_shutdown forgets the array's device address (a caller may reset
    the device after it); the next call looks it up again and gives the same
    result as before."""
    torch.cuda.set_device(DEV)
    spec = dict(B=3, H_q=16, H_kv=2, D=128, bs=16, kv="bf16", free_frac=0.1, steps=1, seed=303,
                ctx=(2500, 900, 3100))
    case = W.make_case(spec, device=DEV)
    bt = case["block_tables"].to(DEV)
    lens = (case["ctx"] + 1).to(DEV)
    max_len = int(lens.max())
    outs = []
    for i in range(2):
        out = torch.full((3, 16, 128), float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(lib, case, bt, lens, max_len, out) == L.PKV_OK, lib.pkv_last_error()
        torch.cuda.synchronize()
        outs.append(out.cpu())
        if i == 0:
            assert lib.pkv_shutdown() == L.PKV_OK
    assert torch.all(torch.isfinite(outs[0])) and torch.equal(outs[0], outs[1])
    assert pkv.device_error(DEV) == 0
