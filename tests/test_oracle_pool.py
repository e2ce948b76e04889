"""The per-unit oracle harness (tests/oracle_pool.py) against the oracle run
on the whole pool: rebuilding one (sequence, KV head) unit with its blocks
renumbered, appending the new tokens and attending must give exactly the
result of appending into the full pool through the block tables and
attending there.  CPU only."""

import numpy as np
import torch

import workloads as W
from oracle import paged_attention as PA
from tests import oracle_pool as OP


def _whole_pool(case, n_new, q_steps):
    """Oracle on the full pool: fill (E4M3), append the first n_new tokens of
    every sequence through the tables, attend with queries q[q_steps]."""
    bt = case["block_tables"].numpy()
    ctx = case["ctx"].numpy().astype(np.int64)
    B, bs = case["B"], case["bs"]
    if case["kv"] == "bf16":
        kc = case["k_cache"].view(torch.int16).numpy().view(np.uint16)
        vc = case["v_cache"].view(torch.int16).numpy().view(np.uint16)
        dt, src, ks, vs = PA.BF16, PA.BF16, None, None
        kn = case["k_new"].view(torch.int16).numpy().view(np.uint16)
        vn = case["v_new"].view(torch.int16).numpy().view(np.uint16)
    else:
        dt, src = PA.E4M3, PA.F32
        kc = np.full(case["k_cache"].shape, 0x7F, dtype=np.uint8)
        vc = kc.copy()
        ks, vs = case["k_scale"].numpy(), case["v_scale"].numpy()
        seq, pos = case["fill_seq"].numpy(), case["fill_pos"].numpy()
        slots = np.array([PA.slot_of(bt[s], int(p), bs) for s, p in zip(seq, pos)])
        kc, vc = PA.append(case["fill_k"].numpy(), case["fill_v"].numpy(), src, slots, kc, vc, dt,
                           ks[seq], vs[seq], scale_row_stride=case["H_kv"])
        kn, vn = case["k_new"].numpy(), case["v_new"].numpy()
    for s in range(n_new):
        slots = np.array([PA.slot_of(bt[b], int(ctx[b]) + s, bs) for b in range(B)])
        kc, vc = PA.append(kn[s], vn[s], src, slots, kc, vc, dt, ks, vs,
                           scale_row_stride=0 if ks is None else case["H_kv"])
    q = case["q"].view(torch.int16).numpy().view(np.uint16)
    lens = ctx + n_new
    if len(q_steps) == 1:
        return PA.decode_attention(q[q_steps[0]], kc, vc, dt, bt, lens, case["scale"], ks, vs)
    qm = np.ascontiguousarray(q[q_steps].transpose(1, 0, 2, 3))
    return PA.multi_query_attention(qm, kc, vc, dt, bt, lens, case["scale"], ks, vs)


def _spec(kv, steps):
    return dict(B=3, ctx=(5, 40, 77), H_q=8, H_kv=2, D=64, bs=16, kv=kv, free_frac=0.3, steps=steps,
                seed=4711 + steps)


def test_units_equal_whole_pool_decode_bf16_and_e4m3():
    for kv in ("bf16", "e4m3"):
        case = W.make_case(_spec(kv, 3))
        src = OP.UnitSource(case)
        units = [(b, h) for b in range(3) for h in range(2)]
        for step in (0, 2):
            res = OP.run_units(src, units, step + 1, [step], procs=2, want_codes=True)
            want = _whole_pool(case, step + 1, [step])
            assert res["units"] == 6
            for (b, h), out in res["outputs"].items():
                assert np.array_equal(out, want[b, h * 4:(h + 1) * 4]), (kv, step, b, h)
            if kv == "e4m3":
                assert set(res["codes"]) == set(units)
                assert res["codes"][(1, 1)][0].shape == (40 + step + 1, 64)


def test_units_equal_whole_pool_multi_token():
    case = W.make_case(_spec("bf16", 4))
    src = OP.UnitSource(case)
    units = [(b, h) for b in range(3) for h in range(2)]
    res = OP.run_units(src, units, 4, [0, 1, 2, 3], procs=2)
    want = _whole_pool(case, 4, [0, 1, 2, 3])
    for (b, h), out in res["outputs"].items():
        assert np.array_equal(out, want[b, :, h * 4:(h + 1) * 4])
    got = np.nan_to_num(want)
    assert OP.max_abs_err(got, res["outputs"], 4, multi=True) == 0.0
