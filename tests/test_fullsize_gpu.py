"""Full-size parity: each workload at its full size, run the way the benchmark runs it (one
sdm_phase1 launch over every chunk, then one sdm_dw launch over every step), checked on samples
the oracle can compute: Phase-1 outputs of sampled chunks (first, last, ragged, random) and the
whole bank of one sampled stream after every step. The other streams' banks start from a seeded
device draw and are checked only for staying finite."""

import numpy as np
import pytest
import torch

import oracle
import sparse_slot_memory_gb300 as sdm
from oracle import bounds
from sdm_testlib import BankStats, compare_p1, host, inputs_to_dev
from synth import WORKLOADS, bf16_bits_to_f32, make_bank_stream, make_inputs

pytestmark = pytest.mark.gpu


def _stream_compact(w, x, p):
    P = x["P"]
    cs = [ti * P + p for ti in range(w.steps)]
    kk, qq = x["k_idx"][cs], x["q_idx"][cs]
    ids = np.concatenate([kk.ravel(), qq.ravel()])
    slots = np.unique(ids[(ids >= 0) & (ids < w.S)])

    def remap(a):
        r = np.searchsorted(slots, a)
        return np.where((a >= 0) & (a < w.S), r, a).astype(np.int32)

    xs = dict(x)
    xs["k_idx"], xs["q_idx"] = x["k_idx"].copy(), x["q_idx"].copy()
    xs["k_idx"][cs], xs["q_idx"][cs] = remap(kk), remap(qq)
    return slots, xs


@pytest.mark.parametrize("name", ["large", "uniform_c128", "zipf_c256", "wide_ragged"])
def test_fullsize_sampled_parity(name):
    w = WORKLOADS[name]
    x = make_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)
    d = inputs_to_dev(x, w)
    ws = sdm.alloc_workspace(shape)
    out = sdm.alloc_outputs(shape)
    P, S, hd = w.P, w.S, w.hd
    p_chk = P - 1
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    bank = (torch.randn(P * S, hd, device="cuda", generator=gen) * w.bank_scale).to(torch.bfloat16)
    init_p = bf16_bits_to_f32(make_bank_stream(w, p_chk))
    bank[p_chk * S:(p_chk + 1) * S] = torch.from_numpy(init_p).cuda().to(torch.bfloat16)

    sdm.phase1(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], out, ws)
    sdm.dw(shape, d["dv"], bank, ws)
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0

    # Phase 1 on sampled chunks
    N = w.N
    rng = np.random.default_rng(5)
    picks = sorted({0, N - 1, N - P, *rng.integers(0, N, size=3).tolist()})
    fp = (w.steps - 1) * P
    for c in picks:
        orc = oracle.phase1(x["k_idx"][c:c + 1], x["q_idx"][c:c + 1], x["k_val"][c:c + 1], x["q_val"][c:c + 1],
                            x["g"][c:c + 1], S=S, val_dtype=w.val_dtype, first_partial=0 if c >= fp else 1,
                            valid_last=w.valid_last)
        compare_p1({k: v[c:c + 1] for k, v in out.items() if k != "repeats"}, orc, 0, 1, w.val_dtype)

    # DW: the sampled stream's whole bank after every step, against the carried rounding intervals
    slots, xs = _stream_compact(w, x, p_chk)
    ref = init_p[slots].astype(np.float64)
    b = bounds.dw_stream_bounds(ref, xs, p_chk, S=len(slots), C=w.C, P=P, steps=w.steps, valid_last=w.valid_last,
                                val_dtype=w.val_dtype, dv_dtype=w.dv_dtype, bank_dtype=w.bank_dtype)
    got = host(bank[torch.from_numpy(p_chk * S + slots.astype(np.int64)).cuda()]).astype(np.float64)
    t = b["writes"] > 0
    assert np.array_equal(got[~t], init_p[slots][~t].astype(np.float64))
    last = {"y": b["y"][t], "lo": b["lo"][t], "hi": b["hi"][t], "relaxed": b["relaxed"][t]}
    r = bounds.check_rows(got[t], last, w.bank_dtype)
    assert r["ok"].all(), f"{name}: {int((~r['ok']).sum())} bank elements of stream {p_chk} outside their interval"
    once = b["writes"][t] == 1
    r1 = bounds.check_rows(got[t][once], {k: v[once] for k, v in last.items()}, w.bank_dtype)
    stats = BankStats(f"{name}_fullsize", "end_to_end", w.bank_dtype)
    stats.add(r, once=r1)
    stats.finish()
    others = np.setdiff1d(rng.integers(0, S, size=4096), slots)
    assert np.array_equal(host(bank[torch.from_numpy(p_chk * S + others.astype(np.int64)).cuda()]),
                          init_p[others].astype(np.float64))
    assert bool(torch.isfinite(bank.float()).all())
