"""The bank rounding intervals (oracle/bounds.py) against what they claim, on the CPU.

* round_to agrees with the oracle C code's own bfloat16 rounding and with a neighbour search;
* a float32 evaluation of the DW update, emulated here step by step in the order the kernels take
  (sc = k * expf(rex) rounded, an fma chain over the group's write entries in sorted order, then
  fma(base, cpe, acc), rounded to the bank type), always lands inside the interval, over many steps
  with the carried bound;
* the intervals are tight: with no carry almost every element's interval holds only y's two
  bank-type neighbours (within 1 ulp of the exact y);
* a planted mistake in the emulation (the cpe dropped for one step) leaves the interval.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import bounds
from synth import WORKLOADS, bf16_bits_to_f32, make_bank_stream, make_inputs, scaled


def test_round_to_matches_a_neighbour_search():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                        [0.0, 1.0, -1.0, 1.00390625, 1.005859375, 2.0 ** -130, -(2.0 ** -133) * 1.5]])
    r = bounds.round_to(x, "bf16")
    for xi, ri in zip(x, r):
        if xi == 0.0:
            assert ri == 0.0
            continue
        e = math.floor(math.log2(abs(xi)))
        step = 2.0 ** max(e - 7, -133)
        lo = math.floor(xi / step) * step
        cands = [lo, lo + step]
        best = min(cands, key=lambda c: (abs(c - xi), int(round(c / step)) & 1))
        assert ri == best, (xi, ri, best)
    assert np.array_equal(bounds.round_to(x, "f32"), x.astype(np.float32).astype(np.float64))


def _f32(x):
    return np.float64(np.float32(x))


def _emulate_step(bank32, x, c, C, S, hd, V, val_dtype, dv_dtype, bank_dtype, drop_cpe=False):
    """A float32 DW step, emulated: per slot group in sorted order (slot, then token, then lane)."""
    kv = oracle.as_f64(x["k_val"][c], val_dtype)
    dv = oracle.as_f64(x["dv"][c * C:(c + 1) * C], dv_dtype)
    ki, g = x["k_idx"][c], x["g"][c]
    o = oracle.phase1(ki[None], x["q_idx"][c][None], x["k_val"][c][None], x["q_val"][c][None], g[None], S=S,
                      val_dtype=val_dtype, first_partial=0, valid_last=V, pairs=False)
    rex32 = o["rex"][0].astype(np.float32)
    cpe = o["cpe"][0]
    cpe = bounds.round_to(cpe, "bf16") if val_dtype == "bf16" else cpe.astype(np.float32).astype(np.float64)
    for s in np.unique(ki[:V]):
        members = [(t, a) for t in range(V) for a in range(ki.shape[1]) if ki[t, a] == s]
        acc = np.zeros(hd)
        for (t, a) in members:
            sc = _f32(_f32(kv[t, a]) * _f32(np.exp(np.float64(rex32[t, a]))))
            acc = (sc * dv[t] + acc).astype(np.float32).astype(np.float64)
        cp = 1.0 if drop_cpe else cpe[members[-1]]
        new = (bank32[s] * cp + acc).astype(np.float32).astype(np.float64)
        bank32[s] = bounds.round_to(new, bank_dtype)


@pytest.mark.parametrize("name", ["bf16", "f32"])
def test_float32_evaluation_lies_in_the_intervals(name):
    base = WORKLOADS["uniform_c128"] if name == "bf16" else WORKLOADS["tiny"]
    w = scaled(base, P=1, T=10 * 32, C=32, S=24, hd=8, W=4, R=2, name=f"bounds_{name}")
    x = make_inputs(w)
    init = make_bank_stream(w, 0)
    init = bf16_bits_to_f32(init).astype(np.float64) if w.bank_dtype == "bf16" else init.astype(np.float64)
    bank = init.copy()
    emu = init.copy()
    carry = np.zeros_like(bank)
    tot = {"over_1ulp_unrelaxed": 0, "elements": 0, "relaxed": 0}
    max_rel = 0.0
    for ti in range(w.steps):
        c = ti
        V = w.valid_last if ti == w.steps - 1 else w.C
        dv = oracle.as_f64(x["dv"][c * w.C:(c + 1) * w.C], w.dv_dtype)
        st = bounds.dw_step(bank, carry, x["k_idx"][c], x["q_idx"][c], x["k_val"][c], x["q_val"][c], x["g"][c], dv,
                            S=w.S, V=V, val_dtype=w.val_dtype, bank_dtype=w.bank_dtype)
        _emulate_step(emu, x, c, w.C, w.S, w.hd, V, w.val_dtype, w.dv_dtype, w.bank_dtype)
        r = bounds.check_rows(emu[st["rows"]], st, w.bank_dtype)
        assert r["ok"].all(), f"step {ti}: the emulated float32 rows leave the interval"
        for k in tot:
            tot[k] += r[k]
        max_rel = max(max_rel, r["max_rel"])
    assert tot["over_1ulp_unrelaxed"] == 0
    if w.bank_dtype == "bf16":   # the intervals are tight: mostly within 1 bf16 ulp of y
        assert tot["relaxed"] <= 0.05 * tot["elements"], tot
    else:                        # float32 rows: the 1e-4 relative target, many times over
        assert max_rel <= 1e-6, max_rel


def test_planted_cpe_drop_leaves_the_interval():
    w = scaled(WORKLOADS["uniform_c128"], P=1, T=64, C=32, S=24, hd=8, W=4, R=2, gate_mu=0.0, name="bounds_plant")
    x = make_inputs(w)
    bank = bf16_bits_to_f32(make_bank_stream(w, 0)).astype(np.float64)
    emu = bank.copy()
    carry = np.zeros_like(bank)
    dv = oracle.as_f64(x["dv"][0:w.C], w.dv_dtype)
    st = bounds.dw_step(bank, carry, x["k_idx"][0], x["q_idx"][0], x["k_val"][0], x["q_val"][0], x["g"][0], dv,
                        S=w.S, V=w.C, val_dtype=w.val_dtype, bank_dtype=w.bank_dtype)
    _emulate_step(emu, x, 0, w.C, w.S, w.hd, w.C, w.val_dtype, w.dv_dtype, w.bank_dtype, drop_cpe=True)
    r = bounds.check_rows(emu[st["rows"]], st, w.bank_dtype)
    assert not r["ok"].all()
