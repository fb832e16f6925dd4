"""GPU parity of Phase 1 and DW against the float64 oracle, through the C ABI.

Workloads are the five synthetic workloads at sizes the oracle finishes in seconds (several
tiles, ragged tails), plus degenerate chunks (one slot for a whole chunk: 127 / 4095
saturations; tiny chunks; a single column). Full-size runs are in test_fullsize_gpu.py.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import sparse_slot_memory_gb300 as sdm
from oracle import bounds
from sdm_testlib import BankStats, compare_p1, host, inputs_to_dev, oracle_p1, run_phase1
from synth import WORKLOADS, bf16_bits_to_f32, make_bank_stream, make_inputs, scaled

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": WORKLOADS["tiny"],
    "uniform_c128": scaled(WORKLOADS["uniform_c128"], P=2, T=1024),
    "zipf_c256": scaled(WORKLOADS["zipf_c256"], P=2, T=1024),
    "large": scaled(WORKLOADS["large"], P=2, T=1024),
    "wide_ragged": scaled(WORKLOADS["wide_ragged"], P=2, T=300),
    "one_slot": scaled(WORKLOADS["large"], P=1, T=512, S=1, hd=8, name="one_slot"),
    "few_slots": scaled(WORKLOADS["tiny"], P=3, T=200, C=64, S=8, hd=16, W=5, R=3, name="few_slots"),
    "c1_w1_r1": scaled(WORKLOADS["tiny"], P=3, T=5, C=1, S=16, hd=4, W=1, R=1, name="c1_w1_r1"),
    "bf16_hd4_ragged": scaled(WORKLOADS["uniform_c128"], P=2, T=100, C=48, S=64, hd=4, W=3, R=7,
                              name="bf16_hd4_ragged"),
    # ~32 write entries per slot and chunk over 64 slots: more hot groups than the dense pair path
    # takes (the rest keep the exact walk)
    "many_hot": scaled(WORKLOADS["zipf_c256"], P=1, T=512, S=64, hd=8, idx="uniform", name="many_hot"),
    # strongly decaying gates (logsigmoid(N(-3, 1))) over 4 slots: the groups' log-cumsums span far
    # more than the dense path's exponent range, so they keep the exact walk
    "wide_span": scaled(WORKLOADS["uniform_c128"], P=1, T=256, S=4, hd=8, W=4, R=4, gate_mu=-3.0,
                        name="wide_span"),
    # ~32 write entries per slot and chunk in rows of two column slices (the second partial) with a
    # ragged last step: long groups (summed ahead of the DW) next to short ones, every slice
    "wide_hot": scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=16, hd=200, name="wide_hot"),
    # one gate per write entry (g [N, C, W]): few slots, so a token often writes one slot on several
    # lanes and only its first lane's gate may count; and the skewed workload's hot slots
    "tiny_pe": scaled(WORKLOADS["tiny"], P=2, T=256, S=48, hd=16, gate_per_entry=True, name="tiny_pe"),
    "zipf_pe": scaled(WORKLOADS["zipf_c256"], P=2, T=1024, gate_per_entry=True, name="zipf_pe"),
}


def _setup(name):
    w = CASES[name]
    x = make_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)
    d = inputs_to_dev(x, w)
    ws = sdm.alloc_workspace(shape)
    return w, x, shape, d, ws


@pytest.mark.parametrize("name", list(CASES))
def test_phase1_parity(name):
    w, x, shape, d, ws = _setup(name)
    out = run_phase1(shape, d, ws)
    assert sdm.device_status(ws) == 0
    orc, lo, hi = oracle_p1(x, w)
    rep = compare_p1(out, orc, lo, hi, w.val_dtype)
    assert int(out["repeats"][0]) == orc["repeats"]
    print(name, rep)


def _expected_stats(x, w):
    """The Phase-1 counters from their definitions, by plain loops over each chunk's valid entries
    in entry order (the stable sort keeps it inside a slot group): valid write groups; pair terms
    (a write entry with an earlier valid write entry of another token: A; a read entry with an
    earlier valid write entry: QK); rows the pair phase writes (a token with an entry that has an
    earlier valid write entry in its group, per triangle)."""
    P, W, R = x["P"], w.W, w.R
    groups = terms = rows = 0
    for c in range(x["k_idx"].shape[0]):
        V = w.valid_last if c // P == w.steps - 1 else w.C
        seen = {}   # slot -> tokens of its valid write entries so far, in entry order
        arow, qrow = set(), set()
        for t in range(V):
            for a in range(W):
                s_ = int(x["k_idx"][c][t, a])
                if 0 <= s_ < w.S:
                    prev = seen.setdefault(s_, [])
                    terms += sum(1 for tf in prev if tf != t)
                    if prev:
                        arow.add(t)
                    prev.append(t)
            for b in range(R):
                s_ = int(x["q_idx"][c][t, b])
                if 0 <= s_ < w.S and seen.get(s_):
                    terms += len(seen[s_])
                    qrow.add(t)
        groups += len(seen)
        rows += len(arow) + len(qrow)
    return groups, terms, rows


@pytest.mark.parametrize("name", ["tiny", "uniform_c128", "few_slots", "c1_w1_r1", "bf16_hd4_ragged", "tiny_pe",
                                  "many_hot"])
def test_phase1_stats(name):
    """out.stats against the counts of the definitions; with dense groups (many_hot) the groups
    exactly and the dense count positive (their pairs are then not counted one by one)."""
    w, x, shape, d, ws = _setup(name)
    out = run_phase1(shape, d, ws, fields=("A", "QK", "stats"))
    st = [int(v) for v in host(out["stats"])]
    groups, terms, rows = _expected_stats(x, w)
    assert st[0] == groups, (st, groups)
    if name in ("many_hot", "few_slots"):   # dense groups: their pairs are not counted one by one, and a
        assert st[1] > 0 and st[2] < terms and st[3] >= rows, (st, terms, rows)   # row they reach is written
    else:
        assert st[1] == 0 and st[2] == terms and st[3] == rows, (st, terms, rows)
    print(name, dict(zip(sdm.STATS, st)))


def _init_bank(w, P):
    """Initial bank rows of every stream as float32 [P, S, hd] (exact for either bank type)."""
    rows = []
    for p in range(P):
        b = make_bank_stream(w, p)
        rows.append(bf16_bits_to_f32(b) if w.bank_dtype == "bf16" else b)
    return np.stack(rows, 0)


def _bank_dev(rows64: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(rows64, np.float32)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def _stream_compact(w, x, p):
    """The slots stream p touches, and its chunks' ids relabelled to [0, U) by rank (a monotone
    relabelling keeps every sort order and group, so the oracle can run on U rows)."""
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


@pytest.mark.parametrize("name", list(CASES))
def test_dw_parity_stepwise(name):
    """Each step from the oracle's own pre-step rows (copied into the GPU bank first): every
    touched element inside the interval of values a float32 evaluation can store (within 1 ulp of
    the exact update of the bank type unless the interval says otherwise: counted and reported),
    every other row bitwise unchanged."""
    w, x, shape, d, ws = _setup(name)
    run_phase1(shape, d, ws, fields=("repeats",))
    P, S, hd, C = x["P"], w.S, w.hd, w.C
    init = _init_bank(w, P)
    gpu_bank = _bank_dev(init.reshape(P * S, hd), w.bank_dtype)
    comp = [_stream_compact(w, x, p) for p in range(P)]
    banks = [init[p][comp[p][0]].astype(np.float64) for p in range(P)]    # oracle state on the touched slots
    rng = np.random.default_rng(0)
    stats = BankStats(name, "per_step", w.bank_dtype)
    for ti in range(w.steps):
        for p in range(P):
            rows = torch.from_numpy(p * S + comp[p][0].astype(np.int64)).cuda()
            gpu_bank.index_copy_(0, rows, _bank_dev(banks[p], w.bank_dtype))
        snapshot = gpu_bank.clone()
        sdm.dw(shape, d["dv"], gpu_bank, ws, ti, ti + 1)
        torch.cuda.synchronize()
        assert sdm.device_status(ws) == 0
        changed = (gpu_bank != snapshot).any(dim=1).cpu().numpy()
        for p in range(P):
            slots, xs = comp[p]
            U = len(slots)
            before = banks[p].copy()
            c = ti * P + p
            V = w.valid_last if ti == w.steps - 1 else C
            dvr = oracle.as_f64(x["dv"][c * C:(c + 1) * C], w.dv_dtype)
            st = bounds.dw_step(banks[p], np.zeros_like(banks[p]), xs["k_idx"][c], xs["q_idx"][c], x["k_val"][c],
                                x["q_val"][c], x["g"][c], dvr, S=U, V=V, val_dtype=w.val_dtype,
                                bank_dtype=w.bank_dtype)
            got = host(gpu_bank[torch.from_numpy(p * S + slots.astype(np.int64)).cuda()]).astype(np.float64)
            t = np.zeros(U, bool)
            t[st["rows"]] = True
            assert np.array_equal(got[~t], before[~t]), f"step {ti} stream {p}: an untouched row changed"
            r = bounds.check_rows(got[st["rows"]], st, w.bank_dtype)
            assert r["ok"].all(), (f"step {ti} stream {p}: {int((~r['ok']).sum())} bank elements outside their "
                                   f"interval; first gpu {got[st['rows']][~r['ok']][0]} exact {st['y'][~r['ok']][0]}")
            stats.add(r)
            # rows of the stream that no entry names are never written
            others = np.setdiff1d(rng.integers(0, S, size=min(S, 4096)), slots)
            assert not changed[p * S + others].any()
    stats.finish()


@pytest.mark.parametrize("name", ["tiny", "uniform_c128", "zipf_c256", "wide_ragged", "few_slots", "large", "tiny_pe",
                                  "zipf_pe"])
def test_forward_end_to_end(name):
    """sdm_forward_chunks over every step vs the oracle run step after step in its own state.
    A difference of one rounding can carry into a row's later writes: a row written k times is
    allowed k times the one-step tolerance."""
    w, x, shape, d, ws = _setup(name)
    P, S, hd = x["P"], w.S, w.hd
    init = _init_bank(w, P)
    gpu_bank = _bank_dev(init.reshape(P * S, hd), w.bank_dtype)
    out = sdm.alloc_outputs(shape)
    sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], gpu_bank, out, ws)
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0
    orc, lo, hi = oracle_p1(x, w)
    compare_p1(out, orc, lo, hi, w.val_dtype)
    stats = BankStats(name, "end_to_end", w.bank_dtype)
    for p in range(P):
        slots, xs = _stream_compact(w, x, p)
        bank = init[p][slots].astype(np.float64)
        b = bounds.dw_stream_bounds(bank, xs, p, S=len(slots), C=w.C, P=P, steps=w.steps, valid_last=w.valid_last,
                                    val_dtype=w.val_dtype, dv_dtype=w.dv_dtype, bank_dtype=w.bank_dtype)
        got = host(gpu_bank[torch.from_numpy(p * S + slots.astype(np.int64)).cuda()]).astype(np.float64)
        t = b["writes"] > 0
        assert np.array_equal(got[~t], init[p][slots][~t])
        last = {"y": b["y"][t], "lo": b["lo"][t], "hi": b["hi"][t], "relaxed": b["relaxed"][t]}
        r = bounds.check_rows(got[t], last, w.bank_dtype)
        assert r["ok"].all(), f"stream {p}: {int((~r['ok']).sum())} elements outside their carried interval"
        # a row written once starts from the same row on both sides: no carry, the per-step bound
        once = b["writes"][t] == 1
        r1 = bounds.check_rows(got[t][once], {k: v[once] for k, v in last.items()}, w.bank_dtype)
        assert r1["over_1ulp_unrelaxed"] == 0
        stats.add(r, once=r1)
    stats.finish()


def _forward_bits(w, shape, d, init, split=None):
    """Every output and the bank of one forward (optionally in two calls split at step `split`),
    as raw bytes."""
    ws = sdm.alloc_workspace(shape)
    bank = _bank_dev(init, w.bank_dtype)
    out = sdm.alloc_outputs(shape)
    if split is None:
        sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, out, ws)
    else:
        sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, out, ws, 0,
                           split)
        sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, out, ws,
                           split, w.steps)
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0
    out["repeats"].zero_()
    return {"bank": bank.view(torch.int16 if w.bank_dtype == "bf16" else torch.int32).cpu().numpy(),
            **{k: v.view(torch.uint8).cpu().numpy() for k, v in out.items()}}


@pytest.mark.parametrize("name", ["uniform_c128", "zipf_c256", "few_slots", "tiny_pe", "wide_hot"])
def test_launch_geometry_does_not_change_bits(name):
    """The same forward with other launch geometries: every Phase-1 block widened by a quarter of its
    warps (at least one; the extra warps hold padding entries: other scan trees over the warps,
    other warps taking the pair rows and the dense groups) and the DW walk over 2 hashed slot buckets per stream, or the
    most the shape allows (each bucket a different warp's walk). Every output bit and the bank agree."""
    w, x, shape, d, ws = _setup(name)
    init = _init_bank(w, x["P"]).reshape(x["P"] * w.S, w.hd)
    ref = _forward_bits(w, shape, d, init)
    kb = max(1, int(np.ceil(np.log2(w.S))))
    warps = -(-w.C * (w.W + w.R) // (8 * 32))   # the automatic Phase-1 warps per block
    for geo in (dict(p1_warps=min(32, warps + max(1, warps // 4)), dw_log_buckets=1),
                dict(dw_log_buckets=min(11, kb))):
        other = _forward_bits(w, dataclasses.replace(shape, **geo), d, init)
        for k in ref:
            assert np.array_equal(ref[k], other[k]), f"{k} differs with geometry {geo}"


@pytest.mark.parametrize("name", ["uniform_c128", "zipf_c256", "wide_ragged", "large"])
def test_resume_and_determinism(name):
    """[0, k) then [k, steps) equals [0, steps) bit for bit; five repeated runs are bitwise identical."""
    w, x, shape, d, ws = _setup(name)
    P = x["P"]
    init = _init_bank(w, P).reshape(P * w.S, w.hd)
    results = [_forward_bits(w, shape, d, init, split)
               for split in (None, None, None, None, None, max(1, w.steps // 2))]
    for r in results[1:]:
        for k in r:
            assert np.array_equal(r[k], results[0][k]), f"{k} differs between runs"


def test_bad_slot_sets_status_without_fault():
    w = scaled(WORKLOADS["tiny"], P=1, T=128, name="bad")
    x = make_inputs(w)
    x["k_idx"][1, 3, 2] = w.S + 5      # out of range
    x["q_idx"][0, 0, 0] = -7
    shape = sdm.ShapeSpec.from_workload(w)
    d = inputs_to_dev(x, w)
    ws = sdm.alloc_workspace(shape)
    bank = torch.zeros(w.P * w.S, w.hd, device="cuda")
    sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, None, ws)
    code = sdm.device_status(ws, clear=True)
    assert code & 0x1
    assert sdm.device_status(ws) == 0   # cleared
    assert torch.isfinite(bank).all()


def test_empty_range_is_noop():
    w, x, shape, d, ws = _setup("tiny")
    bank = torch.ones(w.P * w.S, w.hd, device="cuda")
    sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, None, ws, 3, 3)
    torch.cuda.synchronize()
    assert bool((bank == 1).all())


def test_host_checks_before_launch():
    w, x, shape, d, ws = _setup("tiny")
    bank = torch.zeros(w.P * w.S, w.hd, device="cuda")
    with pytest.raises(sdm.SdmError) as e:
        sdm.dw(shape, d["dv"], bank, ws[:1024], 0, 1)
    assert e.value.status == -5
    big = torch.zeros(w.P * w.S * w.hd + 64, device="cuda")   # a full-size bank one element off alignment
    with pytest.raises(sdm.SdmError) as e:
        sdm.dw(shape, d["dv"], big[1:1 + w.P * w.S * w.hd].view(-1, w.hd), ws, 0, 1)
    assert e.value.status == -4
    with pytest.raises(sdm.SdmError) as e:
        sdm.dw(shape, d["dv"], bank, ws, 2, 1)
    assert e.value.status == -1


@pytest.mark.parametrize("name", ["uniform_c128", "zipf_c256", "few_slots", "one_slot"])
def test_one_launch_equals_per_step_launches(name):
    """One DW launch over every step (windows of records spanning steps, sub-batches cut before a
    repeated slot) gives the bits of one launch per step (each step's loads after the previous
    step's stores): the per-step definition, in program order."""
    w, x, shape, d, ws = _setup(name)
    run_phase1(shape, d, ws, fields=("repeats",))
    P, S, hd = x["P"], w.S, w.hd
    init = _init_bank(w, P).reshape(P * S, hd)
    b1 = _bank_dev(init, w.bank_dtype)
    b2 = _bank_dev(init, w.bank_dtype)
    sdm.dw(shape, d["dv"], b1, ws)
    for t in range(w.steps):
        sdm.dw(shape, d["dv"], b2, ws, t, t + 1)
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0
    assert torch.equal(b1, b2)
