"""Pins of the float64 oracle against definitions other than its own code.

* A hand-worked chunk (tests/golden/hand_chunk.json), derived on paper from the definitions of
  sparse-delta-memory 2.0.0 (phase1_cuda.py module docstring, p1_keys_zw_kernel, p1_scan_kernel,
  the p1_pairs_kernel comment; DW from the mover_da2_cuda.py / mover_fx_cuda.py docstrings).
* Sort positions, group peers, the position pack and the sorted-row elements against Python's
  ``sorted`` and direct counting over all entries.
* log_k / log_q / rex / cpe against the token form: G_s(t) = sum of the gates of the tokens
  t' <= t that write slot s, each token once (phase1_cuda.py docstring: log-cumsum of the gates,
  rex = gates of the later writes, cpe = exp(total gate of the slot)).
* A and QK against a brute force over all lane pairs, O(C^2 W^2).
* DW against the token-sequential recurrence: token by token, decay each slot the token writes
  once by exp(g_t), then add k * dv_t per write lane. The chunk form is the same in exact
  arithmetic; a single write gives base * exp(g) + k * dv.
* Rounding to bfloat16 against a neighbour search.
* Planted mistakes in the oracle's C source fail these pins.
"""

import json
import math
import os
import shutil

import numpy as np
import pytest

import oracle
from synth import WORKLOADS, f32_to_bf16_bits, make_bank_stream, make_inputs, scaled

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- brute-force definitions

def bf_sorted(k_idx, q_idx, V):
    """Sorted order of one chunk: entries e = t*(W+R)+j keyed by (slot, e); invalid last."""
    C, W = k_idx.shape
    R = q_idx.shape[1]
    ents = []
    for t in range(C):
        for j in range(W + R):
            q = j >= W
            a = j - W if q else j
            slot = int(q_idx[t, a] if q else k_idx[t, a])
            valid = t < V
            ents.append(dict(e=t * (W + R) + j, t=t, a=a, q=q, slot=slot, valid=valid))
    order = sorted(ents, key=lambda d: ((0, d["slot"]) if d["valid"] else (1, 0), d["e"]))
    return order


def bf_peers(order, d):
    """(before, after): valid entries of the same kind and slot before / after d in sorted order."""
    if not d["valid"]:
        return 0, 0
    r = order.index(d)
    same = [i for i, x in enumerate(order) if x["valid"] and x["slot"] == d["slot"] and x["q"] == d["q"]]
    return sum(1 for i in same if i < r), sum(1 for i in same if i > r)


def token_gate(k_idx, g, t, s):
    """Token t's gate on slot s: g[t] (one gate per token), or with one gate per write entry
    (g [C, W]) the gate of t's first write lane on s -- a later lane of t on s is a repeat and
    adds nothing."""
    if np.ndim(g) == 1:
        return float(g[t])
    first = min(a for a in range(k_idx.shape[1]) if int(k_idx[t, a]) == s)
    return float(g[t, first])


def token_G(k_idx, g, V):
    """G[s][t] = sum of the gates of the tokens t' <= t (t' < V) that write slot s (each token once,
    with its gate on s)."""
    C, W = k_idx.shape
    G = {}
    for s in set(int(x) for x in k_idx[:V].ravel()):
        run, col = 0.0, []
        for t in range(C):
            if t < V and s in set(int(x) for x in k_idx[t]):
                run += token_gate(k_idx, g, t, s)
            col.append(run)
        G[s] = col
    return G


def Gs(G, s, t):
    return G[s][t] if s in G else 0.0


def random_chunk(rng, C, W, R, S, V, per_entry=False):
    k_idx = rng.integers(0, S, size=(C, W)).astype(np.int32)
    q_idx = rng.integers(0, S, size=(C, R)).astype(np.int32)
    k_idx[V:] = -1
    q_idx[V:] = -1
    k_val = rng.standard_normal((C, W)).astype(np.float32)
    q_val = rng.standard_normal((C, R)).astype(np.float32)
    z = rng.standard_normal((C, W) if per_entry else C) + 1.0
    g = (np.minimum(z, 0) - np.log1p(np.exp(-np.abs(z)))).astype(np.float32)
    return k_idx, q_idx, k_val, q_val, g


CASES = [  # (C, W, R, S, V): small S gives collisions and repeated slots within a token
    (8, 3, 2, 5, 8), (8, 3, 2, 5, 6), (6, 4, 4, 3, 6), (10, 2, 3, 7, 4), (5, 1, 1, 2, 5), (7, 5, 1, 4, 7),
]
# the same shapes with one gate per write entry (g [C, W]); the repeated slots within a token make
# "which lane's gate" observable
GATES = ["token", "entry"]


def run_oracle_chunk(k_idx, q_idx, k_val, q_val, g, S, V, lib=None):
    return oracle.phase1(k_idx[None], q_idx[None], k_val[None], q_val[None], g[None], S=S,
                         val_dtype="f32", first_partial=0, valid_last=V, lib=lib)


# ---------------------------------------------------------------- pins

@pytest.mark.parametrize("fixture", ["hand_chunk.json", "hand_chunk_per_entry.json"])
def test_hand_chunk_golden(fixture):
    fx = json.load(open(os.path.join(HERE, "golden", fixture)))
    ev = lambda s: eval(s, {"exp": math.exp})  # noqa: E731  (expressions written in the fixture)
    k_idx = np.array(fx["k_idx"], np.int32)
    q_idx = np.array(fx["q_idx"], np.int32)
    k_val = np.array(fx["k_val"], np.float32)
    q_val = np.array(fx["q_val"], np.float32)
    g = np.array(fx["g"], np.float32)
    o = run_oracle_chunk(k_idx, q_idx, k_val, q_val, g, fx["S"], fx["V"])
    for f in ("log_k", "rex", "cpe", "k_eff", "log_q", "q_w", "A", "QK"):
        want = np.array([[ev(x) for x in row] for row in fx[f]])
        np.testing.assert_allclose(o[f][0], want, rtol=1e-12, atol=1e-12, err_msg=f)
    for f in ("is_last", "is_only", "pos_k", "pos_q", "q_last", "q_only"):
        np.testing.assert_array_equal(o[f][0], np.array(fx[f]), err_msg=f)
    assert o["repeats"] == fx["repeats"]
    np.testing.assert_array_equal(o["sorted_k"][0].view(np.uint32), [int(h, 16) for h in fx["sorted_k_hex"]])
    np.testing.assert_array_equal(o["sorted_q"][0].view(np.uint32), [int(h, 16) for h in fx["sorted_q_hex"]])
    bank = np.array(fx["bank_in"], np.float64)
    oracle.dw_chunk(bank, k_idx, q_idx, k_val, q_val, g, np.array(fx["dv"], np.float64), S=fx["S"],
                    V=fx["V"], val_dtype="f32", bank_dtype="f32", round_cpe=False, round_bank=False)
    want = np.array([[ev(x) for x in row] for row in fx["bank_out"]])
    np.testing.assert_allclose(bank, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", CASES)
def test_sort_positions_and_rows_bruteforce(case):
    C, W, R, S, V = case
    rng = np.random.default_rng(hash(case) % 2**32)
    k_idx, q_idx, k_val, q_val, g = random_chunk(rng, C, W, R, S, V)
    o = run_oracle_chunk(k_idx, q_idx, k_val, q_val, g, S, V)
    order = bf_sorted(k_idx, q_idx, V)
    sk, sq = [], []
    for r, d in enumerate(order):
        b, a = bf_peers(order, d)
        if d["valid"]:
            asat = min(a, 127)
            want = r | asat << 17 | min(b + 1 + asat, 127) << 24
        else:
            want = r
        got = o["pos_q" if d["q"] else "pos_k"][0, d["t"], d["a"]]
        assert got == want, (d, got, want)
        last, only = (a == 0 and d["valid"]), (a == 0 and b == 0 and d["valid"])
        if d["q"]:
            assert o["q_last"][0, d["t"], d["a"]] == last and o["q_only"][0, d["t"], d["a"]] == only
        else:
            assert o["is_last"][0, d["t"], d["a"]] == last and o["is_only"][0, d["t"], d["a"]] == only
        el = d["t"] << 9 | int(d["q"]) << 8 | d["a"] | (0 if d["valid"] else 0x20000)
        if d["valid"]:
            el |= min(b, 4095) << 18 | (1 << 31 if b == 0 else 0) | (1 << 30 if a == 0 else 0)
        else:
            el |= 3 << 30
        (sq if d["q"] else sk).append(el)
    np.testing.assert_array_equal(o["sorted_k"][0].view(np.uint32), np.array(sk, np.uint64).astype(np.uint32))
    np.testing.assert_array_equal(o["sorted_q"][0].view(np.uint32), np.array(sq, np.uint64).astype(np.uint32))
    # repeated write entries: a token's write lanes beyond the first on one slot
    reps = sum(len(k_idx[t]) - len(set(k_idx[t].tolist())) for t in range(V))
    assert o["repeats"] == reps


@pytest.mark.parametrize("gate", GATES)
@pytest.mark.parametrize("case", CASES)
def test_logs_rex_cpe_token_form(case, gate):
    C, W, R, S, V = case
    rng = np.random.default_rng(1 + hash(case) % 2**32)
    k_idx, q_idx, k_val, q_val, g = random_chunk(rng, C, W, R, S, V, per_entry=gate == "entry")
    o = run_oracle_chunk(k_idx, q_idx, k_val, q_val, g, S, V)
    G = token_G(k_idx, g, V)
    for t in range(C):
        for a in range(W):
            s = int(k_idx[t, a])
            if t >= V:
                assert o["log_k"][0, t, a] == 0 and o["rex"][0, t, a] == 0 and o["cpe"][0, t, a] == 1
                assert o["k_eff"][0, t, a] == 0
                continue
            tot = G[s][C - 1]
            assert o["log_k"][0, t, a] == pytest.approx(G[s][t], abs=1e-12)
            assert o["rex"][0, t, a] == pytest.approx(tot - G[s][t], abs=1e-12)
            assert o["cpe"][0, t, a] == pytest.approx(math.exp(tot), rel=1e-12)
            assert o["k_eff"][0, t, a] == pytest.approx(float(k_val[t, a]) * math.exp(G[s][t]), rel=1e-12)
            if o["is_last"][0, t, a]:
                assert o["rex"][0, t, a] == 0.0
        for a in range(R):
            s = int(q_idx[t, a])
            if t >= V:
                assert o["log_q"][0, t, a] == 0 and o["q_w"][0, t, a] == 0
                continue
            assert o["log_q"][0, t, a] == pytest.approx(Gs(G, s, t), abs=1e-12)
            assert o["q_w"][0, t, a] == pytest.approx(float(q_val[t, a]) * math.exp(Gs(G, s, t)), rel=1e-12)


def bf_pairs(k_idx, q_idx, k_val, q_val, g, V):
    C, W = k_idx.shape
    R = q_idx.shape[1]
    G = token_G(k_idx, g, V)
    A = np.zeros((C, C))
    QK = np.zeros((C, C))
    for i in range(V):
        for j in range(V):
            for b in range(W):
                s = int(k_idx[j, b])
                if j < i:
                    for a in range(W):
                        if int(k_idx[i, a]) == s:
                            A[i, j] += float(k_val[i, a]) * float(k_val[j, b]) * math.exp(G[s][i] - G[s][j])
                if j <= i:
                    for a in range(R):
                        if int(q_idx[i, a]) == s:
                            QK[i, j] += float(q_val[i, a]) * float(k_val[j, b]) * math.exp(G[s][i] - G[s][j])
    return A, QK


@pytest.mark.parametrize("gate", GATES)
@pytest.mark.parametrize("case", CASES)
def test_pairs_bruteforce(case, gate):
    C, W, R, S, V = case
    rng = np.random.default_rng(2 + hash(case) % 2**32)
    k_idx, q_idx, k_val, q_val, g = random_chunk(rng, C, W, R, S, V, per_entry=gate == "entry")
    o = run_oracle_chunk(k_idx, q_idx, k_val, q_val, g, S, V)
    A, QK = bf_pairs(k_idx, q_idx, k_val, q_val, g, V)
    np.testing.assert_allclose(o["A"][0], A, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o["QK"][0], QK, rtol=1e-12, atol=1e-12)
    assert np.all(np.triu(o["A"][0]) == 0) and np.all(np.triu(o["QK"][0], 1) == 0)


def token_recurrence(bank, k_idx, k_val, g, dv, V):
    for t in range(V):
        for s in set(int(x) for x in k_idx[t]):
            bank[s] *= math.exp(token_gate(k_idx, g, t, s))
        for a in range(k_idx.shape[1]):
            bank[int(k_idx[t, a])] += float(k_val[t, a]) * dv[t]


@pytest.mark.parametrize("gate", GATES)
@pytest.mark.parametrize("case", CASES)
def test_dw_token_recurrence(case, gate):
    C, W, R, S, V = case
    hd = 4
    rng = np.random.default_rng(3 + hash(case) % 2**32)
    bank = rng.standard_normal((S, hd))
    want = bank.copy()
    for step in range(3):   # a stream of three chunks, the last one ragged when V < C
        Vs = V if step == 2 else C
        k_idx, q_idx, k_val, q_val, g = random_chunk(rng, C, W, R, S, Vs, per_entry=gate == "entry")
        dv = rng.standard_normal((C, hd)).astype(np.float32).astype(np.float64)
        oracle.dw_chunk(bank, k_idx, q_idx, k_val, q_val, g, dv, S=S, V=Vs, val_dtype="f32",
                        bank_dtype="f32", round_cpe=False, round_bank=False)
        token_recurrence(want, k_idx, k_val, g, dv, Vs)
    np.testing.assert_allclose(bank, want, rtol=1e-11, atol=1e-11)


def test_dw_single_entry_closed_form():
    C, W, R, S, hd = 4, 2, 1, 64, 3
    k_idx = np.array([[10, 11], [12, 13], [14, 15], [16, 17]], np.int32)
    q_idx = np.array([[10], [20], [21], [22]], np.int32)
    k_val = np.array([[0.5, -1.5], [2.0, 0.25], [1.0, 1.0], [-3.0, 0.125]], np.float32)
    q_val = np.ones((C, R), np.float32)
    g = np.array([-0.1, -0.7, -2.0, -0.3], np.float32)
    dv = np.arange(C * hd, dtype=np.float64).reshape(C, hd) - 5.0
    base = np.random.default_rng(5).standard_normal((S, hd))
    bank = base.copy()
    oracle.dw_chunk(bank, k_idx, q_idx, k_val, q_val, g, dv, S=S, V=C, val_dtype="f32", bank_dtype="f32",
                    round_cpe=False, round_bank=False)
    for t in range(C):
        for a in range(W):
            s = k_idx[t, a]
            want = base[s] * math.exp(float(g[t])) + float(k_val[t, a]) * dv[t]
            np.testing.assert_allclose(bank[s], want, rtol=1e-13)
    untouched = np.setdiff1d(np.arange(S), k_idx.ravel())
    np.testing.assert_array_equal(bank[untouched], base[untouched])


def nearest_bf16(x):
    """Nearest bfloat16 of a float64 by a neighbour search (ties to the even pattern)."""
    f = np.float32(x)
    b = int(f32_to_bf16_bits(np.array([f]))[0])
    cands = [(c & 0xFFFF) for c in (b - 1, b, b + 1)]
    vals = [float((np.array([c], np.uint32) << 16).view(np.float32)[0]) for c in cands]
    best = min(range(3), key=lambda i: (abs(vals[i] - x), cands[i] & 1))
    return vals[best]


def test_bank_rounding_bf16():
    """Singleton groups on a zero base store round(k * dv) exactly (rex = 0)."""
    rng = np.random.default_rng(9)
    C, W, R, S, hd = 16, 1, 1, 64, 8
    k_idx = np.arange(C, dtype=np.int32).reshape(C, 1)
    q_idx = np.full((C, 1), 40, np.int32)
    k_val = rng.standard_normal((C, 1)).astype(np.float32)
    q_val = np.ones((C, 1), np.float32)
    g = np.full(C, -0.5, np.float32)
    dv = rng.standard_normal((C, hd)) * 3.0
    bank = np.zeros((S, hd))
    oracle.dw_chunk(bank, k_idx, q_idx, k_val, q_val, g, dv, S=S, V=C, val_dtype="f32", bank_dtype="bf16",
                    round_cpe=True, round_bank=True)
    for t in range(C):
        for i in range(hd):
            x = float(k_val[t, 0]) * dv[t, i]
            assert bank[t, i] == nearest_bf16(x)


def test_cpe_rounding_feeds_dw():
    """DW uses cpe as stored in the value type (bf16): base * round(exp(G)) enters the sum."""
    C, W, R, S, hd = 2, 1, 1, 8, 2
    k_idx = np.array([[3], [3]], np.int32)
    q_idx = np.array([[0], [0]], np.int32)
    k_val = np.zeros((C, 1), np.float32)
    q_val = np.zeros((C, 1), np.float32)
    g = np.array([-0.3, -0.45], np.float32)
    dv = np.zeros((C, hd))
    bank = np.zeros((S, hd))
    bank[3] = [1.0, -2.0]
    oracle.dw_chunk(bank, k_idx, q_idx, f32_to_bf16_bits(k_val), f32_to_bf16_bits(q_val), g, dv, S=S, V=C,
                    val_dtype="bf16", bank_dtype="f32", round_cpe=True, round_bank=False)
    cp = nearest_bf16(math.exp(float(g[0]) + float(g[1])))
    np.testing.assert_array_equal(bank[3], [cp, -2.0 * cp])


def test_flag_invariants_zipf():
    w = scaled(WORKLOADS["zipf_c256"], P=1, T=512)
    x = make_inputs(w)
    o = oracle.phase1(x["k_idx"], x["q_idx"], x["k_val"], x["q_val"], x["g"], S=w.S, val_dtype=w.val_dtype,
                      pairs=False)
    for c in range(x["k_idx"].shape[0]):
        ki = x["k_idx"][c]
        for s in np.unique(ki):
            m = ki == s
            assert o["is_last"][c][m].sum() == 1
            assert o["is_only"][c][m].sum() == (1 if m.sum() == 1 else 0)
        assert np.all(o["is_last"][c] >= o["is_only"][c])
        pk = o["pos_k"][c].view(np.uint32)
        after, size = (pk >> 17) & 127, (pk >> 24) & 127
        assert np.all(size >= np.minimum(after + 1, 127))   # both saturate at 127
        # positions are a permutation of the sorted row
        r = np.concatenate([pk.ravel() & 0x1FFFF, o["pos_q"][c].view(np.uint32).ravel() & 0x1FFFF])
        assert np.array_equal(np.sort(r), np.arange(r.size))


def test_ragged_tail_invalid_entries():
    w = scaled(WORKLOADS["wide_ragged"], P=2, T=200, C=64, hd=8)
    x = make_inputs(w)
    assert w.valid_last == 200 - 3 * 64
    fp = (w.steps - 1) * w.P
    o = oracle.phase1(x["k_idx"], x["q_idx"], x["k_val"], x["q_val"], x["g"], S=w.S, val_dtype=w.val_dtype,
                      first_partial=fp, valid_last=w.valid_last, pairs=True)
    V, C, W, R = w.valid_last, w.C, w.W, w.R
    for c in range(fp, x["k_idx"].shape[0]):
        assert np.all(o["log_k"][c, V:] == 0) and np.all(o["cpe"][c, V:] == 1) and np.all(o["is_last"][c, V:] == 0)
        r = o["pos_k"][c, V:].view(np.uint32)
        assert np.all(r >> 17 == 0) and np.all(r >= V * (W + R) - 0)   # invalid entries sort last
        assert np.all(o["A"][c, V:] == 0) and np.all(o["QK"][c, V:] == 0) and np.all(o["QK"][c, :, V:] == 0)
        tail = o["sorted_k"][c].view(np.uint32)[V * W:]
        assert np.all(tail >> 30 == 3) and np.all(tail & 0x20000)


# ---------------------------------------------------------------- planted mistakes

MUTATIONS = {
    "decay_sign": ("exp(ch.logv[e] - ch.logv[f])", "exp(ch.logv[f] - ch.logv[e])"),
    "repeat_rule_dropped": ("if (!prev_same) xe =", "if (1) xe ="),
    "rex_includes_own": ("for (int u = s + 1; u < r1; ++u) after", "for (int u = s; u < r1; ++u) after"),
    "qk_diagonal_dropped": ("ch.isq[e] && j <= i", "ch.isq[e] && j < i"),
    "pos_after_before_swapped": ("(uint32_t)asat << 17", "(uint32_t)imin(before, 127) << 17"),
    "dw_cpe_dropped": ("double nv = base * cp + acc[i]", "double nv = base + acc[i]"),
    "dw_rex_dropped": ("const double sc = ch.val[e] * exp(ch.rex[e])", "const double sc = ch.val[e]"),
    "after_count_off_by_one": ("ch->ka[e] = nk - kseen;", "ch->ka[e] = nk - kseen + 1;"),
    "group_total_drops_last": ("tot += xe;", "tot += (s + 1 < r1) ? xe : 0.0;"),
    # per-entry gates: the gate of the token's last write lane (every entry reads lane W - 1) ...
    "gate_lane_last": ("g[ch->tok[e] * g_width + ch->lane[e] * g_lane_stride]",
                       "g[ch->tok[e] * g_width + (W - 1) * g_lane_stride]"),
    # ... of lane 0 whatever the entry's lane ...
    "gate_lane_zero": ("g[ch->tok[e] * g_width + ch->lane[e] * g_lane_stride]", "g[ch->tok[e] * g_width]"),
    # ... or of a token's LAST write entry on the slot (the repeat rule looking forward, not back)
    "gate_of_last_repeat": (
        "const int prev_same = s > r && !ch->isq[ch->order[s - 1]] && ch->valid[ch->order[s - 1]] &&\n"
        "                                      ch->tok[ch->order[s - 1]] == ch->tok[e];",
        "const int prev_same = s + 1 < r1 && !ch->isq[ch->order[s + 1]] && ch->valid[ch->order[s + 1]] &&\n"
        "                                      ch->tok[ch->order[s + 1]] == ch->tok[e];"),
}


def _pins_pass(lib):
    try:
        for case, per_entry in [(c, pe) for c in CASES[:4] for pe in (False, True)]:
            C, W, R, S, V = case
            rng = np.random.default_rng(11 + hash(case) % 2**32)
            k_idx, q_idx, k_val, q_val, g = random_chunk(rng, C, W, R, S, V, per_entry=per_entry)
            o = run_oracle_chunk(k_idx, q_idx, k_val, q_val, g, S, V, lib=lib)
            A, QK = bf_pairs(k_idx, q_idx, k_val, q_val, g, V)
            if not (np.allclose(o["A"][0], A, 1e-12, 1e-12) and np.allclose(o["QK"][0], QK, 1e-12, 1e-12)):
                return False
            G = token_G(k_idx, g, V)
            order = bf_sorted(k_idx, q_idx, V)
            for r, d in enumerate(order):
                b, a = bf_peers(order, d)
                if d["valid"]:
                    want = r | min(a, 127) << 17 | min(b + 1 + min(a, 127), 127) << 24
                    if o["pos_q" if d["q"] else "pos_k"][0, d["t"], d["a"]] != want:
                        return False
                    lg = o["log_q" if d["q"] else "log_k"][0, d["t"], d["a"]]
                    if abs(lg - Gs(G, d["slot"], d["t"])) > 1e-12:
                        return False
                    if not d["q"] and abs(o["rex"][0, d["t"], d["a"]] - (G[d["slot"]][C - 1] - G[d["slot"]][d["t"]])) > 1e-12:
                        return False
            hd = 3
            bank = rng.standard_normal((S, hd))
            want = bank.copy()
            dv = rng.standard_normal((C, hd))
            oracle.dw_chunk(bank, k_idx, q_idx, k_val, q_val, g, dv, S=S, V=V, val_dtype="f32", bank_dtype="f32",
                            round_cpe=False, round_bank=False, lib=lib)
            token_recurrence(want, k_idx, k_val, g, dv, V)
            if not np.allclose(bank, want, 1e-11, 1e-11):
                return False
        return True
    except Exception:
        return False


def test_pins_pass_on_the_oracle():
    assert _pins_pass(oracle._load())


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "sdm_oracle.c")).read()
    assert old in src, f"mutation anchor missing: {old}"
    mutated = tmp_path / "sdm_oracle.c"
    mutated.write_text(src.replace(old, new, 1))
    so = oracle.build(str(mutated), str(tmp_path))
    lib = oracle.load_variant(so)
    assert not _pins_pass(lib), f"planted mistake '{name}' was not caught by the pins"
    shutil.rmtree(tmp_path, ignore_errors=True)


def test_snapshot_order_hand_example():
    """The dense snapshot's rows follow the chunk's valid write groups in slot order: ids of invalid
    tokens (t >= V), -1 and ids outside [0, S) form no group (mover_da2_cuda.py, WR mode)."""
    k = np.array([[3, 7, 3], [11, -1, 0], [5, 5, 5]], np.int32)
    assert oracle.snapshot_slots(k, S=10, V=2).tolist() == [0, 3, 7]
    assert oracle.snapshot_slots(k, S=10, V=3).tolist() == [0, 3, 5, 7]


@pytest.mark.parametrize("case", ["tiny_scaled", "zipf_small"])
def test_snapshot_order_matches_sorted_row_groups(case):
    """The dense ordinal of a group (valid write groups before it in the sorted write row, from the
    oracle's Phase-1 sorted_k FIRST flags) is the slot's rank in snapshot_slots."""
    w = {"tiny_scaled": scaled(WORKLOADS["tiny"], T=256), "zipf_small": scaled(WORKLOADS["zipf_c256"], P=1, T=512)}[case]
    x = make_inputs(w)
    orc = oracle.phase1(x["k_idx"], x["q_idx"], x["k_val"], x["q_val"], x["g"], S=w.S, val_dtype=w.val_dtype,
                        valid_last=w.valid_last, first_partial=(w.steps - 1) * w.P)
    for c in range(w.N):
        V = w.valid_last if c >= (w.steps - 1) * w.P else w.C
        el = orc["sorted_k"][c].astype(np.int64) & 0xFFFFFFFF
        first = ((el >> 31) & 1 == 1) & ((el >> 17) & 1 == 0)
        e = el[first] & 0x3FFFF
        t, lane = e >> 9, e & 0xFF
        heads = x["k_idx"][c][t, lane]
        assert heads.tolist() == oracle.snapshot_slots(x["k_idx"][c], S=w.S, V=V).tolist()


def test_snapshot_rows_are_the_pre_step_bank():
    """The captured rows of step t are the stream's rows after the DW of steps [0, t)."""
    w = scaled(WORKLOADS["tiny"], T=512, S=256)
    x = make_inputs(w)
    init = make_bank_stream(w, 0).astype(np.float64)
    kw = dict(S=w.S, C=w.C, P=w.P, steps=w.steps, valid_last=w.valid_last, val_dtype=w.val_dtype,
              dv_dtype=w.dv_dtype, bank_dtype=w.bank_dtype)
    snaps = []
    oracle.dw_stream(init.copy(), x, 0, snaps=snaps, **kw)
    for t in (0, 3, w.steps - 1):
        b = init.copy()
        oracle.dw_stream(b, x, 0, step_end=t, **kw)
        sn = snaps[t]
        assert sn["c"] == t and np.array_equal(sn["rows"], b[sn["slots"]])


def _pa_hand_case():
    # 3 tokens, 2 write lanes, 8 slots; token 1's lane 1 is an invalid id (-1).
    # valid groups by slot: 1 <- (0,0),(1,0),(2,1); 2 <- (0,1); 5 <- (2,0): ordinals 0, 1, 2
    k = np.array([[1, 2], [1, -1], [5, 1]], np.int32)
    kv = np.full((3, 2), 0.5)
    lk = np.zeros((3, 2))            # exp(log_k) = 1
    cpe = np.full((3, 2), 0.9)
    beta = np.array([1.0, 2.0, 3.0])
    dva = np.arange(12, dtype=float).reshape(3, 4)       # rows [0..3], [4..7], [8..11]
    snap = np.arange(12, dtype=float).reshape(3, 4)      # group rows [0..3], [4..7], [8..11]
    return k, kv, lk, cpe, beta, dva, snap


def test_pa_hand_example():
    """Phase A on a hand-worked chunk (pa_dc_cuda.py module docstring, "PA per write group"):
    slot 1: sc = -beta*k*e^0 = -0.5, -1.0, -1.5 for tokens 0, 1, 2, so
      grad[1] = 1*0.9 - 0.5*[0,1,2,3] - 1.0*[4,5,6,7] - 1.5*[8,9,10,11] = [-15.1, -18.1, -21.1, -24.1];
    d_k_eff = -beta * <dva[tok], snap of its group>:
      (0,0): -1*<[0,1,2,3],[0,1,2,3]> = -14; (1,0): -2*<[4..7],[0..3]> = -76; (2,1): -3*<[8..11],[0..3]> = -186;
      (0,1) slot 2: -1*<[0..3],[4..7]> = -38; (2,0) slot 5: -3*<[8..11],[8..11]> = -1098;
    grad_g = cpe * <gdw, snap> with gdw = ones: slot 1: 0.9*6 = 5.4, slot 2: 0.9*22 = 19.8, slot 5: 0.9*38 = 34.2."""
    k, kv, lk, cpe, beta, dva, snap = _pa_hand_case()
    grad = np.ones((8, 4))
    bank = np.full((8, 4), 7.0)
    d_eff, g_g, mag, _, _ = oracle.pa_chunk(grad, bank, snap, k, kv, lk, cpe, beta, dva, S=8, V=3)
    assert np.allclose(d_eff, [[-14, -38], [-76, 0], [-1098, -186]])
    assert np.allclose(g_g, [[5.4, 19.8], [5.4, 0], [34.2, 5.4]])
    assert np.allclose(grad[1], [-15.1, -18.1, -21.1, -24.1])
    # slot 2: 0.9 - 0.5*[0,1,2,3]; slot 5: 0.9 - 1.5*[8,9,10,11]
    assert np.allclose(grad[2], [0.9, 0.4, -0.1, -0.6]) and np.allclose(grad[5], [-11.1, -12.6, -14.1, -15.6])
    # restore: the groups' rows are the snapshot rows, every other row is untouched
    assert np.array_equal(bank[[1, 2, 5]], snap) and np.all(bank[[0, 3, 4, 6, 7]] == 7.0)
    assert np.all(grad[[0, 3, 4, 6, 7]] == 1.0) and np.all(mag[[0, 3, 4, 6, 7]] == 0.0)


def test_pa_single_entry_closed_form():
    """One write entry per group: grad = gdw * cpe - beta * k * exp(log_k) * dva, with cpe = exp(g) of
    the one writer: e.g. g = log(0.5), k = 0.25, beta = 2: grad = 0.5 gdw - 0.25 dva."""
    k = np.array([[3]], np.int32)
    gdw = np.array([[2.0, -4.0]])
    grad = np.zeros((4, 2)); grad[3] = gdw
    bank = np.zeros((4, 2))
    dva = np.array([[8.0, 1.0]])
    d_eff, g_g, *_ = oracle.pa_chunk(grad, bank, np.array([[1.0, 1.0]]), k, np.array([[0.25]]),
                                     np.array([[np.log(0.5)]]), np.array([[0.5]]), np.array([2.0]), dva, S=4, V=1)
    assert np.allclose(grad[3], 0.5 * gdw[0] - 0.25 * dva[0])   # [1 - 2, -2 - 0.25]
    assert np.allclose(grad[3], [-1.0, -2.25])
    assert np.isclose(d_eff[0, 0], -2.0 * 9.0) and np.isclose(g_g[0, 0], 0.5 * (-2.0))


def test_pa_linear_in_grad_and_dva():
    """Phase A is linear in (grad, dva) for fixed records and snapshot (a dropped term, a wrong
    sign or a swapped operand breaks one of these)."""
    rng = np.random.default_rng(3)
    S, C, W, hd = 16, 6, 3, 5
    k = rng.integers(0, 5, size=(C, W)).astype(np.int32)
    kv, lk = rng.standard_normal((C, W)), -rng.random((C, W))
    cpe = np.broadcast_to(rng.random((1, 1)) + 0.2, (C, W)).copy()
    beta, snap = rng.random(C), rng.standard_normal((S, hd))
    g1, g2 = rng.standard_normal((S, hd)), rng.standard_normal((S, hd))
    d1, d2 = rng.standard_normal((C, hd)), rng.standard_normal((C, hd))

    def run(gr, dv):
        gr = gr.copy()
        out = oracle.pa_chunk(gr, np.zeros((S, hd)), snap, k, kv, lk, cpe, beta, dv, S=S, V=C)
        return gr, out[0], out[1]

    a, b = 1.5, -0.75
    rs = run(a * g1 + b * g2, a * d1 + b * d2)
    r1, r2 = run(g1, d1), run(g2, d2)
    for x, y1, y2 in zip(rs, r1, r2):
        assert np.allclose(x, a * y1 + b * y2)


def test_pa_decay_uses_last_members_cpe():
    """The group's grad row decays by cpe_last, the last member's cpe (pa_dc_cuda.py module docstring,
    "PA per write group"), while grad_g of each entry uses its own cpe_e: two members of slot 0 with
    cpe 0.5 then 0.25, gdw = [1, 2], dva = 0: grad[0] = [0.25, 0.5]; snap = [3, 4]: grad_g = 0.5 * 11 and
    0.25 * 11."""
    k = np.array([[0], [0]], np.int32)
    grad = np.zeros((2, 2)); grad[0] = [1.0, 2.0]
    _, g_g, *_ = oracle.pa_chunk(grad, np.zeros((2, 2)), np.array([[3.0, 4.0]]), k, np.ones((2, 1)),
                                 np.zeros((2, 1)), np.array([[0.5], [0.25]]), np.ones(2), np.zeros((2, 2)), S=2, V=2)
    assert np.array_equal(grad[0], [0.25, 0.5]) and np.array_equal(g_g[:, 0], [5.5, 2.75])


def test_gds_hand_example():
    """GDS on a hand-worked chunk (mover_da2_cuda.py, "GDS, split by data need"): 3 tokens, 2 read lanes,
    V = 2 (token 2 is padding). Entries: (0,0) slot 1, (0,1) slot 3, (1,0) slot 1, (1,1) id 9 (outside S = 4).
    gr = [[1, 2], [3, -1], [7, 7]], bank rows 1 = [2, 0], 3 = [1, 1]; q = 0.5 everywhere, log_q = 0 except
    (1,0) with log_q = log 2 (sc = 1):
      d_q_w = [[<[1,2],[2,0]> = 2, <[1,2],[1,1]> = 3], [<[3,-1],[2,0]> = 6, 0], [0, 0]];
      slot 1: acc = 0.5 [1, 2] + 1 [3, -1] = [3.5, 0]; slot 3: acc = 0.5 [1, 2] = [0.5, 1]."""
    q_idx = np.array([[1, 3], [1, 9], [2, 2]], np.int32)
    q_val = np.full((3, 2), 0.5)
    log_q = np.zeros((3, 2)); log_q[1, 0] = np.log(2.0)
    gr = np.array([[1.0, 2.0], [3.0, -1.0], [7.0, 7.0]])
    bank = np.zeros((4, 2)); bank[1] = [2, 0]; bank[3] = [1, 1]; bank[2] = [5, 5]
    grad = np.full((4, 2), 10.0)
    d, mag, _ = oracle.gds_chunk(grad, bank, q_idx, q_val, log_q, gr, S=4, V=2)
    assert np.allclose(d, [[2, 3], [6, 0], [0, 0]])
    assert np.allclose(grad, [[10, 10], [13.5, 10], [10, 10], [10.5, 11]])
    assert np.all(mag[[0, 2]] == 0) and np.allclose(mag[1], [10 + 0.5 + 3, 10 + 1 + 1])


def test_gds_scatter_is_the_adjoint_of_the_weighted_read():
    """The scatter is the transpose of the read: for any rows B, sum_s <grad_after[s] - grad_before[s], B[s]>
    equals sum over valid entries of sc * <gr[t], B[slot]>, and with B = bank that is sum sc * d_q_w. A
    wrong slot, token, lane or scale on either side breaks it."""
    rng = np.random.default_rng(11)
    S, C, R, hd, V = 12, 9, 3, 6, 7
    q_idx = rng.integers(-1, S + 1, size=(C, R)).astype(np.int32)   # some ids outside [0, S)
    q_val, log_q = rng.standard_normal((C, R)), -rng.random((C, R))
    gr, bank = rng.standard_normal((C, hd)), rng.standard_normal((S, hd))
    g0 = rng.standard_normal((S, hd))
    grad = g0.copy()
    d, *_ = oracle.gds_chunk(grad, bank, q_idx, q_val, log_q, gr, S=S, V=V)
    sc = q_val * np.exp(log_q)
    valid = (q_idx >= 0) & (q_idx < S) & (np.arange(C)[:, None] < V)
    assert np.isclose(np.sum((grad - g0) * bank), np.sum(sc[valid] * d[valid]))
    B = rng.standard_normal((S, hd))
    rhs = sum(sc[t, r] * np.dot(gr[t], B[q_idx[t, r]]) for t in range(C) for r in range(R) if valid[t, r])
    assert np.isclose(np.sum((grad - g0) * B), rhs)
    assert np.all(d[~valid] == 0.0)
    # rows no valid entry reads are untouched
    unread = np.setdiff1d(np.arange(S), q_idx[valid])
    assert np.array_equal(grad[unread], g0[unread])


def test_gwr_hand_example():
    """GWR on a hand-worked chunk (pa_dc_cuda.py module docstring, "GWR"): 3 tokens, 2 write lanes, V = 2.
    grad rows 0 = [1, 0], 2 = [0, 2], 3 = [1, 1]; k_idx = [[0, 2], [3, 7 (outside S = 4)], [2, 2]];
    w = [[2, 3], [-1, 5], [9, 9]]; dv = [[1, 1], [2, -1], [4, 4]]:
      d_delta_v[0] = 2 [1, 0] + 3 [0, 2] = [2, 6]; d_delta_v[1] = -1 [1, 1] = [-1, -1]; token 2: 0;
      d_k_pd = [[<[1,1],[1,0]> = 1, <[1,1],[0,2]> = 2], [<[2,-1],[1,1]> = 1, 0], [0, 0]]."""
    grad = np.zeros((4, 2)); grad[0] = [1, 0]; grad[2] = [0, 2]; grad[3] = [1, 1]; grad[1] = [7, 7]
    k_idx = np.array([[0, 2], [3, 7], [2, 2]], np.int32)
    w = np.array([[2.0, 3.0], [-1.0, 5.0], [9.0, 9.0]])
    dv = np.array([[1.0, 1.0], [2.0, -1.0], [4.0, 4.0]])
    dd, pd, *_ = oracle.gwr_chunk(grad, k_idx, w, dv, S=4, V=2)
    assert np.allclose(dd, [[2, 6], [-1, -1], [0, 0]])
    assert np.allclose(pd, [[1, 2], [1, 0], [0, 0]])


def test_gwr_matches_a_dense_gather_matrix():
    """d_delta_v = M @ grad with M[t, s] = sum of w[t, n] over the valid lanes n with k_idx[t, n] = s (a
    library matmul), and sum_t <d_delta_v[t], dv[t]> = sum of w * d_k_pd (the two outputs agree)."""
    rng = np.random.default_rng(12)
    S, C, W, hd, V = 10, 8, 4, 5, 6
    k_idx = rng.integers(-1, S + 2, size=(C, W)).astype(np.int32)
    w, dv, grad = rng.standard_normal((C, W)), rng.standard_normal((C, hd)), rng.standard_normal((S, hd))
    dd, pd, *_ = oracle.gwr_chunk(grad, k_idx, w, dv, S=S, V=V)
    M = np.zeros((C, S))
    for t in range(V):
        for n in range(W):
            if 0 <= k_idx[t, n] < S:
                M[t, k_idx[t, n]] += w[t, n]
    assert np.allclose(dd, M @ grad)
    assert np.isclose(np.sum(dd * dv), np.sum(w * pd))
    valid = (k_idx >= 0) & (k_idx < S) & (np.arange(C)[:, None] < V)
    assert np.all(pd[~valid] == 0.0)


def _dw_vjp_case(seed=21):
    """A small chunk with repeated slots and a repeated write entry of one token, its Phase-1 rex / cpe."""
    rng = np.random.default_rng(seed)
    C, W, R, S, hd = 7, 3, 2, 5, 4
    k_idx = rng.integers(0, S, size=(C, W)).astype(np.int32)
    k_idx[2, 1] = k_idx[2, 0]                       # a token writing one slot twice
    q_idx = rng.integers(0, S, size=(C, R)).astype(np.int32)
    k_val = rng.standard_normal((C, W)).astype(np.float32)
    q_val = rng.standard_normal((C, R)).astype(np.float32)
    g = (-rng.random(C) * 0.5).astype(np.float32)
    o = oracle.phase1(k_idx[None], q_idx[None], k_val[None], q_val[None], g[None], S=S, val_dtype="f32", pairs=False)
    return C, W, S, hd, k_idx, q_idx, k_val, q_val, g, o, rng


def _dw(base, dv, k_idx, q_idx, k_val, q_val, g, S, C):
    b = base.copy()
    oracle.dw_chunk(b, k_idx, q_idx, k_val, q_val, g, dv, S=S, V=C, val_dtype="f32", bank_dtype="f32",
                    round_cpe=False, round_bank=False)
    return b


def test_gwr_is_the_vjp_of_dw_in_the_token_rows():
    """GWR with write weights k * exp(rex) (the DW record's scale) is the vector-Jacobian product of the
    forward DW (oracle.dw_chunk, exact arithmetic) with respect to the token rows dv: the DW is linear in
    dv, so <grad, DW(dv + e_ti) - DW(dv)> is d_delta_v[t, i] exactly (up to rounding)."""
    C, W, S, hd, k_idx, q_idx, k_val, q_val, g, o, rng = _dw_vjp_case()
    base = rng.standard_normal((S, hd))
    dv = rng.standard_normal((C, hd))
    grad = rng.standard_normal((S, hd))
    b0 = _dw(base, dv, k_idx, q_idx, k_val, q_val, g, S, C)
    vjp = np.zeros((C, hd))
    for t in range(C):
        for i in range(hd):
            d1 = dv.copy()
            d1[t, i] += 1.0
            vjp[t, i] = np.sum(grad * (_dw(base, d1, k_idx, q_idx, k_val, q_val, g, S, C) - b0))
    write_w = k_val.astype(np.float64) * np.exp(o["rex"][0])
    dd, *_ = oracle.gwr_chunk(grad, k_idx, write_w, dv, S=S, V=C)
    assert np.allclose(dd, vjp, rtol=1e-9, atol=1e-9)


def test_pa_decay_term_is_the_vjp_of_dw_in_the_base_rows():
    """Phase A's grad update with d_dva = 0 is the vector-Jacobian product of the forward DW with
    respect to the bank rows before the write: grad[s] * cpe_last for written slots (cpe = exp of the
    group's gate total), grad[s] unchanged elsewhere."""
    C, W, S, hd, k_idx, q_idx, k_val, q_val, g, o, rng = _dw_vjp_case(22)
    base = rng.standard_normal((S, hd))
    dv = rng.standard_normal((C, hd))
    grad = rng.standard_normal((S, hd))
    b0 = _dw(base, dv, k_idx, q_idx, k_val, q_val, g, S, C)
    vjp = np.zeros((S, hd))
    for s in range(S):
        for i in range(hd):
            b1 = base.copy()
            b1[s, i] += 1.0
            vjp[s, i] = np.sum(grad * (_dw(b1, dv, k_idx, q_idx, k_val, q_val, g, S, C) - b0))
    slots = oracle.snapshot_slots(k_idx, S=S, V=C)
    got = grad.copy()
    oracle.pa_chunk(got, np.zeros((S, hd)), np.zeros((len(slots), hd)), k_idx, k_val.astype(np.float64),
                    o["log_k"][0], o["cpe"][0], np.ones(C), np.zeros((C, hd)), S=S, V=C)
    assert np.allclose(got, vjp, rtol=1e-9, atol=1e-9)


def test_gds_is_the_vjp_of_the_weighted_read():
    """GDS is the vector-Jacobian product of the chunk's weighted read y[t] = sum_r q_w[t, r] bank[q_idx[t, r]]
    (q_w = q exp(log_q), valid tokens only) for the loss L = sum_t <gr[t], y[t]>: the scatter's change of
    the grad rows is dL/dbank, and d_q_w is dL/dq_w; both checked by unit perturbations of a read written
    here as a plain double loop."""
    rng = np.random.default_rng(13)
    S, C, R, hd, V = 6, 5, 3, 4, 4
    q_idx = rng.integers(0, S, size=(C, R)).astype(np.int32)
    q_val, log_q = rng.standard_normal((C, R)), -rng.random((C, R))
    gr, bank = rng.standard_normal((C, hd)), rng.standard_normal((S, hd))

    def loss(bk, qw):
        return sum(float(np.dot(gr[t], qw[t, r] * bk[q_idx[t, r]])) for t in range(V) for r in range(R))

    qw = q_val * np.exp(log_q)
    base = loss(bank, qw)
    d_bank = np.zeros((S, hd))
    for s in range(S):
        for i in range(hd):
            b1 = bank.copy()
            b1[s, i] += 1.0
            d_bank[s, i] = loss(b1, qw) - base
    d_qw = np.zeros((C, R))
    for t in range(C):
        for r in range(R):
            q1 = qw.copy()
            q1[t, r] += 1.0
            d_qw[t, r] = loss(bank, q1) - base
    grad = np.zeros((S, hd))
    dq, *_ = oracle.gds_chunk(grad, bank, q_idx, q_val, log_q, gr, S=S, V=V)
    assert np.allclose(grad, d_bank, rtol=1e-9, atol=1e-9)
    assert np.allclose(dq, d_qw, rtol=1e-9, atol=1e-9)


# ---- the forward's read-side gather (oracle.read_chunk) ------------------------------------------

def test_read_hand_chunk_golden():
    """The hand-worked chunk of tests/golden/hand_read_chunk.json (expressions evaluated here)."""
    fx = json.load(open(os.path.join(HERE, "golden", "hand_read_chunk.json")))
    y, _ = oracle.read_chunk(np.array(fx["bank"]), np.array(fx["q_idx"], np.int32), np.array(fx["q_w"]),
                             S=fx["S"], V=fx["V"])
    want = np.array([[eval(e) for e in row] for row in fx["y"]])   # noqa: S307 (fixture arithmetic)
    assert np.array_equal(y, want), (y, want)


def _read_by_matrix(bank, q_idx, q_w, S, V):
    """The read as one dense gather matrix G [C, S] (G[t, s] = sum of token t's q_w on slot s) applied
    to the bank by a library matmul."""
    C, R = q_idx.shape
    G = np.zeros((C, S))
    for t in range(V):
        for r in range(R):
            if 0 <= q_idx[t, r] < S:
                G[t, q_idx[t, r]] += q_w[t, r]
    return G @ bank


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_read_equals_a_dense_gather_matrix(seed):
    rng = np.random.default_rng(seed)
    S, C, R, hd, V = 11, 9, 5, 6, 7
    q_idx = rng.integers(-1, S + 2, size=(C, R)).astype(np.int32)   # some ids outside [0, S)
    q_w, bank = rng.standard_normal((C, R)), rng.standard_normal((S, hd))
    y, mag = oracle.read_chunk(bank, q_idx, q_w, S=S, V=V)
    assert np.allclose(y, _read_by_matrix(bank, q_idx, q_w, S, V), rtol=1e-12, atol=1e-12)
    assert np.all(mag >= np.abs(y) - 1e-12) and np.all(y[V:] == 0.0)


def test_read_is_the_adjoint_of_the_gds_dots():
    """<gr, read(q_w)> = sum_{t, r} d_q_w[t, r] q_w[t, r], d_q_w the GDS dots of the same chunk (GDS is
    pinned on its own: hand chunk, VJP of a plain read loop)."""
    rng = np.random.default_rng(7)
    S, C, R, hd, V = 8, 6, 4, 5, 5
    q_idx = rng.integers(0, S, size=(C, R)).astype(np.int32)
    q_val, log_q = rng.standard_normal((C, R)), -rng.random((C, R))
    gr, bank = rng.standard_normal((C, hd)), rng.standard_normal((S, hd))
    q_w = q_val * np.exp(log_q)
    y, _ = oracle.read_chunk(bank, q_idx, q_w, S=S, V=V)
    d_q_w, *_ = oracle.gds_chunk(np.zeros((S, hd)), bank, q_idx, q_val, log_q, gr, S=S, V=V)
    assert np.isclose(float(np.sum(gr * y)), float(np.sum(d_q_w * q_w)), rtol=1e-12, atol=1e-12)


def test_planted_read_mistakes_fail_the_pins():
    """A read that takes the next lane's slot, or drops the last lane, fails the matrix pin."""
    rng = np.random.default_rng(3)
    S, C, R, hd, V = 9, 6, 4, 3, 6
    q_idx = rng.integers(0, S, size=(C, R)).astype(np.int32)
    q_w, bank = rng.standard_normal((C, R)), rng.standard_normal((S, hd))
    ref = _read_by_matrix(bank, q_idx, q_w, S, V)
    shifted = oracle.read_chunk(bank, np.roll(q_idx, 1, axis=1), q_w, S=S, V=V)[0]
    dropped = oracle.read_chunk(bank, np.where(np.arange(R) == R - 1, -1, q_idx), q_w, S=S, V=V)[0]
    assert not np.allclose(shifted, ref) and not np.allclose(dropped, ref)
