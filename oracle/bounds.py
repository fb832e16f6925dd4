"""Rounding intervals of the stored bank rows: which stored values a float32 evaluation of the DW
update may produce, next to the exact update of the float64 oracle.

TEST INFRASTRUCTURE ONLY (like the rest of this package): only ``tests/``, the package's smoke check
and the benchmark's CPU-baseline leg may import it. It shares no code with the CUDA path.

The DW update of one bank element (mover_da2_cuda.py and mover_fx_cuda.py module docstrings) is
y = base * cpe_last + sum_m sc_m * dv[tok_m], sc_m = k_m * exp(rex_m), stored in the bank type. A
float32 evaluation -- an fmaf chain over the group's n write entries, sc = k * expf(rex) from a
float32 rex, then fmaf(base, cpe, acc) -- lands within

    delta = (n + 14 + 4 * gabs) * 2^-24 * mag,   mag = |base * cpe| + sum_m |sc_m * dv[tok_m]|,

of y, where gabs is the sum of |gate| over the group: n + 1 roundings of the chain, each at most one
unit of 2^-24 of a partial sum bounded by mag; sc within (6 + 2 * gabs) units (expf within two
float32 ulps, two roundings, rex within 2^-23 * gabs); with float32 values also cpe itself within
(6 + 2 * gabs) units of exp(group total). With bfloat16 values cpe is stored as bfloat16, the same
value as the oracle's unless exp(group total) lies within 2^-17 (relative) of a rounding boundary;
there the other rounding is a second candidate (``alt`` of the oracle's DW).

The stored value is RN(y') for some y' within Delta = carry + delta of a candidate y, carry being
the bound on the stored row's distance from the oracle's stored row before the step (0 when both
start from the same row; a later step scales it by cpe <= 1). Rounding is monotone, so the stored
value lies in [RN(y - Delta), RN(y + Delta)] (the hull over the candidates). The interval holds at
most the two bank-type neighbours of y, i.e. the stored value is within 1 ulp of the exact y,
unless Delta itself reaches past them (heavy cancellation: mag >> |y|); such elements are counted
as "relaxed".
"""

from __future__ import annotations

import numpy as np

from . import dw_chunk

U = 2.0 ** -24


def round_to(x, dtype: str) -> np.ndarray:
    """Nearest bfloat16 or float32 value (ties to even) of float64 values, as float64."""
    x = np.asarray(x, np.float64)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    shift = np.where(e - 8 < -133, e + 133, 8)   # bfloat16 subnormals: spacing 2^-133
    return np.ldexp(np.rint(np.ldexp(m, shift)), e - shift)


def ulp(x, dtype: str) -> np.ndarray:
    """Spacing of the bank type at |x| (its smallest subnormal spacing at 0)."""
    ax = np.abs(np.asarray(x, np.float64))
    bits, tiny = (8, 2.0 ** -133) if dtype == "bf16" else (24, 2.0 ** -149)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.maximum(np.exp2(e - (bits - 1)), tiny), tiny)


def group_stats(k_idx_c, g_c, *, S: int, V: int):
    """Per slot of one chunk: n = its valid write entries, gabs = the sum over the tokens writing it of
    |the token's gate on it| (g [C] per token, or [C, W] per write entry: the token's first lane)."""
    ids = np.asarray(k_idx_c, np.int64)
    n = np.zeros(S, np.int64)
    gabs = np.zeros(S)
    per_entry = np.ndim(g_c) == 2
    for t in range(V):
        row = ids[t]
        lanes = np.nonzero((row >= 0) & (row < S))[0]
        if lanes.size == 0:
            continue
        np.add.at(n, row[lanes], 1)
        slots, first = np.unique(row[lanes], return_index=True)
        gv = np.abs(np.asarray(g_c[t], np.float64)[lanes[first]]) if per_entry else np.full(slots.size, abs(float(g_c[t])))
        np.add.at(gabs, slots, gv)
    return n, gabs


def dw_step(bank, carry, k_idx_c, q_idx_c, k_val_c, q_val_c, g_c, dv_c, *, S, V, val_dtype, bank_dtype, lib=None):
    """One chunk's DW on the oracle's stored rows ``bank`` ([S, hd] float64, updated in place to the
    oracle's new stored rows) with ``carry`` ([S, hd]: bound on a GPU row's distance from ``bank``,
    updated in place). Returns, for the rows the step writes, their indices ``rows``, the exact
    update ``y``, the interval ``lo`` .. ``hi`` of the values a float32 evaluation may store and
    ``relaxed`` (elements whose interval reaches past y's bank-type neighbours)."""
    y = bank.copy()
    yalt = bank.copy()
    amb = np.zeros(S, np.int32)
    touched = np.zeros(S, np.int32)
    mag = np.zeros_like(bank)
    dw_chunk(y, k_idx_c, q_idx_c, k_val_c, q_val_c, g_c, dv_c, S=S, V=V, val_dtype=val_dtype,
             bank_dtype=bank_dtype, round_cpe=True, round_bank=False, alt=yalt, amb=amb, touched=touched,
             mag=mag, amb_rel=2.0 ** -17 if val_dtype == "bf16" else 0.0, lib=lib)
    rows = np.nonzero(touched > 0)[0]
    n, gabs = group_stats(k_idx_c, g_c, S=S, V=V)
    yr, ya = y[rows], yalt[rows]
    delta = (n[rows, None] + 14 + 4.0 * gabs[rows, None]) * U * mag[rows]
    big = carry[rows] + delta
    lo = np.minimum(round_to(yr - big, bank_dtype), round_to(ya - big, bank_dtype))
    hi = np.maximum(round_to(yr + big, bank_dtype), round_to(ya + big, bank_dtype))
    stored = round_to(yr, bank_dtype)
    u = ulp(yr, bank_dtype)
    relaxed = (hi - yr > u) | (yr - lo > u)
    carry[rows] = np.maximum(hi - stored, stored - lo)
    bank[rows] = stored
    return {"rows": rows, "y": yr, "lo": lo, "hi": hi, "relaxed": relaxed, "mag": mag[rows]}


def check_rows(got, step: dict, bank_dtype: str) -> dict:
    """Compares a GPU's stored rows (float64 values of the rows ``step['rows']``) with a step's
    interval. Returns ok (bool array), max_ulp and over_1ulp (distance from the exact y in units of
    y's spacing), relaxed (elements allowed past 1 ulp), over_1ulp_unrelaxed, max_rel (distance
    from y over mag, the scale of the float32 evaluation) and elements."""
    got = np.asarray(got, np.float64)
    y = step["y"]
    ok = (got >= step["lo"]) & (got <= step["hi"])
    d = np.abs(got - y) / ulp(y, bank_dtype)
    rel = np.abs(got - y) / np.maximum(step["mag"], 1e-300) if "mag" in step else np.zeros_like(d)
    return {"ok": ok, "max_ulp": float(d.max()) if d.size else 0.0, "over_1ulp": int((d > 1.0).sum()),
            "relaxed": int(step["relaxed"].sum()), "elements": int(d.size),
            "over_1ulp_unrelaxed": int(((d > 1.0) & ~step["relaxed"]).sum()),
            "max_rel": float(rel.max()) if rel.size else 0.0}


def dw_stream_bounds(bank, inputs, p_local, *, S, C, P, steps, valid_last, val_dtype, dv_dtype, bank_dtype,
                     step_begin=0, step_end=None, lib=None):
    """DW of steps [step_begin, step_end) of one stream on the oracle's stored rows ``bank`` (updated in
    place), from rows that a GPU shares at the start. Returns, per bank element, the interval of its
    last write (``lo``, ``hi``; the start value where never written), the exact value of that write
    ``y``, ``relaxed`` and ``writes`` (writes per row)."""
    from . import as_f64

    step_end = steps if step_end is None else step_end
    hd = bank.shape[1]
    carry = np.zeros_like(bank)
    lo, hi, y = bank.copy(), bank.copy(), bank.copy()
    relaxed = np.zeros(bank.shape, bool)
    writes = np.zeros(S, np.int32)
    for ti in range(step_begin, step_end):
        c = ti * P + p_local
        V = valid_last if ti == steps - 1 else C
        dv = as_f64(inputs["dv"][c * C:(c + 1) * C], dv_dtype).reshape(C, hd)
        st = dw_step(bank, carry, inputs["k_idx"][c], inputs["q_idx"][c], inputs["k_val"][c], inputs["q_val"][c],
                     inputs["g"][c], dv, S=S, V=V, val_dtype=val_dtype, bank_dtype=bank_dtype, lib=lib)
        r = st["rows"]
        lo[r], hi[r], y[r], relaxed[r] = st["lo"], st["hi"], st["y"], st["relaxed"]
        writes[r] += 1
    return {"lo": lo, "hi": hi, "y": y, "relaxed": relaxed, "writes": writes}
