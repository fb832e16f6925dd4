"""Shared helpers of the parity tests: move seeded inputs to the GPU, run the library through its
C ABI, and compare with the float64 oracle within the tolerances the method's arithmetic allows.

Tolerances (derived from the arithmetic; the forward's target is 1e-4 relative for float32 and
1 bfloat16 ulp):
  * integer / index / flag outputs: bit-exact.
  * log_k, log_q, rex (float32 compensated sums of gates): |d| <= 1e-5 * sum|gate| of the group.
  * cpe, k_eff, q_w: float32 -> 1e-5 relative; bfloat16 -> 1 ulp of the exact value.
  * A, QK (float32 sums of rounded products): |d| <= 1e-4 * sum|term| of the cell (+1e-30).
  * bank, one step from the oracle's own pre-step rows: float32 -> 1e-5 * mag; bfloat16 ->
    1 ulp of the exact result + 2^-17 * mag, where mag = |base * cpe| + sum |sc * dv| bounds the
    float32 evaluation error. A row whose cpe lies within 2^-17 (relative) of a bfloat16 rounding
    boundary may round either way: it also passes against the oracle's other rounding.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_slot_memory_gb300 as sdm

P1_FLOAT = ("log_k", "rex", "log_q")
P1_VAL = ("cpe", "k_eff", "q_w")
P1_INT = ("is_last", "is_only", "pos_k", "q_last", "q_only", "pos_q", "sorted_k", "sorted_q")


def ulp_bf16(x):
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    u = np.exp2(e - 7)
    return np.where(ax > 0, np.maximum(u, 2.0 ** -133), 2.0 ** -133)


def dev_array(x: np.ndarray, dtype: str = "f32") -> torch.Tensor:
    """A numpy input array on the GPU; bfloat16 arrays arrive as uint16 bit patterns."""
    x = np.ascontiguousarray(x)
    if dtype == "bf16":
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(x).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def inputs_to_dev(x: dict, w) -> dict:
    return {
        "k_idx": dev_array(x["k_idx"]), "q_idx": dev_array(x["q_idx"]),
        "k_val": dev_array(x["k_val"], w.val_dtype), "q_val": dev_array(x["q_val"], w.val_dtype),
        "g": dev_array(x["g"]), "dv": dev_array(x["dv"], w.dv_dtype),
    }


def run_phase1(shape, d: dict, ws, fields=None, step_begin=0, step_end=None):
    out = sdm.alloc_outputs(shape, fields=fields) if fields is not None else sdm.alloc_outputs(shape)
    sdm.phase1(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], out, ws, step_begin, step_end)
    torch.cuda.synchronize()
    return out


def oracle_p1(x: dict, w, chunks=None, pairs=True):
    sel = slice(None) if chunks is None else chunks
    n_all = x["k_idx"].shape[0]
    idx = np.arange(n_all)[sel]
    fp = (w.steps - 1) * x["P"]
    # the oracle takes a contiguous block of chunks; first_partial relative to the block
    lo, hi = int(idx[0]), int(idx[-1]) + 1
    return oracle.phase1(x["k_idx"][lo:hi], x["q_idx"][lo:hi], x["k_val"][lo:hi], x["q_val"][lo:hi], x["g"][lo:hi],
                         S=w.S, val_dtype=w.val_dtype, first_partial=fp - lo, valid_last=w.valid_last,
                         pairs=pairs), lo, hi


def compare_p1(gpu: dict, orc: dict, lo: int, hi: int, val_dtype: str, report: dict | None = None):
    """Asserts parity of every Phase-1 output present in ``gpu`` for chunks [lo, hi)."""
    rep = {} if report is None else report
    for f in P1_INT:
        if f not in gpu:
            continue
        g = host(gpu[f])[lo:hi]
        o = orc[f]
        bad = np.argwhere(g != o)
        assert bad.size == 0, f"{f}: {len(bad)} mismatches, first at {bad[0].tolist()}: gpu {g[tuple(bad[0])]} oracle {o[tuple(bad[0])]}"
    for f in P1_FLOAT:
        if f not in gpu:
            continue
        g = host(gpu[f])[lo:hi].astype(np.float64)
        o = orc[f]
        gabs = orc["gabs_q" if f == "log_q" else "gabs_k"]
        d = np.abs(g - o)
        tol = 1e-5 * gabs + 1e-30
        rep[f] = float(np.max(d / np.maximum(gabs, 1e-30))) if d.size else 0.0
        bad = np.argwhere(d > tol)
        assert bad.size == 0, f"{f}: {len(bad)} beyond tolerance, first {bad[0].tolist()}: gpu {g[tuple(bad[0])]} oracle {o[tuple(bad[0])]}"
    for f in P1_VAL:
        if f not in gpu:
            continue
        g = host(gpu[f])[lo:hi].astype(np.float64)
        o = orc[f]
        d = np.abs(g - o)
        if val_dtype == "bf16":
            u = ulp_bf16(o)
            rep[f + "_ulp"] = float(np.max(d / u)) if d.size else 0.0
            bad = np.argwhere(d > u)
        else:
            rep[f + "_rel"] = float(np.max(d / np.maximum(np.abs(o), 1e-30))) if d.size else 0.0
            bad = np.argwhere(d > 1e-5 * np.abs(o) + 1e-30)
        assert bad.size == 0, f"{f}: {len(bad)} beyond tolerance, first {bad[0].tolist()}: gpu {g[tuple(bad[0])]} oracle {o[tuple(bad[0])]}"
    for f in ("A", "QK"):
        if f not in gpu or f not in orc:
            continue
        g = host(gpu[f])[lo:hi].astype(np.float64)
        o = orc[f]
        a = orc[f + "_abs"]
        d = np.abs(g - o)
        rep[f] = float(np.max(d / np.maximum(a, 1e-30))) if d.size else 0.0
        bad = np.argwhere(d > 1e-4 * a + 1e-30)
        assert bad.size == 0, f"{f}: {len(bad)} beyond tolerance, first {bad[0].tolist()}: gpu {g[tuple(bad[0])]} oracle {o[tuple(bad[0])]}"
    return rep


def bank_tolerance_ok(gpu_rows, exact_rows, alt_rows, mag_rows, bank_dtype, amb_rows=None):
    """Per-element acceptance of bank rows (see the module docstring). Returns a bool mask."""
    d = np.abs(gpu_rows - exact_rows)
    if bank_dtype == "bf16":
        tol = ulp_bf16(exact_rows) + 2.0 ** -17 * mag_rows
    else:
        tol = 1e-5 * mag_rows + 1e-30
    ok = d <= tol
    if alt_rows is not None:
        da = np.abs(gpu_rows - alt_rows)
        tol_a = (ulp_bf16(alt_rows) + 2.0 ** -17 * mag_rows) if bank_dtype == "bf16" else tol
        ok |= da <= tol_a
    return ok
