"""Shared helpers of the parity tests: move seeded inputs to the GPU, run the library through its
C ABI, and compare with the float64 oracle within the tolerances the method's arithmetic allows.

Tolerances (derived from the arithmetic; the forward's target is 1e-4 relative for float32 and
1 bfloat16 ulp):
  * integer / index / flag outputs: bit-exact.
  * log_k, log_q, rex (float32 compensated sums of gates): |d| <= 1e-5 * sum|gate| of the group.
  * cpe, k_eff, q_w: float32 -> 1e-5 relative; bfloat16 -> 1 ulp of the exact value.
  * A, QK (float32 sums of rounded products): |d| <= 1e-4 * sum|term| of the cell (+1e-30).
  * bank: every stored element inside the interval of values a float32 evaluation of the update
    can store (oracle/bounds.py: RN of the exact update +- the derived float32 error and the error
    carried from earlier steps), which is within 1 ulp of the exact update of the bank type except
    where the derivation itself allows more (heavy cancellation, or an error carried from an earlier
    write of the row); those elements are counted. BankStats records the distance from the exact
    update in ulps and, with SDM_REPORT_DIR set, appends it to bank_ulp.jsonl there.
"""

from __future__ import annotations

import json
import os

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


class BankStats:
    """Distances of a test's stored bank elements from the exact updates (oracle/bounds.py
    check_rows results), summed over its checks; printed and, with SDM_REPORT_DIR set, appended as
    one JSON line to $SDM_REPORT_DIR/bank_ulp.jsonl."""

    def __init__(self, case: str, kind: str, bank_dtype: str):
        self.rec = {"case": case, "kind": kind, "bank_dtype": bank_dtype, "elements": 0, "max_ulp": 0.0,
                    "over_1ulp": 0, "relaxed": 0, "over_1ulp_unrelaxed": 0, "max_rel": 0.0}
        self.once = None

    def add(self, r: dict, once: dict | None = None):
        for k in ("elements", "over_1ulp", "relaxed", "over_1ulp_unrelaxed"):
            self.rec[k] += r[k]
        for k in ("max_ulp", "max_rel"):
            self.rec[k] = max(self.rec[k], r[k])
        if once is not None:
            if self.once is None:
                self.once = {"elements": 0, "max_ulp": 0.0, "over_1ulp": 0}
            self.once["elements"] += once["elements"]
            self.once["over_1ulp"] += once["over_1ulp"]
            self.once["max_ulp"] = max(self.once["max_ulp"], once["max_ulp"])

    def finish(self):
        rec = dict(self.rec)
        if self.once is not None:
            rec["rows_written_once"] = self.once
        assert rec["over_1ulp_unrelaxed"] == 0, rec
        print("bank parity", json.dumps(rec))
        d = os.environ.get("SDM_REPORT_DIR")
        if d:
            os.makedirs(d, exist_ok=True)
            with open(os.path.join(d, "bank_ulp.jsonl"), "a") as f:
                f.write(json.dumps(rec) + "\n")
        return rec
