"""Float64 CPU oracle of the sparse-delta-memory forward hot path (Phase 1 + DW), the saving
forward's snapshot order and the backward's Phase A, GWR and GDS.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package. It shares no code with the CUDA path and never
imports it. The forward's arithmetic lives in ``sdm_oracle.c`` (plain C, float64, straight
loops); this module builds it with the host C compiler on first use and marshals numpy arrays.
``snapshot_slots``, ``pa_chunk`` (Phase A), ``gwr_chunk`` (GWR), ``gds_chunk`` (GDS) and ``read_chunk`` (the
forward's read-side gather) are plain numpy / Python loops here.

Every function is pinned by ``tests/test_oracle_pins.py`` against brute-force and closed-form
definitions (pair sums over lane pairs, the token-sequential bank recurrence, sort positions by
Python's ``sorted``, rex/cpe closed forms, flag invariants; for Phase A a hand-worked chunk, the
single-entry closed form, linearity and the cpe_last rule; for GDS a hand-worked chunk, the
adjoint identity between the scatter and the weighted read, and the vector-Jacobian product of a
plain read loop; for GWR a hand-worked chunk and a
dense gather matrix applied by a library matmul; GWR and Phase A's decay term also as the
vector-Jacobian products of the forward DW oracle in the token rows and in the base rows; for the
read a hand-worked chunk, a dense gather matrix applied by a library matmul, and the adjoint
identity with the GDS dots).
"""

from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdm_oracle.c")
_lib = None


def build(src: str = _SRC, out_dir: str = None) -> str:
    """Compile sdm_oracle.c into oracle/_build/ (cached by source hash); returns the .so path."""
    with open(src, "rb") as f:
        tag = hashlib.sha1(f.read()).hexdigest()[:12]
    out_dir = out_dir or os.path.join(_HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, f"libsdm_oracle_{tag}.so")
    if not os.path.exists(so):
        tmp = so + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, src, "-lm"])
        os.replace(tmp, so)
    return so


def _bind(lib):
    P = ctypes.c_void_p
    i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.sdm_oracle_phase1.restype = ctypes.c_int
    lib.sdm_oracle_phase1.argtypes = [i64, i32, i32, i32, i64, i32, i32, i64] + [P] * 26
    lib.sdm_oracle_dw_chunk.restype = ctypes.c_int
    lib.sdm_oracle_dw_chunk.argtypes = ([i32, i32, i32, i32, i32, i64, i32] + [P] * 11 +
                                        [i32, i32, i32, i32, f64])
    return lib


def load_variant(so_path: str):
    """Load another build of the oracle (the pin tests use this to check that planted
    mistakes in the C source are caught)."""
    return _bind(ctypes.CDLL(so_path))


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        _lib = _bind(lib)
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Decode an input array (float32, or bfloat16 stored as uint16 bits) exactly to float64."""
    if dtype == "bf16":
        return (np.ascontiguousarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.ascontiguousarray(x, np.float32).astype(np.float64)


def phase1(k_idx, q_idx, k_val, q_val, g, *, S, val_dtype, first_partial=None, valid_last=None,
           pairs=True, lib=None):
    """Phase 1 of every chunk in the arrays (chunk-major [n, C, W] / [n, C, R], g [n, C] or [n, C, W]).

    Returns a dict of float64 / integer arrays in the output layouts of the method, plus
    ``gabs_k`` / ``gabs_q`` (sum of |gate| over each entry's group) and ``A_abs`` / ``QK_abs``
    (sum of |term| per cell) for tolerances.
    """
    lib = _load(lib)
    n, C, W = k_idx.shape
    R = q_idx.shape[2]
    g_per_entry = 1 if g.ndim == 3 else 0
    if valid_last is None:
        valid_last = C
    if first_partial is None:
        first_partial = n
    k_idx = np.ascontiguousarray(k_idx, np.int32)
    q_idx = np.ascontiguousarray(q_idx, np.int32)
    kv, qv = as_f64(k_val, val_dtype), as_f64(q_val, val_dtype)
    gg = np.ascontiguousarray(g, np.float32).astype(np.float64)
    o = {
        "log_k": np.zeros((n, C, W)), "rex": np.zeros((n, C, W)), "cpe": np.zeros((n, C, W)),
        "k_eff": np.zeros((n, C, W)), "is_last": np.zeros((n, C, W), np.int8),
        "is_only": np.zeros((n, C, W), np.int8), "pos_k": np.zeros((n, C, W), np.int32),
        "gabs_k": np.zeros((n, C, W)),
        "log_q": np.zeros((n, C, R)), "q_w": np.zeros((n, C, R)), "pos_q": np.zeros((n, C, R), np.int32),
        "q_last": np.zeros((n, C, R), np.int8), "q_only": np.zeros((n, C, R), np.int8),
        "gabs_q": np.zeros((n, C, R)),
        "sorted_k": np.zeros((n, C * W), np.int32), "sorted_q": np.zeros((n, C * R), np.int32),
    }
    if pairs:
        for k in ("A", "QK", "A_abs", "QK_abs"):
            o[k] = np.zeros((n, C, C))
    reps = np.zeros(1, np.int64)
    st = lib.sdm_oracle_phase1(
        n, C, W, R, first_partial, valid_last, g_per_entry, S, _ptr(k_idx), _ptr(q_idx), _ptr(kv),
        _ptr(qv), _ptr(gg), _ptr(o["log_k"]), _ptr(o["rex"]), _ptr(o["cpe"]), _ptr(o["k_eff"]),
        _ptr(o["is_last"]), _ptr(o["is_only"]), _ptr(o["pos_k"]), _ptr(o["gabs_k"]),
        _ptr(o["log_q"]), _ptr(o["q_w"]), _ptr(o["pos_q"]), _ptr(o["q_last"]), _ptr(o["q_only"]),
        _ptr(o["gabs_q"]), _ptr(o["sorted_k"]), _ptr(o["sorted_q"]), _ptr(o.get("A")),
        _ptr(o.get("QK")), _ptr(o.get("A_abs")), _ptr(o.get("QK_abs")), _ptr(reps))
    if st != 0:
        raise ValueError("oracle: a valid slot id is outside [0, S)")
    o["repeats"] = int(reps[0])
    return o


def dw_chunk(bank, k_idx, q_idx, k_val, q_val, g, dv, *, S, V, val_dtype, bank_dtype,
             round_cpe=True, round_bank=True, alt=None, amb=None, touched=None, mag=None, amb_rel=2.0 ** -17,
             lib=None):
    """Decay-and-write of one chunk ([C, W] / [C, R] inputs, dv [C, hd] float64) into ``bank``
    ([S, hd] float64, in place). See sdm_oracle_dw_chunk for ``alt`` / ``amb`` / ``touched``."""
    lib = _load(lib)
    C, W = k_idx.shape
    R = q_idx.shape[1]
    hd = bank.shape[1]
    assert bank.dtype == np.float64 and bank.flags.c_contiguous and bank.shape[0] == S
    g_per_entry = 1 if np.ndim(g) == 2 else 0
    k_idx = np.ascontiguousarray(k_idx, np.int32)
    q_idx = np.ascontiguousarray(q_idx, np.int32)
    kv, qv = as_f64(k_val, val_dtype), as_f64(q_val, val_dtype)
    gg = np.ascontiguousarray(g, np.float32).astype(np.float64)
    dvv = np.ascontiguousarray(dv, np.float64)
    st = lib.sdm_oracle_dw_chunk(C, W, R, V, g_per_entry, S, hd, _ptr(k_idx), _ptr(q_idx), _ptr(kv),
                                 _ptr(qv), _ptr(gg), _ptr(dvv), _ptr(bank), _ptr(alt), _ptr(amb),
                                 _ptr(touched), _ptr(mag), int(round_cpe), int(val_dtype == "bf16"),
                                 int(round_bank), int(bank_dtype == "bf16"), float(amb_rel))
    if st != 0:
        raise ValueError("oracle: a valid slot id is outside [0, S)")


def snapshot_slots(k_idx_c, *, S, V):
    """The dense compact snapshot's row order of one chunk (mover_da2_cuda.py, the WR mode of the DW
    walk; mover_fx_cuda.py module docstring): a valid write group's row is its dense ordinal, the
    number of the chunk's valid write groups before it in sorted order. Groups are slots with at
    least one valid write entry (token t < V, id in [0, S)); sorted order is slot order. Returns the
    slots by ordinal."""
    ids = np.asarray(k_idx_c)[:V].ravel().astype(np.int64)
    return np.unique(ids[(ids >= 0) & (ids < S)])


def dw_stream(bank, inputs, p_local, *, S, C, P, steps, valid_last, val_dtype, dv_dtype, bank_dtype,
              step_begin=0, step_end=None, round_cpe=True, round_bank=True, track=False, snaps=None):
    """DW of every step in [step_begin, step_end) of one stream, in step order.

    ``inputs`` holds chunk-major arrays of P streams (as synth.make_inputs returns); ``p_local`` is
    the stream's index among them. ``bank`` is that stream's [S, hd] float64 rows (updated in place).
    With ``track`` returns (alt, amb, touched, mag) for tolerance bookkeeping.
    With ``snaps`` (a list) appends, per chunk, its snapshot slots and their rows before the chunk's
    DW (and, with ``track``, the same bookkeeping for those rows plus ``peak``, the largest |value|
    each row has held so far).
    """
    step_end = steps if step_end is None else step_end
    hd = bank.shape[1]
    alt = bank.copy() if track else None
    amb = np.zeros(S, np.int32) if track else None
    touched = np.zeros(S, np.int32) if track else None
    mag = np.zeros_like(bank) if track else None
    peak = np.abs(bank) if (snaps is not None and track) else None   # largest |value| each row has held
    for ti in range(step_begin, step_end):
        c = ti * P + p_local
        V = valid_last if ti == steps - 1 else C
        dv = as_f64(inputs["dv"][c * C:(c + 1) * C], dv_dtype).reshape(C, hd)
        if snaps is not None:   # the saving forward: the groups' base rows before this step
            sl = snapshot_slots(inputs["k_idx"][c], S=S, V=V)
            snaps.append({"c": c, "slots": sl, "rows": bank[sl].copy(),
                          **({"alt": alt[sl].copy(), "amb": amb[sl].copy(), "touched": touched[sl].copy(),
                              "mag": mag[sl].copy(), "peak": peak[sl].copy()} if track else {})})
        dw_chunk(bank, inputs["k_idx"][c], inputs["q_idx"][c], inputs["k_val"][c], inputs["q_val"][c],
                 inputs["g"][c], dv, S=S, V=V, val_dtype=val_dtype, bank_dtype=bank_dtype,
                 round_cpe=round_cpe, round_bank=round_bank, alt=alt, amb=amb, touched=touched, mag=mag)
        if peak is not None:
            np.maximum(peak, np.abs(bank), out=peak)
    if track:
        return alt, amb, touched, mag
    return None


def pa_chunk(grad, bank, snap_rows, k_idx_c, k_val_c, log_k_c, cpe_c, beta_c, dva_c, *, S, V):
    """Phase A, the backward of DW, for one chunk (pa_dc_cuda.py, module docstring: "PA per write
    group"). Float64, plain loops over the chunk's slot groups.

    Per valid write group (slot s with valid write entries; members in sorted order, i.e. token then
    lane), with gdw = grad[s] before this step and snap = the group's row of the dense snapshot
    (snap_rows[g], g = the group's ordinal in slot order):
      sc_m = -beta[tok_m] * k_m * exp(log_k_m)            (the records' scale)
      grad[s] = gdw * cpe_last + sum_m sc_m * dva[tok_m]  (cpe_last: the last member's cpe)
      bank[s] = snap                                      (the pre-write row restored)
      grad_g[e] = cpe_e * <gdw, snap>,  d_k_eff[e] = -beta[tok_e] * <dva[tok_e], snap>
    Inputs: grad / bank [S, hd] float64 (updated in place), snap_rows [G, hd], k_idx_c / k_val_c /
    log_k_c / cpe_c [C, W], beta_c [C], dva_c [C, hd]; tokens t >= V and ids outside [0, S) have
    no group. Returns (d_k_eff [C, W], grad_g [C, W], mag [S, hd], dmag_eff [C, W], dmag_g [C, W]):
    mag = |gdw * cpe_last| + sum_m |sc_m * dva| of each written grad row (zero elsewhere), dmag_* = the
    dots' sums of |products| (tolerance bookkeeping).
    """
    C, W = k_idx_c.shape
    hd = grad.shape[1]
    ids = np.asarray(k_idx_c, np.int64)
    d_k_eff = np.zeros((C, W))
    grad_g = np.zeros((C, W))
    dmag_eff = np.zeros((C, W))
    dmag_g = np.zeros((C, W))
    mag = np.zeros_like(grad)
    slots = snapshot_slots(ids, S=S, V=V)
    groups = {int(s): [] for s in slots}
    for t in range(V):                    # entry order (token, then lane) is the sorted order within a slot
        for j in range(W):
            if int(ids[t, j]) in groups:
                groups[int(ids[t, j])].append((t, j))
    for g, s in enumerate(slots):
        members = groups[int(s)]
        gdw = grad[s].copy()
        snap = np.asarray(snap_rows[g], np.float64)
        cpe = float(cpe_c[members[-1]])     # cpe_last
        acc = np.zeros(hd)
        aabs = np.zeros(hd)
        for (t, j) in members:
            sc = -float(beta_c[t]) * float(k_val_c[t, j]) * np.exp(float(log_k_c[t, j]))
            acc += sc * dva_c[t]
            aabs += np.abs(sc * dva_c[t])
        gdot = float(np.dot(gdw, snap))
        for (t, j) in members:
            grad_g[t, j] = float(cpe_c[t, j]) * gdot
            dmag_g[t, j] = abs(float(cpe_c[t, j])) * float(np.sum(np.abs(gdw * snap)))
            d_k_eff[t, j] = -float(beta_c[t]) * float(np.dot(dva_c[t], snap))
            dmag_eff[t, j] = abs(float(beta_c[t])) * float(np.sum(np.abs(dva_c[t] * snap)))
        grad[s] = gdw * cpe + acc
        mag[s] = np.abs(gdw * cpe) + aabs
        bank[s] = snap
    return d_k_eff, grad_g, mag, dmag_eff, dmag_g


def gds_chunk(grad, bank, q_idx_c, q_val_c, log_q_c, gr_c, *, S, V):
    """GDS, the read side of the backward, for one chunk (mover_da2_cuda.py, module docstring and the
    "GDS, split by data need" comment; the read records of its qrec kernel). Float64, plain loops.

    (1) dots in token order: d_q_w[t, r] = <gr[t], bank[q_idx[t, r]]> for every valid token t < V
        (0 for padding tokens and for ids outside [0, S));
    (2) the grad scatter: per read group (slot s with valid read entries; members in sorted order, i.e.
        token then lane) acc = sum_m sc_m * gr[tok_m], sc = q * exp(log_q) (the read record's scale),
        and grad[s] = grad[s] + acc, once per group.
    Inputs: grad / bank [S, hd] float64 (grad updated in place), q_idx_c / q_val_c / log_q_c [C, R],
    gr_c [C, hd]. Returns (d_q_w [C, R], mag [S, hd], dmag [C, R]): mag = |grad before| + sum |sc * gr|
    of each updated row (zero elsewhere), dmag = sum |products| of each dot (tolerance bookkeeping).
    """
    C, R = q_idx_c.shape
    ids = np.asarray(q_idx_c, np.int64)
    d_q_w = np.zeros((C, R))
    dmag = np.zeros((C, R))
    groups = {}
    for t in range(V):
        for r in range(R):
            s = int(ids[t, r])
            if 0 <= s < S:
                d_q_w[t, r] = float(np.dot(gr_c[t], bank[s]))
                dmag[t, r] = float(np.sum(np.abs(gr_c[t] * bank[s])))
                groups.setdefault(s, []).append((t, r))
    mag = np.zeros_like(grad)
    for s in sorted(groups):
        acc = np.zeros(grad.shape[1])
        aabs = np.zeros(grad.shape[1])
        for (t, r) in groups[s]:
            sc = float(q_val_c[t, r]) * np.exp(float(log_q_c[t, r]))
            acc += sc * gr_c[t]
            aabs += np.abs(sc * gr_c[t])
        mag[s] = np.abs(grad[s]) + aabs
        grad[s] = grad[s] + acc
    return d_q_w, mag, dmag


def gwr_chunk(grad, k_idx_c, write_w_c, dv_c, *, S, V):
    """GWR, the write side's token gather of the backward, for one chunk (pa_dc_cuda.py, module
    docstring: "GWR"). Float64, plain loops over tokens and their write lanes in order.

    For every valid token t < V: d_delta_v[t] = sum over lanes n of write_w[t, n] * grad[k_idx[t, n]]
    and d_k_pd[t, n] = <dv[t], grad[k_idx[t, n]]> (ids outside [0, S) add nothing and get 0); padding
    tokens get zeros. Inputs: grad [S, hd] (read only), k_idx_c / write_w_c [C, W], dv_c [C, hd].
    Returns (d_delta_v [C, hd], d_k_pd [C, W], mag [C, hd], dmag [C, W]): mag = sum |w * grad row| per
    token, dmag = sum |products| per dot (tolerance bookkeeping).
    """
    C, W = k_idx_c.shape
    hd = grad.shape[1]
    d_delta_v = np.zeros((C, hd))
    mag = np.zeros((C, hd))
    d_k_pd = np.zeros((C, W))
    dmag = np.zeros((C, W))
    for t in range(V):
        for n in range(W):
            s = int(k_idx_c[t, n])
            if 0 <= s < S:
                d_delta_v[t] += float(write_w_c[t, n]) * grad[s]
                mag[t] += np.abs(float(write_w_c[t, n]) * grad[s])
                d_k_pd[t, n] = float(np.dot(dv_c[t], grad[s]))
                dmag[t, n] = float(np.sum(np.abs(dv_c[t] * grad[s])))
    return d_delta_v, d_k_pd, mag, dmag


def read_chunk(bank, q_idx_c, q_w_c, *, S, V):
    """The forward's read-side token gather for one chunk: the weighted read of the bank rows at the
    chunk's read entries, the operand of the GDS dots (mover_da2_cuda.py, module docstring: GDS
    d_q_w[t, r] = <gr[t], bank[slot]>, the vector-Jacobian product of this read in q_w; the same
    token_gather form as GWR's d_delta_v in pa_dc_cuda.py's module docstring). Float64, plain loops
    over tokens and their read lanes in order.

    For every valid token t < V: y[t] = sum over lanes r of q_w[t, r] * bank[q_idx[t, r]] (ids outside
    [0, S) add nothing); padding tokens get zeros. Inputs: bank [S, hd] (the rows as they are before
    the chunk's DW), q_idx_c / q_w_c [C, R]. Returns (y [C, hd], mag [C, hd]): mag = sum |q_w * bank
    row| per token (tolerance bookkeeping).
    """
    C, R = q_idx_c.shape
    hd = bank.shape[1]
    y = np.zeros((C, hd))
    mag = np.zeros((C, hd))
    for t in range(V):
        for r in range(R):
            s = int(q_idx_c[t, r])
            if 0 <= s < S:
                y[t] += float(q_w_c[t, r]) * bank[s]
                mag[t] += np.abs(float(q_w_c[t, r]) * bank[s])
    return y, mag
