"""Phase A of the backward (sdm_pa, the backward of DW) against the oracle.

Contract (pa_dc_cuda.py, module docstring, "PA per write group"): per valid write group of a chunk,
grad[s] = gdw * cpe_last + sum of -beta * k * exp(log_k) * d_dva over the members in sorted order,
bank[s] = the group's snapshot row, grad_g[e] = cpe_e <gdw, snap>, d_k_eff[e] = -beta <d_dva, snap>.
The steps run last to first, each reading the grad rows the later step wrote.

Inputs are the oracle's own: sorted_k, log_k and cpe from oracle.phase1 (log_k rounded to float32,
cpe to the value type, as the forward stores them), beta / d_dva / grad / snapshot rows from the
seeded generators; both sides get the same values.

Tolerances (float32 evaluation, u = 2^-24): a grad row after a step, n members, within
(n + 8) u * mag of the exact value (mag = |gdw cpe_last| + sum |sc d_dva|; the fmaf chain, plus the
rounding of sc = -beta (k expf(log_k)) to a few u); with bfloat16 grad rows one more bfloat16 ulp of
the result per step. Earlier steps' errors carry into later ones scaled by cpe <= 1, so the bounds
add over the steps. Dots: (hd + 8) u * sum |products| (+ |cpe_e| sum tol(gdw) |snap| for grad_g,
whose gdw carries the earlier steps' error). Bank rows, invalid entries and untouched rows: exact.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_slot_memory_gb300 as sdm
from sparse_slot_memory_gb300 import _abi
from sdm_testlib import dev_array, host, ulp_bf16
from synth import (WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_backward_inputs, make_bank_stream,
                   make_grad_stream, make_inputs, make_snapshot_chunk, scaled)

pytestmark = pytest.mark.gpu

U = 2.0 ** -24

CASES = {
    "tiny": (WORKLOADS["tiny"], "f32"),
    "uniform_c128": (scaled(WORKLOADS["uniform_c128"], P=2, T=384, S=4096), "f32"),
    "uniform_c128_bf16grad": (scaled(WORKLOADS["uniform_c128"], P=2, T=384, S=4096), "bf16"),
    "zipf_c256": (scaled(WORKLOADS["zipf_c256"], P=2, T=512, S=4096), "f32"),
    "wide_ragged": (scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=8192), "f32"),
    "wide_ragged_bf16grad": (scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=8192), "bf16"),
    # every slot of a chunk holds a group of ~40 members: groups of several 32-member windows
    "few_slots": (scaled(WORKLOADS["tiny"], P=3, T=200, C=64, S=8, hd=16, W=5, R=3, name="few_slots"), "f32"),
    # one slot per stream: one group of C*W members per chunk, two slices of 128 columns
    "one_slot": (scaled(WORKLOADS["tiny"], P=2, T=130, C=64, S=1, hd=200, W=3, R=2, name="one_slot"), "bf16"),
    # edge shapes: rows of 4 columns (one lane), single-token chunks with one read lane
    "edge_hd4": (scaled(WORKLOADS["tiny"], P=1, T=70, C=64, S=64, hd=4, W=2, R=2, name="edge_hd4"), "f32"),
    "edge_c1": (scaled(WORKLOADS["tiny"], P=2, T=3, C=1, S=16, hd=8, W=3, R=1, name="edge_c1"), "bf16"),
}


def _rnd_bf16(a):
    return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


def make_case(w, grad_dtype):
    """The inputs of both sides: a dict of numpy arrays (float64 values exactly as the GPU sees them)."""
    x = make_inputs(w)
    b = make_backward_inputs(w)
    fp = (w.steps - 1) * w.P
    o = oracle.phase1(x["k_idx"], x["q_idx"], x["k_val"], x["q_val"], x["g"], S=w.S, val_dtype=w.val_dtype,
                      first_partial=fp, valid_last=w.valid_last, pairs=False)
    rv = _rnd_bf16 if w.val_dtype == "bf16" else (lambda a: np.asarray(a, np.float32).astype(np.float64))
    kv = bf16_bits_to_f32(x["k_val"]).astype(np.float64) if w.val_dtype == "bf16" else x["k_val"].astype(np.float64)
    grad = np.stack([make_grad_stream(w, p) for p in range(w.P)], 0).astype(np.float64)
    if grad_dtype == "bf16":
        grad = _rnd_bf16(grad)
    bank = np.stack([make_bank_stream(w, p) for p in range(w.P)], 0)
    bank = bf16_bits_to_f32(bank).astype(np.float64) if w.bank_dtype == "bf16" else bank.astype(np.float64)
    snap = np.stack([make_snapshot_chunk(w, c) for c in range(w.N)], 0)
    snap = bf16_bits_to_f32(snap).astype(np.float64) if w.bank_dtype == "bf16" else snap.astype(np.float64)
    return {"x": x, "k_idx": x["k_idx"], "kv": kv, "sorted_k": o["sorted_k"],
            "log_k": np.asarray(o["log_k"], np.float32).astype(np.float64), "cpe": rv(o["cpe"]),
            "beta": b["beta"].astype(np.float64), "dva": b["dva"].astype(np.float64), "grad": grad, "bank": bank,
            "snap": snap, "grad_dtype": grad_dtype}


def to_device(w, k):
    """The case's arrays as the GPU inputs of sdm_pa."""
    def val(a):
        return dev_array(f32_to_bf16_bits(a.astype(np.float32)), "bf16") if w.val_dtype == "bf16" else \
            dev_array(a.astype(np.float32))

    def rows(a, dt):
        t = torch.from_numpy(a.astype(np.float32)).cuda()
        return t.to(torch.bfloat16) if dt == "bf16" else t

    nk = w.C * w.W
    return {
        "sorted_k": dev_array(k["sorted_k"].astype(np.int32)), "k_idx": dev_array(k["k_idx"]),
        "k_val": dev_array(k["x"]["k_val"], w.val_dtype), "log_k": dev_array(k["log_k"].astype(np.float32)),
        "cpe": val(k["cpe"]), "beta": dev_array(k["beta"].astype(np.float32)),
        "dva": dev_array(k["dva"].astype(np.float32)),
        "grad": rows(k["grad"].reshape(w.P * w.S, w.hd), k["grad_dtype"]),
        "bank": rows(k["bank"].reshape(w.P * w.S, w.hd), w.bank_dtype),
        "snap": rows(k["snap"].reshape(w.N * nk, w.hd), w.bank_dtype),
        "d_k_eff": torch.full((w.N, w.C, w.W), float("nan"), device="cuda"),
        "grad_g": torch.full((w.N, w.C, w.W), float("nan"), device="cuda"),
    }


def run_gpu(w, d, step_begin=0, step_end=None, status=None):
    shape = sdm.ShapeSpec.from_workload(w)
    step_end = w.steps if step_end is None else step_end
    nk = w.C * w.W
    snap = d["snap"][step_begin * w.P * nk:]
    sdm.pa(shape, d["sorted_k"], d["k_idx"], d["k_val"], d["log_k"], d["cpe"], d["beta"], d["dva"], d["grad"],
           d["bank"], snap, d["d_k_eff"], d["grad_g"], step_begin, step_end, status)


def run_oracle(w, k):
    """Every stream's steps last to first through oracle.pa_chunk, with the tolerance bookkeeping."""
    P, S, C, W, hd, nk = w.P, w.S, w.C, w.W, w.hd, w.C * w.W
    grad, bank = k["grad"].copy(), k["bank"].copy()
    tol = np.zeros_like(grad)             # bound on |gpu - exact| of every grad element
    d_eff = np.zeros((w.N, C, W))
    g_g = np.zeros((w.N, C, W))
    t_eff = np.zeros((w.N, C, W))
    t_g = np.zeros((w.N, C, W))
    for p in range(P):
        for ti in range(w.steps - 1, -1, -1):
            c = ti * P + p
            V = w.valid_last if ti == w.steps - 1 else C
            ids = k["k_idx"][c]
            slots = oracle.snapshot_slots(ids, S=S, V=V)
            tprev = tol[p].copy()
            de, gg, mag, dme, dmg = oracle.pa_chunk(grad[p], bank[p], k["snap"][c][:len(slots)], ids, k["kv"][c],
                                                    k["log_k"][c], k["cpe"][c], k["beta"][c], k["dva"][c], S=S, V=V)
            d_eff[c], g_g[c] = de, gg
            t_eff[c] = (hd + 8) * U * dme
            # gdw's own error, carried into <gdw, snap>
            sn = np.zeros((S, hd))
            sn[slots] = np.abs(k["snap"][c][:len(slots)])
            valid = (ids >= 0) & (ids < S) & (np.arange(C)[:, None] < V)
            carry = np.zeros((C, W))
            carry[valid] = np.sum(tprev[ids[valid]] * sn[ids[valid]], axis=1)
            t_g[c] = (hd + 8) * U * dmg + np.abs(k["cpe"][c]) * carry
            counts = np.bincount(ids[valid], minlength=S)
            step_tol = (counts[:, None] + 8) * U * mag
            if k["grad_dtype"] == "bf16":
                step_tol = step_tol + np.where(counts[:, None] > 0, ulp_bf16(np.abs(grad[p]) + step_tol), 0.0)
            tol[p] += step_tol
    return {"grad": grad, "bank": bank, "tol": tol, "d_k_eff": d_eff, "grad_g": g_g, "t_eff": t_eff, "t_g": t_g}


def check(w, k, d, ref, label):
    P, S, hd = w.P, w.S, w.hd
    got_grad = host(d["grad"]).astype(np.float64).reshape(P, S, hd)
    got_bank = host(d["bank"]).astype(np.float64).reshape(P, S, hd)
    assert np.array_equal(got_bank, ref["bank"]), f"{label}: bank rows differ from the restored snapshot rows"
    untouched = ref["tol"] == 0
    assert np.array_equal(got_grad[untouched], ref["grad"][untouched]), f"{label}: an unwritten grad row changed"
    dg = np.abs(got_grad - ref["grad"])
    bad = dg > ref["tol"]
    assert not bad.any(), f"{label}: {int(bad.sum())} grad elements beyond tolerance, worst {float(np.max(dg - ref['tol']))}"
    for f, t in (("d_k_eff", "t_eff"), ("grad_g", "t_g")):
        got = host(d[f]).astype(np.float64)
        assert np.isfinite(got).all(), f"{label}: {f} has unwritten entries"
        zero = ref[t] == 0
        assert np.array_equal(got[zero], ref[f][zero]), f"{label}: {f} of invalid entries"
        diff = np.abs(got - ref[f])
        assert (diff <= ref[t]).all(), f"{label}: {f}: {int((diff > ref[t]).sum())} entries beyond tolerance"


@pytest.mark.parametrize("name", list(CASES))
def test_pa_parity(name):
    w, gdt = CASES[name]
    k = make_case(w, gdt)
    d = to_device(w, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, d, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check(w, k, d, run_oracle(w, k), name)


def test_pa_deterministic_and_split_ranges():
    """Two runs give the same bits; [k, steps) then [0, k) gives the bits of [0, steps)."""
    w, gdt = CASES["zipf_c256"]
    k = make_case(w, gdt)
    d1, d2, d3 = to_device(w, k), to_device(w, k), to_device(w, k)
    run_gpu(w, d1)
    run_gpu(w, d2)
    split = w.steps // 2
    run_gpu(w, d3, split, w.steps)
    run_gpu(w, d3, 0, split)
    run_gpu(w, d3, 0, 0)   # an empty range does nothing
    torch.cuda.synchronize()
    for f in ("grad", "bank", "d_k_eff", "grad_g"):
        a = d1[f].view(torch.int16 if d1[f].dtype == torch.bfloat16 else torch.int32)
        for other in (d2, d3):
            b = other[f].view(torch.int16 if other[f].dtype == torch.bfloat16 else torch.int32)
            assert torch.equal(a, b), f


def test_pa_bad_slot_sets_status_and_skips_group():
    """A group whose first member's slot lies outside [0, S) (k_idx changed after the sort) is skipped
    and reported; the other groups are unaffected."""
    w, gdt = CASES["tiny"]
    k = make_case(w, gdt)
    d = to_device(w, k)
    ref_d = to_device(w, k)
    c, nk = w.N - 1, w.C * w.W
    first = int(k["sorted_k"][c][0])
    t, j = (first >> 9) & 0xFF, first & 0xFF
    s = int(k["k_idx"][c, t, j])
    d["k_idx"][c, t, j] = w.S + 5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, d, w.steps - 1, w.steps, st)
    run_gpu(w, ref_d, w.steps - 1, w.steps)
    torch.cuda.synchronize()
    assert int(st.item()) & _abi.SDM_DEV_BAD_SLOT
    g, gr = host(d["grad"]).reshape(w.P, w.S, w.hd), host(ref_d["grad"]).reshape(w.P, w.S, w.hd)
    assert np.array_equal(g[0, s], k["grad"][0, s].astype(np.float32))   # the skipped group's row
    others = np.setdiff1d(np.arange(w.S), [s])
    assert np.array_equal(g[0, others], gr[0, others])
    del nk


def test_pa_argument_errors():
    w, gdt = CASES["tiny"]
    k = make_case(w, gdt)
    d = to_device(w, k)
    shape = sdm.ShapeSpec.from_workload(w)
    args = [d[f] for f in ("sorted_k", "k_idx", "k_val", "log_k", "cpe", "beta", "dva", "grad", "bank", "snap",
                           "d_k_eff", "grad_g")]
    with pytest.raises(sdm.SdmError) as e:
        sdm.pa(shape, *args, 0, w.steps + 1)
    assert e.value.status == -1
    bad = list(args)
    bad[6] = d["dva"].view(-1)[1:]   # 4 bytes past a 16-byte boundary
    with pytest.raises(sdm.SdmError) as e:
        sdm.pa(shape, *bad)
    assert e.value.status == -4
    bad = list(args)
    bad[7] = d["grad"].to(torch.float16)
    with pytest.raises(TypeError):
        sdm.pa(shape, *bad)
    lib = _abi.load()
    import ctypes
    st = lib.sdm_pa(ctypes.byref(shape.c()), 0, *([None] * 12), 0, w.steps, None, None)
    assert st == -1
    st = lib.sdm_pa(ctypes.byref(shape.c()), 2, *[ctypes.c_void_p(a.data_ptr()) for a in args], 0, w.steps, None,
                    None)
    assert st == -3


def test_pa_fullsize_sampled():
    """The large workload (P = 32 streams, C = 256, W = 16, S = 2^20, hd = 128, f32 grad rows) at full
    size, the last two steps in one call (one launch per step, the bench's configuration): stream 31
    against the oracle on the rows it touches, every stream's outputs finite."""
    w = WORKLOADS["large"]
    P, S, C, W, hd, nk = w.P, w.S, w.C, w.W, w.hd, w.C * w.W
    b0, b1 = w.steps - 2, w.steps
    lo, hi = b0 * P, b1 * P
    x = make_inputs(w)
    bw = make_backward_inputs(w)
    o = oracle.phase1(x["k_idx"][lo:hi], x["q_idx"][lo:hi], x["k_val"][lo:hi], x["q_val"][lo:hi], x["g"][lo:hi],
                      S=S, val_dtype=w.val_dtype, first_partial=hi - lo, valid_last=w.valid_last, pairs=False)
    log_k = np.asarray(o["log_k"], np.float32)
    cpe_bits = f32_to_bf16_bits(np.asarray(o["cpe"], np.float32))
    full = lambda a, dt: np.concatenate([np.zeros((lo,) + a.shape[1:], dt), a.astype(dt)], 0)
    snap_bits = np.stack([make_snapshot_chunk(w, c) for c in range(lo, hi)], 0)
    p_chk = P - 1
    ids_p = np.concatenate([x["k_idx"][ti * P + p_chk].ravel() for ti in range(b0, b1)])
    slots = np.unique(ids_p[ids_p >= 0])
    g_rows = make_grad_stream(w, p_chk, slots)

    gen = torch.Generator(device="cuda")
    gen.manual_seed(91)
    grad = torch.randn(P * S, hd, device="cuda", generator=gen)
    rows_dev = torch.from_numpy(p_chk * S + slots.astype(np.int64)).cuda()
    grad[rows_dev] = torch.from_numpy(g_rows).cuda()
    bank = (torch.randn(P * S, hd, device="cuda", generator=gen) * w.bank_scale).to(torch.bfloat16)
    d = {"sorted_k": dev_array(full(o["sorted_k"], np.int32)), "k_idx": dev_array(x["k_idx"]),
         "k_val": dev_array(x["k_val"], "bf16"), "log_k": dev_array(full(log_k, np.float32)),
         "cpe": dev_array(full(cpe_bits, np.uint16), "bf16"), "beta": dev_array(bw["beta"]),
         "dva": dev_array(bw["dva"]), "snap": dev_array(snap_bits.reshape(-1, hd), "bf16")}
    d_k_eff = torch.full((w.N, C, W), float("nan"), device="cuda")
    grad_g = torch.full((w.N, C, W), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = sdm.ShapeSpec.from_workload(w)
    sdm.pa(shape, d["sorted_k"], d["k_idx"], d["k_val"], d["log_k"], d["cpe"], d["beta"], d["dva"], grad, bank,
           d["snap"], d_k_eff, grad_g, b0, b1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    # the oracle: stream p_chk, compact rows (slot -> its rank among the touched slots)
    kk = {c: np.where(x["k_idx"][c] >= 0, np.searchsorted(slots, x["k_idx"][c]), -1).astype(np.int32)
          for c in range(lo, hi)}
    gr = g_rows.astype(np.float64)
    bk = np.zeros_like(gr)
    kv = bf16_bits_to_f32(x["k_val"]).astype(np.float64)
    cpe = bf16_bits_to_f32(cpe_bits).astype(np.float64)
    snap = bf16_bits_to_f32(snap_bits).astype(np.float64)
    tol = np.zeros_like(gr)
    got_eff, got_g = host(d_k_eff), host(grad_g)
    for ti in range(b1 - 1, b0 - 1, -1):
        c = ti * P + p_chk
        ng = len(oracle.snapshot_slots(kk[c], S=len(slots), V=C))
        tprev = tol.copy()
        de, gg, mag, dme, dmg = oracle.pa_chunk(gr, bk, snap[c - lo][:ng], kk[c], kv[c], log_k[c - lo].astype(np.float64),
                                                cpe[c - lo], bw["beta"][c].astype(np.float64),
                                                bw["dva"][c].astype(np.float64), S=len(slots), V=C)
        counts = np.bincount(kk[c].ravel(), minlength=len(slots))
        tol += (counts[:, None] + 8) * U * mag
        assert np.all(np.abs(got_eff[c] - de) <= (hd + 8) * U * dme), f"d_k_eff of chunk {c}"
        carry = np.sum(tprev[kk[c]] * np.abs(snap[c - lo][:ng])[np.searchsorted(np.unique(kk[c]), kk[c])], axis=2)
        assert np.all(np.abs(got_g[c] - gg) <= (hd + 8) * U * dmg + np.abs(cpe[c - lo]) * carry), f"grad_g of chunk {c}"
    got = grad[rows_dev].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - gr) <= tol), "grad rows of the sampled stream"
    assert np.array_equal(bank[rows_dev].float().cpu().numpy().astype(np.float64), bk), "restored bank rows"
    assert bool(torch.isfinite(d_k_eff[lo:hi]).all()) and bool(torch.isfinite(grad_g[lo:hi]).all())
    assert bool(torch.isfinite(grad).all())
