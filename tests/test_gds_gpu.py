"""GDS, the read side of the backward (sdm_gds), against the oracle.

Contract (mover_da2_cuda.py, module docstring and the "GDS, split by data need" comment): per chunk,
d_q_w[t, r] = <gr[t], bank[q_idx[t, r]]> for the valid tokens (0 for padding tokens), and per read
group grad[s] += sum of q * exp(log_q) * gr[tok] over the members in sorted order, rounded once.
The steps run last to first.

Inputs are the oracle's own: sorted_q and log_q from oracle.phase1 (log_q rounded to float32, as the
forward stores it), gr / grad / bank rows from the seeded generators; both sides get the same values.

Tolerances (float32 evaluation, u = 2^-24): d_q_w within (hd + 8) u * sum |products| (the bank and gr
are exact inputs); a grad row after a step, n read members, within (n + 8) u * mag of the exact value
(mag = |grad before| + sum |sc gr|: the fmaf chain, sc = q expf(log_q) to a few u, the final add);
with bfloat16 grad rows one more bfloat16 ulp of the result per step; the bounds of the steps add.
Rows no valid read entry touches: exact.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_slot_memory_gb300 as sdm
from sparse_slot_memory_gb300 import _abi
from sdm_testlib import dev_array, host, ulp_bf16
from synth import (WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_bank_stream, make_grad_stream, make_inputs,
                   make_read_grads, scaled)

pytestmark = pytest.mark.gpu

U = 2.0 ** -24

CASES = {
    "tiny": (WORKLOADS["tiny"], "f32"),
    "uniform_c128": (scaled(WORKLOADS["uniform_c128"], P=2, T=384, S=4096), "f32"),
    "uniform_c128_bf16grad": (scaled(WORKLOADS["uniform_c128"], P=2, T=384, S=4096), "bf16"),
    # hot read slots: groups of more than 32 members, walked past the warp's positions
    "zipf_c256": (scaled(WORKLOADS["zipf_c256"], P=2, T=512, S=4096), "f32"),
    # 8 slices of 128 columns, a ragged last step (padding tokens)
    "wide_ragged": (scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=8192), "bf16"),
    "few_slots": (scaled(WORKLOADS["tiny"], P=3, T=200, C=64, S=8, hd=16, W=5, R=3, name="few_slots"), "f32"),
    # R = 20: a token's entries span two blocks of 16 dots; two slices, one with half its lanes
    "r20": (scaled(WORKLOADS["tiny"], P=2, T=130, C=64, S=300, hd=200, W=2, R=20, name="r20"), "f32"),
    # edge shapes: rows of 4 columns (one lane), single-token chunks with one read lane
    "edge_hd4": (scaled(WORKLOADS["tiny"], P=1, T=70, C=64, S=64, hd=4, W=2, R=2, name="edge_hd4"), "f32"),
    "edge_c1": (scaled(WORKLOADS["tiny"], P=2, T=3, C=1, S=16, hd=8, W=3, R=1, name="edge_c1"), "bf16"),
}


def _rnd_bf16(a):
    return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


def make_case(w, grad_dtype):
    x = make_inputs(w)
    fp = (w.steps - 1) * w.P
    o = oracle.phase1(x["k_idx"], x["q_idx"], x["k_val"], x["q_val"], x["g"], S=w.S, val_dtype=w.val_dtype,
                      first_partial=fp, valid_last=w.valid_last, pairs=False)
    qv = bf16_bits_to_f32(x["q_val"]).astype(np.float64) if w.val_dtype == "bf16" else x["q_val"].astype(np.float64)
    grad = np.stack([make_grad_stream(w, p) for p in range(w.P)], 0).astype(np.float64)
    if grad_dtype == "bf16":
        grad = _rnd_bf16(grad)
    bank = np.stack([make_bank_stream(w, p) for p in range(w.P)], 0)
    bank = bf16_bits_to_f32(bank).astype(np.float64) if w.bank_dtype == "bf16" else bank.astype(np.float64)
    return {"x": x, "q_idx": x["q_idx"], "qv": qv, "sorted_q": o["sorted_q"],
            "log_q": np.asarray(o["log_q"], np.float32).astype(np.float64),
            "gr": make_read_grads(w).astype(np.float64), "grad": grad, "bank": bank, "grad_dtype": grad_dtype}


def to_device(w, k):
    def rows(a, dt):
        t = torch.from_numpy(a.astype(np.float32)).cuda()
        return t.to(torch.bfloat16) if dt == "bf16" else t

    return {
        "sorted_q": dev_array(k["sorted_q"].astype(np.int32)), "q_idx": dev_array(k["q_idx"]),
        "q_val": dev_array(k["x"]["q_val"], w.val_dtype), "log_q": dev_array(k["log_q"].astype(np.float32)),
        "gr": dev_array(k["gr"].astype(np.float32)),
        "bank": rows(k["bank"].reshape(w.P * w.S, w.hd), w.bank_dtype),
        "grad": rows(k["grad"].reshape(w.P * w.S, w.hd), k["grad_dtype"]),
        "d_q_w": torch.full((w.N, w.C, w.R), float("nan"), device="cuda"),
    }


def run_gpu(w, d, step_begin=0, step_end=None, status=None):
    shape = sdm.ShapeSpec.from_workload(w)
    sdm.gds(shape, d["sorted_q"], d["q_idx"], d["q_val"], d["log_q"], d["gr"], d["bank"], d["grad"], d["d_q_w"],
            step_begin, step_end, status)


def run_oracle(w, k):
    P, S, C, R = w.P, w.S, w.C, w.R
    grad = k["grad"].copy()
    tol = np.zeros_like(grad)
    d = np.zeros((w.N, C, R))
    td = np.zeros((w.N, C, R))
    for p in range(P):
        for ti in range(w.steps - 1, -1, -1):
            c = ti * P + p
            V = w.valid_last if ti == w.steps - 1 else C
            ids = k["q_idx"][c]
            dq, mag, dmag = oracle.gds_chunk(grad[p], k["bank"][p], ids, k["qv"][c], k["log_q"][c], k["gr"][c], S=S, V=V)
            d[c] = dq
            td[c] = (w.hd + 8) * U * dmag
            valid = (ids >= 0) & (ids < S) & (np.arange(C)[:, None] < V)
            counts = np.bincount(ids[valid], minlength=S)
            step_tol = (counts[:, None] + 8) * U * mag
            if k["grad_dtype"] == "bf16":
                step_tol = step_tol + np.where(counts[:, None] > 0, ulp_bf16(np.abs(grad[p]) + step_tol), 0.0)
            tol[p] += step_tol
    return {"grad": grad, "tol": tol, "d_q_w": d, "t_d": td}


def check(w, d, ref, label):
    got = host(d["grad"]).astype(np.float64).reshape(w.P, w.S, w.hd)
    untouched = ref["tol"] == 0
    assert np.array_equal(got[untouched], ref["grad"][untouched]), f"{label}: an unread grad row changed"
    dg = np.abs(got - ref["grad"])
    bad = dg > ref["tol"]
    assert not bad.any(), f"{label}: {int(bad.sum())} grad elements beyond tolerance"
    gq = host(d["d_q_w"]).astype(np.float64)
    assert np.isfinite(gq).all(), f"{label}: d_q_w has unwritten entries"
    zero = ref["t_d"] == 0
    assert np.array_equal(gq[zero], ref["d_q_w"][zero]), f"{label}: d_q_w of padding entries"
    diff = np.abs(gq - ref["d_q_w"])
    assert (diff <= ref["t_d"]).all(), f"{label}: {int((diff > ref['t_d']).sum())} d_q_w entries beyond tolerance"


@pytest.mark.parametrize("name", list(CASES))
def test_gds_parity(name):
    w, gdt = CASES[name]
    k = make_case(w, gdt)
    d = to_device(w, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, d, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check(w, d, run_oracle(w, k), name)


def test_gds_deterministic_and_split_ranges():
    """Two runs give the same bits; [k, steps) then [0, k) gives the bits of [0, steps)."""
    w, gdt = CASES["zipf_c256"]
    k = make_case(w, gdt)
    d1, d2, d3 = to_device(w, k), to_device(w, k), to_device(w, k)
    run_gpu(w, d1)
    run_gpu(w, d2)
    split = w.steps // 2
    run_gpu(w, d3, split, w.steps)
    run_gpu(w, d3, 0, split)
    run_gpu(w, d3, 0, 0)
    torch.cuda.synchronize()
    for f in ("grad", "d_q_w"):
        a = d1[f].view(torch.int32)
        for other in (d2, d3):
            assert torch.equal(a, other[f].view(torch.int32)), f


def test_gds_bad_slot_sets_status():
    """A valid token's read id outside [0, S) (q_idx changed after the sort): the status bit is set, the
    entry's dot is 0, and the other entries are unaffected."""
    w, gdt = CASES["tiny"]
    k = make_case(w, gdt)
    d, ref_d = to_device(w, k), to_device(w, k)
    c, t, r = w.N - 1, 3, 1
    d["q_idx"][c, t, r] = w.S + 7
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, d, w.steps - 1, w.steps, st)
    run_gpu(w, ref_d, w.steps - 1, w.steps)
    torch.cuda.synchronize()
    assert int(st.item()) & _abi.SDM_DEV_BAD_SLOT
    a, b = host(d["d_q_w"]), host(ref_d["d_q_w"])
    assert a[c, t, r] == 0.0
    mask = np.ones(a.shape, bool)
    mask[c, t, r] = False
    assert np.array_equal(a[w.N - w.P:][mask[w.N - w.P:]], b[w.N - w.P:][mask[w.N - w.P:]])


def test_gds_argument_errors():
    import ctypes
    w, gdt = CASES["tiny"]
    k = make_case(w, gdt)
    d = to_device(w, k)
    shape = sdm.ShapeSpec.from_workload(w)
    args = [d[f] for f in ("sorted_q", "q_idx", "q_val", "log_q", "gr", "bank", "grad", "d_q_w")]
    with pytest.raises(sdm.SdmError) as e:
        sdm.gds(shape, *args, 2, 1)
    assert e.value.status == -1
    bad = list(args)
    bad[4] = d["gr"].view(-1)[2:]   # 8 bytes past a 16-byte boundary
    with pytest.raises(sdm.SdmError) as e:
        sdm.gds(shape, *bad)
    assert e.value.status == -4
    lib = _abi.load()
    assert lib.sdm_gds(ctypes.byref(shape.c()), 0, *([None] * 8), 0, w.steps, None, None) == -1
    ptrs = [ctypes.c_void_p(a.data_ptr()) for a in args]
    assert lib.sdm_gds(ctypes.byref(shape.c()), 5, *ptrs, 0, w.steps, None, None) == -3


def test_gds_fullsize_sampled():
    """The large workload (P = 32, C = 256, R = 16, S = 2^20, hd = 128, f32 grad rows) at full size, the
    last two steps in one call (the bench's launch configuration): stream 31 against the oracle on the
    rows it reads, every stream's outputs finite."""
    w = WORKLOADS["large"]
    P, S, C, R, hd = w.P, w.S, w.C, w.R, w.hd
    b0, b1 = w.steps - 2, w.steps
    lo, hi = b0 * P, b1 * P
    x = make_inputs(w)
    o = oracle.phase1(x["k_idx"][lo:hi], x["q_idx"][lo:hi], x["k_val"][lo:hi], x["q_val"][lo:hi], x["g"][lo:hi],
                      S=S, val_dtype=w.val_dtype, first_partial=hi - lo, valid_last=w.valid_last, pairs=False)
    log_q = np.asarray(o["log_q"], np.float32)
    full = lambda a, dt: np.concatenate([np.zeros((lo,) + a.shape[1:], dt), a.astype(dt)], 0)
    gr = make_read_grads(w)
    p_chk = P - 1
    ids_p = np.concatenate([x["q_idx"][ti * P + p_chk].ravel() for ti in range(b0, b1)])
    slots = np.unique(ids_p[ids_p >= 0])
    g_rows = make_grad_stream(w, p_chk, slots)
    b_rows = bf16_bits_to_f32(make_bank_stream(w, p_chk)[slots])

    gen = torch.Generator(device="cuda")
    gen.manual_seed(92)
    grad = torch.randn(P * S, hd, device="cuda", generator=gen)
    bank = (torch.randn(P * S, hd, device="cuda", generator=gen) * w.bank_scale).to(torch.bfloat16)
    rows_dev = torch.from_numpy(p_chk * S + slots.astype(np.int64)).cuda()
    grad[rows_dev] = torch.from_numpy(g_rows).cuda()
    bank[rows_dev] = torch.from_numpy(b_rows).cuda().to(torch.bfloat16)
    d_q_w = torch.full((w.N, C, R), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdm.gds(sdm.ShapeSpec.from_workload(w), dev_array(full(o["sorted_q"], np.int32)), dev_array(x["q_idx"]),
            dev_array(x["q_val"], "bf16"), dev_array(full(log_q, np.float32)), dev_array(gr), bank, grad, d_q_w, b0,
            b1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    kk = {c: np.where(x["q_idx"][c] >= 0, np.searchsorted(slots, x["q_idx"][c]), -1).astype(np.int32)
          for c in range(lo, hi)}
    gref = g_rows.astype(np.float64)
    bref = b_rows.astype(np.float64)
    qv = bf16_bits_to_f32(x["q_val"]).astype(np.float64)
    tol = np.zeros_like(gref)
    got_d = host(d_q_w)
    for ti in range(b1 - 1, b0 - 1, -1):
        c = ti * P + p_chk
        dq, mag, dmag = oracle.gds_chunk(gref, bref, kk[c], qv[c], log_q[c - lo].astype(np.float64),
                                         gr[c].astype(np.float64), S=len(slots), V=C)
        assert np.all(np.abs(got_d[c] - dq) <= (hd + 8) * U * dmag), f"d_q_w of chunk {c}"
        counts = np.bincount(kk[c].ravel(), minlength=len(slots))
        tol += (counts[:, None] + 8) * U * mag
    got = grad[rows_dev].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - gref) <= tol), "grad rows of the sampled stream"
    assert bool(torch.isfinite(d_q_w[lo:hi]).all()) and bool(torch.isfinite(grad).all())
