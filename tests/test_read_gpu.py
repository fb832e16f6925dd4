"""The forward's read-side token gather (sdm_read) against the oracle (oracle.read_chunk).

Contract (include/sdm.h, sdm_read): per valid token, y[t] = sum over the read lanes r, in order, of
q_w[t, r] * bank[q_idx[t, r]] (float32 fmaf chain; ids outside [0, S) add nothing); padding tokens get
zeros. Inputs: the workload's read ids, read weights in the value dtype and bank rows from the seeded
generators; both sides get the same values.

Tolerance (float32 evaluation, u = 2^-24): y within (R + 2) u * sum |q_w * bank row| (one rounding per
fmaf of a partial sum bounded by that sum). Padding tokens: exact zeros.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import sparse_slot_memory_gb300 as sdm
from sparse_slot_memory_gb300 import _abi
from sdm_testlib import dev_array, host
from synth import WORKLOADS, bf16_bits_to_f32, make_bank_stream, make_inputs, make_read_weights, scaled

pytestmark = pytest.mark.gpu

U = 2.0 ** -24

CASES = {
    "tiny": WORKLOADS["tiny"],
    "uniform_c128": scaled(WORKLOADS["uniform_c128"], P=2, T=384, S=4096),
    "zipf_c256": scaled(WORKLOADS["zipf_c256"], P=2, T=512, S=4096),
    "large": scaled(WORKLOADS["large"], P=2, T=1024, S=8192),
    # hd = 960: eight column slices; a ragged last step
    "wide_ragged": scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=8192),
    # R = 20: two blocks of 16 read lanes; hd = 200: a second slice with half its lanes
    "r20": scaled(WORKLOADS["tiny"], P=2, T=130, C=64, S=300, hd=200, W=2, R=20, name="r20"),
    # edge shapes: rows of 4 columns (one lane), single-token chunks with one read lane, bf16 weights
    "edge_hd4": scaled(WORKLOADS["tiny"], P=1, T=70, C=64, S=64, hd=4, W=2, R=3, name="edge_hd4"),
    "edge_c1": scaled(WORKLOADS["uniform_c128"], P=2, T=3, C=1, S=16, hd=8, W=3, R=1, name="edge_c1"),
}


def make_case(w):
    x = make_inputs(w)
    qw = make_read_weights(w)
    bank = np.stack([make_bank_stream(w, p) for p in range(w.P)], 0)
    bank64 = (bf16_bits_to_f32(bank) if w.bank_dtype == "bf16" else bank).astype(np.float64)
    qw64 = (bf16_bits_to_f32(qw) if w.val_dtype == "bf16" else qw).astype(np.float64)
    return {"q_idx": x["q_idx"], "qw_raw": qw, "qw": qw64, "bank_raw": bank, "bank": bank64}


def to_device(w, k):
    return {"q_idx": dev_array(k["q_idx"]), "q_w": dev_array(k["qw_raw"], w.val_dtype),
            "bank": dev_array(k["bank_raw"].reshape(w.P * w.S, w.hd), w.bank_dtype),
            "y": torch.full((w.N, w.C, w.hd), float("nan"), device="cuda")}


def run_gpu(w, d, step_begin=0, step_end=None, status=None):
    sdm.read(sdm.ShapeSpec.from_workload(w), d["q_idx"], d["q_w"], d["bank"], d["y"], step_begin, step_end, status)


def check_chunks(w, k, got, chunks, label):
    for c in chunks:
        p, ti = c % w.P, c // w.P
        V = w.valid_last if ti == w.steps - 1 else w.C
        y, mag = oracle.read_chunk(k["bank"][p], k["q_idx"][c], k["qw"][c], S=w.S, V=V)
        assert np.all(np.abs(got[c] - y) <= (w.R + 2) * U * mag), f"{label}: y of chunk {c}"
        assert np.all(got[c][V:] == 0.0), f"{label}: padding tokens of chunk {c}"


@pytest.mark.parametrize("name", list(CASES))
def test_read_parity(name):
    w = CASES[name]
    k = make_case(w)
    d = to_device(w, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, d, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_chunks(w, k, host(d["y"]), range(w.N), name)


def test_read_ranges_write_only_their_chunks_and_are_deterministic():
    w = CASES["r20"]
    k = make_case(w)
    d1, d2 = to_device(w, k), to_device(w, k)
    run_gpu(w, d1)
    run_gpu(w, d2, 1, w.steps - 1)
    torch.cuda.synchronize()
    a, b = host(d1["y"]), host(d2["y"])
    P = w.P
    assert np.all(np.isnan(b[:P])) and np.all(np.isnan(b[(w.steps - 1) * P:])), "chunks outside the range written"
    assert np.array_equal(a[P:(w.steps - 1) * P].view(np.int32), b[P:(w.steps - 1) * P].view(np.int32))
    run_gpu(w, d2, 0, 1)
    run_gpu(w, d2, w.steps - 1, w.steps)
    torch.cuda.synchronize()
    assert np.array_equal(a.view(np.int32), host(d2["y"]).view(np.int32))


def test_read_bad_slot_and_argument_errors():
    w = CASES["tiny"]
    k = make_case(w)
    k["q_idx"] = k["q_idx"].copy()
    k["q_idx"][w.N - 1, 2, 1] = w.S + 7    # a valid token reads an id outside [0, S): it adds nothing
    d = to_device(w, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, d, w.steps - 1, w.steps, st)
    torch.cuda.synchronize()
    assert int(st.item()) & _abi.SDM_DEV_BAD_SLOT
    check_chunks(w, k, host(d["y"]), [w.N - 1], "bad slot")
    shape = sdm.ShapeSpec.from_workload(w)
    with pytest.raises(sdm.SdmError) as e:
        sdm.read(shape, d["q_idx"], d["q_w"], d["bank"], d["y"], 0, w.steps + 1)
    assert e.value.status == -1
    big = torch.zeros(w.N * w.C * w.hd + 16, device="cuda")   # a full-size output one element off alignment
    with pytest.raises(sdm.SdmError) as e:
        sdm.read(shape, d["q_idx"], d["q_w"], d["bank"], big[1:1 + w.N * w.C * w.hd], 0, w.steps)
    assert e.value.status == -4
    lib = _abi.load()
    assert lib.sdm_read(ctypes.byref(shape.c()), None, None, None, None, 0, w.steps, None, None) == -1


def test_read_fullsize_sampled():
    """The large workload (P = 32, C = 256, R = 16, S = 2^20, hd = 128, bf16 weights and bank) at full
    size, one step per call as in the forward: sampled chunks against the oracle, all outputs finite."""
    w = WORKLOADS["large"]
    P, S, C, hd = w.P, w.S, w.C, w.hd
    x = make_inputs(w)
    qw = make_read_weights(w)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(41)
    bank = (torch.randn(P * S, hd, device="cuda", generator=gen) * w.bank_scale).to(torch.bfloat16)
    y = torch.full((w.N, C, hd), float("nan"), device="cuda")
    shape = sdm.ShapeSpec.from_workload(w)
    dq, dw = dev_array(x["q_idx"]), dev_array(qw, "bf16")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in (0, w.steps - 1):
        sdm.read(shape, dq, dw, bank, y, t, t + 1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(5)
    last = (w.steps - 1) * P
    for c in sorted({0, P - 1, last, w.N - 1, *rng.integers(0, P, size=2).tolist()}):
        p = c % P
        ids = x["q_idx"][c]
        slots = np.unique(ids)
        rows = bank[torch.from_numpy(p * S + slots.astype(np.int64)).cuda()].float().cpu().numpy().astype(np.float64)
        kk = np.searchsorted(slots, ids).astype(np.int32)
        V = w.valid_last if c >= last else C
        yo, mag = oracle.read_chunk(rows, kk, bf16_bits_to_f32(qw[c]).astype(np.float64), S=len(slots), V=V)
        assert np.all(np.abs(host(y[c]) - yo) <= (w.R + 2) * U * mag), f"y of chunk {c}"
    assert bool(torch.isfinite(y[:P]).all()) and bool(torch.isfinite(y[last:]).all())
