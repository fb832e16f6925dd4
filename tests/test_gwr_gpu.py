"""GWR, the write side's token gather of the backward (sdm_gwr), against the oracle.

Contract (pa_dc_cuda.py, module docstring, "GWR"): per valid token, d_delta_v[t] = sum over the write
lanes n, in order, of write_w[t, n] * grad[k_idx[t, n]], and d_k_pd[t, n] = <dv[t], grad[k_idx[t, n]]>;
padding tokens get zeros. Inputs: the workload's ids and token rows, write weights and grad rows from
the seeded generators; both sides get the same values.

Tolerances (float32 evaluation, u = 2^-24): d_delta_v within (W + 4) u * sum |w * grad| (the fmaf
chain over W lanes); d_k_pd within (hd + 8) u * sum |products|. Padding entries: exact zeros.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_slot_memory_gb300 as sdm
from sparse_slot_memory_gb300 import _abi
from sdm_testlib import dev_array, host
from synth import (WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_grad_stream, make_inputs, make_write_weights,
                   scaled)

pytestmark = pytest.mark.gpu

U = 2.0 ** -24

CASES = {
    "tiny": (WORKLOADS["tiny"], "f32"),
    "uniform_c128": (scaled(WORKLOADS["uniform_c128"], P=2, T=384, S=4096), "f32"),
    "uniform_c128_bf16grad": (scaled(WORKLOADS["uniform_c128"], P=2, T=384, S=4096), "bf16"),
    "zipf_c256": (scaled(WORKLOADS["zipf_c256"], P=2, T=512, S=4096), "f32"),
    "wide_ragged": (scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=8192), "bf16"),
    # W = 20: two blocks of 16 write lanes; hd = 200: a second slice with half its lanes
    "w20": (scaled(WORKLOADS["tiny"], P=2, T=130, C=64, S=300, hd=200, W=20, R=2, name="w20"), "f32"),
    # edge shapes: rows of 4 columns (one lane), single-token chunks with one read lane
    "edge_hd4": (scaled(WORKLOADS["tiny"], P=1, T=70, C=64, S=64, hd=4, W=2, R=2, name="edge_hd4"), "f32"),
    "edge_c1": (scaled(WORKLOADS["tiny"], P=2, T=3, C=1, S=16, hd=8, W=3, R=1, name="edge_c1"), "bf16"),
}


def make_case(w, grad_dtype):
    x = make_inputs(w)
    grad = np.stack([make_grad_stream(w, p) for p in range(w.P)], 0)
    if grad_dtype == "bf16":
        grad = bf16_bits_to_f32(f32_to_bf16_bits(grad))
    dv = bf16_bits_to_f32(x["dv"]) if w.dv_dtype == "bf16" else x["dv"]
    return {"x": x, "k_idx": x["k_idx"], "write_w": make_write_weights(w), "grad": grad.astype(np.float64),
            "dv": dv.astype(np.float64).reshape(w.N, w.C, w.hd), "grad_dtype": grad_dtype}


def to_device(w, k):
    g = torch.from_numpy(k["grad"].reshape(w.P * w.S, w.hd).astype(np.float32)).cuda()
    return {"k_idx": dev_array(k["k_idx"]), "write_w": dev_array(k["write_w"]), "dv": dev_array(k["x"]["dv"], w.dv_dtype),
            "grad": g.to(torch.bfloat16) if k["grad_dtype"] == "bf16" else g,
            "d_delta_v": torch.full((w.N, w.C, w.hd), float("nan"), device="cuda"),
            "d_k_pd": torch.full((w.N, w.C, w.W), float("nan"), device="cuda")}


def run_gpu(w, d, step_begin=0, step_end=None, status=None):
    sdm.gwr(sdm.ShapeSpec.from_workload(w), d["k_idx"], d["write_w"], d["dv"], d["grad"], d["d_delta_v"], d["d_k_pd"],
            step_begin, step_end, status)


def check_chunks(w, k, d, chunks, label):
    got_dd, got_pd = host(d["d_delta_v"]), host(d["d_k_pd"])
    for c in chunks:
        p, ti = c % w.P, c // w.P
        V = w.valid_last if ti == w.steps - 1 else w.C
        dd, pd, mag, dmag = oracle.gwr_chunk(k["grad"][p], k["k_idx"][c], k["write_w"][c].astype(np.float64),
                                             k["dv"][c], S=w.S, V=V)
        t_dd = (w.W + 4) * U * mag
        t_pd = (w.hd + 8) * U * dmag
        assert np.all(np.abs(got_dd[c] - dd) <= t_dd), f"{label}: d_delta_v of chunk {c}"
        assert np.all(np.abs(got_pd[c] - pd) <= t_pd), f"{label}: d_k_pd of chunk {c}"
        assert np.all(got_dd[c][V:] == 0.0) and np.all(got_pd[c][V:] == 0.0), f"{label}: padding tokens"


@pytest.mark.parametrize("name", list(CASES))
def test_gwr_parity(name):
    w, gdt = CASES[name]
    k = make_case(w, gdt)
    d = to_device(w, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, d, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_chunks(w, k, d, range(w.N), name)


def test_gwr_deterministic_and_split_ranges():
    w, gdt = CASES["w20"]
    k = make_case(w, gdt)
    d1, d2, d3 = to_device(w, k), to_device(w, k), to_device(w, k)
    run_gpu(w, d1)
    run_gpu(w, d2)
    run_gpu(w, d3, 1, w.steps)
    run_gpu(w, d3, 0, 1)
    torch.cuda.synchronize()
    for f in ("d_delta_v", "d_k_pd"):
        for other in (d2, d3):
            assert torch.equal(d1[f].view(torch.int32), other[f].view(torch.int32)), f


def test_gwr_bad_slot_and_argument_errors():
    import ctypes
    w, gdt = CASES["tiny"]
    k = make_case(w, gdt)
    d = to_device(w, k)
    d["k_idx"][w.N - 1, 2, 1] = -5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, d, w.steps - 1, w.steps, st)
    torch.cuda.synchronize()
    assert int(st.item()) & _abi.SDM_DEV_BAD_SLOT
    assert float(d["d_k_pd"][w.N - 1, 2, 1]) == 0.0
    shape = sdm.ShapeSpec.from_workload(w)
    args = [d[f] for f in ("k_idx", "write_w", "dv", "grad", "d_delta_v", "d_k_pd")]
    with pytest.raises(sdm.SdmError) as e:
        sdm.gwr(shape, *args, 0, w.steps + 1)
    assert e.value.status == -1
    bad = list(args)
    bad[1] = d["write_w"].view(-1)[1:]
    with pytest.raises(sdm.SdmError) as e:
        sdm.gwr(shape, *bad)
    assert e.value.status == -4
    lib = _abi.load()
    assert lib.sdm_gwr(ctypes.byref(shape.c()), 0, *([None] * 6), 0, w.steps, None, None) == -1


def test_gwr_fullsize_sampled():
    """The large workload (P = 32, C = 256, W = 16, S = 2^20, hd = 128, bf16 token rows, f32 grad rows) at
    full size, the last two steps in one call: sampled chunks against the oracle, all outputs finite."""
    w = WORKLOADS["large"]
    P, S, C, W, hd = w.P, w.S, w.C, w.W, w.hd
    x = make_inputs(w)
    ww = make_write_weights(w)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(93)
    grad = torch.randn(P * S, hd, device="cuda", generator=gen)
    d_dd = torch.full((w.N, C, hd), float("nan"), device="cuda")
    d_pd = torch.full((w.N, C, W), float("nan"), device="cuda")
    b0, b1 = w.steps - 2, w.steps
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdm.gwr(sdm.ShapeSpec.from_workload(w), dev_array(x["k_idx"]), dev_array(ww), dev_array(x["dv"], "bf16"), grad,
            d_dd, d_pd, b0, b1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(4)
    for c in sorted({b0 * P, b1 * P - 1, *rng.integers(b0 * P, b1 * P, size=3).tolist()}):
        p = c % P
        ids = x["k_idx"][c]
        slots = np.unique(ids)
        rows = grad[torch.from_numpy(p * S + slots.astype(np.int64)).cuda()].cpu().numpy().astype(np.float64)
        kk = np.searchsorted(slots, ids).astype(np.int32)
        dv = bf16_bits_to_f32(x["dv"][c * C:(c + 1) * C]).astype(np.float64)
        dd, pd, mag, dmag = oracle.gwr_chunk(rows, kk, ww[c].astype(np.float64), dv, S=len(slots), V=C)
        assert np.all(np.abs(host(d_dd[c]) - dd) <= (W + 4) * U * mag), f"d_delta_v of chunk {c}"
        assert np.all(np.abs(host(d_pd[c]) - pd) <= (hd + 8) * U * dmag), f"d_k_pd of chunk {c}"
    assert bool(torch.isfinite(d_dd[b0 * P:]).all()) and bool(torch.isfinite(d_pd[b0 * P:]).all())
