"""The saving forward (sdm_forward_chunks_saving / sdm_dw_saving) against the oracle.

The DW of the saving forward also copies, for every valid write group of a chunk, the group's
base row (the bank row before this step's write) into the dense compact snapshot at row
c * (C*W) + g, g = the group's dense ordinal (mover_da2_cuda.py, the WR mode of the DW walk;
mover_fx_cuda.py module docstring). Checked here:
  * ngroups[c] and the row order: exact against the oracle's group list of the chunk;
  * the snapshot rows: within the bank tolerance of the oracle's rows before the step (the GPU's
    own pre-step bank is within that tolerance of the oracle's), and rows past ngroups untouched;
  * the raw-copy identity: the snapshot rows of step t are bit-equal to the bank rows after a
    forward of steps [0, t) (the same kernels, run to that step);
  * the bank: bit-equal to the plain forward's.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_slot_memory_gb300 as sdm
from sdm_testlib import host, inputs_to_dev, ulp_bf16
from synth import WORKLOADS, bf16_bits_to_f32, make_bank_stream, make_inputs, scaled

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": WORKLOADS["tiny"],
    "uniform_c128": scaled(WORKLOADS["uniform_c128"], P=2, T=768, S=4096),
    "zipf_c256": scaled(WORKLOADS["zipf_c256"], P=2, T=1024, S=4096),
    "wide_ragged": scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=8192),
    "few_slots": scaled(WORKLOADS["tiny"], P=3, T=200, C=64, S=8, hd=16, W=5, R=3, name="few_slots"),
}
SENTINEL = {"bf16": 0x7FC1, "f32": 0x7FC00001}   # NaN bit patterns the DW never writes


def _bank(w):
    rows = [make_bank_stream(w, p) for p in range(w.P)]
    rows = [bf16_bits_to_f32(r) if w.bank_dtype == "bf16" else r for r in rows]
    t = torch.from_numpy(np.stack(rows, 0).reshape(w.P * w.S, w.hd).astype(np.float32)).cuda()
    return t.to(torch.bfloat16) if w.bank_dtype == "bf16" else t


def _raw(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def _snap(shape, w):
    s = sdm.alloc_snapshot(shape)
    _raw(s).fill_(SENTINEL[w.bank_dtype])   # both patterns fit the signed raw views
    return s


@pytest.mark.parametrize("name", list(CASES))
def test_saving_forward_snapshot(name):
    w = CASES[name]
    x = make_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)
    d = inputs_to_dev(x, w)
    P, S, C, hd, nk = w.P, w.S, w.C, w.hd, w.C * w.W
    ws = sdm.alloc_workspace(shape)
    out = sdm.alloc_outputs(shape, fields=("ngroups", "repeats"))
    bank = _bank(w)
    snap = _snap(shape, w)
    sentinel = _raw(snap).clone()
    sdm.forward_chunks_saving(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, snap,
                              out, ws)
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0

    # the bank is the plain forward's, bit for bit
    ws2 = sdm.alloc_workspace(shape)
    bank2 = _bank(w)
    sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank2, None, ws2)
    torch.cuda.synchronize()
    assert torch.equal(_raw(bank), _raw(bank2))

    ng = host(out["ngroups"])
    snap_h = host(snap).astype(np.float64).reshape(w.N, nk, hd)
    snap_raw = host(_raw(snap)).reshape(w.N, nk, hd)
    sent_raw = host(sentinel).reshape(w.N, nk, hd)
    for p in range(P):
        init = make_bank_stream(w, p)
        ref = (bf16_bits_to_f32(init) if w.bank_dtype == "bf16" else init).astype(np.float64)
        snaps = []
        oracle.dw_stream(ref, x, p, S=S, C=C, P=P, steps=w.steps, valid_last=w.valid_last,
                         val_dtype=w.val_dtype, dv_dtype=w.dv_dtype, bank_dtype=w.bank_dtype, track=True,
                         snaps=snaps)
        for sn in snaps:
            c, G = sn["c"], len(sn["slots"])
            assert ng[c] == G, f"chunk {c}: {ng[c]} groups, oracle {G}"
            assert np.array_equal(snap_raw[c, G:], sent_raw[c, G:]), f"chunk {c}: rows past ngroups written"
            got, exact = snap_h[c, :G], sn["rows"]
            # The rows after k earlier writes: each write rounds once on either side (GPU and oracle
            # may land one unit of the last place apart, a unit of the value written then, which can
            # be larger than the row's current one) and carries the earlier difference scaled by
            # cpe <= 1; so k units at the row's largest magnitude so far, plus the f32 accumulation.
            k = sn["touched"][:, None].astype(np.float64)
            if w.bank_dtype == "bf16":
                tol = k * (2.0 ** -7 * sn["peak"] + 2.0 ** -17 * sn["mag"])
            else:
                tol = k * (1e-5 * np.maximum(sn["peak"], sn["mag"])) + 1e-30
            ok = (np.abs(got - exact) <= tol) | ((sn["amb"][:, None] > 0) & (np.abs(got - sn["alt"]) <= tol))
            if not ok.all():
                i, j = np.argwhere(~ok)[0]
                raise AssertionError(f"chunk {c}: {int((~ok).sum())} snapshot elements beyond tolerance, first "
                                     f"[{i},{j}] slot {sn['slots'][i]}: gpu {got[i, j]!r} oracle {exact[i, j]!r} "
                                     f"alt {sn['alt'][i, j]!r} amb {sn['amb'][i]} touched {sn['touched'][i]} "
                                     f"mag {sn['mag'][i, j]!r} tol {tol[i, j]!r}")


@pytest.mark.parametrize("name", ["uniform_c128", "zipf_c256", "few_slots"])
def test_snapshot_is_the_pre_step_bank(name):
    """Raw-copy identity: the rows of step t are the bank rows after a forward of steps [0, t)."""
    w = CASES[name]
    x = make_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)
    d = inputs_to_dev(x, w)
    P, S, C, hd, nk = w.P, w.S, w.C, w.hd, w.C * w.W
    ws = sdm.alloc_workspace(shape)
    bank = _bank(w)
    snap = _snap(shape, w)
    sdm.forward_chunks_saving(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, snap,
                              None, ws)
    for t in (0, w.steps // 2, w.steps - 1):
        ws_t = sdm.alloc_workspace(shape)
        bank_t = _bank(w)
        if t > 0:
            sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank_t, None,
                               ws_t, 0, t)
        torch.cuda.synchronize()
        bt = host(_raw(bank_t)).reshape(P, S, hd)
        sr = host(_raw(snap)).reshape(w.N, nk, hd)
        for p in range(P):
            c = t * P + p
            V = w.valid_last if t == w.steps - 1 else C
            sl = oracle.snapshot_slots(x["k_idx"][c], S=S, V=V)
            assert np.array_equal(sr[c, :len(sl)], bt[p, sl]), f"step {t} stream {p}: snapshot is not the pre-step bank"


def test_saving_argument_errors():
    w = CASES["tiny"]
    shape = sdm.ShapeSpec.from_workload(w)
    ws = sdm.alloc_workspace(shape)
    dv = torch.zeros(shape.N * shape.C * shape.hd, device="cuda")
    bank = torch.zeros(shape.P * shape.S * shape.hd, device="cuda")
    snap = torch.zeros(shape.N * shape.C * shape.W * shape.hd + 64, device="cuda")
    with pytest.raises(sdm.SdmError) as e:
        sdm.dw_saving(shape, dv, bank, None, ws)
    assert e.value.status == -1
    with pytest.raises(sdm.SdmError) as e:   # a full-size snapshot one element off alignment
        sdm.dw_saving(shape, dv, bank, snap[1:], ws)
    assert e.value.status == -4
