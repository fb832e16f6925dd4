"""The backward's step loop: GWR, GDS and Phase A called one step at a time, last step first, as a
backward interleaves them (pa_dc_cuda.py module docstring: "Backward step ti"; mover_da2_cuda.py,
GDS), against the oracle doing the same per stream.

Per step ti: GWR reads the grad rows as the later steps left them; GDS takes its dots on the bank as
Phase A of the later steps restored it and adds its scatter to the grad rows; Phase A then propagates
the grad rows through the step's decay-and-write and restores the step's pre-write bank rows.

Tolerances (u = 2^-24): the grad rows carry the bound of every step before (GDS: (n + 8) u mag, Phase
A: (n + 8) u mag, adding up; cpe <= 1 scales earlier errors down); an output that reads grad rows
adds the carried bound times its coefficients (GWR: sum |w| tol, d_k_pd and grad_g: sum tol |x|);
outputs reading the bank are exact-input dots ((hd + 8) u sum |products|); restored bank rows exact.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_slot_memory_gb300 as sdm
from sdm_testlib import dev_array, host
from synth import (WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_backward_inputs, make_bank_stream,
                   make_grad_stream, make_inputs, make_read_grads, make_snapshot_chunk, make_write_weights, scaled)

pytestmark = pytest.mark.gpu

U = 2.0 ** -24

CASES = {
    "uniform_c128": scaled(WORKLOADS["uniform_c128"], P=2, T=384, S=4096),
    "zipf_c256": scaled(WORKLOADS["zipf_c256"], P=2, T=512, S=4096),
    "wide_ragged": scaled(WORKLOADS["wide_ragged"], P=1, T=300, S=8192),
}


def _bf(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("name", list(CASES))
def test_backward_step_loop(name):
    w = CASES[name]
    P, S, C, W, R, hd, nk = w.P, w.S, w.C, w.W, w.R, w.hd, w.C * w.W
    x = make_inputs(w)
    fp = (w.steps - 1) * P
    o = oracle.phase1(x["k_idx"], x["q_idx"], x["k_val"], x["q_val"], x["g"], S=S, val_dtype=w.val_dtype,
                      first_partial=fp, valid_last=w.valid_last, pairs=False)
    log_k = np.asarray(o["log_k"], np.float32)
    log_q = np.asarray(o["log_q"], np.float32)
    cpe_bits = f32_to_bf16_bits(np.asarray(o["cpe"], np.float32))
    b = make_backward_inputs(w)
    gr = make_read_grads(w)
    ww = make_write_weights(w)
    snap_bits = np.stack([make_snapshot_chunk(w, c) for c in range(w.N)], 0)
    grad0 = np.stack([make_grad_stream(w, p) for p in range(P)], 0)
    bank0 = np.stack([make_bank_stream(w, p) for p in range(P)], 0)

    shape = sdm.ShapeSpec.from_workload(w)
    d = {"sorted_k": dev_array(o["sorted_k"].astype(np.int32)), "sorted_q": dev_array(o["sorted_q"].astype(np.int32)),
         "k_idx": dev_array(x["k_idx"]), "q_idx": dev_array(x["q_idx"]), "k_val": dev_array(x["k_val"], "bf16"),
         "q_val": dev_array(x["q_val"], "bf16"), "dv": dev_array(x["dv"], "bf16"), "log_k": dev_array(log_k),
         "log_q": dev_array(log_q), "cpe": dev_array(cpe_bits, "bf16"), "beta": dev_array(b["beta"]),
         "dva": dev_array(b["dva"]), "gr": dev_array(gr), "ww": dev_array(ww),
         "snap": dev_array(snap_bits.reshape(-1, hd), "bf16")}
    grad = torch.from_numpy(grad0.reshape(P * S, hd)).cuda()
    bank = dev_array(bank0.reshape(P * S, hd), "bf16")
    outs = {k: torch.full(shp, float("nan"), device="cuda") for k, shp in
            (("dd", (w.N, C, hd)), ("pd", (w.N, C, W)), ("dq", (w.N, C, R)), ("de", (w.N, C, W)), ("dg", (w.N, C, W)))}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for ti in range(w.steps - 1, -1, -1):
        sdm.gwr(shape, d["k_idx"], d["ww"], d["dv"], grad, outs["dd"], outs["pd"], ti, ti + 1, st)
        sdm.gds(shape, d["sorted_q"], d["q_idx"], d["q_val"], d["log_q"], d["gr"], bank, grad, outs["dq"], ti, ti + 1,
                st)
        sdm.pa(shape, d["sorted_k"], d["k_idx"], d["k_val"], d["log_k"], d["cpe"], d["beta"], d["dva"], grad, bank,
               d["snap"][ti * P * nk:], outs["de"], outs["dg"], ti, ti + 1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = {k: host(v).astype(np.float64) for k, v in outs.items()}

    ref = reference(w, x, o, b, gr, ww, snap_bits, grad0, bank0)
    for k, (val, t) in ref["outs"].items():
        assert np.all(np.abs(got[k] - val) <= t), f"{name}: {k} beyond tolerance"
    for p in range(P):
        gg_rows = host(grad[p * S:(p + 1) * S]).astype(np.float64)
        assert np.all(np.abs(gg_rows - ref["grad"][p]) <= ref["tol"][p]), f"{name}: grad rows of stream {p}"
        assert np.array_equal(host(bank[p * S:(p + 1) * S]).astype(np.float64), ref["bank"][p]), f"{name}: bank {p}"


def reference(w, x, o, b, gr, ww, snap_bits, grad0, bank0):
    """The oracle's step loop per stream: every output with its bound, the final grad rows with theirs,
    the final bank rows."""
    P, S, C, W, R, hd = w.P, w.S, w.C, w.W, w.R, w.hd
    log_k = np.asarray(o["log_k"], np.float32)
    log_q = np.asarray(o["log_q"], np.float32)
    cpe = _bf(f32_to_bf16_bits(np.asarray(o["cpe"], np.float32)))
    kv, qv = _bf(x["k_val"]), _bf(x["q_val"])
    dvf = _bf(x["dv"]).reshape(w.N, C, hd)
    outs = {k: (np.zeros(shp), np.zeros(shp)) for k, shp in
            (("dd", (w.N, C, hd)), ("pd", (w.N, C, W)), ("dq", (w.N, C, R)), ("de", (w.N, C, W)), ("dg", (w.N, C, W)))}
    grads, tols, banks = [], [], []
    for p in range(P):
        g = grad0[p].astype(np.float64)
        bk = _bf(bank0[p])
        tol = np.zeros_like(g)
        for ti in range(w.steps - 1, -1, -1):
            c = ti * P + p
            V = w.valid_last if ti == w.steps - 1 else C
            kid, qid = x["k_idx"][c], x["q_idx"][c]
            kval = (kid >= 0) & (kid < S) & (np.arange(C)[:, None] < V)
            qval = (qid >= 0) & (qid < S) & (np.arange(C)[:, None] < V)
            # GWR on the grad rows as the later steps left them
            dd, pd, mag, dmag = oracle.gwr_chunk(g, kid, ww[c].astype(np.float64), dvf[c], S=S, V=V)
            carry_dd = np.zeros((C, hd))
            carry_pd = np.zeros((C, W))
            for t in range(V):
                for n in range(W):
                    if kval[t, n]:
                        carry_dd[t] += abs(float(ww[c, t, n])) * tol[kid[t, n]]
                        carry_pd[t, n] = float(np.sum(tol[kid[t, n]] * np.abs(dvf[c, t])))
            outs["dd"][0][c], outs["dd"][1][c] = dd, (W + 4) * U * mag + carry_dd
            outs["pd"][0][c], outs["pd"][1][c] = pd, (hd + 8) * U * dmag + carry_pd
            # GDS: dots on the restored bank, scatter into the grad rows
            dq, gmag, qmag = oracle.gds_chunk(g, bk, qid, qv[c], log_q[c].astype(np.float64), gr[c].astype(np.float64),
                                              S=S, V=V)
            outs["dq"][0][c], outs["dq"][1][c] = dq, (hd + 8) * U * qmag
            tol += (np.bincount(qid[qval], minlength=S)[:, None] + 8) * U * gmag
            # Phase A
            slots = oracle.snapshot_slots(kid, S=S, V=V)
            snap = _bf(snap_bits[c][:len(slots)])
            tprev = tol.copy()
            de, gg, pmag, dme, dmg = oracle.pa_chunk(g, bk, snap, kid, kv[c], log_k[c].astype(np.float64), cpe[c],
                                                     b["beta"][c].astype(np.float64), b["dva"][c].astype(np.float64),
                                                     S=S, V=V)
            tol += (np.bincount(kid[kval], minlength=S)[:, None] + 8) * U * pmag
            sn = np.zeros((S, hd))
            sn[slots] = np.abs(snap)
            carry_g = np.zeros((C, W))
            carry_g[kval] = np.sum(tprev[kid[kval]] * sn[kid[kval]], axis=1)
            outs["de"][0][c], outs["de"][1][c] = de, (hd + 8) * U * dme
            outs["dg"][0][c], outs["dg"][1][c] = gg, (hd + 8) * U * dmg + np.abs(cpe[c]) * carry_g
        grads.append(g)
        tols.append(tol)
        banks.append(bk)
    return {"outs": outs, "grad": grads, "tol": tols, "bank": banks}
