"""The no-allocation forward, sdm_forward_chunks_noalloc, against the workspace forward.

Some callers cannot allocate device memory: code inside a host framework that owns every device
allocation, or a plugin interface that is handed only its input and output buffers. They call
sdm_forward_chunks_noalloc, which runs the same kernels on a scratch array compiled into the
library instead of a caller workspace. These tests call it through the C ABI twice in a row (the
second call finds the first call's bytes in the shared scratch) and compare each result with
sdm_forward_chunks on a caller-allocated workspace. Both run the same kernels with the same
arithmetic, so every output and the bank must agree bit for bit, which is inside every tolerance
the parity tests use. This file is named to be collected last; it also passes on its own.
"""

import ctypes
import numpy as np
import pytest
import torch

import sparse_slot_memory_gb300 as sdm
from sparse_slot_memory_gb300 import _abi
from sdm_testlib import inputs_to_dev
from synth import WORKLOADS, bf16_bits_to_f32, make_bank_stream, make_inputs, scaled

pytestmark = pytest.mark.gpu

W = scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=4096, hd=64, name="noalloc")   # ragged last step


def _bank(w):
    rows = np.stack([bf16_bits_to_f32(make_bank_stream(w, p)) for p in range(w.P)], 0)
    return torch.from_numpy(rows.reshape(w.P * w.S, w.hd)).cuda().to(torch.bfloat16)


def _raw(out, bank):
    res = {k: v.view(torch.uint8).cpu().numpy() for k, v in out.items()}
    res["bank"] = bank.view(torch.int16).cpu().numpy()
    return res


def test_noalloc_matches_workspace_forward_on_two_calls():
    x = make_inputs(W)
    shape = sdm.ShapeSpec.from_workload(W)
    assert sdm.workspace_bytes(shape) <= _abi.NOALLOC_SCRATCH_BYTES
    d = inputs_to_dev(x, W)

    ws = sdm.alloc_workspace(shape)
    bank = _bank(W)
    out = sdm.alloc_outputs(shape)
    sdm.forward_chunks(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, out, ws)
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0
    want = _raw(out, bank)

    for call in range(2):
        bank_n = _bank(W)
        out_n = sdm.alloc_outputs(shape)
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        sdm.forward_chunks_noalloc(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank_n,
                                   out_n, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        got = _raw(out_n, bank_n)
        for k in want:
            assert np.array_equal(got[k], want[k]), f"call {call}: {k} differs from the workspace forward"


def test_noalloc_reports_device_status_and_rejects_large_shapes():
    x = make_inputs(W)
    x["k_idx"][0, 5, 1] = W.S + 3    # a valid token with an out-of-range slot id
    shape = sdm.ShapeSpec.from_workload(W)
    d = inputs_to_dev(x, W)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdm.forward_chunks_noalloc(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], _bank(W),
                               None, status)
    torch.cuda.synchronize()
    assert int(status.item()) & _abi.SDM_DEV_BAD_SLOT
    big = sdm.ShapeSpec.from_workload(WORKLOADS["large"])
    assert sdm.workspace_bytes(big) > _abi.NOALLOC_SCRATCH_BYTES
    one = torch.zeros(16, device="cuda")   # the C entry point rejects the shape before touching any array
    p = ctypes.c_void_p(one.data_ptr())
    st = _abi.load().sdm_forward_chunks_noalloc(ctypes.byref(big.c()), p, p, p, p, p, p, p, None, 0, big.steps, None,
                                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == -5
