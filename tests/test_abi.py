"""The C ABI without a GPU: the library builds and loads, exports every function include/sdm.h
declares, sizes workspaces, and rejects bad arguments before any CUDA call (no launches here)."""

import ctypes
import dataclasses
import os
import re

import pytest

import sparse_slot_memory_gb300 as sdm
from sparse_slot_memory_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sdm.build()
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)
    return _abi.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "sdm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sdm_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_abi.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def shape(**kw):
    base = dict(P=32, C=256, W=16, R=16, hd=128, valid_last=256, steps=32, S=1 << 20, val_dtype=1, dv_dtype=1,
                bank_dtype=1, gate_per_entry=0)
    base.update(kw)
    return _abi.Shape(**base)


def test_workspace_bytes(lib):
    n = lib.sdm_workspace_bytes(ctypes.byref(shape()))
    # DW records (16 B per write entry) dominate
    assert n >= 1024 * 4096 * 16
    assert lib.sdm_workspace_bytes(ctypes.byref(shape(C=257))) == 0
    assert lib.sdm_workspace_bytes(ctypes.byref(shape(W=17, R=16))) == 0   # C * (W + R) > 8192
    assert lib.sdm_workspace_bytes(ctypes.byref(shape(hd=6))) == 0
    assert lib.sdm_workspace_bytes(None) == 0
    # the DW bucket count is part of the workspace layout (its per-step bucket bounds)
    b3 = lib.sdm_workspace_bytes(ctypes.byref(shape(dw_log_buckets=3)))
    b11 = lib.sdm_workspace_bytes(ctypes.byref(shape(dw_log_buckets=11)))
    assert 0 < b3 < b11
    assert lib.sdm_workspace_bytes(ctypes.byref(shape(p1_warps=32))) == n


FAKE = 0x100000  # never dereferenced: every case fails a host check first


@pytest.mark.parametrize("kw,code", [
    (dict(C=0), -2), (dict(C=300), -2), (dict(W=0), -2), (dict(R=300), -2), (dict(W=20, R=20), -2),
    (dict(valid_last=0), -2), (dict(valid_last=257), -2), (dict(steps=0), -2), (dict(S=0), -2),
    (dict(S=1 << 31), -2), (dict(val_dtype=7), -3), (dict(bank_dtype=-1), -3), (dict(hd=126), -4),
    (dict(gate_per_entry=2), -2), (dict(dw_log_buckets=12), -2), (dict(dw_log_buckets=-1), -2),
    (dict(S=16, dw_log_buckets=5), -2), (dict(p1_warps=33), -2), (dict(p1_warps=31), -2),
])
def test_shape_errors(lib, kw, code):
    st = lib.sdm_phase1(ctypes.byref(shape(**kw)), FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 1, FAKE, 1 << 40, None)
    assert st == code
    st = lib.sdm_dw(ctypes.byref(shape(**kw)), FAKE, FAKE, 0, 1, FAKE, 1 << 40, None)
    assert st == code


def test_argument_errors(lib):
    s = ctypes.byref(shape())
    assert lib.sdm_phase1(s, None, FAKE, FAKE, FAKE, FAKE, None, 0, 1, FAKE, 1 << 40, None) == -1
    assert lib.sdm_phase1(s, FAKE + 4, FAKE, FAKE, FAKE, FAKE, None, 0, 1, FAKE, 1 << 40, None) == -4
    assert lib.sdm_phase1(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 1, FAKE, 1 << 40, None) == -1
    assert lib.sdm_phase1(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 33, FAKE, 1 << 40, None) == -1
    assert lib.sdm_phase1(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 1, FAKE, 1024, None) == -5
    assert lib.sdm_phase1(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 1, FAKE + 16, 1 << 40, None) == -5
    assert lib.sdm_phase1(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 1, None, 1 << 40, None) == -5
    out = _abi.P1Out()
    out.A = FAKE + 8
    assert lib.sdm_phase1(s, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(out), 0, 1, FAKE, 1 << 40, None) == -4
    assert lib.sdm_dw(s, None, FAKE, 0, 1, FAKE, 1 << 40, None) == -1
    assert lib.sdm_dw(s, FAKE, FAKE + 2, 0, 1, FAKE, 1 << 40, None) == -4
    assert lib.sdm_forward_chunks(s, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0, 1, FAKE, 1 << 40,
                                  None) == -1
    code = ctypes.c_int32(0)
    assert lib.sdm_device_status(None, ctypes.byref(code), 0, None) == -1
    assert lib.sdm_workspace_init(FAKE + 8, 4096, None) == -5


def test_status_strings(lib):
    for c in range(-8, 1):
        s = lib.sdm_status_string(c).decode()
        assert s.startswith("SDM_")
    assert "unknown" in lib.sdm_status_string(5).decode()


def test_no_cpu_path_for_host_tensors():
    import torch
    spec = sdm.ShapeSpec(P=1, C=4, W=1, R=1, hd=4, steps=1, S=8, valid_last=4)
    with pytest.raises(TypeError):
        sdm.dw(spec, torch.zeros(4, 4), torch.zeros(8, 4), torch.zeros(1 << 16, dtype=torch.uint8))


@pytest.mark.parametrize("fn, nptr", [("sdm_pa", 12), ("sdm_gwr", 6), ("sdm_gds", 8)])
def test_backward_argument_errors(lib, fn, nptr):
    """The backward entry points check shape, grad dtype, step range, null and misaligned arrays
    before any CUDA call (the pointers below are never dereferenced)."""
    f = getattr(lib, fn)
    good = [ctypes.c_void_p(0x10000 + 256 * i) for i in range(nptr)]   # 16-byte aligned, never touched
    s = shape()
    assert f(ctypes.byref(s), 0, *([None] * nptr), 0, 32, None, None) == -1              # null arrays
    assert f(ctypes.byref(s), 7, *good, 0, 32, None, None) == -3                         # grad dtype
    assert f(ctypes.byref(shape(C=257)), 0, *good, 0, 32, None, None) == -2              # shape
    assert f(ctypes.byref(shape(hd=6)), 0, *good, 0, 32, None, None) == -4               # hd % 4
    assert f(ctypes.byref(s), 0, *good, 5, 4, None, None) == -1                          # reversed range
    assert f(ctypes.byref(s), 0, *good, 0, 33, None, None) == -1                         # past the last step
    bad = list(good)
    bad[-1] = ctypes.c_void_p(0x10000 + 8)
    assert f(ctypes.byref(s), 0, *bad, 0, 32, None, None) == -4                          # misaligned
    assert f(ctypes.byref(s), 1, *good, 3, 3, None, None) == 0                           # empty range: no launch


def test_binding_rejects_buffers_of_the_wrong_type_or_extent():
    """The C ABI takes bare pointers; the Python binding checks each tensor's dtype and element count
    against the shape before any call (a bank of the wrong type once let the DW write past its end)."""
    import torch

    from sparse_slot_memory_gb300 import api

    shape = api.ShapeSpec(P=1, C=64, W=4, R=4, hd=64, steps=16, S=4096, valid_last=64,
                          val_dtype="f32", dv_dtype="f32", bank_dtype="f32")
    dv = torch.zeros(shape.N * shape.C * shape.hd, dtype=torch.float32)
    ws = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(TypeError, match="bank: expected torch.float32"):
        api.dw(shape, dv, torch.zeros(shape.P * shape.S * shape.hd, dtype=torch.bfloat16), ws)
    with pytest.raises(ValueError, match="bank: expected at least"):
        api.dw(shape, dv, torch.zeros(shape.P * shape.S * shape.hd - 1, dtype=torch.float32), ws)
    with pytest.raises(TypeError, match="dv: expected torch.float32"):
        api.dw(shape, dv.to(torch.bfloat16), torch.zeros(shape.P * shape.S * shape.hd), ws)
    k_idx = torch.zeros(shape.N * shape.C * shape.W, dtype=torch.int32)
    q_idx = torch.zeros(shape.N * shape.C * shape.R, dtype=torch.int32)
    k_val = torch.zeros(shape.N * shape.C * shape.W)
    q_val = torch.zeros(shape.N * shape.C * shape.R)
    g = torch.zeros(shape.N * shape.C)
    with pytest.raises(ValueError, match="g: expected at least"):
        api.phase1(dataclasses.replace(shape, gate_per_entry=True), k_idx, q_idx, k_val, q_val, g, {}, ws)
    with pytest.raises(TypeError, match=r"out\['A'\]: expected torch.float32"):
        api.phase1(shape, k_idx, q_idx, k_val, q_val, g, {"A": torch.zeros(shape.N * shape.C * shape.C, dtype=torch.float64)}, ws)
    with pytest.raises(TypeError, match="k_idx: expected torch.int32"):
        api.forward_chunks(shape, k_idx.long(), q_idx, k_val, q_val, g, dv, torch.zeros(shape.P * shape.S * shape.hd), {}, ws)


def test_shape_struct_is_built_once_and_matches_the_spec(lib):
    """The binding hands the library one C struct per ShapeSpec (the spec is immutable): the same
    object on every call, with the spec's fields, and the spec's equality and hashing untouched."""
    spec = sdm.ShapeSpec(P=3, C=16, W=2, R=4, hd=8, steps=5, S=1000, valid_last=9, val_dtype="f32",
                         bank_dtype="f32", dw_log_buckets=2, p1_warps=1)
    cs = spec.c()
    assert spec.c() is cs
    assert (cs.P, cs.C, cs.W, cs.R, cs.hd, cs.valid_last, cs.steps, cs.S) == (3, 16, 2, 4, 8, 9, 5, 1000)
    assert (cs.val_dtype, cs.dv_dtype, cs.bank_dtype) == (_abi.SDM_F32, _abi.SDM_BF16, _abi.SDM_F32)
    twin = dataclasses.replace(spec)
    assert twin == spec and hash(twin) == hash(spec) and twin.c() is not cs
    assert lib.sdm_workspace_bytes(ctypes.byref(cs)) == lib.sdm_workspace_bytes(ctypes.byref(twin.c())) > 0


def test_default_bucket_count_is_capped_at_two_to_the_ten(lib):
    """With dw_log_buckets = 0 a stream gets about 32768 / P DW buckets, at most 2^10 (more would push a
    512-thread Phase-1 block past two blocks per SM): the default's workspace equals the explicit 2^10
    one for P = 8 (which would want 2^12) and the explicit 2^9 one for P = 64."""
    def ws(P, k):
        spec = sdm.ShapeSpec(P=P, C=256, W=8, R=8, hd=128, steps=4, S=1 << 16, valid_last=256, dw_log_buckets=k)
        return lib.sdm_workspace_bytes(ctypes.byref(spec.c()))
    assert ws(8, 0) == ws(8, 10) != ws(8, 11)
    assert ws(64, 0) == ws(64, 9) != ws(64, 10)
