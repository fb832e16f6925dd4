"""Python face of the C ABI: argument marshalling only.

Tensors are CUDA tensors owned by the caller; every call passes their device pointers and the
current torch stream to ``libsdm_gb300.so``. Every step of the computation runs in the
library's kernels; there is no host or PyTorch fallback, and a CPU tensor is an error.
"""

from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _abi

_DT = {"f32": _abi.SDM_F32, "bf16": _abi.SDM_BF16}
_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


class SdmError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = _abi.load().sdm_status_string(status).decode()
        super().__init__(f"{what}: {msg} ({status})")
        self.status = status


@dataclasses.dataclass(frozen=True)
class ShapeSpec:
    P: int
    C: int
    W: int
    R: int
    hd: int
    steps: int
    S: int
    valid_last: int
    val_dtype: str = "bf16"
    dv_dtype: str = "bf16"
    bank_dtype: str = "bf16"
    gate_per_entry: bool = False
    # launch geometry (0: chosen from the shape); neither changes any output bit
    dw_log_buckets: int = 0
    p1_warps: int = 0

    @property
    def N(self) -> int:
        return self.steps * self.P

    def c(self) -> _abi.Shape:
        """The C struct of the shape (built once: the spec is immutable and the library only reads it)."""
        cs = self.__dict__.get("_cstruct")
        if cs is None:
            cs = _abi.Shape(self.P, self.C, self.W, self.R, self.hd, self.valid_last, self.steps, self.S,
                            _DT[self.val_dtype], _DT[self.dv_dtype], _DT[self.bank_dtype], int(self.gate_per_entry),
                            int(self.dw_log_buckets), int(self.p1_warps))
            object.__setattr__(self, "_cstruct", cs)
        return cs

    @classmethod
    def from_workload(cls, w, P=None) -> "ShapeSpec":
        return cls(P=w.P if P is None else P, C=w.C, W=w.W, R=w.R, hd=w.hd, steps=w.steps, S=w.S,
                   valid_last=w.valid_last, val_dtype=w.val_dtype, dv_dtype=w.dv_dtype, bank_dtype=w.bank_dtype,
                   gate_per_entry=bool(getattr(w, "gate_per_entry", False)))


def _ptr(t):
    """The device address of a contiguous CUDA tensor (an int: ctypes passes it as void*)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("expected a CUDA tensor (the library runs on the GPU only)")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _need(t, dtype, numel: int, name: str):
    """A caller tensor the library reads or writes ``numel`` elements of ``dtype`` through: checked
    here, because the C ABI takes bare pointers (a smaller or differently typed buffer would be
    accessed out of bounds)."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name}: expected at least {numel} elements, got {t.numel()}")


def _need_inputs(shape: "ShapeSpec", k_idx, q_idx, k_val, q_val, g):
    N, C, W, R = shape.N, shape.C, shape.W, shape.R
    vt = _TORCH_DT[shape.val_dtype]
    _need(k_idx, torch.int32, N * C * W, "k_idx")
    _need(q_idx, torch.int32, N * C * R, "q_idx")
    _need(k_val, vt, N * C * W, "k_val")
    _need(q_val, vt, N * C * R, "q_val")
    _need(g, torch.float32, N * C * (W if shape.gate_per_entry else 1), "g")


def _need_outputs(shape: "ShapeSpec", out):
    if not out:
        return
    for f, (shp, dt) in _out_spec(shape).items():
        if out.get(f) is not None:
            n = 1
            for d in shp:
                n *= d
            _need(out[f], dt, n, f"out[{f!r}]")


def _need_rows(shape: "ShapeSpec", dv, bank, snap=None):
    _need(dv, _TORCH_DT[shape.dv_dtype], shape.N * shape.C * shape.hd, "dv")
    _need(bank, _TORCH_DT[shape.bank_dtype], shape.P * shape.S * shape.hd, "bank")
    _need(snap, _TORCH_DT[shape.bank_dtype], shape.N * shape.C * shape.W * shape.hd, "snap")


# the current stream's handle without building a torch.cuda.Stream object per call (a per-step call
# such as read() is otherwise dominated by it); the public route where torch lacks these
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None and _cur_device is not None:
            return _raw_stream(_cur_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(st: int, what: str):
    if st != _abi.SDM_OK:
        raise SdmError(st, what)


def workspace_bytes(shape: ShapeSpec) -> int:
    n = _abi.load().sdm_workspace_bytes(ctypes.byref(shape.c()))
    if n == 0:
        raise ValueError(f"invalid shape {shape}")
    return int(n)


def alloc_workspace(shape: ShapeSpec, device="cuda", stream=None) -> torch.Tensor:
    """A zero-initialised workspace (torch allocations are 256-byte aligned)."""
    n = workspace_bytes(shape)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(_abi.load().sdm_workspace_init(_ptr(ws), n, _stream(stream)), "sdm_workspace_init")
    return ws


# every Phase-1 output but ngroups (written only by the saving forward's Phase 1) and the
# diagnostic counters (stats: ask for them by name)
PLAIN_FIELDS = tuple(f for f in _abi.P1_FIELDS if f not in ("ngroups", "stats"))
# stats[i]: valid write groups, dense (rank-1) pair groups, exact pair terms, A / QK rows with terms
STATS = ("groups", "dense_groups", "pair_terms", "rows_with_terms")


def _out_spec(shape: ShapeSpec) -> dict:
    N, C, W, R = shape.N, shape.C, shape.W, shape.R
    vt = _TORCH_DT[shape.val_dtype]
    return {
        "log_k": ((N, C, W), torch.float32), "rex": ((N, C, W), torch.float32), "cpe": ((N, C, W), vt),
        "k_eff": ((N, C, W), vt), "is_last": ((N, C, W), torch.int8), "is_only": ((N, C, W), torch.int8),
        "pos_k": ((N, C, W), torch.int32), "log_q": ((N, C, R), torch.float32), "q_w": ((N, C, R), vt),
        "pos_q": ((N, C, R), torch.int32), "q_last": ((N, C, R), torch.int8), "q_only": ((N, C, R), torch.int8),
        "A": ((N, C, C), torch.float32), "QK": ((N, C, C), torch.float32),
        "sorted_k": ((N, C * W), torch.int32), "sorted_q": ((N, C * R), torch.int32), "repeats": ((2,), torch.int64),
        "ngroups": ((N,), torch.int32), "stats": ((4,), torch.int64),
    }


def alloc_outputs(shape: ShapeSpec, device="cuda", fields=PLAIN_FIELDS) -> dict:
    spec = _out_spec(shape)
    out = {}
    for f in fields:
        shp, dt = spec[f]
        out[f] = (torch.zeros(shp, dtype=dt, device=device) if f in ("repeats", "stats")
                  else torch.empty(shp, dtype=dt, device=device))
    return out


def _p1out(out):
    o = _abi.P1Out()
    if out:
        for f in _abi.P1_FIELDS:
            if f in out and out[f] is not None:
                setattr(o, f, _ptr(out[f]))
    return o


def phase1(shape: ShapeSpec, k_idx, q_idx, k_val, q_val, g, out: dict, ws, step_begin=0, step_end=None, stream=None):
    _need_inputs(shape, k_idx, q_idx, k_val, q_val, g)
    _need_outputs(shape, out)
    step_end = shape.steps if step_end is None else step_end
    o = _p1out(out)
    st = _abi.load().sdm_phase1(ctypes.byref(shape.c()), _ptr(k_idx), _ptr(q_idx), _ptr(k_val), _ptr(q_val), _ptr(g),
                                ctypes.byref(o), step_begin, step_end, _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "sdm_phase1")


def dw(shape: ShapeSpec, dv, bank, ws, step_begin=0, step_end=None, stream=None):
    _need_rows(shape, dv, bank)
    step_end = shape.steps if step_end is None else step_end
    st = _abi.load().sdm_dw(ctypes.byref(shape.c()), _ptr(dv), _ptr(bank), step_begin, step_end, _ptr(ws), ws.numel(),
                            _stream(stream))
    _check(st, "sdm_dw")


def forward_chunks(shape: ShapeSpec, k_idx, q_idx, k_val, q_val, g, dv, bank, out, ws, step_begin=0, step_end=None,
                   stream=None):
    _need_inputs(shape, k_idx, q_idx, k_val, q_val, g)
    _need_outputs(shape, out)
    _need_rows(shape, dv, bank)
    step_end = shape.steps if step_end is None else step_end
    o = _p1out(out)
    st = _abi.load().sdm_forward_chunks(ctypes.byref(shape.c()), _ptr(k_idx), _ptr(q_idx), _ptr(k_val), _ptr(q_val),
                                        _ptr(g), _ptr(dv), _ptr(bank), ctypes.byref(o) if out else None, step_begin,
                                        step_end, _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "sdm_forward_chunks")


def alloc_snapshot(shape: ShapeSpec, device="cuda") -> torch.Tensor:
    """The dense compact snapshot of the saving forward: [N, C*W, hd] rows of the bank type."""
    return torch.empty((shape.N, shape.C * shape.W, shape.hd), dtype=_TORCH_DT[shape.bank_dtype], device=device)


def phase1_saving(shape: ShapeSpec, k_idx, q_idx, k_val, q_val, g, out: dict, ws, step_begin=0, step_end=None,
                  stream=None):
    """sdm_phase1_saving: Phase 1 whose records carry the groups' dense ordinals (for dw_saving)."""
    _need_inputs(shape, k_idx, q_idx, k_val, q_val, g)
    _need_outputs(shape, out)
    step_end = shape.steps if step_end is None else step_end
    o = _p1out(out)
    st = _abi.load().sdm_phase1_saving(ctypes.byref(shape.c()), _ptr(k_idx), _ptr(q_idx), _ptr(k_val), _ptr(q_val),
                                       _ptr(g), ctypes.byref(o), step_begin, step_end, _ptr(ws), ws.numel(),
                                       _stream(stream))
    _check(st, "sdm_phase1_saving")


def dw_saving(shape: ShapeSpec, dv, bank, snap, ws, step_begin=0, step_end=None, stream=None):
    """sdm_dw_saving: the DW, also writing each group's pre-write base row to ``snap``."""
    _need_rows(shape, dv, bank, snap)
    step_end = shape.steps if step_end is None else step_end
    st = _abi.load().sdm_dw_saving(ctypes.byref(shape.c()), _ptr(dv), _ptr(bank), _ptr(snap), step_begin, step_end,
                                   _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "sdm_dw_saving")


def forward_chunks_saving(shape: ShapeSpec, k_idx, q_idx, k_val, q_val, g, dv, bank, snap, out, ws, step_begin=0,
                          step_end=None, stream=None):
    """sdm_forward_chunks_saving: Phase 1, then the DW writing the dense compact snapshot."""
    _need_inputs(shape, k_idx, q_idx, k_val, q_val, g)
    _need_outputs(shape, out)
    _need_rows(shape, dv, bank, snap)
    step_end = shape.steps if step_end is None else step_end
    o = _p1out(out)
    st = _abi.load().sdm_forward_chunks_saving(ctypes.byref(shape.c()), _ptr(k_idx), _ptr(q_idx), _ptr(k_val),
                                               _ptr(q_val), _ptr(g), _ptr(dv), _ptr(bank), _ptr(snap),
                                               ctypes.byref(o) if out else None, step_begin, step_end, _ptr(ws),
                                               ws.numel(), _stream(stream))
    _check(st, "sdm_forward_chunks_saving")


def forward_chunks_noalloc(shape: ShapeSpec, k_idx, q_idx, k_val, q_val, g, dv, bank, out, status=None, step_begin=0,
                           step_end=None, stream=None):
    """sdm_forward_chunks_noalloc: the forward on the library's own scratch (no workspace).
    ``status`` (optional) is a CUDA int32 tensor of one element that receives the device status."""
    _need_inputs(shape, k_idx, q_idx, k_val, q_val, g)
    _need_outputs(shape, out)
    _need_rows(shape, dv, bank)
    step_end = shape.steps if step_end is None else step_end
    o = _p1out(out)
    st = _abi.load().sdm_forward_chunks_noalloc(ctypes.byref(shape.c()), _ptr(k_idx), _ptr(q_idx), _ptr(k_val),
                                                _ptr(q_val), _ptr(g), _ptr(dv), _ptr(bank),
                                                ctypes.byref(o) if out else None, step_begin, step_end, _ptr(status),
                                                _stream(stream))
    _check(st, "sdm_forward_chunks_noalloc")


def read(shape: ShapeSpec, q_idx, q_w, bank, y, step_begin=0, step_end=None, status=None, stream=None):
    """sdm_read: the forward's read-side token gather of steps [step_begin, step_end):
    y[c, t] = sum over read lanes (in order, float32) of q_w[c, t, r] * bank[p*S + q_idx[c, t, r]].
    ``bank`` is read as it is (run it for a step before that step's DW); ``y`` is [N, C, hd] float32;
    ``status`` (optional) is a CUDA int32 tensor of one element to which SDM_DEV_* bits are OR-ed."""
    N, C, R = shape.N, shape.C, shape.R
    _need(q_idx, torch.int32, N * C * R, "q_idx")
    _need(q_w, _TORCH_DT[shape.val_dtype], N * C * R, "q_w")
    _need(bank, _TORCH_DT[shape.bank_dtype], shape.P * shape.S * shape.hd, "bank")
    _need(y, torch.float32, N * C * shape.hd, "y")
    step_end = shape.steps if step_end is None else step_end
    st = _abi.load().sdm_read(ctypes.byref(shape.c()), _ptr(q_idx), _ptr(q_w), _ptr(bank), _ptr(y), step_begin,
                              step_end, _ptr(status), _stream(stream))
    _check(st, "sdm_read")


def pa(shape: ShapeSpec, sorted_k, k_idx, k_val, log_k, cpe, beta, dva, grad, bank, snap, d_k_eff, grad_g,
       step_begin=0, step_end=None, status=None, stream=None):
    """sdm_pa: Phase A of the backward for steps [step_begin, step_end), last step first.
    ``grad`` is float32 or bfloat16 (its dtype is passed as grad_dtype); ``snap`` holds the range's
    snapshot rows ([steps in range, P, C*W, hd]); ``status`` (optional) is a CUDA int32 tensor of one
    element to which SDM_DEV_* bits are OR-ed."""
    step_end = shape.steps if step_end is None else step_end
    gdt = {torch.float32: _abi.SDM_F32, torch.bfloat16: _abi.SDM_BF16}.get(grad.dtype)
    if gdt is None:
        raise TypeError("grad must be float32 or bfloat16")
    st = _abi.load().sdm_pa(ctypes.byref(shape.c()), gdt, _ptr(sorted_k), _ptr(k_idx), _ptr(k_val), _ptr(log_k),
                            _ptr(cpe), _ptr(beta), _ptr(dva), _ptr(grad), _ptr(bank), _ptr(snap), _ptr(d_k_eff),
                            _ptr(grad_g), step_begin, step_end, _ptr(status), _stream(stream))
    _check(st, "sdm_pa")


def gwr(shape: ShapeSpec, k_idx, write_w, dv, grad, d_delta_v, d_k_pd, step_begin=0, step_end=None, status=None,
        stream=None):
    """sdm_gwr: the write side's token gather of the backward for steps [step_begin, step_end), last
    step first. ``grad`` is float32 or bfloat16 (passed as grad_dtype)."""
    step_end = shape.steps if step_end is None else step_end
    gdt = {torch.float32: _abi.SDM_F32, torch.bfloat16: _abi.SDM_BF16}.get(grad.dtype)
    if gdt is None:
        raise TypeError("grad must be float32 or bfloat16")
    st = _abi.load().sdm_gwr(ctypes.byref(shape.c()), gdt, _ptr(k_idx), _ptr(write_w), _ptr(dv), _ptr(grad),
                             _ptr(d_delta_v), _ptr(d_k_pd), step_begin, step_end, _ptr(status), _stream(stream))
    _check(st, "sdm_gwr")


def gds(shape: ShapeSpec, sorted_q, q_idx, q_val, log_q, gr, bank, grad, d_q_w, step_begin=0, step_end=None,
        status=None, stream=None):
    """sdm_gds: the read side of the backward for steps [step_begin, step_end), last step first.
    ``grad`` is float32 or bfloat16 (its dtype is passed as grad_dtype); ``status`` (optional) is a CUDA
    int32 tensor of one element to which SDM_DEV_* bits are OR-ed."""
    step_end = shape.steps if step_end is None else step_end
    gdt = {torch.float32: _abi.SDM_F32, torch.bfloat16: _abi.SDM_BF16}.get(grad.dtype)
    if gdt is None:
        raise TypeError("grad must be float32 or bfloat16")
    st = _abi.load().sdm_gds(ctypes.byref(shape.c()), gdt, _ptr(sorted_q), _ptr(q_idx), _ptr(q_val), _ptr(log_q),
                             _ptr(gr), _ptr(bank), _ptr(grad), _ptr(d_q_w), step_begin, step_end, _ptr(status),
                             _stream(stream))
    _check(st, "sdm_gds")


def device_status(ws, clear: bool = True, stream=None) -> int:
    code = _abi.c_i32(0)
    st = _abi.load().sdm_device_status(_ptr(ws), ctypes.byref(code), int(clear), _stream(stream))
    if st not in (_abi.SDM_OK, -8):
        _check(st, "sdm_device_status")
    return int(code.value)
