"""The five synthetic workloads of the sparse-delta-memory forward and their seeded generators.

Layout is chunk-major, as the Phase-1 module of ``sparse_delta_memory`` (phase1_cuda.py, module
docstring and ``p1_keys_zw_kernel``) lays its rows out: chunk ``c = ti * P + p`` holds tokens
``[ti * C, (ti + 1) * C)`` of stream ``p``.

* ``k_idx`` int32 ``[N, C, W]``, ``q_idx`` int32 ``[N, C, R]``: stream-local slot ids in ``[0, S)``;
  tokens past the stream's end (the last step, when ``T % C != 0``) hold ``-1``.
* ``k_val`` / ``q_val``: ``[N, C, W]`` / ``[N, C, R]`` float32, or bfloat16 kept as uint16 bit patterns.
* ``g`` float32 ``[N, C]``: one log-decay gate per token, ``logsigmoid(N(mu, 1))``; with
  ``gate_per_entry`` ``[N, C, W]``, one per write entry, drawn the same way.
* ``dv`` ``[N * C, hd]``: the value delta of every token (row ``c * C + t``).
* bank ``[P * S, hd]``: stream ``p`` owns rows ``[p * S, (p + 1) * S)``; drawn per stream.

Every array comes from its own ``numpy`` generator spawned from the workload's seed, per stream,
so any subset of streams can be generated alone and is identical to the same streams of the full
set. bfloat16 values are float32 draws rounded to nearest even.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    P: int            # independent streams (sequences)
    T: int            # tokens per stream
    C: int            # chunk length (tokens)
    S: int            # bank slots per stream
    hd: int           # bank row width (columns)
    W: int            # write (K) entries per token
    R: int            # read (Q) entries per token
    idx: str          # "uniform" or "zipf"
    val_dtype: str    # "f32" or "bf16" (k_val, q_val)
    val_scale: float
    dv_dtype: str
    dv_scale: float
    bank_dtype: str
    bank_scale: float
    gate_mu: float    # gates are logsigmoid(N(gate_mu, 1))
    seed: int
    zipf_s: float = 1.1
    gate_per_entry: bool = False   # g [N, C, W]: one gate per write entry instead of one per token

    @property
    def steps(self) -> int:
        return -(-self.T // self.C)

    @property
    def N(self) -> int:
        return self.steps * self.P

    @property
    def valid_last(self) -> int:
        """Valid tokens of the last step's chunks (C when T is a multiple of C)."""
        return self.T - (self.steps - 1) * self.C

    @property
    def key_bits(self) -> int:
        return max(1, math.ceil(math.log2(self.S)))

    def describe(self) -> dict:
        return {
            "workload": self.name, "P": self.P, "T": self.T, "C": self.C, "S": self.S, "hd": self.hd,
            "W": self.W, "R": self.R, "idx": self.idx, "val": self.val_dtype, "dv": self.dv_dtype,
            "bank": self.bank_dtype, "steps": self.steps, "valid_last": self.valid_last,
        }


# The five workloads of the forward. Value scales that the workload list leaves open are read
# as 1/sqrt(W) for k/q (the stated scale of the uniform W=8 case) and 0.1 for the bf16 bank.
WORKLOADS = {
    "tiny": Workload("tiny", P=1, T=1024, C=64, S=4096, hd=64, W=4, R=4, idx="uniform",
                     val_dtype="f32", val_scale=1.0, dv_dtype="f32", dv_scale=1.0,
                     bank_dtype="f32", bank_scale=1.0, gate_mu=3.0, seed=0),
    "uniform_c128": Workload("uniform_c128", P=8, T=16384, C=128, S=65536, hd=128, W=8, R=8,
                             idx="uniform", val_dtype="bf16", val_scale=1 / math.sqrt(8),
                             dv_dtype="bf16", dv_scale=1.0, bank_dtype="bf16", bank_scale=0.1,
                             gate_mu=3.0, seed=1),
    "zipf_c256": Workload("zipf_c256", P=8, T=16384, C=256, S=65536, hd=120, W=8, R=8, idx="zipf",
                          val_dtype="bf16", val_scale=1 / math.sqrt(8), dv_dtype="bf16", dv_scale=1.0,
                          bank_dtype="bf16", bank_scale=0.1, gate_mu=3.0, seed=2),
    "large": Workload("large", P=32, T=8192, C=256, S=1 << 20, hd=128, W=16, R=16, idx="uniform",
                      val_dtype="bf16", val_scale=0.25, dv_dtype="bf16", dv_scale=0.25,
                      bank_dtype="bf16", bank_scale=0.1, gate_mu=4.0, seed=3),
    "wide_ragged": Workload("wide_ragged", P=4, T=8000, C=128, S=262144, hd=960, W=4, R=4,
                            idx="uniform", val_dtype="bf16", val_scale=0.5, dv_dtype="bf16",
                            dv_scale=1.0, bank_dtype="bf16", bank_scale=0.1, gate_mu=3.0, seed=4),
}


def scaled(w: Workload, **changes) -> Workload:
    """The same distributions at other sizes (e.g. fewer tokens or streams for a parity case)."""
    return dataclasses.replace(w, **changes)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _vals(rng: np.random.Generator, shape, scale: float, dtype: str) -> np.ndarray:
    x = (rng.standard_normal(shape, dtype=np.float32) * np.float32(scale)).astype(np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def _zipf_cdf(S: int, s: float) -> np.ndarray:
    w = np.arange(1, S + 1, dtype=np.float64) ** (-s)
    c = np.cumsum(w)
    return c / c[-1]


def _stream_rngs(w: Workload, p: int):
    """Independent generators of stream p: idx K, idx Q, k, q, g, dv (bank: make_bank_stream)."""
    ss = np.random.SeedSequence([w.seed, p])
    return [np.random.default_rng(s) for s in ss.spawn(6)]


def make_inputs(w: Workload, streams=None) -> dict:
    """All per-token inputs of the workload (or of a subset of its streams), chunk-major.

    With ``streams`` given, the arrays hold only those streams, in that order, as if P were
    ``len(streams)``; each stream's data is identical to its data in the full set.
    """
    streams = list(range(w.P)) if streams is None else list(streams)
    Ps, st, C, W, R, hd = len(streams), w.steps, w.C, w.W, w.R, w.hd
    k_idx = np.empty((st, Ps, C, W), np.int32)
    q_idx = np.empty((st, Ps, C, R), np.int32)
    vt = np.uint16 if w.val_dtype == "bf16" else np.float32
    dt = np.uint16 if w.dv_dtype == "bf16" else np.float32
    k_val = np.empty((st, Ps, C, W), vt)
    q_val = np.empty((st, Ps, C, R), vt)
    gshape = (st, C, W) if w.gate_per_entry else (st, C)
    g = np.empty((st, Ps) + gshape[1:], np.float32)
    dv = np.empty((st, Ps, C, hd), dt)
    cdf = _zipf_cdf(w.S, w.zipf_s) if w.idx == "zipf" else None
    for i, p in enumerate(streams):
        r_k, r_q, r_kv, r_qv, r_g, r_dv = _stream_rngs(w, p)
        for arr, rng, lanes in ((k_idx, r_k, W), (q_idx, r_q, R)):
            if cdf is None:
                ids = rng.integers(0, w.S, size=(st, C, lanes), dtype=np.int64)
            else:
                u = rng.random(size=(st, C, lanes))
                ids = np.minimum(np.searchsorted(cdf, u, side="right"), w.S - 1)
            arr[:, i] = ids.astype(np.int32)
        k_val[:, i] = _vals(r_kv, (st, C, W), w.val_scale, w.val_dtype)
        q_val[:, i] = _vals(r_qv, (st, C, R), w.val_scale, w.val_dtype)
        z = r_g.standard_normal(gshape) + w.gate_mu
        g[:, i] = (np.minimum(z, 0.0) - np.log1p(np.exp(-np.abs(z)))).astype(np.float32)
        dv[:, i] = _vals(r_dv, (st, C, hd), w.dv_scale, w.dv_dtype)
    if w.valid_last < C:   # the stream's end falls inside the last step's chunks
        k_idx[st - 1, :, w.valid_last:] = -1
        q_idx[st - 1, :, w.valid_last:] = -1
    N = st * Ps
    return {
        "k_idx": k_idx.reshape(N, C, W), "q_idx": q_idx.reshape(N, C, R),
        "k_val": k_val.reshape(N, C, W), "q_val": q_val.reshape(N, C, R),
        "g": g.reshape((N, C, W) if w.gate_per_entry else (N, C)), "dv": dv.reshape(N * C, hd),
        "streams": streams, "P": Ps, "steps": st, "valid_last": w.valid_last,
    }


def make_bank_stream(w: Workload, p: int) -> np.ndarray:
    """Initial bank rows of stream p: [S, hd], normal with the workload's scale."""
    rng = np.random.default_rng(np.random.SeedSequence([w.seed, p, 7]))
    x = (rng.standard_normal((w.S, w.hd), dtype=np.float32) * np.float32(w.bank_scale)).astype(np.float32)
    return f32_to_bf16_bits(x) if w.bank_dtype == "bf16" else x


# ---- inputs of the backward's Phase A (the backward of DW) ------------------------------------
# The Phase-A contract (pa_dc_cuda.py, module docstring) takes, besides the forward's inputs and
# Phase-1 outputs: beta [N, C] (a write strength per token, here sigmoid(N(0, 1))), d_dva [N, C, hd]
# float32 (the gradient of the token rows, normal with dv_scale), the grad rows [P * S, hd] (normal,
# scale 1) and the dense compact snapshot rows (any rows of the bank dtype: normal with bank_scale).

def make_backward_inputs(w: Workload, streams=None) -> dict:
    """beta [N, C] float32 and dva [N, C, hd] float32, chunk-major like make_inputs."""
    streams = list(range(w.P)) if streams is None else list(streams)
    Ps, st, C, hd = len(streams), w.steps, w.C, w.hd
    beta = np.empty((st, Ps, C), np.float32)
    dva = np.empty((st, Ps, C, hd), np.float32)
    for i, p in enumerate(streams):
        r_b, r_d = [np.random.default_rng(s) for s in np.random.SeedSequence([w.seed, p, 11]).spawn(2)]
        z = r_b.standard_normal((st, C))
        beta[:, i] = (1.0 / (1.0 + np.exp(-z))).astype(np.float32)
        dva[:, i] = (r_d.standard_normal((st, C, hd), dtype=np.float32) * np.float32(w.dv_scale)).astype(np.float32)
    N = st * Ps
    return {"beta": beta.reshape(N, C), "dva": dva.reshape(N, C, hd)}


def make_grad_stream(w: Workload, p: int, rows=None) -> np.ndarray:
    """Grad rows of stream p before the backward's first Phase-A step: [S, hd] float32 normal (or
    only the rows ``rows`` of it, drawn the same)."""
    rng = np.random.default_rng(np.random.SeedSequence([w.seed, p, 13]))
    x = rng.standard_normal((w.S, w.hd), dtype=np.float32)
    return x if rows is None else x[rows]


def make_snapshot_chunk(w: Workload, c: int) -> np.ndarray:
    """Dense compact snapshot rows of chunk c: [C * W, hd] in the bank dtype (uint16 bits for bf16)."""
    rng = np.random.default_rng(np.random.SeedSequence([w.seed, c, 17]))
    x = (rng.standard_normal((w.C * w.W, w.hd), dtype=np.float32) * np.float32(w.bank_scale)).astype(np.float32)
    return f32_to_bf16_bits(x) if w.bank_dtype == "bf16" else x


def make_read_grads(w: Workload, streams=None) -> np.ndarray:
    """gr [N, C, hd] float32: the gradient of every token's read result (GDS, the read side of the
    backward), normal with scale 1, chunk-major like make_inputs."""
    streams = list(range(w.P)) if streams is None else list(streams)
    Ps, st, C, hd = len(streams), w.steps, w.C, w.hd
    gr = np.empty((st, Ps, C, hd), np.float32)
    for i, p in enumerate(streams):
        rng = np.random.default_rng(np.random.SeedSequence([w.seed, p, 19]))
        gr[:, i] = rng.standard_normal((st, C, hd), dtype=np.float32)
    return gr.reshape(st * Ps, C, hd)


def make_read_weights(w: Workload, streams=None) -> np.ndarray:
    """q_w [N, C, R]: the weights of the forward's read-side gather, normal with the workload's value
    scale, in the value dtype (uint16 bits for bf16), chunk-major like make_inputs."""
    streams = list(range(w.P)) if streams is None else list(streams)
    Ps, st, C, R = len(streams), w.steps, w.C, w.R
    out = np.empty((st, Ps, C, R), np.float32)
    for i, p in enumerate(streams):
        rng = np.random.default_rng(np.random.SeedSequence([w.seed, p, 29]))
        out[:, i] = (rng.standard_normal((st, C, R), dtype=np.float32) * np.float32(w.val_scale)).astype(np.float32)
    out = out.reshape(st * Ps, C, R)
    return f32_to_bf16_bits(out) if w.val_dtype == "bf16" else out


def make_write_weights(w: Workload, streams=None) -> np.ndarray:
    """write_w [N, C, W] float32: the weights of the backward's token gather (GWR), normal with the
    workload's value scale, chunk-major like make_inputs."""
    streams = list(range(w.P)) if streams is None else list(streams)
    Ps, st, C, W = len(streams), w.steps, w.C, w.W
    out = np.empty((st, Ps, C, W), np.float32)
    for i, p in enumerate(streams):
        rng = np.random.default_rng(np.random.SeedSequence([w.seed, p, 23]))
        out[:, i] = (rng.standard_normal((st, C, W), dtype=np.float32) * np.float32(w.val_scale)).astype(np.float32)
    return out.reshape(st * Ps, C, W)
