"""Benchmark of the sparse-delta-memory forward (Phase 1 + DW over every step) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload large] [--impl ours|reference]

One step = one forward over the whole workload: Phase 1 of every chunk and the decay-and-write
of every step, through the library's C ABI. The default workload is the large one (P = 32
streams x T = 8192 tokens, C = 256, S = 2^20 slots per stream, hd = 128, W = R = 16, bf16; an
8 GiB bank, far larger than L2, so no flush is needed between steps). Under torchrun each rank
runs its own copy of the workload (independent streams: weak scaling, no collective on the data
path); rank 0 prints one JSON line.

--impl reference times the float64 CPU oracle (the only reference this method has) on a bounded
sample of the same workload, on this host's cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import WORKLOADS, make_inputs, scaled  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # the GB300's nominal HBM3e bandwidth (the measured copy peak is the roofline)

METRIC_FWD = "SDM forward (Phase1+DW) tokens/sec and achieved HBM GB/s vs GB300 peak"
METRIC_PA = "SDM backward Phase A (the backward of DW) tokens/sec and achieved HBM GB/s vs GB300 peak"
METRIC_GDS = "SDM backward GDS (read-side dots + grad scatter) tokens/sec and achieved HBM GB/s vs GB300 peak"
METRIC_GWR = "SDM backward GWR (write-side token gather) tokens/sec and achieved HBM GB/s vs GB300 peak"
METRIC_READ = "SDM forward read-side gather tokens/sec and achieved HBM GB/s vs GB300 peak"

# DRAM bytes (read + write) per launch from one ncu capture, keyed by workload, kernel and the
# hash of the kernel's CUDA sources at capture time. A source change voids the figure: the bench
# line then reports null traffic.
NCU_TRAFFIC = {
    # the forward (bench.py): the timed loop's Phase 1 (all outputs) and DW, one launch each at full size
    "large:dw:ef4ffb8f7982": 1162345728 + 979819008,
    "large:phase1:4c17089261ec": 52839680 + 723335680,
    # the read gather (bench.py --read): one launch (one step) of the timed pass
    "large:read:4629bd9f0dbc": 34294528 + 6400,
    # Phase A (bench.py --pa): one launch captured on the large workload with S = 2^18 slots per stream
    # (same grid and group count per chunk), scaled by the groups ratio 4186081 / 4161534
    "large:pa:25bcbddec3cb": round((106349824 + 43558912) * 4186081 / 4161534),
    # GDS (bench.py --gds): the dots and the scatter launch of one step (S = 2^18 capture, same grid),
    # scaled by the read-groups ratio 4185964 / 4161643
    "large:gds:4a65ad955f9a": round((38026752 + 72657920 + 19646208) * 4185964 / 4161643),
    # GWR (bench.py --gwr): one launch (S = 2^18 capture; the same write entries, rows per entry)
    "large:gwr:8ac2b9913f79": 69718784 + 85760,
}


def src_hash(dom: str) -> str:
    """Hash of the code of the sources that build kernel domain ``dom``: its own .cu file, the local
    headers it includes and the launch code of sdm_api.cu. Comment-only and blank lines do not count,
    and a source added for another kernel does not change it."""
    h = hashlib.sha1()
    d = os.path.join(ROOT, "sparse_slot_memory_gb300", "csrc")
    own = f"sdm_{dom}.cu"
    with open(os.path.join(d, own), encoding="utf-8") as fh:
        heads = sorted(set(re.findall(r'#include "([^"/]+\.cuh)"', fh.read())))
    for f in ["sdm_api.cu", own] + heads:
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode())
            for line in fh:
                t = line.strip()
                if t and not t.startswith("//"):
                    h.update(t.encode())
    return h.hexdigest()[:12]


def traffic_source(key: str, traffic) -> str:
    if traffic is None:
        return f"null: no ncu capture of these sources ({key})"
    return f"ncu dram__bytes_read.sum + dram__bytes_write.sum, one capture of sources {key} (profiles/)"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons around and during the timed region.

    The sampler runs every 5 ms from before the warm-up to after the timed region; ``mark`` records
    the host time at the start and end of the timed region. The summary takes the samples inside
    that window, or, when the window is shorter than the sampling period, the nearest sample on each
    side of it (both taken with the GPU busy: the warm-up before, the last launches after)."""

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.window = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "5"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t_end = time.time() + 3.0   # sampling is live before the work starts
            while not self.rows and time.time() < t_end:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.02)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, busy_ms: float | None = None):
        rows = list(self.rows)
        if not rows or self.window is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        t0, t1 = self.window
        inside = [r for (t, r) in rows if t0 <= t <= t1]
        how = "inside the timed region"
        if not inside:
            before = [r for (t, r) in rows if t < t0][-1:]
            after = [r for (t, r) in rows if t > t1][:1]
            inside = before + after
            how = "nearest sample before and after the timed region (shorter than the 5 ms sampling period)"
        sm = [float(r[0]) for r in inside if r and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in inside if len(r) > 1 and r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if len(r) > 3 + i and r[3 + i] == "Active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": reasons, "samples": len(inside), "how": how}
        if busy_ms is not None and sm:
            out["ms_x_mhz"] = busy_ms * statistics.median(sm)
        return out


def count_groups(x, w):
    """Slot groups with at least one valid write entry, per chunk (exactly, from the data)."""
    k = x["k_idx"].reshape(x["k_idx"].shape[0], -1).astype(np.int64)
    N = k.shape[0]
    total = 0
    for c0 in range(0, N, 256):
        blk = np.sort(k[c0:c0 + 256], axis=1)
        valid = blk >= 0
        distinct = np.concatenate([np.ones((blk.shape[0], 1), bool), blk[:, 1:] != blk[:, :-1]], axis=1)
        total += int((distinct & valid).sum())
    return total


def algorithmic_bytes(w, x, groups, saving=False):
    """Algorithmic bytes per forward: inputs read once, outputs written once,
    dv rows read once, per slot group one base-row read and one row write (the saving forward:
    and one snapshot row write)."""
    vt = 2 if w.val_dtype == "bf16" else 4
    dvt = 2 if w.dv_dtype == "bf16" else 4
    bt = 2 if w.bank_dtype == "bf16" else 4
    N, C, W, R = x["k_idx"].shape[0], w.C, w.W, w.R
    tok = N * C
    p1_in = tok * (W * (4 + vt) + R * (4 + vt) + 4)
    p1_out = tok * (W * (4 + 4 + vt + vt + 1 + 1 + 4) + R * (4 + vt + 4 + 1 + 1)) + N * C * C * 4 * 2
    dw = tok * w.hd * dvt + groups * w.hd * bt * (3 if saving else 2)
    return {"phase1": p1_in + p1_out, "dw": dw, "total": p1_in + p1_out + dw}


def valid_tokens(w, P):
    return P * w.T


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sparse_slot_memory_gb300 as sdm

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sdm.build()
    w = WORKLOADS[args.workload]
    if args.streams:
        w = scaled(w, P=args.streams)
    if args.slots:
        w = scaled(w, S=args.slots)
    if getattr(args, "idx", None):
        w = scaled(w, idx=args.idx)
    x = make_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)

    def dev(a, dt):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(a)
        return t.cuda()

    host = {"k_idx": x["k_idx"], "q_idx": x["q_idx"], "k_val": x["k_val"], "q_val": x["q_val"], "g": x["g"],
            "dv": x["dv"]}
    dts = {"k_idx": "i", "q_idx": "i", "g": "f32", "k_val": w.val_dtype, "q_val": w.val_dtype, "dv": w.dv_dtype}
    d = {k: dev(v, dts[k]) for k, v in host.items()}
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + w.seed + rank)
    bdt = torch.bfloat16 if w.bank_dtype == "bf16" else torch.float32
    bank = (torch.randn(w.P * w.S, w.hd, device="cuda", generator=gen) * w.bank_scale).to(bdt)
    ws = sdm.alloc_workspace(shape)
    out = sdm.alloc_outputs(shape)
    stream = torch.cuda.current_stream()
    # the saving forward also writes the dense compact snapshot (one base row per group)
    snap = sdm.alloc_snapshot(shape) if args.saving else None

    def dw():
        if snap is None:
            sdm.dw(shape, d["dv"], bank, ws)
        else:
            sdm.dw_saving(shape, d["dv"], bank, snap, ws)

    p1 = sdm.phase1 if snap is None else sdm.phase1_saving

    def step():
        p1(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], out, ws)
        dw()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0
    # the kernel's own counters of one Phase 1 (untimed): its valid write groups give the DW's bytes
    sout = sdm.alloc_outputs(shape, fields=("A", "QK", "stats"))
    p1(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], sout, ws)
    torch.cuda.synchronize()
    p1_stats = dict(zip(sdm.STATS, (int(v) for v in sout["stats"].cpu())))
    del sout

    # timed region: K forwards back to back (the DW-side kernels launch early, as programmatic
    # dependents, and wait for their predecessor inside); then the per-kernel durations from a second
    # timed loop of K forwards with an event between Phase 1 and the DW (an event there stops that
    # early launch, so the forward's value comes from the first loop)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        h0 = time.time()
        t0.record(stream)
        for i in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        for i in range(args.steps):
            ev[i][0].record(stream)
            p1(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], out, ws)
            ev[i][1].record(stream)
            dw()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        clk.mark(h0, time.time())
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    p1_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    dw_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    assert sdm.device_status(ws) == 0
    if world > 1:
        tt = torch.tensor([ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    tokens = valid_tokens(w, w.P)
    value = tokens * world / (ms / 1e3)

    # End to end through the public API with host buffers: per step, the inputs H2D from pinned host
    # memory, the forward, every Phase-1 output D2H to pinned host memory. The bank is resident state.
    # Two buffer sets pipeline the steps: step i's outputs travel D2H (one copy stream) while step
    # i + 1's inputs travel H2D (another) and step i + 1 computes (the launching stream).
    e2e = None
    if not args.no_e2e:
        pin = [{k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16) if dts[k] == "bf16" else np.ascontiguousarray(v))
                .pin_memory() for k, v in host.items()} for _ in range(2)]
        dbuf = [d, {k: torch.empty_like(v) for k, v in d.items()}]
        obuf = [out, sdm.alloc_outputs(shape)]
        outs_h = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()} for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in pin[0].values())
        d2h = sum(v.numel() * v.element_size() for v in out.values())
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):   # every buffer starts free
            ev_comp[b].record(stream)
            ev_out[b].record(stream)

        def e2e_step(i):
            b = i & 1
            di, oi = dbuf[b], obuf[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_comp[b])            # step i - 2 has read these inputs
                for k, v in pin[b].items():
                    dst = di[k].view(torch.int16) if dts[k] == "bf16" else di[k]
                    dst.copy_(v, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])               # step i - 2's outputs have left
            if snap is None:
                sdm.forward_chunks(shape, di["k_idx"], di["q_idx"], di["k_val"], di["q_val"], di["g"], di["dv"], bank,
                                   oi, ws)
            else:
                sdm.forward_chunks_saving(shape, di["k_idx"], di["q_idx"], di["k_val"], di["q_val"], di["g"], di["dv"],
                                          bank, snap, oi, ws)
            ev_comp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                for k, v in oi.items():
                    outs_h[b][k].copy_(v, non_blocking=True)
                ev_out[b].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        n2 = max(4, min(args.steps, 12))
        a0 = time.perf_counter()
        for i in range(n2):
            e2e_step(i)
        torch.cuda.synchronize()
        e_ms = (time.perf_counter() - a0) * 1e3 / n2
        if world > 1:
            tt = torch.tensor([e_ms], device="cuda")
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e_ms = float(tt.item())
        e2e = {"value": tokens * world / (e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "note": "per step: inputs H2D from pinned host memory, the forward, every Phase-1 output D2H to "
                       "pinned host memory; steps pipelined over two buffer sets and two copy streams; the bank is "
                       "resident state; host wall clock from the first copy to the last byte home"}

    groups = p1_stats["groups"]
    assert groups == count_groups(x, w), (p1_stats, count_groups(x, w))
    ab = algorithmic_bytes(w, x, groups, saving=args.saving)
    peak, peak_kind = peaks()
    dom = "dw" if dw_ms >= p1_ms else "phase1"
    dom_ms = dw_ms if dom == "dw" else p1_ms
    achieved = ab[dom] / (dom_ms / 1e3) / 1e9
    key = f"{args.workload}:{dom}:{src_hash(dom)}"
    traffic = NCU_TRAFFIC.get(key)
    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            x0 = make_inputs(w, streams=[0])
            cpu = cpu_baselines("fwd", args, w, cpu_baseline(w, x0, budget_s=args.cpu_seconds))
        result = {
            "metric": METRIC_FWD,
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.val_dtype, "data": "synthetic (seeded generators of the workload's distributions)",
            "config": {"workload": w.name + ("+saving" if args.saving else ""), **{k: v for k, v in w.describe().items() if k != "workload"},
                       "tokens_per_step_per_gpu": tokens, "parallelism": f"replicas x{world} (independent streams)",
                       "l2": "inputs larger than L2 (8 GiB bank)"},
            "hbm_gbs_total": ab["total"] / (ms / 1e3) / 1e9,
            "kernels_ms": {"phase1": p1_ms, "dw": dw_ms},
            "algorithmic_bytes": ab, "groups": groups, "p1_stats": p1_stats,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                         "peak_kind": f"{peak_kind} (hbm copy GB/s)", "unit": "GB/s", "frac": achieved / peak,
                         "frac_nominal": achieved / NOMINAL_HBM_GBS, "traffic": traffic,
                         "traffic_source": traffic_source(key, traffic),
                         "total_frac": ab["total"] / (ms / 1e3) / 1e9 / peak,
                         "total_frac_nominal": ab["total"] / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 2 * 3 * args.steps,   # per forward: Phase 1, the long-group sums, the DW; two loops
            "clocks": clk.summary(ms * args.steps),
            "impl": "ours",
        }
        print(json.dumps(result))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def pa_algorithmic_bytes(w, groups, grad_bytes):
    """Bytes of one Phase-A pass over every step (the backward of DW): per valid group the grad row
    read and written, the snapshot row read and the bank row written, and the first member's slot
    id; per write entry its sorted-row word and the two f32 outputs, plus k, log_k and cpe; per
    token its d_dva row (f32) and beta."""
    vt = 2 if w.val_dtype == "bf16" else 4
    bt = 2 if w.bank_dtype == "bf16" else 4
    tok = w.N * w.C
    ent = tok * w.W
    return groups * (w.hd * (2 * grad_bytes + 2 * bt) + 4) + ent * (4 + 8 + vt + 4 + vt) + tok * (w.hd * 4 + 4)


def pa_cpu_baseline(w, x, b, budget_s=12.0, max_chunks=None):
    """The oracle's Phase A as it stands (float64, single thread) on a bounded sample: the chunks
    of stream 0, last step first, on the rows that stream touches, until ~budget_s seconds passed.
    ``x`` / ``b`` hold stream 0 alone (make_inputs / make_backward_inputs with streams=[0])."""
    import oracle

    P, C = x["P"], w.C
    p = 0
    ids = x["k_idx"][p::P].ravel()
    slots = np.unique(ids[ids >= 0])
    rng = np.random.default_rng(5)
    grad = rng.standard_normal((len(slots), w.hd))
    bank = np.zeros((len(slots), w.hd))
    kvf = oracle.as_f64(x["k_val"], w.val_dtype)
    t0 = time.perf_counter()
    chunks = 0
    for ti in range(w.steps - 1, -1, -1):
        c = ti * P + p
        V = w.valid_last if ti == w.steps - 1 else C
        kk = np.searchsorted(slots, x["k_idx"][c]).astype(np.int32)
        kk[x["k_idx"][c] < 0] = -1
        ng = len(oracle.snapshot_slots(kk, S=len(slots), V=V))
        lk = -rng.random((C, w.W))
        cpe = np.exp(lk)
        oracle.pa_chunk(grad, bank, rng.standard_normal((ng, w.hd)), kk, kvf[c], lk, cpe, b["beta"][c], b["dva"][c],
                        S=len(slots), V=V)
        chunks += 1
        if time.perf_counter() - t0 > budget_s or (max_chunks and chunks >= max_chunks):
            break
    dt = time.perf_counter() - t0
    toks = chunks * C
    return {"value": toks / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{chunks} chunks ({toks} tokens) of stream 0, last step first: Phase A, float64, "
                      f"{dt:.1f} s single-threaded"}


def run_pa(args):
    """The backward's Phase A over every step of the workload: one bench step = sdm_pa over steps
    [0, steps) (one launch per step, last step first). Its inputs come from one untimed saving
    forward (sorted rows, log_k, cpe, the dense compact snapshot) and the seeded generators (beta,
    d_dva); grad rows are float32 (the --pa-grad bf16 option: the bank's format)."""
    import torch

    import sparse_slot_memory_gb300 as sdm
    from synth import make_backward_inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sdm.build()
    w = WORKLOADS[args.workload]
    if args.streams:
        w = scaled(w, P=args.streams)
    if args.slots:
        w = scaled(w, S=args.slots)
    if getattr(args, "idx", None):
        w = scaled(w, idx=args.idx)
    x = make_inputs(w)
    b = make_backward_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)

    def dev(a, dt):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(a)
        return t.cuda()

    d = {"k_idx": dev(x["k_idx"], "i"), "q_idx": dev(x["q_idx"], "i"), "k_val": dev(x["k_val"], w.val_dtype),
         "q_val": dev(x["q_val"], w.val_dtype), "g": dev(x["g"], "f32"), "dv": dev(x["dv"], w.dv_dtype),
         "beta": dev(b["beta"], "f32"), "dva": dev(b["dva"], "f32")}
    del b
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2000 + w.seed + rank)
    bdt = torch.bfloat16 if w.bank_dtype == "bf16" else torch.float32
    bank = (torch.randn(w.P * w.S, w.hd, device="cuda", generator=gen) * w.bank_scale).to(bdt)
    ws = sdm.alloc_workspace(shape)
    out = sdm.alloc_outputs(shape, fields=("log_k", "cpe", "sorted_k", "ngroups", "repeats"))
    snap = sdm.alloc_snapshot(shape)
    sdm.forward_chunks_saving(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], d["dv"], bank, snap,
                              out, ws)
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0
    groups = int(out["ngroups"].sum().item())
    del ws
    gdt = torch.bfloat16 if args.pa_grad == "bf16" else torch.float32
    grad = torch.randn(w.P * w.S, w.hd, device="cuda", generator=gen).to(gdt)
    d_k_eff = torch.empty((w.N, w.C, w.W), device="cuda")
    grad_g = torch.empty((w.N, w.C, w.W), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        sdm.pa(shape, out["sorted_k"], d["k_idx"], d["k_val"], out["log_k"], out["cpe"], d["beta"], d["dva"], grad,
               bank, snap, d_k_eff, grad_g, 0, w.steps, status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        h0 = time.time()
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        clk.mark(h0, time.time())
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    assert int(status.item()) == 0
    if world > 1:
        tt = torch.tensor([ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    tokens = valid_tokens(w, w.P)
    value = tokens * world / (ms / 1e3)

    # End to end through the public call with host buffers: per pass, every per-token input of the
    # pass H2D from pinned host memory (sorted rows, ids, k, log_k, cpe, beta, d_dva, the snapshot),
    # the pass, both outputs D2H; grad and bank rows are resident state.
    e2e = None
    if not args.no_e2e:
        ins = {"sorted_k": out["sorted_k"], "k_idx": d["k_idx"], "k_val": d["k_val"], "log_k": out["log_k"],
               "cpe": out["cpe"], "beta": d["beta"], "dva": d["dva"], "snap": snap}
        pin = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) for k, v in ins.items()}
        outs_h = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in
                  (("d_k_eff", d_k_eff), ("grad_g", grad_g))}
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = sum(v.numel() * v.element_size() for v in outs_h.values())

        def e2e_step():
            for k, v in pin.items():
                ins[k].copy_(v, non_blocking=True)
            sdm.pa(shape, ins["sorted_k"], ins["k_idx"], ins["k_val"], ins["log_k"], ins["cpe"], ins["beta"],
                   ins["dva"], grad, bank, ins["snap"], d_k_eff, grad_g, 0, w.steps, status)
            outs_h["d_k_eff"].copy_(d_k_eff, non_blocking=True)
            outs_h["grad_g"].copy_(grad_g, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n2 = max(3, min(args.steps, 8))
        a0 = time.perf_counter()
        for _ in range(n2):
            e2e_step()
        torch.cuda.synchronize()
        e_ms = (time.perf_counter() - a0) * 1e3 / n2
        e2e = {"value": tokens * world / (e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "note": "per pass: every per-token input H2D from pinned host memory, the pass, both outputs D2H; "
                       "one stream; grad and bank rows resident; host wall clock"}

    peak, peak_kind = peaks()
    ab = pa_algorithmic_bytes(w, groups, 2 if args.pa_grad == "bf16" else 4)
    kern_ms = ms / w.steps                      # one launch per workload step
    achieved = ab / w.steps / (kern_ms / 1e3) / 1e9
    key = f"{args.workload}:pa{'_bf16grad' if args.pa_grad == 'bf16' else ''}:{src_hash('pa')}"
    result = None
    if rank == 0:
        cpu = None if args.no_cpu_baseline else cpu_baselines(
            "pa", args, w, pa_cpu_baseline(w, make_inputs(w, streams=[0]), make_backward_inputs(w, streams=[0]),
                                           budget_s=args.cpu_seconds))
        result = {
            "metric": METRIC_PA,
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded generators; Phase-1 outputs and snapshot from one saving forward)",
            "config": {"workload": w.name + "+phaseA" + ("+bf16grad" if args.pa_grad == "bf16" else ""),
                       **{k: v for k, v in w.describe().items() if k != "workload"},
                       "grad": args.pa_grad, "tokens_per_step_per_gpu": tokens,
                       "parallelism": f"replicas x{world} (independent streams)",
                       "l2": "inputs larger than L2 (16 GiB f32 grad rows, 8 GiB bank)"},
            "kernels_ms": {"pa_per_launch": kern_ms}, "algorithmic_bytes": ab, "groups": groups,
            "roofline": {"bound": "hbm", "kernel": "pa", "achieved": achieved, "peak": peak,
                         "peak_kind": f"{peak_kind} (hbm copy GB/s)", "unit": "GB/s", "frac": achieved / peak,
                         "frac_nominal": achieved / NOMINAL_HBM_GBS, "traffic": NCU_TRAFFIC.get(key),
                         "traffic_source": traffic_source(key, NCU_TRAFFIC.get(key))},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": w.steps * args.steps,
            "clocks": clk.summary(ms * args.steps), "impl": "ours",
        }
        print(json.dumps(result))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def count_read_groups(x):
    """Slots with at least one valid read entry, per chunk (exactly, from the data)."""
    q = x["q_idx"].reshape(x["q_idx"].shape[0], -1).astype(np.int64)
    total = 0
    for c0 in range(0, q.shape[0], 256):
        blk = np.sort(q[c0:c0 + 256], axis=1)
        distinct = np.concatenate([np.ones((blk.shape[0], 1), bool), blk[:, 1:] != blk[:, :-1]], axis=1)
        total += int((distinct & (blk >= 0)).sum())
    return total


def gds_algorithmic_bytes(w, qgroups, grad_bytes):
    """Bytes of one GDS pass over every step (the read side of the backward): per read group its bank
    row read (the dots) and its grad row read and written (the scatter); per read entry its sorted-row
    word, slot id, q, log_q and d_q_w; per token its reading-gradient row (f32)."""
    vt = 2 if w.val_dtype == "bf16" else 4
    bt = 2 if w.bank_dtype == "bf16" else 4
    tok = w.N * w.C
    return qgroups * w.hd * (bt + 2 * grad_bytes) + tok * w.R * (4 + 4 + vt + 4 + 4) + tok * w.hd * 4


def gds_cpu_baseline(w, x, gr, budget_s=12.0, max_chunks=None):
    """The oracle's GDS as it stands (float64, single thread) on a bounded sample: the chunks of stream 0,
    last step first, on the rows that stream reads. ``x`` / ``gr`` hold stream 0 alone."""
    import oracle

    P, C = x["P"], w.C
    ids = x["q_idx"][0::P].ravel()
    slots = np.unique(ids[ids >= 0])
    rng = np.random.default_rng(6)
    grad = rng.standard_normal((len(slots), w.hd))
    bank = rng.standard_normal((len(slots), w.hd))
    qvf = oracle.as_f64(x["q_val"], w.val_dtype)
    t0 = time.perf_counter()
    chunks = 0
    for ti in range(w.steps - 1, -1, -1):
        c = ti * P
        V = w.valid_last if ti == w.steps - 1 else C
        qq = np.searchsorted(slots, x["q_idx"][c]).astype(np.int32)
        qq[x["q_idx"][c] < 0] = -1
        oracle.gds_chunk(grad, bank, qq, qvf[c], -rng.random((C, w.R)), gr[c], S=len(slots), V=V)
        chunks += 1
        if time.perf_counter() - t0 > budget_s or (max_chunks and chunks >= max_chunks):
            break
    dt = time.perf_counter() - t0
    toks = chunks * C
    return {"value": toks / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{chunks} chunks ({toks} tokens) of stream 0, last step first: GDS, float64, "
                      f"{dt:.1f} s single-threaded"}


def run_gds(args):
    """GDS over every step of the workload: one bench step = sdm_gds over steps [0, steps) (two launches
    per step, last step first). sorted_q and log_q come from one untimed Phase 1 on the GPU, the reading
    gradients from the seeded generator; grad rows are float32 (--pa-grad bf16: the bank's format)."""
    import torch

    import sparse_slot_memory_gb300 as sdm
    from synth import make_read_grads

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sdm.build()
    w = WORKLOADS[args.workload]
    if args.streams:
        w = scaled(w, P=args.streams)
    if args.slots:
        w = scaled(w, S=args.slots)
    if getattr(args, "idx", None):
        w = scaled(w, idx=args.idx)
    x = make_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)

    def dev(a, dt):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(a)
        return t.cuda()

    d = {"k_idx": dev(x["k_idx"], "i"), "q_idx": dev(x["q_idx"], "i"), "k_val": dev(x["k_val"], w.val_dtype),
         "q_val": dev(x["q_val"], w.val_dtype), "g": dev(x["g"], "f32"), "gr": dev(make_read_grads(w), "f32")}
    ws = sdm.alloc_workspace(shape)
    out = sdm.alloc_outputs(shape, fields=("log_q", "sorted_q", "repeats"))
    sdm.phase1(shape, d["k_idx"], d["q_idx"], d["k_val"], d["q_val"], d["g"], out, ws)
    torch.cuda.synchronize()
    assert sdm.device_status(ws) == 0
    del ws
    gen = torch.Generator(device="cuda")
    gen.manual_seed(3000 + w.seed + rank)
    bdt = torch.bfloat16 if w.bank_dtype == "bf16" else torch.float32
    bank = (torch.randn(w.P * w.S, w.hd, device="cuda", generator=gen) * w.bank_scale).to(bdt)
    gdt = torch.bfloat16 if args.pa_grad == "bf16" else torch.float32
    grad = torch.randn(w.P * w.S, w.hd, device="cuda", generator=gen).to(gdt)
    d_q_w = torch.empty((w.N, w.C, w.R), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        sdm.gds(shape, out["sorted_q"], d["q_idx"], d["q_val"], out["log_q"], d["gr"], bank, grad, d_q_w, 0, w.steps,
                status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        h0 = time.time()
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        clk.mark(h0, time.time())
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    assert int(status.item()) == 0
    if world > 1:
        tt = torch.tensor([ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    tokens = valid_tokens(w, w.P)
    value = tokens * world / (ms / 1e3)

    # End to end with host buffers: per pass, every per-token input H2D from pinned host memory (sorted
    # read rows, ids, q, log_q, the reading gradients), the pass, d_q_w D2H; grad and bank rows resident.
    e2e = None
    if not args.no_e2e:
        ins = {"sorted_q": out["sorted_q"], "q_idx": d["q_idx"], "q_val": d["q_val"], "log_q": out["log_q"],
               "gr": d["gr"]}
        pin = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) for k, v in ins.items()}
        out_h = torch.empty(d_q_w.shape, dtype=d_q_w.dtype, pin_memory=True)
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = out_h.numel() * out_h.element_size()

        def e2e_step():
            for k, v in pin.items():
                ins[k].copy_(v, non_blocking=True)
            sdm.gds(shape, ins["sorted_q"], ins["q_idx"], ins["q_val"], ins["log_q"], ins["gr"], bank, grad, d_q_w, 0,
                    w.steps, status)
            out_h.copy_(d_q_w, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n2 = max(3, min(args.steps, 8))
        a0 = time.perf_counter()
        for _ in range(n2):
            e2e_step()
        torch.cuda.synchronize()
        e_ms = (time.perf_counter() - a0) * 1e3 / n2
        e2e = {"value": tokens * world / (e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "note": "per pass: every per-token input H2D from pinned host memory, the pass, d_q_w D2H; one "
                       "stream; grad and bank rows resident; host wall clock"}

    peak, peak_kind = peaks()
    qgroups = count_read_groups(x)
    ab = gds_algorithmic_bytes(w, qgroups, 2 if args.pa_grad == "bf16" else 4)
    step_ms = ms / w.steps                      # one workload step: the dots and the scatter launch
    achieved = ab / w.steps / (step_ms / 1e3) / 1e9
    key = f"{args.workload}:gds{'_bf16grad' if args.pa_grad == 'bf16' else ''}:{src_hash('gds')}"
    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            x0 = make_inputs(w, streams=[0])
            cpu = cpu_baselines("gds", args, w, gds_cpu_baseline(w, x0, make_read_grads(w, streams=[0]).astype(np.float64),
                                                                 budget_s=args.cpu_seconds))
        result = {
            "metric": METRIC_GDS,
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded generators; sorted read rows and log_q from one Phase 1)",
            "config": {"workload": w.name + "+gds" + ("+bf16grad" if args.pa_grad == "bf16" else ""),
                       **{k: v for k, v in w.describe().items() if k != "workload"},
                       "grad": args.pa_grad, "tokens_per_step_per_gpu": tokens,
                       "parallelism": f"replicas x{world} (independent streams)",
                       "l2": "inputs larger than L2 (16 GiB f32 grad rows, 8 GiB bank)"},
            "kernels_ms": {"gds_per_workload_step": step_ms}, "algorithmic_bytes": ab, "read_groups": qgroups,
            "roofline": {"bound": "hbm", "kernel": "gds (dots + scatter launches of one step)", "achieved": achieved,
                         "peak": peak, "peak_kind": f"{peak_kind} (hbm copy GB/s)", "unit": "GB/s",
                         "frac": achieved / peak, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                         "traffic": NCU_TRAFFIC.get(key), "traffic_source": traffic_source(key, NCU_TRAFFIC.get(key))},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 2 * w.steps * args.steps,
            "clocks": clk.summary(ms * args.steps), "impl": "ours",
        }
        print(json.dumps(result))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def gwr_algorithmic_bytes(w, grad_bytes):
    """Bytes of one GWR pass over every step: per write entry its grad row read, slot id, weight and
    d_k_pd; per token its dv row read and its d_delta_v row (f32) written."""
    dvt = 2 if w.dv_dtype == "bf16" else 4
    tok = w.N * w.C
    return tok * w.W * (w.hd * grad_bytes + 4 + 4 + 4) + tok * w.hd * (dvt + 4)


def gwr_cpu_baseline(w, x, ww, budget_s=12.0, max_chunks=None):
    """The oracle's GWR as it stands (float64, single thread) on a bounded sample: the chunks of stream
    0 on the rows that stream writes. ``x`` / ``ww`` hold stream 0 alone."""
    import oracle

    C = w.C
    ids = x["k_idx"].ravel()
    slots = np.unique(ids[ids >= 0])
    grad = np.random.default_rng(7).standard_normal((len(slots), w.hd))
    dvf = oracle.as_f64(x["dv"], w.dv_dtype)
    t0 = time.perf_counter()
    chunks = 0
    for ti in range(w.steps - 1, -1, -1):
        V = w.valid_last if ti == w.steps - 1 else C
        kk = np.searchsorted(slots, x["k_idx"][ti]).astype(np.int32)
        kk[x["k_idx"][ti] < 0] = -1
        oracle.gwr_chunk(grad, kk, ww[ti].astype(np.float64), dvf[ti * C:(ti + 1) * C], S=len(slots), V=V)
        chunks += 1
        if time.perf_counter() - t0 > budget_s or (max_chunks and chunks >= max_chunks):
            break
    dt = time.perf_counter() - t0
    toks = chunks * C
    return {"value": toks / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{chunks} chunks ({toks} tokens) of stream 0: GWR, float64, {dt:.1f} s single-threaded"}


def run_gwr(args):
    """GWR over every step of the workload: one bench step = sdm_gwr over steps [0, steps) (one launch per
    step). Ids and token rows are the workload's, write weights from the seeded generator, grad rows
    float32 (--pa-grad bf16: the bank's format)."""
    import torch

    import sparse_slot_memory_gb300 as sdm
    from synth import make_write_weights

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sdm.build()
    w = WORKLOADS[args.workload]
    if args.streams:
        w = scaled(w, P=args.streams)
    if args.slots:
        w = scaled(w, S=args.slots)
    if getattr(args, "idx", None):
        w = scaled(w, idx=args.idx)
    x = make_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)

    def dev(a, dt):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(a)
        return t.cuda()

    d = {"k_idx": dev(x["k_idx"], "i"), "write_w": dev(make_write_weights(w), "f32"), "dv": dev(x["dv"], w.dv_dtype)}
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4000 + w.seed + rank)
    gdt = torch.bfloat16 if args.pa_grad == "bf16" else torch.float32
    grad = torch.randn(w.P * w.S, w.hd, device="cuda", generator=gen).to(gdt)
    d_dd = torch.empty((w.N, w.C, w.hd), device="cuda")
    d_pd = torch.empty((w.N, w.C, w.W), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        sdm.gwr(shape, d["k_idx"], d["write_w"], d["dv"], grad, d_dd, d_pd, 0, w.steps, status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        h0 = time.time()
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        clk.mark(h0, time.time())
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    if world > 1:
        tt = torch.tensor([ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    tokens = valid_tokens(w, w.P)
    value = tokens * world / (ms / 1e3)

    # End to end with host buffers: per pass the ids, weights and token rows H2D from pinned memory, the
    # pass, both outputs D2H; grad rows resident.
    e2e = None
    if not args.no_e2e:
        pin = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) for k, v in d.items()}
        outs = {"d_delta_v": d_dd, "d_k_pd": d_pd}
        outs_h = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = sum(v.numel() * v.element_size() for v in outs_h.values())

        def e2e_step():
            for k, v in pin.items():
                d[k].copy_(v, non_blocking=True)
            step()
            for k, v in outs.items():
                outs_h[k].copy_(v, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n2 = max(3, min(args.steps, 8))
        a0 = time.perf_counter()
        for _ in range(n2):
            e2e_step()
        torch.cuda.synchronize()
        e_ms = (time.perf_counter() - a0) * 1e3 / n2
        e2e = {"value": tokens * world / (e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "note": "per pass: ids, weights and token rows H2D from pinned host memory, the pass, both outputs "
                       "D2H; one stream; grad rows resident; host wall clock"}

    peak, peak_kind = peaks()
    ab = gwr_algorithmic_bytes(w, 2 if args.pa_grad == "bf16" else 4)
    kern_ms = ms / w.steps
    achieved = ab / w.steps / (kern_ms / 1e3) / 1e9
    key = f"{args.workload}:gwr{'_bf16grad' if args.pa_grad == 'bf16' else ''}:{src_hash('gwr')}"
    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            cpu = cpu_baselines("gwr", args, w, gwr_cpu_baseline(w, make_inputs(w, streams=[0]),
                                                                 make_write_weights(w, streams=[0]),
                                                                 budget_s=args.cpu_seconds))
        result = {
            "metric": METRIC_GWR,
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded generators)",
            "config": {"workload": w.name + "+gwr" + ("+bf16grad" if args.pa_grad == "bf16" else ""),
                       **{k: v for k, v in w.describe().items() if k != "workload"},
                       "grad": args.pa_grad, "tokens_per_step_per_gpu": tokens,
                       "parallelism": f"replicas x{world} (independent streams)",
                       "l2": "inputs larger than L2 (16 GiB f32 grad rows)"},
            "kernels_ms": {"gwr_per_launch": kern_ms}, "algorithmic_bytes": ab,
            "roofline": {"bound": "hbm", "kernel": "gwr", "achieved": achieved, "peak": peak,
                         "peak_kind": f"{peak_kind} (hbm copy GB/s)", "unit": "GB/s", "frac": achieved / peak,
                         "frac_nominal": achieved / NOMINAL_HBM_GBS, "traffic": NCU_TRAFFIC.get(key),
                         "traffic_source": traffic_source(key, NCU_TRAFFIC.get(key))},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": w.steps * args.steps,
            "clocks": clk.summary(ms * args.steps), "impl": "ours",
        }
        print(json.dumps(result))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def read_algorithmic_bytes(w, x):
    """Bytes of one read pass over every step: per token its R ids and weights and its f32 output row;
    per read entry of a valid token with an id in [0, S) one bank row."""
    vt = 2 if w.val_dtype == "bf16" else 4
    bt = 2 if w.bank_dtype == "bf16" else 4
    ids = x["q_idx"]
    P = x["P"]
    rows = 0
    for c in range(ids.shape[0]):
        V = w.valid_last if c // P == w.steps - 1 else w.C
        q = ids[c][:V]
        rows += int(((q >= 0) & (q < w.S)).sum())
    tok = w.N * w.C
    return tok * (w.R * (4 + vt) + w.hd * 4) + rows * w.hd * bt


def read_cpu_baseline(w, x, qw, budget_s=12.0, max_chunks=None):
    """The oracle's read as it stands (float64, single thread) on a bounded sample: the chunks of stream
    0 on the rows that stream reads. ``x`` / ``qw`` hold stream 0 alone."""
    import oracle

    C = w.C
    ids = x["q_idx"].ravel()
    slots = np.unique(ids[ids >= 0])
    bank = np.random.default_rng(7).standard_normal((len(slots), w.hd))
    qwf = oracle.as_f64(qw, w.val_dtype)
    t0 = time.perf_counter()
    chunks = 0
    for ti in range(w.steps):
        V = w.valid_last if ti == w.steps - 1 else C
        kk = np.searchsorted(slots, x["q_idx"][ti]).astype(np.int32)
        kk[x["q_idx"][ti] < 0] = -1
        oracle.read_chunk(bank, kk, qwf[ti], S=len(slots), V=V)
        chunks += 1
        if time.perf_counter() - t0 > budget_s or (max_chunks and chunks >= max_chunks):
            break
    dt = time.perf_counter() - t0
    toks = chunks * C
    return {"value": toks / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{chunks} chunks ({toks} tokens) of stream 0: the read gather, float64, {dt:.1f} s single-threaded"}


def run_read(args):
    """The forward's read-side gather over every step: one bench step = sdm_read of each step in turn
    (one launch per step, as the forward runs it before each step's DW). Read ids are the workload's,
    weights from the seeded generator in the value dtype, bank rows normal in the bank dtype."""
    import torch

    import sparse_slot_memory_gb300 as sdm
    from synth import make_read_weights

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sdm.build()
    w = WORKLOADS[args.workload]
    if args.streams:
        w = scaled(w, P=args.streams)
    if args.slots:
        w = scaled(w, S=args.slots)
    if getattr(args, "idx", None):
        w = scaled(w, idx=args.idx)
    x = make_inputs(w)
    shape = sdm.ShapeSpec.from_workload(w)

    def dev(a, dt):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(a)
        return t.cuda()

    d = {"q_idx": dev(x["q_idx"], "i"), "q_w": dev(make_read_weights(w), w.val_dtype)}
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5000 + w.seed + rank)
    bank = (torch.randn(w.P * w.S, w.hd, device="cuda", generator=gen) * w.bank_scale).to(
        torch.bfloat16 if w.bank_dtype == "bf16" else torch.float32)
    y = torch.empty((w.N, w.C, w.hd), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        for t in range(w.steps):
            sdm.read(shape, d["q_idx"], d["q_w"], bank, y, t, t + 1, status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        h0 = time.time()
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        clk.mark(h0, time.time())
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    if world > 1:
        tt = torch.tensor([ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    tokens = valid_tokens(w, w.P)
    value = tokens * world / (ms / 1e3)

    # End to end with host buffers: per pass the ids and weights H2D from pinned memory, the pass, the
    # output D2H; bank rows resident.
    e2e = None
    if not args.no_e2e:
        pin = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) for k, v in d.items()}
        y_h = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = y_h.numel() * y_h.element_size()

        def e2e_step():
            for k, v in pin.items():
                d[k].copy_(v, non_blocking=True)
            step()
            y_h.copy_(y, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n2 = max(3, min(args.steps, 8))
        a0 = time.perf_counter()
        for _ in range(n2):
            e2e_step()
        torch.cuda.synchronize()
        e_ms = (time.perf_counter() - a0) * 1e3 / n2
        e2e = {"value": tokens * world / (e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "note": "per pass: ids and weights H2D from pinned host memory, the pass, the output D2H; one "
                       "stream; bank rows resident; host wall clock"}

    peak, peak_kind = peaks()
    ab = read_algorithmic_bytes(w, x)
    kern_ms = ms / w.steps
    achieved = ab / w.steps / (kern_ms / 1e3) / 1e9
    key = f"{args.workload}:read:{src_hash('read')}"
    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            cpu = cpu_baselines("read", args, w, read_cpu_baseline(w, make_inputs(w, streams=[0]),
                                                                   make_read_weights(w, streams=[0]),
                                                                   budget_s=args.cpu_seconds))
        result = {
            "metric": METRIC_READ,
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded generators)",
            "config": {"workload": w.name + "+read", **{k: v for k, v in w.describe().items() if k != "workload"},
                       "tokens_per_step_per_gpu": tokens, "parallelism": f"replicas x{world} (independent streams)",
                       "l2": "inputs larger than L2"},
            "kernels_ms": {"read_per_launch": kern_ms}, "algorithmic_bytes": ab,
            "roofline": {"bound": "hbm", "kernel": "read", "achieved": achieved, "peak": peak,
                         "peak_kind": f"{peak_kind} (hbm copy GB/s)", "unit": "GB/s", "frac": achieved / peak,
                         "frac_nominal": achieved / NOMINAL_HBM_GBS, "traffic": NCU_TRAFFIC.get(key),
                         "traffic_source": traffic_source(key, NCU_TRAFFIC.get(key))},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": w.steps * args.steps,
            "clocks": clk.summary(ms * args.steps), "impl": "ours",
        }
        print(json.dumps(result))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def cpu_baseline(w, x, budget_s=15.0, max_chunks=None):
    """The oracle as it stands (float64, single thread) on a bounded sample: whole steps of one
    stream (Phase 1 with the pair triangles, then DW), until ~budget_s seconds have passed."""
    import oracle

    P, C = x["P"], w.C
    oracle.build()
    t0 = time.perf_counter()
    chunks = 0
    p = 0
    S = w.S
    # the oracle's DW runs on the rows the sampled stream touches (compacted: same arithmetic)
    ids = x["k_idx"][p::P].ravel()
    slots = np.unique(ids[ids >= 0])
    bank = np.zeros((len(slots), w.hd))
    for ti in range(w.steps):
        c = ti * P + p
        V = w.valid_last if ti == w.steps - 1 else C
        oracle.phase1(x["k_idx"][c:c + 1], x["q_idx"][c:c + 1], x["k_val"][c:c + 1], x["q_val"][c:c + 1],
                      x["g"][c:c + 1], S=S, val_dtype=w.val_dtype, first_partial=0 if V < C else 1, valid_last=V)
        kk = np.searchsorted(slots, x["k_idx"][c]).astype(np.int32)
        kk[x["k_idx"][c] < 0] = -1
        qq = np.zeros_like(x["q_idx"][c])
        dvr = oracle.as_f64(x["dv"][c * C:(c + 1) * C], w.dv_dtype)
        oracle.dw_chunk(bank, kk, qq, x["k_val"][c], x["q_val"][c], x["g"][c], dvr, S=len(slots), V=V,
                        val_dtype=w.val_dtype, bank_dtype=w.bank_dtype)
        chunks += 1
        if time.perf_counter() - t0 > budget_s or (max_chunks and chunks >= max_chunks):
            break
    dt = time.perf_counter() - t0
    toks = chunks * C
    return {"value": toks / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{chunks} chunks ({toks} tokens) of stream 0: Phase 1 with A/QK + DW, float64, "
                      f"{dt:.1f} s single-threaded"}


def host_cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


_WORKER = {}


def _stream_sample(job):
    """One process of the all-cores CPU baseline: the single-thread oracle sample of mode ``kind`` on
    stream ``p`` of the workload for ``budget`` seconds (the stream's inputs are drawn once per
    process and kept)."""
    kind, wname, over, p, budget, mc = job
    key = (kind, wname, over, p)
    if key not in _WORKER:
        w = scaled(WORKLOADS[wname], **dict(over)) if over else WORKLOADS[wname]
        x = make_inputs(w, streams=[p])
        extra = None
        if kind == "pa":
            from synth import make_backward_inputs
            extra = make_backward_inputs(w, streams=[p])
        elif kind == "gds":
            from synth import make_read_grads
            extra = make_read_grads(w, streams=[p]).astype(np.float64)
        elif kind == "gwr":
            from synth import make_write_weights
            extra = make_write_weights(w, streams=[p])
        elif kind == "read":
            from synth import make_read_weights
            extra = make_read_weights(w, streams=[p])
        _WORKER[key] = (w, x, extra)
    w, x, extra = _WORKER[key]
    if kind == "pa":
        return pa_cpu_baseline(w, x, extra, budget_s=budget, max_chunks=mc)
    if kind == "gds":
        return gds_cpu_baseline(w, x, extra, budget_s=budget, max_chunks=mc)
    if kind == "gwr":
        return gwr_cpu_baseline(w, x, extra, budget_s=budget, max_chunks=mc)
    if kind == "read":
        return read_cpu_baseline(w, x, extra, budget_s=budget, max_chunks=mc)
    return cpu_baseline(w, x, budget_s=budget, max_chunks=mc)


class CpuPool:
    """Every host core running the oracle at once: one spawned process per core, each timing its own
    single-thread sample on its own stream; the aggregate is the sum of their rates."""

    def __init__(self, kind: str, wname: str, over: tuple, P: int):
        import multiprocessing as mp

        self.kind, self.wname, self.over, self.P = kind, wname, over, P
        self.n = os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.n)
        self.sample(1.0, 1)   # each process draws its stream and loads the oracle first (untimed)

    def sample(self, budget: float, max_chunks=None) -> dict:
        jobs = [(self.kind, self.wname, self.over, i % self.P, budget, max_chunks) for i in range(self.n)]
        res = self.pool.map(_stream_sample, jobs, chunksize=1)
        return {"value": sum(r["value"] for r in res), "unit": "tokens/s", "cores": self.n, "kind": "oracle",
                "cpu_count": os.cpu_count(), "cpu_model": host_cpu_model(),
                "sample": f"{self.n} processes at once (one per host core), each on its own stream: "
                          + res[0]["sample"].replace("stream 0", "its stream").replace(" single-threaded", "")}

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baselines(kind: str, args, w, single: dict) -> dict:
    """The two CPU rows of a GPU arm's line: the oracle on all host cores (the row's value) and on one
    core (``single_core``)."""
    over = tuple(sorted({k: v for k, v in (("P", args.streams), ("S", args.slots), ("idx", getattr(args, "idx", None)))
                         if v}.items()))
    pool = CpuPool(kind, args.workload, over, w.P)
    try:
        allc = pool.sample(args.cpu_seconds)
    finally:
        pool.close()
    single = dict(single, cpu_count=os.cpu_count(), cpu_model=host_cpu_model())
    return dict(allc, single_core=single)


def run_reference(args):
    """The reference arm: the float64 oracle of the same mode (forward, or --pa / --gds / --gwr / --read) on
    bounded samples of the same workload, on this host's cores; rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    grad_sfx = "+bf16grad" if args.pa_grad == "bf16" else ""
    if args.pa:
        metric, name = METRIC_PA, w.name + "+phaseA" + grad_sfx
    elif args.gds:
        metric, name = METRIC_GDS, w.name + "+gds" + grad_sfx
    elif args.gwr:
        metric, name = METRIC_GWR, w.name + "+gwr" + grad_sfx
    elif args.read:
        metric, name = METRIC_READ, w.name + "+read"
    else:
        metric, name = METRIC_FWD, w.name
    kind = "pa" if args.pa else "gds" if args.gds else "gwr" if args.gwr else "read" if args.read else "fwd"
    pool = CpuPool(kind, args.workload, (), w.P)   # every host core, one stream each
    try:
        for _ in range(args.warmup):
            pool.sample(1.0, 1)
        vals = []
        t0 = time.perf_counter()
        for _ in range(args.steps):
            vals.append(pool.sample(args.cpu_seconds / max(1, args.steps)))
        el = time.perf_counter() - t0
    finally:
        pool.close()
    v = statistics.mean(r["value"] for r in vals)
    print(json.dumps({
        "impl": "reference", "metric": metric,
        "value": v, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": {**w.describe(), "workload": name},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": vals[0]["cores"], "kind": "oracle",
                         "cpu_count": vals[0]["cpu_count"], "cpu_model": vals[0]["cpu_model"],
                         "sample": vals[0]["sample"]},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="large", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--streams", type=int, default=0, help="override the workload's stream count (profiling runs)")
    ap.add_argument("--slots", type=int, default=0, help="override the workload's slots per stream (profiling runs)")
    ap.add_argument("--idx", choices=["uniform", "zipf"], default=None,
                    help="override the workload's slot-id distribution (the same shape with other ids)")
    ap.add_argument("--saving", action="store_true", help="time the saving forward (DW writes the dense snapshot)")
    ap.add_argument("--pa", action="store_true", help="time the backward's Phase A over every step instead")
    ap.add_argument("--gds", action="store_true", help="time the backward's GDS (read side) over every step instead")
    ap.add_argument("--gwr", action="store_true", help="time the backward's GWR (write-side gather) over every step")
    ap.add_argument("--read", action="store_true", help="time the forward's read-side gather over every step")
    ap.add_argument("--pa-grad", default="f32", choices=["f32", "bf16"], help="grad row format of --pa / --gds")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.pa:
        run_pa(args)
    elif args.gds:
        run_gds(args)
    elif args.gwr:
        run_gwr(args)
    elif args.read:
        run_read(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
