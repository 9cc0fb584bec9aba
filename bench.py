#!/usr/bin/env python3
"""Benchmark of one absorbed-MLA decode step (absorb_q -> decode_attn -> out_proj).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config dsv3] [--impl ours|reference]

Prints ONE JSON line on rank 0.  A step is one pass of the whole hot path over
one batch of synthetic inputs already resident in HBM.  Under torchrun each rank
runs an independent replica on its own GPU (sequences never read each other's
cache, so the batch shards with no data-path collective: weak scaling); the
step time is the maximum over ranks.

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the slow baseline arm)."""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mla_decode_attention_absorbed_gb300.workloads import CONFIGS, KV_FP8_SCALE, make_inputs, to_fp8_cache  # noqa: E402

METRIC = "MLA decode TFLOP/s, HBM TB/s & roofline fraction (H=128, d_c=512+64, 1×GB300)"
DEFAULT_CONFIG = "dsv3"
L2_BYTES = 129 * 2 ** 20


# ------------------------------------------------------------------------- distributed plumbing
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return False
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return True


def barrier(active: bool):
    if active:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, active: bool, device="cpu") -> float:
    """Maximum of a host scalar over ranks (timing only: no data-path collective)."""
    if not active:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(cfg_seed: int, rank: int) -> int:
    """Each rank decodes its own independent batch."""
    return cfg_seed + 1000 * rank


# ------------------------------------------------------------------------- algorithmic work
def work(cfg, seq_lens, kv_bytes: int = 2):
    """Algorithmic FLOPs and bytes of one step; kv_bytes = bytes per cached element
    (2 for bf16, 1 for an FP8 cache: the query, o_lat and lse stay as they are)."""
    from oracle import counts  # closed-form counters, pinned against the pages
    lens = [int(x) for x in seq_lens]
    B, H, s_q = cfg.B, cfg.H, cfg.s_q
    attn_f = counts.attention_flops(H, cfg.d_c, cfg.d_rope, lens, s_q)
    attn_b = counts.attention_bytes(H, cfg.d_c, cfg.d_rope, lens, s_q) - sum(lens) * cfg.W * (2 - kv_bytes)
    abs_f = counts.absorb_flops(B, s_q, H, cfg.d_nope, cfg.d_c)
    abs_b = counts.absorb_bytes(B, s_q, H, cfg.d_nope, cfg.d_c, cfg.d_rope)
    out_f = counts.out_proj_flops(B, s_q, H, cfg.d_c, cfg.d_v)
    out_b = counts.out_proj_bytes(B, s_q, H, cfg.d_c, cfg.d_v)
    pairs = sum(counts.visible_pairs(L, s_q) for L in lens)
    return dict(attn_flops=attn_f, attn_bytes=attn_b, step_flops=attn_f + abs_f + out_f,
                step_bytes=attn_b + abs_b + out_b, pairs=pairs, tokens=B * s_q,
                cache_bytes=sum(lens) * (cfg.d_c + cfg.d_rope) * kv_bytes)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def traffic_for(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d:
        return None
    if d.get("source_sha256") != source_hash():
        return None
    return d.get("bytes_per_launch")


# The sources the attention launches are built and planned from: its kernel, the
# headers it includes, the merge, and the entry points that choose grid and plan.
# A change elsewhere (the projections, the expansion, the naive path) leaves the
# attention kernel, and so its captured DRAM traffic, as it was.
ATTN_SOURCES = ("api.cu", "attn_common.cuh", "attn_persist.cu", "attn_tc.cu", "attn_tc.cuh", "combine.cu", "common.cuh", "launch.h", "sm100.cuh", "tmap.h")


def source_hash() -> str:
    """Hash of the attention's sources with comments and blank space taken out (an
    edited comment leaves the kernel as it was)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_decode_attention_absorbed_gb300", "csrc")
    for name in ATTN_SOURCES:
        with open(os.path.join(csrc, name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", "", text)                  # line comments
        text = "\n".join(line.strip() for line in text.splitlines() if line.strip())
        h.update(name.encode())
        h.update(text.encode())
    return h.hexdigest()


# ------------------------------------------------------------------------- clocks
def nvsmi_gpu_id(local: int) -> str:
    """The id nvidia-smi should sample for CUDA device `local`: its UUID (else its
    PCI bus id).  nvidia-smi numbers GPUs its own way and ignores
    CUDA_VISIBLE_DEVICES, so an ordinal could name another user's GPU."""
    try:
        props = torch.cuda.get_device_properties(local)
        u = str(getattr(props, "uuid", "") or "")
        u = u[4:] if u.startswith("GPU-") else u
        if re.fullmatch(r"[0-9a-fA-F]{8}(-[0-9a-fA-F]{4}){3}-[0-9a-fA-F]{12}", u):
            return "GPU-" + u
        bus, devid = getattr(props, "pci_bus_id", None), getattr(props, "pci_device_id", None)
        if bus is not None and devid is not None:  # a UUID the process may not see in full
            return f"{getattr(props, 'pci_domain_id', 0):08x}:{bus:02x}:{devid:02x}.0"
    except Exception:  # noqa: BLE001 - no device properties: fall back to the ordinal
        pass
    return str(local)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.gpu = gpu_id
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "gpu": self.gpu}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "gpu": self.gpu,
                "window": "nvidia-smi every 100 ms over 1 s of the same steps untimed, then the timed steps"}


class L2Flush:
    """What runs between timed steps: a write of a buffer larger than L2, so that no
    line a step reads is left in L2, then a read of another buffer as large, so
    that the write's dirty lines go back to HBM now and not during the next timed
    step (after the write alone, a tiny kernel measured 6.7 us between its events).
    `zero_()` keeps the call sites of a plain flush tensor."""

    def __init__(self, dev):
        self.w = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.zeros((), dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)
        return self


L2_NOTE = "L2 flushed between steps (256 MB write, then a 256 MB read of another buffer)"


def soak(step, dev, seconds=1.0, flush=None):
    """Runs the step, untimed, for about `seconds` right before the timed region, so
    that the clock samples (every 100 ms) see the clocks under this very load and
    the timed steps start from a warm, sustained state."""
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(20):
            if flush is not None:
                flush.zero_()
            step()
        torch.cuda.synchronize(dev)


def capture(fn, dev):
    """fn's launches captured once as a CUDA graph (its host-side argument checks and
    tensor-map encoding done at capture), returned as a replay callable; None where
    capture is refused."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            fn()
        g.replay()
        torch.cuda.synchronize(dev)
    except RuntimeError:
        torch.cuda.synchronize(dev)
        return None
    return g.replay


def roofline_of(w, attn_ms, pk):
    """The attention kernel against the slower of its FLOPs at the bf16 peak and its
    bytes at the HBM copy bandwidth (both measured)."""
    attn_s = attn_ms * 1e-3
    tensor_bound = w["attn_flops"] / (pk["bf16_tflops"] * 1e12) > w["attn_bytes"] / (pk["hbm_gbs"] * 1e9)
    if tensor_bound:
        achieved = w["attn_flops"] / attn_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"]}
    else:
        achieved = w["attn_bytes"] / attn_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"]}
    roof["peak_source"] = pk["source"] + (" burst bf16" if tensor_bound else " HBM copy")
    roof["roofline_time_us"] = max(w["attn_flops"] / (pk["bf16_tflops"] * 1e12),
                                   w["attn_bytes"] / (pk["hbm_gbs"] * 1e9)) * 1e6
    roof["kernel_us"] = attn_ms * 1e3
    return roof


# ------------------------------------------------------------------------- our arm
def plan_is_balanced(prob, cache, splits):
    """Whether mla_decode_attn runs the balanced plan for this split request: asked
    for, or the library's choice when its workspace is the balanced plan's."""
    from mla_decode_attention_absorbed_gb300 import mla
    if splits == mla.SPLITS_BALANCED:
        return True
    if splits != 0:
        return False
    try:
        bal = mla.decode_workspace_size(prob, cache, mla.SPLITS_BALANCED)
    except ValueError:  # not available for these dims
        return False
    return mla.decode_workspace_size(prob, cache, 0) == bal


class DecodeRun:
    """One decode workload on this rank's GPU: inputs, a Decoder, and the decode
    step and the attention alone each captured as a CUDA graph."""

    def __init__(self, cfg, args, rank, dev, kv="bf16"):
        from mla_decode_attention_absorbed_gb300 import mla
        self.c = c = cfg.with_(seed=replica_seed(cfg.seed, rank))
        self.inp = inp = make_inputs(c)
        self.kv_scale = None
        if kv == "fp8":
            inp["kv"] = to_fp8_cache(inp["kv"])
            self.kv_scale = inp["kv_scale"] = KV_FP8_SCALE
        self.w = work(c, inp["seq_lens"].tolist(), 1 if kv == "fp8" else 2)
        self.d = d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        self.prob = prob = mla.Problem.of(c)
        self.dec = mla.Decoder(prob, d["kv"], d["seq_lens"], d["w_uk"], d["w_uv"], d["block_table"], c.page_size,
                               max_seq_len=int(inp["seq_lens"].max()), num_splits=args.splits, kv_scale=self.kv_scale)
        self.splits = mla.decode_num_splits(prob, self.dec.cache) if args.splits == 0 else args.splits
        self.balanced = plan_is_balanced(prob, self.dec.cache, args.splits)
        self.plan = ((f"balanced ({self.splits} tile ranges per 128-row block)" if self.splits > 0
                      else "balanced (asked for)") if self.balanced
                     else f"split plan ({self.splits} pieces a split sequence)" if self.splits > 1 else "unsplit")
        self.dev = dev
        self.eager_step = lambda: self.dec.step(d["q_nope"], d["q_rope"])
        self.eager_attend = lambda: self.dec.attend()
        self.step = self.attend = None

    def warm(self, warmup, flush):
        from mla_decode_attention_absorbed_gb300 import mla
        for _ in range(warmup):
            if flush is not None:
                flush.zero_()
            self.eager_step()
        torch.cuda.synchronize(self.dev)
        st = mla.read_status(self.dec.workspace)
        if st != 0:
            raise RuntimeError(f"{self.c.name}: device status after warm-up: {mla.status_string(st)}")
        self.step = capture(self.eager_step, self.dev)
        self.step_mode = "graph" if self.step is not None else "eager"
        self.step = self.step or self.eager_step
        self.attend = capture(self.eager_attend, self.dev) or self.eager_attend
        if mla.read_status(self.dec.workspace) != 0:
            raise RuntimeError(f"{self.c.name}: device status after the captured calls")

    def release(self):
        for k in ("dec", "d", "inp", "step", "attend", "eager_step", "eager_attend"):
            if hasattr(self, k):
                delattr(self, k)
        torch.cuda.empty_cache()


def config_line(run, steps, stream, dev, flush, pk):
    """Step time, attention time (each from its graph), roofline and rates of one
    secondary workload; short, for the default run's `configs` key."""
    w = run.w
    fl = flush if w["cache_bytes"] < 2 * L2_BYTES else None
    step_ms = statistics.median(_timed_steps(run.step, steps, fl, stream, dev))
    attn_ms = statistics.median(_timed_steps(run.attend, steps, fl, stream, dev))
    roof = roofline_of(w, attn_ms, pk)
    return {"workload": workload_name(run.c), "steps": steps, "ms_per_step": step_ms, "kernel_us": attn_ms * 1e3,
            "num_splits": run.splits, "plan": run.plan,
            "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "roofline_time_us")},
            "tflops_step": w["step_flops"] / (step_ms * 1e-3) / 1e12,
            "attn_tflops": w["attn_flops"] / (attn_ms * 1e-3) / 1e12,
            "attn_tbps": w["attn_bytes"] / (attn_ms * 1e-3) / 1e12,
            "attended_tokens_per_s": w["pairs"] / (step_ms * 1e-3),
            "decode_tokens_per_s": w["tokens"] / (step_ms * 1e-3),
            "l2": "inputs larger than L2" if fl is None else L2_NOTE,
            "launch": f"median of {steps} graph replays each of the step and of the attention alone"}


def naive_line(run, absorbed_ms, dev, stream, reps=3):
    """The decompress-then-attend path on the same inputs (mla_naive_decode), timed
    beside the absorbed step: wall-time ratio next to the algorithmic FLOP ratio."""
    from mla_decode_attention_absorbed_gb300 import mla
    from oracle import counts
    c, d = run.c, run.d
    lens = run.inp["seq_lens"].tolist()
    cache = mla.make_cache(run.prob, d["kv"], d["seq_lens"], d["block_table"], c.page_size, max(lens))
    out, lse, ws = mla.naive_decode(run.prob, d["q_nope"], d["q_rope"], cache, d["w_uk"], d["w_uv"])
    torch.cuda.synchronize(dev)
    if mla.read_status(ws) != 0:
        raise RuntimeError("naive path: device status")
    call = lambda: mla.naive_decode(run.prob, d["q_nope"], d["q_rope"], cache, d["w_uk"], d["w_uv"],  # noqa: E731
                                    out=out, lse=lse, workspace=ws)
    ms = statistics.median(_timed_steps(call, reps, None, stream, dev))
    nf = counts.naive_flops(c.H, c.d_c, c.d_rope, c.d_nope, c.d_v, lens, c.s_q)
    af = run.w["step_flops"]
    res = {"workload": workload_name(c), "ms": ms, "absorbed_ms": absorbed_ms, "ratio_wall": ms / absorbed_ms,
           "flops": nf, "absorbed_flops": af, "ratio_flops": nf / af, "tflops": nf / (ms * 1e-3) / 1e12,
           "workspace_gb": ws.numel() / 1e9, "reps": reps,
           "path": "tcgen05 expansion GEMM (K_h, V_h of every cached token and head) + per-head attention"}
    del out, lse, ws
    torch.cuda.empty_cache()
    return res


def naive_oracle_line(budget_s=12.0):
    """The naive form of the fp64 oracle on the host cores: the whole tiny workload,
    and a seeded subset of the long workload's query rows (each row re-expands its
    head's K and V over the whole history); rates of the sample, no extrapolation."""
    import numpy as np

    import oracle
    from oracle import counts
    res = {"cores": oracle.threads(), "kind": "oracle"}
    tiny = CONFIGS["tiny"]
    inp = make_inputs(tiny)
    t = time.perf_counter()
    oracle.naive(tiny, inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"], inp["w_uv"])
    t = time.perf_counter() - t
    f = counts.naive_flops(tiny.H, tiny.d_c, tiny.d_rope, tiny.d_nope, tiny.d_v, inp["seq_lens"].tolist(), tiny.s_q)
    res["tiny"] = {"seconds": t, "tflops": f / t / 1e12, "sample": "the whole workload"}
    long = CONFIGS["long"].with_(B=1)
    inp = make_inputs(long)
    rows_total = long.s_q * long.H
    n = max(1, min(rows_total, oracle.threads()))
    rows = sorted(np.random.default_rng(3).choice(rows_total, size=n, replace=False).tolist())
    t = time.perf_counter()
    oracle.naive(long, inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"], inp["w_uv"], rows=rows)
    t = time.perf_counter() - t
    L = int(inp["seq_lens"][0])
    per_row = counts.naive_flops(1, long.d_c, long.d_rope, long.d_nope, long.d_v, [L], long.s_q)
    res["long"] = {"seconds": t, "tflops": per_row * n / t / 1e12,
                   "sample": f"{n} seeded query rows of the first sequence (L={L}), each re-expanding its head"}
    return res


def run_ours(cfg, args, rank, world, local, active):
    from mla_decode_attention_absorbed_gb300 import mla

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mla.load()
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)
    run = DecodeRun(cfg, args, rank, dev, args.kv)
    w = run.w
    fl = flush if w["cache_bytes"] < 2 * L2_BYTES else None
    run.warm(args.warmup, fl)
    step = run.step

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(nvsmi_gpu_id(local)).start()
    soak(step, dev, 1.0, fl)
    barrier(active)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    for k in range(K):
        if fl is not None:
            fl.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(active)
    t_wall = time.perf_counter() - t_wall
    # the attention kernel alone (its own launch from a graph, same inputs), for its roofline
    attn_ms_list = _timed_steps(run.attend, K, fl, stream, dev)
    clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(step_ms) / K
    ms = reduce_max(ms_local, active, "cuda" if active and args.backend == "nccl" else "cpu")
    attn_avg = sum(attn_ms_list) / K

    # end to end through the public API: every step copies its inputs from pinned host
    # memory (queries, lengths, block table) and reads its result back
    c, d, inp, prob = run.c, run.d, run.inp, run.prob
    q_nope, q_rope = d["q_nope"], d["q_rope"]
    h_qn = inp["q_nope"].pin_memory()
    h_qr = inp["q_rope"].pin_memory()
    h_lens = inp["seq_lens"].pin_memory()
    h_bt = inp["block_table"].pin_memory() if inp["block_table"] is not None else None
    host_in = [h_qn, h_qr, h_lens] + ([h_bt] if h_bt is not None else [])
    sets = []
    for j in range(2):
        lens_j = d["seq_lens"].clone()
        bt_j = d["block_table"].clone() if d["block_table"] is not None else None
        dec_j = mla.Decoder(prob, d["kv"], lens_j, d["w_uk"], d["w_uv"], bt_j, c.page_size,
                            max_seq_len=int(inp["seq_lens"].max()), num_splits=args.splits, kv_scale=run.kv_scale)
        qn_j, qr_j = torch.empty_like(q_nope), torch.empty_like(q_rope)
        sets.append(dict(dec=dec_j, ins=[qn_j, qr_j, lens_j] + ([bt_j] if bt_j is not None else []),
                         out=dec_j.out, h_out=torch.empty(dec_j.out.shape, dtype=dec_j.out.dtype).pin_memory(),
                         step=lambda dec_j=dec_j, qn_j=qn_j, qr_j=qr_j: dec_j.step(qn_j, qr_j)))
    e2e_steps = max(3, min(K, 50))
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sets[0]["h_out"].numel() * 2
    torch.cuda.synchronize(dev)
    barrier(active)
    e2e_local, e2e_mode = pipelined_e2e(dev, host_in, sets, e2e_steps)
    e2e_ms = reduce_max(e2e_local, active, "cuda" if active and args.backend == "nccl" else "cpu")
    if any(mla.read_status(sj["dec"].workspace) != 0 for sj in sets):
        raise RuntimeError("device status after the end-to-end loop")
    del sets
    res = dict(w=w, ms=ms, attn_ms=attn_avg, e2e_ms=e2e_ms, e2e_mode=e2e_mode + " (%d steps)" % e2e_steps,
               step_mode=run.step_mode, h2d=h2d, d2h=d2h, splits=run.splits, clocks=clocks,
               step_ms=step_ms, attn_ms_list=attn_ms_list, wall_s=t_wall, inp=inp, c=c,
               plan=run.plan, launches_per_step=3 + (1 if run.splits > 1 and not run.balanced else 0))
    run.release()
    # the other workloads of the method, each on its own (this rank's replica)
    configs, naive = {}, None
    if not args.headline_only and args.kv == "bf16" and cfg.name == DEFAULT_CONFIG:
        pk = peaks()
        steps = max(3, min(K, 20))
        for name in SECONDARY:
            r2 = DecodeRun(CONFIGS[name], args, rank, dev, "bf16")
            fl2 = flush if r2.w["cache_bytes"] < 2 * L2_BYTES else None
            r2.warm(3, fl2)
            configs[name] = config_line(r2, steps, stream, dev, flush, pk)
            if name == "long" and not args.no_naive:
                naive = naive_line(r2, configs[name]["ms_per_step"], dev, stream)
            r2.release()
    res["configs"], res["naive"] = configs, naive
    return res
def cpu_baseline(cfg, inp, budget_s: float = 12.0):
    """The oracle as it stands, absorbed form, on whole sequences of the same
    workload until about ``budget_s`` of host time is spent."""
    import oracle
    from oracle import counts
    threads = oracle.threads()
    B = cfg.B
    done_flops, t_used, n = 0, 0.0, 0
    for b in range(B):
        sub = cfg.with_(B=1)
        one = {k: inp[k][b:b + 1] for k in ("q_nope", "q_rope", "seq_lens")}
        if inp["block_table"] is None:
            kv = inp["kv"][b:b + 1]
            bt = None
        else:
            kv, bt = inp["kv"], inp["block_table"][b:b + 1]
        t0 = time.perf_counter()
        oracle.decode(sub, one["q_nope"], one["q_rope"], kv, one["seq_lens"], inp["w_uk"], inp["w_uv"],
                      block_table=bt, page_size=cfg.page_size, kv_scale=inp.get("kv_scale"))
        t_used += time.perf_counter() - t0
        L = int(one["seq_lens"][0])
        done_flops += (counts.attention_flops(cfg.H, cfg.d_c, cfg.d_rope, [L], cfg.s_q)
                       + counts.absorb_flops(1, cfg.s_q, cfg.H, cfg.d_nope, cfg.d_c)
                       + counts.out_proj_flops(1, cfg.s_q, cfg.H, cfg.d_c, cfg.d_v))
        n += 1
        if t_used >= budget_s:
            break
    return {"value": done_flops / t_used / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {B} sequences of the {cfg.name} workload, whole absorbed step (fp64), "
                      f"{t_used:.1f} s"}


def workload_name(cfg, kv: str = "bf16"):
    lens = f"T={cfg.T}" if not cfg.len_lo else f"L~U[{cfg.len_lo},{cfg.len_hi}]"
    lay = f"paged{cfg.page_size}" if cfg.paged else "contiguous"
    cache = "bf16 cache" if kv == "bf16" else "FP8 E4M3 cache (scale 1/16)"
    return (f"{cfg.name}: B={cfg.B} H={cfg.H} d_c={cfg.d_c} d_rope={cfg.d_rope} d_nope={cfg.d_nope} "
            f"d_v={cfg.d_v} {lens} s_q={cfg.s_q} {lay} {cache}")


# the other workloads of the method, each measured in the default run beside the headline
SECONDARY = ("tiny", "long", "spec", "ragged_paged")


def main_ours(args):
    rank, world, local = dist_env()
    active = init_dist(world, args.backend)
    cfg = CONFIGS[args.config]
    r = run_ours(cfg, args, rank, world, local, active)
    if rank != 0:
        return
    w, ms = r["w"], r["ms"]
    pk = peaks()
    total_flops = w["step_flops"] * world
    value = total_flops / (ms * 1e-3) / 1e12
    roof = roofline_of(w, r["attn_ms"], pk)
    roof["traffic"] = traffic_for(f"attn{'_fp8' if args.kv == 'fp8' else ''}:{cfg.name}")
    roof["kernel"] = ("mla_decode_attn, balanced plan (persistent pair kernel, in-launch merge)" if "balanced" in r["plan"]
                      else "mla_decode_attn (split-T attention + LSE combine)") + (
        ", FP8 E4M3 cache dequantised on chip, fp16 MMAs" if args.kv == "fp8" else "")
    roof["kernel_timing"] = (f"CUDA events around each of {args.steps} replays of the attention call captured "
                             "as a CUDA graph (no host launch work inside)")
    cpu = cpu_baseline(r["c"], r["inp"], args.cpu_budget) if not args.no_cpu_baseline else None
    naive = r["naive"]
    if naive is not None and not args.no_cpu_baseline:
        naive["oracle"] = naive_oracle_line()
    clk = r["clocks"].summary()
    attn_s = r["attn_ms"] * 1e-3
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if args.kv == "bf16" else "e4m3 cache, f16 MMAs, bf16 projections",
        "data": "synthetic (seeded N(0,1) queries and latent cache, N(0,1/d_c) weights)",
        "config": {"workload": workload_name(cfg, args.kv),
                   "num_splits": r["splits"], "plan": r["plan"],
                   "l2": ("inputs larger than L2: the cache alone is "
                          f"{w['cache_bytes'] / 1e6:.0f} MB per replica") if w["cache_bytes"] >= 2 * L2_BYTES
                   else L2_NOTE,
                   "parallelism": f"{world} independent replica(s), sequences sharded by rank",
                   "launch": f"one mla_decode_step per step ({r['step_mode']}: the call's three launches "
                             "captured once and replayed)" if r["step_mode"] == "graph" else
                             "one mla_decode_step per step (eager launches)"},
        "hbm_tbps": (w["step_bytes"] * world) / (ms * 1e-3) / 1e12,
        "attn_tflops": w["attn_flops"] / attn_s / 1e12,
        "attn_tbps": w["attn_bytes"] / attn_s / 1e12,
        "attended_tokens_per_s": w["pairs"] * world / (ms * 1e-3),
        "decode_tokens_per_s": w["tokens"] * world / (ms * 1e-3),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": total_flops / (r["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": r["e2e_ms"], "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "note": "pinned host q_nope/q_rope/seq_lens(/block_table) in, out back, every step, on a copy "
                        "stream overlapping the neighbouring steps' compute (two alternating buffer sets); "
                        "latent cache and weights stay resident in HBM",
                "launch": r["e2e_mode"]},
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": clk,
        "step_ms_min": min(r["step_ms"]),
        "step_ms_median": statistics.median(r["step_ms"]),
        "configs": r["configs"],
        "naive": naive,
    }
    print(json.dumps(line))


# ------------------------------------------------------------------------- other rows of the path
D_MODEL = 7168  # DeepSeek-V3 hidden width (the down-projection's contraction)


def _timed_steps(step, K, flush, stream, dev):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize(dev)
    for k in range(K):
        if flush is not None:
            flush.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) for a, b in ev]


def pipelined_e2e(dev, host_in, sets, n_steps):
    """End-to-end time per step through the public API: step i copies host_in (pinned)
    into its set's device inputs and reads its set's output back to pinned memory, on a
    copy stream that overlaps the neighbouring steps' compute (two alternating sets, so
    that a set is refilled only after its step ran and its result was read).  The loop
    is captured once as a CUDA graph, so that the host's launch work does not pace the
    GPU; where capture is refused the same loop runs eagerly.
    sets: two dicts with "ins" (device tensors in host_in's order), "out" (device),
    "h_out" (pinned host) and "step" (issues the step on the current stream).
    Returns (ms per step, "graph" | "eager")."""
    copy = torch.cuda.Stream(dev)

    def copy_in(j):
        with torch.cuda.stream(copy):
            for dst, src in zip(sets[j]["ins"], host_in):
                dst.copy_(src, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(copy)
        return ev

    def loop(n):
        cur = torch.cuda.current_stream(dev)
        fork = torch.cuda.Event()
        fork.record(cur)
        copy.wait_event(fork)
        ev_in = copy_in(0)
        for i in range(n):
            j = i % 2
            cur.wait_event(ev_in)
            sets[j]["step"]()
            done = torch.cuda.Event()
            done.record(cur)
            if i + 1 < n:
                ev_in = copy_in(1 - j)  # queued behind the read-back of step i-1, which used that set
            with torch.cuda.stream(copy):
                copy.wait_event(done)
                sets[j]["h_out"].copy_(sets[j]["out"], non_blocking=True)
        join = torch.cuda.Event()
        join.record(copy)
        cur.wait_event(join)

    stream = torch.cuda.current_stream(dev)
    mode = "graph"
    graph = torch.cuda.CUDAGraph()
    try:
        loop(2)  # the copy paths, eagerly, before the capture
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph, capture_error_mode="relaxed"):
            loop(n_steps)
        graph.replay()
        torch.cuda.synchronize(dev)
    except RuntimeError:
        torch.cuda.synchronize(dev)
        mode = "eager"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if mode == "graph":
        graph.replay()
    else:
        loop(n_steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / n_steps, mode


TOPK = 2048  # DeepSeek-V3.2's index_topk


def main_op(args):
    """One JSON line for a non-headline row of the path, same contract as the decode line."""
    rank, world, local = dist_env()
    active = init_dist(world, args.backend)
    default = {"sparse": "sparse", "prefill": "prefill"}.get(args.op, DEFAULT_CONFIG)
    cfg = CONFIGS[default if args.config == DEFAULT_CONFIG else args.config]
    if args.op == "sparse":
        return main_sparse(args, cfg, rank, world, local, active)
    if args.op == "prefill":
        return main_prefill(args, cfg, rank, world, local, active)
    from mla_decode_attention_absorbed_gb300 import mla
    from mla_decode_attention_absorbed_gb300.workloads import make_append_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    mla.load()
    c = cfg.with_(seed=replica_seed(cfg.seed, rank))
    inp = make_inputs(c)
    kv_scale, eb = None, 2
    if args.kv == "fp8":
        inp["kv"] = to_fp8_cache(inp["kv"])
        kv_scale, eb = KV_FP8_SCALE, 1
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    prob = mla.Problem.of(c)
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], d["block_table"], c.page_size, kv_scale=kv_scale)
    flush = L2Flush(dev)
    pk = peaks()
    assert args.op == "append"
    app = make_append_inputs(c, D_MODEL)
    a = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in app.items()}
    ws = mla.alloc_workspace(mla.cache_append_workspace_size(prob, D_MODEL), dev)
    M = c.B * c.s_q
    # algorithmic work: every W_DKV, x and k_rope byte read once, the new cache rows written once
    bytes_ = (D_MODEL * c.d_c + M * D_MODEL + M * c.d_rope) * 2 + M * c.W * eb + c.B * 4
    flops = 2 * M * D_MODEL * c.d_c

    def step():
        mla.cache_append(prob, a["x"], a["w_dkv"], a["k_rope"], cache, workspace=ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    st = mla.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {mla.status_string(st)}")
    # the step's launches (host-side argument checks and tensor-map encoding done
    # once at capture) replayed as one CUDA graph: the device time of the op, not
    # the Python call around it
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(nvsmi_gpu_id(local)).start()
    soak(graph.replay, dev, 1.0, flush)
    barrier(active)
    step_ms = _timed_steps(graph.replay, args.steps, flush, stream, dev)
    barrier(active)
    clocks.stop()
    ms = reduce_max(sum(step_ms) / len(step_ms), active, "cuda" if active and args.backend == "nccl" else "cpu")
    achieved = bytes_ / (ms * 1e-3) / 1e9

    # end to end: pinned x / k_rope in, the appended rows out, every step
    h_x, h_kr = app["x"].pin_memory(), app["k_rope"].pin_memory()
    lens = inp["seq_lens"].to(torch.long)
    pos = lens.repeat_interleave(c.s_q) - c.s_q + torch.arange(c.s_q).repeat(c.B)
    if inp["block_table"] is None:
        flat = torch.arange(c.B).repeat_interleave(c.s_q) * inp["kv"].shape[1] + pos
    else:
        page = inp["block_table"].to(torch.long)[torch.arange(c.B).repeat_interleave(c.s_q), pos // c.page_size]
        flat = page * c.page_size + pos % c.page_size
    flat = flat.to(dev)
    kv_rows = d["kv"].view(-1, c.W)
    gather = lambda: kv_rows.index_select(0, flat)  # noqa: E731
    h_rows = torch.empty(M, c.W, dtype=d["kv"].dtype).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))
    sets = []
    for _ in range(2):
        bufs = dict(x=torch.empty_like(a["x"]), kr=torch.empty_like(a["k_rope"]), ws=torch.empty_like(ws),
                    rows=torch.empty(M, c.W, dtype=d["kv"].dtype, device=dev))

        def append_step(b=bufs):
            mla.cache_append(prob, b["x"], a["w_dkv"], b["kr"], cache, workspace=b["ws"])
            b["rows"].copy_(gather())
        sets.append(dict(ins=[bufs["x"], bufs["kr"]], out=bufs["rows"], h_out=torch.empty_like(h_rows).pin_memory(),
                         step=append_step))
    del bufs
    torch.cuda.synchronize(dev)
    e2e_local, e2e_mode = pipelined_e2e(dev, [h_x, h_kr], sets, e2e_steps)
    e2e_ms = reduce_max(e2e_local, active, "cuda" if active and args.backend == "nccl" else "cpu")
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        t = time.perf_counter()
        oracle.down_proj(app["x"], app["w_dkv"])
        t = time.perf_counter() - t
        cpu = {"value": bytes_ / t / 1e9, "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
               "sample": f"the whole step: {M} tokens x d_model {D_MODEL} x d_c {c.d_c} in fp64, {t:.2f} s"}
    line = {
        "metric": "MLA cache append (latent down-projection of the new tokens) GB/s",
        "value": bytes_ * world / (ms * 1e-3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if args.kv == "bf16" else "bf16 GEMM, e4m3 cache rows",
        "data": "synthetic (seeded N(0,1) hidden states, N(0,1/d_model) W_DKV)",
        "config": {"workload": f"append to {workload_name(c, args.kv)}, d_model={D_MODEL}",
                   "l2": L2_NOTE,
                   "launch": "the step's kernels replayed as a CUDA graph",
                   "parallelism": f"{world} independent replica(s)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": None,
                     "kernel": "mla_cache_append (split-K tcgen05 GEMM + scatter)",
                     "peak_source": pk["source"] + " HBM copy",
                     "roofline_time_us": bytes_ / (pk["hbm_gbs"] * 1e9) * 1e6, "kernel_us": ms * 1e3,
                     "tflops": flops / (ms * 1e-3) / 1e12},
        "cpu_baseline": cpu,
        "e2e": {"value": bytes_ * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": (h_x.numel() + h_kr.numel()) * 2, "d2h_bytes_per_step": h_rows.numel() * h_rows.element_size(),
                "note": "pinned host x / k_rope in, the appended cache rows back, every step, on a copy stream "
                        "overlapping the neighbouring steps' compute (two alternating buffer sets)",
                "launch": e2e_mode},
        "gpu_launches": 2 * args.steps,  # split-K GEMM + scatter (the accumulator memset is a driver op)
        "clocks": clocks.summary(),
        "step_ms_min": min(step_ms),
        "step_ms_median": statistics.median(step_ms),
    }
    print(json.dumps(line))


def prefill_flops(cfg, lens):
    """Algorithmic FLOPs of one prefill step in the expand form ("Why MLA and MTP
    Fight Each Other", 5.3/5.5): K_h, V_h for every cached token of every head,
    then causal attention over the visible pairs with a (d_nope + d_rope)-wide
    score and a d_v-wide sum; and in the absorbed form (5.3 / the decode counters)."""
    from oracle import counts
    toks = sum(int(L) for L in lens)
    pairs = sum(counts.visible_pairs(int(L), cfg.s_q) for L in lens)
    expand = (2 * toks * cfg.H * cfg.d_c * (cfg.d_nope + cfg.d_v)
              + 2 * pairs * cfg.H * (cfg.d_nope + cfg.d_rope + cfg.d_v))
    absorbed = (counts.attention_flops(cfg.H, cfg.d_c, cfg.d_rope, lens, cfg.s_q)
                + counts.absorb_flops(cfg.B, cfg.s_q, cfg.H, cfg.d_nope, cfg.d_c)
                + counts.out_proj_flops(cfg.B, cfg.s_q, cfg.H, cfg.d_c, cfg.d_v))
    return expand, absorbed


def main_prefill(args, cfg, rank, world, local, active):
    """Prefill through mla_prefill (expand form above the crossover); the
    absorbed form is timed beside it where its row limit allows."""
    from mla_decode_attention_absorbed_gb300 import mla

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    mla.load()
    c = cfg.with_(seed=replica_seed(cfg.seed, rank))
    inp = make_inputs(c)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    prob = mla.Problem.of(c)
    lens = inp["seq_lens"].tolist()
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], d["block_table"], c.page_size, max_seq_len=max(lens))
    f_exp, f_abs = prefill_flops(c, lens)
    out = torch.empty(c.B, c.s_q, c.H, c.d_v, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(c.B, c.s_q, c.H, dtype=torch.float32, device=dev)
    ws = mla.alloc_workspace(mla.load().mla_prefill_workspace_size(ctypes.byref(prob.dims()), ctypes.byref(cache)), dev)
    path = [None]

    def step():
        path[0] = mla.prefill(prob, d["q_nope"], d["q_rope"], cache, d["w_uk"], d["w_uv"], out=out, lse=lse,
                              workspace=ws)[3]

    flush = L2Flush(dev)
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    st = mla.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {mla.status_string(st)}")
    clocks = ClockSampler(nvsmi_gpu_id(local)).start()
    soak(step, dev, 1.0, flush)
    barrier(active)
    step_ms = _timed_steps(step, args.steps, flush, stream, dev)
    barrier(active)
    clocks.stop()
    ms = reduce_max(sum(step_ms) / len(step_ms), active, "cuda" if active and args.backend == "nccl" else "cpu")
    flops = f_exp if path[0] == mla.PATH_EXPAND else f_abs
    # the absorbed form on the same step, where the absorbed kernels' row limit allows
    absorbed_ms = None
    if c.s_q * c.H <= 65536:
        dec = mla.Decoder(prob, d["kv"], d["seq_lens"], d["w_uk"], d["w_uv"], d["block_table"], c.page_size,
                          max_seq_len=max(lens))
        for _ in range(args.warmup):
            flush.zero_()
            dec(d["q_nope"], d["q_rope"])
        absorbed_ms = sum(_timed_steps(lambda: dec(d["q_nope"], d["q_rope"]), args.steps, flush, stream, dev)) / args.steps
    # end to end: pinned q_nope / q_rope in, out back, every step
    h_qn, h_qr = inp["q_nope"].pin_memory(), inp["q_rope"].pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    sets = []
    for _ in range(2):
        bufs = dict(qn=torch.empty_like(d["q_nope"]), qr=torch.empty_like(d["q_rope"]), out=torch.empty_like(out),
                    lse=torch.empty_like(lse), ws=torch.empty_like(ws))

        def prefill_step(b=bufs):
            mla.prefill(prob, b["qn"], b["qr"], cache, d["w_uk"], d["w_uv"], out=b["out"], lse=b["lse"],
                        workspace=b["ws"])
        sets.append(dict(ins=[bufs["qn"], bufs["qr"]], out=bufs["out"],
                         h_out=torch.empty(out.shape, dtype=out.dtype).pin_memory(), step=prefill_step))
    del bufs
    torch.cuda.synchronize(dev)
    e2e_local, e2e_mode = pipelined_e2e(dev, [h_qn, h_qr], sets, e2e_steps)
    e2e_ms = reduce_max(e2e_local, active, "cuda" if active and args.backend == "nccl" else "cpu")
    if rank != 0:
        return
    pk = peaks()
    ach = flops / (ms * 1e-3) / 1e12
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        rows = list(range(0, c.B * c.s_q * c.H, max(1, c.B * c.s_q * c.H // 32)))[:32]
        t = time.perf_counter()
        oracle.naive(c, inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"], inp["w_uv"],
                     inp["block_table"], c.page_size, rows=rows)
        t = time.perf_counter() - t
        rows_total = c.B * c.s_q * c.H
        cpu = {"value": flops * len(rows) / rows_total / t / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
               "kind": "oracle",
               "sample": f"{len(rows)} of {rows_total} query rows, decompress-then-attend in fp64, {t:.1f} s "
                         "(the oracle re-expands each row's history: far more work than the sampled share)"}
    line = {
        "metric": "MLA prefill TFLOP/s (expand form above the crossover S*, H=128, d_c=512+64, 1xGB300)",
        "value": flops * world / (ms * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) queries and latent cache, N(0,1/d_c) weights)",
        "config": {"workload": workload_name(c), "path": "expand" if path[0] == mla.PATH_EXPAND else "absorbed",
                   "crossover_S": mla.prefill_crossover(prob, max(lens)),
                   "l2": L2_NOTE,
                   "parallelism": f"{world} independent replica(s)"},
        "flops_expand_form": f_exp,
        "flops_absorbed_form": f_abs,
        "absorbed_form_ms": absorbed_ms,
        "roofline": {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": ach / pk["bf16_tflops"], "traffic": None,
                     "kernel": "mla_prefill (expand GEMM + per-head attention) as one step",
                     "peak_source": pk["source"] + " burst bf16",
                     "roofline_time_us": flops / (pk["bf16_tflops"] * 1e12) * 1e6, "kernel_us": ms * 1e3},
        "cpu_baseline": cpu,
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": (h_qn.numel() + h_qr.numel()) * 2, "d2h_bytes_per_step": h_out.numel() * 2,
                "note": "pinned host q_nope/q_rope in, out back, every step, on a copy stream overlapping the "
                        "neighbouring steps' compute (two alternating buffer sets); cache and weights resident",
                "launch": e2e_mode},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
        "step_ms_min": min(step_ms),
        "step_ms_median": statistics.median(step_ms),
    }
    print(json.dumps(line))


def cpu_baseline_sparse(cfg, inp, idx, per_pair_flops, budget_s: float = 12.0):
    """The oracle as it stands: absorb, sparse attention and out_proj in fp64 on
    whole sequences of the same workload until about ``budget_s`` of host time."""
    import oracle
    from oracle import counts
    done, t_used, n = 0, 0.0, 0
    sub = cfg.with_(B=1)
    for b in range(cfg.B):
        bt = None if inp["block_table"] is None else inp["block_table"][b:b + 1]
        kv = inp["kv"][b:b + 1] if bt is None else inp["kv"]
        L = inp["seq_lens"][b:b + 1]
        t0 = time.perf_counter()
        q_cat = oracle.absorb_q(sub, inp["q_nope"][b:b + 1], inp["q_rope"][b:b + 1], inp["w_uk"])
        o_lat, _ = oracle.attend_sparse(sub, q_cat, kv, L, idx[b:b + 1], bt, cfg.page_size,
                                        kv_scale=inp.get("kv_scale"))
        oracle.out_proj(sub, o_lat, inp["w_uv"])
        t_used += time.perf_counter() - t0
        lim = int(L[0]) - cfg.s_q + torch.arange(cfg.s_q).view(-1, 1)
        pairs = int(((idx[b] >= 0) & (idx[b] <= lim)).sum())
        done += (pairs * per_pair_flops + counts.absorb_flops(1, cfg.s_q, cfg.H, cfg.d_nope, cfg.d_c)
                 + counts.out_proj_flops(1, cfg.s_q, cfg.H, cfg.d_c, cfg.d_v))
        n += 1
        if t_used >= budget_s:
            break
    return {"value": done / t_used / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{n} of {cfg.B} sequences of the sparse top-{TOPK} step (fp64), {t_used:.1f} s"}


def main_sparse(args, cfg, rank, world, local, active):
    """The decode step with the attention over k = TOPK listed tokens per query token."""
    from mla_decode_attention_absorbed_gb300 import mla
    from mla_decode_attention_absorbed_gb300.workloads import make_sparse_indices

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    mla.load()
    c = cfg.with_(seed=replica_seed(cfg.seed, rank))
    inp = make_inputs(c)
    kv_scale, eb = None, 2
    if args.kv == "fp8":
        inp["kv"] = to_fp8_cache(inp["kv"])
        kv_scale, eb = KV_FP8_SCALE, 1
        inp["kv_scale"] = kv_scale
    idx = make_sparse_indices(c, inp["seq_lens"], TOPK)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    d_idx = idx.to(dev)
    prob = mla.Problem.of(c)
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], d["block_table"], c.page_size, kv_scale=kv_scale)
    q_cat = torch.empty(c.B, c.s_q, c.H, c.W, dtype=torch.bfloat16, device=dev)
    o_lat = torch.empty(c.B, c.s_q, c.H, c.d_c, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(c.B, c.s_q, c.H, dtype=torch.float32, device=dev)
    out = torch.empty(c.B, c.s_q, c.H, c.d_v, dtype=torch.bfloat16, device=dev)
    ws = mla.alloc_workspace(mla.decode_sparse_workspace_size(prob, cache, TOPK, args.splits), dev)
    # algorithmic work: the visible listed pairs, each listed cache row read once per query token
    n_pairs = int(((idx >= 0) & (idx <= (inp["seq_lens"].view(-1, 1, 1) - c.s_q
                                        + torch.arange(c.s_q).view(1, -1, 1)))).sum())
    per_pair_flops = 2 * c.H * (c.W + c.d_c)
    attn_flops = n_pairs * per_pair_flops
    attn_bytes = n_pairs * c.W * eb + q_cat.numel() * 2 + o_lat.numel() * 2 + lse.numel() * 4 + idx.numel() * 4
    proj_flops = 2 * c.B * c.s_q * c.H * c.d_nope * c.d_c + 2 * c.B * c.s_q * c.H * c.d_c * c.d_v
    step_flops = attn_flops + proj_flops

    def absorb():
        mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"], q_cat=q_cat)

    def attend():
        mla.decode_attn_sparse(prob, q_cat, cache, d_idx, num_splits=args.splits, o_lat=o_lat, lse=lse,
                               workspace=ws)

    def project():
        mla.out_proj(prob, o_lat, d["w_uv"], out=out)

    flush = L2Flush(dev)
    for _ in range(args.warmup):
        flush.zero_()
        absorb(); attend(); project()
    torch.cuda.synchronize(dev)
    st = mla.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {mla.status_string(st)}")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    ev_a = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(nvsmi_gpu_id(local)).start()
    soak(lambda: (absorb(), attend(), project()), dev, 1.0, flush)
    barrier(active)
    torch.cuda.synchronize(dev)
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        absorb()
        ev_a[k][0].record(stream)
        attend()
        ev_a[k][1].record(stream)
        project()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(active)
    clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    attn_ms = sum(a.elapsed_time(b) for a, b in ev_a) / K
    ms = reduce_max(sum(step_ms) / K, active, "cuda" if active and args.backend == "nccl" else "cpu")
    # end to end: pinned q_nope / q_rope / index lists in, out back, every step
    h_qn, h_qr, h_idx = inp["q_nope"].pin_memory(), inp["q_rope"].pin_memory(), idx.pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e_steps = max(3, min(K, 50))
    sets = []
    for _ in range(2):
        bufs = dict(qn=torch.empty_like(d["q_nope"]), qr=torch.empty_like(d["q_rope"]), idx=torch.empty_like(d_idx),
                    q_cat=torch.empty_like(q_cat), o_lat=torch.empty_like(o_lat), lse=torch.empty_like(lse),
                    out=torch.empty_like(out), ws=torch.empty_like(ws))

        def sparse_step(b=bufs):
            mla.absorb_q(prob, b["qn"], b["qr"], d["w_uk"], q_cat=b["q_cat"])
            mla.decode_attn_sparse(prob, b["q_cat"], cache, b["idx"], num_splits=args.splits, o_lat=b["o_lat"],
                                   lse=b["lse"], workspace=b["ws"])
            mla.out_proj(prob, b["o_lat"], d["w_uv"], out=b["out"])
        sets.append(dict(ins=[bufs["qn"], bufs["qr"], bufs["idx"]], out=bufs["out"],
                         h_out=torch.empty(out.shape, dtype=out.dtype).pin_memory(), step=sparse_step))
    torch.cuda.synchronize(dev)
    e2e_local, e2e_mode = pipelined_e2e(dev, [h_qn, h_qr, h_idx], sets, e2e_steps)
    e2e_ms = reduce_max(e2e_local, active, "cuda" if active and args.backend == "nccl" else "cpu")
    if rank != 0:
        return
    pk = peaks()
    attn_s = attn_ms * 1e-3
    tensor_bound = attn_flops / (pk["bf16_tflops"] * 1e12) > attn_bytes / (pk["hbm_gbs"] * 1e9)
    if tensor_bound:
        ach = attn_flops / attn_s / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"]}
    else:
        ach = attn_bytes / attn_s / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"]}
    roof.update({"traffic": traffic_for(f"attn_sparse{'_fp8' if args.kv == 'fp8' else ''}:{cfg.name}"),
                 "kernel": "mla_decode_attn_sparse (gathered top-k attention)",
                 "peak_source": pk["source"] + (" burst bf16" if tensor_bound else " HBM copy"),
                 "roofline_time_us": max(attn_flops / (pk["bf16_tflops"] * 1e12),
                                         attn_bytes / (pk["hbm_gbs"] * 1e9)) * 1e6,
                 "kernel_us": attn_ms * 1e3})
    cpu = None if args.no_cpu_baseline else cpu_baseline_sparse(c, inp, idx, per_pair_flops)
    line = {
        "metric": f"MLA sparse top-{TOPK} decode TFLOP/s (H=128, d_c=512+64, 1xGB300)",
        "value": step_flops * world / (ms * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if args.kv == "bf16" else "e4m3 cache, f16 MMAs, bf16 projections",
        "data": "synthetic (seeded N(0,1) queries and latent cache, N(0,1/d_c) weights, uniform random top-k lists)",
        "config": {"workload": f"{workload_name(c, args.kv)}, top-{TOPK} lists",
                   "num_splits": args.splits,
                   "l2": L2_NOTE,
                   "parallelism": f"{world} independent replica(s), sequences sharded by rank"},
        "attn_tflops": attn_flops / attn_s / 1e12,
        "attn_tbps": attn_bytes / attn_s / 1e12,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": step_flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": (h_qn.numel() + h_qr.numel()) * 2 + h_idx.numel() * 4,
                "d2h_bytes_per_step": h_out.numel() * 2,
                "note": "pinned host q_nope/q_rope/index lists in, out back, every step, on a copy stream "
                        "overlapping the neighbouring steps' compute (two alternating buffer sets); cache and "
                        "weights resident", "launch": e2e_mode},
        "gpu_launches": 3 * K,
        "clocks": clocks.summary(),
        "step_ms_min": min(step_ms),
        "step_ms_median": statistics.median(step_ms),
    }
    print(json.dumps(line))


# ------------------------------------------------------------------------- reference arm
def main_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    from oracle import counts
    cfg = CONFIGS[args.config]
    inp = make_inputs(cfg)
    threads = oracle.threads()
    # each step: the whole absorbed step for one sequence of the workload (bounded sample)
    def one(b):
        sub = cfg.with_(B=1)
        kv = inp["kv"][b:b + 1] if inp["block_table"] is None else inp["kv"]
        bt = None if inp["block_table"] is None else inp["block_table"][b:b + 1]
        oracle.decode(sub, inp["q_nope"][b:b + 1], inp["q_rope"][b:b + 1], kv, inp["seq_lens"][b:b + 1],
                      inp["w_uk"], inp["w_uv"], block_table=bt, page_size=cfg.page_size)
        L = int(inp["seq_lens"][b])
        return (counts.attention_flops(cfg.H, cfg.d_c, cfg.d_rope, [L], cfg.s_q)
                + counts.absorb_flops(1, cfg.s_q, cfg.H, cfg.d_nope, cfg.d_c)
                + counts.out_proj_flops(1, cfg.s_q, cfg.H, cfg.d_c, cfg.d_v))

    for k in range(args.warmup):
        one(k % cfg.B)
    flops, t = 0, 0.0
    times = []
    for k in range(args.steps):
        t0 = time.perf_counter()
        flops += one(k % cfg.B)
        dt = time.perf_counter() - t0
        times.append(dt)
        t += dt
    value = flops / t / 1e12
    ms = t / args.steps * 1e3
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": workload_name(cfg),
                   "sample": "each step = the whole absorbed decode of one sequence (all heads) of this workload"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} sequence(s) of {cfg.B}, one per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--splits", type=int, default=0, help="split count (0 = the library's choice)")
    ap.add_argument("--backend", default="nccl", choices=["nccl", "gloo"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="decode: time the headline workload only (no `configs`, no naive leg)")
    ap.add_argument("--no-naive", action="store_true", help="decode: skip the naive comparison leg")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="latent cache format of the decode and sparse ops (fp8: E4M3 codes, scale 1/16)")
    ap.add_argument("--op", default="decode", choices=["decode", "append", "sparse", "prefill"],
                    help="decode: the absorbed decode step (headline); append: the cache append "
                         "(latent down-projection of the new tokens, d_model = 7168); sparse: the decode "
                         "step with sparse top-k attention (k = 2048, workload 'sparse' by default)")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        a.warmup = 3
    if a.steps is None:
        a.steps = 2 if a.impl == "reference" else 200
    return a


if __name__ == "__main__":
    args = parse()
    if args.op != "decode":
        main_op(args)
    elif args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)
