"""Benchmark of the NSA forward hot path on B300 (libnsa.so, sm_103a).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one NSA prefill forward over a 65,536-token sequence (64 query heads
in 4 GQA groups, dk=192, dv=128, bf16, seed 2): compression, compressed
attention with block scores and top-16 selection, selected-block attention,
sliding-window attention and the gated combine.  ``value`` is whole-job
prefill tokens/s (all ranks) with inputs resident in HBM; ``e2e`` repeats the
measurement through the same C-ABI call with inputs copied from pinned host
memory and the output copied back inside the timed region.  The decode step
(16 x 64k caches) and the DSA decode step (8 x 128k) are timed in the same run
and reported under ``decode`` / ``dsa`` when the library provides them.

Inputs (q: 1.6 GB) are larger than the 126 MB L2, so no flush is needed
between steps.  Under torchrun every rank runs its own sequence (independent
problems: weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import NSAParams, PREFILL_CONFIGS, decode_config, dsa_config, dsa_prefill_config, \
    make_prefill, make_decode, make_dsa, make_dsa_prefill  # noqa: E402

PARAMS = NSAParams()


# ---------------------------------------------------------------- work counts
def prefill_counts(T, H, G, dk, dv, B=1, p=PARAMS):
    """Attended keys per branch summed over query rows, and useful FLOPs:
    2*(dk+dv)*H*keys per branch plus the compression GEMM."""
    t = np.arange(T, dtype=np.int64)
    Nc = 0 if T < p.l else (T - p.l) // p.d + 1
    cmp_k = np.where(t >= p.l - 1, np.minimum((t - (p.l - 1)) // p.d + 1, Nc), 0).sum()
    jt = t // p.lsel
    sel_k = ((np.minimum(p.n, jt + 1) - 1) * p.lsel + (t - p.lsel * jt + 1)).sum()
    win_k = np.minimum(p.w, t + 1).sum()
    per_key = 2 * (dk + dv) * H * B
    f = dict(cmp=float(per_key * cmp_k), sel=float(per_key * sel_k), win=float(per_key * win_k),
             phi=float(2 * Nc * (p.l * dk * dk + p.l * dv * dv) * G * B))
    f["total"] = sum(f.values())
    return f, Nc


def decode_bytes(B, G, T, dk, dv, p=PARAMS):
    """Bytes one decode step must read: per KV head the visible compressed
    entries, the n selected blocks and the window (K and V, bf16)."""
    Nc = 0 if T < p.l else (T - p.l) // p.d + 1
    ncmp = min(Nc, (T - 1 - (p.l - 1)) // p.d + 1)
    jt = (T - 1) // p.lsel
    nsel = (min(p.n, jt + 1) - 1) * p.lsel + (T - p.lsel * jt)
    nwin = min(p.w, T)
    return (ncmp + nsel + nwin) * (dk + dv) * 2 * G * B


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["unsampled"], samples=0)
        sm = [float(r[1]) for r in rows]
        smax = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v and "Not" not in v})
        load = [s for s in sm if s > 0.5 * smax] or sm
        return dict(sm_mhz=statistics.median(load), sm_max_mhz=smax, reasons=reasons, samples=len(rows),
                    power_w_max=max(float(r[3]) for r in rows if r[3].strip() not in ("", "[N/A]")))


# ---------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")   # host-only runs of this bookkeeping
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, ms_max: float, ws: int) -> float:
    """Replicas: every rank processes ``units_per_rank``; the job takes the
    slowest rank's time."""
    return ws * units_per_rank / (ms_max * 1e-3)


# DRAM bytes (read + write) per launch or step, from one-pass ncu captures of
# the same launches (dram__bytes_read.sum + dram__bytes_write.sum).  A figure
# is reported only while the kernel sources it was taken from are unchanged
# (sha256 prefix of the listed files); otherwise the bench line says null.
_CSRC = "sparse_attention_long_10_b300/csrc/"
NCU_TRAFFIC = {
    "cmp_win": {"files": ["prefill_cmp_win.cu", "common.cuh"], "sha": "e959ad480b14df14",
                "bytes": (1857.92 + 2115.24) * 1e6, "how": "full-size capture (one pass)"},
    "sel": {"files": ["prefill_sel.cu", "common.cuh"], "sha": "10bdbff3281aef65",
            "bytes": (4423.19 + 1073.58) * 1e6, "how": "full-size capture (one pass)"},
    # both kernels of one decode step
    "decode": {"files": ["decode.cu", "common.cuh"], "sha": "e50108f99388e6fe",
               "bytes": (189.29 + 9.81 + 52.01 + 0.01) * 1e6, "how": "full-size capture, both kernels"},
    # the four kernels of one DSA step
    "dsa": {"files": ["dsa.cu", "common.cuh", "warp_mma.cuh"], "sha": "32d048ff48605774",
            "bytes": (134.26 + 4.10 + 4.40 + 36.96 + 8.43) * 1e6, "how": "full-size capture, four kernels"},
    # the nine largest kernels of one backward step (dq x 2, dK/dV x 3, dx x 2, dw x 2)
    "backward": {"files": ["backward.cu", "common.cuh"], "sha": "2680b909956a1c8b",
                 "bytes": (2984.45 + 8892.27 + 3190.17 + 39265.95 + 12238.97 + 217.73 + 118.14 + 143.73 + 77.62) * 1e6 +
                          (3291.44 + 3293.89 + 42.27 + 492.96 + 323.55 + 140.83 + 0.38 + 73.53 + 0.11) * 1e6,
                 "how": "full-size capture (one pass), the step's nine largest kernels"},
    "dsa_latent": {"files": ["dsa.cu", "common.cuh", "warp_mma.cuh"], "sha": "32d048ff48605774",
                   "bytes": (134.25 + 4.04 + 4.40 + 20.18 + 8.43) * 1e6,
                   "how": "full-size capture, four kernels"},
}

def ncu_traffic(key: str):
    import hashlib
    ent = NCU_TRAFFIC[key]
    h = hashlib.sha256()
    root = os.path.dirname(os.path.abspath(__file__))
    for f in ent["files"]:
        with open(os.path.join(root, _CSRC, f), "rb") as fh:
            h.update(fh.read())
    return ent["bytes"] if h.hexdigest()[:16] == ent["sha"] else None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return dict(hbm=m["hbm_gbs"], bf16=m["bf16_tflops"], bf16_sus=m["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


# ---------------------------------------------------------------- CPU oracle baseline
def oracle_prefill_rate(inp, rows_per_step: int, steps: int, seed: int = 0):
    """Time the fp64 oracle on the host: compression of every KV head once, then
    ``steps`` steps of ``rows_per_step`` uniformly sampled query rows (all
    heads, all three branches).  Returns projected tokens/s for the whole
    sequence and the timing details."""
    from oracle import nsa as O
    B, T, H, dk = inp["q"].shape
    G = inp["k"].shape[2]
    t0 = time.perf_counter()
    pe_k, pe_v = O.to_f64(inp["pe_k"]), O.to_f64(inp["pe_v"])
    w_k, w_v = O.to_f64(inp["w_k"]), O.to_f64(inp["w_v"])
    kc = np.stack([O.compress(O.to_f64(inp["k"][0, :, g]), pe_k, w_k, PARAMS.l, PARAMS.d) for g in range(G)])
    vc = np.stack([O.compress(O.to_f64(inp["v"][0, :, g]), pe_v, w_v, PARAMS.l, PARAMS.d) for g in range(G)])
    t_compress = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    step_times = []
    for _ in range(steps):
        rows = np.sort(rng.integers(0, T, rows_per_step))
        s0 = time.perf_counter()
        O.nsa_prefill_reference(inp, rows=rows, kc=kc, vc=vc)
        step_times.append(time.perf_counter() - s0)
    t_row = sum(step_times) / (steps * rows_per_step)
    rate = T / (t_compress + T * t_row)
    return rate, dict(t_compress_s=t_compress, t_row_s=t_row, step_times=step_times)


def cpu_cores():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        blas = max((i.get("num_threads", 1) for i in info), default=1)
    except Exception:
        blas = 1
    return blas, os.cpu_count()


# ---------------------------------------------------------------- our arm
def run_ours(args, ws, rank):
    import sparse_attention_long_10_b300 as nsa
    wl = PREFILL_CONFIGS[args.workload]
    B, T, H, G, dk, dv = wl.B, wl.T, wl.H, wl.G, wl.dk, wl.dv
    inp = make_prefill(wl)
    dev = {k: v.cuda() for k, v in inp.items()}
    cfg = nsa.make_cfg(B, T, H, G, dk, dv, phi=dev)
    Nc = nsa.nsa_num_compressed(cfg)
    kc = torch.empty(B, G, Nc, dk, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty(B, G, Nc, dv, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(B, T, H, dv, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(B, T, G, PARAMS.n, dtype=torch.int32, device="cuda")
    wsp = nsa.workspace(nsa.nsa_prefill_workspace_size(cfg))
    stream = torch.cuda.current_stream()

    def step():
        nsa.nsa_prefill_fwd(cfg, dev["q"], dev["k"], dev["v"], dev["gates"], kc, vc, out, idx, wsp, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("device status set during warm-up")

    # ---- device-resident timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, ws)
    status = nsa.nsa_device_status(wsp)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # ---- same steps with per-launch events: kernel shares and the roofline
    nsa.nsa_profile_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = nsa.nsa_profile_read()
    nsa.nsa_profile_enable(False)
    launches = sum(c for c, _ in prof.values())

    # ---- end to end through host buffers: every step uploads its inputs from
    # pinned host memory and downloads its output, pipelined as a serving
    # loop runs it: step i+1's inputs upload (one copy stream) and step i-1's
    # output downloads (another) while step i computes, over two device sets
    keys_in = ("q", "k", "v", "gates", "pe_k", "pe_v", "w_k", "w_v")
    host = {k: inp[k].pin_memory() for k in keys_in}
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys_in)
    d2h = out.numel() * out.element_size()
    sets = [dev, {k: torch.empty_like(dev[k]) for k in keys_in}]
    cfgs = [cfg, nsa.make_cfg(B, T, H, G, dk, dv, phi=sets[1])]
    outs = [out, torch.empty_like(out)]
    outs_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]

    def upload(j):
        for k in keys_in:
            sets[j][k].copy_(host[k], non_blocking=True)

    def compute(j):
        nsa.nsa_prefill_fwd(cfgs[j], sets[j]["q"], sets[j]["k"], sets[j]["v"], sets[j]["gates"], kc, vc,
                            outs[j], idx, wsp, stream)

    def download(j):
        outs_h[j].copy_(outs[j], non_blocking=True)

    barrier(ws)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(pipelined_e2e(upload, compute, download, max(3, args.steps), stream), ws)
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("device status set in the end-to-end region")

    flops, _ = prefill_counts(T, H, G, dk, dv, B)
    pk = peaks()
    dense = run_dense_arm(nsa, cfg, dev, B, T, H, G, dk, dv, ms, stream, args)
    dom = max(prof.items(), key=lambda kv: kv[1][1])
    dom_name, (dom_n, dom_ms) = dom
    dom_avg_ms = dom_ms / dom_n
    dom_flops = dict(cmp_win=flops["cmp"] + flops["win"], sel=flops["sel"],
                     compress_gemm=flops["phi"] / 2).get(dom_name, float("nan"))
    achieved = dom_flops / (dom_avg_ms * 1e-3) / 1e12
    tok_s = whole_job_rate(B * T, ms, ws)
    res = {
        "metric": "NSA 64k prefill tokens/s" if T == 65536 else f"NSA prefill tokens/s (T={T})",
        "value": tok_s,
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, learned-map-like phi draws, sigmoid gates)",
        "config": {"workload": wl.name, "B": B, "T": T, "H": H, "G": G, "dk": dk, "dv": dv,
                   "l": PARAMS.l, "d": PARAMS.d, "lsel": PARAMS.lsel, "n": PARAMS.n, "w": PARAMS.w,
                   "parallelism": f"replicas x{ws} (independent sequences)",
                   "l2_flush": "inputs larger than L2 (q 1.6 GB)"},
        "useful_tflops": flops["total"] / (ms * 1e-3) / 1e12,
        "useful_tflop_per_step": flops["total"] / 1e12,
        "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": achieved,
                     "peak": pk["bf16_sus"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_sus"],
                     "peak_kind": f"bf16 dense sustained ({pk['src']})",
                     "algorithmic_tflop_per_launch": dom_flops / 1e12, "avg_launch_ms": dom_avg_ms,
                     "traffic": ncu_traffic(dom_name) if dom_name in NCU_TRAFFIC else None,
                     "traffic_how": NCU_TRAFFIC[dom_name]["how"] if dom_name in NCU_TRAFFIC else None},
        "kernels": {k: {"launches_per_step": c / args.steps, "ms_per_step": t / args.steps,
                        "share": t / sum(x[1] for x in prof.values())} for k, (c, t) in prof.items()},
        "gpu_launches": int(launches),
        "dense": dense,
        "e2e": {"value": whole_job_rate(B * T, ms_e2e, ws), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e, "how": PIPELINE_HOW},
        "clocks": clk.summary(),
    }
    return res, inp


def run_dense_arm(nsa, cfg, dev, B, T, H, G, dk, dv, nsa_ms, stream, args):
    """Exact causal full attention on the same q/k/v (nsa_full_attn_fwd): the
    dense comparison the pages quote NSA's 9.0x forward speed-up against."""
    out = torch.empty(B, T, H, dv, dtype=torch.bfloat16, device="cuda")
    wsp = nsa.workspace(nsa.nsa_full_attn_workspace_size(cfg))

    def step():
        nsa.nsa_full_attn_fwd(cfg, dev["q"], dev["k"], dev["v"], out, wsp, stream)

    step()
    torch.cuda.synchronize()
    n = max(2, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("dense arm: device status set")
    ms = e0.elapsed_time(e1) / n
    fl = 2.0 * (dk + dv) * H * B * T * (T + 1) / 2
    return {"what": "exact causal full attention on the same inputs (nsa_full_attn_fwd: one-pass online "
                    "softmax, tcgen05, 8 queries x 16 heads per 128-row tile)",
            "ms_per_step": ms, "steps": n, "useful_tflop_per_step": fl / 1e12,
            "useful_tflops": fl / (ms * 1e-3) / 1e12,
            "nsa_speedup": ms / nsa_ms, "pages_forward_speedup_64k_context": 9.0}


# ---------------------------------------------------------------- decode leg
class L2Flush:
    """Evicts a step's data from the 126 MB L2 before a timed replay: writes a
    256 MB buffer, then reads a second 256 MB one.  The read pushes the lines
    the write left dirty back to HBM, so their write-back happens here, outside
    the timed interval, and the step starts with an L2 of clean lines that it
    never reads."""

    def __init__(self):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(64 << 20, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.w.add_(1)
        self.r.sum()


L2_FLUSH_NOTE = "256 MB written, then another 256 MB read, before every step (outside the timed interval)"


def time_graph_steps(graph, steps, flush):
    """Device time of ``steps`` replays of ``graph`` (ms each), with the L2
    flushed by ``flush`` (an L2Flush) before every replay and outside the
    timed interval."""
    times = []
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        times.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def pipelined_e2e(upload, compute, download, n_steps, stream):
    """Per-step time (ms) of ``n_steps`` end-to-end steps run as a serving loop
    runs them, over two device input / output sets j = i % 2: upload(j) on
    one copy stream, compute(j) on ``stream``, download(j) on another copy
    stream; step i+1's upload and step i-1's download overlap step i's
    compute, and events order every reuse of a set."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in_ready", "in_free", "out_ready", "out_free")}

    def run(n):
        for e in ev["in_free"] + ev["out_free"]:
            e.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(n):
            j = i & 1
            s_in.wait_event(ev["in_free"][j])       # step i-2 has read set j
            with torch.cuda.stream(s_in):
                upload(j)
            ev["in_ready"][j].record(s_in)
            stream.wait_event(ev["in_ready"][j])
            stream.wait_event(ev["out_free"][j])    # step i-2's output is downloaded
            compute(j)
            ev["in_free"][j].record(stream)
            ev["out_ready"][j].record(stream)
            s_out.wait_event(ev["out_ready"][j])
            with torch.cuda.stream(s_out):
                download(j)
            ev["out_free"][j].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(n_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n_steps


PIPELINE_HOW = ("per step: inputs uploaded from pinned host memory, the C-ABI call, output downloaded; uploads and "
                "downloads on their own streams overlap the neighbouring steps' compute (two device input / output "
                "sets)")


class PackedInputs:
    """A step's small inputs packed into one pinned host buffer, uploaded with
    one copy into one device buffer whose slices (256-byte aligned) are the
    tensors the C-ABI call reads."""

    def __init__(self, tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off = (off + t.numel() * t.element_size() + 255) // 256 * 256
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device="cuda")
        self.views = []
        for t, o in zip(tensors, offs):
            n = t.numel() * t.element_size()
            self.host[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
            self.views.append(self.dev[o:o + n].view(t.dtype).view(t.shape))
        self.nbytes = sum(t.numel() * t.element_size() for t in tensors)

    def upload(self):
        self.dev.copy_(self.host, non_blocking=True)


def time_e2e_graph(step_e2e, steps, flush, ws):
    """End-to-end time of a decode-type step (ms): the step's host-to-device
    input copies, the C-ABI call and the device-to-host copy of its result,
    captured once in a CUDA graph (as a serving loop runs a step) and
    replayed ``steps`` times with the L2 flushed before each replay; the
    copies run inside every timed replay."""
    for _ in range(3):
        step_e2e()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step_e2e()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    return max_over_ranks(statistics.mean(time_graph_steps(g, steps, flush)), ws)


E2E_HOW = ("CUDA graph replay of the step's input upload from pinned host memory (one packed copy), the C-ABI "
           "call and the result copy back")


def run_decode_leg(args, ws):
    """One NSA decode step for 16 sequences with 65,536-token caches: the
    query at t = T-1 reads 4095 compressed entries, 16 kept blocks and the
    512-token window per KV head.  The compressed caches are precomputed once
    (they are decode-time state, like the KV cache)."""
    import sparse_attention_long_10_b300 as nsa
    wl = decode_config()
    B, T, H, G, dk, dv = wl.B, wl.T, wl.H, wl.G, wl.dk, wl.dv
    inp = make_decode(wl)
    dev = {k: v.cuda() for k, v in inp.items()}
    cfg = nsa.make_cfg(B, T, H, G, dk, dv, phi=dev)
    Nc = nsa.nsa_num_compressed(cfg)
    kc = torch.empty(B, G, Nc, dk, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty(B, G, Nc, dv, dtype=torch.bfloat16, device="cuda")
    cws = nsa.workspace(nsa.nsa_compress_workspace_size(cfg))
    nsa.nsa_compress_kv(cfg, nsa.NSA_LAYOUT_BGTD, dev["kcache"], dev["vcache"], kc, vc, cws)
    out = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
    wsp = nsa.workspace(nsa.nsa_decode_workspace_size(cfg))

    def step(stream=None):
        nsa.nsa_decode_step(cfg, dev["q"], dev["kcache"], dev["vcache"], kc, vc, dev["gates"], out, None,
                            wsp, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("decode: device status set during warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    flush = L2Flush()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    ms = statistics.mean(time_graph_steps(graph, args.steps, flush))
    ms = max_over_ranks(ms, ws)
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("decode: device status set in the timed region")
    # per-kernel split (eager launches bracketed by events, L2 flushed between steps)
    nsa.nsa_profile_enable(True)
    for _ in range(args.steps):
        flush()
        step()
    torch.cuda.synchronize()
    prof = nsa.nsa_profile_read()
    nsa.nsa_profile_enable(False)
    # end to end: the new token's q, gates and K/V row uploaded in one copy
    # (the rows then placed into the caches on the device), out copied back
    pk_in = PackedInputs([inp["q"], inp["gates"], inp["kcache"][:, :, T - 1], inp["vcache"][:, :, T - 1]])
    q_v, g_v, krow_v, vrow_v = pk_in.views
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = pk_in.nbytes
    d2h = out_h.numel() * out_h.element_size()

    def step_e2e():
        pk_in.upload()
        dev["kcache"][:, :, T - 1].copy_(krow_v, non_blocking=True)
        dev["vcache"][:, :, T - 1].copy_(vrow_v, non_blocking=True)
        nsa.nsa_decode_step(cfg, q_v, dev["kcache"], dev["vcache"], kc, vc, g_v, out, None, wsp, None)
        out_h.copy_(out, non_blocking=True)

    ms_e2e = time_e2e_graph(step_e2e, args.steps, flush, ws)
    nbytes = decode_bytes(B, G, T, dk, dv)
    pk = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    kern = {k: {"launches_per_step": c / args.steps, "us_per_step": 1e3 * t / args.steps}
            for k, (c, t) in prof.items()}
    return {
        "metric": "NSA decode step latency (16 seqs x 65,536-token caches)",
        "value": ms * 1e3, "unit": "us", "higher_is_better": False,
        "workload": wl.name, "steps": args.steps, "l2_flush": L2_FLUSH_NOTE,
        "bytes_per_step": nbytes,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm"], "unit": "GB/s",
                     "frac": gbs / pk["hbm"], "peak_kind": f"HBM copy ({pk['src']})",
                     "frac_of_8TBs": gbs / 8000.0, "traffic": ncu_traffic("decode"),
                     "note": "whole step (memset + 2 kernels, CUDA graph replay), L2 flushed before each step; "
                             "traffic: " + NCU_TRAFFIC["decode"]["how"]},
        "kernels": kern,
        "gpu_launches_per_step": int(sum(c for c, _ in prof.values()) / args.steps),
        "e2e": {"value": ms_e2e * 1e3, "unit": "us", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "how": E2E_HOW},
    }


# ---------------------------------------------------------------- multi-token decode leg
def run_decode_multi_leg(args, ws, m=4):
    """m new tokens per sequence (positions T-m .. T-1) for the 16 sequences
    with 65,536-token caches, in one nsa_decode_multi call: each token keeps
    its own selection; the chunk shares the compressed and window tiles."""
    import sparse_attention_long_10_b300 as nsa
    from workloads import make_decode_multi
    wl = decode_config()
    B, T, H, G, dk, dv = wl.B, wl.T, wl.H, wl.G, wl.dk, wl.dv
    inp = make_decode_multi(wl, m)
    dev = {k: v.cuda() for k, v in inp.items()}
    cfg = nsa.make_cfg(B, T, H, G, dk, dv, phi=dev)
    Nc = nsa.nsa_num_compressed(cfg)
    kc = torch.empty(B, G, Nc, dk, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty(B, G, Nc, dv, dtype=torch.bfloat16, device="cuda")
    cws = nsa.workspace(nsa.nsa_compress_workspace_size(cfg))
    nsa.nsa_compress_kv(cfg, nsa.NSA_LAYOUT_BGTD, dev["kcache"], dev["vcache"], kc, vc, cws)
    out = torch.empty(B, m, H, dv, dtype=torch.bfloat16, device="cuda")
    wsp = nsa.workspace(nsa.nsa_decode_multi_workspace_size(cfg, m))

    def step():
        nsa.nsa_decode_multi(cfg, m, dev["q"], dev["kcache"], dev["vcache"], kc, vc, dev["gates"], out, None, wsp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("decode multi: device status set during warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    flush = L2Flush()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    ms = max_over_ranks(statistics.mean(time_graph_steps(graph, args.steps, flush)), ws)
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("decode multi: device status set in the timed region")
    nsa.nsa_profile_enable(True)
    for _ in range(args.steps):
        flush()
        step()
    torch.cuda.synchronize()
    prof = nsa.nsa_profile_read()
    nsa.nsa_profile_enable(False)
    return {
        "metric": f"NSA multi-token decode step latency (16 seqs x 65,536-token caches, {m} new tokens each)",
        "value": ms * 1e3, "unit": "us", "higher_is_better": False, "workload": f"{wl.name}_m{m}",
        "steps": args.steps, "l2_flush": L2_FLUSH_NOTE, "tokens_per_step": B * m, "tokens_per_s": B * m / (ms * 1e-3),
        "kernels": {k: {"launches_per_step": c / args.steps, "us_per_step": 1e3 * t / args.steps}
                    for k, (c, t) in prof.items()},
        "gpu_launches_per_step": int(sum(c for c, _ in prof.values()) / args.steps),
        "note": "CUDA graph replay, L2 flushed before each step",
    }


# ---------------------------------------------------------------- DSA decode leg
def run_dsa_prefill_leg(args, ws):
    """DSA over a whole sequence: one 8,192-token sequence, every position a
    query with its own indexer query and weights, keeping min(2048, t+1)
    positions of its causal prefix; latent keys (576 columns, the first 512
    are the values)."""
    import sparse_attention_long_10_b300 as nsa
    wl = dsa_prefill_config()
    inp = make_dsa_prefill(wl)
    inp["v"] = None
    dev = {k: v.cuda() for k, v in inp.items() if v is not None}
    cfg = nsa.make_dsa_cfg(wl.B, wl.T, wl.HI, wl.dI, wl.H, wl.dk, wl.dv, wl.topk)
    out = torch.empty(wl.B, wl.T, wl.H, wl.dv, dtype=torch.bfloat16, device="cuda")
    wsp = nsa.workspace(nsa.dsa_prefill_workspace_size(cfg))

    def step():
        nsa.dsa_prefill_fwd(cfg, dev["qI"], dev["wI"], dev["kI"], dev["q"], dev["k"], None, out, None, wsp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("dsa prefill: device status set during warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    flush = L2Flush()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    ms = max_over_ranks(statistics.mean(time_graph_steps(graph, args.steps, flush)), ws)
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("dsa prefill: device status set in the timed region")
    nsa.nsa_profile_enable(True)
    for _ in range(args.steps):
        flush()
        step()
    torch.cuda.synchronize()
    prof = nsa.nsa_profile_read()
    nsa.nsa_profile_enable(False)
    # end to end: the sequence's inputs uploaded (one packed copy), out back,
    # pipelined over two device sets
    packs = [PackedInputs([inp["qI"], inp["wI"], inp["kI"], inp["q"], inp["k"]]) for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    outs_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = packs[0].nbytes
    d2h = out.numel() * out.element_size()
    stream = torch.cuda.current_stream()

    def compute(j):
        qI_v, wI_v, kI_v, q_v, k_v = packs[j].views
        nsa.dsa_prefill_fwd(cfg, qI_v, wI_v, kI_v, q_v, k_v, None, outs[j], None, wsp, stream)

    barrier(ws)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(pipelined_e2e(lambda j: packs[j].upload(), compute,
                                          lambda j: outs_h[j].copy_(outs[j], non_blocking=True),
                                          max(3, args.steps), stream), ws)
    # useful work: the indexer over every causal prefix, the attention over the kept positions
    t1 = torch.arange(1, wl.T + 1, dtype=torch.float64)
    idx_flop = float(t1.sum()) * wl.HI * wl.dI * 2 * wl.B
    att_flop = float(torch.clamp(t1, max=wl.topk).sum()) * wl.H * (wl.dk + wl.dv) * 2 * wl.B
    pk = peaks()
    tf = (idx_flop + att_flop) / (ms * 1e-3) / 1e12
    return {
        "metric": "DSA prefill (1 x 8,192 tokens, every position a query, top-2048, latent KV)",
        "value": wl.B * wl.T / (ms * 1e-3), "unit": "tokens/s", "higher_is_better": True,
        "ms_per_step": ms, "workload": wl.name, "steps": args.steps, "l2_flush": L2_FLUSH_NOTE,
        "useful_tflop_per_step": (idx_flop + att_flop) / 1e12,
        "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_sus"], "unit": "TFLOP/s",
                     "frac": tf / pk["bf16_sus"], "peak_kind": f"bf16 dense sustained ({pk['src']})",
                     "traffic": None,
                     "note": "indexer + attention FLOPs over the step (memset + 4 kernels, CUDA graph replay); "
                             "the attention's MMAs have N = 16 heads"},
        "kernels": {k: {"launches_per_step": c / args.steps, "us_per_step": 1e3 * t / args.steps}
                    for k, (c, t) in prof.items()},
        "gpu_launches_per_step": int(sum(c for c, _ in prof.values()) / args.steps),
        "e2e": {"value": wl.B * wl.T / (ms_e2e * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "how": PIPELINE_HOW},
    }


def run_backward_leg(args, ws):
    """NSA backward over the 64k prefill (B=1, T=65,536, H=64, G=4, dk=192,
    dv=128): gradients of every input (q, k, v, gates, W_c, PE) given the
    forward's compressed cache, kept blocks and saved selected-branch
    statistics, and a bf16 upstream gradient.  The forward runs before the
    timed region; every step is one nsa_prefill_bwd call (inputs far above
    the L2 size, so no flush)."""
    import sparse_attention_long_10_b300 as nsa
    from workloads import make_prefill_dout
    wl = PREFILL_CONFIGS["prefill_64k"]
    inp = make_prefill(wl)
    dev = {k: v.cuda() for k, v in inp.items()}
    dout = make_prefill_dout(wl).cuda()
    B, T, H, G, dk, dv = wl.B, wl.T, wl.H, wl.G, wl.dk, wl.dv
    cfg = nsa.make_cfg(B, T, H, G, dk, dv, phi=dev)
    Nc = nsa.nsa_num_compressed(cfg)
    kc = torch.empty(B, G, Nc, dk, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty(B, G, Nc, dv, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(B, T, H, dv, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(B, T, G, PARAMS.n, dtype=torch.int32, device="cuda")
    wsf = nsa.workspace(nsa.nsa_prefill_workspace_size(cfg))
    f32 = dict(dtype=torch.float32, device="cuda")
    slc_lse = torch.empty(B, T, H, **f32)
    slc_o = torch.empty(B, T, H, dv, **f32)

    def fwd():
        nsa.nsa_prefill_fwd_train(cfg, dev["q"], dev["k"], dev["v"], dev["gates"], kc, vc, out, idx, slc_lse,
                                  slc_o, wsf)
    for _ in range(2):
        fwd()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    for _ in range(3):
        fwd()
    f1.record()
    torch.cuda.synchronize()
    ms_fwd_train = f0.elapsed_time(f1) / 3
    grads = [torch.empty(B, T, H, dk, **f32), torch.empty(B, T, G, dk, **f32), torch.empty(B, T, G, dv, **f32),
             torch.empty(B, T, H, 3, **f32), torch.empty(32 * dk, dk, **f32), torch.empty(32 * dv, dv, **f32),
             torch.empty(32, dk, **f32), torch.empty(32, dv, **f32)]
    wsb = nsa.workspace(nsa.nsa_prefill_bwd_workspace_size(cfg))

    def step():
        nsa.nsa_prefill_bwd(cfg, dev["q"], dev["k"], dev["v"], dev["gates"], kc, vc, idx, dout, *grads, wsb,
                            slc_lse=slc_lse, slc_o=slc_o)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if nsa.nsa_device_status(wsb) != 0:
        raise RuntimeError("backward: device status set during warm-up")
    steps = max(2, min(args.steps, 5))
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, ws)
    if nsa.nsa_device_status(wsb) != 0:
        raise RuntimeError("backward: device status set in the timed region")
    nsa.nsa_profile_enable(True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    prof = nsa.nsa_profile_read()
    nsa.nsa_profile_enable(False)
    # algorithmic work: 2.5x the forward's attention FLOPs (S recomputed, dP,
    # dV, dK, dq) plus twice the compression GEMM (dX and dW)
    f, _ = prefill_counts(T, H, G, dk, dv, B)
    att_fwd = f["cmp"] + f["sel"] + f["win"]
    flops = 2.5 * att_fwd + 2 * f["phi"]
    pk = peaks()
    tf = flops / (ms * 1e-3) / 1e12
    return {
        "metric": "NSA 64k backward tokens/s", "value": B * T / (ms * 1e-3), "unit": "tokens/s",
        "higher_is_better": True, "ms_per_step": ms, "workload": wl.name + "_backward", "steps": steps,
        "forward_train_ms": ms_fwd_train,
        "how": "nsa_prefill_bwd reading the selected branch's statistics that nsa_prefill_fwd_train saved "
               "(the forward, outside the timed region, takes forward_train_ms)",
        "useful_tflop_per_step": flops / 1e12,
        "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_sus"], "unit": "TFLOP/s",
                     "frac": tf / pk["bf16_sus"], "peak_kind": f"bf16 dense sustained ({pk['src']})",
                     "traffic": ncu_traffic("backward"), "traffic_how": NCU_TRAFFIC["backward"]["how"],
                     "note": "2.5 x the forward's attention FLOPs + 2 x the compression GEMM over the whole call; "
                             "traffic is DRAM bytes per step"},
        "kernels": {k: {"launches_per_step": c / steps, "ms_per_step": t / steps} for k, (c, t) in prof.items()},
        # profiled spans: the list building is 3 kernels, the compression backward 8
        "gpu_launches_per_step": int(sum(c * {"bwd_lists": 3, "bwd_compress": 8}.get(k, 1)
                                         for k, (c, _) in prof.items()) / steps),
    }


def run_dsa_leg(args, ws, latent=False):
    """One DSA-style decode step: batch 8, 131,072-token context, indexer of 4
    heads x 64 dims, top-2048 positions, attention of 16 heads (dk=576,
    dv=512) over the kept positions only.  latent: the values are the first
    512 columns of the 576-column key rows (latent KV), so only keys are
    gathered."""
    import sparse_attention_long_10_b300 as nsa
    wl = dsa_config()
    inp = make_dsa(wl)
    if latent:
        inp["v"] = None
    dev = {k: v.cuda() for k, v in inp.items() if v is not None}
    cfg = nsa.make_dsa_cfg(wl.B, wl.T, wl.HI, wl.dI, wl.H, wl.dk, wl.dv, wl.topk)
    out = torch.empty(wl.B, wl.H, wl.dv, dtype=torch.bfloat16, device="cuda")
    wsp = nsa.workspace(nsa.dsa_decode_workspace_size(cfg))

    def step():
        nsa.dsa_decode_step(cfg, dev["qI"], dev["wI"], dev["kI"], dev["q"], dev["k"], dev.get("v"), out, None,
                            wsp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("dsa: device status set during warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    flush = L2Flush()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    ms = max_over_ranks(statistics.mean(time_graph_steps(graph, args.steps, flush)), ws)
    if nsa.nsa_device_status(wsp) != 0:
        raise RuntimeError("dsa: device status set in the timed region")
    nsa.nsa_profile_enable(True)
    for _ in range(args.steps):
        flush()
        step()
    torch.cuda.synchronize()
    prof = nsa.nsa_profile_read()
    nsa.nsa_profile_enable(False)
    # end to end: the new token's queries and indexer weights uploaded in one
    # copy, out copied back
    pk_in = PackedInputs([inp["qI"], inp["wI"], inp["q"]])
    qI_v, wI_v, q_v = pk_in.views
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = pk_in.nbytes
    d2h = out_h.numel() * out_h.element_size()

    def step_e2e():
        pk_in.upload()
        nsa.dsa_decode_step(cfg, qI_v, wI_v, dev["kI"], q_v, dev["k"], dev.get("v"), out, None, wsp)
        out_h.copy_(out, non_blocking=True)

    ms_e2e = time_e2e_graph(step_e2e, args.steps, flush, ws)
    kk = min(wl.topk, wl.T)
    nbytes = wl.B * wl.T * wl.dI * 2 + wl.B * kk * (wl.dk + (0 if latent else wl.dv)) * 2
    pk = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {
        "metric": ("DSA decode step latency, latent KV (values = first 512 key columns)" if latent else
                   "DSA decode step latency") + " (8 rows x 131,072-token context, top-2048)",
        "value": ms * 1e3, "unit": "us", "higher_is_better": False,
        "workload": wl.name + ("_latent" if latent else ""), "steps": args.steps, "l2_flush": L2_FLUSH_NOTE,
        "bytes_per_step": nbytes,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm"], "unit": "GB/s",
                     "frac": gbs / pk["hbm"], "peak_kind": f"HBM copy ({pk['src']})",
                     "traffic": ncu_traffic("dsa_latent" if latent else "dsa"),
                     "note": "whole step (memset + 4 kernels, CUDA graph replay), L2 flushed before each step; "
                             "traffic: " + NCU_TRAFFIC["dsa_latent" if latent else "dsa"]["how"]},
        "kernels": {k: {"launches_per_step": c / args.steps, "us_per_step": 1e3 * t / args.steps}
                    for k, (c, t) in prof.items()},
        "gpu_launches_per_step": int(sum(c for c, _ in prof.values()) / args.steps),
        "e2e": {"value": ms_e2e * 1e3, "unit": "us", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "how": E2E_HOW},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode and DSA decode legs")
    ap.add_argument("--workload", default="prefill_64k",
                    choices=sorted(PREFILL_CONFIGS) + ["decode_64k", "dsa_128k", "dsa_latent_128k",
                                                       "dsa_prefill_8k", "backward_64k"],
                    help="prefill workload (the headline is prefill_64k; smaller ones serve profiling) or "
                         "decode_64k / dsa_128k / dsa_latent_128k / dsa_prefill_8k / backward_64k: one of the other legs "
                         "alone")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws, rank, _ = dist_setup()

    if args.impl == "reference":
        if rank != 0:
            return
        wl = PREFILL_CONFIGS["prefill_64k"]
        inp = make_prefill(wl)
        blas, ncpu = cpu_cores()
        rate, info = oracle_prefill_rate(inp, rows_per_step=8, steps=args.steps + args.warmup)
        st = info["step_times"][args.warmup:]
        res = {"impl": "reference", "metric": "NSA 64k prefill tokens/s", "value": rate, "unit": "tokens/s",
               "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": 1e3 * sum(st) / len(st), "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f64", "data": "synthetic",
               "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "G": wl.G, "dk": wl.dk, "dv": wl.dv},
               "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": blas, "host_cpus": ncpu,
                                "kind": "oracle",
                                "sample": f"compression of all {wl.G} KV heads once "
                                          f"({info['t_compress_s']:.1f} s) + 8 sampled query rows per step; "
                                          f"projected to the {wl.T}-token sequence"},
               "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(res), flush=True)
        return

    if args.workload in ("decode_64k", "dsa_128k", "dsa_latent_128k", "dsa_prefill_8k", "backward_64k"):
        if args.workload == "decode_64k":
            res = run_decode_leg(args, ws)
        elif args.workload == "backward_64k":
            res = run_backward_leg(args, ws)
        elif args.workload == "dsa_prefill_8k":
            res = run_dsa_prefill_leg(args, ws)
        else:
            res = run_dsa_leg(args, ws, latent=args.workload == "dsa_latent_128k")
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    res, inp = run_ours(args, ws, rank)
    if not args.no_decode:
        res["decode"] = run_decode_leg(args, ws)
        res["gpu_launches"] += res["decode"]["gpu_launches_per_step"] * args.steps
        res["decode_multi"] = run_decode_multi_leg(args, ws)
        res["gpu_launches"] += res["decode_multi"]["gpu_launches_per_step"] * args.steps
        res["dsa"] = run_dsa_leg(args, ws)
        res["gpu_launches"] += res["dsa"]["gpu_launches_per_step"] * args.steps
        res["dsa_latent"] = run_dsa_leg(args, ws, latent=True)
        res["gpu_launches"] += res["dsa_latent"]["gpu_launches_per_step"] * args.steps
        res["dsa_prefill"] = run_dsa_prefill_leg(args, ws)
        res["gpu_launches"] += res["dsa_prefill"]["gpu_launches_per_step"] * args.steps
        res["backward"] = run_backward_leg(args, ws)
        res["gpu_launches"] += res["backward"]["gpu_launches_per_step"] * res["backward"]["steps"]
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        blas, ncpu = cpu_cores()
        rate, info = oracle_prefill_rate(inp, rows_per_step=16, steps=2)
        res["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": blas, "host_cpus": ncpu,
                               "kind": "oracle",
                               "sample": f"compression of all KV heads ({info['t_compress_s']:.1f} s) + 32 "
                                         f"sampled query rows ({info['t_row_s'] * 1e3:.1f} ms/row), "
                                         f"projected to 65,536 rows"}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
