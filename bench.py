"""Benchmark of the decode-attention hot path on one B300 (replicas on N).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the absorbed-MLA pipeline over one batch of the
DeepSeek-V3-like decode workload (b=32, h=128, d=128, k=512, p=64, t=4096,
s=1): query absorption GEMM, tcgen05 latent attention (+ split combine) and
the W_uv projection. Inputs are seeded synthetic tensors already resident in
HBM; three full input sets (about 555 MB, far above the 126 MB L2) rotate
between steps so no step reads another step's data from L2. Steps are
replayed from CUDA graphs captured once per input set.

Printed: one JSON line (rank 0). `value` is microseconds per pipeline call of
the whole job (the timed time divided by the calls all ranks made), so lower
is better. `roofline` is for the latent-attention call (kernel + combine),
timed in its own loop of graph replays with CUDA events on its stream.
`e2e` times the public Python API with every step's queries and lengths copied
in from pinned host memory and its outputs copied back, the copies on their own
streams overlapping the neighbouring steps' compute. `cpu_baseline` times the
fp64 oracle on a bounded sample on the host cores.

--impl reference runs that oracle as the reference arm (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn µs/call, TFLOP/s, HBM GB/s and % roofline (MLA h128 k512 t4096)"
UNIT = "us/call"
WORKLOAD = "mla_dsv3"
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
E2E_STEPS = 400


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the grouped-head and s-sweep side measurements")
    ap.add_argument("--profile", default=None, metavar="WORKLOAD",
                    help="profiling mode: run --warmup + --steps calls of one op on one input set of the named "
                         "workload (mla_dsv3, mla_mtp_s8, gqa_64_8, gqa_paged_hkv4, gqa_64_8_fp8, gqa_paged_hkv1_tc ...: _tc pins "
                         "the tensor-core grouped-head kernel, _split the split-KV kernels) and exit; "
                         "MLA workloads run whole pipeline steps; prints no "
                         "bench line (numbers taken under a profiler are not bench values)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


class ClockSampler:
    """Samples SM clocks and clock-event reasons with nvidia-smi (every
    100 ms) while the timed region runs. `gpu` is the device's UUID (or
    index) as nvidia-smi knows it."""

    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu: str, period_ms: int = 100):
        self.gpu, self.period = gpu, period_ms
        self.proc = None
        self.lines = []
        self.error = None

    def __enter__(self):
        import subprocess

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
            time.sleep(0.3)  # let the first sample land before the timed region
        except Exception as e:  # no nvidia-smi: reported, not fatal
            self.error = repr(e)
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, err = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, err = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]
        if not self.lines and err:
            self.error = err.strip()[:200]

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < len(self.FIELDS):
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, val in zip(self.REASONS, f[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0, "error": self.error}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "sm_mhz_min": min(sm), "source": "nvidia-smi -lms %d" % self.period}


def cost_numbers(wl):
    from oracle import cost

    L = wl.seqlens()
    f = cost.mla_flops_exact(wl.heads, wl.k, wl.p, L, wl.s)
    by = cost.mla_bytes_exact(wl.heads, wl.k, wl.p, L, wl.s)
    fa = cost.proj_flops(wl.b, wl.heads, wl.s, wl.d, wl.k)
    ba = cost.proj_bytes(wl.b, wl.heads, wl.s, wl.d, wl.k)
    return f, by, fa, ba


def cpu_baseline(wl, seconds_target=15.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload:
    whole sequences (all heads) of the absorbed pipeline until about
    `seconds_target` seconds of CPU work; scaled to a full call."""
    import numpy as np
    import torch

    from decode_attention_18_b300 import workloads as W
    from oracle import attention as A

    inp = W.make_mla(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, wl.seqlens(), seed=wl.seed, device="cpu")
    f = lambda t: t.float().double().numpy()  # noqa: E731
    wuk, wuv = f(inp.w_uk), f(inp.w_uv)
    n, t_total = 0, 0.0
    while t_total < seconds_target and n < wl.b:
        i = n
        L = inp.seqlens[i]
        zs, kp = [f(inp.z[i, :L])], [f(inp.k_pe[i, :L])]
        qn, qp = f(inp.q_nope[i:i + 1]), f(inp.q_pe[i:i + 1])
        t0 = time.perf_counter()
        A.mla_absorbed_ref(qn, qp, zs, kp, wuk, wuv, [inp.seqlens[i]], inp.scale)
        t_total += time.perf_counter() - t0
        n += 1
    cores = torch.get_num_threads()
    try:
        from threadpoolctl import threadpool_info

        blas = [x.get("num_threads") for x in threadpool_info() if x.get("user_api") == "blas"]
        if blas:
            cores = max(blas)
    except Exception:
        pass
    us_per_call = t_total / n * wl.b * 1e6
    return {"value": us_per_call, "unit": UNIT, "cores": int(cores), "kind": "oracle",
            "sample": f"{n} of {wl.b} sequences (all {wl.heads} heads, absorb + latent attention + W_uv "
                      f"in float64), {t_total:.1f} s of CPU time, scaled x{wl.b / n:.1f} to one call"}


def traffic_record():
    """DRAM bytes (read + write) per launch of the latent kernel from the committed
    ncu summary, if that summary was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "mla_pair_dsv3_b32_h128_k512_t4096_s1.md")
    src = os.path.join(ROOT, "decode_attention_18_b300", "csrc", "mla_decode.cu")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith(("|", "#", " ")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if fields.get("source_sha256_16") != h or "dram_bytes_per_launch" not in fields:
        return None
    return int(fields["dram_bytes_per_launch"])


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np

    from decode_attention_18_b300 import workloads as W
    from oracle import attention as A

    wl = W.WORKLOADS[WORKLOAD]
    inp = W.make_mla(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, wl.seqlens(), seed=wl.seed, device="cpu")
    f = lambda t: t.float().double().numpy()  # noqa: E731
    wuk, wuv = f(inp.w_uk), f(inp.w_uv)
    seqs = [(f(inp.z[i, :inp.seqlens[i]]), f(inp.k_pe[i, :inp.seqlens[i]])) for i in range(2)]

    def step(k):
        i = k % 2
        j = ((k // 2) * heads_per_step) % (wl.heads - heads_per_step + 1)
        hsl = slice(j, j + heads_per_step)
        A.mla_absorbed_ref(f(inp.q_nope[i:i + 1, hsl]), f(inp.q_pe[i:i + 1, hsl]), [seqs[i][0]], [seqs[i][1]],
                           wuk[hsl], wuv[hsl], [inp.seqlens[i]], inp.scale)

    heads_per_step = 1
    t0 = time.perf_counter()
    for k in range(3):
        step(k)
    per_head = (time.perf_counter() - t0) / 3
    budget = 90.0
    heads_per_step = max(1, min(wl.heads, int(budget / max(1, args.steps) / per_head)))
    for k in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(k)
    dt = time.perf_counter() - t0
    sample_units = heads_per_step
    full_units = wl.b * wl.heads
    value = dt / args.steps * (full_units / sample_units) * 1e6
    import torch

    cores = torch.get_num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "step_sample": f"{heads_per_step} head(s) of one sequence per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": int(cores), "kind": "oracle",
                         "sample": f"{heads_per_step} of {full_units} (sequence, head) pairs per step, "
                                   f"scaled x{full_units / sample_units:.0f} to one call"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import build as dabuild
    from decode_attention_18_b300 import workloads as W

    if not os.path.exists(dabuild.LIB):
        raise RuntimeError("libdecattn.so is not built (run: python -m decode_attention_18_b300.build)")
    wl = W.WORKLOADS[WORKLOAD]
    seqlens = wl.seqlens()
    L = max(seqlens)
    NBUF = 3
    sets = [W.make_mla(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, seqlens, seed=wl.seed + 17 * r, device=dev)
            for r in range(NBUF)]
    sl = torch.tensor(seqlens, dtype=torch.int32, device=dev)
    scale = sets[0].scale
    ws_bytes = da.ops.load().mla_decode_workspace_size(wl.b, wl.s, wl.heads, wl.k, L)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    outs = []
    for s_ in sets:
        outs.append(dict(
            qz=torch.empty((wl.b, wl.heads, wl.s, wl.k), dtype=torch.bfloat16, device=dev),
            o_lat=torch.empty((wl.b, wl.heads, wl.s, wl.k), dtype=torch.bfloat16, device=dev),
            lse=torch.empty((wl.b, wl.heads, wl.s), dtype=torch.float32, device=dev),
            out=torch.empty((wl.b, wl.heads, wl.s, wl.d), dtype=torch.bfloat16, device=dev)))

    stream = torch.cuda.Stream(device=dev)

    def step(r, parts=("absorb", "decode", "proj"), seq=None):
        s_, o = sets[r], outs[r]
        sl_ = sl if seq is None else seq
        if "absorb" in parts:
            da.mla_absorb_q(s_.q_nope, s_.w_uk, sl_, out=o["qz"], stream=stream)
        if "decode" in parts:
            da.mla_decode(o["qz"], s_.q_pe, s_.z, s_.k_pe, sl_, scale=scale, max_seqlen=L, out=o["o_lat"],
                          lse=o["lse"], workspace=ws, stream=stream)
        if "proj" in parts:
            da.mla_out_proj(o["o_lat"], s_.w_uv, sl_, out=o["out"], stream=stream)

    # warm (first-call set-up happens outside capture), then capture one graph per input set
    with torch.cuda.stream(stream):
        for r in range(NBUF):
            step(r)
    torch.cuda.synchronize()
    nsplit = da.last_num_splits()
    assert da.check_errors(stream) == 0
    graphs, dgraphs = [], []
    for r in range(NBUF):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(r)
        graphs.append(g)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            step(r, ("decode",))
        dgraphs.append(g2)
    # the same steps back to back: one graph per rotation (a step on each input set in
    # turn), so that programmatic dependent launch also overlaps consecutive steps, as
    # inside a graph of a whole decode step; reported beside the one-step graphs
    rot, drot = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(rot, stream=stream):
        for r in range(NBUF):
            step(r)
    with torch.cuda.graph(drot, stream=stream):
        for r in range(NBUF):
            step(r, ("decode",))
    launches_per_step = 3 + (1 if nsplit > 1 else 0)

    def timed(gs, k_steps, w_steps):
        with torch.cuda.stream(stream):
            for k in range(w_steps):
                gs[k % NBUF].replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for k in range(k_steps):
                gs[k % NBUF].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        if world > 1:
            t = torch.tensor([ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    gpu_id = str(local) if uuid is None else (str(uuid) if str(uuid).startswith("GPU-") else "GPU-" + str(uuid))
    with ClockSampler(gpu_id) as clk:
        total_ms = timed(graphs, args.steps, args.warmup)
    dec_steps = max(args.steps, 500)
    dec_ms = timed(dgraphs, dec_steps, max(3, args.warmup // 4))
    b2b_reps = max(dec_steps // NBUF, 100)
    b2b_ms = timed([rot] * NBUF, b2b_reps, 3) / (b2b_reps * NBUF)
    dec_b2b_ms = timed([drot] * NBUF, b2b_reps, 3) / (b2b_reps * NBUF)

    def per_call(gs, n):
        """Per-replay durations (an event pair around each replay): median, p10, p90."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for k in range(n):
                gs[k % NBUF].replay()
                ev[k + 1].record(stream)
        torch.cuda.synchronize()
        return distribution_us([ev[k].elapsed_time(ev[k + 1]) * 1e-3 for k in range(n)])

    step_dist = per_call(graphs, 300)
    dec_dist = per_call(dgraphs, 300)
    assert da.check_errors(stream) == 0

    ms_per_step = total_ms / args.steps
    value = total_ms * 1e3 / (args.steps * world)  # us per call over the whole job

    # end to end through the public API: every step copies its queries and lengths in from
    # pinned host memory and its outputs (out, LSE) back. The copies run on their own streams,
    # ordered by events, so step k+1's inputs upload while step k computes and step k's
    # outputs download while step k+1 computes, as a serving loop overlaps them; each
    # input set's buffers are reused only after the step that last used them is done.
    # a fixed step count, independent of --steps: long enough that the pipeline fill and
    # the first calls' host set-up do not dominate the per-step figure
    e2e_steps = E2E_STEPS
    h2d_stream = torch.cuda.Stream(device=dev)  # uploads and downloads on their own streams:
    d2h_stream = torch.cuda.Stream(device=dev)  # the two directions use separate copy engines
    hq_nope = [s_.q_nope.cpu().pin_memory() for s_ in sets]
    hq_pe = [s_.q_pe.cpu().pin_memory() for s_ in sets]
    hsl = torch.tensor(seqlens, dtype=torch.int32).pin_memory()
    sls = [torch.empty_like(sl) for _ in range(NBUF)]
    hout = [torch.empty((wl.b, wl.heads, wl.s, wl.d), dtype=torch.bfloat16).pin_memory() for _ in range(NBUF)]
    hlse = [torch.empty((wl.b, wl.heads, wl.s), dtype=torch.float32).pin_memory() for _ in range(NBUF)]
    ev_in = [torch.cuda.Event() for _ in range(NBUF)]
    ev_done = [torch.cuda.Event() for _ in range(NBUF)]
    ev_out = [torch.cuda.Event() for _ in range(NBUF)]
    used = [False] * NBUF

    def upload(k):
        r = k % NBUF
        if used[r]:
            h2d_stream.wait_event(ev_done[r])  # the step that last read set r has finished
        with torch.cuda.stream(h2d_stream):
            sets[r].q_nope.copy_(hq_nope[r], non_blocking=True)
            sets[r].q_pe.copy_(hq_pe[r], non_blocking=True)
            sls[r].copy_(hsl, non_blocking=True)
        ev_in[r].record(h2d_stream)

    # the attention step of each input set captured once from the same public API calls, as
    # a serving loop captures its decode step; replayed every step (the copies stay eager)
    step_graphs = []
    with torch.cuda.stream(stream):
        for r in range(NBUF):
            step(r, seq=sls[r])
    torch.cuda.synchronize()
    for r in range(NBUF):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(r, seq=sls[r])
        step_graphs.append(g)
    use_graph = [True]

    def compute(k):
        r = k % NBUF
        stream.wait_event(ev_in[r])
        if used[r]:
            stream.wait_event(ev_out[r])  # set r's outputs of the earlier step are downloaded
        with torch.cuda.stream(stream):
            if use_graph[0]:
                step_graphs[r].replay()
            else:
                step(r, seq=sls[r])
        ev_done[r].record(stream)
        used[r] = True

    def download(k):
        r = k % NBUF
        d2h_stream.wait_event(ev_done[r])
        with torch.cuda.stream(d2h_stream):
            hout[r].copy_(outs[r]["out"], non_blocking=True)
            hlse[r].copy_(outs[r]["lse"], non_blocking=True)
        ev_out[r].record(d2h_stream)

    def e2e_run(n):
        upload(0)
        for k in range(n):
            compute(k)
            if k + 1 < n:
                upload(k + 1)
            download(k)

    def e2e_timed(graphed):
        use_graph[0] = graphed
        e2e_run(5)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(h2d_stream)  # the first upload is the first timed operation
        th0 = time.perf_counter()
        e2e_run(e2e_steps)
        host = time.perf_counter() - th0  # host time to enqueue every step (API calls and copies)
        e1.record(d2h_stream)  # after the last download
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        if world > 1:
            t = torch.tensor([ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms = float(t.item())
        return ms, host

    eager_ms, eager_host_s = e2e_timed(False)

    # The whole pipelined step as one graph per rotation phase: step k uploads input set
    # k+1 (h2d stream), computes set k (compute stream) and downloads set k-1's outputs
    # (d2h stream), joined at the end; every replay copies the pinned host buffers anew.
    # Set k was uploaded by step k-1 and set k-1 computed by it (replays on one stream run
    # in order); set k+1 was last read by step k-2 and downloaded by step k-1.
    def capture_phase(r):
        nxt, prv = (r + 1) % NBUF, (r - 1) % NBUF
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fork = torch.cuda.Event()
            fork.record(stream)
            h2d_stream.wait_event(fork)
            d2h_stream.wait_event(fork)
            with torch.cuda.stream(h2d_stream):
                sets[nxt].q_nope.copy_(hq_nope[nxt], non_blocking=True)
                sets[nxt].q_pe.copy_(hq_pe[nxt], non_blocking=True)
                sls[nxt].copy_(hsl, non_blocking=True)
            step(r, seq=sls[r])
            with torch.cuda.stream(d2h_stream):
                hout[prv].copy_(outs[prv]["out"], non_blocking=True)
                hlse[prv].copy_(outs[prv]["lse"], non_blocking=True)
            j1, j2 = torch.cuda.Event(), torch.cuda.Event()
            j1.record(h2d_stream)
            j2.record(d2h_stream)
            stream.wait_event(j1)
            stream.wait_event(j2)
        return g

    torch.cuda.synchronize()
    phase_graphs = [capture_phase(r) for r in range(NBUF)]

    def piped_run(n):
        with torch.cuda.stream(stream):
            sets[0].q_nope.copy_(hq_nope[0], non_blocking=True)  # step 0's inputs
            sets[0].q_pe.copy_(hq_pe[0], non_blocking=True)
            sls[0].copy_(hsl, non_blocking=True)
            for k in range(n):
                phase_graphs[k % NBUF].replay()
            last = (n - 1) % NBUF  # the last step's outputs
            hout[last].copy_(outs[last]["out"], non_blocking=True)
            hlse[last].copy_(outs[last]["lse"], non_blocking=True)

    piped_run(6)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    th0 = time.perf_counter()
    piped_run(e2e_steps)
    host_s = time.perf_counter() - th0
    p1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = p0.elapsed_time(p1)
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    graph_step_ms, graph_step_host_s = e2e_timed(True)
    h2d = sum(t.numel() * t.element_size() for t in (hq_nope[0], hq_pe[0], hsl))
    d2h = hout[0].numel() * hout[0].element_size() + hlse[0].numel() * hlse[0].element_size()

    f_core, b_core, f_proj, b_proj = cost_numbers(wl)
    hbm, tfl, tfl_sus, peak_src = peaks()
    dec_s = dec_ms / dec_steps * 1e-3
    t_roof = max(f_core / (tfl * 1e12), b_core / (hbm * 1e9))
    bound = "hbm" if b_core / (hbm * 1e9) >= f_core / (tfl * 1e12) else "tensor"
    if bound == "hbm":
        achieved, peak, unit = b_core / dec_s / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = f_core / dec_s / 1e12, tfl, "TFLOP/s"
    step_s = ms_per_step * 1e-3
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "global_batch": wl.b * world, "seq_len": wl.t, "new_tokens": wl.s,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"{NBUF} rotating input sets of {sum(t.numel() * t.element_size() for t in (sets[0].z, sets[0].k_pe, sets[0].w_uk, sets[0].w_uv, sets[0].q_nope, sets[0].q_pe)) / 1e6:.0f} MB each (> 126 MB L2)",
                   "num_splits": nsplit, "graphs": "one CUDA graph per input set"},
        "step_breakdown": {
            "pipeline_us": ms_per_step * 1e3,
            "latent_call_us": dec_s * 1e6,
            "back_to_back": {"pipeline_us": b2b_ms * 1e3, "latent_call_us": dec_b2b_ms * 1e3,
                             "graphs": f"one graph of {NBUF} steps (one per input set), replayed {b2b_reps} times"},
            "pipeline_per_call": step_dist,
            "latent_per_call": dec_dist,
            "pipeline_tflops": (f_core + 2 * f_proj) / step_s / 1e12,
            "pipeline_hbm_gbs": (b_core + 2 * b_proj) / step_s / 1e9,
            "latent_tflops": f_core / dec_s / 1e12,
            "latent_hbm_gbs": b_core / dec_s / 1e9,
            "latent_roofline_us": t_roof * 1e6,
            "latent_frac_of_roofline": t_roof / dec_s,
            "latent_algorithmic": {"flops": f_core, "bytes": b_core, "ai": f_core / b_core},
        },
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": traffic_record(), "kernel": "mla_decode call (tcgen05 CTA-pair latent kernel + combine)",
                     "peak_source": peak_src,
                     "note": "frac of measured peak; the call's roofline time is max(FLOPs/tensor peak, bytes/HBM peak)"},
        "e2e": {"value": e2e_ms * 1e3 / (e2e_steps * world), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "host_enqueue_us_per_step": host_s * 1e6 / e2e_steps,
                "step": "the public API calls and the step's copies (upload of the next input set, download "
                        "of the previous outputs, on their own streams) captured once per rotation phase in a "
                        "CUDA graph and replayed each step; every replay copies the pinned host buffers",
                "graphed_compute_eager_copies_us": graph_step_ms * 1e3 / (e2e_steps * world),
                "eager_api_us": eager_ms * 1e3 / (e2e_steps * world),
                "eager_api_host_enqueue_us_per_step": eager_host_s * 1e6 / e2e_steps,
                "copies": "every step's inputs in and outputs out, overlapping the neighbouring steps' compute "
                          "(three input/output sets)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0 and not args.no_extras:
        line["extras"] = extras(dev, stream, hbm, tfl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile(args):
    """A few calls of one op on one input set, for ncu (no timing, no JSON)."""
    import torch

    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.profile == "mla_expanded_s128_b4":
        # the expanded form's attention at s = 128 (tensor-core grouped-head kernel) on 4
        # sequences of 4096 + 128 keys, 128 heads (decompressed cache 1.4 GB, > L2)
        b, h, s, L = 4, 128, 128, 4096 + 128
        x = W.make_mla(b, h, 128, 512, 64, s, [L] * b, capacity=L, seed=5, device=dev)
        kf, vf = da.mla_decompress_kv(x.z, x.k_pe, x.w_uk, x.w_uv)
        q = torch.cat([x.q_nope, x.q_pe], dim=-1).contiguous()
        sl = torch.tensor([L] * b, dtype=torch.int32, device=dev)
        for _ in range(args.warmup + args.steps):
            da.gqa_decode_dv(q, kf, vf, sl, scale=x.scale, max_seqlen=L)
        torch.cuda.synchronize()
        assert da.check_errors() == 0
        print(f"profiled {args.profile}: {args.warmup + args.steps} calls, splits {da.last_num_splits()}", flush=True)
        return 0
    name = args.profile
    if name.endswith("_tc"):  # grouped-head workload pinned to the tensor-core kernel
        da.set_grouped_kernel(2)
        name = name[:-3]
    elif name.endswith("_split"):  # grouped-head workload pinned to the split-KV kernels
        da.set_grouped_kernel(1)
        name = name[:-6]
    fp8 = name.endswith("_fp8")  # grouped-head workload over an FP8 cache
    wl = W.WORKLOADS[name[:-4] if fp8 else name]
    seqlens = wl.seqlens()
    L = max(seqlens)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=dev)
    if wl.kind == "gqa" and fp8:
        q, c, ks, vs = W.make_gqa_fp8(wl.b, wl.heads, wl.hkv, wl.d, wl.s, seqlens, paged=wl.paged, seed=wl.seed,
                                      device=dev)

        def fn():
            da.gqa_decode_fp8(q, c.k, c.v, sl, k_scale=ks, v_scale=vs, max_seqlen=L,
                              block_table=c.block_table if wl.paged else None)
    elif wl.kind == "gqa":
        q, c = W.make_gqa(wl.b, wl.heads, wl.hkv, wl.d, wl.s, seqlens, paged=wl.paged, seed=wl.seed, device=dev)

        def fn():
            da.gqa_decode(q, c.k, c.v, sl, max_seqlen=L, block_table=c.block_table if wl.paged else None)
    else:
        # one pipeline step per call: absorb, latent attention (+ combine), W_uv
        x = W.make_mla(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, seqlens, seed=wl.seed, device=dev)

        def fn():
            qz = da.mla_absorb_q(x.q_nope, x.w_uk, sl)
            o_lat, _ = da.mla_decode(qz, x.q_pe, x.z, x.k_pe, sl, scale=x.scale, max_seqlen=L)
            da.mla_out_proj(o_lat, x.w_uv, sl)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    print(f"profiled {args.profile}: {args.warmup + args.steps} calls, splits {da.last_num_splits()}", flush=True)
    return 0


def extras(dev, stream, hbm, tfl):
    """Side measurements (not the headline): the grouped-head workloads and the
    MLA s-sweep, each as us per call with its roofline fraction."""
    import torch

    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W
    from oracle import cost

    res = {}

    def time_calls(fns, n=100, w=6):
        """Seconds per call: one CUDA graph per input set (captured after an eager
        warm-up call), replayed round-robin, an event pair around every replay on
        the stream. Returns the mean; the per-call median, p10 and p90, and the mean
        per call with all input sets' calls back to back in one graph, are kept in
        `dist` for the caller's record."""
        with torch.cuda.stream(stream):
            for f in fns:
                f()
        torch.cuda.synchronize()
        graphs = []
        for f in fns:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                f()
            graphs.append(g)
        with torch.cuda.stream(stream):
            for i in range(w):
                graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(n):
                graphs[i % len(graphs)].replay()
                ev[i + 1].record(stream)
        torch.cuda.synchronize()
        per = [ev[i].elapsed_time(ev[i + 1]) * 1e-3 for i in range(n)]
        dist.clear()
        dist.update(distribution_us(per))
        # the same calls back to back in one graph (one call per input set), so that
        # programmatic dependent launch overlaps consecutive calls as inside a larger graph
        g_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_all, stream=stream):
            for f in fns:
                f()
        reps = max(2, n // len(fns))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g_all.replay()
            e0.record(stream)
            for _ in range(reps):
                g_all.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        dist["back_to_back_us"] = e0.elapsed_time(e1) * 1e3 / (reps * len(fns))
        del g_all
        return ev[0].elapsed_time(ev[n]) / n * 1e-3

    dist = {}
    for name in ("gqa_64_8", "gqa_paged_hkv24", "gqa_paged_hkv4", "gqa_paged_hkv1"):
        wl = W.WORKLOADS[name]
        seqlens = wl.seqlens()
        nb = 2
        qs = []
        for r in range(nb):
            q, c = W.make_gqa(wl.b, wl.heads, wl.hkv, wl.d, wl.s, seqlens, paged=wl.paged, seed=wl.seed + r, device=dev)
            qs.append((q, c))
        sl = torch.tensor(seqlens, dtype=torch.int32, device=dev)
        outs = [torch.empty_like(q) for q, _ in qs]
        lses = [torch.empty(q.shape[:3], dtype=torch.float32, device=dev) for q, _ in qs]
        wsb = da.ops.load().gqa_decode_workspace_size(wl.b, wl.s, wl.heads, wl.hkv, wl.d, max(seqlens))
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        def call(r):
            def f():
                q, c = qs[r]
                da.gqa_decode(q, c.k, c.v, sl, max_seqlen=max(seqlens),
                              block_table=c.block_table if wl.paged else None, out=outs[r], lse=lses[r],
                              workspace=ws, stream=stream)
            return f

        t = time_calls([call(r) for r in range(nb)])
        by = cost.gqa_bytes_exact(wl.heads, wl.hkv, wl.d, seqlens, wl.s)
        fl = cost.gqa_flops_exact(wl.heads, wl.d, seqlens, wl.s)
        res[name] = {"us": t * 1e6, **dist, "hbm_gbs": by / t / 1e9, "frac_hbm": by / t / 1e9 / hbm,
                     "tflops": fl / t / 1e12, "bytes": by, "num_splits": da.last_num_splits(),
                     "l2": f"{nb} rotating caches of {by / 1e6:.0f} MB", "timing": "CUDA graph replays"}
        del qs, ws
        # the same workload over an FP8 (E4M3) cache: half the cache bytes
        f8 = [W.make_gqa_fp8(wl.b, wl.heads, wl.hkv, wl.d, wl.s, seqlens, paged=wl.paged, seed=wl.seed + r, device=dev)
              for r in range(nb)]
        wsb = da.ops.load().gqa_decode_fp8_workspace_size(wl.b, wl.s, wl.heads, wl.hkv, wl.d, max(seqlens))
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)

        def call8(r):
            def f():
                q, c, ks, vs = f8[r]
                da.gqa_decode_fp8(q, c.k, c.v, sl, k_scale=ks, v_scale=vs, max_seqlen=max(seqlens),
                                  block_table=c.block_table if wl.paged else None, out=outs[r], lse=lses[r],
                                  workspace=ws, stream=stream)
            return f

        t8 = time_calls([call8(r) for r in range(nb)])
        by8 = cost.gqa_fp8_bytes_exact(wl.heads, wl.hkv, wl.d, seqlens, wl.s)
        res[name + "_fp8"] = {"us": t8 * 1e6, **dist, "hbm_gbs": by8 / t8 / 1e9, "frac_hbm": by8 / t8 / 1e9 / hbm,
                              "bytes": by8, "speedup_over_bf16": t / t8, "num_splits": da.last_num_splits(),
                              "cache": "E4M3 bytes, per-tensor scales"}
        del f8, outs, lses, ws
        torch.cuda.empty_cache()

    # the two projection GEMMs of the headline pipeline, each alone
    wl = W.WORKLOADS["mla_dsv3"]
    seqlens = wl.seqlens()
    inp = [W.make_mla(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, seqlens, seed=wl.seed + r, device=dev) for r in range(3)]
    sl = torch.tensor(seqlens, dtype=torch.int32, device=dev)
    qzs = [torch.empty((wl.b, wl.heads, wl.s, wl.k), dtype=torch.bfloat16, device=dev) for _ in inp]
    outs = [torch.empty((wl.b, wl.heads, wl.s, wl.d), dtype=torch.bfloat16, device=dev) for _ in inp]
    olats = [torch.randn((wl.b, wl.heads, wl.s, wl.k), device=dev).to(torch.bfloat16) for _ in inp]
    pb = cost.proj_bytes(wl.b, wl.heads, wl.s, wl.d, wl.k)
    t_abs = time_calls([(lambda r=r: da.mla_absorb_q(inp[r].q_nope, inp[r].w_uk, sl, out=qzs[r], stream=stream))
                        for r in range(3)], n=300)
    res["proj_absorb"] = {"us": t_abs * 1e6, **dist, "hbm_gbs": pb / t_abs / 1e9, "frac_hbm": pb / t_abs / 1e9 / hbm,
                          "bytes": pb, "l2": "3 rotating weight sets of 16.8 MB"}
    t_out = time_calls([(lambda r=r: da.mla_out_proj(olats[r], inp[r].w_uv, sl, out=outs[r], stream=stream))
                        for r in range(3)], n=300)
    res["proj_out"] = {"us": t_out * 1e6, **dist, "hbm_gbs": pb / t_out / 1e9, "frac_hbm": pb / t_out / 1e9 / hbm,
                       "bytes": pb, "l2": "3 rotating weight sets of 16.8 MB"}
    del inp, qzs, outs, olats
    torch.cuda.empty_cache()

    for s in SWEEP_S:
        wl = W.WORKLOADS["mla_dsv3"] if s == 1 else W.WORKLOADS[f"mla_mtp_s{s}"]
        seqlens = wl.seqlens()
        inp = [W.make_mla(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, seqlens, seed=wl.seed + r, device=dev)
               for r in range(2)]
        sl = torch.tensor(seqlens, dtype=torch.int32, device=dev)
        qzs = [da.mla_absorb_q(x.q_nope, x.w_uk, sl) for x in inp]
        o = [torch.empty_like(q) for q in qzs]
        lse = [torch.empty(q.shape[:3], dtype=torch.float32, device=dev) for q in qzs]
        wsb = da.ops.load().mla_decode_workspace_size(wl.b, wl.s, wl.heads, wl.k, max(seqlens))
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        def call(r):
            def f():
                da.mla_decode(qzs[r], inp[r].q_pe, inp[r].z, inp[r].k_pe, sl, scale=inp[r].scale,
                              max_seqlen=max(seqlens), out=o[r], lse=lse[r], workspace=ws, stream=stream)
            return f

        t = time_calls([call(r) for r in range(2)], n=60 if s <= 4 else (20 if s <= 32 else 6))
        fl = cost.mla_flops_exact(wl.heads, wl.k, wl.p, seqlens, wl.s)
        by = cost.mla_bytes_exact(wl.heads, wl.k, wl.p, seqlens, wl.s)
        troof = max(fl / (tfl * 1e12), by / (hbm * 1e9))
        res[f"mla_s{s}"] = {"us": t * 1e6, **dist, "tflops": fl / t / 1e12, "hbm_gbs": by / t / 1e9, "ai": fl / by,
                            "roofline_us": troof * 1e6, "frac_roofline": troof / t,
                            "bound": "tensor" if fl / (tfl * 1e12) > by / (hbm * 1e9) else "hbm",
                            "num_splits": da.last_num_splits()}
        del inp, qzs, o, lse, ws
        torch.cuda.empty_cache()

    # expanded form ("Mla Analysis", Cost Models - FlashAttention; Regime Selection):
    # the latent cache of 32 sequences of 4096 + 128 keys decompressed once into per-head
    # keys [nope || rope] (192 values) and values (128) for all 128 heads (11.1 GB), then
    # grouped-head decode with Hkv = Hq = 128 at each s, beside the absorbed call above
    b, h, d, k, p, smax, t0 = 32, 128, 128, 512, 64, max(SWEEP_S), 4096
    cap = t0 + smax
    x = W.make_mla(b, h, d, k, p, smax, [cap] * b, capacity=cap, seed=5, device=dev)
    kf = torch.empty((b, cap, h, d + p), dtype=torch.bfloat16, device=dev)
    vf = torch.empty((b, cap, h, d), dtype=torch.bfloat16, device=dev)
    t_dec = time_calls([lambda: da.mla_decompress_kv(x.z, x.k_pe, x.w_uk, x.w_uv, k_out=kf, v_out=vf, stream=stream)],
                       n=5, w=1)
    rows = b * cap
    dfl, dby = cost.decompress_flops(rows, h, d, k), cost.decompress_bytes(rows, h, d, k, p)
    res["mla_decompress"] = {"us": t_dec * 1e6, **dist, "rows": rows, "tflops": dfl / t_dec / 1e12,
                             "frac_tensor": dfl / t_dec / 1e12 / tfl, "hbm_gbs": dby / t_dec / 1e9,
                             "bound": "tensor" if dfl / (tfl * 1e12) > dby / (hbm * 1e9) else "hbm",
                             "note": "once per cached token, not per decode step"}
    q_all = torch.cat([x.q_nope, x.q_pe], dim=-1).contiguous()  # the expanded query [q_nope || q_pe]
    crossover = {}
    for s in SWEEP_S:
        L = t0 + (s if s > 1 else 0)  # the latent sweep's lengths
        seqlens = [L] * b
        sl = torch.tensor(seqlens, dtype=torch.int32, device=dev)
        q = q_all[:, :, :s].contiguous()
        o = torch.empty((b, h, s, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((b, h, s), dtype=torch.float32, device=dev)
        wsb = da.ops.load().gqa_decode_dv_workspace_size(b, s, h, h, d + p, d, L)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        t = time_calls([lambda: da.gqa_decode_dv(q, kf, vf, sl, scale=x.scale, max_seqlen=L, out=o, lse=lse,
                                                 workspace=ws, stream=stream)], n=10 if s <= 8 else 4, w=1)
        fl = cost.fa_flops_exact(h, d, p, seqlens, s)
        by = cost.fa_bytes_exact(h, d, p, seqlens, s)
        troof = max(fl / (tfl * 1e12), by / (hbm * 1e9))
        res[f"mla_expanded_s{s}"] = {"us": t * 1e6, **dist, "tflops": fl / t / 1e12, "hbm_gbs": by / t / 1e9,
                                     "ai": fl / by, "roofline_us": troof * 1e6, "frac_roofline": troof / t,
                                     "bound": "tensor" if fl / (tfl * 1e12) > by / (hbm * 1e9) else "hbm",
                                     "num_splits": da.last_num_splits(), "bytes": by}
        crossover[f"s{s}"] = {"absorbed_us": res[f"mla_s{s}"]["us"], "expanded_us": t * 1e6,
                              "expanded_over_absorbed": t * 1e6 / res[f"mla_s{s}"]["us"]}
        del o, lse, ws
    res["expanded_vs_absorbed"] = crossover
    del x, kf, vf, q_all
    torch.cuda.empty_cache()

    # hybrid form ("Mla Analysis", MLAvar6+ Design): the n most recent keys decompressed,
    # the o = L - n older ones latent, merged by LSE; the whole step (absorb, latent part,
    # W_uv, expanded part, merge) against the absorbed pipeline (absorb, latent, W_uv) at
    # the same s, and against the pages' cost model of the split
    for s in (1, 32):
        L = t0 + (s if s > 1 else 0)
        seqlens = [L] * b
        x = W.make_mla(b, h, d, k, p, s, seqlens, capacity=L, seed=7, device=dev)
        sl = torch.tensor(seqlens, dtype=torch.int32, device=dev)
        q_full = torch.cat([x.q_nope, x.q_pe], dim=-1).contiguous()
        absorbed = time_calls([lambda: da.mla_forward(x.q_nope, x.q_pe, x.z, x.k_pe, x.w_uk, x.w_uv, sl,
                                                      scale=x.scale, max_seqlen=L, stream=stream)], n=20, w=2)
        res[f"mla_absorbed_pipeline_s{s}"] = {"us": absorbed * 1e6, **dist}
        for n in (s, 256, 1024):
            kr, vr = da.mla_decompress_kv(x.z[:, L - n:].contiguous(), x.k_pe[:, L - n:].contiguous(), x.w_uk, x.w_uv)
            sl_old = torch.full((b,), L - n, dtype=torch.int32, device=dev)
            sl_rec = torch.full((b,), n, dtype=torch.int32, device=dev)
            t = time_calls([lambda: da.mla_split_forward(x.q_nope, x.q_pe, q_full, x.z, x.k_pe, kr, vr, x.w_uk, x.w_uv,
                                                         sl_old, sl_rec, scale=x.scale, max_old=L - n, max_recent=n,
                                                         stream=stream)], n=20, w=2)
            fl = cost.split_latent_flops(b, h, s, L - n, n, d, p, k)
            by = cost.split_latent_bytes(b, h, s, L - n, n, d, p, k)
            troof = max(fl / (tfl * 1e12), by / (hbm * 1e9))
            res[f"mla_split_s{s}_n{n}"] = {"us": t * 1e6, **dist, "old": L - n, "recent": n,
                                           "model_flops": fl, "model_bytes": by, "roofline_us": troof * 1e6,
                                           "frac_roofline": troof / t, "over_absorbed_pipeline": t / absorbed,
                                           "note": "cost model counts the attention core only, as the pages do"}
            del kr, vr
        del x, q_full
        torch.cuda.empty_cache()
    return res


# new tokens per sequence of the absorbed / expanded sweep: decode (1), speculative (2 .. 32)
# and the start of the prefill-sized regime, where the two forms cross
SWEEP_S = (1, 2, 4, 8, 16, 32, 64, 128)


def distribution_us(per_call_s):
    """Median, p10 and p90 of per-call times (seconds in, microseconds out)."""
    import numpy as np

    a = np.asarray(per_call_s, dtype=np.float64) * 1e6
    return {"p10_us": float(np.percentile(a, 10)), "p50_us": float(np.percentile(a, 50)),
            "p90_us": float(np.percentile(a, 90)), "calls": int(a.size)}


if __name__ == "__main__":
    sys.exit(main())
