"""Benchmark of the EP dispatch/combine hot path on GB300.

One step = layout -> dispatch -> combine over one batch of the DeepSeek-V3-shaped
prefill workload (T=4096 tokens, H=7168 bf16, E=256 experts, top-8, R=32
virtual ranks = 8 nodes x 4), inputs resident in HBM. The expert between
dispatch and combine is the identity (combine reads the dispatch buffer), so
no harness work sits in the timed region. L2 is flushed between steps, outside
the timed events, by a 256 MiB write followed by a 256 MiB read: every step
starts with a cold L2 that holds only clean lines, so the write-back of the
flush itself is not charged to the step.

Prints ONE JSON line (rank 0): value = algorithmic HBM GB/s of the step
(whole job, summed over ranks), plus tokens/s, the roofline of the dominant
kernel, per-stage times for the other workloads (FP8 dispatch, restripe and
node dispatch, skewed routing), an end-to-end number through host buffers,
the CPU oracle as a baseline, and SM clocks sampled during the timed region.

--impl reference times the oracle (plain single-threaded C) on the host on
the same workload and prints the same line with "impl": "reference".

Multi-GPU (torchrun): each rank runs an independent replica of the workload on
its own GPU (token batches are independent; no collective on the data path);
timing is bracketed by barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "dispatch+combine HBM GB/s & tokens/s at T=4096,H=7168,E=256,k=8; % of HBM peak"
UNIT = "GB/s"
FLUSH_BYTES = 256 << 20
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_HBM_GBS = 6800.0
STAGE_ITERATIONS = 50  # timed replays per extra stage (median, p10 and p90 reported)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------------- byte accounting

def step_bytes(T, H, k, E, R, N, pairs, row_bytes_out=None):
    """Algorithmic HBM bytes of each stage (what the method must move).

    pairs = number of (token, rank) deliveries = sum of tokens_per_rank.
    layout:   read topk_idx T*k*8; write is_token_in_rank T*R, slot 4*T*R,
              is_token_in_node T*N, counts 4*(E+R+N)
    dispatch: read x T*2H (+ slot row 4*T*R, topk 12*T*k); write per delivery the row
              plus src index 4 + topk ids/weights 8k
    combine:  read one row per delivery + slot 4*T*R; write T*2H
    """
    row = 2 * H if row_bytes_out is None else row_bytes_out
    layout = T * k * 8 + T * R * 5 + T * N + 4 * (E + R + N)
    dispatch = T * 2 * H + 4 * T * R + 12 * T * k + pairs * (row + 4 + 8 * k)
    combine = pairs * 2 * H + 4 * T * R + T * 2 * H
    return {"layout": layout, "dispatch": dispatch, "combine": combine}


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(name):
    """Hash of a kernel's translation unit and every shared internal header."""
    csrc = os.path.join(ROOT, "combine_ep_get_05_gb300", "csrc")
    h = hashlib.sha256()
    for p in [os.path.join(csrc, name)] + sorted(os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith(".cuh")):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, source):
    """dram read+write bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f)
        e = t.get(kernel)
        if e and e.get("source_sha") == source_digest(source):
            return e.get("dram_bytes_per_launch_full"), e.get("note")
    except Exception:
        pass
    return None, None


# --------------------------------------------------------------------------- L2 flush

class L2Flush:
    """Evict L2 (129 MB on GB300) between timed launches: write one 256 MiB buffer, then read
    another, so L2 is cold and holds no dirty lines whose write-back a timed kernel would pay."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            self.uuid = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.uuid and self.uuid.replace("GPU-", "") not in parts[0]:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        try:
            sm = [float(r[1]) for r in rows]
            mx = max(float(r[2]) for r in rows)
        except ValueError:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, value):
    if world == 1:
        return value
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- oracle (CPU) timing

@contextlib.contextmanager
def one_core():
    """Pin the calling thread (the oracle runs single-threaded in it) to one host core while
    it is timed, and restore its affinity afterwards. Yields the core's index, or None where
    the platform has no affinity call."""
    try:
        old = os.sched_getaffinity(0)
    except (AttributeError, OSError):
        yield None
        return
    core = max(old)  # the highest allowed core: away from core 0's interrupt load
    try:
        os.sched_setaffinity(0, {core})
        yield core
    finally:
        os.sched_setaffinity(0, old)


def oracle_step_seconds(w, max_tokens, tokens):
    """One oracle step (layout -> dispatch -> identity combine) on the first `tokens` tokens."""
    import oracle

    topk = np.ascontiguousarray(w.topk_idx[:tokens])
    x = np.ascontiguousarray(w.x[:tokens])
    tw = np.ascontiguousarray(w.topk_w[:tokens])
    t0 = time.perf_counter()
    L = oracle.layout(topk, w.E, w.R, w.ranks_per_node)
    D = oracle.dispatch(x, topk, tw, L["slot"], w.E, w.R, max_tokens)
    oracle.combine(D["recv_x"], L["slot"], max_tokens)
    dt = time.perf_counter() - t0
    return dt, int(L["tokens_per_rank"].sum())


def cpu_baseline(w, budget_s=12.0, tokens=None):
    import oracle

    oracle.build()
    tokens = tokens or w.T
    N = w.num_nodes
    spent, steps, pairs = 0.0, 0, 0
    with one_core() as core:
        while spent < budget_s and steps < 50:
            dt, pairs = oracle_step_seconds(w, tokens, tokens)
            spent += dt
            steps += 1
    b = step_bytes(tokens, w.H, w.k, w.E, w.R, N, pairs)
    total = sum(b.values())
    return {
        "value": round(total / (spent / steps) / 1e9, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
        "host": host_cpu(), "pinned_core": core,
        "sample": f"{steps} oracle steps (layout+dispatch+identity combine) on {tokens} of the {w.T} tokens, "
                  f"single-threaded C, {spent:.1f} s",
        "tokens_per_s": round(tokens / (spent / steps), 1),
    }


def host_cpu():
    """The host's core count and CPU model, as /proc/cpuinfo (or the platform) gives them."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model Name", "cpu model"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key:
                    model = line.split(":", 1)[1].strip()
                    break
            if model:
                break
        if model is None:  # Arm: implementer / part numbers
            imp = [line.split(":")[1].strip() for line in info.splitlines() if line.startswith("CPU implementer")]
            part = [line.split(":")[1].strip() for line in info.splitlines() if line.startswith("CPU part")]
            if imp and part:
                known = {("0x41", "0xd4f"): "Arm Neoverse V2", ("0x41", "0xd40"): "Arm Neoverse V1",
                         ("0x41", "0xd0c"): "Arm Neoverse N1", ("0x41", "0xd49"): "Arm Neoverse N2"}
                model = known.get((imp[0].lower(), part[0].lower()), f"Arm implementer {imp[0]} part {part[0]}")
    except OSError:
        pass
    import platform

    return {"nproc": os.cpu_count(), "model": model or platform.processor() or platform.machine()}


def oracle_stage_baselines():
    """The oracle (single-threaded C, one host core) on a bounded sample of each extra stage's
    workload, in the same unit (algorithmic GB/s by the same formulas, scaled to the sample)."""
    with one_core() as core:
        res = _oracle_stage_baselines()
    res["pinned_core"] = core
    return res


def _oracle_stage_baselines():
    import oracle

    oracle.build()
    res = {"host": host_cpu(), "cores_used": 1}

    def timed(fn, min_s=0.25):
        """Mean seconds per call over as many calls as fill min_s (at least one)."""
        n, spent, out = 0, 0.0, None
        while n == 0 or spent < min_s:
            t0 = time.perf_counter()
            out = fn()
            spent += time.perf_counter() - t0
            n += 1
        return spent / n, out

    def entry(bytes_, sec, sample):
        return {"gbs": round(bytes_ / sec / 1e9, 3), "s": round(sec, 3), "sample": sample}

    S = 512  # tokens per sample for the large-row stages
    w = workloads.make("dsv3_fp8")
    x, ti, tw = w.x[:S], w.topk_idx[:S], w.topk_w[:S]
    L = oracle.layout(ti, w.E, w.R, w.ranks_per_node)
    pairs = int(L["tokens_per_rank"].sum())
    sec, D = timed(lambda: oracle.dispatch(x, ti, tw, L["slot"], w.E, w.R, S, fp8=True))
    row = w.H + 4 * (w.H // 128)
    res["dsv3_fp8_dispatch"] = entry(step_bytes(S, w.H, w.k, w.E, w.R, w.num_nodes, pairs, row)["dispatch"], sec,
                                     f"first {S} of {w.T} tokens")
    sec, _ = timed(lambda: oracle.combine_fp8(D["recv_x"], D["recv_scales"], L["slot"], S))
    res["dsv3_fp8_combine"] = entry(pairs * row + 4 * S * w.R + 2 * S * w.H, sec, f"first {S} of {w.T} tokens")
    sec, _ = timed(lambda: oracle.combine_weights(D["recv_topk_w"], L["slot"], S))
    res["dsv3_combine_weights"] = entry(pairs * 4 * w.k + 4 * S * w.R + 4 * S * w.k, sec, f"first {S} of {w.T} tokens")
    del D

    w = workloads.make("restripe")
    Nn, P = w.num_nodes, w.prob.shape[2]
    sec, st = timed(lambda: oracle.restripe_prob(w.prob, w.T))
    res["restripe_prob"] = entry(2 * w.T * Nn * P * 4, sec, f"all {w.T} tokens")
    L = oracle.layout(w.topk_idx[:S], w.E, w.R, w.ranks_per_node)
    stS = np.ascontiguousarray(st[:, :S])
    routed = int(L["is_token_in_node"].sum())
    for name, dense, dests in (("node_dispatch_sparse", False, routed), ("node_dispatch_dense", True, Nn * S)):
        sec, _ = timed(lambda dense=dense: oracle.dispatch_nodes(w.x[:S], stS, L["is_token_in_node"], S,
                                                                 w.chunk_tokens, dense=dense))
        b = S * 2 * w.H + dests * (2 * w.H + 2 * P * 4) + (0 if dense else S * Nn)
        res[name] = entry(b, sec, f"first {S} of {w.T} tokens (2 chunks)")
    del st, stS

    w = workloads.make("dsv3")
    T, H, k, E, R = w.T, w.H, w.k, w.E, w.R
    sec, EL = timed(lambda: oracle.expert_layout(w.topk_idx, E))
    res["expert_layout"] = entry(T * k * 12 + 4 * (E + 1), sec, f"all {T} tokens")
    ti, x, tw = w.topk_idx[:S], w.x[:S], w.topk_w[:S]
    ELs = oracle.expert_layout(ti, E)
    Mp = int(oracle.rows_per_rank(ELs["expert_offsets"], E, R).max())
    entries = int(ELs["expert_offsets"][E])
    sec, PX = timed(lambda: oracle.dispatch_permuted(x, ti, tw, ELs, E, R, Mp))
    res["dispatch_permuted"] = entry(S * 2 * H + S * k * 16 + entries * (2 * H + 8), sec, f"first {S} of {T} tokens")
    L = oracle.layout(ti, E, R, w.ranks_per_node)
    pairs = int(L["tokens_per_rank"].sum())
    D = oracle.dispatch(x, ti, tw, L["slot"], E, R, S)
    sec, _ = timed(lambda: oracle.permute_received(D, L["tokens_per_rank"], ELs, S, E, R, Mp))
    res["permute_received"] = entry(pairs * (2 * H + 4 + 8 * k) + S * k * 4 + entries * (2 * H + 8), sec,
                                    f"first {S} of {T} tokens")
    sec, _ = timed(lambda: oracle.combine_permuted(PX["perm_x"], ti, tw, ELs, E, R))
    res["combine_permuted_weighted"] = entry(entries * 2 * H + S * k * 16 + S * 2 * H, sec, f"first {S} of {T} tokens")
    sec, _ = timed(lambda: oracle.combine_send(PX["perm_x"], D, L["tokens_per_rank"], ELs, S, E, R))
    res["combine_send_weighted"] = entry(entries * 2 * H + pairs * (2 * H + 4 + 8 * k) + S * k * 4 + 4 * (E + 1), sec,
                                         f"first {S} of {T} tokens")
    del PX, D

    w = workloads.make("dsv3", T=128)
    sec, ELd = timed(lambda: oracle.expert_layout(w.topk_idx, E))
    Mp = int(oracle.rows_per_rank(ELd["expert_offsets"], E, R).max())
    entries = int(ELd["expert_offsets"][E])
    sec2, PX = timed(lambda: oracle.dispatch_permuted(w.x, w.topk_idx, w.topk_w, ELd, E, R, Mp))
    res["decode128_dispatch_permuted"] = entry(128 * 2 * H + 128 * k * 8 + 4 * (E + 1) + 128 * k * 4 +
                                               entries * (2 * H + 8), sec + sec2, "all 128 tokens")
    sec, _ = timed(lambda: oracle.combine_permuted(PX["perm_x"], w.topk_idx, w.topk_w, ELd, E, R))
    res["decode128_combine_weighted"] = entry(entries * 2 * H + 128 * k * 16 + 128 * 2 * H, sec, "all 128 tokens")
    del PX

    w = workloads.make("skewed")
    ti, x, tw = w.topk_idx[:S], w.x[:S], w.topk_w[:S]
    sec, L = timed(lambda: oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node))
    b = step_bytes(w.T, w.H, w.k, w.E, w.R, w.num_nodes, int(L["tokens_per_rank"].sum()))
    res["skewed_layout"] = entry(b["layout"], sec, f"all {w.T} tokens")
    L = oracle.layout(ti, w.E, w.R, w.ranks_per_node)
    pairs = int(L["tokens_per_rank"].sum())
    b = step_bytes(S, w.H, w.k, w.E, w.R, w.num_nodes, pairs)
    sec, D = timed(lambda: oracle.dispatch(x, ti, tw, L["slot"], w.E, w.R, S))
    res["skewed_dispatch"] = entry(b["dispatch"], sec, f"first {S} of {w.T} tokens")
    sec, _ = timed(lambda: oracle.combine(D["recv_x"], L["slot"], S))
    res["skewed_combine"] = entry(b["combine"], sec, f"first {S} of {w.T} tokens")
    del D

    w = workloads.make("tiny")
    sec, L = timed(lambda: oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node))
    sec2, D = timed(lambda: oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, w.R, w.T))
    sec3, _ = timed(lambda: oracle.combine(D["recv_x"], L["slot"], w.T))
    pairs = int(L["tokens_per_rank"].sum())
    res["tiny_step"] = entry(sum(step_bytes(w.T, w.H, w.k, w.E, w.R, w.num_nodes, pairs).values()), sec + sec2 + sec3,
                             f"all {w.T} tokens")
    return res


# --------------------------------------------------------------------------- GPU arm

def capture(fn, warm=2):
    """Capture fn (library launches on the current stream) into a CUDA graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def run_ours(args, world, rank):
    import combine_ep_get_05_gb300 as ep

    ep.build_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = workloads.make("dsv3")
    T, H, E, k, R, rpn = w.T, w.H, w.E, w.k, w.R, w.ranks_per_node
    N = w.num_nodes
    M = w.max_tokens
    x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(w.topk_idx).to(dev)
    tw = torch.from_numpy(w.topk_w).to(dev)
    lay = ep.alloc_layout(T, E, R, rpn, dev)
    disp = ep.alloc_dispatch(R, M, H, k, fp8=False, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    cstatus = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def do_layout():
        ep.get_layout(topk, E, R, rpn, out=lay)

    def do_dispatch():
        ep.dispatch(x, topk, tw, lay, M, out=disp)

    def do_combine():
        ep.combine(disp.recv_x, lay, M, out=out, status=cstatus)

    def step():
        do_layout()
        do_dispatch()
        do_combine()

    step()
    torch.cuda.synchronize()
    g_step = capture(step)
    g_stage = {"layout": capture(do_layout), "dispatch": capture(do_dispatch), "combine": capture(do_combine)}

    for _ in range(args.warmup):
        flush()
        g_step.replay()
    torch.cuda.synchronize()
    pairs = int(lay.tokens_per_rank.sum().item())
    flags = ep.read_flags(lay.status) | ep.read_flags(disp.status) | ep.read_flags(cstatus)
    if flags:
        raise RuntimeError(f"kernels raised status flags {flags}")

    clocks = ClockSampler(dev.index)
    clocks.start()
    soak_end = time.perf_counter() + args.soak_s  # untimed load so the sampled clocks are under load
    while time.perf_counter() < soak_end:
        for _ in range(20):
            flush()
            g_step.replay()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for a, z in ev:
        flush()
        a.record(stream)
        g_step.replay()
        z.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    step_ms = [a.elapsed_time(z) for a, z in ev]

    # per-kernel durations: each stage's graph alone, L2 flushed before it
    stage_ms = {s: [] for s in g_stage}
    for _ in range(args.steps):
        for s, g in g_stage.items():
            flush()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            z.record(stream)
            stage_ms[s].append((a, z))
    torch.cuda.synchronize()
    clk = clocks.stop()
    stage_ms = {s: [a.elapsed_time(z) for a, z in v] for s, v in stage_ms.items()}

    ms = max_over_ranks(world, statistics.mean(step_ms))
    b = step_bytes(T, H, k, E, R, N, pairs)
    total_bytes = sum(b.values())
    value = world * total_bytes / (ms * 1e-3) / 1e9
    peak, peak_kind = load_peaks()
    mean = {s: statistics.mean(v) for s, v in stage_ms.items()}
    dom = max(("dispatch", "combine"), key=lambda s: mean[s])
    dom_kernel = {"dispatch": "scatter_rows_tma_kernel<DispatchScatter>", "combine": "combine_kernel"}[dom]
    dom_src = {"dispatch": "ep_dispatch.cu", "combine": "ep_combine.cu"}[dom]
    achieved = b[dom] / (mean[dom] * 1e-3) / 1e9
    traffic, traffic_note = committed_traffic(dom_kernel, dom_src)
    stages = {s: {"ms": round(mean[s], 4), "ms_p10": round(float(np.percentile(stage_ms[s], 10)), 4),
                  "ms_p90": round(float(np.percentile(stage_ms[s], 90)), 4),
                  "alg_bytes": b[s], "gbs": round(b[s] / (mean[s] * 1e-3) / 1e9, 1),
                  "frac_of_hbm_peak": round(b[s] / (mean[s] * 1e-3) / 1e9 / peak, 4)} for s in stage_ms}

    e2e = None if args.no_e2e else run_e2e(ep, w, dev, lay, disp, out, cstatus, flush, args, world, total_bytes)
    sustained = None if args.skip_extra else sustained_step(ep, dev, args, flush, peak)
    extra = {} if args.skip_extra else extra_stages(ep, dev, args, flush, peak)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "ms_per_step_median": round(statistics.median(step_ms), 4),
        "ms_per_step_p10": round(float(np.percentile(step_ms, 10)), 4),
        "ms_per_step_p90": round(float(np.percentile(step_ms, 90)), 4),
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "dsv3 prefill: T=4096 H=7168 bf16, E=256 top-8, R=32 virtual ranks "
                               "(8 nodes x 4), max_tokens=4096, identity expert",
                   "T": T, "H": H, "E": E, "k": k, "R": R, "nodes": N, "max_tokens": M,
                   "pairs": pairs, "parallelism": f"replicas x{world}",
                   "launch": "each step is one CUDA graph replay of the three library kernels",
                   "l2": "flushed between steps: 256 MiB write then 256 MiB read, outside the timed events",
                   "soak_s": args.soak_s},
        "tokens_per_s": round(world * T / (ms * 1e-3), 1),
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "stages": stages,
        "roofline": {"bound": "hbm", "kernel": dom_kernel, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} (copy bandwidth, hbm_gbs)"
                     if peak_kind == "measured" else "fallback", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "alg_bytes_per_launch": b[dom], "traffic_note": traffic_note},
        "sustained": sustained,
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
        "extra_workloads": extra,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
        if not args.skip_extra:
            line["cpu_baseline"]["per_stage"] = oracle_stage_baselines()
    return line


def run_e2e(ep, w, dev, lay, disp, out, cstatus, flush, args, world, total_bytes):
    """The same step through the public API as a user pipeline calls it, with every step's
    inputs copied in from pinned host memory and its combined result copied back. Steps are
    double-buffered on two copy streams: step i+1's inputs travel host -> device while step
    i computes and its result travels device -> host (the link is full duplex). The timed
    region holds K whole steps, copies included; the value is K steps' bytes over it."""
    T, H, E, R, rpn, M = w.T, w.H, w.E, w.R, w.ranks_per_node, w.max_tokens
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    x_h = torch.from_numpy(w.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    topk_h = torch.from_numpy(w.topk_idx).pin_memory()
    tw_h = torch.from_numpy(w.topk_w).pin_memory()
    nb = 2
    out_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    x_d = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(nb)]
    topk_d = [torch.empty_like(topk_h, device=dev) for _ in range(nb)]
    tw_d = [torch.empty_like(tw_h, device=dev) for _ in range(nb)]
    out_d = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(nb)]
    ev = {n: [torch.cuda.Event() for _ in range(nb)] for n in ("in", "used", "done", "out")}

    def step(i):
        b = i % nb
        with torch.cuda.stream(s_in):
            if i >= nb:
                s_in.wait_event(ev["used"][b])  # step i-2 no longer reads these inputs
            topk_d[b].copy_(topk_h, non_blocking=True)
            tw_d[b].copy_(tw_h, non_blocking=True)
            x_d[b].copy_(x_h, non_blocking=True)
            ev["in"][b].record(s_in)
        main.wait_event(ev["in"][b])
        ep.get_layout(topk_d[b], E, R, rpn, out=lay)
        ep.dispatch(x_d[b], topk_d[b], tw_d[b], lay, M, out=disp)
        ev["used"][b].record(main)
        if i >= nb:
            main.wait_event(ev["out"][b])  # step i-2's result has left out_d[b]
        ep.combine(disp.recv_x, lay, M, out=out_d[b], status=cstatus)
        ev["done"][b].record(main)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["done"][b])
            out_h[b].copy_(out_d[b], non_blocking=True)
            ev["out"][b].record(s_out)

    for i in range(2 * nb):
        step(i)
    torch.cuda.synchronize()
    K = max(args.steps, 2 * nb)
    flush()
    torch.cuda.synchronize()
    barrier(world)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    s_in.wait_event(a)  # the first copy starts after the start event
    for i in range(K):
        step(i)
    main.wait_stream(s_out)
    z.record(main)
    z.synchronize()
    last = (K - 1) % nb
    assert torch.equal(out_h[last], out_d[last].cpu())
    assert torch.equal(out_h[last], out.cpu())  # the same step as the device-timed one
    t = max_over_ranks(world, a.elapsed_time(z) / K)
    return {"value": round(world * total_bytes / (t * 1e-3) / 1e9, 2), "unit": UNIT, "ms_per_step": round(t, 4),
            "h2d_bytes_per_step": x_h.numel() * 2 + topk_h.numel() * 8 + tw_h.numel() * 4,
            "d2h_bytes_per_step": out_h[0].numel() * 2, "steps": K,
            "path": "pinned host -> cudaMemcpyAsync (copy stream) -> ep_get_layout, ep_dispatch, ep_combine -> "
                    "pinned host (second copy stream); double-buffered, step i+1's input copy overlapping step i's "
                    "compute and output copy; L2 flushed once before the timed steps"}


def sustained_step(ep, dev, args, flush, peak, K=8):
    """K whole steps (layout -> dispatch -> combine) back to back in one graph, each on its
    own input and output buffers (K x 505 MB touched, far beyond L2), L2 flushed only before
    the replay: every step's writes are written back to HBM inside the timed region (by the
    steps that follow; the last step's output is the only data possibly left in L2)."""
    stream = torch.cuda.current_stream()
    w = workloads.make("dsv3")
    T, H, E, k, R, rpn, M = w.T, w.H, w.E, w.k, w.R, w.ranks_per_node, w.max_tokens
    x0 = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
    topk0 = torch.from_numpy(w.topk_idx).to(dev)
    tw0 = torch.from_numpy(w.topk_w).to(dev)
    sets = []
    for _ in range(K):
        sets.append({"x": x0.clone(), "topk": topk0.clone(), "tw": tw0.clone(),
                     "lay": ep.alloc_layout(T, E, R, rpn, dev), "d": ep.alloc_dispatch(R, M, H, k, device=dev),
                     "out": torch.empty((T, H), dtype=torch.bfloat16, device=dev)})

    def run():
        for st in sets:
            ep.get_layout(st["topk"], E, R, rpn, out=st["lay"])
            ep.dispatch(st["x"], st["topk"], st["tw"], st["lay"], M, out=st["d"])
            ep.combine(st["d"].recv_x, st["lay"], M, out=st["out"])

    side = torch.cuda.Stream()
    ev_lay = [torch.cuda.Event() for _ in range(K)]

    def run_pipelined():
        """The same K steps as a stream of batches: the layouts (routing only, latency-bound)
        run on a second stream, each step's dispatch waiting for its own layout, so that
        step i + 1's layout overlaps step i's dispatch and combine."""
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            for i, st in enumerate(sets):
                ep.get_layout(st["topk"], E, R, rpn, out=st["lay"])
                ev_lay[i].record(side)
        for i, st in enumerate(sets):
            main.wait_event(ev_lay[i])
            ep.dispatch(st["x"], st["topk"], st["tw"], st["lay"], M, out=st["d"])
            ep.combine(st["d"].recv_x, st["lay"], M, out=st["out"])
        main.wait_stream(side)

    n_rep = max(3, min(args.steps, 10))
    times = time_events(run, n_rep, flush, stream)
    ms = float(times) / K
    pairs = int(sets[0]["lay"].tokens_per_rank.sum().item())
    assert torch.equal(sets[-1]["out"], sets[0]["out"])
    for st in sets:
        st["out"].zero_()
    ptimes = time_events(run_pipelined, n_rep, flush, stream)
    pms = float(ptimes) / K
    assert all(torch.equal(st["out"], sets[0]["out"]) for st in sets) and bool(sets[0]["out"].any())
    total = sum(step_bytes(T, H, k, E, R, w.num_nodes, pairs).values())
    del sets
    gb = lambda t: total / (t * 1e-3) / 1e9
    return {"steps_per_replay": K, "ms_per_step": round(ms, 4), "ms_per_step_p10": round(times.p10 / K, 4),
            "ms_per_step_p90": round(times.p90 / K, 4), "replays": times.n, "alg_bytes_per_step": total,
            "gbs": round(gb(ms), 1), "frac_of_hbm_peak": round(gb(ms) / peak, 4),
            "tokens_per_s": round(T / (ms * 1e-3), 1),
            "timing": f"{K} steps on {K} distinct buffer sets in one graph; L2 flushed before each replay only",
            "pipelined": {"ms_per_step": round(pms, 4), "ms_per_step_p10": round(ptimes.p10 / K, 4),
                          "ms_per_step_p90": round(ptimes.p90 / K, 4), "gbs": round(gb(pms), 1),
                          "frac_of_hbm_peak": round(gb(pms) / peak, 4), "tokens_per_s": round(T / (pms * 1e-3), 1),
                          "timing": "the same steps with the layouts on a second stream, each dispatch waiting "
                                    "for its own layout (a stream of batches: step i+1's routing layout overlaps "
                                    "step i's dispatch and combine); every byte still charged"}}


class Times(float):
    """Mean device time (ms) of timed replays, carrying their median, 10th and 90th
    percentiles and count."""

    def __new__(cls, samples):
        obj = float.__new__(cls, statistics.mean(samples))
        obj.median = statistics.median(samples)
        obj.p10 = float(np.percentile(samples, 10))
        obj.p90 = float(np.percentile(samples, 90))
        obj.n = len(samples)
        return obj


def time_events(fn, n, flush, stream):
    """Device time of fn, captured in a CUDA graph, L2 flushed before each of n replays."""
    g = capture(fn)
    ms = []
    for _ in range(n):
        flush()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        z.record(stream)
        ms.append((a, z))
    torch.cuda.synchronize()
    return Times([a.elapsed_time(z) for a, z in ms])


def extra_stages(ep, dev, args, flush, peak):
    """Per-stage device times of the other workloads (FP8 dispatch and combine, combined weights,
    restripe + node dispatch,
    skewed routing). Each is timed with CUDA events, L2 flushed before every launch."""
    stream = torch.cuda.current_stream()
    n = STAGE_ITERATIONS
    res = {"iterations_per_stage": n}

    def gbs(bytes_, ms, per=1):
        """ms: the mean (and, from time_events, the distribution) of one timed replay, which
        holds `per` launches of the stage."""
        t = float(ms) / per
        out = {"ms": round(t, 4), "alg_bytes": bytes_, "gbs": round(bytes_ / (t * 1e-3) / 1e9, 1),
               "frac_of_hbm_peak": round(bytes_ / (t * 1e-3) / 1e9 / peak, 4)}
        if isinstance(ms, Times):
            out.update({"ms_median": round(ms.median / per, 4), "ms_p10": round(ms.p10 / per, 4),
                        "ms_p90": round(ms.p90 / per, 4)})
        return out

    # FP8 dispatch (dsv3 shape)
    w = workloads.make("dsv3_fp8")
    x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(w.topk_idx).to(dev)
    tw = torch.from_numpy(w.topk_w).to(dev)
    lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node)
    d = ep.alloc_dispatch(w.R, w.max_tokens, w.H, w.k, fp8=True, device=dev)
    ep.dispatch(x, topk, tw, lay, w.max_tokens, fp8=True, out=d)
    pairs = int(lay.tokens_per_rank.sum().item())
    ms = time_events(lambda: ep.dispatch(x, topk, tw, lay, w.max_tokens, fp8=True, out=d), n, flush, stream)
    row = w.H + 4 * (w.H // 128)
    b = step_bytes(w.T, w.H, w.k, w.E, w.R, w.num_nodes, pairs, row_bytes_out=row)["dispatch"]
    res["dsv3_fp8_dispatch"] = gbs(b, ms)
    # combine of the FP8 rows (the identity expert: the dispatch output itself) and the
    # combined top-k weights, dsv3 shape
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    ms = time_events(lambda: ep.combine_fp8(d.recv_x, d.recv_scales, lay, w.max_tokens, out=out), n, flush, stream)
    res["dsv3_fp8_combine"] = gbs(pairs * row + 4 * w.T * w.R + 2 * w.T * w.H, ms)
    cw = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
    ms = time_events(lambda: ep.combine_weights(d.recv_topk_w, lay, w.max_tokens, out=cw), n, flush, stream)
    res["dsv3_combine_weights"] = gbs(pairs * 4 * w.k + 4 * w.T * w.R + 4 * w.T * w.k, ms)
    del d, x, lay, out, cw

    # restripe + node dispatch (T=8192, H=7168, 8 nodes, P=128)
    w = workloads.make("restripe")
    x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(w.topk_idx).to(dev)
    lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node)
    prob = torch.from_numpy(w.prob).to(dev)
    Nn, T, M, P, H = w.num_nodes, w.T, w.max_tokens, w.prob.shape[2], w.H
    staging = torch.empty((Nn, M, P), dtype=torch.float32, device=dev)
    ms1 = time_events(lambda: ep.ep_restripe_prob(prob, M, staging), n, flush, stream)
    # the kernel's own rate: 8 restripes back to back on 8 distinct buffer pairs (536 MB, well
    # beyond L2) in one graph, so each launch also pays the write-back of the previous one's
    # output; a single launch after a flush is dominated by the ~6 us event/launch floor
    NB = 8
    probs = [prob] + [prob.clone() for _ in range(NB - 1)]
    stagings = [staging] + [torch.empty_like(staging) for _ in range(NB - 1)]
    ms8 = time_events(lambda: [ep.ep_restripe_prob(probs[i], M, stagings[i]) for i in range(NB)], n, flush, stream)
    res["restripe_prob"] = gbs(2 * T * Nn * P * 4, ms8, per=NB)
    res["restripe_prob"].update({"timing": f"{NB} launches back to back on distinct buffers in one graph, per launch",
                                 "single_launch_ms": round(ms1, 4),
                                 "single_launch_gbs": round(2 * T * Nn * P * 4 / (ms1 * 1e-3) / 1e9, 1)})
    del probs, stagings
    rx = torch.empty((Nn, M, H), dtype=torch.bfloat16, device=dev)
    rp = torch.empty((Nn, M, P), dtype=torch.float32, device=dev)
    routed = int(lay.is_token_in_node.sum().item())
    for name, mode, dests in (("node_dispatch_sparse", ep.NODES_SPARSE, routed),
                              ("node_dispatch_dense", ep.NODES_DENSE, Nn * T)):
        fn = lambda mode=mode: ep.ep_dispatch_nodes(x, staging, lay.is_token_in_node, Nn, M, w.chunk_tokens, mode,
                                                    rx, rp)
        fn()
        ms = time_events(fn, n, flush, stream)
        res[name] = gbs(T * 2 * H + dests * (2 * H + 2 * P * 4) + (T * Nn if mode == ep.NODES_SPARSE else 0), ms)
    del rx, rp, staging, prob, x, lay

    # expert-major path on the dsv3 shape: expert layout, fused dispatch + permute, the split
    # path's receive phase, and the weighted combine from the expert-major slabs
    w = workloads.make("dsv3")
    T, H, k, E, R = w.T, w.H, w.k, w.E, w.R
    x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(w.topk_idx).to(dev)
    tw = torch.from_numpy(w.topk_w).to(dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    eslot = torch.empty((T, k), dtype=torch.int32, device=dev)
    ews = torch.zeros(ep.ep_expert_layout_workspace_size(T, E), dtype=torch.uint8, device=dev)
    ep.ep_get_expert_layout(topk, E, off, eslot, ews)
    offs = off.cpu().numpy()
    epr = E // R
    Mp = int(max(offs[(r + 1) * epr] - offs[r * epr] for r in range(R)))
    entries = int(offs[E])
    px = torch.empty((R, Mp, H), dtype=torch.bfloat16, device=dev)
    ps = torch.empty((R, Mp), dtype=torch.int32, device=dev)
    pw = torch.empty((R, Mp), dtype=torch.float32, device=dev)
    lay = ep.get_layout(topk, E, R, w.ranks_per_node)
    pairs = int(lay.tokens_per_rank.sum().item())
    d = ep.alloc_dispatch(R, w.max_tokens, H, k, device=dev)
    ep.dispatch(x, topk, tw, lay, w.max_tokens, out=d)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ms = time_events(lambda: ep.ep_get_expert_layout(topk, E, off, eslot, ews), n, flush, stream)
    res["expert_layout"] = gbs(T * k * 12 + 4 * (E + 1), ms)
    ms = time_events(lambda: ep.ep_dispatch_permuted(x, topk, tw, off, eslot, E, R, Mp, px, ps, pw), n, flush, stream)
    res["dispatch_permuted"] = gbs(T * 2 * H + T * k * 16 + entries * (2 * H + 8), ms)
    ms = time_events(lambda: ep.ep_permute_received(d.recv_x, d.recv_src_idx, d.recv_topk_idx, d.recv_topk_w,
                                                    lay.tokens_per_rank, off, eslot, E, Mp, px, ps, pw),
                     n, flush, stream)
    res["permute_received"] = gbs(pairs * (2 * H + 4 + 8 * k) + T * k * 4 + entries * (2 * H + 8), ms)
    ms = time_events(lambda: ep.ep_combine_permuted(px, topk, tw, off, eslot, E, out), n, flush, stream)
    res["combine_permuted_weighted"] = gbs(entries * 2 * H + T * k * 16 + T * 2 * H, ms)
    res["permuted_entries"] = entries
    # split (hook-mode) combine: send phase back into the rank slabs, then the rank combine
    yr = torch.empty((R, w.max_tokens, H), dtype=torch.bfloat16, device=dev)
    send = lambda: ep.ep_combine_send(px, d.recv_src_idx, d.recv_topk_idx, d.recv_topk_w, lay.tokens_per_rank, off,
                                      eslot, E, yr)
    # read the expert-major rows, each received row's metadata, the expert slots and offsets;
    # write one rank-level row per received row
    b_send = entries * 2 * H + pairs * (2 * H + 4 + 8 * k) + T * k * 4 + 4 * (E + 1)
    ms = time_events(send, n, flush, stream)
    res["combine_send_weighted"] = gbs(b_send, ms)

    def split():
        send()
        ep.combine(yr, lay, w.max_tokens, out=out)

    ms = time_events(split, n, flush, stream)
    res["split_combine_weighted"] = gbs(b_send + pairs * 2 * H + 4 * T * R + T * 2 * H, ms)
    del px, ps, pw, d, x, lay, out, yr

    # decode-sized batch (T=128 of the same shape): expert layout + dispatch + permute as two
    # launches (one graph) against the single low-latency launch, then the weighted combine
    Td = 128
    w = workloads.make("dsv3", T=Td)
    x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(w.topk_idx).to(dev)
    tw = torch.from_numpy(w.topk_w).to(dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    eslot = torch.empty((Td, k), dtype=torch.int32, device=dev)
    ews = torch.zeros(ep.ep_expert_layout_workspace_size(Td, E), dtype=torch.uint8, device=dev)
    ep.ep_get_expert_layout(topk, E, off, eslot, ews)
    offs = off.cpu().numpy()
    Mp = int(max(offs[(r + 1) * epr] - offs[r * epr] for r in range(R)))
    entries = int(offs[E])
    px = torch.empty((R, Mp, H), dtype=torch.bfloat16, device=dev)
    ps = torch.empty((R, Mp), dtype=torch.int32, device=dev)
    pw = torch.empty((R, Mp), dtype=torch.float32, device=dev)
    out = torch.empty((Td, H), dtype=torch.bfloat16, device=dev)
    b_dp = Td * 2 * H + Td * k * 8 + 4 * (E + 1) + Td * k * 4 + entries * (2 * H + 8)

    def two_launches():
        ep.ep_get_expert_layout(topk, E, off, eslot, ews)
        ep.ep_dispatch_permuted(x, topk, tw, off, eslot, E, R, Mp, px, ps, pw)

    ms = time_events(two_launches, n, flush, stream)
    res["decode128_layout_plus_dispatch_permuted"] = gbs(b_dp, ms)
    ms = time_events(lambda: ep.ep_dispatch_permuted_ll(x, topk, tw, E, R, Mp, off, eslot, px, ps, pw), n, flush,
                     stream)
    res["decode128_dispatch_permuted_ll"] = gbs(b_dp, ms)
    ms = time_events(lambda: ep.ep_combine_permuted(px, topk, tw, off, eslot, E, out), n, flush, stream)
    res["decode128_combine_permuted_weighted"] = gbs(entries * 2 * H + Td * k * 16 + Td * 2 * H, ms)
    ms = time_events(lambda: ep.ep_combine_permuted_ll(px, topk, tw, off, eslot, E, out), n, flush, stream)
    res["decode128_combine_ll_weighted"] = gbs(entries * 2 * H + Td * k * 16 + Td * 2 * H, ms)
    # the decode round trip (dispatch + permute, then the weighted combine of the permuted
    # rows as the identity expert's output), in one graph: the normal kernels (expert layout,
    # dispatch + permute, combine) against the two low-latency launches, whose combine is
    # scheduled while the dispatch still runs
    b_rt = b_dp + entries * 2 * H + Td * k * 16 + Td * 2 * H

    def normal_rt():
        two_launches()
        ep.ep_combine_permuted(px, topk, tw, off, eslot, E, out)

    def ll_rt():
        ep.ep_dispatch_permuted_ll(x, topk, tw, E, R, Mp, off, eslot, px, ps, pw)
        ep.ep_combine_permuted_ll(px, topk, tw, off, eslot, E, out)

    res["decode128_roundtrip_normal"] = gbs(b_rt, time_events(normal_rt, n, flush, stream))
    res["decode128_roundtrip_ll"] = gbs(b_rt, time_events(ll_rt, n, flush, stream))
    floor = torch.zeros(4, device=dev)
    res["event_floor_ms"] = round(time_events(lambda: floor.add_(1), n, flush, stream), 4)
    del px, ps, pw, x, out

    # the tiny workload's whole step (T=128, H=1024, E=16, k=4, R=4), one graph
    w = workloads.make("tiny")
    x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(w.topk_idx).to(dev)
    tw = torch.from_numpy(w.topk_w).to(dev)
    lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node)
    d = ep.alloc_dispatch(w.R, w.max_tokens, w.H, w.k, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)

    def tiny_step():
        ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay)
        ep.dispatch(x, topk, tw, lay, w.max_tokens, out=d)
        ep.combine(d.recv_x, lay, w.max_tokens, out=out)

    tiny_step()
    pairs = int(lay.tokens_per_rank.sum().item())
    ms = time_events(tiny_step, n, flush, stream)
    res["tiny_step"] = gbs(sum(step_bytes(w.T, w.H, w.k, w.E, w.R, w.num_nodes, pairs).values()), ms)
    del x, lay, d, out

    # skewed routing dispatch + combine (T=16384, H=4096, R=64, max_tokens = hottest rank)
    w = workloads.make("skewed")
    x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(w.topk_idx).to(dev)
    tw = torch.from_numpy(w.topk_w).to(dev)
    lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node)
    M = int(lay.tokens_per_rank.max().item())
    pairs = int(lay.tokens_per_rank.sum().item())
    d = ep.alloc_dispatch(w.R, M, w.H, w.k, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    ms_l = time_events(lambda: ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay), n, flush, stream)
    ep.dispatch(x, topk, tw, lay, M, out=d)
    ms_d = time_events(lambda: ep.dispatch(x, topk, tw, lay, M, out=d), n, flush, stream)
    ms_c = time_events(lambda: ep.combine(d.recv_x, lay, M, out=out), n, flush, stream)
    b = step_bytes(w.T, w.H, w.k, w.E, w.R, w.num_nodes, pairs)
    res["skewed_layout"] = gbs(b["layout"], ms_l)
    res["skewed_dispatch"] = gbs(b["dispatch"], ms_d)
    res["skewed_combine"] = gbs(b["combine"], ms_c)
    res["skewed_hottest_rank_tokens"] = M
    res["skewed_mean_rank_tokens"] = round(pairs / w.R, 1)
    return res


# --------------------------------------------------------------------------- profiling runs

PROFILE_STAGES = ("step", "sustained", "restripe", "send", "fp8", "decode", "nodes", "permuted", "skewed")


def profile_stage(name):
    """Run one stage's kernels three times, L2 flushed before each, and exit: a small, fixed
    program for ncu captures (no timing, no JSON line). step: the dsv3 layout, dispatch and
    combine; sustained: the dsv3 step on 8 distinct buffer sets back to back; restripe: the
    prob restripe (T=8192, 8 nodes, P=128); send: the dsv3 send phase of the split combine;
    fp8: the dsv3 FP8 dispatch, then the FP8-input combine of its rows; decode: the
    low-latency dispatch + permute of a T=128 dsv3 batch, then its low-latency weighted
    combine; nodes: the restripe, then the sparse and the dense node dispatch (T=8192,
    H=7168, 8 nodes, P=128); permuted: the dsv3 expert layout, fused dispatch + permute,
    receive-side permute and weighted combine from the expert-major slabs; skewed: the
    skewed layout, dispatch and combine (T=16384, H=4096, R=64, max_tokens = hottest rank)."""
    import combine_ep_get_05_gb300 as ep

    ep.build_library()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    flush = L2Flush(dev)

    def load(wname, **over):
        w = workloads.make(wname, **over)
        x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
        return w, x, torch.from_numpy(w.topk_idx).to(dev), torch.from_numpy(w.topk_w).to(dev)

    if name in ("step", "sustained"):
        w, x, topk, tw = load("dsv3")
        M = w.max_tokens
        sets = [(x.clone(), topk.clone(), tw.clone(), ep.alloc_layout(w.T, w.E, w.R, w.ranks_per_node, dev),
                 ep.alloc_dispatch(w.R, M, w.H, w.k, device=dev), torch.empty((w.T, w.H), dtype=torch.bfloat16,
                                                                              device=dev))
                for _ in range(8 if name == "sustained" else 1)]
        for _ in range(3):
            flush()
            for xx, tk, ww, lay, d, out in sets:
                ep.get_layout(tk, w.E, w.R, w.ranks_per_node, out=lay)
                ep.dispatch(xx, tk, ww, lay, M, out=d)
                ep.combine(d.recv_x, lay, M, out=out)
    elif name == "restripe":
        w = workloads.make("restripe")
        prob = torch.from_numpy(w.prob).to(dev)
        out = torch.empty((w.num_nodes, w.max_tokens, w.prob.shape[2]), dtype=torch.float32, device=dev)
        for _ in range(3):
            flush()
            ep.ep_restripe_prob(prob, w.max_tokens, out)
    elif name == "send":
        w, x, topk, tw = load("dsv3")
        E, R, T, H, k = w.E, w.R, w.T, w.H, w.k
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        eslot = torch.empty((T, k), dtype=torch.int32, device=dev)
        ews = torch.zeros(ep.ep_expert_layout_workspace_size(T, E), dtype=torch.uint8, device=dev)
        ep.ep_get_expert_layout(topk, E, off, eslot, ews)
        offs = off.cpu().numpy()
        Mp = int(max(offs[(r + 1) * (E // R)] - offs[r * (E // R)] for r in range(R)))
        px = torch.empty((R, Mp, H), dtype=torch.bfloat16, device=dev)
        ep.ep_dispatch_permuted(x, topk, tw, off, eslot, E, R, Mp, px)
        lay = ep.get_layout(topk, E, R, w.ranks_per_node)
        d = ep.dispatch(x, topk, tw, lay, w.max_tokens)
        yr = torch.empty((R, w.max_tokens, H), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            flush()
            ep.ep_combine_send(px, d.recv_src_idx, d.recv_topk_idx, d.recv_topk_w, lay.tokens_per_rank, off, eslot,
                               E, yr)
    elif name == "fp8":
        w, x, topk, tw = load("dsv3_fp8")
        lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node)
        d = ep.alloc_dispatch(w.R, w.max_tokens, w.H, w.k, fp8=True, device=dev)
        out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            flush()
            ep.dispatch(x, topk, tw, lay, w.max_tokens, fp8=True, out=d)
            flush()
            ep.combine_fp8(d.recv_x, d.recv_scales, lay, w.max_tokens, out=out)
    elif name == "decode":
        w, x, topk, tw = load("dsv3", T=128)
        E, R, T, H, k = w.E, w.R, w.T, w.H, w.k
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        eslot = torch.empty((T, k), dtype=torch.int32, device=dev)
        ews = torch.zeros(ep.ep_expert_layout_workspace_size(T, E), dtype=torch.uint8, device=dev)
        ep.ep_get_expert_layout(topk, E, off, eslot, ews)
        offs = off.cpu().numpy()
        Mp = int(max(offs[(r + 1) * (E // R)] - offs[r * (E // R)] for r in range(R)))
        px = torch.empty((R, Mp, H), dtype=torch.bfloat16, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            flush()
            ep.ep_dispatch_permuted_ll(x, topk, tw, E, R, Mp, off, eslot, px)
            ep.ep_combine_permuted_ll(px, topk, tw, off, eslot, E, out)
    elif name == "nodes":
        w, x, topk, tw = load("restripe")
        lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node)
        prob = torch.from_numpy(w.prob).to(dev)
        Nn, M, P, H = w.num_nodes, w.max_tokens, w.prob.shape[2], w.H
        staging = torch.empty((Nn, M, P), dtype=torch.float32, device=dev)
        rx = torch.empty((Nn, M, H), dtype=torch.bfloat16, device=dev)
        rp = torch.empty((Nn, M, P), dtype=torch.float32, device=dev)
        for _ in range(3):
            flush()
            ep.ep_restripe_prob(prob, M, staging)
            for mode in (ep.NODES_SPARSE, ep.NODES_DENSE):
                flush()
                ep.ep_dispatch_nodes(x, staging, lay.is_token_in_node, Nn, M, w.chunk_tokens, mode, rx, rp)
    elif name == "permuted":
        w, x, topk, tw = load("dsv3")
        E, R, T, H, k = w.E, w.R, w.T, w.H, w.k
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        eslot = torch.empty((T, k), dtype=torch.int32, device=dev)
        ews = torch.zeros(ep.ep_expert_layout_workspace_size(T, E), dtype=torch.uint8, device=dev)
        ep.ep_get_expert_layout(topk, E, off, eslot, ews)
        offs = off.cpu().numpy()
        Mp = int(max(offs[(r + 1) * (E // R)] - offs[r * (E // R)] for r in range(R)))
        px = torch.empty((R, Mp, H), dtype=torch.bfloat16, device=dev)
        ps = torch.empty((R, Mp), dtype=torch.int32, device=dev)
        pw = torch.empty((R, Mp), dtype=torch.float32, device=dev)
        lay = ep.get_layout(topk, E, R, w.ranks_per_node)
        d = ep.dispatch(x, topk, tw, lay, w.max_tokens)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            flush()
            ep.ep_get_expert_layout(topk, E, off, eslot, ews)
            flush()
            ep.ep_dispatch_permuted(x, topk, tw, off, eslot, E, R, Mp, px, ps, pw)
            flush()
            ep.ep_permute_received(d.recv_x, d.recv_src_idx, d.recv_topk_idx, d.recv_topk_w, lay.tokens_per_rank,
                                   off, eslot, E, Mp, px, ps, pw)
            flush()
            ep.ep_combine_permuted(px, topk, tw, off, eslot, E, out)
    elif name == "skewed":
        w, x, topk, tw = load("skewed")
        lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node)
        M = int(lay.tokens_per_rank.max().item())
        d = ep.alloc_dispatch(w.R, M, w.H, w.k, device=dev)
        out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            flush()
            ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay)
            ep.dispatch(x, topk, tw, lay, M, out=d)
            ep.combine(d.recv_x, lay, M, out=out)
    else:
        raise ValueError(f"unknown stage {name!r}; expected one of {PROFILE_STAGES}")
    torch.cuda.synchronize()
    log(f"profile stage {name}: done")


# --------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    """The oracle (plain single-threaded C) on the host cores, same metric and workload."""
    import oracle

    oracle.build()
    w = workloads.make("dsv3")
    tokens = w.T
    times = []
    pairs = 0
    with one_core() as core:
        for _ in range(args.warmup):
            oracle_step_seconds(w, tokens, tokens)
        for _ in range(args.steps):
            dt, pairs = oracle_step_seconds(w, tokens, tokens)
            times.append(dt)
    s = statistics.mean(times)
    b = step_bytes(tokens, w.H, w.k, w.E, w.R, w.num_nodes, pairs)
    value = sum(b.values()) / s / 1e9
    sample = (f"each step: the oracle's layout+dispatch+identity combine on all {tokens} tokens of the "
              f"dsv3 workload, single-threaded C on one host core")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "dsv3 prefill: T=4096 H=7168 bf16, E=256 top-8, R=32 virtual ranks "
                               "(8 nodes x 4), max_tokens=4096, identity expert"},
        "tokens_per_s": round(tokens / s, 1),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                         "host": host_cpu(), "pinned_core": core},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--skip-extra", action="store_true", help="skip the other workloads' stage timings")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end host-buffer measurement")
    ap.add_argument("--soak-s", type=float, default=1.0, help="untimed load before the timed steps (clocks)")
    ap.add_argument("--profile", choices=PROFILE_STAGES, default=None,
                    help="run one stage's kernels three times for a profiler capture, then exit (no timing)")
    args = ap.parse_args(argv)
    if args.profile is not None:
        profile_stage(args.profile)
        return 0
    if args.warmup < 3:
        log("warmup raised to 3 (minimum)")
        args.warmup = 3
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks have no work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        print(json.dumps(run_reference(args, world, 0)), flush=True)
        return 0
    world, rank, _ = dist_setup()
    line = run_ours(args, world, rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
