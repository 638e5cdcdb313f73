"""Benchmark: the whole indexed sparse attention layer (indexer -> Top-K ->
sparse MLA) on the batched-decode workload, 64 sequences x 32768 history,
64x128 indexer heads, K = 2048, 128 MLA heads over a 576-wide bf16 latent cache.

One step = one dsi_indexed_attention call over the batch (one query token per
sequence), inputs resident in HBM.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--config C]

--impl reference times the CPU oracle (fp64 numpy) on a bounded sample of the
same workload; it is the baseline arm, not a GPU implementation.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

# the oracle's numpy BLAS runs single-threaded unless told otherwise (its core
# count is reported with the CPU baseline)
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from indexed_sparse_attention_indexer_gb300 import workloads as W  # noqa: E402

METRIC = "fused indexer+TopK+sparse-MLA tokens/s; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------
# algorithmic work per step (only what the method must move)
# ----------------------------------------------------------------------------

def algorithmic_bytes(ws) -> dict:
    """Bytes the layer must move per step: every visible index key (+ scale),
    the query tensors, the K selected latent rows, the outputs and indices.
    The score row (4 B per position) is written and read back once by the
    unfused scoring/select pair; it is listed separately."""
    B = ws.T
    lens = ws.seq_lens.to(torch.int64).cpu()
    if ws.mode == "decode":
        vis = decode_visible(ws)
    else:
        vis = torch.arange(1, B + 1, dtype=torch.int64) + ws.q_offset
    kel = ws.k_idx.element_size()
    # index keys are read once per sequence: the candidate rows of a
    # multi-token step see nested prefixes of one history (the longest is the
    # sequence's length); every other row reads its own
    kv = torch.clamp(lens, max=ws.s_max) if (ws.mode == "decode" and ws.tokens_per_seq > 1) else vis
    key = int(kv.sum()) * ws.d * kel
    # scale bytes per key: one fp32 (FP8) or d/G E8M0 bytes (MXFP8)
    if ws.k_scale is None:
        per_key_scale = 0
    elif ws.k_scale.dim() == ws.k_idx.dim():
        per_key_scale = ws.k_scale.shape[-1] * ws.k_scale.element_size()
    else:
        per_key_scale = ws.k_scale.element_size()
    scale = int(kv.sum()) * per_key_scale
    sel = torch.clamp(vis, max=ws.K)
    # one latent row: 576 bf16, or 576 E4M3 codes + 5 fp32 tile scales
    row_bytes = W.D_QK * ws.latent.element_size()
    if getattr(ws, "latent_scale", None) is not None:
        row_bytes += ws.latent_scale.shape[-1] * ws.latent_scale.element_size()
    gather = int(sel.sum()) * row_bytes
    q_bytes = ws.q_idx.numel() * 2 + ws.w.numel() * 4 + ws.q.numel() * 2
    out = B * ws.H * W.D_LATENT * 2 + B * ws.H * 4
    idx = B * ws.K * 4
    scores = int(vis.sum()) * 4 * 2
    return {"index_keys": key + scale, "gather": gather, "queries": q_bytes, "outputs": out,
            "indices": idx, "score_rows": scores,
            "total": key + scale + gather + q_bytes + out + idx}


def scoring_kernel_bytes(ws) -> int:
    """Algorithmic bytes of one scoring launch: index keys (+ scales), q_idx,
    head weights, and the fp32 score row it writes."""
    a = algorithmic_bytes(ws)
    return a["index_keys"] + ws.q_idx.numel() * 2 + ws.w.numel() * 4 + a["score_rows"] // 2


def decode_visible(ws) -> torch.Tensor:
    """Visible history of every decode row: T candidate rows per sequence, row
    (b, t) sees seq_lens[b] - (T - 1 - t) positions (T = 1: seq_lens)."""
    T = ws.tokens_per_seq
    lens = ws.seq_lens.to(torch.int64).cpu()
    if T == 1:
        return lens
    t = torch.arange(T, dtype=torch.int64)
    return torch.clamp(lens.view(-1, 1) - (T - 1 - t).view(1, -1), min=0).reshape(-1)


def algorithmic_flops(ws) -> dict:
    vis = decode_visible(ws) if ws.mode == "decode" else torch.arange(1, ws.T + 1) + ws.q_offset
    idx_fl = 2 * int(vis.sum()) * ws.H_i * ws.d
    sel = torch.clamp(vis, max=ws.K)
    mla_fl = 2 * int(sel.sum()) * ws.H * (W.D_QK + W.D_LATENT)
    return {"indexer": idx_fl, "mla": mla_fl}


# ----------------------------------------------------------------------------
# measured peaks, clocks, profiles
# ----------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, on: bool):
        if on:
            self.t_on = time.time()
        else:
            self.t_off = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        inside = [s for t, s in self.samples if self.t_on and self.t_off and
                  self.t_on - 0.06 <= t <= self.t_off + 0.06]
        used = inside if inside else [s for _, s in self.samples]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in used:
            parts = [x.strip() for x in s.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0])); mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_timed_region": len(inside)}


_HEADERS = ("common.cuh", "tc_common.cuh", "tma_host.h", "kernels.h")
KERNEL_SOURCES = {
    "index_score": ("index_score.cu", "index_score_tc.cu") + _HEADERS,
    "index_topk_prefill": ("index_topk_prefill.cu",) + _HEADERS,
    "mla_tc": ("sparse_mla_tc.cu",) + _HEADERS,
}


def kernel_source_sha(kernel: str = "index_score") -> str:
    """Hash of a kernel's sources (traffic figures go stale when they change)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "indexed_sparse_attention_indexer_gb300", "csrc", f),
                      "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it is now (profiles/traffic.txt: kernel workload bytes sha)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    sha = kernel_source_sha(kernel)
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) == 4 and f[0] == kernel and f[1] == workload and f[3] == sha:
            return float(f[2])
    return None


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def time_alone(launch, stream, n: int) -> float:
    """Average ms of one launch, timed with CUDA events on the launching stream
    over n back-to-back launches after three untimed ones."""
    for _ in range(3):
        launch()
    torch.cuda.synchronize()
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    for _ in range(n):
        launch()
    k1.record(stream)
    torch.cuda.synchronize()
    return k0.elapsed_time(k1) / n


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over the ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank: int, world: int, steps: int, ms_max: float) -> float:
    """Tokens all ranks processed in the timed region / the slowest rank's time
    (replicas: every rank runs its own batch, weak scaling)."""
    return tokens_per_rank * world * steps / (ms_max / 1e3)


def run_gpu(args):
    from indexed_sparse_attention_indexer_gb300 import binding

    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.config]
    # seeded per config; each rank its own replica (--rows: a smaller decode batch
    # for profiling captures, never a bench line)
    ws = W.make_config(args.config, device=dev, rows=args.rows, tokens_per_seq=args.tokens_per_seq,
                       k_mx_group=getattr(args, "k_mx_group", 0),
                       latent_fp8=getattr(args, "latent_fp8", False))
    tps = ws.tokens_per_seq
    wname = ws.name   # the config's workload, or its MXFP8-key variant
    torch.cuda.synchronize()
    binding.load()
    stream = torch.cuda.current_stream()
    cache = binding.Cache.of(ws)
    decode = ws.mode == "decode"
    span = cache.struct.s_max if decode else ws.q_offset + ws.T
    wsp = binding.alloc_workspace(
        binding.workspace_size(ws.T, ws.H_i, ws.H, ws.K, span, decode), dev)
    out = torch.empty((ws.T, ws.H, W.D_LATENT), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((ws.T, ws.H), dtype=torch.float32, device=dev)
    idx = torch.empty((ws.T, ws.K), dtype=torch.int32, device=dev)
    cnt = torch.empty((ws.T,), dtype=torch.int32, device=dev)

    def step():
        if tps > 1:
            binding.indexed_attention_multi(ws.q_idx, ws.w, ws.q, cache, tps, ws.K, ws.scale,
                                            out=out, lse=lse, idx=idx, count=cnt, workspace=wsp,
                                            stream=stream)
        else:
            binding.indexed_attention(ws.q_idx, ws.w, ws.q, cache, ws.K, ws.scale, decode,
                                      ws.q_offset, out=out, lse=lse, idx=idx, count=cnt,
                                      workspace=wsp, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    # keep the GPU busy while the sampler starts, then time exactly K steps
    t_end = time.time() + 0.3
    while time.time() < t_end:
        step()
        torch.cuda.synchronize()
    l0 = binding.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark(True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    barrier(world)
    launches = binding.launch_count() - l0
    ms_local = e0.elapsed_time(e1)
    clk = clocks.stop()
    ms = max_over_ranks(ms_local, world)
    ms_step = ms / args.steps
    value = whole_job_tokens_per_s(ws.T, world, args.steps, ms)

    hbm, tfl, src = peaks()
    extra = {}
    if decode and (tps > 1 or ws.latent_scale is not None):
        # multi-token step (the scoring entry point takes one row per sequence)
        # or FP8 latent cache (the attention core is the changed kernel): the
        # step itself stands in for the kernel (HBM-bound like decode)
        ab_step = algorithmic_bytes(ws)["total"]
        achieved = ab_step / (ms_step / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": "step", "achieved": round(achieved, 1), "peak": hbm,
                    "unit": "GB/s", "frac": round(achieved / hbm, 4), "peak_source": src,
                    "traffic": None, "algorithmic_bytes": ab_step, "kernel_ms": round(ms_step, 5)}
    elif decode:
        # ---- dominant kernel: the indexer scoring launch, timed alone ------
        scores = torch.empty((ws.T, span), dtype=torch.float32, device=dev)
        k_ms = time_alone(lambda: binding.index_score(ws.q_idx, ws.w, cache, decode, ws.q_offset,
                                                      scores=scores, ld=span, stream=stream),
                          stream, max(10, args.steps))
        kbytes = scoring_kernel_bytes(ws)
        achieved = kbytes / (k_ms / 1e3) / 1e9
        kname = "index_score"
        roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": hbm,
                    "unit": "GB/s", "frac": round(achieved / hbm, 4), "peak_source": src,
                    "traffic": recorded_traffic(kname, wname),
                    "algorithmic_bytes": kbytes, "kernel_ms": round(k_ms, 5)}
    else:
        # ---- prefill: both halves are dense contractions on the tensor cores;
        # the attention core dominates, the fused indexer is reported beside it
        fl = algorithmic_flops(ws)
        nk = max(3, min(10, args.steps))
        m_ms = time_alone(lambda: binding.sparse_mla_prefill(ws.q, cache, idx, ws.q_offset, ws.scale,
                                                             out=out, lse=lse, workspace=wsp,
                                                             stream=stream), stream, nk)
        i_ms = time_alone(lambda: binding.index_topk_prefill(ws.q_idx, ws.w, cache, ws.K,
                                                             ws.q_offset, idx=idx, count=cnt,
                                                             stream=stream), stream, nk)

        def tensor_line(kname, flops, ms):
            a_tf = flops / (ms / 1e3) / 1e12
            return {"bound": "tensor", "kernel": kname, "achieved": round(a_tf, 1), "peak": tfl,
                    "unit": "TFLOP/s", "frac": round(a_tf / tfl, 4), "peak_source": src,
                    "traffic": recorded_traffic(kname, cfg["name"]),
                    "algorithmic_flops": flops, "kernel_ms": round(ms, 5)}
        roofline = tensor_line("mla_tc", fl["mla"], m_ms)
        extra["indexer_roofline"] = tensor_line("index_topk_prefill", fl["indexer"], i_ms)
    ab = algorithmic_bytes(ws)
    step_gbs = ab["total"] / (ms_step / 1e3) / 1e9

    # ---- end to end through the public API with host buffers ---------------
    e2e = run_e2e(ws, cache, wsp, decode, args, stream, dev)

    result = None
    if rank == 0:
        fl = algorithmic_flops(ws)
        result = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded generators; integer-valued indexer inputs, N(0,1) latent)",
            "config": {"workload": wname, "batch": ws.T, "history": int(ws.s_max),
                       "indexer": f"{ws.H_i}x{ws.d}", "topk": ws.K, "mla_heads": ws.H,
                       "parallelism": f"replicas x{world} (batch shards, no collective)",
                       "l2": "inputs larger than L2 (537 MB of index keys streamed per step)"},
            "hbm_gbs_step": round(step_gbs, 1),
            "hbm_frac_step": round(step_gbs / hbm, 4),
            "algorithmic_bytes_per_step": ab, "algorithmic_flops_per_step": fl,
            "roofline": roofline, **extra, "e2e": e2e, "gpu_launches": int(launches),
            "gpu_launches_per_step": launches / args.steps, "clocks": clk,
        }
        if args.rows:
            result["config"]["profiling_rows"] = args.rows
        if tps > 1:
            result["config"]["tokens_per_seq"] = tps
        if ws.latent_scale is not None:
            result["config"]["latent_cache"] = "fp8 (E4M3 + fp32 scale per 128-dim tile)"
        mxg = getattr(args, "k_mx_group", 0)
        if mxg:
            result["config"]["index_keys"] = f"mxfp8 (E4M3 + E8M0 per {mxg})"
            result["config"]["l2"] = "inputs larger than L2 (MXFP8 index keys streamed per step)"
        if world == 1 and not args.no_cpu:
            result["cpu_baseline"] = cpu_baseline(ws, budget_s=args.cpu_seconds)
    barrier(world)
    return result


def run_e2e(ws, cache, wsp, decode, args, stream, dev):
    """Same metric through binding.indexed_attention with the per-step inputs
    (q_idx, w, q) copied from pinned host memory and the output read back every
    step; the caches stay resident as they would in serving.  As a server
    would, the copies of one step overlap the computation of its neighbour:
    two device input/output sets alternate, host-to-device copies run on one
    side stream and device-to-host reads on another, ordered by events."""
    from indexed_sparse_attention_indexer_gb300 import binding
    h_qidx = ws.q_idx.cpu().pin_memory()
    h_w = ws.w.cpu().pin_memory()
    h_q = ws.q.cpu().pin_memory()
    h_out = [torch.empty((ws.T, ws.H, W.D_LATENT), dtype=torch.bfloat16).pin_memory()
             for _ in range(2)]
    sets = [(torch.empty_like(ws.q_idx), torch.empty_like(ws.w), torch.empty_like(ws.q),
             torch.empty((ws.T, ws.H, W.D_LATENT), dtype=torch.bfloat16, device=dev))
            for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    computed = [ev(), ev()]     # step on set i finished computing
    read_back = [ev(), ev()]    # its output has been copied to the host
    for e in computed + read_back:
        e.record(stream)

    def step(k):
        i = k & 1
        d_qidx, d_w, d_q, d_out = sets[i]
        landed = ev()
        with torch.cuda.stream(s_in):
            s_in.wait_event(computed[i])          # step k-2 no longer reads set i
            d_qidx.copy_(h_qidx, non_blocking=True)
            d_w.copy_(h_w, non_blocking=True)
            d_q.copy_(h_q, non_blocking=True)
            landed.record(s_in)
        stream.wait_event(landed)
        stream.wait_event(read_back[i])           # step k-2's output was read
        if ws.tokens_per_seq > 1:
            binding.indexed_attention_multi(d_qidx, d_w, d_q, cache, ws.tokens_per_seq, ws.K,
                                            ws.scale, out=d_out, workspace=wsp, want_lse=False,
                                            want_idx=False, stream=stream)
        else:
            binding.indexed_attention(d_qidx, d_w, d_q, cache, ws.K, ws.scale, decode, ws.q_offset,
                                      out=d_out, workspace=wsp, want_lse=False, want_idx=False,
                                      stream=stream)
        computed[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[i])
            h_out[i].copy_(d_out, non_blocking=True)
            read_back[i].record(s_out)

    for k in range(max(3, args.warmup)):
        step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for k in range(args.steps):
        step(k)
    s_out.synchronize()
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    bi = h_qidx.numel() * 2 + h_w.numel() * 4 + h_q.numel() * 2
    bo = h_out[0].numel() * 2
    return {"value": round(ws.T * args.steps / (ms / 1e3), 1), "unit": UNIT,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": round(ms / args.steps, 5),
            "note": "caches resident; per-step queries in, attention output out; copies of a "
                    "step overlap its neighbour's computation (two buffer sets, side streams)"}


# ----------------------------------------------------------------------------
# the oracle (CPU baseline / reference arm)
# ----------------------------------------------------------------------------

def _cpu_rows(ws_dev, rows):
    """CPU copy of the sampled decode rows (the oracle's inputs)."""
    sub = ws_dev.to(ws_dev.q.device)
    sub.q_idx, sub.w, sub.q = ws_dev.q_idx[rows], ws_dev.w[rows], ws_dev.q[rows]
    sub.seq_lens = ws_dev.seq_lens[rows]
    sub.k_idx, sub.latent = ws_dev.k_idx[rows], ws_dev.latent[rows]
    sub.k_scale = None if ws_dev.k_scale is None else ws_dev.k_scale[rows]
    return sub.to("cpu")


def _oracle_rows(ws, budget_s: float, start: int = 0):
    """Run the oracle row by row (starting at ``start``) until ``budget_s`` has
    passed (at least one row).  Returns (rows done, seconds)."""
    import oracle
    rows_done = 0
    cpu_ws = None if ws.mode == "decode" else ws.to("cpu")
    t0 = time.perf_counter()
    while True:
        r = (start + rows_done) % ws.T
        if cpu_ws is None:
            oracle.decode_row(_cpu_rows(ws, [r]), 0)
        else:
            oracle.prefill_row(cpu_ws, r)
        rows_done += 1
        if time.perf_counter() - t0 >= budget_s or rows_done >= ws.T:
            break
    return rows_done, time.perf_counter() - t0


def cpu_baseline(ws, budget_s: float = 10.0) -> dict:
    rows, el = _oracle_rows(ws, budget_s)
    return {"value": round(rows / el, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{rows} of {ws.T} query rows of the same workload (fp64 numpy oracle, "
                      f"single-threaded BLAS, inputs copied to the host per row), {el:.1f} s"}


def run_reference(args):
    """The baseline arm: the CPU oracle on a bounded sample, same metric and config."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return None
    cfg = W.CONFIGS[args.config]
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    ws = W.make_config(args.config, device=dev, k_mx_group=getattr(args, "k_mx_group", 0),
                       latent_fp8=getattr(args, "latent_fp8", False))
    per_step = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    start = 0
    for _ in range(args.warmup):
        n, _ = _oracle_rows(ws, per_step, start)
        start += n
    tot_rows, tot_s = 0, 0.0
    for _ in range(args.steps):
        n, el = _oracle_rows(ws, per_step, start)
        start += n
        tot_rows += n
        tot_s += el
    value = tot_rows / tot_s
    sample = (f"{tot_rows} query rows over {args.steps} timed steps (each a bounded sample of the "
              f"{ws.T}-row batch, ~{per_step:.1f} s), fp64 numpy oracle, single-threaded BLAS")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot_s / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded generators as the GPU arm)",
            "config": {"workload": ws.name, "batch": ws.T, "history": int(ws.s_max),
                       "indexer": f"{ws.H_i}x{ws.d}", "topk": ws.K, "mla_heads": ws.H},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_crossover():
    """Dense versus sparse attention for a decode batch as the history grows:
    the sparse layer (indexer + Top-K 2048 + attention over 2048 rows) against
    attention over every history row (the same attention kernel given all
    positions, K = S, up to the library's 4096-entry limit).  64 sequences,
    64x128 indexer heads, 128 MLA heads, inputs resident."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from indexed_sparse_attention_indexer_gb300 import binding
    binding.load()
    stream = torch.cuda.current_stream()
    B, K = 64, 2048
    res = []
    for S in (1024, 2048, 2560, 3072, 3584, 4096):
        ws = W.make_decode(B, S, 64, 128, K, 128, seed=0, device=dev, name="crossover")
        cache = binding.Cache.of(ws)
        wsp = binding.alloc_workspace(binding.workspace_size(B, 64, 128, K, S, True), dev)
        out = torch.empty((B, 128, W.D_LATENT), dtype=torch.bfloat16, device=dev)
        sparse_ms = time_alone(lambda: binding.indexed_attention(
            ws.q_idx, ws.w, ws.q, cache, K, ws.scale, True, 0, out=out, workspace=wsp,
            want_lse=False, want_idx=False, stream=stream), stream, 20)
        every = torch.arange(S, dtype=torch.int32, device=dev).repeat(B, 1)
        wsd = binding.alloc_workspace(binding.workspace_size(B, 0, 128, S, 0, True), dev)
        dense_ms = time_alone(lambda: binding.sparse_mla_decode(
            ws.q, cache, every, ws.scale, out=out, want_lse=False, workspace=wsd,
            stream=stream), stream, 20)
        res.append({"history": S, "sparse_ms": round(sparse_ms, 4), "dense_ms": round(dense_ms, 4),
                    "sparse_over_dense": round(sparse_ms / dense_ms, 3)})
        del ws, cache, wsp, wsd, every
        torch.cuda.empty_cache()
    cross = next((r["history"] for r in res if r["sparse_ms"] < r["dense_ms"]), None)
    print(json.dumps({"probe": "dense_vs_sparse_decode", "batch": B, "topk": K,
                      "indexer": "64x128", "mla_heads": 128, "results": res,
                      "first_history_where_sparse_wins": cross}))


def run_mx_scan():
    """MXFP8 group-size scan on the decode workload's shapes (64 sequences x
    32768 positions, 64x128 indexer heads, Top-2048): bf16 keys with outlier
    channels and N(0,1) index queries; for G = 32, 64, 128 the keys go through
    the quantiser, are scored on the MXFP8 path (the query quantised in the
    kernel with the same G) and selected, and the selection is compared with
    the one made from bf16 scores of the unquantised keys.  Reports the Top-K
    recall, the score error, the scoring time and the quantiser's bandwidth.
    G = 128 with 128-wide keys is one power-of-two scale per key.  Two key
    distributions: outlier channels (x32 on four channels), and channels whose
    magnitudes spread over exp(U(-5, 5)) (about 2^14 between the extremes),
    where a key's small channels fall below E4M3's range under one coarse scale."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from indexed_sparse_attention_indexer_gb300 import binding
    binding.load()
    stream = torch.cuda.current_stream()
    B, S, Hi, d, K = 64, 32768, 64, 128, 2048
    hbm, _, src = peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    q_idx = torch.randn((B, Hi, d), generator=g, device=dev).to(torch.bfloat16)
    w = torch.rand((B, Hi), generator=g, device=dev)
    lens = torch.full((B,), S, dtype=torch.int32, device=dev)
    latent = torch.empty((1, 1, W.D_QK), dtype=torch.bfloat16, device=dev)   # not read here
    scores = torch.empty((B, S), dtype=torch.float32, device=dev)
    res = []
    for dist_name, spread in (("outlier channels x32", 0.0), ("channel magnitudes exp(U(-5,5))", 5.0)):
        keys = W.make_mx_input(B * S, d, seed=5, device=dev, special=False, row_spread=1.0,
                               channel_spread=spread)
        c_bf = binding.Cache(keys.view(B, S, d), latent, lens)
        ms_bf = time_alone(lambda: binding.index_score(q_idx, w, c_bf, True, scores=scores, ld=S,
                                                       stream=stream), stream, 20)
        ref = scores.clone()
        ref_idx, _ = binding.topk(ref, K, row_len=lens)
        mask = torch.zeros((B, S), dtype=torch.bool, device=dev)
        mask.scatter_(1, ref_idx.to(torch.int64), True)
        ref_mag = ref.abs().mean(dim=1, keepdim=True)
        res.append({"keys_dist": dist_name, "group": None, "keys": "bf16",
                    "key_bytes_per_position": 2 * d, "score_ms": round(ms_bf, 4)})
        for G in (32, 64, 128):
            codes = torch.empty((B * S, d), dtype=torch.float8_e4m3fn, device=dev)
            sc = torch.empty((B * S, d // G), dtype=torch.uint8, device=dev)
            q_ms = time_alone(lambda: binding.mxfp8_quantize(keys, G, codes=codes, scales=sc,
                                                             stream=stream), stream, 20)
            qbytes = B * S * (2 * d + d + d // G)
            c_mx = binding.Cache(codes.view(B, S, d), latent, lens, k_scale=sc.view(B, S, d // G))
            ms = time_alone(lambda: binding.index_score(q_idx, w, c_mx, True, scores=scores, ld=S,
                                                        stream=stream), stream, 20)
            idx, _ = binding.topk(scores, K, row_len=lens)
            hits = mask.gather(1, idx.to(torch.int64)).sum(dim=1).float() / K
            err = ((scores - ref).abs() / ref_mag).flatten()
            res.append({"keys_dist": dist_name, "group": G, "keys": "mxfp8",
                        "key_bytes_per_position": d + d // G,
                        "topk_recall_vs_bf16": round(float(hits.mean()), 5),
                        "topk_recall_min_row": round(float(hits.min()), 5),
                        "score_err_rel_mean_abs_median": float(err.median()),
                        "score_err_rel_mean_abs_max": float(err.max()),
                        "score_ms": round(ms, 4),
                        "quantize_ms": round(q_ms, 4),
                        "quantize_gbs": round(qbytes / (q_ms / 1e3) / 1e9, 1),
                        "quantize_hbm_frac": round(qbytes / (q_ms / 1e3) / 1e9 / hbm, 4)})
            del codes, sc, c_mx
        del keys, c_bf
        torch.cuda.empty_cache()
    print(json.dumps({"probe": "mxfp8_group_scan", "batch": B, "history": S,
                      "indexer": f"{Hi}x{d}", "topk": K, "peak_source": src,
                      "keys": "bf16 N(0,1) x exp(U(-1,1)) per row, then per-channel scaling",
                      "queries": "N(0,1) bf16", "results": res}))


def run_gather_ceiling():
    """Plain-load bandwidth of the attention core's access pattern: 2048 random
    distinct rows of each of 64 sequences x 32768 rows x 1152 bytes (the decode
    workload's latent cache), L2 flushed before each timed launch."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from indexed_sparse_attention_indexer_gb300 import binding
    binding.load()
    B, S, K, pitch = 64, 32768, 2048, W.D_QK * 2
    base = torch.ones(B * S * pitch // 2, dtype=torch.bfloat16, device=dev)
    g = torch.Generator().manual_seed(0)
    rows = torch.stack([torch.randperm(S, generator=g)[:K] + b * S for b in range(B)])
    rows = rows.to(torch.int32).reshape(-1).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    res = []
    for nbytes in (640, 1152):
        for blocks in (2 * sms, 4 * sms):
            best = math.inf
            for rep_i in range(5):
                flush.fill_(rep_i & 255)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                binding.probe_random_gather(base, pitch, rows, nbytes, blocks)
                e1.record()
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1))
            res.append({"bytes_per_row": nbytes, "blocks": blocks, "us": round(best * 1e3, 1),
                        "gbs": round(rows.numel() * nbytes / (best / 1e3) / 1e9, 1)})
    print(json.dumps({"probe": "random_row_gather", "rows": int(rows.numel()),
                      "cache_bytes": B * S * pitch, "row_pitch": pitch, "results": res,
                      "best_gbs": max(r["gbs"] for r in res)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", type=int, default=2, choices=sorted(W.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--crossover", action="store_true",
                    help="measurement: dense vs sparse attention as the history grows (not a bench line)")
    ap.add_argument("--gather-ceiling", action="store_true",
                    help="diagnostic: random-row gather bandwidth of plain loads (not a bench line)")
    ap.add_argument("--tokens-per-seq", type=int, default=1,
                    help="decode workloads: candidate tokens verified per sequence in one step "
                         "(multi-token decode; the default line is 1)")
    ap.add_argument("--k-mx-group", type=int, default=0, choices=[0, 32, 64, 128],
                    help="contiguous decode workloads: index keys stored as MXFP8 with this "
                         "many elements per scale (0: the workload's own key format)")
    ap.add_argument("--latent-fp8", action="store_true",
                    help="the 64x128-head decode workload with an FP8 latent cache (own bench line)")
    ap.add_argument("--mx-scan", action="store_true",
                    help="measurement: MXFP8 group-size scan, precision and speed (not a bench line)")
    ap.add_argument("--rows", type=int, default=None,
                    help="profiling aid: a smaller decode batch (the printed line is not a bench line)")
    args = ap.parse_args()
    if args.gather_ceiling:
        run_gather_ceiling()
        return
    if args.crossover:
        run_crossover()
        return
    if args.mx_scan:
        run_mx_scan()
        return
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
