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
    # a prefill row with at most K positions of history takes all of them: its
    # scores decide nothing, and the fused indexer does not compute them
    scored = vis if ws.mode == "decode" else vis[vis > ws.K]
    idx_fl = 2 * int(scored.sum()) * ws.H_i * ws.d
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


def _outputs(ws, dev):
    out = torch.empty((ws.T, ws.H, W.D_LATENT), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((ws.T, ws.H), dtype=torch.float32, device=dev)
    idx = torch.empty((ws.T, ws.K), dtype=torch.int32, device=dev)
    cnt = torch.empty((ws.T,), dtype=torch.int32, device=dev)
    return out, lse, idx, cnt


def _layer_step(ws, cache, wsp, bufs, stream):
    """One call of the fused layer over the workload (the bench's step)."""
    from indexed_sparse_attention_indexer_gb300 import binding
    out, lse, idx, cnt = bufs
    decode = ws.mode == "decode"
    tps = ws.tokens_per_seq
    if tps > 1:
        return lambda: binding.indexed_attention_multi(
            ws.q_idx, ws.w, ws.q, cache, tps, ws.K, ws.scale, out=out, lse=lse, idx=idx,
            count=cnt, workspace=wsp, stream=stream)
    return lambda: binding.indexed_attention(
        ws.q_idx, ws.w, ws.q, cache, ws.K, ws.scale, decode, ws.q_offset, out=out, lse=lse,
        idx=idx, count=cnt, workspace=wsp, stream=stream)


def _workspace(ws, cache, dev):
    from indexed_sparse_attention_indexer_gb300 import binding
    return binding.alloc_workspace(binding.layer_workspace_size(
        cache, ws.T, ws.H_i, ws.H, ws.K, ws.q_offset, ws.mode == "decode"), dev)


def time_steps(step, stream, steps: int, warmup: int, local: int, world: int = 1,
               flush=None) -> dict:
    """Warm-up, then exactly ``steps`` steps timed with CUDA events on the
    launching stream between barriers, nvidia-smi clocks sampled meanwhile.
    With ``flush`` (a callable writing a buffer larger than L2) every step is
    timed on its own after a flush, for workloads that would sit in L2."""
    from indexed_sparse_attention_indexer_gb300 import binding
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t_end = time.time() + 0.3        # keep the GPU busy while the sampler starts
    while time.time() < t_end:
        step()
        torch.cuda.synchronize()
    l0 = binding.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark(True)
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_local = e0.elapsed_time(e1)
    else:
        evs = []
        for _ in range(steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ms_local = sum(a.elapsed_time(b) for a, b in evs)
    clocks.mark(False)
    barrier(world)
    launches = binding.launch_count() - l0
    return {"ms_local": ms_local, "clocks": clocks.stop(), "launches": launches}


def _tensor_line(kname, flops, ms, tfl, src, workload):
    a_tf = flops / (ms / 1e3) / 1e12
    return {"bound": "tensor", "kernel": kname, "achieved": round(a_tf, 1), "peak": tfl,
            "unit": "TFLOP/s", "frac": round(a_tf / tfl, 4), "peak_source": src,
            "traffic": recorded_traffic(kname, workload), "algorithmic_flops": flops,
            "kernel_ms": round(ms, 5)}


def _score_roofline(ws, cache, span, stream, dev, n, hbm, src):
    """The indexer scoring launch timed alone (decode: the dominant kernel)."""
    from indexed_sparse_attention_indexer_gb300 import binding
    scores = torch.empty((ws.T, span), dtype=torch.float32, device=dev)
    k_ms = time_alone(lambda: binding.index_score(ws.q_idx, ws.w, cache, True, 0, scores=scores,
                                                  ld=span, stream=stream), stream, n)
    kbytes = scoring_kernel_bytes(ws)
    achieved = kbytes / (k_ms / 1e3) / 1e9
    return {"bound": "hbm", "kernel": "index_score", "achieved": round(achieved, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(achieved / hbm, 4), "peak_source": src,
            "traffic": recorded_traffic("index_score", ws.name), "algorithmic_bytes": kbytes,
            "kernel_ms": round(k_ms, 5)}


def _prefill_rooflines(parts, cache, part_bufs, wsp, stream, n, tfl, src):
    """Both prefill kernels timed alone over the step's calls (one workload,
    or a rank's zigzag segments), against their algorithmic flops."""
    from indexed_sparse_attention_indexer_gb300 import binding
    if not isinstance(parts, (list, tuple)):
        parts, part_bufs = [parts], [part_bufs]
    fl_m = sum(algorithmic_flops(p)["mla"] for p in parts)
    fl_i = sum(algorithmic_flops(p)["indexer"] for p in parts)

    def mla():
        for p, (out, lse, idx, _) in zip(parts, part_bufs):
            binding.sparse_mla_prefill(p.q, cache, idx, p.q_offset, p.scale, out=out, lse=lse,
                                       workspace=wsp, stream=stream)

    def indexer():
        for p, (_, _, idx, cnt) in zip(parts, part_bufs):
            binding.index_topk_prefill(p.q_idx, p.w, cache, p.K, p.q_offset, idx=idx, count=cnt,
                                       stream=stream)
    # the indexer first: the attention core reads the indices it writes
    i_ms = time_alone(indexer, stream, n)
    m_ms = time_alone(mla, stream, n)
    name = parts[0].name
    return (_tensor_line("mla_tc", fl_m, m_ms, tfl, src, name),
            _tensor_line("index_topk_prefill", fl_i, i_ms, tfl, src, name))


def prefill_parts(ws, world: int, rank: int):
    """This rank's zigzag segments of a prefill, each a workload of its own
    (query rows sliced, query offset at the segment's start, cache shared)."""
    from indexed_sparse_attention_indexer_gb300 import partition
    out = []
    for a, b in partition.zigzag_segments(ws.T, world)[rank]:
        out.append(W.Workload(ws.name, "prefill", ws.H_i, ws.d, ws.K, ws.H, ws.scale,
                              ws.q_idx[a:b], ws.w[a:b], ws.q[a:b], ws.k_idx, ws.k_scale,
                              ws.latent, ws.seq_lens, ws.block_table, ws.page_size,
                              ws.q_offset + a, dict(ws.meta), ws.latent_scale))
    return out


def _l2_flusher(dev):
    # 1 GB: far larger than L2, and long enough on the device (~0.15 ms) for
    # the host to enqueue the timed call behind it, so the call's time is
    # device time, not launch latency
    buf = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    state = {"i": 0}

    def flush():
        state["i"] += 1
        buf.fill_(state["i"] & 255)
    return flush


def measure_config(cfg: int, args, stream, dev, local: int) -> dict:
    """One entry of the per-config table (1 GPU, same invocation as the
    headline): step time, tokens/s, rooflines and clocks."""
    from indexed_sparse_attention_indexer_gb300 import binding
    hbm, tfl, src = peaks()
    steps = max(3, min(args.steps, 20))
    n = max(3, min(args.steps, 10))
    entry = {"workload": W.CONFIGS[cfg]["name"]}
    if cfg == 4:
        c = W.CONFIGS[4]
        k_idx, latent = W.make_long_cache(c["S"], c["d"], c["seed"], dev)
        chunks = []
        n_chunks = c["S"] // c["T"]
        for ch in sorted({0, 7, 15, 23, n_chunks - 1}):
            ws = W.make_chunk(k_idx, latent, ch, c["T"], c["H_i"], c["K"], c["H"], c["seed"],
                              name=c["name"])
            cache = binding.Cache.of(ws)
            wsp = _workspace(ws, cache, dev)
            bufs = _outputs(ws, dev)
            tm = time_steps(_layer_step(ws, cache, wsp, bufs, stream), stream, max(3, steps // 4),
                            args.warmup, local)
            ms = tm["ms_local"] / max(3, steps // 4)
            mla, idxr = _prefill_rooflines(ws, cache, bufs, wsp, stream, 3, tfl, src)
            chunks.append({"chunk": ch, "history_end": (ch + 1) * c["T"], "ms_per_step": round(ms, 4),
                           "tokens_per_s": round(ws.T / (ms / 1e3), 1),
                           "roofline": mla, "indexer_roofline": idxr, "clocks": tm["clocks"]})
            del ws, cache, wsp, bufs
            torch.cuda.empty_cache()
        entry.update({"unit": UNIT, "chunk_tokens": c["T"], "chunks": chunks,
                      "note": "chunks sampled across the 32 of the sequence; tokens/s per chunk "
                              "falls as its causal history (indexer work) grows"})
        return entry
    ws = W.make_config(cfg, device=dev)
    cache = binding.Cache.of(ws)
    wsp = _workspace(ws, cache, dev)
    bufs = _outputs(ws, dev)
    decode = ws.mode == "decode"
    flush = _l2_flusher(dev) if cfg == 1 else None   # its 0.4 MB would otherwise sit in L2
    tm = time_steps(_layer_step(ws, cache, wsp, bufs, stream), stream, steps, args.warmup, local,
                    flush=flush)
    ms = tm["ms_local"] / steps
    ab = algorithmic_bytes(ws)
    gbs = ab["total"] / (ms / 1e3) / 1e9
    entry.update({"ms_per_step": round(ms, 5), "tokens_per_s": round(ws.T / (ms / 1e3), 1),
                  "unit": UNIT, "hbm_gbs_step": round(gbs, 1), "hbm_frac_step": round(gbs / hbm, 4),
                  "algorithmic_bytes_per_step": ab["total"], "clocks": tm["clocks"],
                  "gpu_launches_per_step": tm["launches"] / steps})
    if cfg == 1:
        entry["us_per_call"] = round(ms * 1e3, 2)
        entry["l2"] = "1 GB written before every timed call (the workload fits in L2)"
        entry["note"] = "latency-bound: 0.4 MB per call"
    if decode:
        span = cache.struct.s_max
        entry["roofline"] = _score_roofline(ws, cache, span, stream, dev, n, hbm, src)
    else:
        entry["roofline"], entry["indexer_roofline"] = _prefill_rooflines(
            ws, cache, bufs, wsp, stream, n, tfl, src)
    del ws, cache, wsp, bufs
    torch.cuda.empty_cache()
    return entry


def run_gpu(args):
    from indexed_sparse_attention_indexer_gb300 import binding

    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # seeded per config; each rank its own replica (--rows: a smaller decode batch
    # or a shorter prefill for profiling captures, never a bench line)
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
    # decode: every rank runs its own batch (replicas); prefill: the ranks
    # share the query rows of one sequence in zigzag segment pairs, each over
    # the whole (replicated) causal history
    parts = [ws] if (decode or world == 1) else prefill_parts(ws, world, rank)
    wsp = _workspace(max(parts, key=lambda p: p.T), cache, dev)
    part_bufs = [_outputs(p, dev) for p in parts]
    bufs = part_bufs[0]
    steps_of = [_layer_step(p, cache, wsp, b, stream) for p, b in zip(parts, part_bufs)]
    tm = time_steps(lambda: [f() for f in steps_of], stream, args.steps, args.warmup, local,
                    world)
    launches, clk = tm["launches"], tm["clocks"]
    ms = max_over_ranks(tm["ms_local"], world)
    ms_step = ms / args.steps
    rows_job = ws.T * (world if decode else 1)      # query tokens all ranks processed per step
    value = rows_job * args.steps / (ms / 1e3)

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
        roofline = _score_roofline(ws, cache, span, stream, dev, max(10, args.steps), hbm, src)
    else:
        # ---- prefill: both halves are dense contractions on the tensor cores;
        # the attention core dominates, the fused indexer is reported beside it
        nk = max(3, min(10, args.steps))
        roofline, extra["indexer_roofline"] = _prefill_rooflines(parts, cache, part_bufs, wsp,
                                                                 stream, nk, tfl, src)
    ab = algorithmic_bytes(ws)
    step_gbs = ab["total"] / (ms_step / 1e3) / 1e9

    # ---- end to end through the public API with host buffers ---------------
    e2e = run_e2e(parts, cache, wsp, decode, args, stream, dev)
    if world > 1:
        e2e["value"] = round(rows_job * args.steps / (max_over_ranks(e2e["ms_per_step"], world)
                                                      * args.steps / 1e3), 1)

    result = None
    if rank == 0:
        fl = algorithmic_flops(ws)
        result = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak" if decode else "strong",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded generators; integer-valued indexer inputs, N(0,1) latent)",
            "config": config_dict(ws, world),
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
    del wsp, bufs, part_bufs
    torch.cuda.empty_cache()
    plain = (args.config == 2 and not args.rows and tps == 1 and ws.latent_scale is None
             and not getattr(args, "k_mx_group", 0))
    if world == 1 and plain and not args.no_configs:
        # every workload of the table, measured in this same invocation
        table = {}
        for c in sorted(W.CONFIGS):
            if c == args.config:
                table[str(c)] = {"workload": wname, "ms_per_step": round(ms_step, 5),
                                 "tokens_per_s": round(value, 1), "unit": UNIT,
                                 "hbm_gbs_step": round(step_gbs, 1),
                                 "hbm_frac_step": round(step_gbs / hbm, 4),
                                 "roofline": roofline, "clocks": clk, "headline": True}
            else:
                table[str(c)] = measure_config(c, args, stream, dev, local)
        result["configs"] = table
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(ws, budget_s=args.cpu_seconds)
    barrier(world)
    return result


def config_dict(ws, world: int = 1) -> dict:
    """The ``config`` object of a line (shared by the GPU and reference arms)."""
    return {"workload": ws.name, "batch": ws.T, "history": int(ws.s_max),
            "indexer": f"{ws.H_i}x{ws.d}", "topk": ws.K, "mla_heads": ws.H,
            "parallelism": (f"replicas x{world} (batch shards, no collective)" if ws.mode == "decode"
                            else f"query-row shards x{world} (zigzag segment pairs, replicated cache, no collective)"),
            "l2": "inputs larger than L2 (index keys and latent rows streamed per step)"}


def run_e2e(parts, cache, wsp, decode, args, stream, dev):
    """Same metric through binding.indexed_attention with the per-step inputs
    (q_idx, w, q) copied from pinned host memory and the output read back every
    step; the caches stay resident as they would in serving.  As a server
    would, the copies of one step overlap the computation of its neighbour:
    two device input/output sets alternate, host-to-device copies run on one
    side stream and device-to-host reads on another, ordered by events.
    ``parts``: the step's calls (one workload, or a rank's prefill segments)."""
    from indexed_sparse_attention_indexer_gb300 import binding
    host = [(p.q_idx.cpu().pin_memory(), p.w.cpu().pin_memory(), p.q.cpu().pin_memory(),
             [torch.empty((p.T, p.H, W.D_LATENT), dtype=torch.bfloat16).pin_memory()
              for _ in range(2)]) for p in parts]
    sets = [[(torch.empty_like(p.q_idx), torch.empty_like(p.w), torch.empty_like(p.q),
              torch.empty((p.T, p.H, W.D_LATENT), dtype=torch.bfloat16, device=dev))
             for p in parts] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    computed = [ev(), ev()]     # step on set i finished computing
    read_back = [ev(), ev()]    # its output has been copied to the host
    for e in computed + read_back:
        e.record(stream)

    def step(k):
        i = k & 1
        landed = ev()
        with torch.cuda.stream(s_in):
            s_in.wait_event(computed[i])          # step k-2 no longer reads set i
            for (h_qidx, h_w, h_q, _), (d_qidx, d_w, d_q, _) in zip(host, sets[i]):
                d_qidx.copy_(h_qidx, non_blocking=True)
                d_w.copy_(h_w, non_blocking=True)
                d_q.copy_(h_q, non_blocking=True)
            landed.record(s_in)
        stream.wait_event(landed)
        stream.wait_event(read_back[i])           # step k-2's output was read
        for p, (d_qidx, d_w, d_q, d_out) in zip(parts, sets[i]):
            if p.tokens_per_seq > 1:
                binding.indexed_attention_multi(d_qidx, d_w, d_q, cache, p.tokens_per_seq, p.K,
                                                p.scale, out=d_out, workspace=wsp, want_lse=False,
                                                want_idx=False, stream=stream)
            else:
                binding.indexed_attention(d_qidx, d_w, d_q, cache, p.K, p.scale, decode,
                                          p.q_offset, out=d_out, workspace=wsp, want_lse=False,
                                          want_idx=False, stream=stream)
        computed[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[i])
            for (_, _, _, h_out), (_, _, _, d_out) in zip(host, sets[i]):
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
    bi = sum(h[0].numel() * 2 + h[1].numel() * 4 + h[2].numel() * 2 for h in host)
    bo = sum(h[3][0].numel() * 2 for h in host)
    rows = sum(p.T for p in parts)
    return {"value": round(rows * args.steps / (ms / 1e3), 1), "unit": UNIT,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": round(ms / args.steps, 5),
            "note": "caches resident; per-step queries in, attention output out; copies of a "
                    "step overlap its neighbour's computation (two buffer sets, side streams)"}


# ----------------------------------------------------------------------------
# the oracle (CPU baseline / reference arm)
# ----------------------------------------------------------------------------

def _row_bundle(ws, r: int):
    """A CPU workload with only what row r of ``ws`` reads: its sequence (its
    pages gathered in order, for a paged cache; the oracle's paged and
    contiguous results are pinned equal) or, for prefill, the causal prefix."""
    d = ws.q.device
    if ws.mode == "decode":
        T = ws.tokens_per_seq
        b = r // T
        rows = slice(b * T, b * T + T)
        L = int(ws.seq_lens[b])
        if ws.block_table is not None:
            npg = max(1, -(-L // ws.page_size))
            pages = ws.block_table[b, :npg].to(torch.int64)

            def seq(x):
                if x is None:
                    return None
                raw = x.view(torch.uint8) if x.element_size() == 1 else x   # float8 as bytes
                y = raw[pages].reshape((1, -1) + tuple(x.shape[2:]))
                return y.view(x.dtype) if raw is not x else y
        else:
            def seq(x):
                return None if x is None else x[b:b + 1]
        sub = W.Workload(ws.name, "decode", ws.H_i, ws.d, ws.K, ws.H, ws.scale, ws.q_idx[rows],
                         ws.w[rows], ws.q[rows], seq(ws.k_idx), seq(ws.k_scale), seq(ws.latent),
                         torch.tensor([L], dtype=torch.int32, device=d), None, 0, 0,
                         dict(ws.meta), seq(ws.latent_scale))
        return sub.to("cpu"), ("multi", r % T, T) if T > 1 else ("decode", 0, 1)
    n = ws.q_offset + r + 1
    sub = W.Workload(ws.name, "prefill", ws.H_i, ws.d, ws.K, ws.H, ws.scale, ws.q_idx[r:r + 1],
                     ws.w[r:r + 1], ws.q[r:r + 1], ws.k_idx[:, :n],
                     None if ws.k_scale is None else ws.k_scale[:, :n], ws.latent[:, :n],
                     torch.tensor([n], dtype=torch.int32, device=d), None, 0, n - 1, {},
                     None if ws.latent_scale is None else ws.latent_scale[:, :n])
    return sub.to("cpu"), ("prefill", 0, 1)


def _oracle_one(bundle) -> None:
    import oracle
    sub, (kind, t, T) = bundle
    if kind == "decode":
        oracle.decode_row(sub, 0)
    elif kind == "multi":
        oracle.multi_token_row(sub, t, T)
    else:
        oracle.prefill_row(sub, 0)


_POOL_BUNDLES = None


def _pool_init(bundles):
    global _POOL_BUNDLES
    _POOL_BUNDLES = bundles


def _pool_task(i: int) -> int:
    _oracle_one(_POOL_BUNDLES[i % len(_POOL_BUNDLES)])
    return 1


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _sample_rows(ws, n: int):
    """Rows spread evenly over the batch (decode) or the prefill's tokens."""
    n = max(1, min(n, ws.T))
    return sorted({int(i * ws.T // n) for i in range(n)})


def oracle_throughput(ws, budget_s: float, cores: int) -> dict:
    """Oracle rows per second over a bounded sample of the workload's rows:
    first one core, then ``cores`` worker processes (spawned: no GPU state is
    inherited) sharing the sample through shared memory.  The sample's host
    copies are made before either timed region."""
    rows = _sample_rows(ws, 2 * cores)
    bundles = [_row_bundle(ws, r) for r in rows]
    for sub, _ in bundles:
        for f in ("q_idx", "w", "q", "k_idx", "k_scale", "latent", "latent_scale", "seq_lens"):
            x = getattr(sub, f)
            if x is not None:
                x.share_memory_()
    # one core
    t_one = 0.3 * budget_s
    done, t0 = 0, time.perf_counter()
    while True:
        _oracle_one(bundles[done % len(bundles)])
        done += 1
        if time.perf_counter() - t0 >= t_one:
            break
    el1 = time.perf_counter() - t0
    rate1 = done / el1
    res = {"single_core": {"value": round(rate1, 3), "rows": done, "seconds": round(el1, 2)}}
    if cores > 1:
        # spawned workers (never forked from a process that has touched the
        # GPU); a worker that dies breaks the pool with an error, it never
        # hangs the run
        import concurrent.futures as cf
        import torch.multiprocessing as tmp
        with cf.ProcessPoolExecutor(cores, mp_context=tmp.get_context("spawn"),
                                    initializer=_pool_init, initargs=(bundles,)) as pool:
            list(pool.map(_pool_task, range(cores), timeout=600))      # warm: imports, first touch
            n_tasks = max(cores, int(rate1 * cores * 0.7 * budget_s * 0.8))
            t0 = time.perf_counter()
            done = sum(pool.map(_pool_task, range(n_tasks), timeout=600))
            el = time.perf_counter() - t0
        res["all_cores"] = {"value": round(done / el, 3), "rows": done, "seconds": round(el, 2)}
    res["sample_rows"] = len(rows)
    return res


def cpu_baseline(ws, budget_s: float = 10.0) -> dict:
    cores = host_cores()
    r = oracle_throughput(ws, budget_s, cores)
    best = r.get("all_cores", r["single_core"])
    used = cores if "all_cores" in r else 1
    return {"value": best["value"], "unit": UNIT, "cores": used, "kind": "oracle",
            "single_core_value": r["single_core"]["value"], "nproc": cores,
            "sample": f"{r['sample_rows']} of {ws.T} query rows of the same workload, spread "
                      f"evenly, cycled: {best['rows']} rows in {best['seconds']} s on {used} "
                      f"worker processes (fp64 numpy oracle, single-threaded BLAS each); "
                      f"one core: {r['single_core']['rows']} rows in "
                      f"{r['single_core']['seconds']} s; host copies made before timing"}


def run_reference(args):
    """The baseline arm: the CPU oracle on a bounded sample, same metric and config."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return None
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    if args.config == 4:
        raise SystemExit("--impl reference takes the single-batch configs (1, 2, 3, 5)")
    ws = W.make_config(args.config, device=dev, k_mx_group=getattr(args, "k_mx_group", 0),
                       latent_fp8=getattr(args, "latent_fp8", False),
                       tokens_per_seq=args.tokens_per_seq)
    cores = host_cores()
    # each step is a bounded sample: the whole run stays within --cpu-seconds
    per_step = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    r = oracle_throughput(ws, per_step * (args.steps + args.warmup), cores)
    best = r.get("all_cores", r["single_core"])
    used = cores if "all_cores" in r else 1
    value = best["value"]
    sample = (f"{r['sample_rows']} of {ws.T} query rows spread evenly, cycled: {best['rows']} rows "
              f"in {best['seconds']} s on {used} worker processes (fp64 numpy oracle, "
              f"single-threaded BLAS each); one core {r['single_core']['value']} rows/s")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * ws.T / value, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded generators as the GPU arm)",
            "config": config_dict(ws, world),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": used,
                             "kind": "oracle", "sample": sample,
                             "single_core_value": r["single_core"]["value"], "nproc": cores},
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


def relaunch_ranks(n: int) -> int:
    """``--gpus N`` without an outside launcher: start N ranks of this script
    (one per local GPU, NCCL for the timing barrier) through torch's launcher
    and return its exit status; rank 0 prints the line."""
    import socket
    if torch.cuda.device_count() < n:
        print(json.dumps({"error": f"--gpus {n}: only {torch.cuda.device_count()} GPUs visible"}))
        return 2
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__),
           *sys.argv[1:]]
    return subprocess.run(cmd).returncode


def run_appends():
    """The two cache-append kernels at cache scale, HBM-bound: MXFP8
    quantisation of the 64x32768 decode batch's index keys (bf16 in, E4M3 +
    E8M0 out) and the FP8 append of its latent rows (bf16 in, E4M3 + five
    fp32 tile scales out).  Bytes counted once each way; CUDA events, best of
    five after warm-up (not a bench line)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from indexed_sparse_attention_indexer_gb300 import binding
    binding.load()
    stream = torch.cuda.current_stream()
    hbm, _, src = peaks()
    rows, d, G = 64 * 32768, 128, 32
    keys = W.make_mx_input(rows, d, seed=5, device=dev, special=False)
    codes = torch.empty((rows, d), dtype=torch.float8_e4m3fn, device=dev)
    sc = torch.empty((rows, d // G), dtype=torch.uint8, device=dev)
    q_ms = time_alone(lambda: binding.mxfp8_quantize(keys, G, codes=codes, scales=sc,
                                                     stream=stream), stream, 10)
    q_bytes = rows * (2 * d + d + d // G)
    del keys, codes, sc
    lat = torch.randn((rows, W.D_QK), device=dev).to(torch.bfloat16)
    lc = torch.empty((rows, W.D_QK), dtype=torch.float8_e4m3fn, device=dev)
    ls = torch.empty((rows, 5), dtype=torch.float32, device=dev)
    a_ms = time_alone(lambda: binding.latent_fp8_append(lat, codes=lc, scales=ls, stream=stream),
                      stream, 10)
    a_bytes = rows * (2 * W.D_QK + W.D_QK + 5 * 4)
    out = []
    for name, ms, b in (("mxfp8_quantize", q_ms, q_bytes), ("latent_fp8_append", a_ms, a_bytes)):
        gbs = b / (ms / 1e3) / 1e9
        out.append({"kernel": name, "rows": rows, "bytes": b, "ms": round(ms, 4),
                    "gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4), "peak_source": src})
    print(json.dumps({"probe": "cache_appends", "results": out}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", type=int, default=2, choices=sorted(W.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="headline line only (skip the per-config table)")
    ap.add_argument("--crossover", action="store_true",
                    help="measurement: dense vs sparse attention as the history grows (not a bench line)")
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
    ap.add_argument("--appends", action="store_true",
                    help="measurement: the two cache-append kernels at cache scale (not a bench line)")
    ap.add_argument("--rows", type=int, default=None,
                    help="profiling aid: a smaller decode batch or a shorter prefill (the printed "
                         "line is not a bench line)")
    args = ap.parse_args()
    if args.crossover:
        run_crossover()
        return
    if args.mx_scan:
        run_mx_scan()
        return
    if args.appends:
        run_appends()
        return
    args.warmup = max(3, args.warmup)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch_ranks(args.gpus))
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
