"""Seeded synthetic workloads for the indexed sparse attention layer.

This module only draws random numbers and lays them out in the buffers the
library reads.  None of the scoring, selection or attention arithmetic lives
here: the CUDA path (through the binding) and the CPU oracle (in the tests and
the bench's CPU leg) both take their inputs from these functions, and nothing
else is shared between them.

Value recipe (shapes and distributions of the five workloads the layer is
measured on):

* index queries ``q_idx`` and index keys ``k_idx``: integers drawn uniformly
  from {-3..3}, stored in bf16 (keys may instead be FP8 E4M3, which holds these
  integers exactly, with one positive power-of-two scale 2^e, e in {-4..0}, per
  token).  Every dot product of two such vectors is an exact small integer, so
  fp32 scores are exact in any summation order.
* MXFP8 index keys (the microscaled variant): E4M3 codes holding integers
  from {-3..3} plus one E8M0 scale byte per group of G (32 unless stated)
  elements, drawn uniformly from {125, 126, 127} (scales 1/4, 1/2, 1).  With
  integer index queries (whose MXFP8 quantisation is exact) every dot product
  is a multiple of 1/4 below 2^11 and the weighted head sums stay far below
  the 2^15 where fp32 would start to round them.
* inputs of the MXFP8 quantiser: bf16 normal rows with a per-row magnitude
  exp(U(-8, 8)), four outlier channels x32, and special rows (all zero, bf16
  subnormals, magnitudes near 2^120, exact powers of two, group maxima with
  mantissa 1.875 that saturate at 448); the group-size scan also uses rows
  whose channels carry their own magnitudes exp(U(-5, 5)).
* FP8 latent cache (the quantised KV cache variant): E4M3 codes drawn as
  bytes with a random sign, exponent field uniform in {4..10} and mantissa
  uniform in {0..7} (magnitudes 1/8 .. 15), and one fp32 scale per position
  and tile of 128 dims (5 tiles: the rope dims are the fifth) uniform in
  [0.02, 0.2); drawn where the bf16 latent would be, codes then scales.
* head weights ``w``: uniform [0,1) rounded down to a multiple of 2^-7, so that
  every partial sum of ``w_h * relu(u_h)`` is a multiple of 2^-7 below 2^24
  and hence exact in fp32 whatever the order.
* latent cache rows (512 latent + 64 rope dims): bf16 N(0,1).
* attention queries ``q``: bf16 N(0,1)/sqrt(576); softmax scale 1/sqrt(576).
* varlen decode: lengths floor(exp(U(ln 1024, ln 131072))), 64-token pages,
  physical page ids a random permutation.

Draw order for one generator: q_idx, k_idx, (k_scale), w, q, latent, then the
page permutation.  A varlen workload draws its lengths first, from the same
generator, because they size every other buffer.  A chunked prefill draws the
sequence's cache (k_idx, latent) from ``seed`` and each query chunk from its
own stream ``seed + 1_000_003 * (chunk + 1)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

D_LATENT = 512          # value / latent width of one cache row
D_ROPE = 64             # rope part of one cache row
D_QK = D_LATENT + D_ROPE  # key width of one cache row (576)

WEIGHT_GRID = 128       # head weights are multiples of 1/WEIGHT_GRID


@dataclass
class Workload:
    """One batch of inputs for the layer.

    Cache layout: contiguous caches are ``[B, S_max, ...]`` (``block_table`` is
    None); paged caches are pools ``[P, page_size, ...]`` addressed through
    ``block_table[B, max_pages]`` (unused entries are -1).  Decode rows are one
    query token per sequence (T == B) and row b sees positions
    ``0 .. seq_lens[b]-1``.  Prefill is one sequence (B == 1); query token t
    sits at position ``q_offset + t`` and sees positions ``0 .. q_offset+t``.
    """

    name: str
    mode: str                      # "decode" or "prefill"
    H_i: int
    d: int
    K: int
    H: int
    scale: float
    q_idx: torch.Tensor            # [T, H_i, d] bf16
    w: torch.Tensor                # [T, H_i] fp32
    q: torch.Tensor                # [T, H, 576] bf16
    k_idx: torch.Tensor            # [B, S_max, d] or [P, page, d]; bf16 / fp8 e4m3
    k_scale: Optional[torch.Tensor]  # same leading shape as k_idx minus d, fp32, or None
    latent: torch.Tensor           # [B, S_max, 576] or [P, page, 576] bf16
    seq_lens: torch.Tensor         # [B] int32
    block_table: Optional[torch.Tensor] = None  # [B, max_pages] int32
    page_size: int = 0
    q_offset: int = 0
    meta: dict = field(default_factory=dict)
    latent_scale: Optional[torch.Tensor] = None   # FP8 latent: fp32 [..., 5] tile scales

    @property
    def T(self) -> int:
        return int(self.q_idx.shape[0])

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def tokens_per_seq(self) -> int:
        """Decode query rows per sequence (1, or T for a multi-token step)."""
        return int(self.meta.get("tokens_per_seq", 1))

    @property
    def paged(self) -> bool:
        return self.block_table is not None

    @property
    def s_max(self) -> int:
        """Rows per sequence in a contiguous cache; max_pages*page for a paged one."""
        if self.paged:
            return int(self.block_table.shape[1]) * self.page_size
        return int(self.k_idx.shape[1])

    def to(self, device) -> "Workload":
        def mv(x):
            return None if x is None else x.to(device)
        return Workload(self.name, self.mode, self.H_i, self.d, self.K, self.H, self.scale,
                        mv(self.q_idx), mv(self.w), mv(self.q), mv(self.k_idx), mv(self.k_scale),
                        mv(self.latent), mv(self.seq_lens), mv(self.block_table),
                        self.page_size, self.q_offset, dict(self.meta), mv(self.latent_scale))

    def input_bytes(self) -> int:
        n = 0
        for x in (self.q_idx, self.w, self.q, self.k_idx, self.k_scale, self.latent,
                  self.latent_scale, self.seq_lens, self.block_table):
            if x is not None:
                n += x.numel() * x.element_size()
        return n


# ----------------------------------------------------------------------------
# elementary draws
# ----------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


_CHUNK = 1 << 24  # elements per draw, to bound temporary fp32 memory


def _int_values(shape, g, device, dtype=torch.bfloat16) -> torch.Tensor:
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1) if dtype != torch.float8_e4m3fn else None
    n = out.numel()
    if dtype == torch.float8_e4m3fn:
        tmp = torch.empty(n, dtype=torch.float8_e4m3fn, device=device)
        for s in range(0, n, _CHUNK):
            e = min(n, s + _CHUNK)
            tmp[s:e] = torch.randint(-3, 4, (e - s,), generator=g, device=device).to(torch.float32).to(dtype)
        return tmp.view(shape)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        flat[s:e] = torch.randint(-3, 4, (e - s,), generator=g, device=device).to(dtype)
    return out


def _normal_bf16(shape, g, device, std: float = 1.0) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = out.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:e] = x.to(torch.bfloat16)
    return out


def _weights(shape, g, device) -> torch.Tensor:
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return torch.floor(u * WEIGHT_GRID) / WEIGHT_GRID


def _pow2_scales(shape, g, device) -> torch.Tensor:
    e = torch.randint(0, 5, shape, generator=g, device=device)
    return torch.pow(torch.tensor(2.0, device=device), -e.to(torch.float32))


def _e8m0_bytes(shape, g, device, lo: int = 125, hi: int = 127) -> torch.Tensor:
    return torch.randint(lo, hi + 1, shape, generator=g, device=device).to(torch.uint8)


LATENT_TILES = 5   # tiles of 128 dims per latent row; the 64 rope dims are the fifth


def _latent_fp8(shape, g, device):
    """E4M3 latent codes [*shape, 576] (as bytes, viewed as float8) and fp32
    tile scales [*shape, 5]."""
    n = 1
    for v in shape:
        n *= v
    out = torch.empty((n * D_QK,), dtype=torch.uint8, device=device)
    for s in range(0, n * D_QK, _CHUNK):
        e = min(n * D_QK, s + _CHUNK)
        sign = torch.randint(0, 2, (e - s,), generator=g, device=device)
        expo = torch.randint(4, 11, (e - s,), generator=g, device=device)
        mant = torch.randint(0, 8, (e - s,), generator=g, device=device)
        out[s:e] = (sign * 128 + expo * 8 + mant).to(torch.uint8)
    codes = out.view(tuple(shape) + (D_QK,)).view(torch.float8_e4m3fn)
    scales = torch.empty(tuple(shape) + (LATENT_TILES,), dtype=torch.float32,
                         device=device).uniform_(0.02, 0.2, generator=g)
    return codes, scales


def loguniform_lengths(B: int, lo: int, hi: int, g, device) -> torch.Tensor:
    u = torch.rand(B, generator=g, device=device, dtype=torch.float64)
    L = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return L.clamp(lo, hi).to(torch.int32)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

def make_decode(B: int, S: int, H_i: int, d: int, K: int, H: int, seed: int = 0,
                device="cpu", lengths: Optional[Sequence[int]] = None,
                loguniform: Optional[tuple] = None, page_size: int = 0,
                k_fp8: bool = False, scale: Optional[float] = None,
                q_std: Optional[float] = None, name: str = "decode",
                tokens_per_seq: int = 1, k_mx_group: int = 0,
                latent_fp8: bool = False) -> Workload:
    """Decode batch: one query token per sequence, or ``tokens_per_seq`` (T)
    candidate tokens per sequence for a multi-token step (query rows come T to
    a sequence; the candidates' keys are the last T positions of its history).

    ``S`` is the history length of every sequence unless ``lengths`` gives them
    or ``loguniform=(lo, hi)`` draws them.  ``page_size > 0`` stores the caches
    as page pools behind a randomly permuted block table.  ``k_mx_group > 0``
    stores the index keys as MXFP8 (E4M3 codes, one E8M0 byte per group of
    that many elements in ``k_scale``); ``latent_fp8`` stores the latent cache
    as E4M3 codes with per-tile fp32 scales (``latent_scale``).
    """
    R = B * tokens_per_seq
    g = _gen(seed, device)
    if loguniform is not None:
        L = loguniform_lengths(B, loguniform[0], loguniform[1], g, device).cpu()
    elif lengths is not None:
        L = torch.tensor(list(lengths), dtype=torch.int32)
        assert L.numel() == B
    else:
        L = torch.full((B,), S, dtype=torch.int32)
    if page_size > 0:
        pages_per = [(int(l) + page_size - 1) // page_size for l in L]
        n_pages = max(1, sum(pages_per))
        rows_shape = (n_pages, page_size)
    else:
        s_max = max(1, int(L.max()) if L.numel() else 1)
        rows_shape = (B, s_max)
    kdt = torch.float8_e4m3fn if (k_fp8 or k_mx_group) else torch.bfloat16
    q_idx = _int_values((R, H_i, d), g, device)
    k_idx = _int_values(rows_shape + (d,), g, device, kdt)
    if k_mx_group:
        assert d % k_mx_group == 0
        k_scale = _e8m0_bytes(rows_shape + (d // k_mx_group,), g, device)
    else:
        k_scale = _pow2_scales(rows_shape, g, device) if k_fp8 else None
    w = _weights((R, H_i), g, device)
    std = (1.0 / math.sqrt(D_QK)) if q_std is None else q_std
    q = _normal_bf16((R, H, D_QK), g, device, std)
    latent_scale = None
    if latent_fp8:
        latent, latent_scale = _latent_fp8(rows_shape, g, device)
    else:
        latent = _normal_bf16(rows_shape + (D_QK,), g, device)
    block_table = None
    if page_size > 0:
        perm = torch.randperm(n_pages, generator=g, device=device).to(torch.int32).cpu()
        max_pages = max(1, max(pages_per) if pages_per else 1)
        block_table = torch.full((B, max_pages), -1, dtype=torch.int32)
        c = 0
        for b, npg in enumerate(pages_per):
            block_table[b, :npg] = perm[c:c + npg]
            c += npg
        block_table = block_table.to(device)
    return Workload(name=name, mode="decode", H_i=H_i, d=d, K=K, H=H,
                    scale=(1.0 / math.sqrt(D_QK)) if scale is None else scale,
                    q_idx=q_idx, w=w, q=q, k_idx=k_idx, k_scale=k_scale, latent=latent,
                    seq_lens=L.to(device), block_table=block_table, page_size=page_size,
                    meta={"tokens_per_seq": tokens_per_seq} if tokens_per_seq != 1 else {},
                    latent_scale=latent_scale)


def make_prefill(T: int, S: int, H_i: int, d: int, K: int, H: int, seed: int = 0,
                 device="cpu", q_offset: int = 0, scale: Optional[float] = None,
                 q_std: Optional[float] = None, name: str = "prefill",
                 k_mx_group: int = 0, latent_fp8: bool = False) -> Workload:
    """Causal prefill of one sequence: query tokens q_offset .. q_offset+T-1
    against a cache of S >= q_offset+T rows, all from one generator
    (``k_mx_group``: MXFP8 index keys as in ``make_decode``)."""
    assert S >= q_offset + T
    g = _gen(seed, device)
    q_idx = _int_values((T, H_i, d), g, device)
    k_idx = _int_values((1, S, d), g, device,
                        torch.float8_e4m3fn if k_mx_group else torch.bfloat16)
    k_scale = _e8m0_bytes((1, S, d // k_mx_group), g, device) if k_mx_group else None
    w = _weights((T, H_i), g, device)
    std = (1.0 / math.sqrt(D_QK)) if q_std is None else q_std
    q = _normal_bf16((T, H, D_QK), g, device, std)
    latent_scale = None
    if latent_fp8:
        latent, latent_scale = _latent_fp8((1, S), g, device)
    else:
        latent = _normal_bf16((1, S, D_QK), g, device)
    return Workload(name=name, mode="prefill", H_i=H_i, d=d, K=K, H=H,
                    scale=(1.0 / math.sqrt(D_QK)) if scale is None else scale,
                    q_idx=q_idx, w=w, q=q, k_idx=k_idx, k_scale=k_scale, latent=latent,
                    seq_lens=torch.tensor([S], dtype=torch.int32, device=device),
                    q_offset=q_offset, latent_scale=latent_scale)


def make_mx_input(n: int, d: int, seed: int = 0, device="cpu", special: bool = True,
                  row_spread: float = 8.0, channel_spread: float = 0.0) -> torch.Tensor:
    """bf16 rows [n, d] for the MXFP8 quantiser: normal values with a per-row
    magnitude exp(U(-row_spread, row_spread)) and four outlier channels x32
    (with ``channel_spread`` > 0 every channel is scaled instead by its own
    exp(U(-channel_spread, channel_spread)), drawn after the outlier channels);
    with ``special`` and n >= 8 the first rows are special: all zero, bf16
    subnormals, magnitudes near 2^120, exact powers of two, and groups whose
    largest magnitude has mantissa 1.875 (they saturate at 448 after scaling)."""
    g = _gen(seed, device)
    x = torch.empty((n, d), device=device, dtype=torch.bfloat16)
    mag = torch.exp(torch.empty((n, 1), device=device).uniform_(-row_spread, row_spread,
                                                                 generator=g))
    ch = torch.randperm(d, generator=g, device=device)[:4]
    boost = torch.ones(d, device=device)
    boost[ch] = 32.0
    if channel_spread > 0:
        boost = torch.exp(torch.empty(d, device=device).uniform_(-channel_spread, channel_spread,
                                                                  generator=g))
    step = max(1, _CHUNK // max(1, d))
    for s in range(0, n, step):
        e = min(n, s + step)
        x[s:e] = (torch.randn((e - s, d), generator=g, device=device) * mag[s:e] * boost).to(
            torch.bfloat16)
    if not special or n < 8:
        return x
    x = x.float()
    if n >= 8:
        x[0] = 0.0
        x[1] = torch.randn(d, generator=g, device=device) * 2.0 ** -130
        x[2] = torch.randn(d, generator=g, device=device) * 2.0 ** 118
        e = torch.randint(-20, 20, (d,), generator=g, device=device).to(torch.float32)
        x[3] = torch.pow(2.0, e) * torch.where(torch.rand(d, generator=g, device=device) < 0.5,
                                               -1.0, 1.0)
        x[4] = torch.randn(d, generator=g, device=device)
        m = x[4, ::16].numel()
        x[4, ::16] = 1.875 * torch.pow(2.0, torch.randint(-5, 5, (m,), generator=g,
                                                           device=device).to(torch.float32))
        x[5] = -x[4]
    return x.to(torch.bfloat16)


CHUNK_STREAM = 1_000_003


def make_long_cache(S: int, d: int, seed: int = 0, device="cpu"):
    """Cache of one long sequence for chunked prefill: (k_idx [1,S,d], latent [1,S,576])."""
    g = _gen(seed, device)
    k_idx = _int_values((1, S, d), g, device)
    latent = _normal_bf16((1, S, D_QK), g, device)
    return k_idx, latent


def make_chunk(k_idx: torch.Tensor, latent: torch.Tensor, chunk: int, T: int,
               H_i: int, K: int, H: int, seed: int = 0,
               name: str = "chunked-prefill") -> Workload:
    """Query chunk ``chunk`` (tokens chunk*T .. chunk*T+T-1) of a long sequence."""
    device = k_idx.device
    d = int(k_idx.shape[-1])
    S = int(k_idx.shape[1])
    g = _gen(seed + CHUNK_STREAM * (chunk + 1), device)
    q_idx = _int_values((T, H_i, d), g, device)
    w = _weights((T, H_i), g, device)
    q = _normal_bf16((T, H, D_QK), g, device, 1.0 / math.sqrt(D_QK))
    return Workload(name=name, mode="prefill", H_i=H_i, d=d, K=K, H=H,
                    scale=1.0 / math.sqrt(D_QK), q_idx=q_idx, w=w, q=q,
                    k_idx=k_idx, k_scale=None, latent=latent,
                    seq_lens=torch.tensor([S], dtype=torch.int32, device=device),
                    q_offset=chunk * T, meta={"chunk": chunk})


# ----------------------------------------------------------------------------
# the five measured workloads
# ----------------------------------------------------------------------------

CONFIGS = {
    1: dict(name="decode-s2048-hi4x64-k128-h16", mode="decode", B=1, S=2048, H_i=4, d=64,
            K=128, H=16, seed=0),
    2: dict(name="decode-b64-s32768-hi64x128-k2048-h128", mode="decode", B=64, S=32768,
            H_i=64, d=128, K=2048, H=128, seed=0),
    3: dict(name="prefill-t8192-hi64x128-k2048-h128", mode="prefill", T=8192, S=8192,
            H_i=64, d=128, K=2048, H=128, seed=0),
    4: dict(name="chunked-prefill-s131072-c4096-hi64x128-k2048-h128", mode="chunked",
            S=131072, T=4096, H_i=64, d=128, K=2048, H=128, seed=0),
    5: dict(name="paged-decode-b128-loguniform-fp8keys-k2048-h128", mode="decode", B=128,
            S=131072, lo=1024, hi=131072, H_i=64, d=128, K=2048, H=128, page_size=64,
            seed=7),
}


def make_config(cfg: int, device="cpu", chunk: int = 0, rows: int | None = None,
                tokens_per_seq: int = 1, k_mx_group: int = 0,
                latent_fp8: bool = False) -> Workload:
    """The named workload; ``rows`` shrinks a decode batch (same shapes per
    sequence, fewer sequences) or a prefill (fewer tokens) for profiling
    captures that must stay small;
    ``tokens_per_seq`` turns a decode workload into a multi-token step;
    ``k_mx_group`` stores the 64x128-head decode workload's index keys as MXFP8;
    ``latent_fp8`` stores its latent cache as FP8 with per-tile scales."""
    c = CONFIGS[cfg]
    if tokens_per_seq != 1 and cfg not in (1, 2, 5):
        raise ValueError("tokens_per_seq applies to the decode workloads only")
    if rows is not None and cfg not in (1, 2, 3, 5):
        raise ValueError("rows applies to the decode workloads and the prefill")
    if (k_mx_group or latent_fp8) and cfg != 2:
        raise ValueError("MXFP8 keys and the FP8 latent cache apply to the 64x128-head "
                         "contiguous decode workload only")
    if cfg in (1, 2):
        return make_decode(rows or c["B"], c["S"], c["H_i"], c["d"], c["K"], c["H"], c["seed"],
                           device=device,
                           name=c["name"] + ("-mxfp8" if k_mx_group else "")
                           + ("-fp8latent" if latent_fp8 else ""),
                           tokens_per_seq=tokens_per_seq, k_mx_group=k_mx_group,
                           latent_fp8=latent_fp8)
    if cfg == 3:     # rows: a shorter prefill (T = S = rows) for small profiling captures
        T = rows or c["T"]
        return make_prefill(T, rows or c["S"], c["H_i"], c["d"], c["K"], c["H"], c["seed"],
                            device=device, name=c["name"])
    if cfg == 4:
        k_idx, latent = make_long_cache(c["S"], c["d"], c["seed"], device)
        return make_chunk(k_idx, latent, chunk, c["T"], c["H_i"], c["K"], c["H"], c["seed"],
                          name=c["name"])
    if cfg == 5:
        return make_decode(rows or c["B"], 0, c["H_i"], c["d"], c["K"], c["H"], c["seed"],
                           device=device, loguniform=(c["lo"], c["hi"]),
                           page_size=c["page_size"], k_fp8=True, name=c["name"],
                           tokens_per_seq=tokens_per_seq)
    raise ValueError(cfg)
