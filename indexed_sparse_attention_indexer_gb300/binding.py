"""ctypes binding of libdsi (include/dsi.h): argument marshalling only.

Every function here hands device pointers of torch tensors to the C ABI and
allocates the outputs with torch; all computation happens in the library's
CUDA kernels.  A missing library raises ``RuntimeError`` — there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIBS = {}

DSI_OK, DSI_ERR_INVALID_ARG, DSI_ERR_UNSUPPORTED, DSI_ERR_CUDA = 0, 1, 2, 3
DSI_ERR_TIMEOUT, DSI_ERR_BOUNDS, DSI_ERR_WORKSPACE = 4, 5, 6
DSI_BF16, DSI_FP8_E4M3, DSI_MXFP8_E4M3 = 0, 1, 2
D_QK, D_LATENT = 576, 512

c_void_p, c_int32, c_int64, c_float, c_size_t = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.c_float, ctypes.c_size_t)


class DsiCache(ctypes.Structure):
    """Mirror of ``struct dsi_cache``."""
    _fields_ = [("k_idx", c_void_p), ("k_dtype", c_int32), ("d", c_int32), ("k_scale", c_void_p),
                ("latent", c_void_p), ("block_table", c_void_p), ("page_size", c_int32),
                ("max_pages", c_int32), ("seq_lens", c_void_p), ("batch", c_int32),
                ("s_max", c_int64), ("num_pages", c_int64), ("k_group", c_int32),
                ("latent_dtype", c_int32), ("latent_scale", c_void_p)]


# name -> (restype, argtypes); the exported surface of include/dsi.h
SIGNATURES = {
    "dsi_index_score": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(DsiCache), c_int32, c_int32,
                                  c_int32, c_int64, c_void_p, c_int64, c_void_p]),
    "dsi_topk": (c_int32, [c_void_p, c_int64, c_int32, c_void_p, c_int64, c_int32, c_void_p,
                           c_void_p, c_void_p]),
    "dsi_index_topk_prefill": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(DsiCache), c_int32,
                                         c_int32, c_int64, c_int32, c_void_p, c_void_p,
                                         c_void_p]),
    "dsi_sparse_mla_decode": (c_int32, [c_void_p, ctypes.POINTER(DsiCache), c_void_p, c_int32,
                                        c_int32, c_int32, c_float, c_void_p, c_void_p, c_void_p,
                                        c_size_t, c_void_p]),
    "dsi_sparse_mla_prefill": (c_int32, [c_void_p, ctypes.POINTER(DsiCache), c_void_p, c_int32,
                                         c_int32, c_int32, c_int64, c_float, c_void_p, c_void_p,
                                         c_void_p, c_size_t, c_void_p]),
    "dsi_indexed_attention": (c_int32, [c_void_p, c_void_p, c_void_p, ctypes.POINTER(DsiCache),
                                        c_int32, c_int32, c_int32, c_int32, c_int64, c_float,
                                        c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_size_t, c_void_p]),
    "dsi_indexed_attention_multi": (c_int32, [c_void_p, c_void_p, c_void_p, ctypes.POINTER(DsiCache),
                                              c_int32, c_int32, c_int32, c_int32, c_float, c_void_p,
                                              c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                              c_void_p]),
    "dsi_indexed_attention_static": (c_int32, [c_void_p, c_void_p, c_void_p,
                                               ctypes.POINTER(DsiCache), c_int32, c_int32,
                                               c_int32, c_int32, c_int64, c_float, c_int32,
                                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "dsi_mxfp8_quantize": (c_int32, [c_void_p, c_int64, c_int32, c_int64, c_int32, c_void_p,
                                     c_void_p, c_void_p, c_void_p]),
    "dsi_latent_fp8_append": (c_int32, [c_void_p, c_int64, c_int64, c_void_p, c_void_p, c_void_p,
                                        c_void_p]),
    "dsi_workspace_size": (c_size_t, [c_int32, c_int32, c_int32, c_int32, c_int64, c_int32]),
    "dsi_layer_workspace_size": (c_size_t, [ctypes.POINTER(DsiCache), c_int32, c_int32, c_int32,
                                            c_int32, c_int64, c_int32]),
    "dsi_get_device_status": (c_int32, [c_void_p]),
    "dsi_selftest_wait_timeout": (c_int32, [ctypes.c_uint64, c_void_p]),
    "dsi_status_string": (ctypes.c_char_p, [c_int32]),
    "dsi_version": (c_int32, []),
    "dsi_launch_count": (ctypes.c_uint64, []),
}


class DsiError(RuntimeError):
    def __init__(self, fn: str, status: int, lib=None):
        msg = lib.dsi_status_string(status).decode() if lib is not None else str(status)
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def lib_path(checked: bool = False) -> str:
    return os.path.join(_PKG, "libdsi_checked.so" if checked else "libdsi.so")


def load(checked: bool = False):
    """Load (once) and return the library with typed entry points."""
    key = bool(checked)
    if key in _LIBS:
        return _LIBS[key]
    path = lib_path(checked)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run __graft_entry__.build() (no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIBS[key] = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _rows_contiguous(t: torch.Tensor, name: str):
    """The C ABI takes a row pitch: elements within a row must be contiguous."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with contiguous rows")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(lib, fn: str, status: int):
    if status != DSI_OK:
        raise DsiError(fn, status, lib)


class Cache:
    """Device tensors of one cache plus the ``dsi_cache`` struct that points at them."""

    def __init__(self, k_idx: Optional[torch.Tensor], latent: Optional[torch.Tensor],
                 seq_lens: Optional[torch.Tensor] = None, k_scale: Optional[torch.Tensor] = None,
                 block_table: Optional[torch.Tensor] = None, page_size: int = 0,
                 latent_scale: Optional[torch.Tensor] = None):
        self.k_idx, self.latent, self.seq_lens = k_idx, latent, seq_lens
        self.k_scale, self.block_table, self.page_size = k_scale, block_table, page_size
        self.latent_scale = latent_scale
        ref = k_idx if k_idx is not None else latent
        s = DsiCache()
        s.k_idx = k_idx.data_ptr() if k_idx is not None else None
        s.d = int(k_idx.shape[-1]) if k_idx is not None else 0
        s.k_dtype = DSI_BF16
        s.k_group = 0
        if k_idx is not None and k_idx.dtype == torch.float8_e4m3fn:
            # uint8 scales [.., d/G] are MXFP8 group scales; fp32 [..] per-position scales
            if k_scale is not None and k_scale.dtype == torch.uint8:
                s.k_dtype = DSI_MXFP8_E4M3
                s.k_group = s.d // int(k_scale.shape[-1])
            else:
                s.k_dtype = DSI_FP8_E4M3
        s.k_scale = k_scale.data_ptr() if k_scale is not None else None
        s.latent = latent.data_ptr() if latent is not None else None
        # an E4M3 latent cache is FP8 with per-tile scales
        s.latent_dtype = DSI_FP8_E4M3 if (latent is not None and latent.dtype == torch.float8_e4m3fn) else DSI_BF16
        s.latent_scale = latent_scale.data_ptr() if latent_scale is not None else None
        if block_table is not None:
            s.block_table = block_table.data_ptr()
            s.page_size = int(page_size)
            s.max_pages = int(block_table.shape[1])
            s.batch = int(block_table.shape[0])
            s.s_max = s.max_pages * s.page_size
            s.num_pages = int(ref.shape[0])
        else:
            s.block_table = None
            s.batch = int(ref.shape[0])
            s.s_max = int(ref.shape[1])
            s.num_pages = 0
        s.seq_lens = seq_lens.data_ptr() if seq_lens is not None else None
        self.struct = s

    @classmethod
    def of(cls, ws) -> "Cache":
        """Cache of a workload whose tensors are on the device."""
        return cls(ws.k_idx, ws.latent, ws.seq_lens, ws.k_scale, ws.block_table, ws.page_size,
                   getattr(ws, "latent_scale", None))

    def ref(self):
        return ctypes.byref(self.struct)


# ----------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ----------------------------------------------------------------------------

def index_score(q_idx, w, cache: Cache, decode: bool, q_offset: int = 0, scores=None,
                ld: Optional[int] = None, stream=None, checked: bool = False):
    lib = load(checked)
    rows, H_i = int(q_idx.shape[0]), int(q_idx.shape[1])
    if ld is None:
        ld = cache.struct.s_max if decode else q_offset + rows
    if scores is None:
        scores = torch.empty((rows, ld), dtype=torch.float32, device=q_idx.device)
    st = lib.dsi_index_score(_ptr(q_idx), _ptr(w), cache.ref(), rows, H_i, int(bool(decode)),
                             int(q_offset), _ptr(scores), int(ld), _stream(stream))
    _check(lib, "dsi_index_score", st)
    return scores


def index_topk_prefill(q_idx, w, cache: Cache, K: int, q_offset: int = 0, idx=None, count=None,
                       stream=None, checked: bool = False):
    """Fused prefill indexer: the causal Top-K indices of every query token,
    computed without writing the score matrix."""
    lib = load(checked)
    T, H_i = int(q_idx.shape[0]), int(q_idx.shape[1])
    if idx is None:
        idx = torch.empty((T, K), dtype=torch.int32, device=q_idx.device)
    if count is None:
        count = torch.empty((T,), dtype=torch.int32, device=q_idx.device)
    st = lib.dsi_index_topk_prefill(_ptr(q_idx), _ptr(w), cache.ref(), T, H_i, int(q_offset),
                                    int(K), _ptr(idx), _ptr(count), _stream(stream))
    _check(lib, "dsi_index_topk_prefill", st)
    return idx, count


def mxfp8_quantize(x, group: int = 32, dst_rows=None, codes=None, scales=None, stream=None,
                   checked: bool = False):
    """MXFP8 codes (float8_e4m3fn) and E8M0 scale bytes (uint8) of bf16 rows
    ``x [n, d]``; with ``dst_rows`` (int64 [n]) row i goes to row dst_rows[i]
    of the given ``codes``/``scales`` (an append into a cache)."""
    lib = load(checked)
    n, d = int(x.shape[0]), int(x.shape[1])
    _rows_contiguous(x, "x")
    if codes is None:
        codes = torch.empty((n, d), dtype=torch.float8_e4m3fn, device=x.device)
    if scales is None:
        scales = torch.empty((n, d // group), dtype=torch.uint8, device=x.device)
    st = lib.dsi_mxfp8_quantize(_ptr(x), n, d, int(x.stride(0)), int(group), _ptr(dst_rows),
                                _ptr(codes), _ptr(scales), _stream(stream))
    _check(lib, "dsi_mxfp8_quantize", st)
    return codes, scales


def latent_fp8_append(x, dst_rows=None, codes=None, scales=None, stream=None,
                      checked: bool = False):
    """FP8 latent codes (float8_e4m3fn [*, 576]) and fp32 tile scales ([*, 5]) of
    bf16 latent rows ``x [n, 576]``; with ``dst_rows`` (int64 [n]) row i goes to
    row dst_rows[i] of the given ``codes``/``scales`` (an append into a cache)."""
    lib = load(checked)
    n = int(x.shape[0])
    _rows_contiguous(x, "x")
    if int(x.shape[1]) != D_QK:
        raise ValueError(f"latent rows are {D_QK} wide, got {int(x.shape[1])}")
    if codes is None:
        codes = torch.empty((n, D_QK), dtype=torch.float8_e4m3fn, device=x.device)
    if scales is None:
        scales = torch.empty((n, 5), dtype=torch.float32, device=x.device)
    st = lib.dsi_latent_fp8_append(_ptr(x), n, int(x.stride(0)), _ptr(dst_rows), _ptr(codes),
                                   _ptr(scales), _stream(stream))
    _check(lib, "dsi_latent_fp8_append", st)
    return codes, scales


def topk(scores, K: int, row_len=None, q_offset: int = 0, idx=None, count=None, stream=None,
         checked: bool = False):
    lib = load(checked)
    rows, ld = int(scores.shape[0]), int(scores.stride(0)) if scores.dim() == 2 else 0
    if idx is None:
        idx = torch.empty((rows, K), dtype=torch.int32, device=scores.device)
    if count is None:
        count = torch.empty((rows,), dtype=torch.int32, device=scores.device)
    st = lib.dsi_topk(_ptr(scores), ld, rows, _ptr(row_len), int(q_offset), int(K), _ptr(idx),
                      _ptr(count), _stream(stream))
    _check(lib, "dsi_topk", st)
    return idx, count


def sparse_mla_decode(q, cache: Cache, idx, scale: float, out=None, lse=None, want_lse=True,
                      workspace=None, stream=None, checked: bool = False):
    lib = load(checked)
    B, H = int(q.shape[0]), int(q.shape[1])
    K = int(idx.shape[1])
    if out is None:
        out = torch.empty((B, H, D_LATENT), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    wsz = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.dsi_sparse_mla_decode(_ptr(q), cache.ref(), _ptr(idx), B, H, K, float(scale),
                                   _ptr(out), _ptr(lse), _ptr(workspace), wsz, _stream(stream))
    _check(lib, "dsi_sparse_mla_decode", st)
    return out, lse


def sparse_mla_prefill(q, cache: Cache, idx, q_offset: int, scale: float, out=None, lse=None,
                       want_lse=True, workspace=None, stream=None, checked: bool = False):
    lib = load(checked)
    T, H = int(q.shape[0]), int(q.shape[1])
    K = int(idx.shape[1])
    if out is None:
        out = torch.empty((T, H, D_LATENT), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    wsz = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.dsi_sparse_mla_prefill(_ptr(q), cache.ref(), _ptr(idx), T, H, K, int(q_offset),
                                    float(scale), _ptr(out), _ptr(lse), _ptr(workspace), wsz,
                                    _stream(stream))
    _check(lib, "dsi_sparse_mla_prefill", st)
    return out, lse


def workspace_size(rows: int, n_heads_idx: int, n_heads: int, K: int, s_max: int,
                   decode: bool, checked: bool = False) -> int:
    return int(load(checked).dsi_workspace_size(rows, n_heads_idx, n_heads, K, s_max,
                                                 int(bool(decode))))


def layer_workspace_size(cache: "Cache", rows: int, n_heads_idx: int, n_heads: int, K: int,
                         q_offset: int, decode: bool, checked: bool = False) -> int:
    """Exact workspace bytes of one fused-layer call (no score rows when a
    prefill takes the fused indexer)."""
    return int(load(checked).dsi_layer_workspace_size(cache.ref(), rows, n_heads_idx, n_heads, K,
                                                       int(q_offset), int(bool(decode))))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty((max(256, nbytes),), dtype=torch.uint8, device=device)


def indexed_attention(q_idx, w, q, cache: Cache, K: int, scale: float, decode: bool,
                      q_offset: int = 0, out=None, lse=None, idx=None, count=None,
                      workspace=None, want_lse=True, want_idx=True, stream=None,
                      checked: bool = False):
    """The whole layer (indexer -> Top-K -> sparse MLA) through ``dsi_indexed_attention``."""
    lib = load(checked)
    rows, H_i, H = int(q_idx.shape[0]), int(q_idx.shape[1]), int(q.shape[1])
    dev = q.device
    if workspace is None:
        workspace = alloc_workspace(
            layer_workspace_size(cache, rows, H_i, H, K, q_offset, decode, checked), dev)
    if out is None:
        out = torch.empty((rows, H, D_LATENT), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((rows, H), dtype=torch.float32, device=dev)
    if idx is None and want_idx:
        idx = torch.empty((rows, K), dtype=torch.int32, device=dev)
    if count is None and want_idx:
        count = torch.empty((rows,), dtype=torch.int32, device=dev)
    st = lib.dsi_indexed_attention(_ptr(q_idx), _ptr(w), _ptr(q), cache.ref(), rows, H_i, H, int(K),
                                   int(q_offset), float(scale), int(bool(decode)), _ptr(idx),
                                   _ptr(count), _ptr(out), _ptr(lse), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    _check(lib, "dsi_indexed_attention", st)
    return out, lse, idx, count


def indexed_attention_multi(q_idx, w, q, cache: Cache, tokens_per_seq: int, K: int, scale: float,
                            out=None, lse=None, idx=None, count=None, workspace=None,
                            want_lse=True, want_idx=True, stream=None, checked: bool = False):
    """A multi-token decode step through ``dsi_indexed_attention_multi``: rows
    come ``tokens_per_seq`` to a sequence (row r is candidate r % T of
    sequence r // T)."""
    lib = load(checked)
    rows, H_i, H = int(q_idx.shape[0]), int(q_idx.shape[1]), int(q.shape[1])
    dev = q.device
    if workspace is None:
        workspace = alloc_workspace(workspace_size(rows, H_i, H, K, cache.struct.s_max, True,
                                                   checked), dev)
    if out is None:
        out = torch.empty((rows, H, D_LATENT), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((rows, H), dtype=torch.float32, device=dev)
    if idx is None and want_idx:
        idx = torch.empty((rows, K), dtype=torch.int32, device=dev)
    if count is None and want_idx:
        count = torch.empty((rows,), dtype=torch.int32, device=dev)
    st = lib.dsi_indexed_attention_multi(_ptr(q_idx), _ptr(w), _ptr(q), cache.ref(),
                                         int(tokens_per_seq), H_i, H, int(K), float(scale),
                                         _ptr(idx), _ptr(count), _ptr(out), _ptr(lse),
                                         _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream))
    _check(lib, "dsi_indexed_attention_multi", st)
    return out, lse, idx, count


def device_status(stream=None, checked: bool = False) -> int:
    """Synchronise the stream and read/clear the device status word."""
    lib = load(checked)
    return int(lib.dsi_get_device_status(_stream(stream)))


def selftest_wait_timeout(limit_ns: int, stream=None, checked: bool = False) -> None:
    """Launch the bounded-wait self-test (one warp waits on a barrier nothing
    completes, for ``limit_ns``); ``device_status()`` then reports the timeout."""
    lib = load(checked)
    _check(lib, "dsi_selftest_wait_timeout", lib.dsi_selftest_wait_timeout(int(limit_ns),
                                                                          _stream(stream)))


def launch_count(checked: bool = False) -> int:
    """Kernels the library has launched in this process."""
    return int(load(checked).dsi_launch_count())


def layer(ws, workspace=None, stream=None, checked: bool = False, **kw):
    """Run the whole layer on a device-resident workload."""
    return indexed_attention(ws.q_idx, ws.w, ws.q, Cache.of(ws), ws.K, ws.scale,
                             ws.mode == "decode", ws.q_offset, workspace=workspace,
                             stream=stream, checked=checked, **kw)
