"""The C-ABI library on a machine without a GPU: it loads, exports every symbol
include/dsi.h declares, matches the header's struct layout, and rejects bad
arguments on the host before launching anything."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from indexed_sparse_attention_indexer_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsi.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsi_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module", params=[False, True], ids=["release", "checked"])
def L(request):
    path = binding.lib_path(request.param)
    if not os.path.exists(path):
        pytest.skip("library not built (run __graft_entry__.build())")
    return binding.load(request.param)


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(binding.SIGNATURES), "binding and header disagree"


def test_version_and_status_strings(L):
    assert L.dsi_version() == 2
    for code in range(7):
        s = L.dsi_status_string(code)
        assert s and s != b"unknown status"
    assert L.dsi_status_string(99) == b"unknown status"


def test_struct_layout_matches_header(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "dsi.h"\n'
        "#define O(f) printf(\"%s %zu\\n\", #f, offsetof(dsi_cache, f));\n"
        "int main(void){ printf(\"size %zu\\n\", sizeof(dsi_cache));"
        + "".join(f"O({f})" for f, _ in binding.DsiCache._fields_) + "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(line.split() for line in out if line)
    assert int(got["size"]) == ctypes.sizeof(binding.DsiCache)
    for f, _ in binding.DsiCache._fields_:
        assert int(got[f]) == getattr(binding.DsiCache, f).offset, f


FAKE = 1 << 20  # an aligned, never dereferenced stand-in for a device pointer


def _cache(**kw):
    c = binding.DsiCache()
    c.k_idx, c.k_dtype, c.d, c.k_scale = FAKE, 0, 128, None
    c.latent, c.block_table, c.page_size, c.max_pages = FAKE, None, 0, 0
    c.seq_lens, c.batch, c.s_max, c.num_pages = FAKE, 4, 1024, 0
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _score(L, c, rows=4, heads=64, decode=1, q_offset=0, ld=1024, q=FAKE, w=FAKE, s=FAKE):
    return L.dsi_index_score(q, w, ctypes.byref(c), rows, heads, decode, q_offset, s, ld, None)


def test_index_score_validation(L):
    E, U = binding.DSI_ERR_INVALID_ARG, binding.DSI_ERR_UNSUPPORTED
    assert _score(L, _cache(), q=None) == E
    assert _score(L, _cache(), w=None) == E
    assert _score(L, _cache(), s=None) == E
    assert _score(L, _cache(), rows=-1) == E
    assert _score(L, _cache(), heads=0) == U
    assert _score(L, _cache(), heads=129) == U
    assert _score(L, _cache(k_idx=None)) == E
    assert _score(L, _cache(d=12)) == U                       # not a multiple of 8
    assert _score(L, _cache(k_dtype=1, d=24, k_scale=FAKE)) == U  # fp8 needs multiples of 16
    assert _score(L, _cache(k_dtype=1)) == E                  # fp8 without scales
    assert _score(L, _cache(k_dtype=7)) == U
    assert _score(L, _cache(k_idx=FAKE + 2)) == E             # misaligned
    assert _score(L, _cache(), rows=3) == E                   # decode rows != batch
    assert _score(L, _cache(seq_lens=None)) == E
    assert _score(L, _cache(), ld=1000) == E                  # ld < s_max
    # prefill: one sequence, q_offset + rows <= s_max
    assert _score(L, _cache(batch=1), decode=0, rows=8, q_offset=1020, ld=2048) == E
    assert _score(L, _cache(batch=2), decode=0, rows=8, ld=2048) == E
    # paged: s_max must be max_pages * page_size, page size a multiple of 8
    assert _score(L, _cache(block_table=FAKE, page_size=64, max_pages=8, num_pages=10)) == E
    assert _score(L, _cache(block_table=FAKE, page_size=60, max_pages=16, num_pages=10,
                            s_max=960), ld=960) == U
    # zero rows: nothing to launch, success
    assert _score(L, _cache(batch=0), rows=0) == binding.DSI_OK


def _itp(L, c, T=8, heads=64, q_offset=0, K=16, q=FAKE, w=FAKE, idx=FAKE):
    return L.dsi_index_topk_prefill(q, w, ctypes.byref(c), T, heads, q_offset, K, idx, None, None)


def test_index_topk_prefill_validation(L):
    """Host checks of the fused prefill indexer: errors before any launch."""
    E, U = binding.DSI_ERR_INVALID_ARG, binding.DSI_ERR_UNSUPPORTED
    one = dict(batch=1, seq_lens=None)
    assert _itp(L, _cache(**one), q=None) == E
    assert _itp(L, _cache(**one), w=None) == E
    assert _itp(L, _cache(**one), idx=None) == E
    assert _itp(L, _cache(**one), T=-1) == E
    assert _itp(L, _cache(**one), K=0) == E
    assert _itp(L, _cache(**one), K=4097) == U
    assert _itp(L, _cache(**one), heads=0) == U
    assert _itp(L, _cache(batch=2, seq_lens=None)) == E       # prefill is one sequence
    assert _itp(L, _cache(**one), T=8, q_offset=1020) == E    # beyond s_max
    assert _itp(L, _cache(**one), heads=32) == U              # the fused kernel needs 64 x 128
    assert _itp(L, _cache(d=64, **one)) == U
    assert _itp(L, _cache(k_dtype=1, k_scale=FAKE, **one)) == U
    assert _itp(L, _cache(**one), K=2049) == U
    assert _itp(L, _cache(**one), T=0) == binding.DSI_OK


def test_indexed_attention_multi_validation(L):
    """Host checks of the multi-token decode entry (rows = batch x T)."""
    E = binding.DSI_ERR_INVALID_ARG
    M = L.dsi_indexed_attention_multi
    c = _cache(batch=4)
    args = lambda **kw: dict(dict(q_idx=FAKE, w=FAKE, q=FAKE, T=2, Hi=64, H=128, K=16, out=FAKE,
                                  ws=FAKE, wsb=1 << 30), **kw)
    def call(cache, **kw):
        a = args(**kw)
        return M(a["q_idx"], a["w"], a["q"], ctypes.byref(cache), a["T"], a["Hi"], a["H"], a["K"],
                 0.04, None, None, a["out"], None, a["ws"], a["wsb"], None)
    assert M(FAKE, FAKE, FAKE, None, 2, 64, 128, 16, 0.04, None, None, FAKE, None, FAKE, 1 << 30,
             None) == E
    assert call(c, T=0) == E
    assert call(c, q_idx=None) == E
    assert call(c, out=None) == E
    assert call(c, K=0) == E
    assert call(_cache(batch=4, seq_lens=None)) == E
    assert call(c, ws=None) == binding.DSI_ERR_WORKSPACE
    assert call(_cache(batch=0)) == binding.DSI_OK     # no rows: nothing to launch


def test_mxfp8_validation(L):
    """Host checks of the MXFP8 quantiser and of MXFP8 key caches."""
    E, U = binding.DSI_ERR_INVALID_ARG, binding.DSI_ERR_UNSUPPORTED
    Q = L.dsi_mxfp8_quantize
    assert Q(None, 4, 128, 128, 32, None, FAKE, FAKE, None) == E
    assert Q(FAKE, 4, 128, 128, 32, None, None, FAKE, None) == E
    assert Q(FAKE, 4, 128, 128, 32, None, FAKE, None, None) == E
    assert Q(FAKE, -1, 128, 128, 32, None, FAKE, FAKE, None) == E
    assert Q(FAKE, 4, 128, 128, 16, None, FAKE, FAKE, None) == U     # group size
    assert Q(FAKE, 4, 96, 96, 64, None, FAKE, FAKE, None) == U       # d not a multiple of group
    assert Q(FAKE, 4, 128, 120, 32, None, FAKE, FAKE, None) == E     # ld_x < d
    assert Q(FAKE, 4, 128, 132, 32, None, FAKE, FAKE, None) == E     # ld_x not a multiple of 8
    assert Q(FAKE + 8, 4, 128, 128, 32, None, FAKE, FAKE, None) == E
    assert Q(FAKE, 4, 128, 128, 32, None, FAKE + 4, FAKE, None) == E
    assert Q(FAKE, 0, 128, 128, 32, None, FAKE, FAKE, None) == binding.DSI_OK
    mx = dict(k_dtype=binding.DSI_MXFP8_E4M3, k_scale=FAKE)
    assert _score(L, _cache(k_dtype=binding.DSI_MXFP8_E4M3)) == E          # no scales
    assert _score(L, _cache(**mx, k_group=48)) == U
    assert _score(L, _cache(**dict(mx, k_scale=FAKE + 4))) == E            # misaligned scales
    assert _score(L, _cache(**mx, d=96, k_group=64)) == U
    # MXFP8 keys only on the tensor-core shape (64 heads x 128 dims)
    assert _score(L, _cache(**mx), heads=32) == U
    c = _cache(**mx)
    args = [FAKE, FAKE, FAKE, ctypes.byref(c), 4, 32, 128, 2048, 0, 0.04, 1, None, None, FAKE,
            None]
    assert L.dsi_indexed_attention(*args, FAKE, 1 << 40, None) == U


def test_latent_fp8_validation(L):
    """Host checks of the FP8 latent append and of FP8 latent caches."""
    E, U = binding.DSI_ERR_INVALID_ARG, binding.DSI_ERR_UNSUPPORTED
    A = L.dsi_latent_fp8_append
    assert A(None, 4, 576, None, FAKE, FAKE, None) == E
    assert A(FAKE, 4, 576, None, None, FAKE, None) == E
    assert A(FAKE, 4, 576, None, FAKE, None, None) == E
    assert A(FAKE, -1, 576, None, FAKE, FAKE, None) == E
    assert A(FAKE, 4, 512, None, FAKE, FAKE, None) == E      # ld_x < 576
    assert A(FAKE, 4, 580, None, FAKE, FAKE, None) == E      # ld_x not a multiple of 8
    assert A(FAKE + 8, 4, 576, None, FAKE, FAKE, None) == E
    assert A(FAKE, 4, 576, None, FAKE + 8, FAKE, None) == E
    assert A(FAKE, 4, 576, None, FAKE, FAKE + 2, None) == E
    assert A(FAKE, 0, 576, None, FAKE, FAKE, None) == binding.DSI_OK
    f = L.dsi_sparse_mla_decode
    c = _cache(latent_dtype=binding.DSI_FP8_E4M3)             # FP8 latent without scales
    assert f(FAKE, ctypes.byref(c), FAKE, 4, 16, 64, 0.1, FAKE, None, None, 0, None) == E
    c = _cache(latent_dtype=7)
    assert f(FAKE, ctypes.byref(c), FAKE, 4, 16, 64, 0.1, FAKE, None, None, 0, None) == U
    c = _cache(latent_dtype=binding.DSI_FP8_E4M3, latent_scale=FAKE + 2)
    assert f(FAKE, ctypes.byref(c), FAKE, 4, 16, 64, 0.1, FAKE, None, None, 0, None) == E


def test_selftest_wait_timeout_validation(L):
    E = binding.DSI_ERR_INVALID_ARG
    assert L.dsi_selftest_wait_timeout(999, None) == E            # below 1 us
    assert L.dsi_selftest_wait_timeout(1000000001, None) == E     # above 1 s


def test_topk_validation(L):
    E, U = binding.DSI_ERR_INVALID_ARG, binding.DSI_ERR_UNSUPPORTED
    assert L.dsi_topk(None, 16, 2, None, 0, 4, FAKE, None, None) == E
    assert L.dsi_topk(FAKE, 16, 2, None, 0, 0, FAKE, None, None) == E
    assert L.dsi_topk(FAKE, 16, 2, None, 0, 4, None, None, None) == E
    assert L.dsi_topk(FAKE, 16, 2, None, -1, 4, FAKE, None, None) == E
    assert L.dsi_topk(FAKE, 16, 2, None, 0, 4097, FAKE, None, None) == U
    assert L.dsi_topk(FAKE, 16, 0, None, 0, 4, FAKE, None, None) == binding.DSI_OK


def test_mla_validation(L):
    E, U = binding.DSI_ERR_INVALID_ARG, binding.DSI_ERR_UNSUPPORTED
    c = _cache()
    f = L.dsi_sparse_mla_decode
    assert f(None, ctypes.byref(c), FAKE, 4, 128, 64, 0.1, FAKE, None, None, 0, None) == E
    assert f(FAKE, ctypes.byref(c), FAKE, 4, 129, 64, 0.1, FAKE, None, None, 0, None) == U
    assert f(FAKE, ctypes.byref(c), FAKE, 4, 40, 64, 0.1, FAKE, None, None, 0, None) == U
    assert f(FAKE, ctypes.byref(c), FAKE, 4, 128, 0, 0.1, FAKE, None, None, 0, None) == E
    assert f(FAKE, ctypes.byref(c), FAKE, 4, 128, 64, float("nan"), FAKE, None, None, 0, None) == E
    assert f(FAKE, ctypes.byref(_cache(latent=None)), FAKE, 4, 128, 64, 0.1, FAKE, None, None, 0,
             None) == E
    assert f(FAKE, ctypes.byref(c), FAKE, 4, 128, 64, 0.1, FAKE, None, FAKE + 16, 1 << 20,
             None) == E  # workspace not 256-byte aligned
    g = L.dsi_sparse_mla_prefill
    assert g(FAKE, ctypes.byref(_cache(batch=1)), FAKE, 8, 128, 64, 1020, 0.1, FAKE, None, None,
             0, None) == E


def test_fused_validation(L):
    c = _cache()
    f = L.dsi_indexed_attention
    args = [FAKE, FAKE, FAKE, ctypes.byref(c), 4, 64, 128, 2048, 0, 0.04, 1, None, None, FAKE,
            None]
    assert f(*args, None, 0, None) == binding.DSI_ERR_WORKSPACE
    assert f(*args, FAKE, 16, None) == binding.DSI_ERR_WORKSPACE
    bad = list(args); bad[7] = 5000
    assert f(*bad, None, 0, None) == binding.DSI_ERR_UNSUPPORTED
    bad = list(args); bad[2] = None
    assert f(*bad, None, 0, None) == binding.DSI_ERR_INVALID_ARG


def test_workspace_size(L):
    a = L.dsi_workspace_size(64, 64, 128, 2048, 32768, 1)
    # at least the fp32 score rows and the index rows
    assert a >= 64 * 32768 * 4 + 64 * 2048 * 4
    assert L.dsi_workspace_size(64, 64, 128, 2048, 65536, 1) > a
    assert L.dsi_workspace_size(0, 64, 128, 2048, 32768, 1) == 256


def test_layer_workspace_size(L):
    """The exact size of one call: a decode call needs what the upper bound
    gives; no call needs more than it; degenerate sizes give 256."""
    c = _cache(batch=64, s_max=32768)
    ws = L.dsi_layer_workspace_size
    assert ws(ctypes.byref(c), 64, 64, 128, 2048, 0, 1) == L.dsi_workspace_size(64, 64, 128, 2048,
                                                                                32768, 1)
    p = _cache(batch=1, s_max=8192, seq_lens=None)
    for T, off in ((8192, 0), (4096, 4096), (100, 7)):
        assert ws(ctypes.byref(p), T, 64, 128, 2048, off, 0) <= L.dsi_workspace_size(
            T, 64, 128, 2048, off + T, 0)
        # an index row per token at least
        assert ws(ctypes.byref(p), T, 64, 128, 2048, off, 0) >= T * 2048 * 4
    assert ws(None, 64, 64, 128, 2048, 0, 1) == 256
    assert ws(ctypes.byref(c), 0, 64, 128, 2048, 0, 1) == 256


def test_binding_rejects_strided_rows():
    """The quantiser bindings pass a row pitch: rows must be contiguous (checked
    before anything reaches the library)."""
    import torch
    x = torch.zeros((128, 4), dtype=torch.bfloat16).t()      # 4 rows with stride 1 between rows
    with pytest.raises(ValueError):
        binding.mxfp8_quantize(x)
    with pytest.raises(ValueError):
        binding.latent_fp8_append(torch.zeros((2, 512), dtype=torch.bfloat16))
