"""Plant plausible mistakes in copies of the oracle (CPU) and check that the pins
catch every one of them.  Nothing here touches the CUDA path."""
import math
import types

import numpy as np
import pytest

import oracle
from oracle import dsi_oracle as real
from tests import oracle_pins


def _ns(**overrides):
    ns = types.SimpleNamespace(**{k: getattr(real, k) for k in dir(real) if not k.startswith("__")})
    for k, v in overrides.items():
        setattr(ns, k, v)
    # layer_row must call the namespace's own pieces
    def layer_row(q_idx_t, w_t, q_t, k_hist, k_scale_hist, latent_of, n_hist, K, scale):
        I = ns.index_scores(q_idx_t, w_t, k_hist, k_scale_hist)
        idx, count = ns.topk_select(I, K)
        o, lse = ns.sparse_mla(q_t, latent_of(idx[:count]), scale)
        return {"scores": I, "idx": idx, "count": count, "out": o, "lse": lse}
    if "layer_row" not in overrides:
        ns.layer_row = layer_row
    return ns


def _scores_no_relu(q_idx, w, k_rows, k_scale=None):
    q = real._f64(q_idx); k = real._f64(k_rows)
    if k_scale is not None:
        k = k * real._f64(k_scale)[:, None]
    return (k @ q.T) @ real._f64(w)


def _scores_relu_after_sum(q_idx, w, k_rows, k_scale=None):
    return np.maximum(_scores_no_relu(q_idx, w, k_rows, k_scale), 0.0)


def _scores_ignore_scale(q_idx, w, k_rows, k_scale=None):
    return real.index_scores(q_idx, w, k_rows, None)


def _scores_reversed_weights(q_idx, w, k_rows, k_scale=None):
    return real.index_scores(q_idx, real._f64(w)[::-1].copy(), k_rows, k_scale)


def _scores_first_head_only_weight(q_idx, w, k_rows, k_scale=None):
    ww = real._f64(w).copy(); ww[:] = ww[0]
    return real.index_scores(q_idx, ww, k_rows, k_scale)


def _topk_high_tie(scores, K):
    I = real._f64(scores); n = I.shape[0]
    order = np.lexsort((-np.arange(n), -I))
    keep = np.sort(order[:min(K, n)])
    out = np.full(K, -1, dtype=np.int64); out[:keep.shape[0]] = keep
    return out, int(keep.shape[0])


def _topk_score_order(scores, K):
    I = real._f64(scores); n = I.shape[0]
    order = np.lexsort((np.arange(n), -I))[:min(K, n)]
    out = np.full(K, -1, dtype=np.int64); out[:order.shape[0]] = order
    return out, int(order.shape[0])


def _topk_off_by_one(scores, K):
    return real.topk_select(scores, max(1, K - 1))[0].tolist() + [-1], max(0, min(K - 1, len(scores)))


def _mla_values_tail(q, rows, scale, d_v=512):
    qq = real._f64(q); c = real._f64(rows)
    l = scale * (qq @ c.T); e = np.exp(l - l.max(1, keepdims=True)); z = e.sum(1, keepdims=True)
    return (e @ c[:, -d_v:]) / z, l.max(1) + np.log(z[:, 0])


def _mla_keys_latent_only(q, rows, scale, d_v=512):
    qq = real._f64(q); c = real._f64(rows)
    kd = max(1, c.shape[1] - 64)
    l = scale * (qq[:, :kd] @ c[:, :kd].T); e = np.exp(l - l.max(1, keepdims=True)); z = e.sum(1, keepdims=True)
    return (e @ c[:, :d_v]) / z, l.max(1) + np.log(z[:, 0])


def _mla_no_scale(q, rows, scale, d_v=512):
    return real.sparse_mla(q, rows, 1.0, d_v)


def _mla_lse_log2(q, rows, scale, d_v=512):
    o, lse = real.sparse_mla(q, rows, scale, d_v)
    return o, lse / math.log(2.0)


def _mla_unnormalised(q, rows, scale, d_v=512):
    qq = real._f64(q); c = real._f64(rows)
    l = scale * (qq @ c.T); e = np.exp(l - l.max(1, keepdims=True))
    return e @ c[:, :d_v], l.max(1)


def _mx_quantize_with(exponent, rounding=None):
    """An MXFP8 quantiser with a planted change in the exponent rule or rounding."""
    def quantize(x, group=32):
        a = real._f64(x); d = a.shape[-1]
        blocks = a.reshape(a.shape[:-1] + (d // group, group))
        amax = np.abs(blocks).max(axis=-1)
        X = np.vectorize(exponent, otypes=[np.int64])(amax)
        y = blocks / np.ldexp(1.0, X)[..., None]
        c = real.e4m3_round(y) if rounding is None else rounding(y)
        return c.reshape(a.shape), X
    return quantize


def _exp_rounded_log2(amax):
    return -127 if amax == 0 else max(-127, int(round(math.log2(amax))) - 8)


def _exp_emax7(amax):
    return -127 if amax == 0 else max(-127, math.frexp(amax)[1] - 1 - 7)


def _exp_zero_group_0(amax):
    return 0 if amax == 0 else real.mx_exponent(amax)


def _e4m3_truncate(y):
    """Toward-zero rounding onto the E4M3 grid (saturating at 448)."""
    import torch
    codes = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn)
    mags = np.sort(codes.to(torch.float64).numpy())      # 0 .. 448
    a = np.minimum(np.abs(y), 448.0)
    return np.sign(y) * mags[np.searchsorted(mags, a, side="right") - 1]


def _mx_scores(q_quant=True, per_row_scale=False):
    def scores(q_idx, w, k_rows, k_scale=None):
        if k_scale is None or np.ndim(real._f64(k_scale)) != 2:
            return real.index_scores(q_idx, w, k_rows, k_scale)
        byt = real._f64(k_scale).astype(np.int64)
        k = real._f64(k_rows); group = k.shape[-1] // byt.shape[-1]
        if per_row_scale:
            byt = np.repeat(byt[:, :1], byt.shape[1], axis=1)
        q = real._f64(q_idx)
        if q_quant:
            q = real.mxfp8_dequantize(*real.mxfp8_quantize(q, group), group)
        kk = real.mxfp8_dequantize(k, byt - 127, group)
        return np.maximum(kk @ q.T, 0.0) @ real._f64(w)
    return scores


def _latent_quantize_with(tiles=None, qmax=448.0):
    """An FP8 latent quantiser with a planted change in the tiling or the scale."""
    tl = tiles or real.LATENT_TILES
    def quantize(rows):
        x = real._f64(rows).astype(np.float32)
        codes = np.zeros(x.shape)
        scales = np.zeros(x.shape[:-1] + (len(real.LATENT_TILES),))
        for t, (a, b) in enumerate(tl):
            seg = x[..., a:b]
            sc = (np.abs(seg).max(axis=-1) / np.float32(qmax)).astype(np.float32)
            safe = np.where(sc > 0, sc, np.float32(1.0)).astype(np.float32)
            codes[..., a:b] = real.e4m3_round((seg / safe[..., None]).astype(np.float64))
            scales[..., min(t, len(real.LATENT_TILES) - 1)] = sc
        return codes, scales
    return quantize


MUTANTS = {
    "no_relu": dict(index_scores=_scores_no_relu),
    "relu_after_head_sum": dict(index_scores=_scores_relu_after_sum),
    "fp8_scale_ignored": dict(index_scores=_scores_ignore_scale),
    "head_weights_reversed": dict(index_scores=_scores_reversed_weights),
    "one_weight_for_all_heads": dict(index_scores=_scores_first_head_only_weight),
    "ties_to_higher_position": dict(topk_select=_topk_high_tie),
    "indices_in_score_order": dict(topk_select=_topk_score_order),
    "k_minus_one": dict(topk_select=_topk_off_by_one),
    "values_from_row_tail": dict(sparse_mla=_mla_values_tail, dense_mla=_mla_values_tail),
    "keys_without_rope": dict(sparse_mla=_mla_keys_latent_only, dense_mla=_mla_keys_latent_only),
    "softmax_scale_dropped": dict(sparse_mla=_mla_no_scale, dense_mla=_mla_no_scale),
    "lse_base_2": dict(sparse_mla=_mla_lse_log2, dense_mla=_mla_lse_log2),
    "softmax_not_normalised": dict(sparse_mla=_mla_unnormalised, dense_mla=_mla_unnormalised),
    "mx_exponent_rounded": dict(mxfp8_quantize=_mx_quantize_with(_exp_rounded_log2)),
    "mx_emax_7": dict(mxfp8_quantize=_mx_quantize_with(_exp_emax7)),
    "mx_zero_group_exponent_0": dict(mxfp8_quantize=_mx_quantize_with(_exp_zero_group_0)),
    "mx_round_toward_zero": dict(mxfp8_quantize=_mx_quantize_with(real.mx_exponent,
                                                                   _e4m3_truncate)),
    "mx_query_not_quantised": dict(index_scores=_mx_scores(q_quant=False)),
    "mx_one_scale_per_row": dict(index_scores=_mx_scores(per_row_scale=True)),
    "latent_scale_over_240": dict(latent_fp8_quantize=_latent_quantize_with(qmax=240.0)),
    "latent_rope_in_last_tile": dict(latent_fp8_quantize=_latent_quantize_with(
        tiles=((0, 128), (128, 256), (256, 384), (384, 576)))),
    "latent_tiles_of_64": dict(latent_fp8_quantize=_latent_quantize_with(
        tiles=tuple((a, a + 64) for a in range(0, 576, 64))[:5])),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    ns = _ns(**MUTANTS[name])
    failed = []
    for check in oracle_pins.all_checks():
        try:
            check(ns)
        except AssertionError:
            failed.append(check.__name__)
        except Exception:   # a crash on a pin input also counts as caught
            failed.append(check.__name__ + "(error)")
    assert failed, f"no pin catches the planted mistake '{name}'"


def test_real_oracle_passes_all_pins():
    for check in oracle_pins.all_checks():
        check(oracle)
