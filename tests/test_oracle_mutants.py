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
