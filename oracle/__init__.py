"""CPU oracle of the indexed sparse attention layer — test infrastructure only.

Imported by the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline
leg; never by the library.
"""
from .dsi_oracle import (mx_exponent, mxfp8_quantize, mxfp8_dequantize, index_scores,
                         topk_select, sparse_mla, dense_mla, latent_fp8_quantize,
                         latent_fp8_dequantize, history_rows, layer_row, decode_row,
                         multi_token_row, prefill_row, row_scores, layer)

__all__ = ["mx_exponent", "mxfp8_quantize", "mxfp8_dequantize", "index_scores", "topk_select",
           "sparse_mla", "dense_mla", "latent_fp8_quantize", "latent_fp8_dequantize",
           "history_rows", "layer_row", "decode_row",
           "multi_token_row", "prefill_row", "row_scores", "layer"]
