"""The oracle: a plain, slow, float64 CPU statement of the paged quantized-KV
hot path (E4M3 / INT8 encode and decode, quantize-and-append into pages, paged
decode / verify attention, split-KV log-sum-exp merge).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it.  It shares no code with the CUDA
library and never imports it.
"""
from .codec import (E4M3_MAX, INT8_MAX, INT8_TOKEN, dequantize, e4m3_decode, e4m3_encode,
                    int8_decode, int8_encode, int8_row_scale, quantize, scaled_input)
from .attention import (attention_partial, dense_attention, gather_kv,
                        kv_append_quant, lse_merge, merge_lse, new_pool, new_scale_pool,
                        paged_attention, paged_attention_partial)

__all__ = [
    "E4M3_MAX", "INT8_MAX", "INT8_TOKEN", "dequantize", "e4m3_decode", "e4m3_encode",
    "int8_decode", "int8_encode", "int8_row_scale", "quantize", "scaled_input",
    "attention_partial", "dense_attention", "gather_kv", "kv_append_quant", "lse_merge",
    "merge_lse", "new_pool", "new_scale_pool", "paged_attention", "paged_attention_partial",
]
