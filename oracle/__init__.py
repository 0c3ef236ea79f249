"""CPU oracle (float64 numpy) for the context-parallel attention path.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
legs of ``bench.py``; never by the product library or its Python binding.
"""
from .cp_attention import (E4M3_MAX, attention, attention_chunked, attention_fp8,
                           attention_online, attention_ring, chunk_bounds, e4m3_decode,
                           e4m3_encode, e4m3_quantize, e4m3_round, fp8_p_rounding_bound, head2seq,
                           lse_merge, seq2head, softmax_weights, to_f64, ulysses_attention)

__all__ = ["E4M3_MAX", "attention_fp8", "e4m3_decode", "e4m3_encode", "e4m3_quantize",
           "e4m3_round", "fp8_p_rounding_bound",
           "attention", "attention_chunked", "attention_online", "attention_ring", "chunk_bounds",
           "head2seq",
           "lse_merge", "seq2head", "softmax_weights", "to_f64", "ulysses_attention"]
