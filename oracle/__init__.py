"""CPU oracle (float64 numpy) for the context-parallel attention path.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
legs of ``bench.py``; never by the product library or its Python binding.
"""
from .cp_attention import (attention, attention_chunked, attention_online, attention_ring,
                           chunk_bounds, head2seq, lse_merge, seq2head, softmax_weights, to_f64,
                           ulysses_attention)

__all__ = ["attention", "attention_chunked", "attention_online", "attention_ring", "chunk_bounds",
           "head2seq",
           "lse_merge", "seq2head", "softmax_weights", "to_f64", "ulysses_attention"]
