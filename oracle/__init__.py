"""Test infrastructure: the float64 CPU oracle for the attention library.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
package.  The CUDA library and its Python binding never import it, and it imports nothing from
them.  See ``oracle/attention_fp64.py`` for the definitions and the readings of the pages.
"""
from .attention_fp64 import (  # noqa: F401
    LATENT_DIM, LATENT_ROPE_DIM, as_f64, attention, attention_backward, attention_probs, combine_partials, decode,
    decode_append, latent_decode, prefill_chunk, merge_one_key, prefill, prefill_rows, rope_inv_freq, rope_rotate_half,
    ROPE_STYLES, rope_rotate, rope_rotate_interleaved,
    scores, softmax_rows, split_decode_partials,
)
