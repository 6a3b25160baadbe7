"""CPU oracle for static-KV-cache GQA decode attention and causal prefill.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain, fp64 statement of
what the CUDA path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and ``bench.py --impl reference``) may import
it.  The product library never calls it, and it shares no code with the CUDA
path: it takes plain numpy arrays holding the exact values of the bf16 inputs.

Every function is pinned by ``tests/test_oracle_pins.py`` against things other
than itself: a pure-Python brute force (``oracle.brute``), PyTorch's library
``scaled_dot_product_attention`` in fp64 (the call the decode page makes, with
and without its full-length boolean mask), closed forms (position 0 returns
V[0]; identical keys or a zero query return the mean of V), and invariances
(key-row permutation, GQA equal to repeat-KV MHA, prefill of one token equal to
a decode step, prefix prefill equal to the tail of a full causal prefill),
and for the rotary embedding: a hand-worked rotation, the identity at angle
0, norm preservation, and dot products that depend only on the position
difference; for the local window: a window of one returning V[pos], any
window of pos + 1 or more equal to the full decode, and the windowed decode
equal to the full decode of the shifted slice; for multi-token decode: one
token equal to the decode, and a sequence's tokens equal to a prefill over
its cache rows from their first position.
"""

from .attention import (  # noqa: F401
    kv_append,
    decode,
    decode_masked_full,
    decode_rows,
    prefill,
    prefill_rows,
    decode_bytes,
    decode_flops,
    prefill_flops,
    rope_f32,
    round_bf16,
    decode_rope_step,
    decode_window,
    decode_multi,
)
