"""The failure path of a wait that runs out, made on purpose without a fault.

attn_test_skip_tile makes a decode launch skip one tile's bulk copy, so the
waits for that tile never complete.  Every wait in the
kernels gives up after 500 ms: the launch must end by itself with
ATTN_DEV_TIMEOUT in the status word, and the CUDA context must stay usable --
a normal step right after gives the oracle's result.  Covers cluster mode
and stream-K on both kernel families: per-warp MMAs (g <= 8) and tcgen05
(g = 16).
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, f64

pytestmark = pytest.mark.gpu


# per-warp MMAs: clusters (g=2), stream-K (g=4), stream-K (g=8), clusters
# (g=8); tcgen05: clusters at g=16 (at most 9 CTAs), stream-K at g=16
@pytest.mark.parametrize("B,Hq,Hkv", [(1, 16, 8), (16, 8, 2), (16, 16, 2), (1, 64, 8),
                                      (4, 32, 2), (16, 32, 2)])
def test_wait_runs_out_and_the_context_stays_usable(B, Hq, Hkv):
    positions = [700 + 37 * b for b in range(B)]
    case = synth.decode_case(B=B, Hq=Hq, Hkv=Hkv, D=128, L=2048, positions=positions,
                             fill="all", seed=400 + B + Hq, device="cuda")
    ws = ga.decode_workspace(B, Hq, Hkv, 2048, 128)
    ga.attn_test_skip_tile(0)
    try:
        ga.attn_decode_step(case.q, case.positions, case.k_cache, case.v_cache, case.scale,
                            workspace=ws)
        bits = ga.attn_read_device_status(ws)  # synchronises: the launch ended by itself
    finally:
        ga.attn_test_skip_tile(-1)
    assert bits & ga.ATTN_DEV_TIMEOUT
    # the same step again, on a fresh workspace: the context still works
    ws2 = ga.decode_workspace(B, Hq, Hkv, 2048, 128)
    out = ga.attn_decode_step(case.q, case.positions, case.k_cache, case.v_cache, case.scale,
                              workspace=ws2)
    assert ga.attn_read_device_status(ws2) == 0
    want = oracle.decode(f64(case.q), f64(case.k_cache), f64(case.v_cache), positions, case.scale)
    assert_attn_close(f64(out), want, f"after a timeout B={B} Hq={Hq}")
