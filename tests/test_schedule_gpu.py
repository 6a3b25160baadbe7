"""Split-schedule invariance: the same decode under every way of splitting
its segments over CTAs.

The decode page's split-KV attention (section 3: partial results per key
range, combined with their running maxima and sums) gives the same output
whatever the key ranges are; only the rounding of the merge order may
differ.  attn_test_force_schedule forces stream-K (flat tile list over the
persistent grid, split segments merged through the workspace by the last
CTA to arrive) or cluster mode with clusters of C CTAs (rank r takes tiles
r, r+C, ...; partials merged in rank 0's shared memory).  Each schedule must
match the oracle, and all schedules must agree with each other closely.
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, f64

pytestmark = pytest.mark.gpu

SCHEDULES = [-1, 0, 1, 2, 3, 5, 8, 9, 12, 16]


def _run(case, sched, fused):
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    ga.attn_test_force_schedule(sched)
    try:
        if fused:
            out = ga.attn_decode_step_append(case.q, case.k_new, case.v_new, case.positions,
                                             kc, vc, case.scale)
        else:
            ga.attn_kv_append(case.k_new, case.v_new, case.positions, kc, vc)
            out = ga.attn_decode_step(case.q, case.positions, kc, vc, case.scale)
        torch.cuda.synchronize()
    except ga.AttnError:
        return None  # a cluster size this kernel cannot launch
    finally:
        ga.attn_test_force_schedule(-1)
    return out


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("fused", [False, True])
def test_every_schedule_matches_the_oracle_and_the_others(g, fused):
    Hkv = 2
    positions = [4095, 130, 8191]  # 32, 2 and 64 tiles: ragged splits
    case = synth.decode_case(B=3, Hq=g * Hkv, Hkv=Hkv, D=128, L=8192, positions=positions,
                             fill="all", poison=True, seed=100 + g, device="cuda")
    pos = case.positions.cpu().numpy()
    kc, vc = oracle.kv_append(f64(case.k_cache), f64(case.v_cache), f64(case.k_new),
                              f64(case.v_new), pos)
    want = oracle.decode(f64(case.q), kc, vc, pos, case.scale)
    outs = {}
    for sched in SCHEDULES:
        out = _run(case, sched, fused)
        if out is None:
            assert sched >= 9, f"g={g}: schedule {sched} refused"
            continue
        assert_attn_close(f64(out), want, f"g={g} schedule={sched} fused={fused}")
        outs[sched] = f64(out)
    assert 0 in outs and 8 in outs and -1 in outs
    ref = outs[-1]
    for sched, o in outs.items():
        # the same sums in another order: far inside the oracle tolerance
        assert float(np.abs(o - ref).max()) <= 4e-3, (g, sched)
