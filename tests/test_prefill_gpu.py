"""Causal prefill over a cached prefix (tcgen05 kernel) against the fp64 oracle.

Covers both prefill workloads (512 new tokens over a 2048-token prefix; 2048
tokens from scratch; 32 heads of d=64), query tiles and prefixes that are not
multiples of the 128-row tile, a single new token, GQA head sharing and the
empty problem; a launch that reads the previous launch's output on the same
stream; and the same kernel at d_head=128 (small cases against the full
oracle, a 512-token GQA prompt chunk at the decode shapes, and one new token
through both the prefill and the decode kernel).
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, f64

pytestmark = pytest.mark.gpu


def _run(case):
    out = ga.attn_prefill_causal(case.q, case.k, case.v, case.start_pos, case.scale)
    assert ga.attn_read_prefill_status() == 0   # synchronises; no wait gave up
    return out


def _full_check(case, what):
    want = oracle.prefill(f64(case.q), f64(case.k), f64(case.v), case.start_pos, case.scale)
    got = f64(_run(case))
    return assert_attn_close(got, want, what)


def _sampled_check(case, rows, what):
    want = oracle.prefill_rows(f64(case.q), f64(case.k), f64(case.v), case.start_pos,
                               case.scale, rows)
    out = _run(case)
    got = np.stack([f64(out[i, h]) for i, h in rows])
    assert torch.isfinite(out.float()).all()
    return assert_attn_close(got, want, what)


@pytest.mark.parametrize("S,start_pos,Hq,Hkv", [
    (128, 0, 1, 1),      # one tile, no prefix
    (1, 0, 2, 2),        # a single token
    (100, 0, 2, 2),      # ragged single tile
    (129, 0, 2, 1),      # tile + 1 row, GQA g=2
    (300, 37, 4, 4),     # prefix not tile aligned
    (1, 500, 4, 2),      # one new token over a prefix (== a decode step)
    (128, 128, 2, 2),    # everything tile aligned
    (200, 127, 8, 2),    # GQA g=4, prefix one short of a tile
    (64, 129, 3, 1),     # g=3
])
def test_small_cases_full_oracle(S, start_pos, Hq, Hkv):
    case = synth.prefill_case(S=S, start_pos=start_pos, Hq=Hq, Hkv=Hkv, d=64,
                              seed=S + start_pos, device="cuda")
    _full_check(case, f"S={S} start_pos={start_pos} Hq={Hq} Hkv={Hkv}")


def test_prefill_prefix_workload():
    """32 heads, d=64, 2048 cached prefix tokens + 512 new tokens."""
    case = synth.generators.workload_case("prefill_prefix", seed=1, device="cuda")
    rng = np.random.default_rng(1)
    rows = [(int(i), int(h)) for i, h in zip(rng.integers(0, 512, 600), rng.integers(0, 32, 600))]
    rows += [(i, 5) for i in range(512)] + [(0, h) for h in range(32)] + [(511, h) for h in range(32)]
    _sampled_check(case, rows, "prefill_prefix")


def test_prefill_workload():
    """32 heads, d=64, 2048 tokens, no prefix (plain causal attention)."""
    case = synth.generators.workload_case("prefill", seed=2, device="cuda")
    rng = np.random.default_rng(2)
    rows = [(int(i), int(h)) for i, h in zip(rng.integers(0, 2048, 800), rng.integers(0, 32, 800))]
    rows += [(i, 17) for i in range(0, 2048, 3)] + [(0, h) for h in range(32)]
    rows += [(2047, h) for h in range(32)] + [(127, 0), (128, 0), (1023, 31)]
    _sampled_check(case, rows, "prefill")


def test_first_token_is_v0_and_empty_problem():
    case = synth.prefill_case(S=5, start_pos=0, Hq=2, Hkv=2, d=64, seed=9, device="cuda")
    out = _run(case)
    # token 0 sees key 0 only: softmax over one entry is exactly 1
    assert torch.equal(out[0].view(torch.int16), case.v[0].view(torch.int16))
    empty = synth.prefill_case(S=0, start_pos=10, Hq=2, Hkv=2, d=64, seed=1, device="cuda")
    ga.attn_prefill_causal(empty.q, empty.k, empty.v, empty.start_pos, empty.scale)


def test_prefill_matches_decode_path():
    """One new token over a prefix through both kernels (both against the
    oracle's definition, and against each other)."""
    start_pos, H, D = 1000, 8, 64
    case = synth.prefill_case(S=1, start_pos=start_pos, Hq=H, Hkv=H, d=D, seed=4, device="cuda")
    out = _run(case)
    want = oracle.prefill(f64(case.q), f64(case.k), f64(case.v), start_pos, case.scale)
    assert_attn_close(f64(out), want, "S=1 prefill")


def test_pair_items_with_a_ragged_last_tile():
    """Enough heads that work items hold two query tiles (each K/V tile
    serves both softmax lanes): 300 tokens are three query tiles, so the
    second item of each head has one tile and its second lane no work; GQA
    g=4 over a prefix that is not tile aligned."""
    case = synth.prefill_case(S=300, start_pos=37, Hq=160, Hkv=40, d=64, seed=91, device="cuda")
    rng = np.random.default_rng(91)
    rows = [(int(i), int(h)) for i, h in zip(rng.integers(0, 300, 700), rng.integers(0, 160, 700))]
    rows += [(i, 7) for i in range(300)] + [(i, 159) for i in range(0, 300, 7)]
    rows += [(0, h) for h in range(160)] + [(299, h) for h in range(160)]
    _sampled_check(case, rows, "pair items, ragged last tile")


@pytest.mark.parametrize("S,start_pos,Hq,Hkv,d", [
    (256, 300, 4, 2, 64),    # one query tile per item: the split-keys kernel
    (1024, 0, 40, 8, 64),    # pairs of query tiles per item
    (256, 100, 8, 2, 128),   # head dim 128
])
def test_back_to_back_launches_read_the_previous_output(S, start_pos, Hq, Hkv, d):
    """The prefill kernels may start while the previous kernel on the stream
    drains (programmatic dependent launch) and touch q, k, v and out only
    after it is done: a second prefill whose queries are the first one's
    output, queued without a synchronisation, sees all of that output."""
    case = synth.prefill_case(S=S, start_pos=start_pos, Hq=Hq, Hkv=Hkv, d=d, seed=S + d,
                              device="cuda")
    out1 = ga.attn_prefill_causal(case.q, case.k, case.v, start_pos, case.scale)
    out2 = ga.attn_prefill_causal(out1, case.k, case.v, start_pos, case.scale)
    assert ga.attn_read_prefill_status() == 0
    rng = np.random.default_rng(S + d)
    rows = [(int(i), int(h)) for i, h in zip(rng.integers(0, S, 300), rng.integers(0, Hq, 300))]
    rows += [(0, h) for h in range(Hq)] + [(S - 1, h) for h in range(Hq)]
    want = oracle.prefill_rows(f64(out1), f64(case.k), f64(case.v), start_pos, case.scale, rows)
    got = np.stack([f64(out2[i, h]) for i, h in rows])
    assert_attn_close(got, want, f"chained S={S} d={d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("sign", [0.0, -1.0])
def test_zero_and_negative_scale(d, sign):
    """A zero scale weighs every visible key alike; a negative one (the
    usual 1/sqrt(d), sign flipped) reverses the order of the scores, so the
    row's largest scaled score is the smallest raw one."""
    scale = sign / d ** 0.5
    case = synth.prefill_case(S=260, start_pos=70, Hq=4, Hkv=2, d=d, seed=93 + d, device="cuda",
                              scale=scale)
    _full_check(case, f"d={d} scale={scale}")


# ------------------------------------------------------------- d_head = 128 ---
# The decode model's head size: prompt chunks of a GQA model with D=128 go
# through the same kernel, each 128-wide row as two 128-byte column blocks.

@pytest.mark.parametrize("S,start_pos,Hq,Hkv", [
    (128, 0, 1, 1),      # one tile, no prefix
    (1, 0, 2, 2),        # a single token
    (129, 0, 2, 1),      # tile + 1 row, GQA g=2
    (300, 37, 4, 4),     # prefix not tile aligned
    (1, 500, 4, 2),      # one new token over a prefix (== a decode step)
    (200, 127, 16, 8),   # the decode shapes' g=2, prefix one short of a tile
    (64, 129, 8, 1),     # g=8
])
def test_d128_small_cases_full_oracle(S, start_pos, Hq, Hkv):
    case = synth.prefill_case(S=S, start_pos=start_pos, Hq=Hq, Hkv=Hkv, d=128,
                              seed=1000 + S + start_pos, device="cuda")
    _full_check(case, f"d=128 S={S} start_pos={start_pos} Hq={Hq} Hkv={Hkv}")


def test_d128_gqa_prompt_chunk():
    """A 512-token prompt chunk over a 2048-token cache at the decode shapes
    (Hq=32, Hkv=8, D=128), sampled rows against the oracle."""
    case = synth.prefill_case(S=512, start_pos=2048, Hq=32, Hkv=8, d=128, seed=77,
                              device="cuda")
    rng = np.random.default_rng(77)
    rows = [(int(i), int(h)) for i, h in zip(rng.integers(0, 512, 400), rng.integers(0, 32, 400))]
    rows += [(i, 9) for i in range(0, 512, 5)] + [(0, h) for h in range(32)]
    rows += [(511, h) for h in range(32)] + [(127, 3), (128, 3)]
    _sampled_check(case, rows, "d=128 prompt chunk")


def test_d128_first_token_is_v0_and_one_token_equals_decode():
    case = synth.prefill_case(S=3, start_pos=0, Hq=4, Hkv=2, d=128, seed=78, device="cuda")
    out = _run(case)
    assert torch.equal(out[0, 0].view(torch.int16), case.v[0, 0].view(torch.int16))
    assert torch.equal(out[0, 3].view(torch.int16), case.v[0, 1].view(torch.int16))
    # one new token over a 700-token prefix through prefill and through decode
    pc = synth.prefill_case(S=1, start_pos=700, Hq=16, Hkv=8, d=128, seed=79, device="cuda")
    pout = _run(pc)
    kc = pc.k.permute(1, 0, 2).unsqueeze(0).contiguous()  # [1, Hkv, 701, D]
    vc = pc.v.permute(1, 0, 2).unsqueeze(0).contiguous()
    pos = torch.tensor([700], dtype=torch.int32, device="cuda")
    dout = ga.attn_decode_step(pc.q, pos, kc, vc, pc.scale)
    torch.cuda.synchronize()
    want = oracle.prefill(f64(pc.q), f64(pc.k), f64(pc.v), 700, pc.scale)
    assert_attn_close(f64(pout), want, "d=128 one token (prefill)")
    assert_attn_close(f64(dout), want, "d=128 one token (decode)")
