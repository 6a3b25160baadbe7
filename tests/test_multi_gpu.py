"""Multi-token decode (attn_decode_multi) against the fp64 oracle's
decode_multi: S new tokens per sequence, token t at positions[b] + t attends
rows 0 .. positions[b] + t.

The S new rows are appended by the call (bit-exact) and every row past the
last new token holds NaN.  Covers both schedules (clusters for one or two
sequences, stream-K for many), S x g of 2, 4 and 8, new tokens straddling
128-row tile edges, one token equal to the plain decode bit for bit, a
sequence running off the end of the cache, and an unsupported S x g.
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, bits, f64

pytestmark = pytest.mark.gpu


def _case(B, S, Hq, Hkv, positions, seed, L=8192):
    """A decode case with S new tokens: q/k_new/v_new carry a token axis;
    the cache is NaN from the first new row on (the call writes the new rows,
    everything past them must never be read)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    rn = lambda *shape: torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    kc, vc = rn(B, Hkv, L, 128), rn(B, Hkv, L, 128)
    rows = torch.arange(L, device="cuda").view(1, 1, L)
    bad = (rows >= pos.view(B, 1, 1)).unsqueeze(-1).expand_as(kc)
    kc.masked_fill_(bad, float("nan"))
    vc.masked_fill_(bad, float("nan"))
    return rn(B, S, Hq, 128), rn(B, S, Hkv, 128), rn(B, S, Hkv, 128), pos, kc, vc


def _run_and_check(B, S, Hq, Hkv, positions, seed, what):
    q, kn, vn, pos, kc, vc = _case(B, S, Hq, Hkv, positions, seed)
    scale = 128 ** -0.5
    # oracle: the cache after writing the S new rows, up to the last new row
    want = {}
    for b, p in enumerate(positions):
        kcb = f64(kc[b:b + 1, :, : p + S])
        vcb = f64(vc[b:b + 1, :, : p + S])
        kcb[0, :, p:p + S] = f64(kn[b]).transpose(1, 0, 2)
        vcb[0, :, p:p + S] = f64(vn[b]).transpose(1, 0, 2)
        want[b] = oracle.decode_multi(f64(q[b:b + 1]), kcb, vcb, [p], scale)[0]
    out = ga.attn_decode_multi(q, pos, kc, vc, scale, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    for b, p in enumerate(positions):
        assert torch.equal(bits(kc[b, :, p:p + S].transpose(0, 1)), bits(kn[b])), f"{what} k b={b}"
        assert torch.equal(bits(vc[b, :, p:p + S].transpose(0, 1)), bits(vn[b])), f"{what} v b={b}"
        assert_attn_close(f64(out[b]), want[b], f"{what} b={b}")


POS16 = [0, 1, 60, 124, 125, 126, 127, 128, 250, 253, 1000, 4093, 4094, 8000, 7, 3001]


@pytest.mark.parametrize("S,Hq,Hkv", [(2, 4, 2), (4, 4, 2), (8, 2, 2), (2, 8, 2), (4, 2, 2),
                                      (2, 16, 2), (4, 8, 2), (16, 2, 2)])
def test_multi_stream_k(S, Hq, Hkv):
    """16 sequences (stream-K); S x g = 4, 8, 8, 8, 4, 16, 16, 16."""
    _run_and_check(16, S, Hq, Hkv, [min(p, 8192 - S) for p in POS16], 300 + S * Hq,
                   f"multi S={S} Hq={Hq} Hkv={Hkv} stream-K")


@pytest.mark.parametrize("S,Hq,Hkv", [(2, 16, 8), (4, 16, 8), (2, 32, 8), (2, 64, 8)])
def test_multi_clusters(S, Hq, Hkv):
    """One or two sequences at the decode shapes (cluster mode)."""
    _run_and_check(1, S, Hq, Hkv, [4094], 310 + S, f"multi S={S} Hq={Hq} B=1")
    _run_and_check(2, S, Hq, Hkv, [126, 8190 - S], 311 + S, f"multi S={S} Hq={Hq} B=2")


@pytest.mark.parametrize("Hq,Hkv", [(16, 8), (64, 8), (32, 2)])
def test_one_token_is_the_plain_decode(Hq, Hkv):
    """S = 1 writes the same cache bits as the fused append step.  At g = 2
    and 8 (the per-warp MMA kernels) the outputs are the same bits too.  At
    g = 16 (tcgen05 kernels) the fused step folds its new row in fp32 on the
    side, while the multi-token path reads it back through the tile, so
    there the two agree to rounding, within the attention tolerance."""
    q, kn, vn, pos, kc, vc = _case(3, 1, Hq, Hkv, [5, 700, 8191], 320)
    kc2, vc2 = kc.clone(), vc.clone()
    out = ga.attn_decode_multi(q, pos, kc, vc, 0.088, k_new=kn, v_new=vn)
    ref = ga.attn_decode_step_append(q[:, 0].contiguous(), kn[:, 0].contiguous(),
                                     vn[:, 0].contiguous(), pos, kc2, vc2, 0.088)
    torch.cuda.synchronize()
    assert torch.equal(bits(kc), bits(kc2))
    assert torch.equal(bits(vc), bits(vc2))
    if Hq // Hkv <= 8:
        assert torch.equal(bits(out[:, 0]), bits(ref))
    else:
        assert_attn_close(f64(out[:, 0]), f64(ref), "multi S=1 against the fused step")


def test_multi_out_of_range_and_unsupported():
    L = 512
    q, kn, vn, pos, kc, vc = _case(3, 4, 8, 4, [10, L - 3, 200], 330, L=L)
    k_before = kc.clone()
    ws = ga.decode_workspace(3, 4 * 8, 4, L, 128)
    out = ga.attn_decode_multi(q, pos, kc, vc, 0.088, k_new=kn, v_new=vn, workspace=ws)
    assert ga.attn_read_device_status(ws) & ga.ATTN_DEV_BAD_POSITION
    assert torch.isnan(out[1].float()).all()
    assert torch.equal(bits(kc[1]), bits(k_before[1]))
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(out[2].float()).all()
    with pytest.raises(ga.AttnError):
        ga.attn_decode_multi(torch.zeros(1, 3, 16, 128, dtype=torch.bfloat16, device="cuda"),
                             pos[:1], kc[:1], vc[:1], 0.088)


@pytest.mark.parametrize("B,S,Hq,Hkv", [(1, 2, 16, 8), (1, 4, 16, 8), (12, 2, 8, 4),
                                        (12, 2, 16, 2)])
def test_multi_positions_near_int_max(B, S, Hq, Hkv):
    """A first-token position so large that position + S - 1 overflows a
    32-bit int must be rejected like any other out-of-range position: status
    bit, NaN output rows, and no byte of the cache written (the row index
    of such a token, taken in 64 bits, would lie far outside the cache).
    Covers a cluster launch (B=1), stream-K (B=12) and the tensor-core
    kernels (S x g = 16)."""
    L = 1024
    big = [2 ** 31 - 1, 2 ** 31 - 2, 2 ** 31 - S + 1]
    positions = [(big[b % 3] if b % 2 == 0 else 100 + 37 * b) for b in range(B)]
    q, kn, vn, pos, kc, vc = _case(B, S, Hq, Hkv, [min(p, L - S) for p in positions], 340 + B,
                                   L=L)
    pos.copy_(torch.tensor(positions, dtype=torch.int32, device="cuda"))
    k_before, v_before = kc.clone(), vc.clone()
    ws = ga.decode_workspace(B, S * Hq, Hkv, L, 128)
    out = ga.attn_decode_multi(q, pos, kc, vc, 0.088, k_new=kn, v_new=vn, workspace=ws)
    assert ga.attn_read_device_status(ws) & ga.ATTN_DEV_BAD_POSITION
    for b, p in enumerate(positions):
        if p >= L:
            assert torch.isnan(out[b].float()).all(), f"b={b}"
            assert torch.equal(bits(kc[b]), bits(k_before[b])), f"k b={b}"
            assert torch.equal(bits(vc[b]), bits(v_before[b])), f"v b={b}"
        else:
            assert torch.isfinite(out[b].float()).all(), f"b={b}"
            assert torch.equal(bits(kc[b, :, p:p + S].transpose(0, 1)), bits(kn[b])), f"b={b}"
