"""attn_kv_append against the oracle: bit-exact, and no other byte changes."""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import bits

pytestmark = pytest.mark.gpu


def _guarded(shape, fill_bits, device="cuda"):
    """A bf16 tensor embedded in a larger buffer whose guard regions hold a
    known pattern; returns (view, whole buffer)."""
    n = int(np.prod(shape))
    guard = 4096
    buf = torch.full((n + 2 * guard,), fill_bits, dtype=torch.int16, device=device)
    view = buf[guard:guard + n].view(torch.bfloat16).view(shape)
    return view, buf, guard


@pytest.mark.parametrize("B,Hkv,L,D,positions", [
    (1, 8, 8192, 128, [100]),
    (4, 8, 64, 128, [0, 63, 17, 1]),
    (3, 2, 33, 64, [32, 0, 5]),
    (64, 8, 512, 128, "uniform"),
])
def test_append_bit_exact(B, Hkv, L, D, positions):
    case = synth.decode_case(B=B, Hq=Hkv, Hkv=Hkv, D=D, L=L, positions=positions,
                             fill="all", poison=True, seed=7, device="cuda")
    kc, kbuf, guard = _guarded(case.k_cache.shape, 0x1234)
    vc, vbuf, _ = _guarded(case.v_cache.shape, 0x4321)
    kc.copy_(case.k_cache)
    vc.copy_(case.v_cache)
    ga.attn_kv_append(case.k_new, case.v_new, case.positions, kc, vc)
    torch.cuda.synchronize()
    # oracle on raw 16-bit patterns (the copy must be exact, NaN payloads too)
    pos = case.positions.cpu().numpy()
    wk, wv = oracle.kv_append(bits(case.k_cache).cpu().numpy(), bits(case.v_cache).cpu().numpy(),
                              bits(case.k_new).cpu().numpy(), bits(case.v_new).cpu().numpy(), pos)
    assert np.array_equal(bits(kc).cpu().numpy(), wk)
    assert np.array_equal(bits(vc).cpu().numpy(), wv)
    # guard regions untouched
    assert torch.all(kbuf[:guard] == 0x1234) and torch.all(kbuf[-guard:] == 0x1234)
    assert torch.all(vbuf[:guard] == 0x4321) and torch.all(vbuf[-guard:] == 0x4321)


def test_append_skips_out_of_range_positions():
    case = synth.decode_case(B=3, Hq=2, Hkv=2, D=128, L=16, positions=[3, 16, -1],
                             fill="all", seed=3, device="cuda")
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    ga.attn_kv_append(case.k_new, case.v_new, case.positions, kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(bits(kc[1:]), bits(case.k_cache[1:]))
    assert torch.equal(bits(vc[1:]), bits(case.v_cache[1:]))
    assert torch.equal(bits(kc[0, :, 3]), bits(case.k_new[0]))
