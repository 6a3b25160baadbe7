"""Local-window decode (attn_decode_step_window) against the fp64 oracle's
decode_window: each sequence attends rows max(0, pos - W + 1) .. pos only.

Every row outside the window (before it and after the position) holds NaN,
so a read outside the window shows up in the output.  Covers both schedules
(clusters for a few sequences, stream-K for many), every group size, windows
of 1, across tile edges and wider than the position, the fused append, the
full-size ragged batch, and a wide window being bit-identical to the plain
decode.
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, bits, f64

pytestmark = pytest.mark.gpu

POSITIONS = [0, 1, 63, 127, 128, 129, 255, 256, 700, 1000, 4095, 4096, 8000, 8191, 5, 3000]


def _poison_outside(case, window):
    """NaN into every row outside [pos - W + 1, pos] (the rows after pos are
    already NaN when the case was drawn with poison=True)."""
    for b, p in enumerate(case.positions.tolist()):
        lo = max(0, p - window + 1)
        if lo > 0:
            case.k_cache[b, :, :lo] = float("nan")
            case.v_cache[b, :, :lo] = float("nan")


def _want(case, window, bs=None):
    B = case.q.shape[0]
    bs = range(B) if bs is None else bs
    pos = case.positions.tolist()
    out = {}
    for b in bs:
        p = pos[b]
        lo = max(0, p - window + 1)
        # the window rows only (finite), shifted to start at row 0
        kc = f64(case.k_cache[b:b + 1, :, lo:p + 1])
        vc = f64(case.v_cache[b:b + 1, :, lo:p + 1])
        out[b] = oracle.decode_window(f64(case.q[b:b + 1]), kc, vc, [p - lo], case.scale, window)[0]
    return out


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("window", [1, 7, 128, 129, 1000])
def test_window_stream_k(g, window):
    """16 sequences x 2 KV heads (stream-K)."""
    Hkv = 2
    case = synth.decode_case(B=16, Hq=g * Hkv, Hkv=Hkv, D=128, L=8192, positions=POSITIONS,
                             fill="all", poison=True, seed=200 + g, device="cuda")
    _poison_outside(case, window)
    want = _want(case, window)
    out = ga.attn_decode_step_window(case.q, case.positions, case.k_cache, case.v_cache,
                                     case.scale, window)
    torch.cuda.synchronize()
    got = np.stack([f64(out[b]) for b in range(16)])
    ref = np.stack([want[b] for b in range(16)])
    assert_attn_close(got, ref, f"window={window} g={g} stream-K")


@pytest.mark.parametrize("g", [2, 8])
@pytest.mark.parametrize("window", [1, 300, 4096])
def test_window_clusters_with_append(g, window):
    """2 sequences x 4 KV heads (cluster mode), new rows appended first."""
    Hkv = 4
    case = synth.decode_case(B=2, Hq=g * Hkv, Hkv=Hkv, D=128, L=8192, positions=[4200, 8191],
                             fill="all", poison=True, seed=210 + g, device="cuda")
    _poison_outside(case, window)
    pos = case.positions.tolist()
    kc = case.k_cache.clone()  # the oracle's cache after the append
    vc = case.v_cache.clone()
    for b in range(2):
        kc[b, :, pos[b]] = case.k_new[b]
        vc[b, :, pos[b]] = case.v_new[b]
    want = {}
    for b in range(2):
        lo = max(0, pos[b] - window + 1)
        want[b] = oracle.decode_window(f64(case.q[b:b + 1]), f64(kc[b:b + 1, :, lo:pos[b] + 1]),
                                       f64(vc[b:b + 1, :, lo:pos[b] + 1]), [pos[b] - lo],
                                       case.scale, window)[0]
    out = ga.attn_decode_step_window(case.q, case.positions, case.k_cache, case.v_cache,
                                     case.scale, window, k_new=case.k_new, v_new=case.v_new)
    torch.cuda.synchronize()
    for b in range(2):
        assert torch.equal(bits(case.k_cache[b, :, pos[b]]), bits(case.k_new[b]))
        assert torch.equal(bits(case.v_cache[b, :, pos[b]]), bits(case.v_new[b]))
        assert_attn_close(f64(out[b]), want[b], f"window={window} g={g} clusters b={b}")


def test_window_ragged_workload_full_size():
    """B=64, Hq=32, Hkv=8, L=8192, positions uniform, W=1024: 6 sequences."""
    case = synth.generators.workload_case("ragged", seed=220, device="cuda")
    W = 1024
    _poison_outside(case, W)
    bs = [0, 9, 27, 38, 51, 63]
    want = _want(case, W, bs)
    out = ga.attn_decode_step_window(case.q, case.positions, case.k_cache, case.v_cache,
                                     case.scale, W)
    torch.cuda.synchronize()
    assert_attn_close(np.stack([f64(out[b]) for b in bs]), np.stack([want[b] for b in bs]),
                      "window ragged")


def test_wide_window_is_bit_identical_to_plain_decode():
    case = synth.decode_case(B=5, Hq=32, Hkv=8, D=128, L=8192, positions=[0, 99, 1234, 5000, 8191],
                             fill="all", seed=221, device="cuda")
    plain = ga.attn_decode_step(case.q, case.positions, case.k_cache, case.v_cache, case.scale)
    for W in (8192, 10 ** 6):
        win = ga.attn_decode_step_window(case.q, case.positions, case.k_cache, case.v_cache,
                                         case.scale, W)
        torch.cuda.synchronize()
        assert torch.equal(bits(win), bits(plain))
