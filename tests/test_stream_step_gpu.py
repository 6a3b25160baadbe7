"""Streaming step with the position advanced on the device
(attn_decode_stream_step): one captured CUDA graph replayed step after step.

Checks against the fp64 oracle: the appended (and, with rotation tables,
rotated) rows bit-exact, sampled outputs within tolerance, positions advanced
by one per step, both schedules (clusters for B=1, stream-K for a ragged
batch), a position that runs off the end of the cache (NaN rows, status bit,
still advanced), and bit-identity with the fused step at host-side positions.
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, bits, f64

pytestmark = pytest.mark.gpu


def _tables(L, D=128, base=10000.0):
    return synth.rope_tables(torch.arange(L), D, base=base, device="cuda")


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("Hq", [16, 64])
def test_graph_replayed_stream_b1(rope, Hq):
    """B=1, Hkv=8: one captured step replayed 200 times from position 0, fresh
    q/k/v copied in before each replay.  Hq=16 (g=2, the streaming shapes)
    runs the per-warp MMA kernels; Hq=64 (g=8) runs them too without the
    rotation, and the tcgen05 kernels with it."""
    steps, Hkv, D, L = 200, 8, 128, 1024
    q, kn, vn, _ = synth.streaming_inputs(steps=steps, B=1, Hq=Hq, Hkv=Hkv, D=D, seed=90,
                                          device="cuda")
    cos, sin = _tables(L) if rope else (None, None)
    kc = torch.zeros((1, Hkv, L, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    qb, kb, vb = q[0].clone(), kn[0].clone(), vn[0].clone()
    ob = torch.empty_like(qb)
    ws = ga.decode_workspace(1, Hq, Hkv, L, D)
    scale = D ** -0.5
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up launch at position 0 (re-done by replay 0)
        ga.attn_decode_stream_step(qb, kb, vb, pos, kc, vc, scale, cos, sin, out=ob, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    pos.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ga.attn_decode_stream_step(qb, kb, vb, pos, kc, vc, scale, cos, sin, out=ob, workspace=ws)
    torch.cuda.synchronize()
    assert int(pos.item()) == 0  # capture does not run the step
    outs = []
    for t in range(steps):
        qb.copy_(q[t])
        kb.copy_(kn[t])
        vb.copy_(vn[t])
        g.replay()
        outs.append(ob.clone())
    torch.cuda.synchronize()
    assert int(pos.item()) == steps
    # cache rows 0..steps-1: the (rotated) keys, the values as given
    if rope:
        kr = oracle.round_bf16(oracle.rope_f32(f64(kn[:, 0]), cos[:steps, None].cpu().numpy(),
                                               sin[:steps, None].cpu().numpy()))
    else:
        kr = f64(kn[:, 0])
    want_k = torch.from_numpy(np.ascontiguousarray(kr.transpose(1, 0, 2))).to(torch.bfloat16)
    assert torch.equal(bits(kc[0, :, :steps].cpu()), bits(want_k))
    assert torch.equal(bits(vc[0, :, :steps].cpu()), bits(vn[:, 0].transpose(0, 1).cpu()))
    assert not kc[0, :, steps:].any()
    for t in (0, 1, 127, 128, 129, steps - 1):
        qt = f64(q[t])
        if rope:
            qt = oracle.rope_f32(qt, cos[t].cpu().numpy(), sin[t].cpu().numpy()).astype(np.float64)
        want = oracle.decode(qt, f64(kc[:, :, : t + 1]), f64(vc[:, :, : t + 1]), [t], scale)
        assert_attn_close(f64(outs[t]), want, f"stream step {t} rope={rope}")


@pytest.mark.parametrize("rope", [False, True])
def test_stream_steps_ragged_batch(rope):
    """B=64, Hq=32, Hkv=8 at ragged positions (stream-K), three steps; one
    sequence starts at L-1 and runs off the end of the cache on step 2."""
    L = 2048
    case = synth.decode_case(B=64, Hq=32, Hkv=8, D=128, L=L, positions="uniform", fill="all",
                             seed=91, device="cuda")
    case.positions[5] = L - 1
    start = case.positions.clone()
    cos, sin = _tables(L, base=5e5) if rope else (None, None)
    ws = ga.decode_workspace(64, 32, 8, L, 128)
    check_b = [0, 5, 17, 40, 63]
    for step in range(3):
        pos_now = (start + step).cpu()
        kc0 = case.k_cache.clone()
        vc0 = case.v_cache.clone()
        out = ga.attn_decode_stream_step(case.q, case.k_new, case.v_new, case.positions,
                                         case.k_cache, case.v_cache, case.scale, cos, sin,
                                         workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(case.positions.cpu(), pos_now + 1)
        status = ga.attn_read_device_status(ws)
        assert bool(status & ga.ATTN_DEV_BAD_POSITION) == (step >= 1)
        for b in check_b:
            p = int(pos_now[b])
            if p >= L:
                assert torch.isnan(out[b].float()).all()
                assert torch.equal(bits(case.k_cache[b]), bits(kc0[b]))
                continue
            qb_ = f64(case.q[b:b + 1])
            kn_ = f64(case.k_new[b:b + 1])
            if rope:
                c = cos[p].cpu().numpy()[None, None]
                s_ = sin[p].cpu().numpy()[None, None]
                qb_ = oracle.rope_f32(qb_, c, s_).astype(np.float64)
                kn_ = oracle.round_bf16(oracle.rope_f32(kn_, c, s_))
            kc, vc = oracle.kv_append(f64(kc0[b:b + 1, :, : p + 1]), f64(vc0[b:b + 1, :, : p + 1]),
                                      kn_, f64(case.v_new[b:b + 1]), [p])
            assert torch.equal(bits(case.k_cache[b, :, p].cpu()),
                               bits(torch.from_numpy(kc[0, :, p]).to(torch.bfloat16)))
            want = oracle.decode(qb_, kc, vc, [p], case.scale)
            assert_attn_close(f64(out[b:b + 1]), want, f"ragged stream step {step} b={b}")


def test_stream_step_equals_fused_step():
    """Same inputs: attn_decode_stream_step and attn_decode_step_rope_append
    (with the table rows gathered at the positions) give bit-identical
    outputs and caches; only the positions differ (advanced by one)."""
    L = 4096
    mk = lambda: synth.decode_case(B=3, Hq=16, Hkv=8, D=128, L=L, positions=[7, 1500, 4095],
                                   fill="all", seed=92, device="cuda")
    a, b = mk(), mk()
    cos, sin = _tables(L)
    pl = b.positions.long()
    out_a = ga.attn_decode_stream_step(a.q, a.k_new, a.v_new, a.positions, a.k_cache, a.v_cache,
                                       a.scale, cos, sin)
    out_b = ga.attn_decode_step_rope_append(b.q, b.k_new, b.v_new, cos[pl].contiguous(),
                                            sin[pl].contiguous(), b.positions, b.k_cache,
                                            b.v_cache, b.scale)
    torch.cuda.synchronize()
    assert torch.equal(bits(out_a), bits(out_b))
    assert torch.equal(bits(a.k_cache), bits(b.k_cache))
    assert torch.equal(bits(a.v_cache), bits(b.v_cache))
    assert torch.equal(a.positions, b.positions + 1)
