"""Decode step with the rotary embedding (attn_decode_step_rope_append)
against the fp64 oracle's decode_rope_step.

The cache row written at positions[b] must equal the oracle's rotated key,
rounded to bf16, bit for bit; the value row is the unrotated v_new; the output
is attention of the rotated query over rows 0..positions[b] within the decode
tolerance.  Covers both schedules (clusters for a few sequences, stream-K for
many), every group size, tile boundaries with NaN-poisoned rows past each
position, the ragged B=64 workload at full size (sampled outputs, every
appended row), a run of consecutive steps whose rotated rows are read back
from the cache, the identity rotation (bit-identical to the plain fused
step) and an out-of-range position.
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, bits, f64

pytestmark = pytest.mark.gpu


def _oracle(case, cos, sin, bs):
    """Oracle outputs {(b, h): row} and rotated key rows {b: [Hkv, D]} for
    sequences bs, from the pre-append inputs (call before the kernel runs)."""
    Hq = case.q.shape[1]
    out, krow = {}, {}
    cos_n, sin_n = cos.cpu().numpy(), sin.cpu().numpy()
    for b in bs:
        p = int(case.positions[b])
        o, kc, _ = oracle.decode_rope_step(
            f64(case.q[b:b + 1]), f64(case.k_new[b:b + 1]), f64(case.v_new[b:b + 1]),
            cos_n[b:b + 1], sin_n[b:b + 1], f64(case.k_cache[b:b + 1, :, : p + 1]),
            f64(case.v_cache[b:b + 1, :, : p + 1]), [p], case.scale)
        for h in range(Hq):
            out[(b, h)] = o[0, h]
        krow[b] = kc[0, :, p]
    return out, krow


def _rotated_keys(case, cos, sin):
    """The oracle's rotated new key rows of every sequence, as bf16 values."""
    kr = oracle.rope_f32(f64(case.k_new), cos.cpu().numpy()[:, None, :], sin.cpu().numpy()[:, None, :])
    return oracle.round_bf16(kr)


def _step(case, cos, sin, workspace=None):
    out = ga.attn_decode_step_rope_append(case.q, case.k_new, case.v_new, cos, sin,
                                          case.positions, case.k_cache, case.v_cache,
                                          case.scale, workspace=workspace)
    torch.cuda.synchronize()
    return out


def _check_out(want, out, what):
    keys = sorted(want)
    got = np.stack([f64(out[b, h]) for b, h in keys])
    ref = np.stack([want[k] for k in keys])
    assert_attn_close(got, ref, what)


def _check_rows(case, krow, v_new, bs):
    for b in bs:
        p = int(case.positions[b])
        want = torch.from_numpy(krow[b]).to(torch.bfloat16)
        assert torch.equal(bits(case.k_cache[b, :, p].cpu()), bits(want)), f"k row b={b}"
        assert torch.equal(bits(case.v_cache[b, :, p].cpu()), bits(v_new[b].cpu())), f"v row b={b}"


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_rope_boundaries_stream_k(g):
    """16 sequences x 2 KV heads (stream-K), positions at tile edges."""
    Hkv = 2
    positions = [0, 1, 62, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 4095, 4096, 8191]
    case = synth.decode_case(B=len(positions), Hq=g * Hkv, Hkv=Hkv, D=128, L=8192,
                             positions=positions, fill="all", poison=True, seed=40 + g,
                             device="cuda")
    cos, sin = synth.rope_tables(case.positions, 128, device="cuda")
    want, krow = _oracle(case, cos, sin, range(len(positions)))
    v_new = case.v_new.clone()
    out = _step(case, cos, sin)
    _check_out(want, out, f"rope stream-K g={g}")
    _check_rows(case, krow, v_new, range(len(positions)))


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_rope_few_sequences_cluster(g):
    """3 sequences x 2 KV heads (cluster mode)."""
    Hkv = 2
    positions = [0, 129, 8191]
    case = synth.decode_case(B=3, Hq=g * Hkv, Hkv=Hkv, D=128, L=8192, positions=positions,
                             fill="all", poison=True, seed=50 + g, device="cuda")
    cos, sin = synth.rope_tables(case.positions, 128, device="cuda")
    want, krow = _oracle(case, cos, sin, range(3))
    v_new = case.v_new.clone()
    out = _step(case, cos, sin)
    _check_out(want, out, f"rope cluster g={g}")
    _check_rows(case, krow, v_new, range(3))


def test_rope_ragged_workload_full_size():
    """B=64, Hq=32, Hkv=8, L=8192, positions uniform: every appended key row
    bit-exact, outputs of 6 sequences against the oracle."""
    case = synth.generators.workload_case("ragged", seed=61, device="cuda")
    cos, sin = synth.rope_tables(case.positions, 128, base=1e6, device="cuda")
    bs = [0, 7, 21, 33, 50, 63]
    want, _ = _oracle(case, cos, sin, bs)
    kr = _rotated_keys(case, cos, sin)
    v_new = case.v_new.clone()
    out = _step(case, cos, sin)
    _check_out(want, out, "rope ragged")
    pos = case.positions.long().cpu()
    idx = torch.arange(64, device="cuda")
    got = case.k_cache[idx, :, pos.cuda()].cpu()  # [B, Hkv, D]
    assert torch.equal(bits(got), bits(torch.from_numpy(kr).to(torch.bfloat16)))
    assert torch.equal(bits(case.v_cache[idx, :, pos.cuda()].cpu()), bits(v_new.cpu()))


def test_rope_consecutive_steps_read_back_rotated_rows():
    """B=1, Hq=16, Hkv=8: 300 steps from position 0 (the streaming shape),
    then the cache prefix and the last output against the oracle."""
    steps, Hq, Hkv, D, L = 300, 16, 8, 128, 8192
    q, kn, vn, pos = synth.streaming_inputs(steps=steps, B=1, Hq=Hq, Hkv=Hkv, D=D, seed=62,
                                            device="cuda")
    cos, sin = synth.rope_tables(torch.arange(steps), D, device="cuda")
    kc = torch.zeros((1, Hkv, L, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ws = ga.decode_workspace(1, Hq, Hkv, L, D)
    scale = D ** -0.5
    for s in range(steps):
        out = ga.attn_decode_step_rope_append(q[s], kn[s], vn[s], cos[s:s + 1], sin[s:s + 1],
                                              pos[s], kc, vc, scale, workspace=ws)
    torch.cuda.synchronize()
    cos_n, sin_n = cos.cpu().numpy(), sin.cpu().numpy()
    kr = oracle.round_bf16(oracle.rope_f32(f64(kn[:, 0]), cos_n[:, None, :], sin_n[:, None, :]))
    assert torch.equal(bits(kc[0, :, :steps].cpu()),
                       bits(torch.from_numpy(kr.transpose(1, 0, 2).copy()).to(torch.bfloat16)))
    assert torch.equal(bits(vc[0, :, :steps].cpu()), bits(vn[:, 0].transpose(0, 1).cpu()))
    qr = oracle.rope_f32(f64(q[steps - 1]), cos_n[steps - 1][None, None, :],
                         sin_n[steps - 1][None, None, :])
    want = oracle.decode(qr.astype(np.float64), f64(kc[:, :, :steps]), f64(vc[:, :, :steps]),
                         [steps - 1], scale)
    assert_attn_close(f64(out), want, "rope steps")


def test_rope_identity_equals_plain_fused_step():
    """cos = 1, sin = 0: q and k are unchanged, so output and cache are bit
    for bit those of attn_decode_step_append."""
    positions = [5, 300, 4100]
    a = synth.decode_case(B=3, Hq=32, Hkv=8, D=128, L=8192, positions=positions, fill="all",
                          seed=63, device="cuda")
    b = synth.decode_case(B=3, Hq=32, Hkv=8, D=128, L=8192, positions=positions, fill="all",
                          seed=63, device="cuda")
    one = torch.ones((3, 128), dtype=torch.float32, device="cuda")
    zero = torch.zeros_like(one)
    out_r = _step(a, one, zero)
    out_p = ga.attn_decode_step_append(b.q, b.k_new, b.v_new, b.positions, b.k_cache, b.v_cache,
                                       b.scale)
    torch.cuda.synchronize()
    assert torch.equal(bits(out_r), bits(out_p))
    assert torch.equal(bits(a.k_cache), bits(b.k_cache))
    assert torch.equal(bits(a.v_cache), bits(b.v_cache))


def test_rope_out_of_range_position():
    """positions[1] = L: NaN rows for sequence 1, no cache write, status bit;
    the other sequences are unaffected."""
    L = 512
    case = synth.decode_case(B=3, Hq=8, Hkv=2, D=128, L=L, positions=[10, L, 300], fill="all",
                             seed=64, device="cuda")
    cos, sin = synth.rope_tables(torch.tensor([10, 0, 300]), 128, device="cuda")
    want, krow = _oracle(case, cos, sin, [0, 2])
    k_before = case.k_cache.clone()
    v_new = case.v_new.clone()
    ws = ga.decode_workspace(3, 8, 2, L, 128)
    out = _step(case, cos, sin, workspace=ws)
    assert torch.isnan(out[1].float()).all()
    assert torch.equal(bits(case.k_cache[1]), bits(k_before[1]))
    assert ga.attn_read_device_status(ws) & ga.ATTN_DEV_BAD_POSITION
    _check_out(want, out, "rope bad position")
    _check_rows(case, krow, v_new, [0, 2])


def test_rope_rejects_bad_tables():
    case = synth.decode_case(B=2, Hq=8, Hkv=2, D=128, L=64, positions=[1, 2], device="cuda")
    cos, sin = synth.rope_tables(case.positions, 128, device="cuda")
    with pytest.raises(ValueError):
        ga.attn_decode_step_rope_append(case.q, case.k_new, case.v_new, cos[:1], sin[:1],
                                        case.positions, case.k_cache, case.v_cache, case.scale)
    with pytest.raises(TypeError):
        ga.attn_decode_step_rope_append(case.q, case.k_new, case.v_new, cos.double(),
                                        sin.double(), case.positions, case.k_cache,
                                        case.v_cache, case.scale)
