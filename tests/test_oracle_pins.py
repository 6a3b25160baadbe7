"""Pins for the CPU oracle: it is checked against things other than itself.

* hand-derived closed forms (tests/golden/closed_form.json);
* a pure-Python brute force (oracle.brute) on tiny shapes, every position;
* PyTorch's library scaled_dot_product_attention in fp64 on CPU, called the
  two ways the decode page calls it (sliced cache with enable_gqa, section
  4.1; full-length cache with the boolean mask arange(L) <= pos, section
  2.1/2.3) and the way the prefill page calls it (is_causal for a prompt with
  no prefix);
* closed forms: position 0 returns V[0] exactly; identical keys or a zero
  query return the mean of V[0..pos];
* invariances: key-row permutation, GQA == repeat-KV MHA, prefill of one
  token == a decode step, prefix prefill == tail rows of a full prefill.

``test_planted_mistakes_are_caught`` plants plausible mistakes in the oracle
(monkeypatching its named steps) and checks that the pins above catch each.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import attention as oatt
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def _nested(x):
    if isinstance(x, list):
        return np.array([_nested(e) for e in x], dtype=np.float64)
    return float(x)  # handles "nan"


def _rand(rng, shape, bf16=True):
    x = rng.standard_normal(shape).astype(np.float32)
    if bf16:
        x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    return x.astype(np.float64)


def _poison_after(cache, positions):
    c = cache.copy()
    for b, p in enumerate(positions):
        c[b, :, int(p) + 1:, :] = np.nan
    return c


# ---------------------------------------------------------------- golden ----

def test_golden_closed_forms():
    with open(GOLDEN) as f:
        g = json.load(f)
    for case in g["decode"]:
        out = oracle.decode(_nested(case["q"]), _nested(case["k_cache"]),
                            _nested(case["v_cache"]), case["positions"], case["scale"])
        np.testing.assert_allclose(out, _nested(case["expected"]), rtol=0, atol=1e-12,
                                   err_msg=case["why"])
    for case in g["prefill"]:
        out = oracle.prefill(_nested(case["q"]), _nested(case["k"]), _nested(case["v"]),
                             case["start_pos"], case["scale"])
        np.testing.assert_allclose(out, _nested(case["expected"]), rtol=0, atol=1e-12,
                                   err_msg=case["why"])


# ------------------------------------------------------------ brute force ---

@pytest.mark.parametrize("B,Hq,Hkv,D", [(1, 1, 1, 4), (2, 4, 2, 8), (1, 4, 1, 3), (2, 2, 2, 5)])
def test_brute_force_decode_every_position(B, Hq, Hkv, D):
    rng = np.random.default_rng(B * 100 + Hq * 10 + D)
    L = 7
    for pos in range(L):
        positions = [pos] * B if B == 1 else [pos, (pos * 3) % L]
        q = _rand(rng, (B, Hq, D))
        kc = _rand(rng, (B, Hkv, L, D))
        vc = _rand(rng, (B, Hkv, L, D))
        scale = 1.0 / math.sqrt(D)
        got = oracle.decode(q, kc, vc, positions, scale)
        want = np.array(brute.decode(q.tolist(), kc.tolist(), vc.tolist(), positions, scale))
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("S,start_pos,Hq,Hkv,d", [(1, 0, 1, 1, 4), (4, 0, 2, 2, 3),
                                                  (3, 2, 4, 2, 4), (5, 3, 2, 1, 2)])
def test_brute_force_prefill(S, start_pos, Hq, Hkv, d):
    rng = np.random.default_rng(S * 7 + start_pos)
    T = start_pos + S
    q = _rand(rng, (S, Hq, d))
    k = _rand(rng, (T, Hkv, d))
    v = _rand(rng, (T, Hkv, d))
    got = oracle.prefill(q, k, v, start_pos, 0.37)
    want = np.array(brute.prefill(q.tolist(), k.tolist(), v.tolist(), start_pos, 0.37))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ library SDPA pins ---

def _sdpa_decode_sliced(q, kc, vc, positions, scale):
    """The decode page's patched call, section 4.1, per sequence."""
    outs = []
    for b, p in enumerate(positions):
        qq = torch.from_numpy(q[b]).view(1, q.shape[1], 1, q.shape[2])
        kk = torch.from_numpy(kc[b, :, : int(p) + 1]).unsqueeze(0)
        vv = torch.from_numpy(vc[b, :, : int(p) + 1]).unsqueeze(0)
        o = F.scaled_dot_product_attention(qq, kk, vv, scale=scale, enable_gqa=True)
        outs.append(o.view(q.shape[1], q.shape[2]).numpy())
    return np.stack(outs)


def _sdpa_decode_masked(q, kc, vc, positions, scale):
    """The decode page's original call, section 2.1/2.3: full cache, bool mask."""
    L = kc.shape[2]
    outs = []
    for b, p in enumerate(positions):
        mask = (torch.arange(L) <= int(p)).view(1, L)
        qq = torch.from_numpy(q[b]).view(1, q.shape[1], 1, q.shape[2])
        kk = torch.from_numpy(kc[b]).unsqueeze(0)
        vv = torch.from_numpy(vc[b]).unsqueeze(0)
        o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale,
                                           enable_gqa=True)
        outs.append(o.view(q.shape[1], q.shape[2]).numpy())
    return np.stack(outs)


@pytest.mark.parametrize("B,Hq,Hkv,D,L", [(1, 16, 8, 128, 300), (3, 8, 2, 64, 64),
                                          (2, 8, 8, 32, 40), (2, 8, 1, 16, 33)])
def test_library_sdpa_decode(B, Hq, Hkv, D, L):
    rng = np.random.default_rng(L + Hq)
    positions = [int(x) for x in rng.integers(0, L, size=B)]
    positions[0] = L - 1
    q = _rand(rng, (B, Hq, D))
    kc = _rand(rng, (B, Hkv, L, D))
    vc = _rand(rng, (B, Hkv, L, D))
    scale = 1.0 / math.sqrt(D)
    got = oracle.decode(q, kc, vc, positions, scale)
    np.testing.assert_allclose(got, _sdpa_decode_sliced(q, kc, vc, positions, scale),
                               rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(got, _sdpa_decode_masked(q, kc, vc, positions, scale),
                               rtol=1e-11, atol=1e-12)


def test_masked_full_equals_sliced_with_poisoned_tail():
    """Section 3 of the decode page: slicing 0..pos is the same as masking."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, L = 3, 4, 2, 16, 50
    positions = [0, 17, 49]
    q = _rand(rng, (B, Hq, D))
    kc = _poison_after(_rand(rng, (B, Hkv, L, D)), positions)
    vc = _poison_after(_rand(rng, (B, Hkv, L, D)), positions)
    a = oracle.decode(q, kc, vc, positions, 0.25)
    b = oracle.decode_masked_full(q, kc, vc, positions, 0.25)
    assert np.all(np.isfinite(a))
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("S,H,d", [(37, 4, 64), (128, 2, 32)])
def test_library_sdpa_prefill_no_prefix_is_causal(S, H, d):
    """Decode page section 5 / prefill page: a prompt with no prefix is plain
    is_causal attention."""
    rng = np.random.default_rng(S)
    q = _rand(rng, (S, H, d))
    k = _rand(rng, (S, H, d))
    v = _rand(rng, (S, H, d))
    scale = 1.0 / math.sqrt(d)
    got = oracle.prefill(q, k, v, 0, scale)
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1).unsqueeze(0),
        torch.from_numpy(k).transpose(0, 1).unsqueeze(0),
        torch.from_numpy(v).transpose(0, 1).unsqueeze(0),
        is_causal=True, scale=scale).squeeze(0).transpose(0, 1).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_library_sdpa_prefill_with_prefix_gqa():
    """Prefix prefill: new token i sees keys 0..start_pos+i (bottom-right
    aligned causal mask), GQA via enable_gqa."""
    rng = np.random.default_rng(11)
    S, start_pos, Hq, Hkv, d = 20, 13, 8, 2, 16
    T = start_pos + S
    q = _rand(rng, (S, Hq, d))
    k = _rand(rng, (T, Hkv, d))
    v = _rand(rng, (T, Hkv, d))
    mask = torch.arange(T).view(1, T) <= (start_pos + torch.arange(S)).view(S, 1)
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1).unsqueeze(0),
        torch.from_numpy(k).transpose(0, 1).unsqueeze(0),
        torch.from_numpy(v).transpose(0, 1).unsqueeze(0),
        attn_mask=mask, scale=0.3, enable_gqa=True).squeeze(0).transpose(0, 1).numpy()
    np.testing.assert_allclose(oracle.prefill(q, k, v, start_pos, 0.3), ref,
                               rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------ closed forms ---

def test_position_zero_is_v0_exactly():
    rng = np.random.default_rng(0)
    B, Hq, Hkv, D, L = 2, 8, 4, 128, 16
    q = _rand(rng, (B, Hq, D)) * 50
    kc = _poison_after(_rand(rng, (B, Hkv, L, D)), [0, 0])
    vc = _poison_after(_rand(rng, (B, Hkv, L, D)), [0, 0])
    out = oracle.decode(q, kc, vc, [0, 0], 1.0 / math.sqrt(D))
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(out[b, h], vc[b, h // 2, 0])


def test_identical_keys_or_zero_query_give_mean_of_v():
    rng = np.random.default_rng(1)
    B, Hq, Hkv, D, L = 1, 4, 2, 32, 64
    pos = 40
    kc = _rand(rng, (B, Hkv, L, D))
    kc[:, :, : pos + 1, :] = kc[:, :, :1, :]       # every attended key equal
    vc = _rand(rng, (B, Hkv, L, D))
    q = _rand(rng, (B, Hq, D))
    out = oracle.decode(q, kc, vc, [pos], 0.1)
    mean = vc[0, :, : pos + 1, :].mean(axis=1)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], mean[h // 2], rtol=1e-12, atol=1e-13)
    kc2 = _rand(rng, (B, Hkv, L, D))
    out0 = oracle.decode(np.zeros_like(q), kc2, vc, [pos], 0.1)
    for h in range(Hq):
        np.testing.assert_allclose(out0[0, h], mean[h // 2], rtol=1e-12, atol=1e-13)


# -------------------------------------------------------------- invariances ---

def test_key_row_permutation_invariance():
    rng = np.random.default_rng(2)
    B, Hq, Hkv, D, L = 1, 4, 2, 16, 30
    pos = 25
    q = _rand(rng, (B, Hq, D))
    kc = _rand(rng, (B, Hkv, L, D))
    vc = _rand(rng, (B, Hkv, L, D))
    perm = rng.permutation(pos + 1)
    kp, vp = kc.copy(), vc.copy()
    kp[:, :, : pos + 1] = kc[:, :, perm]
    vp[:, :, : pos + 1] = vc[:, :, perm]
    np.testing.assert_allclose(oracle.decode(q, kc, vc, [pos], 0.2),
                               oracle.decode(q, kp, vp, [pos], 0.2), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("g", [2, 4, 8])
def test_gqa_equals_repeat_kv_mha(g):
    rng = np.random.default_rng(g)
    B, Hkv, D, L = 2, 2, 16, 20
    Hq = g * Hkv
    positions = [19, 6]
    q = _rand(rng, (B, Hq, D))
    kc = _rand(rng, (B, Hkv, L, D))
    vc = _rand(rng, (B, Hkv, L, D))
    gqa = oracle.decode(q, kc, vc, positions, 0.25)
    mha = oracle.decode(q, np.repeat(kc, g, axis=1), np.repeat(vc, g, axis=1), positions, 0.25)
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=0)


def test_prefill_one_token_equals_decode_step():
    rng = np.random.default_rng(3)
    start_pos, Hq, Hkv, d = 33, 8, 2, 64
    T = start_pos + 1
    q = _rand(rng, (1, Hq, d))
    k = _rand(rng, (T, Hkv, d))
    v = _rand(rng, (T, Hkv, d))
    pre = oracle.prefill(q, k, v, start_pos, 0.125)
    kc = k.transpose(1, 0, 2)[None]          # [1, Hkv, T, d]
    vc = v.transpose(1, 0, 2)[None]
    dec = oracle.decode(q, kc, vc, [start_pos], 0.125)
    np.testing.assert_allclose(pre, dec, rtol=1e-13, atol=1e-14)


def test_prefix_prefill_equals_tail_of_full_prefill():
    rng = np.random.default_rng(4)
    start_pos, S, H, d = 9, 7, 3, 8
    T = start_pos + S
    q_all = _rand(rng, (T, H, d))
    k = _rand(rng, (T, H, d))
    v = _rand(rng, (T, H, d))
    full = oracle.prefill(q_all, k, v, 0, 0.35)
    tail = oracle.prefill(q_all[start_pos:], k, v, start_pos, 0.35)
    np.testing.assert_allclose(tail, full[start_pos:], rtol=1e-13, atol=1e-14)


def test_kv_append_writes_only_the_target_rows():
    B, Hkv, L, D = 3, 2, 9, 4
    kc = np.full((B, Hkv, L, D), 7.0)
    vc = np.full((B, Hkv, L, D), -7.0)
    kn = np.arange(B * Hkv * D, dtype=np.float64).reshape(B, Hkv, D)
    vn = -kn - 1
    positions = [0, 8, 4]
    k2, v2 = oracle.kv_append(kc, vc, kn, vn, positions)
    want_k, want_v = kc.copy(), vc.copy()
    for b, p in enumerate(positions):
        want_k[b, :, p] = kn[b]
        want_v[b, :, p] = vn[b]
    assert np.array_equal(k2, want_k) and np.array_equal(v2, want_v)
    assert np.all(kc == 7.0)  # inputs not modified


def test_kv_append_hand_written_case():
    """A 2-sequence, 2-head, 3-row, D=2 cache written out by hand: sequence 0
    takes its new rows at position 2, sequence 1 at position 0; every other
    entry keeps its value."""
    kc = np.array([[[[1, 2], [3, 4], [5, 6]], [[7, 8], [9, 10], [11, 12]]],
                   [[[13, 14], [15, 16], [17, 18]], [[19, 20], [21, 22], [23, 24]]]],
                  dtype=np.float64)
    vc = -kc
    kn = np.array([[[101, 102], [103, 104]], [[105, 106], [107, 108]]], dtype=np.float64)
    vn = -kn
    k2, v2 = oracle.kv_append(kc, vc, kn, vn, [2, 0])
    want_k = np.array([[[[1, 2], [3, 4], [101, 102]], [[7, 8], [9, 10], [103, 104]]],
                       [[[105, 106], [15, 16], [17, 18]], [[107, 108], [21, 22], [23, 24]]]],
                      dtype=np.float64)
    assert np.array_equal(k2, want_k)
    assert np.array_equal(v2, -want_k)


def test_kv_append_matches_library_indexed_assignment():
    """The same write as PyTorch's index_put_ with (sequence, head, position)
    index tensors on the CPU, on bf16 bit patterns."""
    g = torch.Generator().manual_seed(5)
    B, Hkv, L, D = 4, 3, 11, 8
    kc = torch.randn(B, Hkv, L, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, Hkv, L, D, generator=g).to(torch.bfloat16)
    kn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    positions = torch.tensor([10, 0, 5, 5])
    bi = torch.arange(B).repeat_interleave(Hkv)
    hi = torch.arange(Hkv).repeat(B)
    pi = positions.repeat_interleave(Hkv)
    want_k = kc.clone().index_put_((bi, hi, pi), kn.reshape(B * Hkv, D))
    want_v = vc.clone().index_put_((bi, hi, pi), vn.reshape(B * Hkv, D))
    k2, v2 = oracle.kv_append(kc.view(torch.int16).numpy(), vc.view(torch.int16).numpy(),
                              kn.view(torch.int16).numpy(), vn.view(torch.int16).numpy(),
                              positions.tolist())
    assert np.array_equal(k2, want_k.view(torch.int16).numpy())
    assert np.array_equal(v2, want_v.view(torch.int16).numpy())


def test_work_counts():
    """Algorithmic bytes/flops used by the roofline: hand-counted small cases."""
    # one sequence at position 3: 4 rows of K and V, 2 KV heads, D=2, bf16
    assert oracle.decode_bytes([3], Hq=4, Hkv=2, D=2) == 2 * 2 * 4 * 2 * 2 + 2 * 4 * 2 * 2
    assert oracle.decode_flops([3], Hq=4, D=2) == 4 * 2 * 4 * 4
    # S=2, start_pos=1: token 0 sees 2 keys, token 1 sees 3 keys
    assert oracle.prefill_flops(2, 1, H=1, d=2) == 4 * 2 * 5


# ------------------------------------------------------- planted mistakes ---

def _pins_pass():
    """Re-run a compact set of the independent pins; False if any fails."""
    try:
        test_golden_closed_forms()
        test_brute_force_decode_every_position(2, 4, 2, 8)
        test_brute_force_prefill(3, 2, 4, 2, 4)
        test_library_sdpa_decode(3, 8, 2, 64, 64)
        test_library_sdpa_prefill_with_prefix_gqa()
        test_position_zero_is_v0_exactly()
    except (AssertionError, IndexError, ValueError):
        return False
    return True


def test_pins_pass_on_the_real_oracle():
    assert _pins_pass()


@pytest.mark.parametrize("mutant", ["head_mod", "exclusive_range", "top_left_causal",
                                    "dropped_scale", "keys_as_values", "no_normalise"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "head_mod":          # h % Hkv instead of h // g
        monkeypatch.setattr(oatt, "_kv_head", lambda h, g, Hkv: h % Hkv)
    elif mutant == "exclusive_range":  # 0..pos-1 instead of 0..pos
        monkeypatch.setattr(oatt, "_attended_rows", lambda p: range(0, max(p, 1)))
    elif mutant == "top_left_causal":  # mask aligned to the top-left corner
        monkeypatch.setattr(oatt, "_causal_keys", lambda s, i: range(0, i + 1))
    elif mutant == "dropped_scale":
        orig = oatt._attend
        monkeypatch.setattr(oatt, "_attend", lambda q, K, V, scale: orig(q, K, V, 1.0))
    elif mutant == "keys_as_values":
        orig = oatt._attend
        monkeypatch.setattr(oatt, "_attend", lambda q, K, V, scale: orig(q, K, K, scale))
    elif mutant == "no_normalise":
        monkeypatch.setattr(oatt, "_softmax", lambda s: np.exp(s - np.max(s)))
    assert not _pins_pass(), f"mutant {mutant} slipped past every pin"


# ------------------------------------------------------ rotary embedding ---

def test_rope_hand_example():
    """D=4: rotate_half([1,2,3,4]) = [-3,-4,1,2]; x' = x*cos + rot*sin."""
    x = np.array([1.0, 2.0, 3.0, 4.0])
    cos = np.array([0.5, 0.25, 0.5, 0.25], dtype=np.float32)
    sin = np.array([0.75, -1.0, 0.75, -1.0], dtype=np.float32)
    want = [1 * 0.5 - 3 * 0.75, 2 * 0.25 - 4 * -1.0, 3 * 0.5 + 1 * 0.75, 4 * 0.25 + 2 * -1.0]
    np.testing.assert_array_equal(oracle.rope_f32(x, cos, sin), np.array(want, dtype=np.float32))


def _angles(pos, D, base=10000.0):
    inv = base ** (-np.arange(0, D, 2) / D)
    ang = np.outer(np.atleast_1d(pos), inv)
    ang = np.concatenate([ang, ang], axis=-1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(21)
    D = 128
    x = _rand(rng, (3, D))
    c0, s0 = np.ones((3, D), np.float32), np.zeros((3, D), np.float32)
    np.testing.assert_array_equal(oracle.rope_f32(x, c0, s0), x.astype(np.float32))
    c, s = _angles([5, 900, 7000], D)
    xr = oracle.rope_f32(x, c, s).astype(np.float64)
    np.testing.assert_allclose(np.linalg.norm(xr, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-5)
    # q at position m and k at position n: q'.k' depends only on m - n
    q, k = _rand(rng, (D,)), _rand(rng, (D,))
    dots = []
    for m, n in [(10, 3), (107, 100), (5007, 5000)]:
        cq, sq = _angles(m, D)
        ck, sk = _angles(n, D)
        dots.append(float(oracle.rope_f32(q, cq[0], sq[0]).astype(np.float64)
                          @ oracle.rope_f32(k, ck[0], sk[0]).astype(np.float64)))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-4, atol=1e-4)


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(10000) * 10).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0]  # ties go to even
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), want)


def test_rope_step_without_rotation_is_plain_decode():
    rng = np.random.default_rng(8)
    B, Hq, Hkv, D, L = 2, 8, 2, 16, 12
    q, kn, vn = _rand(rng, (B, Hq, D)), _rand(rng, (B, Hkv, D)), _rand(rng, (B, Hkv, D))
    kc, vc = _rand(rng, (B, Hkv, L, D)), _rand(rng, (B, Hkv, L, D))
    pos = [11, 4]
    ones, zeros = np.ones((B, D), np.float32), np.zeros((B, D), np.float32)
    out, kc2, vc2 = oracle.decode_rope_step(q, kn, vn, ones, zeros, kc, vc, pos, 0.25)
    k3, v3 = oracle.kv_append(kc, vc, kn, vn, pos)
    np.testing.assert_array_equal(kc2, k3)
    np.testing.assert_allclose(out, oracle.decode(q, k3, v3, pos, 0.25), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ local window ---

def test_window_of_one_is_v_at_position():
    rng = np.random.default_rng(31)
    B, Hq, Hkv, D, L = 2, 4, 2, 16, 40
    q = _rand(rng, (B, Hq, D))
    kc, vc = _rand(rng, (B, Hkv, L, D)), _rand(rng, (B, Hkv, L, D))
    pos = [0, 33]
    out = oracle.decode_window(q, kc, vc, pos, 0.3, 1)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_array_equal(out[b, h], vc[b, h // 2, pos[b]])


def test_wide_window_is_full_decode_and_window_is_shifted_slice():
    rng = np.random.default_rng(32)
    B, Hq, Hkv, D, L = 3, 8, 2, 16, 300
    q = _rand(rng, (B, Hq, D))
    kc, vc = _rand(rng, (B, Hkv, L, D)), _rand(rng, (B, Hkv, L, D))
    pos = [5, 130, 299]
    full = oracle.decode(q, kc, vc, pos, 0.25)
    for W in (300, 301, 10 ** 6):
        np.testing.assert_allclose(oracle.decode_window(q, kc, vc, pos, 0.25, W), full,
                                   rtol=1e-13, atol=1e-14)
    for W in (1, 2, 6, 64, 131):
        got = oracle.decode_window(q, kc, vc, pos, 0.25, W)
        for b, p in enumerate(pos):
            lo = max(0, p - W + 1)
            want = oracle.decode(q[b:b + 1], kc[b:b + 1, :, lo:p + 1], vc[b:b + 1, :, lo:p + 1],
                                 [p - lo], 0.25)
            np.testing.assert_allclose(got[b:b + 1], want, rtol=1e-13, atol=1e-14)


def test_window_matches_brute_force():
    rng = np.random.default_rng(33)
    B, Hq, Hkv, D, L = 2, 4, 2, 8, 20
    q = _rand(rng, (B, Hq, D))
    kc, vc = _rand(rng, (B, Hkv, L, D)), _rand(rng, (B, Hkv, L, D))
    for pos in ([19, 3], [0, 12]):
        for W in (1, 3, 7, 25):
            want = np.array(brute.decode_window(q.tolist(), kc.tolist(), vc.tolist(), pos, 0.5, W))
            np.testing.assert_allclose(oracle.decode_window(q, kc, vc, pos, 0.5, W), want,
                                       rtol=1e-12, atol=1e-12)


def test_window_pin_catches_an_off_by_one():
    """A window one row too wide (a plausible mistake) fails the shifted-slice
    pin: the pins are not vacuous."""
    rng = np.random.default_rng(34)
    q = _rand(rng, (1, 2, 8))
    kc, vc = _rand(rng, (1, 1, 30, 8)), _rand(rng, (1, 1, 30, 8))
    good = oracle.decode_window(q, kc, vc, [20], 0.5, 5)
    saved = oatt._window_rows
    try:
        oatt._window_rows = lambda position, window: range(max(0, position - window), position + 1)
        bad = oracle.decode_window(q, kc, vc, [20], 0.5, 5)
    finally:
        oatt._window_rows = saved
    assert np.abs(good - bad).max() > 1e-3


# ------------------------------------------------------- multi-token decode ---

def test_multi_token_one_token_is_decode():
    rng = np.random.default_rng(41)
    B, Hq, Hkv, D, L = 2, 8, 2, 16, 50
    q = _rand(rng, (B, 1, Hq, D))
    kc, vc = _rand(rng, (B, Hkv, L, D)), _rand(rng, (B, Hkv, L, D))
    pos = [0, 37]
    np.testing.assert_allclose(oracle.decode_multi(q, kc, vc, pos, 0.3)[:, 0],
                               oracle.decode(q[:, 0], kc, vc, pos, 0.3), rtol=1e-13, atol=1e-14)


def test_multi_token_equals_prefill_over_the_cache():
    """Sequence b's S tokens at positions p..p+S-1 are a causal prefill of S
    tokens with start_pos = p over the cache rows 0..p+S-1 (token-major)."""
    rng = np.random.default_rng(42)
    B, S, Hq, Hkv, D, L = 3, 4, 8, 2, 16, 60
    q = _rand(rng, (B, S, Hq, D))
    kc, vc = _rand(rng, (B, Hkv, L, D)), _rand(rng, (B, Hkv, L, D))
    pos = [0, 9, 56]
    got = oracle.decode_multi(q, kc, vc, pos, 0.25)
    for b, p in enumerate(pos):
        k_tok = kc[b, :, : p + S].transpose(1, 0, 2)  # [T, Hkv, D]
        v_tok = vc[b, :, : p + S].transpose(1, 0, 2)
        want = oracle.prefill(q[b], k_tok, v_tok, p, 0.25)
        np.testing.assert_allclose(got[b], want, rtol=1e-13, atol=1e-14)


def test_multi_token_matches_brute_force():
    rng = np.random.default_rng(43)
    B, S, Hq, Hkv, D, L = 2, 3, 4, 2, 8, 12
    q = _rand(rng, (B, S, Hq, D))
    kc, vc = _rand(rng, (B, Hkv, L, D)), _rand(rng, (B, Hkv, L, D))
    pos = [0, 8]
    got = oracle.decode_multi(q, kc, vc, pos, 0.5)
    for t in range(S):
        want = np.array(brute.decode(q[:, t].tolist(), kc.tolist(), vc.tolist(),
                                     [p + t for p in pos], 0.5))
        np.testing.assert_allclose(got[:, t], want, rtol=1e-12, atol=1e-12)
