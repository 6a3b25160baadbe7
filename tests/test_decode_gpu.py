"""Decode step (attn_kv_append then attn_decode_step) against the fp64 oracle.

Covers the five decode workloads' shapes (the single step at position 100,
the 8192-step streaming loop, the ragged B=64 batch, the B=256 g=8 stress
batch with peaky keys), tile/split boundaries, position 0, out-of-range
positions, NaN-poisoned rows past each position (any over-read would show up
as NaN), every supported group size, workspace reuse, and the largest batch.
"""

import math

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, bits, f64

pytestmark = pytest.mark.gpu


def _oracle_rows(case, bs, heads=None):
    """Oracle output for sequences `bs` (all heads, or `heads`), computed from
    the pre-append cache and the new rows (call before the kernels run)."""
    Hq = case.q.shape[1]
    Hkv = case.k_cache.shape[1]
    out = {}
    for b in bs:
        p = int(case.positions[b])
        kc = f64(case.k_cache[b:b + 1, :, : p + 1])
        vc = f64(case.v_cache[b:b + 1, :, : p + 1])
        kc, vc = oracle.kv_append(kc, vc, f64(case.k_new[b:b + 1]), f64(case.v_new[b:b + 1]), [p])
        hs = list(range(Hq)) if heads is None else heads
        rows = oracle.decode_rows(f64(case.q[b:b + 1]), kc, vc, [p], case.scale,
                                  [(0, h) for h in hs])
        for h, r in zip(hs, rows):
            out[(b, h)] = r
    assert Hkv >= 1
    return out


def _run_step(case, workspace=None):
    ga.attn_kv_append(case.k_new, case.v_new, case.positions, case.k_cache, case.v_cache)
    out = ga.attn_decode_step(case.q, case.positions, case.k_cache, case.v_cache, case.scale,
                              workspace=workspace)
    torch.cuda.synchronize()
    return out


def _check(case, want, out, what):
    keys = sorted(want)
    got = np.stack([f64(out[b, h]) for b, h in keys])
    ref = np.stack([want[k] for k in keys])
    return assert_attn_close(got, ref, what)


def test_single_step_workload():
    """B=1, Hq=16, Hkv=8, rows 0..99 filled, new row at position 100."""
    case = synth.generators.workload_case("single_step", seed=1, device="cuda")
    want = _oracle_rows(case, [0])
    out = _run_step(case)
    _check(case, want, out, "single_step")


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_tile_and_split_boundaries_poisoned(g):
    Hkv = 2
    positions = [0, 1, 62, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 4095, 4096, 8191]
    case = synth.decode_case(B=len(positions), Hq=g * Hkv, Hkv=Hkv, D=128, L=8192,
                             positions=positions, fill="all", poison=True, seed=g,
                             device="cuda")
    want = _oracle_rows(case, range(len(positions)))
    out = _run_step(case)
    _check(case, want, out, f"boundaries g={g}")


def test_position_zero_is_v0_bit_exact():
    case = synth.decode_case(B=3, Hq=16, Hkv=8, D=128, L=64, positions=[0, 0, 0],
                             fill="all", poison=True, seed=5, device="cuda")
    out = _run_step(case)
    for h in range(16):
        assert torch.equal(bits(out[:, h]), bits(case.v_new[:, h // 2]))


def test_ragged_workload_sampled():
    """B=64, Hq=32, Hkv=8, positions uniform in [0, 8191], every row N(0,1)."""
    case = synth.generators.workload_case("ragged", seed=2, device="cuda")
    pos = case.positions.cpu().numpy()
    order = np.argsort(pos)
    bs = sorted(set([int(order[0]), int(order[1]), int(order[-1]), int(order[-2])] +
                    [int(x) for x in np.random.default_rng(0).choice(64, 8, replace=False)]))
    want = _oracle_rows(case, bs)
    out = _run_step(case)
    assert torch.isfinite(out.float()).all()
    _check(case, want, out, "ragged")


def test_ragged_small_full_oracle_poisoned():
    case = synth.decode_case(B=16, Hq=32, Hkv=8, D=128, L=700, positions="uniform",
                             fill="all", poison=True, seed=9, device="cuda")
    want = _oracle_rows(case, range(16))
    out = _run_step(case)
    _check(case, want, out, "ragged small")


def test_stress_workload_sampled():
    """B=256, Hq=64, Hkv=8 (g=8), all at position 8191, 1% of key rows x8."""
    case = synth.generators.workload_case("stress", seed=3, device="cuda")
    bs = [0, 97, 255]
    want = _oracle_rows(case, bs)
    out = _run_step(case)
    assert torch.isfinite(out.float()).all()
    _check(case, want, out, "stress")
    del case
    torch.cuda.empty_cache()


def test_peaky_keys_small_full_oracle():
    case = synth.decode_case(B=4, Hq=64, Hkv=8, D=128, L=1500, positions=[1499, 700, 64, 3],
                             fill="all", peaky=0.01, poison=True, seed=4, device="cuda")
    want = _oracle_rows(case, range(4))
    out = _run_step(case)
    _check(case, want, out, "peaky")


def test_streaming_workload_sampled_steps():
    """8192 consecutive append+decode steps from position 0 (B=1, Hq=16, Hkv=8)."""
    steps, Hq, Hkv, D, L = 8192, 16, 8, 128, 8192
    q, k, v, pos = synth.streaming_inputs(steps=steps, Hq=Hq, Hkv=Hkv, D=D, seed=11,
                                          device="cuda")
    kc = torch.zeros((1, Hkv, L, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ws = ga.decode_workspace(1, Hq, Hkv, L, D)
    outs = torch.empty((steps, 1, Hq, D), dtype=torch.bfloat16, device="cuda")
    scale = 1.0 / math.sqrt(D)
    for s in range(steps):
        ga.attn_kv_append(k[s], v[s], pos[s], kc, vc)
        ga.attn_decode_step(q[s], pos[s], kc, vc, scale, out=outs[s], workspace=ws)
    torch.cuda.synchronize()
    assert ga.attn_read_device_status(ws) == 0
    kk = f64(k[:, 0])   # [steps, Hkv, D]: row s of the cache is step s's k
    vv = f64(v[:, 0])
    for s in [0, 1, 63, 64, 65, 100, 1000, 4000, 8000, 8191]:
        # cache state after the appends of steps 0..s: row j holds step j's k/v
        kc_o = kk[: s + 1].transpose(1, 0, 2)[None]
        vc_o = vv[: s + 1].transpose(1, 0, 2)[None]
        want = oracle.decode(f64(q[s]), kc_o, vc_o, [s], scale)
        assert_attn_close(f64(outs[s]), want, f"streaming step {s}")


def test_out_of_range_positions_flag_and_nan():
    case = synth.decode_case(B=4, Hq=16, Hkv=8, D=128, L=256, positions=[10, 256, -3, 255],
                             fill="all", seed=6, device="cuda")
    ws = ga.decode_workspace(4, 16, 8, 256, 128)
    want = _oracle_rows(case, [0, 3])
    out = _run_step(case, workspace=ws)
    assert torch.isnan(out[1].float()).all() and torch.isnan(out[2].float()).all()
    _check(case, want, out, "valid rows next to invalid ones")
    assert ga.attn_read_device_status(ws) & ga.ATTN_DEV_BAD_POSITION
    assert ga.attn_read_device_status(ws) == 0  # cleared by the read


def test_workspace_reuse_across_calls():
    """Counters are left at zero, so one workspace serves call after call of
    the same sizes (re-zeroed when the sizes change)."""
    ws = ga.decode_workspace(32, 32, 8, 4096, 128)
    for seed, (B, positions) in enumerate([(32, "uniform"), (32, [4095] * 32),
                                           (32, "uniform"), (5, [4095, 0, 64, 2000, 3]),
                                           (5, [3, 4095, 64, 2000, 1])]):
        if seed == 3:
            ws.zero_()
        case = synth.decode_case(B=B, Hq=32, Hkv=8, D=128, L=4096, positions=positions,
                                 fill="all", poison=True, seed=100 + seed, device="cuda")
        want = _oracle_rows(case, range(min(B, 6)))
        out = _run_step(case, workspace=ws)
        _check(case, want, out, f"reuse call {seed}")
    assert ga.attn_read_device_status(ws) == 0


def test_max_batch_tiny_positions():
    """B=8192 (the largest batch): exercises the multi-chunk position scan."""
    B, L = 8192, 4
    case = synth.decode_case(B=B, Hq=8, Hkv=4, D=128, L=L, positions="uniform", fill="all",
                             poison=True, seed=12, device="cuda")
    bs = [0, 1, 255, 256, 4097, 8191]
    want = _oracle_rows(case, bs)
    out = _run_step(case)
    assert torch.isfinite(out.float()).all()
    _check(case, want, out, "B=8192")


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("Hq", [16, 32])
def test_max_batch_eight_and_sixteen_heads(fused, Hq):
    """B=8192 with 8 heads per KV head (per-warp MMA kernels) and 16 (the
    tcgen05 kernels; there, above B=4287 the stream-K prefix array leaves
    room for two K/V stages only, so this runs the 2-stage ring).  Plain
    step, and the fused append step."""
    B, L = 8192, 300
    case = synth.decode_case(B=B, Hq=Hq, Hkv=2, D=128, L=L, positions="uniform", fill="all",
                             poison=True, seed=13 + int(fused) + Hq, device="cuda")
    bs = [0, 1, 127, 2048, 4287, 4288, 8191]
    want = _oracle_rows(case, bs)
    if fused:
        out = ga.attn_decode_step_append(case.q, case.k_new, case.v_new, case.positions,
                                         case.k_cache, case.v_cache, case.scale)
        torch.cuda.synchronize()
    else:
        out = _run_step(case)
    assert torch.isfinite(out.float()).all()
    _check(case, want, out, f"B=8192 g={Hq // 2} fused={fused}")


def test_single_row_cache_and_odd_scale():
    case = synth.decode_case(B=2, Hq=4, Hkv=1, D=128, L=1, positions=[0, 0], fill="all",
                             seed=13, device="cuda", scale=3.7)
    want = _oracle_rows(case, [0, 1])
    out = _run_step(case)
    _check(case, want, out, "L=1")
    case = synth.decode_case(B=2, Hq=8, Hkv=2, D=128, L=300, positions=[299, 150],
                             fill="all", seed=14, device="cuda", scale=0.01)
    want = _oracle_rows(case, [0, 1])
    _check(case, want, _run_step(case), "scale 0.01")


# ---- fused append + decode (attn_decode_step_append) ------------------------

def _fused_step(case, workspace=None):
    out = ga.attn_decode_step_append(case.q, case.k_new, case.v_new, case.positions,
                                     case.k_cache, case.v_cache, case.scale, workspace=workspace)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_fused_append_decode_boundaries_poisoned(g):
    Hkv = 2
    positions = [0, 1, 62, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 4095, 4096, 8191]
    case = synth.decode_case(B=len(positions), Hq=g * Hkv, Hkv=Hkv, D=128, L=8192,
                             positions=positions, fill="all", poison=True, seed=20 + g,
                             device="cuda")
    want = _oracle_rows(case, range(len(positions)))
    pos = case.positions.cpu().numpy()
    wk, wv = oracle.kv_append(bits(case.k_cache).cpu().numpy(), bits(case.v_cache).cpu().numpy(),
                              bits(case.k_new).cpu().numpy(), bits(case.v_new).cpu().numpy(), pos)
    out = _fused_step(case)
    _check(case, want, out, f"fused g={g}")
    assert np.array_equal(bits(case.k_cache).cpu().numpy(), wk)
    assert np.array_equal(bits(case.v_cache).cpu().numpy(), wv)


def test_fused_position_zero_and_bad_positions():
    case = synth.decode_case(B=4, Hq=16, Hkv=8, D=128, L=64, positions=[0, 64, 0, -1],
                             fill="all", poison=True, seed=31, device="cuda")
    k_before = bits(case.k_cache).clone()
    ws = ga.decode_workspace(4, 16, 8, 64, 128)
    out = _fused_step(case, workspace=ws)
    for h in range(16):
        assert torch.equal(bits(out[0, h]), bits(case.v_new[0, h // 2]))
        assert torch.equal(bits(out[2, h]), bits(case.v_new[2, h // 2]))
    assert torch.isnan(out[1].float()).all() and torch.isnan(out[3].float()).all()
    assert torch.equal(bits(case.k_cache[1]), k_before[1])
    assert torch.equal(bits(case.k_cache[3]), k_before[3])
    assert ga.attn_read_device_status(ws) & ga.ATTN_DEV_BAD_POSITION


def test_fused_streaming_loop_matches_two_call_loop():
    """The streaming workload through the fused call; sampled steps against
    the oracle and every step against the append-then-decode pair."""
    steps, Hq, Hkv, D, L = 1500, 16, 8, 128, 2048
    q, k, v, pos = synth.streaming_inputs(steps=steps, Hq=Hq, Hkv=Hkv, D=D, seed=12,
                                          device="cuda")
    scale = 1.0 / math.sqrt(D)
    caches = [torch.full((1, Hkv, L, D), float("nan"), dtype=torch.bfloat16, device="cuda")
              for _ in range(4)]
    ws = [ga.decode_workspace(1, Hq, Hkv, L, D) for _ in range(2)]
    outs = [torch.empty((steps, 1, Hq, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for s in range(steps):
        ga.attn_decode_step_append(q[s], k[s], v[s], pos[s], caches[0], caches[1], scale,
                                   out=outs[0][s], workspace=ws[0])
        ga.attn_kv_append(k[s], v[s], pos[s], caches[2], caches[3])
        ga.attn_decode_step(q[s], pos[s], caches[2], caches[3], scale, out=outs[1][s],
                            workspace=ws[1])
    torch.cuda.synchronize()
    assert torch.equal(bits(caches[0][:, :, :steps]), bits(caches[2][:, :, :steps]))
    assert torch.equal(bits(caches[1][:, :, :steps]), bits(caches[3][:, :, :steps]))
    assert torch.equal(bits(outs[0]), bits(outs[1]))
    kk, vv = f64(k[:, 0]), f64(v[:, 0])
    for s in [0, 63, 64, 777, 1499]:
        kc_o = kk[: s + 1].transpose(1, 0, 2)[None]
        vc_o = vv[: s + 1].transpose(1, 0, 2)[None]
        want = oracle.decode(f64(q[s]), kc_o, vc_o, [s], scale)
        assert_attn_close(f64(outs[0][s]), want, f"fused streaming step {s}")


@pytest.mark.parametrize("g,Hkv,positions", [
    (2, 8, [8191]), (2, 8, [0]), (2, 8, [65]), (8, 1, [5000]), (1, 4, [1023, 64]),
    (4, 2, [63, 3000]), (2, 8, [130, 7000]),
    # tensor-core kernels: position 0 (with the fused append the tile holds
    # only the appended row) and the first tile boundaries
    (4, 8, [0]), (8, 8, [0]), (8, 2, [127, 128]), (4, 4, [1, 8191]),
    # g = 16: clusters of at most 9 (rank 0's 16-head landing slots)
    (16, 2, [5000]), (16, 1, [0, 8191]), (16, 4, [127, 128, 3000]),
])
def test_small_batches_one_cluster_per_segment(g, Hkv, positions):
    """Few (sequence, KV head) segments: each gets a cluster of CTAs that
    merge through distributed shared memory.  Plain and fused calls."""
    B = len(positions)
    for fused in (False, True):
        case = synth.decode_case(B=B, Hq=g * Hkv, Hkv=Hkv, D=128, L=8192, positions=positions,
                                 fill="all", poison=True, seed=50 + g + int(fused), device="cuda")
        want = _oracle_rows(case, range(B))
        out = _fused_step(case) if fused else _run_step(case)
        _check(case, want, out, f"small batch g={g} fused={fused}")


@pytest.mark.parametrize("g", [1, 2, 4])
@pytest.mark.parametrize("L,positions", [(100, [99, 0]), (300, [299, 255]), (1500, [1499, 1407])])
def test_short_caches_in_cluster_mode(g, L, positions):
    """Caches whose length is not a multiple of the 128-row tile, few
    segments (one cluster each): a rank's first tile is copied before the
    position is known when it starts inside the cache, its box may reach past
    L (those rows arrive as zeros), and ranks that the position leaves without
    tiles drop that copy.  Plain and fused calls, rows past each position
    NaN-poisoned, the appended rows checked bit for bit."""
    B, Hkv = len(positions), 2
    for fused in (False, True):
        case = synth.decode_case(B=B, Hq=g * Hkv, Hkv=Hkv, D=128, L=L, positions=positions,
                                 fill="all", poison=True, seed=70 + g + L + int(fused),
                                 device="cuda")
        want = _oracle_rows(case, range(B))
        pos = case.positions.cpu().numpy()
        wk, wv = oracle.kv_append(bits(case.k_cache).cpu().numpy(),
                                  bits(case.v_cache).cpu().numpy(),
                                  bits(case.k_new).cpu().numpy(), bits(case.v_new).cpu().numpy(),
                                  pos)
        out = _fused_step(case) if fused else _run_step(case)
        _check(case, want, out, f"L={L} g={g} fused={fused}")
        assert np.array_equal(bits(case.k_cache).cpu().numpy(), wk)
        assert np.array_equal(bits(case.v_cache).cpu().numpy(), wv)


@pytest.mark.parametrize("B,Hq,positions", [(1, 16, [70000]), (3, 16, [100, 8000, 70000]),
                                            (1, 128, [4000])])
def test_max_len_of_a_million_rows(B, Hq, positions):
    """max_len = 2^20 with short positions: the step reads rows 0..pos only
    (every row past each position is NaN, so a read of any of them would show
    in the output) and matches the oracle, on a cluster launch (B=1), on
    stream-K (B=3) and on the tensor-core kernels (g = 16)."""
    L = 1 << 20
    case = synth.decode_case(B=B, Hq=Hq, Hkv=8, D=128, L=L, positions=positions, fill="all",
                             poison=True, seed=77 + B + Hq, device="cuda")
    want = _oracle_rows(case, range(B))
    out = _run_step(case)
    _check(case, want, out, f"L=2^20 B={B} Hq={Hq}")
    del case
    torch.cuda.empty_cache()
