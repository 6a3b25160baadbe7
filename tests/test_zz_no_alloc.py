"""attn_decode_step_noalloc: decode without any device allocation.

Some callers cannot call cudaMalloc: plugin or embedded hosts that own all
device memory and hand the library none, and real-time streaming loops that
must not stall on the device-wide synchronisation an allocation can imply.
For them the library offers a decode entry point whose split-KV scratch is a
fixed device array inside the library.

This test calls that entry point through the C ABI (ctypes, raw pointers) on
two calls in a row (the second with other sizes, so the shared scratch's
leftovers from the first call must not leak into it) and checks its output,
within the attention tolerance used by every other test, against the
workspace-taking attn_decode_step on the same inputs and against the fp64
oracle on sampled sequences.  The file name makes pytest collect it last.
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
import oracle
import synth
from _helpers import assert_attn_close, f64

pytestmark = pytest.mark.gpu


def _noalloc(lib, case, out):
    B, Hq, D = case.q.shape
    Hkv, L = case.k_cache.shape[1], case.k_cache.shape[2]
    return lib.attn_decode_step_noalloc(
        case.q.data_ptr(), case.positions.data_ptr(), case.k_cache.data_ptr(),
        case.v_cache.data_ptr(), B, Hq, Hkv, L, D, case.scale, out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _oracle_sample(case, bs):
    """Oracle rows (all heads) of sequences bs, from the cache before the
    append and the new rows; call before the kernels run."""
    want = {}
    for b in bs:
        p = int(case.positions[b])
        kc = f64(case.k_cache[b:b + 1, :, : p + 1])
        vc = f64(case.v_cache[b:b + 1, :, : p + 1])
        kc, vc = oracle.kv_append(kc, vc, f64(case.k_new[b:b + 1]), f64(case.v_new[b:b + 1]), [p])
        want[b] = oracle.decode(f64(case.q[b:b + 1]), kc, vc, [p], case.scale)[0]
    return want


def test_noalloc_matches_workspace_entry_point_two_calls():
    lib = ga.load_library()
    shapes = [
        dict(B=64, Hq=32, Hkv=8, L=8192, positions="uniform"),   # split segments, combine
        dict(B=3, Hq=16, Hkv=8, L=600, positions=[599, 0, 130]),  # other layout of scratch
    ]
    for i, sh in enumerate(shapes):
        case = synth.decode_case(D=128, fill="all", poison=True, seed=40 + i, device="cuda", **sh)
        sample = [0, 17, 40, 63] if sh["B"] == 64 else [0, 1, 2]
        want = _oracle_sample(case, sample)
        ga.attn_kv_append(case.k_new, case.v_new, case.positions, case.k_cache, case.v_cache)
        ref = ga.attn_decode_step(case.q, case.positions, case.k_cache, case.v_cache, case.scale)
        out = torch.full_like(case.q, float("nan"))
        code = _noalloc(lib, case, out)
        assert code == 0, ga.attn_status_string(code)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert_attn_close(f64(out).reshape(-1, 128), f64(ref).reshape(-1, 128),
                          f"no-alloc call {i} against attn_decode_step")
        for b in sample:
            assert_attn_close(f64(out[b]), want[b], f"no-alloc call {i} b={b} against the oracle")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = ga.load_library()
    P = 0x1000  # aligned fake pointers: the size check returns before any launch
    # B=8192, Hkv=8, g=8 needs far more than the built-in 16 MiB
    assert lib.attn_decode_step_noalloc(P, P, P, P, 8192, 64, 8, 64, 128, 1.0, P, None) == 3
