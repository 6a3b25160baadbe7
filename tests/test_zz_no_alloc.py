"""attn_decode_step_noalloc: decode without any device allocation.

Some callers cannot call cudaMalloc -- code that runs while a CUDA graph is
being captured, real-time streaming loops that must not stall on the
device-wide synchronisation an allocation implies, and plugin or embedded
hosts that own all device memory.  For them the library offers a decode entry
point whose split-KV scratch is a fixed device array inside the library.

This test calls that entry point through the C ABI (ctypes, raw pointers) and
checks its output against the workspace-taking attn_decode_step on the same
inputs, within the attention tolerance used by every other test, on two calls
in a row (the second with other sizes, so the shared scratch's leftovers from
the first call must not leak into it).  The file name makes pytest collect it
last.
"""

import numpy as np
import pytest
import torch

import gqa_decode_attention_place_gb300 as ga
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


def test_noalloc_matches_workspace_entry_point_two_calls():
    lib = ga.load_library()
    shapes = [
        dict(B=64, Hq=32, Hkv=8, L=8192, positions="uniform"),   # split segments, combine
        dict(B=3, Hq=16, Hkv=8, L=600, positions=[599, 0, 130]),  # other layout of scratch
    ]
    for i, sh in enumerate(shapes):
        case = synth.decode_case(D=128, fill="all", poison=True, seed=40 + i, device="cuda", **sh)
        ga.attn_kv_append(case.k_new, case.v_new, case.positions, case.k_cache, case.v_cache)
        ref = ga.attn_decode_step(case.q, case.positions, case.k_cache, case.v_cache, case.scale)
        out = torch.full_like(case.q, float("nan"))
        code = _noalloc(lib, case, out)
        assert code == 0, ga.attn_status_string(code)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert_attn_close(f64(out).reshape(-1, 128), f64(ref).reshape(-1, 128),
                          f"no-alloc call {i}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = ga.load_library()
    P = 0x1000  # aligned fake pointers: the size check returns before any launch
    # B=8192, Hkv=8, g=8 needs far more than the built-in 16 MiB
    assert lib.attn_decode_step_noalloc(P, P, P, P, 8192, 64, 8, 64, 128, 1.0, P, None) == 3
