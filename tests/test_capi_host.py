"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function include/gqa_attn.h declares, and
reject bad arguments on the host before any CUDA call.  Only calls that
return before touching the GPU are made here.
"""

import ctypes
import os
import re

import pytest

import gqa_decode_attention_place_gb300 as ga

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(attn_[a-z0-9_]+)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return ga.load_library()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ["attn_kv_append", "attn_decode_workspace_size", "attn_decode_step",
                 "attn_prefill_causal", "attn_read_device_status", "attn_status_string",
                 "attn_last_cuda_error", "attn_decode_step_append",
                 "attn_decode_step_rope_append", "attn_decode_step_noalloc",
                 "attn_decode_stream_step", "attn_decode_step_window", "attn_decode_multi",
                 "attn_test_skip_tile", "attn_read_prefill_status", "attn_debug_build",
                 "attn_read_prefill_skips", "attn_test_force_schedule"]:
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_release_and_range_checked_builds():
    """The default library has no range checks; the -DGQA_DEBUG build exports
    the same functions and reports that it has them."""
    from gqa_decode_attention_place_gb300 import _build
    rel = ctypes.CDLL(_build.build())
    dbg = ctypes.CDLL(_build.build(debug=True))
    assert rel.attn_debug_build() == 0
    assert dbg.attn_debug_build() == 1
    for name in _declared_functions():
        assert hasattr(dbg, name), f"{name} missing from the range-checked build"


def test_status_strings(lib):
    assert ga.attn_status_string(0) == "ok"
    for c in range(1, 6):
        assert ga.attn_status_string(c) not in ("ok", "unknown status")
    assert ga.attn_status_string(99) == "unknown status"


def test_workspace_size_rules(lib):
    n1 = ga.attn_decode_workspace_size(1, 16, 8, 8192, 128)
    n2 = ga.attn_decode_workspace_size(64, 32, 8, 8192, 128)
    n3 = ga.attn_decode_workspace_size(256, 64, 8, 8192, 128)
    assert 0 < n1 < n2 < n3
    assert n3 < 64 << 20  # bounded by grid + B*Hkv partials, not by B*Hq*L
    assert n1 % 256 == 0
    # independent of max_len: the split is chosen on the device from positions
    assert ga.attn_decode_workspace_size(1, 16, 8, 1 << 20, 128) == n1
    assert ga.attn_decode_workspace_size(1, 16, 8, 8192, 64) == 0      # D unsupported
    assert ga.attn_decode_workspace_size(1, 12, 8, 8192, 128) == 0     # Hq % Hkv
    assert ga.attn_decode_workspace_size(1, 48, 3, 8192, 128) > 0      # g = 16
    assert ga.attn_decode_workspace_size(1, 96, 3, 8192, 128) == 0     # g = 32
    assert ga.attn_decode_workspace_size(0, 16, 8, 8192, 128) == 0


def test_host_validation_happens_before_any_launch(lib):
    P = 0x1000  # fake but 16-byte aligned "device" pointer: never dereferenced
    # null pointers
    assert lib.attn_kv_append(None, P, P, P, P, 1, 8, 16, 128, None) == 1
    assert lib.attn_decode_step(P, P, P, P, 1, 16, 8, 16, 128, 1.0, None, P, 1 << 20, None) == 1
    # misaligned tensor pointer
    assert lib.attn_kv_append(P + 2, P, P, P, P, 1, 8, 16, 128, None) == 1
    # non-positive sizes, Hq % Hkv
    assert lib.attn_decode_step(P, P, P, P, 1, 12, 8, 16, 128, 1.0, P, P, 1 << 20, None) == 1
    assert lib.attn_kv_append(P, P, P, P, P, 0, 8, 16, 128, None) == 1
    # unsupported D / g
    assert lib.attn_decode_step(P, P, P, P, 1, 16, 8, 16, 96, 1.0, P, P, 1 << 20, None) == 2
    assert lib.attn_decode_step(P, P, P, P, 1, 64, 2, 16, 128, 1.0, P, P, 1 << 20, None) == 2
    assert lib.attn_kv_append(P, P, P, P, P, 1, 8, 16, 12, None) == 2
    # workspace too small / missing
    need = ga.attn_decode_workspace_size(1, 16, 8, 16, 128)
    assert lib.attn_decode_step(P, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P, need - 1, None) == 3
    assert lib.attn_decode_step(P, P, P, P, 1, 16, 8, 16, 128, 1.0, P, None, need, None) == 3
    # prefill: bad sizes, unsupported head dim, empty problem is a no-op
    assert lib.attn_prefill_causal(P, P, P, -1, 0, 32, 32, 64, 0.125, P, None) == 1
    assert lib.attn_prefill_causal(P, P, P, 4, -1, 32, 32, 64, 0.125, P, None) == 1
    assert lib.attn_prefill_causal(P, P, P, 4, 0, 32, 7, 64, 0.125, P, None) == 1
    assert lib.attn_prefill_causal(P, P, P, 4, 0, 32, 32, 80, 0.125, P, None) == 2
    assert lib.attn_read_device_status(None, None, None) == 1
    # rotary step: null or misaligned cos/sin, then the append step's own checks
    rope = lib.attn_decode_step_rope_append
    assert rope(P, P, P, None, P, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P, 1 << 20, None) == 1
    assert rope(P, P, P, P, P + 4, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P, 1 << 20, None) == 1
    assert rope(P, None, P, P, P, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P, 1 << 20, None) == 1
    # g = 16 decodes, but not with the rotation (two operand rows per head)
    assert rope(P, P, P, P, P, P, P, P, 1, 32, 2, 16, 128, 1.0, P, P, 1 << 20, None) == 2
    assert rope(P, P, P, P, P, P, P, P, 1, 64, 2, 16, 128, 1.0, P, P, 1 << 20, None) == 2
    assert rope(P, P, P, P, P, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P, need - 1, None) == 3
    # streaming step: tables both or neither, aligned; then the append step's checks
    stream = lib.attn_decode_stream_step
    assert stream(P, P, P, P, None, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P, 1 << 20, None) == 1
    assert stream(P, P, P, P + 8, P, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P, 1 << 20, None) == 1
    assert stream(P, P, P, None, None, None, P, P, 1, 16, 8, 16, 128, 1.0, P, P, 1 << 20,
                  None) == 1
    assert stream(P, P, P, None, None, P, P, P, 1, 16, 8, 16, 96, 1.0, P, P, 1 << 20, None) == 2
    assert stream(P, P, P, P, P, P, P, P, 1, 32, 2, 16, 128, 1.0, P, P, 1 << 20, None) == 2
    assert stream(P, P, P, None, None, P, P, P, 1, 16, 8, 16, 128, 1.0, P, None, need,
                  None) == 3
    assert stream(P, None, None, None, None, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P, need,
                  None) == 1
    # local window: window > 0, new rows both or neither
    win = lib.attn_decode_step_window
    assert win(P, None, None, P, P, P, 1, 16, 8, 16, 128, 0, 1.0, P, P, need, None) == 1
    assert win(P, P, None, P, P, P, 1, 16, 8, 16, 128, 4, 1.0, P, P, need, None) == 1
    assert win(P, None, None, P, P, P, 1, 64, 2, 16, 128, 4, 1.0, P, P, need, None) == 2
    assert win(P, None, None, P, P, P, 1, 16, 8, 16, 128, 4, 1.0, P, P, need - 1, None) == 3
    # multi-token decode: S * g must be 1, 2, 4, 8 or 16; workspace for S * Hq heads
    multi = lib.attn_decode_multi
    need2 = ga.attn_decode_workspace_size(1, 32, 8, 16, 128)
    assert need2 > need
    assert multi(P, None, None, P, P, P, 1, 3, 16, 8, 16, 128, 1.0, P, P, 1 << 24, None) == 2
    assert multi(P, None, None, P, P, P, 1, 4, 64, 8, 16, 128, 1.0, P, P, 1 << 24, None) == 2
    assert multi(P, None, None, P, P, P, 1, 0, 16, 8, 16, 128, 1.0, P, P, 1 << 24, None) == 1
    assert multi(P, P, None, P, P, P, 1, 2, 16, 8, 16, 128, 1.0, P, P, 1 << 24, None) == 1
    assert multi(P, None, None, P, P, P, 1, 2, 16, 8, 16, 128, 1.0, P, P, need2 - 1, None) == 3
    assert lib.attn_test_skip_tile(-2) == 1
    assert lib.attn_test_skip_tile(-1) == 0
    assert lib.attn_test_force_schedule(-2) == 1
    assert lib.attn_test_force_schedule(17) == 1
    assert lib.attn_test_force_schedule(-1) == 0
    # the append entry points still refuse missing new rows
    assert lib.attn_decode_step_append(P, None, None, P, P, P, 1, 16, 8, 16, 128, 1.0, P, P,
                                       need, None) == 1


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ga.attn_kv_append(x, x, torch.zeros(1, dtype=torch.int32),
                          torch.zeros(1, 8, 4, 128, dtype=torch.bfloat16),
                          torch.zeros(1, 8, 4, 128, dtype=torch.bfloat16))
