import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(autouse=True)
def _range_checked_build_clean(request):
    """Under GQA_ATTN_DEBUG=1 (the range-checked library): a GPU test also
    fails if any of its launches skipped an access that failed a range check."""
    if os.environ.get("GQA_ATTN_DEBUG", "0") in ("", "0") or "gpu" not in request.keywords:
        yield
        return
    import torch
    import gqa_decode_attention_place_gb300 as ga
    assert ga.attn_debug_build(), "GQA_ATTN_DEBUG=1 but the release library was loaded"
    ga.debug_collect_range_bits()
    yield
    torch.cuda.synchronize()
    assert ga.debug_collect_range_bits() == 0, "a range check failed (ATTN_DEV_RANGE)"
