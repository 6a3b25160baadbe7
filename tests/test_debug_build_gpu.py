"""The range-checked build (-DGQA_DEBUG) on the boundary and ragged cases.

Compute-sanitizer is not available here, so the library has a second build in
which every decode kernel checks its index-derived addresses (bulk-copy tile
coordinates, cluster landing slots, partial-result slots, output and new-row
addresses) and both prefill kernels check their tile coordinates and output
rows before use; a failed check skips the access and is recorded
(ATTN_DEV_RANGE in the decode status word, a count for prefill).  This test
builds that library and runs the decode, append, rotary, window, multi-token,
streaming, prefill and split-schedule parity tests against it in a child
process
(GQA_ATTN_DEBUG=1): each must match the oracle as before, and the autouse
fixture in conftest.py fails any test after which a check had failed.
"""

import os
import re
import subprocess
import sys

import pytest

from gqa_decode_attention_place_gb300 import _build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
FILES = ["test_decode_gpu.py", "test_append_gpu.py", "test_rope_gpu.py", "test_window_gpu.py",
         "test_multi_gpu.py", "test_stream_step_gpu.py", "test_prefill_gpu.py",
         "test_schedule_gpu.py"]
# the 2^20-row caches are left out for memory and time; nothing else
DESELECT = "not million"


def test_range_checked_build_parity():
    _build.build(debug=True)
    env = dict(os.environ, GQA_ATTN_DEBUG="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "-k", DESELECT] + [os.path.join(HERE, f) for f in FILES]
    r = subprocess.run(cmd, cwd=os.path.dirname(HERE), env=env, capture_output=True, text=True,
                       timeout=1200)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, f"range-checked build:\n{tail}"
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 100 and " failed" not in r.stdout, tail
    print(f"range-checked build: {m.group(0)}")
