"""The opt-in device check of request offset arrays (pkm_validate_row_offsets and the
PKM_DEBUG_VALIDATE switch).  The pages give buffer_row_offsets / input_row_offsets as prefix
offsets (rows of request b = [offsets[b], offsets[b+1])), so the entry points require them
non-decreasing; the check reports an array that decreases, and writes nothing else."""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_mla_gb300  # noqa: F401


def _check(offsets):
    import paged_kv_mla_gb300 as pkm
    off = torch.tensor(np.asarray(offsets, np.uint32).view(np.int32), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = off.clone()
    pkm.pkm_validate_row_offsets(off, st)
    torch.cuda.synchronize()
    assert torch.equal(off, before)
    return int(st.item())


def test_non_decreasing_offsets_pass():
    assert _check([0, 5, 5, 16]) == 0                        # an empty request is fine
    rng = np.random.default_rng(5)
    assert _check(np.concatenate([[0], np.cumsum(rng.integers(0, 4, 5000))])) == 0
    assert _check([7]) == 0                                   # no requests


def test_a_decrease_anywhere_is_reported():
    import paged_kv_mla_gb300 as pkm
    assert _check([0, 12, 8, 30]) == pkm.PKM_ERR_INVALID_ARG
    big = np.concatenate([[0], np.cumsum(np.full(6000, 3))]).astype(np.int64)
    big[-1] = big[-2] - 1                                     # the last request only
    assert _check(big) == pkm.PKM_ERR_INVALID_ARG
    big = np.concatenate([[0], np.cumsum(np.full(6000, 3))]).astype(np.int64)
    big[1] = 5                                                # 0, 5, 6: fine
    assert _check(big) == 0


_DEBUG_CHILD = r"""
import sys, numpy as np, torch
sys.path[:0] = [{root!r}, {tests!r}]
import workloads
from gpu_util import DeviceDecompress
d = workloads.make_decompress("dbg", 1301, [20, 20, 20], [0, 0, 0], 16, 64, 16, 128)
d.buffer_row_offsets = np.array([0, 12, 8, 30], np.uint32)   # decreases after request 0
d.buffer_length = 30
g = DeviceDecompress(d)
g.run()
torch.cuda.synchronize()
print(int(g.status.item()))
"""


@pytest.mark.parametrize("debug", ["0", "1"])
def test_debug_switch_checks_every_call(debug):
    """With PKM_DEBUG_VALIDATE=1 the decompress reports the decreasing offsets in its status
    word; without it the same call (every lookup in range) reports nothing."""
    env = dict(os.environ, PKM_DEBUG_VALIDATE=debug)
    code = _DEBUG_CHILD.format(root=os.path.dirname(HERE), tests=HERE)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert int(out.stdout.strip().splitlines()[-1]) == (1 if debug == "1" else 0)
