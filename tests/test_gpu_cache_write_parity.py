"""GPU parity of the cache-write side (RMSNorm with kv_norm_gamma, RoPE with freqs_cis,
stored into the paged latent cache), called through the C ABI, against the CPU oracle on
the same seeded inputs.  The cache starts filled with a NaN sentinel: the set of slots
written must equal the oracle's bit for bit, and their values agree within
|gpu - oracle| <= 1e-2 |oracle| + 2e-3 (one bf16 rounding of an fp32 result against one of
an fp64 result).  Inputs whose arithmetic is exact in fp32 must match bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from gpu_util import BF16_TOL, DeviceCacheWrite, assert_close_bf16
from util import oracle_cache_write

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_mla_gb300  # noqa: F401  (raises if the library is missing)


def check_full(c, expect_status=0):
    g = DeviceCacheWrite(c)
    g.run()
    out, status = g.results()
    st, ref = oracle_cache_write(c)
    assert st == expect_status and status == expect_status
    changed_ref = ref != c.cache
    changed_gpu = out != c.cache
    assert np.array_equal(changed_ref, changed_gpu), "written cache elements differ"
    assert_close_bf16(out[changed_ref], ref[changed_ref], BF16_TOL, "cache values")
    return out, ref


@pytest.mark.parametrize("new,lens,R,P,ps", [
    ([7, 1, 300, 0, 45], [5, 0, 17, 3, 128], 512, 64, 16),   # DeepSeek-V3 latent, ragged
    ([130, 129], [0, 250], 512, 64, 128),
    ([64, 11, 3], [1, 2, 127], 128, 32, 32),
    ([40], [9], 1024, 256, 8),                                # largest supported R and P
    ([33, 2], [0, 5], 8, 8, 4),                               # smallest R and P
    ([17, 9], [3, 60], 256, 0, 16),                           # no rope columns
    ([50, 50], [0, 0], 96, 24, 64),                           # R, P not powers of two
])
def test_cache_write_mid(new, lens, R, P, ps):
    c = workloads.make_cache_write("cwmid", 700 + R + P + ps, new, lens, R, P, ps, num_layers=2,
                                   layer_idx=1, extra_pages=3)
    check_full(c)


def test_cache_write_exact_inputs_bit_exact():
    """Rows of +-2^e (mean square 4^e: the norm factor is an exact power of two), gamma
    small dyadic values, epsilon 0 and rotations by multiples of 90 degrees: every result is
    exact in fp32 and fp64, so the cache must match the oracle bit for bit."""
    c = workloads.make_cache_write("cwexact", 731, [70, 200, 1], [9, 0, 64], 512, 64, 32)
    g = np.random.default_rng(731)
    M, C = c.latent.shape
    e = g.integers(-3, 4, size=(M, 1))
    sign = np.where(g.random((M, C)) < 0.5, -1.0, 1.0)
    vals = (sign * np.power(2.0, e)).astype(np.float32)
    vals[:, 512:] = g.integers(-64, 65, size=(M, 64)) / 8.0
    c.latent = (vals.view(np.uint32) >> 16).astype(np.uint16)
    c.gamma = (g.integers(1, 33, size=512) / 16.0).astype(np.float32)
    c.epsilon = 0.0
    q = g.integers(0, 4, size=c.freqs_cis.shape[:1] + (32,))
    cs = np.stack([np.choose(q, [1.0, 0.0, -1.0, 0.0]), np.choose(q, [0.0, 1.0, 0.0, -1.0])], -1)
    c.freqs_cis = cs.reshape(c.freqs_cis.shape).astype(np.float32)
    gpu = DeviceCacheWrite(c)
    gpu.run()
    out, status = gpu.results()
    st, ref = oracle_cache_write(c)
    assert status == 0 and st == 0
    assert np.array_equal(out, ref)


def test_cache_write_out_of_range_rows_skipped():
    c = workloads.make_cache_write("cwoor", 733, [40, 70, 9], [0, 100, 3], 512, 64, 32,
                                   extra_pages=2)
    c.page_table = c.page_table.copy()
    c.page_table[1, 4] = c.num_pages + 9     # positions 128..159 of request 1
    check_full(c, expect_status=4)
    # positions past freqs_cis (max_seq_len) are out of range too
    c2 = workloads.make_cache_write("cwoor2", 735, [20, 30], [4, 10], 128, 32, 16,
                                    max_seq_len=30, extra_pages=2)
    check_full(c2, expect_status=4)


def test_cache_write_empty_and_stream():
    import paged_kv_mla_gb300 as pkm
    c = workloads.make_cache_write("cwempty", 737, [0, 0], [3, 4], 512, 64, 16, extra_pages=1)
    g = DeviceCacheWrite(c)
    assert g.run() == pkm.PKM_OK
    out, status = g.results()
    assert status == 0 and np.array_equal(out, c.cache)
    c = workloads.make_cache_write("cwstream", 739, [300, 5], [1, 0], 512, 64, 64)
    g = DeviceCacheWrite(c)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.run(stream=s)
    s.synchronize()
    out, status = g.results()
    st, ref = oracle_cache_write(c)
    changed = ref != c.cache
    assert status == 0 and np.array_equal(changed, out != c.cache)
    assert_close_bf16(out[changed], ref[changed], BF16_TOL, "cache values")


def test_cache_write_deterministic():
    c = workloads.make_cache_write("cwdet", 741, [500, 77], [3, 900], 512, 64, 128)
    a = DeviceCacheWrite(c)
    a.run()
    b = DeviceCacheWrite(c)
    b.run()
    assert np.array_equal(a.results()[0], b.results()[0])


def test_cache_write_path_full_size():
    """DeepSeek-V3 prefill write (32 requests, ~80k new rows): every element of both layers
    against the whole oracle."""
    c = workloads.WORKLOADS["cache_write_path"]()
    out, ref = check_full(c)
    assert np.array_equal(out[0], c.cache[0])      # layer 0 untouched
