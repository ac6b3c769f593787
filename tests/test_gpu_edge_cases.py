"""GPU parity on degenerate and extreme shapes, through the C ABI against the oracle:
one token per page (page_size 1), decode-shaped batches (thousands of requests of one or two
rows, so every tile mixes many requests and pages), and rows that start mid-page.  Same
comparison rules as the other parity tests (bit for bit for gathered rows, codes, scales
and addresses; tolerance for products)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from gpu_util import BF16_TOL, FP8_TOL, DeviceCacheWrite, DeviceKvMatmul, assert_close_bf16
from test_gpu_parity import check_full_decompress, check_full_fp8
from util import oracle_cache_write, oracle_kv_matmul, oracle_kv_matmul_fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_mla_gb300  # noqa: F401  (raises if the library is missing)


def _decode_batch(seed, batch, max_len, page_size):
    """`batch` requests of 1-2 copied tokens at the end of histories up to max_len."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(2, max_len, batch)
    offsets = lengths - rng.integers(1, 3, batch)
    return lengths.tolist(), offsets.tolist()


@pytest.mark.parametrize("fp8", [False, True])
def test_decompress_one_token_per_page(fp8):
    d = workloads.make_decompress("ps1", 801, [37, 300, 5], [0, 41, 2], 1, 512, 64, 256, fp8=fp8,
                                  extra_pages=7)
    (check_full_fp8 if fp8 else check_full_decompress)(d)


@pytest.mark.parametrize("fp8", [False, True])
def test_decompress_decode_shaped_batch(fp8):
    lengths, offsets = _decode_batch(803, 1000, 512, 64)
    d = workloads.make_decompress("decode", 805, lengths, offsets, 64, 512, 64, 256, fp8=fp8)
    (check_full_fp8 if fp8 else check_full_decompress)(d)


def test_qcache_decompress_decode_shaped_batch():
    from test_gpu_qcache_parity import check_decompress
    lengths, offsets = _decode_batch(807, 1200, 512, 32)
    d = workloads.make_qcache_decompress("qdecode", 809, lengths, offsets, 32, 512, 64, 256)
    check_decompress(d)


@pytest.mark.parametrize("page_size", [1, 64])
def test_cache_write_decode_shaped_batch(page_size):
    rng = np.random.default_rng(811)
    new = rng.integers(0, 3, 900)
    lens = rng.integers(0, 3000, 900)
    c = workloads.make_cache_write("cwdec", 813, new, lens, 512, 64, page_size, extra_pages=3)
    g = DeviceCacheWrite(c)
    g.run()
    out, status = g.results()
    st, ref = oracle_cache_write(c)
    changed = ref != c.cache
    assert status == st == 0 and np.array_equal(changed, out != c.cache)
    assert_close_bf16(out[changed], ref[changed], BF16_TOL, "cache values")


@pytest.mark.parametrize("fp8", [False, True])
def test_kv_matmul_one_token_per_page_and_decode_batch(fp8):
    rng = np.random.default_rng(815)
    new = rng.integers(1, 3, 300)
    lens = rng.integers(0, 500, 300)
    k = workloads.make_kv_matmul("kvdec", 817, new, lens, 512, 2, 128, 1, fp8=fp8, extra_pages=2)
    g = DeviceKvMatmul(k)
    g.run()
    out, status = g.results()
    st, ref = (oracle_kv_matmul_fp8(k)[:2] if fp8 else oracle_kv_matmul(k))
    changed = ref != k.cache
    assert status == st == 0 and np.array_equal(changed, out != k.cache)
    assert_close_bf16(out[changed], ref[changed], FP8_TOL if fp8 else BF16_TOL, "kv cache values")
