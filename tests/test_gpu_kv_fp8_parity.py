"""GPU parity of the FP8 kv_matmul (hidden rows quantised per 128 columns, e4m3 weight with
128 x 128 fp32 block scales, block-scaled product written into the paged K/V cache), called
through the C ABI, against the CPU oracle on the same seeded inputs.  The quantised rows and
the set of cache elements written are compared bit for bit; values within the FP8 tolerance
(3e-2 |oracle| + 5e-3)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import FP8_TOL, DeviceKvMatmul, assert_close_bf16
from util import e4m3_midpoint_bf16_values, kv_cache_view, oracle_kv_matmul_fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_mla_gb300  # noqa: F401  (raises if the library is missing)


def check_full(k, expect_status=0):
    g = DeviceKvMatmul(k)
    g.run()
    out, status = g.results()
    q, s = g.quantised_rows()
    st, ref, oq, os_ = oracle_kv_matmul_fp8(k)
    assert status == expect_status and st == expect_status
    changed_ref = ref != k.cache
    assert np.array_equal(changed_ref, out != k.cache), "written cache elements differ"
    assert_close_bf16(out[changed_ref], ref[changed_ref], FP8_TOL, "fp8 kv cache values")
    rows = (oq != 0).any(1) | (os_ != 0).any(1)          # rows the oracle wrote
    assert np.array_equal(q[rows], oq[rows]) and np.array_equal(s[rows], os_[rows])
    return out


@pytest.mark.parametrize("new,lens,k_in,hkv,d,ps,k_only", [
    ([7, 1, 300, 0, 45], [5, 0, 17, 3, 128], 512, 2, 128, 16, False),
    ([130, 129], [0, 250], 1024, 8, 128, 128, False),
    ([64, 11], [1, 2], 384, 1, 256, 32, True),           # odd number of 128-column blocks
    ([90, 3], [0, 7], 256, 3, 64, 8, False),             # HD = 192: K/V boundary inside a tile
])
def test_kv_matmul_fp8_mid(new, lens, k_in, hkv, d, ps, k_only):
    k = workloads.make_kv_matmul("kvf8", 600 + k_in + hkv, new, lens, k_in, hkv, d, ps,
                                 num_layers=2, layer_idx=1, k_only=k_only, extra_pages=4,
                                 fp8=True)
    check_full(k)


def test_kv_matmul_fp8_out_of_range():
    k = workloads.make_kv_matmul("kvf8oor", 623, [40, 70], [0, 100], 256, 2, 64, 32, fp8=True)
    k.page_table = k.page_table.copy()
    k.page_table[1, 4] = k.num_pages + 9   # positions 128..159 of request 1
    check_full(k, expect_status=4)


def test_kv_matmul_fp8_empty():
    import paged_kv_mla_gb300 as pkm
    k = workloads.make_kv_matmul("kvf8e", 625, [0, 0], [3, 4], 128, 1, 64, 16, extra_pages=1,
                                 fp8=True)
    g = DeviceKvMatmul(k)
    assert g.run() == pkm.PKM_OK
    out, status = g.results()
    assert status == 0 and np.array_equal(out, k.cache)


def test_kv_matmul_fp8_write_path_full_size():
    """6 496 rows, K = 4096, N = 2048: addressing of every row and the quantised rows bit for
    bit, values of three whole requests against the oracle."""
    k = workloads.WORKLOADS["kv_matmul_fp8_write_path"]()
    g = DeviceKvMatmul(k)
    g.run()
    out, status = g.results()
    q, s = g.quantised_rows()
    assert status == 0
    view = kv_cache_view(k)
    dest = oracle.kv_row_dest(k.input_row_offsets, k.batch, k.total_rows, k.cache_lengths, view)
    assert (dest >= 0).all()
    _, _, P, S, E = k.cache.shape
    expect = np.zeros((P * S,), bool)
    expect[dest // E] = True
    changed = (out[0] != k.cache[0]).any(axis=-1).reshape(2, P * S)
    assert np.array_equal(changed[0], expect) and np.array_equal(changed[1], expect)
    for r in range(0, k.total_rows, 7):
        q1, s1 = oracle.quantize_row_e4m3(k.hidden_state[r], k.k_in)
        assert np.array_equal(q[r], q1) and np.array_equal(s[r], s1)
    pick = [0, 13, 31]
    iro = k.input_row_offsets.astype(np.int64)
    rows = np.concatenate([np.arange(iro[b], iro[b + 1]) for b in pick])
    sub = workloads.KvMatmulInputs(
        name="sub", hidden_state=k.hidden_state[rows],
        input_row_offsets=np.concatenate([[0], np.cumsum([iro[b + 1] - iro[b] for b in pick])]).astype(np.uint32),
        weight=None, cache=k.cache, page_table=k.page_table[pick],
        cache_lengths=k.cache_lengths[pick], head_elems=k.head_elems, layer_idx=k.layer_idx,
        w_e4m3=k.w_e4m3, w_scale=k.w_scale)
    st, ref, _, _ = oracle_kv_matmul_fp8(sub)
    changed_ref = ref != k.cache
    assert_close_bf16(out[changed_ref], ref[changed_ref], FP8_TOL, "fp8 kv cache values")


def test_kv_matmul_fp8_quantisation_at_e4m3_midpoints_bit_exact():
    """Hidden blocks with a power-of-two scale (amax = 448 * 2^k) whose other values sit on
    e4m3 rounding midpoints or one bf16 step beside them (normal and subnormal e4m3 range):
    the quantised rows must equal the oracle's bit for bit."""
    k = workloads.make_kv_matmul("kvmid", 641, [40, 25], [0, 3], 512, 1, 128, 16, fp8=True)
    vals = bf16_bits = e4m3_midpoint_bf16_values()
    rng = np.random.default_rng(641)
    h = np.empty_like(k.hidden_state)
    for r in range(h.shape[0]):
        for kb in range(4):
            j = int(rng.integers(-4, 3))
            blk = workloads.bf16_bits_to_float(rng.choice(bf16_bits, 128)).astype(np.float64)
            blk *= np.where(rng.random(128) < 0.5, -1.0, 1.0) * 2.0 ** j
            blk[int(rng.integers(0, 128))] = 448.0 * 2.0 ** j
            h[r, kb * 128:(kb + 1) * 128] = [oracle.double_to_bf16(v) for v in blk]
    k.hidden_state = h
    check_full(k)
