"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU oracle on the
same seeded inputs.  k_latent_buffer, quantised codes / scales and every cache address are
compared bit for bit; floating-point outputs within |gpu - oracle| <= rtol*|oracle| + atol
(bf16: 1e-2, 2e-3; FP8: 3e-2, 5e-3).  Outputs start filled with sentinels so that rows /
slots the operation must not touch are checked too.  Full-size workloads are checked on
sampled rows (the oracle computes them one by one) plus properties over every row."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import (BF16_TOL, FP8_TOL, DeviceDecompress, DeviceKvMatmul, assert_close_bf16,
                      dev, host_u16)
from util import cache_view, kv_cache_view, oracle_decompress, oracle_decompress_fp8, oracle_kv_matmul

pytestmark = pytest.mark.gpu

SENT = workloads.SENTINEL_OUT


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_mla_gb300  # noqa: F401  (raises if the library is missing)


def _sentinel(shape):
    return np.full(shape, SENT, np.uint16)


def check_full_decompress(d, expect_status=0):
    """Runs the GPU and the whole oracle; compares everything."""
    g = DeviceDecompress(d)
    g.run()
    lat, kb, status = g.results()
    L = d.buffer_length
    st, olat, ok, written = oracle_decompress(d, k_latent=_sentinel((L, d.latent_cols)),
                                              k_buffer=_sentinel((L, d.n_out)))
    assert status == expect_status and st == expect_status
    assert np.array_equal(lat, olat), "k_latent_buffer differs from the oracle"
    assert (kb[~written] == SENT).all(), "rows no request covers were written"
    assert_close_bf16(kb[written], ok[written], BF16_TOL, "k_buffer")
    return g, kb, ok, written


def test_tiny_decompress():
    check_full_decompress(workloads.tiny_decompress())


@pytest.mark.parametrize("R,P,N,ps,lengths,offsets,layers", [
    (512, 64, 1024, 16, [300, 0, 517, 64, 129], [7, 0, 100, 0, 1], 2),   # 8 m-tiles, ragged tail
    (128, 64, 384, 128, [1000, 77], [31, 5], 1),                          # bn = 128
    (256, 0, 320, 64, [250, 3, 190], [0, 0, 17], 1),                      # bn = 64, no rope
    (64, 16, 256, 4, [40, 90, 1], [3, 0, 0], 3),                          # tiny pages
    (192, 64, 256, 32, [600, 45, 211], [0, 3, 9], 1),                     # odd k-block count
])
def test_decompress_mid(R, P, N, ps, lengths, offsets, layers):
    d = workloads.make_decompress("mid", 200 + R + N, lengths, offsets, ps, R, P, N,
                                  num_layers=layers, layer_idx=layers - 1, extra_pages=5)
    check_full_decompress(d)


def test_decompress_rows_past_the_requests_are_untouched_and_clipped():
    d = workloads.make_decompress("edges", 301, [200, 131], [0, 9], 32, 512, 64, 512)
    covered = int(d.buffer_row_offsets[-1])
    d.buffer_length = covered + 77       # 77 rows that no request covers
    check_full_decompress(d)
    d.buffer_length = covered - 45       # the last request is clipped
    check_full_decompress(d)


def test_decompress_out_of_range_page_sets_status_and_skips_rows():
    d = workloads.make_decompress("oor", 303, [150, 260], [0, 10], 64, 512, 64, 256)
    d.page_table = d.page_table.copy()
    d.page_table[1, 1] = d.num_pages + 3     # tokens 64..127 of request 1
    check_full_decompress(d, expect_status=oracle_status_out_of_range())


def oracle_status_out_of_range():
    return 4


def test_decompress_small_integers_bit_exact():
    d = workloads.make_decompress("ints", 305, [333, 95], [1, 0], 16, 512, 64, 768, int_values=True)
    g = DeviceDecompress(d)
    g.run()
    lat, kb, status = g.results()
    st, olat, ok, written = oracle_decompress(d)
    assert status == 0 and written.all()
    assert np.array_equal(lat, olat) and np.array_equal(kb, ok)


def test_decompress_identity_weight_is_gather():
    d = workloads.make_decompress("eye", 307, [129, 200], [0, 3], 32, 256, 64, 256)
    eye = np.eye(256, dtype=np.float32)
    d.w_k = (eye.view(np.uint32) >> 16).astype(np.uint16)
    g = DeviceDecompress(d)
    g.run()
    lat, kb, status = g.results()
    assert status == 0
    assert np.array_equal(kb, lat[:, :256])


def test_decompress_repeatable_and_on_a_side_stream():
    d = workloads.make_decompress("rep", 309, [500, 260], [4, 0], 128, 512, 64, 2048)
    g = DeviceDecompress(d)
    g.run()
    lat1, kb1, _ = g.results()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.k_buffer.fill_(0)
        g.run(stream=s)
    s.synchronize()
    lat2, kb2, st = g.results()
    assert st == 0 and np.array_equal(lat1, lat2) and np.array_equal(kb1, kb2)


def _sample_rows(d, n_random, seed):
    """First / last row of every request, rows on both sides of page boundaries, plus
    seeded random rows."""
    bro = d.buffer_row_offsets.astype(np.int64)
    co = d.cache_offsets.astype(np.int64)
    rows = set()
    for b in range(d.batch):
        if bro[b + 1] > bro[b]:
            rows.update([bro[b], bro[b + 1] - 1])
            t0 = co[b]
            first_boundary = (-t0) % d.page_size
            for i in range(first_boundary, bro[b + 1] - bro[b], d.page_size * 7):
                rows.update([bro[b] + i, bro[b] + max(i - 1, 0)])
    g = np.random.default_rng(seed)
    rows.update(g.integers(0, d.buffer_length, n_random).tolist())
    return np.array(sorted(r for r in rows if r < d.buffer_length), np.int64)


def _check_sampled(d, g: DeviceDecompress, n_random, seed, fp8=False):
    L = d.buffer_length
    torch.cuda.synchronize()
    assert int(g.status.item()) == 0
    # k_latent_buffer in full against the oracle's gather
    st, olat, written = oracle.gather_latent(cache_view(d), d.layer_idx, d.buffer_row_offsets,
                                             d.cache_offsets, d.batch, L, d.latent_cols)
    assert st == 0 and written.all()
    assert np.array_equal(host_u16(g.k_latent)[:L], olat)
    rows = _sample_rows(d, n_random, seed)
    idx = torch.from_numpy(rows).cuda()
    kb = host_u16(g.k_buffer.index_select(0, idx))
    ref = np.zeros_like(kb)
    if fp8:
        q, s = g.fp8_workspace()
    for j, r in enumerate(rows):
        if fp8:
            st, lrow, krow, qrow, srow = oracle.decompress_k_fp8_row(
                cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch, L,
                d.kv_lora_rank, d.rope_dim, d.w_k_e4m3, d.w_k_scale, r)
            assert np.array_equal(q[r], qrow) and np.array_equal(s[r], srow), f"row {r} codes"
        else:
            st, lrow, krow = oracle.decompress_k_row(cache_view(d), d.layer_idx,
                                                     d.buffer_row_offsets, d.cache_offsets,
                                                     d.batch, L, d.kv_lora_rank, d.rope_dim,
                                                     d.w_k, r)
        assert st == 0
        ref[j] = krow
    assert_close_bf16(kb, ref, FP8_TOL if fp8 else BF16_TOL, "sampled k_buffer rows")
    return rows


def test_deepseek_v3_bf16_decompress_full_size():
    d = workloads.WORKLOADS["deepseek_v3_bf16_decompress"]()
    g = DeviceDecompress(d)
    g.run()
    _check_sampled(d, g, n_random=256, seed=11)
    # all rows: finite and never the sentinel (every row is covered here)
    kb = g.k_buffer
    assert not bool((kb == int(SENT)).any().item())
    assert bool(torch.isfinite(kb.view(torch.bfloat16).float()).all().item())


def test_long_context_decompress_full_size():
    d = workloads.WORKLOADS["long_context_decompress"]()
    g = DeviceDecompress(d)
    g.run()
    _check_sampled(d, g, n_random=96, seed=13)
    assert not bool((g.k_buffer == int(SENT)).any().item())


# ----------------------------------------------------------------------------------------
# FP8
# ----------------------------------------------------------------------------------------

def check_full_fp8(d, expect_status=0):
    g = DeviceDecompress(d, fp8=True)
    g.run()
    lat, kb, status = g.results()
    q, s = g.fp8_workspace()
    L = d.buffer_length
    st, olat, ok, oq, os_, written = oracle_decompress_fp8(d, k_latent=_sentinel((L, d.latent_cols)),
                                                           k_buffer=_sentinel((L, d.n_out)))
    assert status == expect_status and st == expect_status
    assert np.array_equal(lat, olat)
    assert np.array_equal(q[written], oq[written]), "quantised codes differ"
    assert np.array_equal(s[written], os_[written]), "activation scales differ"
    assert (kb[~written] == SENT).all()
    assert_close_bf16(kb[written], ok[written], FP8_TOL, "fp8 k_buffer")


@pytest.mark.parametrize("R,P,N,ps,lengths,offsets", [
    (512, 64, 1024, 16, [300, 0, 517, 64, 129], [7, 0, 100, 0, 1]),
    (128, 64, 256, 128, [700, 77], [31, 5]),
    (384, 0, 384, 32, [190, 2], [0, 1]),
])
def test_fp8_decompress_mid(R, P, N, ps, lengths, offsets):
    d = workloads.make_decompress("fp8mid", 400 + R + N, lengths, offsets, ps, R, P, N, fp8=True,
                                  num_layers=2, layer_idx=1, extra_pages=3)
    check_full_fp8(d)


def test_fp8_decompress_edges():
    d = workloads.make_decompress("fp8edge", 411, [260, 131], [0, 9], 32, 512, 64, 512, fp8=True)
    d.buffer_length = int(d.buffer_row_offsets[-1]) + 40
    check_full_fp8(d)
    d.page_table = d.page_table.copy()
    d.page_table[0, 2] = d.num_pages + 1
    check_full_fp8(d, expect_status=4)


@pytest.mark.parametrize("fp8", [False, True])
def test_leading_rows_and_empty_requests_are_untouched(fp8):
    """buffer_row_offsets starting above zero (generic_flare_mla_decompress_k_cache_ragged_paged,
    Args buffer_row_offsets_1d: rows below the first offset belong to no request) with empty
    requests between full ones and a request ending mid-page: the leading rows and every
    uncovered row stay untouched, the others match the oracle."""
    d = workloads.make_decompress("lead", 421, [90, 0, 170, 0, 0, 33], [5, 0, 31, 0, 0, 7], 32,
                                  512, 64, 512, fp8=fp8)
    d.buffer_row_offsets = (d.buffer_row_offsets + 37).astype(np.uint32)
    d.buffer_length = int(d.buffer_row_offsets[-1]) + 11
    if fp8:
        check_full_fp8(d)
    else:
        check_full_decompress(d)


def test_deepseek_v3_fp8_decompress_full_size():
    d = workloads.WORKLOADS["deepseek_v3_fp8_decompress"]()
    g = DeviceDecompress(d, fp8=True)
    g.run()
    _check_sampled(d, g, n_random=192, seed=17, fp8=True)


# ----------------------------------------------------------------------------------------
# kv_matmul
# ----------------------------------------------------------------------------------------

def check_full_kv(k, expect_status=0):
    g = DeviceKvMatmul(k)
    g.run()
    out, status = g.results()
    st, ref = oracle_kv_matmul(k)
    assert status == expect_status and st == expect_status
    changed_ref = ref != k.cache
    changed_gpu = out != k.cache
    assert np.array_equal(changed_ref, changed_gpu), "written cache slots differ"
    assert_close_bf16(out[changed_ref], ref[changed_ref], BF16_TOL, "kv cache values")


@pytest.mark.parametrize("new,lens,k_in,hkv,d,ps,k_only", [
    ([7, 1, 300, 0, 45], [5, 0, 17, 3, 128], 512, 2, 128, 16, False),
    ([130, 129], [0, 250], 1024, 8, 128, 128, False),
    ([64, 11], [1, 2], 256, 1, 576, 32, True),       # MLA-shaped latent cache, K only
    ([5], [0], 128, 3, 64, 8, False),                # bn = 128 (n_out 384)
])
def test_kv_matmul_mid(new, lens, k_in, hkv, d, ps, k_only):
    k = workloads.make_kv_matmul("kvmid", 500 + k_in + hkv, new, lens, k_in, hkv, d, ps,
                                 num_layers=2, layer_idx=1, k_only=k_only, extra_pages=4)
    check_full_kv(k)


def test_kv_matmul_small_integers_bit_exact():
    k = workloads.make_kv_matmul("kvint", 521, [77, 200], [9, 0], 256, 2, 64, 32, int_values=True)
    g = DeviceKvMatmul(k)
    g.run()
    out, status = g.results()
    st, ref = oracle_kv_matmul(k)
    assert status == 0 and np.array_equal(out, ref)


def test_kv_matmul_out_of_range():
    k = workloads.make_kv_matmul("kvoor", 523, [40, 70], [0, 100], 256, 2, 64, 32)
    k.page_table = k.page_table.copy()
    k.page_table[1, 4] = k.num_pages + 9   # positions 128..159 of request 1
    check_full_kv(k, expect_status=4)


def test_kv_matmul_write_path_full_size():
    k = workloads.WORKLOADS["kv_matmul_write_path"]()
    g = DeviceKvMatmul(k)
    g.run()
    out, status = g.results()
    assert status == 0
    # addressing of every row, bit for bit: the changed slots are exactly the oracle's
    view = kv_cache_view(k)
    dest = oracle.kv_row_dest(k.input_row_offsets, k.batch, k.total_rows, k.cache_lengths, view)
    assert (dest >= 0).all()
    _, _, P, S, E = k.cache.shape
    expect = np.zeros((P * S,), bool)
    expect[dest // E] = True
    changed = (out[0] != k.cache[0]).any(axis=-1).reshape(2, P * S)
    assert np.array_equal(changed[0], expect) and np.array_equal(changed[1], expect)
    # values of sampled rows of EVERY request against the oracle: each request's first and
    # last new row, the rows on both sides of every page boundary its new tokens cross, and
    # four seeded random rows.  Each sampled row becomes a one-row request of its own with
    # the same page table row and cache position, so the oracle writes the same slot.
    rng = np.random.default_rng(29)
    iro = k.input_row_offsets.astype(np.int64)
    ps = k.page_size
    sel = []
    for b in range(k.batch):
        n = int(iro[b + 1] - iro[b])
        if n == 0:
            continue
        cl = int(k.cache_lengths[b])
        picks = {0, n - 1}
        for i in range(1, n):
            if (cl + i) % ps == 0:
                picks.update({i - 1, i})
        picks.update(int(v) for v in rng.integers(0, n, 4))
        sel.extend((b, i) for i in sorted(picks))
    assert len({b for b, _ in sel}) == int((iro[1:] > iro[:-1]).sum())
    rows = np.array([iro[b] + i for b, i in sel])
    sub = workloads.KvMatmulInputs(
        name="sub", hidden_state=k.hidden_state[rows],
        input_row_offsets=np.arange(len(sel) + 1, dtype=np.uint32),
        weight=k.weight, cache=k.cache, page_table=k.page_table[[b for b, _ in sel]],
        cache_lengths=np.array([int(k.cache_lengths[b]) + i for b, i in sel], np.uint32),
        head_elems=k.head_elems, layer_idx=k.layer_idx)
    st, ref = oracle_kv_matmul(sub)
    assert st == 0
    changed_ref = ref != k.cache
    assert changed_ref.sum() == len(sel) * 2 * k.head_elems  # K and V slot of each row
    assert_close_bf16(out[changed_ref], ref[changed_ref], BF16_TOL, "kv cache values")


# ----------------------------------------------------------------------------------------
# degenerate calls
# ----------------------------------------------------------------------------------------

def test_empty_problems_launch_nothing():
    import paged_kv_mla_gb300 as pkm
    d = workloads.make_decompress("empty", 601, [0, 0], [0, 0], 16, 64, 16, 64, extra_pages=1)
    d.buffer_length = 0
    g = DeviceDecompress(d)
    assert g.run() == pkm.PKM_OK
    d2 = workloads.make_decompress("empty2", 602, [5, 9], [5, 9], 16, 64, 16, 64)
    d2.buffer_length = 8        # no request copies a row: every row stays untouched
    check_full_decompress(d2)
    k = workloads.make_kv_matmul("kvempty", 603, [0, 0], [3, 4], 128, 1, 64, 16, extra_pages=1)
    gk = DeviceKvMatmul(k)
    assert gk.run() == pkm.PKM_OK
    out, status = gk.results()
    assert status == 0 and np.array_equal(out, k.cache)


def test_bounded_wait_times_out_and_context_stays_usable():
    """Failure detection without a fault: a wait that nothing satisfies gives up after its
    limit, reports PKM_ERR_TIMEOUT, and the next launch on the same context is correct."""
    import paged_kv_mla_gb300 as pkm
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkm.pkm_check_wait_timeout(st, 200)
    torch.cuda.synchronize()
    assert int(st.item()) == pkm.PKM_ERR_TIMEOUT
    check_full_decompress(workloads.tiny_decompress())
