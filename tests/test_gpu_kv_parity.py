"""GPU parity of the K-and-V decompress (mla_decompress_kv_paged and its FP8 form) against
the oracle, through the C ABI: whole outputs at sizes the oracle finishes in seconds
(several tiles, ragged tails, both gather paths, every n-tile width), the K half against
the K-only entry point, and sampled rows at the DeepSeek-V3 size."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import BF16_TOL, FP8_TOL, DeviceDecompress, assert_close_bf16, host_u16
from util import cache_view

pytestmark = pytest.mark.gpu

SENT = workloads.SENTINEL_OUT


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_mla_gb300  # noqa: F401  (raises if the library is missing)


def _oracle_kv(d, fp8):
    L = d.buffer_length
    if fp8:
        st, lat, k, v, q, s, written = oracle.decompress_kv_fp8(
            cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch, L,
            d.kv_lora_rank, d.rope_dim, d.w_k_e4m3, d.w_k_scale, d.w_uv_e4m3, d.w_uv_scale)
        return st, lat, k, v, written, (q, s)
    wv = d.w_uv
    st, lat, k, v, written = oracle.decompress_kv(
        cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch, L,
        d.kv_lora_rank, d.rope_dim, d.w_k, wv,
        k_latent=np.full((L, d.latent_cols), SENT, np.uint16),
        k_buffer=np.full((L, d.n_out), SENT, np.uint16),
        v_buffer=np.full((L, wv.shape[0], wv.shape[1]), SENT, np.uint16))
    return st, lat, k, v, written, None


def check_full_kv(d, fp8=False, expect_status=0):
    g = DeviceDecompress(d, fp8=fp8)
    g.run()
    lat, kb, status = g.results()
    vb = g.v_results()
    st, olat, ok, ov, written, codes = _oracle_kv(d, fp8)
    tol = FP8_TOL if fp8 else BF16_TOL
    assert status == expect_status and st == expect_status
    assert np.array_equal(lat[written], olat[written]), "k_latent_buffer differs from the oracle"
    assert (kb[~written] == SENT).all() and (vb[~written] == SENT).all(), "uncovered rows written"
    assert_close_bf16(kb[written], ok[written], tol, "k_buffer")
    assert_close_bf16(vb[written], ov[written], tol, "v_buffer")
    if fp8:
        q, s = g.fp8_workspace()
        assert np.array_equal(q[written], codes[0][written]), "quantised codes differ"
        assert np.array_equal(s[written], codes[1][written]), "activation scales differ"
    return g, kb, vb


@pytest.mark.parametrize("R,P,N,H,Dv,ps,lengths,offsets,layers", [
    (512, 64, 1024, 4, 128, 16, [300, 0, 517, 64, 129], [7, 0, 100, 0, 1], 2),  # TMA gather
    (128, 64, 384, 3, 128, 128, [1000, 77], [31, 5], 1),                         # bn = 128
    (256, 0, 320, 5, 64, 64, [250, 3, 190], [0, 0, 17], 1),                      # bn = 64
    (64, 16, 256, 2, 32, 4, [40, 90, 1], [3, 0, 0], 3),                          # cp.async gather
])
def test_kv_decompress_mid(R, P, N, H, Dv, ps, lengths, offsets, layers):
    d = workloads.make_decompress("kvmid", 500 + R + N, lengths, offsets, ps, R, P, N,
                                  num_layers=layers, layer_idx=layers - 1, extra_pages=5)
    workloads.add_v_weight(d, H, Dv, 600 + H * Dv)
    check_full_kv(d)


def test_kv_decompress_k_half_equals_k_only_call_and_clips_rows():
    d = workloads.make_decompress("kvk", 511, [200, 131], [0, 9], 32, 512, 64, 512)
    workloads.add_v_weight(d, 2, 256, 512)
    d.buffer_length = int(d.buffer_row_offsets[-1]) + 37   # rows past the requests untouched
    g, kb, vb = check_full_kv(d)
    w_uv = d.w_uv
    d.w_uv = None
    g2 = DeviceDecompress(d)
    g2.run()
    lat2, kb2, st2 = g2.results()
    assert st2 == 0 and np.array_equal(kb, kb2), "K half differs from the K-only entry point"
    d.w_uv = w_uv
    d.buffer_length = 150                                   # fewer rows than the requests
    check_full_kv(d)


def test_kv_decompress_out_of_range_page_sets_status():
    d = workloads.make_decompress("kvoor", 513, [260, 131], [0, 9], 32, 256, 64, 256)
    workloads.add_v_weight(d, 2, 128, 514)
    d.page_table = d.page_table.copy()
    d.page_table[1, 1] = d.num_pages + 3
    check_full_kv(d, expect_status=4)


@pytest.mark.parametrize("R,P,N,H,Dv,ps,lengths,offsets", [
    (512, 64, 1024, 4, 128, 16, [300, 0, 517, 64, 129], [7, 0, 100, 0, 1]),
    (128, 64, 256, 2, 64, 128, [700, 77], [31, 5]),      # a scale block spans two heads
    (384, 0, 384, 3, 128, 32, [190, 2], [0, 1]),
])
def test_kv_decompress_fp8_mid(R, P, N, H, Dv, ps, lengths, offsets):
    d = workloads.make_decompress("kvf8", 700 + R + N, lengths, offsets, ps, R, P, N, fp8=True,
                                  num_layers=2, layer_idx=1, extra_pages=3)
    workloads.add_v_weight(d, H, Dv, 800 + H * Dv, fp8=True)
    check_full_kv(d, fp8=True)


def _sampled_rows(d, n, seed):
    g = np.random.default_rng(seed)
    bro = d.buffer_row_offsets.astype(np.int64)
    rows = set(g.integers(0, d.buffer_length, n).tolist())
    for b in range(d.batch):
        if bro[b + 1] > bro[b]:
            rows.update([int(bro[b]), int(bro[b + 1] - 1)])
    return np.array(sorted(r for r in rows if r < d.buffer_length), np.int64)


@pytest.mark.parametrize("fp8", [False, True])
def test_deepseek_v3_kv_decompress_full_size(fp8):
    d = workloads.WORKLOADS["deepseek_v3_fp8_decompress_kv" if fp8 else
                            "deepseek_v3_bf16_decompress_kv"]()
    g = DeviceDecompress(d, fp8=fp8)
    g.run()
    torch.cuda.synchronize()
    assert int(g.status.item()) == 0
    rows = _sampled_rows(d, 96, 21 if fp8 else 19)
    idx = torch.from_numpy(rows).cuda()
    kb = host_u16(g.k_buffer.index_select(0, idx))
    vb = host_u16(g.v_buffer.index_select(0, idx)).reshape(len(rows), -1)
    rk, rv = np.zeros_like(kb), np.zeros_like(vb)
    for j, r in enumerate(rows):
        if fp8:
            st, _, krow, vrow, _, _ = oracle.decompress_kv_fp8_row(
                cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch,
                d.buffer_length, d.kv_lora_rank, d.rope_dim, d.w_k_e4m3, d.w_k_scale,
                d.w_uv_e4m3, d.w_uv_scale, r)
        else:
            st, _, krow, vrow = oracle.decompress_kv_row(
                cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch,
                d.buffer_length, d.kv_lora_rank, d.rope_dim, d.w_k, d.w_uv, r)
        assert st == 0
        rk[j], rv[j] = krow, vrow.reshape(-1)
    tol = FP8_TOL if fp8 else BF16_TOL
    assert_close_bf16(kb, rk, tol, "sampled k_buffer rows")
    assert_close_bf16(vb, rv, tol, "sampled v_buffer rows")
    sent16 = int(np.uint16(SENT).view(np.int16))
    assert not bool((g.v_buffer == sent16).any().item()), "a covered V row was not written"
