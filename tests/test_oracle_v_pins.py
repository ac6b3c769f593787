"""Pins of the oracle's V up-projection (w_uv) against what the pages and the mathematics
fix: a hand-computed worked example through the paged gather (tests/golden), one-hot
latent rows that read w_uv back in its [head, v_dim, latent] order, exact small-integer
products, composition with the K path, and the FP8 block-scale indexing.  No GPU."""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
import workloads
from util import (assert_correctly_rounded_bf16, bf16_to_f64, cache_view, e4m3_decode_table,
                  f32_to_bf16_exact, oracle_decompress, oracle_decompress_fp8)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kv(d, **kw):
    return oracle.decompress_kv(cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets,
                                d.batch, d.buffer_length, d.kv_lora_rank, d.rope_dim, d.w_k, d.w_uv,
                                **kw)


def _kv_fp8(d):
    return oracle.decompress_kv_fp8(cache_view(d), d.layer_idx, d.buffer_row_offsets,
                                    d.cache_offsets, d.batch, d.buffer_length, d.kv_lora_rank,
                                    d.rope_dim, d.w_k_e4m3, d.w_k_scale, d.w_uv_e4m3, d.w_uv_scale)


def test_v_worked_example():
    with open(os.path.join(GOLDEN, "decompress_v_worked_example.json")) as f:
        ex = json.load(f)
    with open(os.path.join(GOLDEN, ex["uses"])) as f:
        base = json.load(f)
    lay1 = np.array(base["cache_layer1"], np.float32)
    cache = np.stack([np.full_like(lay1, base["cache_layer0_fill"]), lay1])
    d = workloads.DecompressInputs(
        name="worked_v", cache=f32_to_bf16_exact(cache),
        page_table=np.array(base["page_table"], np.uint32),
        buffer_row_offsets=np.array(base["buffer_row_offsets"], np.uint32),
        cache_offsets=np.array(base["cache_offsets"], np.uint32), buffer_length=base["buffer_length"],
        kv_lora_rank=base["kv_lora_rank"], rope_dim=base["rope_dim"], n_out=2,
        layer_idx=base["layer_idx"], w_k=f32_to_bf16_exact(np.array(base["w_k"], np.float32)),
        w_uv=f32_to_bf16_exact(np.array(ex["w_uv"], np.float32)))
    st, lat, k, v, written = _kv(d)
    assert st == 0 and written.all()
    assert np.array_equal(bf16_to_f64(lat), np.array(base["expected_k_latent"], np.float64))
    assert np.array_equal(bf16_to_f64(k), np.array(base["expected_k_buffer"], np.float64))
    assert v.shape == (4, ex["num_heads"], ex["v_head_dim"])
    assert np.array_equal(bf16_to_f64(v), np.array(ex["expected_v_buffer"], np.float64))
    for r in range(d.buffer_length):
        st, lrow, krow, vrow = oracle.decompress_kv_row(
            cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch,
            d.buffer_length, d.kv_lora_rank, d.rope_dim, d.w_k, d.w_uv, r)
        assert st == 0 and np.array_equal(krow, k[r]) and np.array_equal(vrow, v[r])


def test_v_one_hot_rows_read_w_uv_in_head_vdim_latent_order():
    H, Dv, R = 3, 5, 8
    g = workloads._gen(7)
    w_uv = workloads.bf16_normal((H, Dv, R), 1.0, g)
    lat = f32_to_bf16_exact(np.concatenate([np.eye(R, dtype=np.float32),
                                            np.full((R, 2), 7.0, np.float32)], axis=1))
    v = oracle.up_project_v_bf16(lat, R + 2, w_uv, R)
    for k in range(R):
        assert np.array_equal(v[k], w_uv[:, :, k])  # a single exact product per output


def test_v_small_integers_exact_and_k_path_unchanged():
    d = workloads.make_decompress("ints_v", 43, [30, 61], [3, 7], 8, 64, 16, 64, int_values=True)
    workloads.add_v_weight(d, 4, 16, 44, int_values=True)
    st, lat, k, v, written = _kv(d)
    assert st == 0 and written.all()
    a = bf16_to_f64(lat[:, :64]).astype(np.int64)
    w = bf16_to_f64(d.w_uv).astype(np.int64)
    assert np.array_equal(bf16_to_f64(v).astype(np.int64), np.einsum("rk,hdk->rhd", a, w))
    _, lat2, k2, _ = oracle_decompress(d)
    assert np.array_equal(lat, lat2) and np.array_equal(k, k2)


def test_v_untouched_rows_and_row_form():
    d = workloads.make_decompress("edges_v", 53, [9, 0, 12, 5], [2, 0, 12, 0], 4, 128, 64, 128)
    workloads.add_v_weight(d, 2, 128, 54)
    L = int(d.buffer_row_offsets[-1])
    d.buffer_length = L + 3
    sent_v = np.full((L + 3, 2, 128), workloads.SENTINEL_OUT, np.uint16)
    st, lat, k, v, written = _kv(d, v_buffer=sent_v)
    assert st == 0 and written[:L].all() and not written[L:].any()
    assert (v[L:] == workloads.SENTINEL_OUT).all() and not (v[:L] == workloads.SENTINEL_OUT).all()
    exact = np.einsum("rk,hdk->rhd", bf16_to_f64(lat[:L, :128]), bf16_to_f64(d.w_uv))
    assert_correctly_rounded_bf16(v[:L], exact)
    for r in [0, 5, L - 1]:
        st, _, krow, vrow = oracle.decompress_kv_row(
            cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch,
            d.buffer_length, d.kv_lora_rank, d.rope_dim, d.w_k, d.w_uv, r)
        assert st == 0 and np.array_equal(vrow, v[r]) and np.array_equal(krow, k[r])


def test_fp8_v_block_scales_index_heads_by_rows_of_128():
    # v_head_dim 64: each 128-row block of w_uv_scale spans two heads
    for Dv in (64, 128):
        d = workloads.make_decompress("f8v", 83, [150, 61], [20, 0], 32, 256, 64, 256, fp8=True)
        workloads.add_v_weight(d, 4, Dv, 84, fp8=True)
        st, lat, k, v, q, qs, written = _kv_fp8(d)
        assert st == 0 and written.all()
        table = e4m3_decode_table()
        a = table[q] * np.repeat(qs.astype(np.float64), 128, axis=1)
        wv = table[d.w_uv_e4m3.reshape(4 * Dv, 256)] * np.repeat(
            np.repeat(d.w_uv_scale.astype(np.float64), 128, axis=0), 128, axis=1)
        exact = (a @ wv.T).reshape(-1, 4, Dv)
        assert_correctly_rounded_bf16(v, exact, rel_slack=1e-9)
        # K part, codes and scales identical to the K-only FP8 decompress
        st2, lat2, k2, q2, qs2, _ = oracle_decompress_fp8(d)
        assert np.array_equal(k, k2) and np.array_equal(q, q2) and np.array_equal(qs, qs2)
        for r in [0, 129, d.buffer_length - 1]:
            st, _, krow, vrow, qrow, _ = oracle.decompress_kv_fp8_row(
                cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch,
                d.buffer_length, d.kv_lora_rank, d.rope_dim, d.w_k_e4m3, d.w_k_scale,
                d.w_uv_e4m3, d.w_uv_scale, r)
            assert st == 0 and np.array_equal(vrow, v[r]) and np.array_equal(krow, k[r])
