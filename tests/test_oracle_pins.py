"""Pins of the CPU oracle against facts fixed outside it: the number-format definitions
(via torch's casts), hand-computed worked examples (tests/golden), closed forms (identity
page table = a plain GEMM computed by numpy; W = I = a pure gather), invariances
(permuting physical pages, splitting / reordering requests, linearity) and exact integer
arithmetic.  No GPU."""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from util import (assert_correctly_rounded_bf16, bf16_to_f64, cache_view, e4m3_decode_table,
                  f32_to_bf16_exact, kv_cache_view, oracle_decompress, oracle_decompress_fp8,
                  oracle_kv_matmul)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------------------

def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_round_from_float_matches_torch_rne():
    g = np.random.default_rng(7)
    # random finite float32 bit patterns over the whole range, incl. subnormals
    u = g.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    extra = np.array([0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895314e38, 1e-40,
                      -2.5e-39, 65504.0], np.float32)
    f = np.concatenate([f, extra])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.double_to_bf16(float(x)) for x in f], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_round_from_double_is_single_rounding():
    # 1 + 2^-8 + 2^-30: a float intermediate would land on the tie 1 + 2^-8 and round to
    # even (0x3F80); the correctly rounded bf16 is 0x3F81.
    assert oracle.double_to_bf16(1.0 + 2 ** -8 + 2 ** -30) == 0x3F81
    assert oracle.double_to_bf16(1.0 + 2 ** -8) == 0x3F80          # tie -> even
    assert oracle.double_to_bf16(1.0 + 3 * 2 ** -8) == 0x3F82      # tie -> even
    assert oracle.double_to_bf16(-(1.0 + 2 ** -8 + 2 ** -30)) == 0xBF81
    assert oracle.double_to_bf16(3.4e38) == 0x7F80                 # overflow -> inf
    assert oracle.double_to_bf16(2.0 ** -134) == 0x0000            # half of min subnormal, tie -> 0
    assert oracle.double_to_bf16(1.5 * 2.0 ** -133) == 0x0002      # tie -> even (2 quanta)


def test_e4m3_decode_table_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_decode_table()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e4m3_encode_grid_midpoints_and_saturation():
    table = e4m3_decode_table()
    pos = table[:0x7F]  # 0 .. 448, increasing
    assert np.all(np.diff(pos) > 0)
    for code in range(0x7F):
        assert oracle.float_to_e4m3(pos[code]) == code
        assert oracle.float_to_e4m3(-pos[code]) == (code | 0x80)
    for code in range(0x7E):
        mid = np.float32((pos[code] + pos[code + 1]) / 2)  # exact in fp32
        even = code if code % 2 == 0 else code + 1
        assert oracle.float_to_e4m3(mid) == even
        assert oracle.float_to_e4m3(np.nextafter(mid, np.float32(1e9))) == code + 1
        assert oracle.float_to_e4m3(np.nextafter(mid, np.float32(-1e9))) == code
    for big in [448.0, 448.5, 463.9, 464.0, 500.0, 1e30, math.inf]:
        assert oracle.float_to_e4m3(big) == 0x7E
        assert oracle.float_to_e4m3(-big) == 0xFE
    assert oracle.float_to_e4m3(math.nan) == 0x7F


def test_e4m3_encode_matches_torch_in_range():
    g = np.random.default_rng(11)
    x = np.concatenate([g.uniform(-448, 448, 5000), g.normal(0, 1, 5000),
                        g.normal(0, 1e-2, 2000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.float_to_e4m3(v) for v in x], np.uint8)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------------------
# decompress: worked example, closed forms, invariances
# ---------------------------------------------------------------------------------------

def _golden_decompress():
    with open(os.path.join(GOLDEN, "decompress_worked_example.json")) as f:
        return json.load(f)


def test_decompress_worked_example():
    ex = _golden_decompress()
    lay1 = np.array(ex["cache_layer1"], np.float32)
    cache = np.stack([np.full_like(lay1, ex["cache_layer0_fill"]), lay1])
    d = workloads.DecompressInputs(
        name="worked", cache=f32_to_bf16_exact(cache), page_table=np.array(ex["page_table"], np.uint32),
        buffer_row_offsets=np.array(ex["buffer_row_offsets"], np.uint32),
        cache_offsets=np.array(ex["cache_offsets"], np.uint32), buffer_length=ex["buffer_length"],
        kv_lora_rank=ex["kv_lora_rank"], rope_dim=ex["rope_dim"], n_out=2, layer_idx=ex["layer_idx"],
        w_k=f32_to_bf16_exact(np.array(ex["w_k"], np.float32)))
    st, lat, k, written = oracle_decompress(d)
    assert st == 0 and written.all()
    assert np.array_equal(bf16_to_f64(lat), np.array(ex["expected_k_latent"], np.float64))
    assert np.array_equal(bf16_to_f64(k), np.array(ex["expected_k_buffer"], np.float64))
    for r in range(ex["buffer_length"]):
        st, lrow, krow = oracle.decompress_k_row(cache_view(d), d.layer_idx, d.buffer_row_offsets,
                                                 d.cache_offsets, d.batch, d.buffer_length,
                                                 d.kv_lora_rank, d.rope_dim, d.w_k, r)
        assert st == 0
        assert np.array_equal(lrow, lat[r]) and np.array_equal(krow, k[r])


def _identity_problem(L, R, P, N, seed):
    """One request, cache_offsets 0, one page of page_size = L, identity page table."""
    return workloads.make_decompress("identity", seed, [L], [0], L, R, P, N,
                                     page_table=np.array([[0]], np.uint32), num_pages=1)


@pytest.mark.parametrize("L,R,P,N", [(16, 64, 16, 64), (37, 128, 64, 256), (130, 512, 64, 200)])
def test_identity_page_table_is_plain_gemm(L, R, P, N):
    d = _identity_problem(L, R, P, N, seed=20 + L)
    st, lat, k, written = oracle_decompress(d)
    assert st == 0 and written.all()
    # the gather of an identity table with page_size = buffer_length is the page itself
    assert np.array_equal(lat, d.cache[0, 0, :, : R + P])
    exact = bf16_to_f64(d.cache[0, 0, :, :R]) @ bf16_to_f64(d.w_k).T  # numpy fp64 GEMM
    assert_correctly_rounded_bf16(k, exact)


def test_page_permutation_leaves_output_unchanged():
    lengths, co = workloads.deepseek_lengths(1001)
    # the DeepSeek-shaped length mix, shrunk to keep the oracle fast
    d = workloads.make_decompress("perm", 5, lengths[:3] // 8 + 5, co[:3] // 8, 16, 128, 64, 256,
                                  extra_pages=7)
    st, lat, k, written = oracle_decompress(d)
    perm = np.random.default_rng(3).permutation(d.num_pages)
    cache2 = np.empty_like(d.cache)
    cache2[:, perm] = d.cache                       # physical page p moves to perm[p]
    pt2 = d.page_table.copy()
    valid = pt2 != workloads.PAGE_TABLE_PAD
    pt2[valid] = perm[pt2[valid]]
    d2 = workloads.DecompressInputs(**{**d.__dict__, "cache": cache2, "page_table": pt2})
    st2, lat2, k2, written2 = oracle_decompress(d2)
    assert st == st2 == 0
    assert np.array_equal(lat, lat2) and np.array_equal(k, k2) and np.array_equal(written, written2)
    # and a moved page really moves the data: with the old table the result differs
    d3 = workloads.DecompressInputs(**{**d.__dict__, "cache": cache2})
    _, lat3, _, _ = oracle_decompress(d3)
    assert not np.array_equal(lat, lat3)


def test_weight_identity_is_pure_gather():
    d = workloads.make_decompress("eye", 9, [40, 3, 77], [5, 0, 13], 8, 64, 16, 64, extra_pages=3)
    d.w_k = f32_to_bf16_exact(np.eye(64, dtype=np.float32))
    st, lat, k, written = oracle_decompress(d)
    assert st == 0 and written.all()
    assert np.array_equal(k, lat[:, :64])


def test_split_and_reorder_requests_invariance():
    d = workloads.make_decompress("split", 31, [50, 20, 33], [10, 0, 4], 8, 64, 16, 128)
    st, lat, k, _ = oracle_decompress(d)
    # split request 0 (40 rows, tokens 10..49) into tokens 10..24 and 25..49 sharing its pages
    pt = d.page_table
    pt2 = np.concatenate([pt[:1], pt[:1], pt[1:]])
    co2 = np.array([10, 25, 0, 4, 0], np.uint32)
    bro2 = np.array([0, 15, 40, 60, 89], np.uint32)
    d2 = workloads.DecompressInputs(**{**d.__dict__, "page_table": pt2, "cache_offsets": co2,
                                       "buffer_row_offsets": bro2})
    st2, lat2, k2, _ = oracle_decompress(d2)
    assert np.array_equal(lat, lat2) and np.array_equal(k, k2)
    # reorder requests (2, 0, 1): row blocks move with their request
    order = [2, 0, 1]
    rows = np.diff(d.buffer_row_offsets.astype(np.int64))
    bro3 = np.concatenate([[0], np.cumsum(rows[order])]).astype(np.uint32)
    d3 = workloads.DecompressInputs(**{**d.__dict__, "page_table": pt[order],
                                       "cache_offsets": np.concatenate([d.cache_offsets[order], [0]]).astype(np.uint32),
                                       "buffer_row_offsets": bro3})
    st3, lat3, k3, _ = oracle_decompress(d3)
    blocks = [np.arange(d.buffer_row_offsets[b], d.buffer_row_offsets[b + 1]) for b in order]
    idx = np.concatenate(blocks)
    assert np.array_equal(lat3, lat[idx]) and np.array_equal(k3, k[idx])


def test_small_integers_exact_and_linear():
    d = workloads.make_decompress("ints", 41, [30, 61], [3, 7], 8, 64, 16, 64, int_values=True)
    st, lat, k, _ = oracle_decompress(d)
    a = bf16_to_f64(lat[:, :64]).astype(np.int64)
    w = bf16_to_f64(d.w_k).astype(np.int64)
    assert np.array_equal(bf16_to_f64(k).astype(np.int64), a @ w.T)  # |sums| < 256: exact
    # linearity in W
    w2 = workloads.bf16_small_ints((64, 64), -1, 1, workloads._gen(5))
    d2 = workloads.DecompressInputs(**{**d.__dict__, "w_k": w2})
    wsum = f32_to_bf16_exact(bf16_to_f64(d.w_k).astype(np.float32) + bf16_to_f64(w2).astype(np.float32))
    d3 = workloads.DecompressInputs(**{**d.__dict__, "w_k": wsum})
    _, _, k2, _ = oracle_decompress(d2)
    _, _, k3, _ = oracle_decompress(d3)
    assert np.array_equal(bf16_to_f64(k3), bf16_to_f64(k) + bf16_to_f64(k2))


def test_ragged_edges_untouched_rows_and_errors():
    d = workloads.make_decompress("edges", 51, [9, 0, 12, 5], [2, 0, 12, 0], 4, 64, 16, 64)
    # request 1 empty, request 2 copies nothing (offset == length)
    L = int(d.buffer_row_offsets[-1])
    assert L == 7 + 0 + 0 + 5
    sent_l = np.full((L + 3, d.latent_cols), workloads.SENTINEL_OUT, np.uint16)
    sent_k = np.full((L + 3, d.n_out), workloads.SENTINEL_OUT, np.uint16)
    d.buffer_length = L + 3  # three rows past the last request stay untouched
    st, lat, k, written = oracle_decompress(d, k_latent=sent_l, k_buffer=sent_k)
    assert st == 0 and written[:L].all() and not written[L:].any()
    assert (lat[L:] == workloads.SENTINEL_OUT).all() and (k[L:] == workloads.SENTINEL_OUT).all()
    # buffer_length shorter than the rows: rows are clipped
    d.buffer_length = 4
    st, lat, k, written = oracle_decompress(d)
    assert written.all() and lat.shape[0] == 4
    # a page id past the cache: error code, that row skipped
    d.buffer_length = L
    d.page_table = d.page_table.copy()
    d.page_table[3, 0] = d.num_pages + 5
    st, lat, k, written = oracle_decompress(d)
    assert st == 4 and written.sum() == L - 4  # request 3's first page holds its 4 tokens


def test_row_form_matches_full_form():
    d = workloads.make_decompress("rows", 61, [70, 33], [6, 1], 16, 128, 64, 128)
    st, lat, k, _ = oracle_decompress(d)
    for r in [0, 1, 63, 64, 65, d.buffer_length - 1]:
        st, lrow, krow = oracle.decompress_k_row(cache_view(d), d.layer_idx, d.buffer_row_offsets,
                                                 d.cache_offsets, d.batch, d.buffer_length,
                                                 d.kv_lora_rank, d.rope_dim, d.w_k, r)
        assert st == 0 and np.array_equal(lrow, lat[r]) and np.array_equal(krow, k[r])


# ---------------------------------------------------------------------------------------
# FP8
# ---------------------------------------------------------------------------------------

def test_fp8_worked_example():
    with open(os.path.join(GOLDEN, "fp8_worked_example.json")) as f:
        ex = json.load(f)
    R, N = ex["kv_lora_rank"], ex["n_out"]
    row = np.where(np.arange(R) % 2 == 0, ex["x_even"], ex["x_odd"]).astype(np.float32)
    q, s = oracle.quantize_row_e4m3(f32_to_bf16_exact(row), R)
    assert s[0] == np.float32(1.0) / np.float32(448.0)
    assert (q[0::2] == ex["expected_q_even"]).all() and (q[1::2] == ex["expected_q_odd"]).all()
    d = workloads.DecompressInputs(
        name="fp8w", cache=f32_to_bf16_exact(row.reshape(1, 1, 1, R)), page_table=np.zeros((1, 1), np.uint32),
        buffer_row_offsets=np.array([0, 1], np.uint32), cache_offsets=np.array([0, 0], np.uint32),
        buffer_length=1, kv_lora_rank=R, rope_dim=0, n_out=N, layer_idx=0,
        w_k_e4m3=np.full((N, R), ex["w_code"], np.uint8),
        w_k_scale=np.full((N // 128, R // 128), ex["w_scale"], np.float32))
    st, lat, k, qq, qs, written = oracle_decompress_fp8(d)
    assert st == 0 and written.all()
    assert (bf16_to_f64(k) == ex["expected_k"]).all()


def test_fp8_quantisation_exact_on_representable_blocks():
    table = e4m3_decode_table()
    g = np.random.default_rng(5)
    for j in [-6, 0, 3]:
        codes = g.integers(0, 0x7F, 128)
        codes[17] = 0x7E  # amax = 448 * 2^j
        vals = table[codes] * np.where(g.random(128) < 0.5, -1, 1) * 2.0 ** j
        bits = f32_to_bf16_exact(vals.astype(np.float32))
        q, s = oracle.quantize_row_e4m3(bits, 128)
        assert s[0] == 2.0 ** j
        assert np.array_equal(table[q] * s[0], bf16_to_f64(bits))
    q, s = oracle.quantize_row_e4m3(np.zeros(256, np.uint16), 256)
    assert (s == 1.0).all() and (q == 0).all()


def test_fp8_quantisation_error_bound_and_rope_excluded():
    d = workloads.make_decompress("q", 71, [200], [0], 64, 512, 64, 128, fp8=True)
    table = e4m3_decode_table()
    for r in range(0, 200, 17):
        slot = d.cache[0, d.page_table[0, r // 64], r % 64]
        q, s = oracle.quantize_row_e4m3(slot, 512)
        x = bf16_to_f64(slot[:512]).reshape(4, 128)
        amax = np.abs(x).max(axis=1)
        assert np.array_equal(s, (amax.astype(np.float32) / np.float32(448.0)))
        y = (x / s[:, None].astype(np.float64))
        dq = table[q].reshape(4, 128)
        # round-to-nearest on the e4m3 grid: error <= half the local quantum
        e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
        half_q = 0.5 * np.exp2(e - 3)
        assert (np.abs(dq - y) <= half_q * (1 + 1e-6) + 1e-7).all()
        slot2 = slot.copy()
        slot2[512:] = f32_to_bf16_exact(np.full(64, 1024.0, np.float32))
        q2, s2 = oracle.quantize_row_e4m3(slot2, 512)
        assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_fp8_block_product_matches_numpy_on_dequantised_values():
    d = workloads.make_decompress("f8", 81, [150, 61], [20, 0], 32, 256, 64, 384, fp8=True)
    st, lat, k, q, qs, written = oracle_decompress_fp8(d)
    assert st == 0 and written.all()
    table = e4m3_decode_table()
    a = table[q] * np.repeat(qs.astype(np.float64), 128, axis=1)
    w = table[d.w_k_e4m3] * np.repeat(np.repeat(d.w_k_scale.astype(np.float64), 128, axis=0), 128, axis=1)
    exact = a @ w.T
    assert_correctly_rounded_bf16(k, exact, rel_slack=1e-9)
    # bf16 gather part identical to the bf16 path's gather
    st2, lat2, _ = oracle.gather_latent(cache_view(d), d.layer_idx, d.buffer_row_offsets,
                                        d.cache_offsets, d.batch, d.buffer_length, d.latent_cols)
    assert np.array_equal(lat, lat2)
    for r in [0, 77, 129, 130, 190]:
        st, lrow, krow, qrow, srow = oracle.decompress_k_fp8_row(
            cache_view(d), 0, d.buffer_row_offsets, d.cache_offsets, d.batch, d.buffer_length,
            d.kv_lora_rank, d.rope_dim, d.w_k_e4m3, d.w_k_scale, r)
        assert st == 0 and np.array_equal(krow, k[r]) and np.array_equal(qrow, q[r])
        assert np.array_equal(srow, qs[r]) and np.array_equal(lrow, lat[r])


# ---------------------------------------------------------------------------------------
# kv_matmul
# ---------------------------------------------------------------------------------------

def test_kv_matmul_worked_example():
    with open(os.path.join(GOLDEN, "kv_matmul_worked_example.json")) as f:
        ex = json.load(f)
    ps, P, HD = ex["page_size"], ex["num_pages"], ex["head_elems"]
    cache = np.empty((1, 2, P, ps, HD), np.uint16)
    cache[:, 0] = workloads.SENTINEL_K
    cache[:, 1] = workloads.SENTINEL_V
    k = workloads.KvMatmulInputs(
        name="worked", hidden_state=f32_to_bf16_exact(np.array(ex["hidden_state"], np.float32)),
        input_row_offsets=np.array(ex["input_row_offsets"], np.uint32),
        weight=f32_to_bf16_exact(np.array(ex["weight"], np.float32)), cache=cache,
        page_table=np.array(ex["page_table"], np.uint32),
        cache_lengths=np.array(ex["cache_lengths"], np.uint32), head_elems=HD, layer_idx=0)
    st, out = oracle_kv_matmul(k)
    assert st == 0
    expected = cache.copy()
    for w in ex["expected_writes"]:
        expected[0, 0 if w["plane"] == "K" else 1, w["page"], w["slot"]] = \
            f32_to_bf16_exact(np.array(w["values"], np.float32))
    assert np.array_equal(out, expected)


def test_kv_matmul_identity_weight_is_copy_into_pages():
    k = workloads.make_kv_matmul("copy", 91, [7, 1, 30], [5, 0, 17], 64, 1, 64, 8, num_layers=2,
                                 layer_idx=1)
    eye = np.eye(64, dtype=np.float32)
    k.weight = f32_to_bf16_exact(np.concatenate([eye, eye], axis=1))
    st, out = oracle_kv_matmul(k)
    assert st == 0
    assert np.array_equal(out[0], k.cache[0])  # other layer untouched
    seen = np.zeros(out.shape[1:4], bool)
    for b in range(k.batch):
        for i in range(int(k.new_tokens[b])):
            r = k.input_row_offsets[b] + i
            pos = k.cache_lengths[b] + i
            page, slot = k.page_table[b, pos // 8], pos % 8
            assert np.array_equal(out[1, 0, page, slot], k.hidden_state[r])
            assert np.array_equal(out[1, 1, page, slot], k.hidden_state[r])
            seen[:, page, slot] = True
    assert (out[1, 0][~seen[0]] == workloads.SENTINEL_K).all()
    assert (out[1, 1][~seen[1]] == workloads.SENTINEL_V).all()


def test_kv_matmul_identity_table_is_plain_gemm():
    k = workloads.make_kv_matmul("gemm", 93, [45], [0], 256, 2, 64, 64)
    k.page_table = np.array([[0]], np.uint32)
    k.cache = k.cache[:, :, :1].copy()
    st, out = oracle_kv_matmul(k)
    exact = bf16_to_f64(k.hidden_state) @ bf16_to_f64(k.weight)
    got = np.concatenate([out[0, 0, 0, :45], out[0, 1, 0, :45]], axis=1)
    assert_correctly_rounded_bf16(got, exact)
    assert (out[0, 0, 0, 45:] == workloads.SENTINEL_K).all()  # slots past the new rows
    assert (out[0, 1, 0, 45:] == workloads.SENTINEL_V).all()


def test_kv_matmul_then_decompress_composes():
    """A K-only kv_matmul into an MLA-shaped cache (1 kv head of 576 columns), then a
    decompress of the same tokens, equals bf16(X W)[:, :512] W_k^T."""
    km = workloads.make_kv_matmul("mla", 95, [20, 9], [0, 0], 128, 1, 576, 16, k_only=True)
    st, out = oracle_kv_matmul(km)
    assert st == 0
    y = out[0, 0]  # [pages, 16, 576] K plane only
    d = workloads.DecompressInputs(
        name="compose", cache=y[None], page_table=km.page_table,
        buffer_row_offsets=km.input_row_offsets, cache_offsets=np.zeros(3, np.uint32),
        buffer_length=29, kv_lora_rank=512, rope_dim=64, n_out=128, layer_idx=0,
        w_k=workloads.bf16_normal((128, 512), 1 / math.sqrt(512), workloads._gen(3)))
    st, lat, kb, _ = oracle_decompress(d)
    yx = bf16_to_f64(km.hidden_state) @ bf16_to_f64(km.weight)
    assert_correctly_rounded_bf16(lat, yx)
    exact = bf16_to_f64(lat[:, :512]) @ bf16_to_f64(d.w_k).T
    assert_correctly_rounded_bf16(kb, exact)


def test_kv_row_dest_matches_worked_example():
    with open(os.path.join(GOLDEN, "kv_matmul_worked_example.json")) as f:
        ex = json.load(f)
    ps, P, HD = ex["page_size"], ex["num_pages"], ex["head_elems"]
    view = oracle.PagedCacheView(np.zeros(2 * P * ps * HD, np.uint16), 2 * P * ps * HD, ps * HD, HD,
                                 P, ps, np.array(ex["page_table"], np.uint32), 2, kv_stride=P * ps * HD)
    dest = oracle.kv_row_dest(np.array(ex["input_row_offsets"], np.uint32), 2, 3,
                              np.array(ex["cache_lengths"], np.uint32), view)
    k_writes = [w for w in ex["expected_writes"] if w["plane"] == "K"]
    assert list(dest) == [w["page"] * ps * HD + w["slot"] * HD for w in k_writes]
