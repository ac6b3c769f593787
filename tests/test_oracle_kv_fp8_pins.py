"""Pins of the oracle's FP8 kv_matmul (block-scaled e4m3 GEMM of the ragged hidden state,
written into the paged K/V cache) against what the pages and the mathematics fix: a
hand-derived worked example (tests/golden), exact equality with the bf16 kv_matmul when
every quantisation is exact (power-of-two scales, e4m3-representable values), the
addressing of the bf16 kv_matmul, and the quantised rows it reports.  No GPU."""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
import workloads
from util import kv_cache_view

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_fp8(k, data=None):
    v = kv_cache_view(k, data=k.cache.copy() if data is None else data)
    st, q, s = oracle.kv_matmul_fp8(k.hidden_state, k.input_row_offsets, k.batch, k.total_rows,
                                    k.w_e4m3, k.w_scale, v, k.head_elems, k.cache_lengths,
                                    k.layer_idx)
    return st, v.data.reshape(k.cache.shape), q, s


def test_kv_matmul_fp8_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_matmul_fp8_worked_example.json")))
    K, N, HD, PS = g["k_in"], g["n_out"], g["head_elems"], g["page_size"]
    k_idx = np.arange(K)
    rows = [np.ones(K), np.where(k_idx < 80, 2.0, -2.0)]
    hidden = np.array([[oracle.double_to_bf16(v) for v in r] for r in rows], np.uint16)
    cache = np.empty((1, 2, g["num_pages"], PS, HD), np.uint16)
    cache[:, 0] = workloads.SENTINEL_K
    cache[:, 1] = workloads.SENTINEL_V
    w = np.empty((N, K), np.uint8)
    w[:HD] = int(g["w_codes"]["k_columns"], 16)
    w[HD:] = int(g["w_codes"]["v_columns"], 16)
    k = workloads.KvMatmulInputs(
        name="golden", hidden_state=hidden, input_row_offsets=np.array(g["input_row_offsets"], np.uint32),
        weight=None, cache=cache, page_table=np.array(g["page_table"], np.uint32),
        cache_lengths=np.array(g["cache_lengths"], np.uint32), head_elems=HD, layer_idx=0,
        w_e4m3=w, w_scale=np.array(g["w_scale"], np.float32))
    st, out, q, s = run_fp8(k)
    assert st == 0
    touched = np.zeros(out.shape, bool)
    for e in g["expected"]:
        kv = out[0, 0, e["page"], e["slot"]], out[0, 1, e["page"], e["slot"]]
        assert (kv[0] == int(e["k_bf16"], 16)).all() and (kv[1] == int(e["v_bf16"], 16)).all()
        touched[0, :, e["page"], e["slot"]] = True
    assert (out[~touched] == cache[~touched]).all()
    assert (q[0] == 0x7E).all() and np.array_equal(q[1], np.where(k_idx < 80, 0x7E, 0xFE))
    assert s[0, 0] == np.float32(1) / np.float32(448) and s[1, 0] == np.float32(2) / np.float32(448)


def _exact_problem(seed, new, lens, k_in, heads, d, ps):
    """Hidden rows whose 128-column blocks hold e4m3 grid values times 2^j with one element
    448 * 2^j (so the block scale is 2^j and quantisation is exact), and an e4m3 weight with
    power-of-two block scales; returns the FP8 problem and the bf16 problem with the
    dequantised weight (exact in bf16)."""
    k = workloads.make_kv_matmul("ex", seed, new, lens, k_in, heads, d, ps, fp8=True)
    rng = np.random.default_rng(seed)
    grid = np.array([oracle.e4m3_to_double(c) for c in range(0x7F) if c != 0x7F])
    M = k.total_rows
    h = rng.choice(grid, (M, k_in)) * np.where(rng.random((M, k_in)) < 0.5, -1, 1)
    for r in range(M):
        for kb in range(k_in // 128):
            j = int(rng.integers(-6, 4))
            blk = h[r, kb * 128:(kb + 1) * 128] * 2.0 ** j
            blk[int(rng.integers(0, 128))] = 448.0 * 2.0 ** j
            h[r, kb * 128:(kb + 1) * 128] = blk
    k.hidden_state = np.array([[oracle.double_to_bf16(v) for v in row] for row in h], np.uint16)
    codes = rng.integers(0, 0x7F, (k.n_out, k_in)).astype(np.uint8) | (
        (rng.random((k.n_out, k_in)) < 0.5).astype(np.uint8) << 7)
    scales = (2.0 ** rng.integers(-8, 2, (k.n_out // 128, k_in // 128))).astype(np.float32)
    k.w_e4m3, k.w_scale = codes, scales
    table = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    deq = table[codes] * np.repeat(np.repeat(scales, 128, 0), 128, 1)
    wb = np.array([[oracle.double_to_bf16(v) for v in row] for row in deq.T], np.uint16)
    kb = workloads.KvMatmulInputs(name="exb", hidden_state=k.hidden_state,
                                  input_row_offsets=k.input_row_offsets, weight=wb, cache=k.cache,
                                  page_table=k.page_table, cache_lengths=k.cache_lengths,
                                  head_elems=k.head_elems, layer_idx=k.layer_idx)
    return k, kb


def test_exact_quantisation_gives_the_bf16_kv_matmul_bit_for_bit():
    k, kb = _exact_problem(4711, [9, 4], [3, 0], 256, 1, 128, 8)
    st, out, q, s = run_fp8(k)
    vb = kv_cache_view(kb, data=kb.cache.copy())
    stb = oracle.kv_matmul(kb.hidden_state, kb.input_row_offsets, kb.batch, kb.total_rows,
                           kb.weight, vb, kb.head_elems, kb.cache_lengths, kb.layer_idx)
    assert st == stb == 0
    assert np.array_equal(out, vb.data.reshape(kb.cache.shape))
    # quantisation was exact: q * s reproduces the hidden rows
    table = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    x = workloads.bf16_bits_to_float(k.hidden_state).astype(np.float64)
    assert np.array_equal(table[q] * np.repeat(s, 128, 1), x)


def test_addressing_and_reported_rows_match_kv_matmul():
    k = workloads.make_kv_matmul("addr", 4713, [30, 0, 17], [5, 9, 120], 128, 2, 64, 16, fp8=True,
                                 num_layers=2, layer_idx=1, extra_pages=2)
    st, out, q, s = run_fp8(k)
    assert st == 0
    dest = oracle.kv_row_dest(k.input_row_offsets, k.batch, k.total_rows, k.cache_lengths,
                              kv_cache_view(k))
    _, two, P, S, E = k.cache.shape
    written = (out[1] != k.cache[1]).any(-1).reshape(2, P * S)
    expect = np.zeros(P * S, bool)
    expect[dest // E] = True
    assert np.array_equal(written[0], expect) and np.array_equal(written[1], expect)
    assert (out[0] == k.cache[0]).all()
    for r in range(k.total_rows):
        q1, s1 = oracle.quantize_row_e4m3(k.hidden_state[r], 128)
        assert np.array_equal(q[r], q1) and np.array_equal(s[r], s1)


def test_out_of_range_rows_are_skipped():
    k = workloads.make_kv_matmul("oor", 4715, [40, 70], [0, 100], 256, 2, 64, 32, fp8=True)
    k.page_table = k.page_table.copy()
    k.page_table[1, 4] = k.num_pages + 9
    st, out, q, s = run_fp8(k)
    assert st == 4
    assert (q[40 + 28:40 + 60] == 0).all()      # positions 128..159 of request 1
