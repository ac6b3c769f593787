"""Pins of the oracle's cache-write side (RMSNorm with kv_norm_gamma, RoPE with freqs_cis,
stored into the paged latent cache at each new token's position) against what the pages
and the mathematics fix: a hand-computed worked example (tests/golden), closed forms of
the normalisation, exact rotations, scale invariance, the destination slots of the
kv_matmul position rule, and out-of-range rows.  No GPU."""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
import workloads
from util import assert_correctly_rounded_bf16, bf16_to_f64, f32_to_bf16_exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SENT = workloads.SENTINEL_CACHE


def view(c: workloads.CacheWriteInputs, data):
    ls, ps, ss = c.strides
    return oracle.PagedCacheView(data, ls, ps, ss, c.num_pages, c.page_size, c.page_table,
                                 c.page_table.shape[1])


def run(c: workloads.CacheWriteInputs):
    v = view(c, c.cache.copy())
    st = oracle.cache_write(c.latent, c.input_row_offsets, c.batch, c.total_rows, c.kv_lora_rank,
                            c.rope_dim, c.gamma, c.epsilon, c.freqs_cis, v, c.cache_lengths,
                            c.layer_idx)
    return st, v.data.reshape(c.cache.shape)


def dests(c):
    ls, ps, ss = c.strides
    return oracle.kv_row_dest(c.input_row_offsets, c.batch, c.total_rows, c.cache_lengths,
                              view(c, c.cache))


def test_cache_write_worked_example():
    with open(os.path.join(GOLDEN, "cache_write_worked_example.json")) as f:
        ex = json.load(f)
    R, P, ps = ex["kv_lora_rank"], ex["rope_dim"], ex["page_size"]
    c = workloads.CacheWriteInputs(
        name="worked", latent=f32_to_bf16_exact(np.array(ex["latent"], np.float32)),
        input_row_offsets=np.array(ex["input_row_offsets"], np.uint32),
        cache_lengths=np.array(ex["cache_lengths"], np.uint32),
        page_table=np.array(ex["page_table"], np.uint32),
        cache=np.full((ex["num_layers"], ex["num_pages"], ps, R + P), SENT, np.uint16),
        gamma=np.array(ex["gamma"], np.float32), epsilon=ex["epsilon"],
        freqs_cis=np.array(ex["freqs_cis"], np.float32), kv_lora_rank=R, rope_dim=P,
        layer_idx=ex["layer_idx"])
    st, cache = run(c)
    assert st == 0
    expect = np.full(cache.shape, SENT, np.uint16)
    for e in ex["expected_slots"]:
        expect[ex["layer_idx"], e["page"], e["slot"]] = f32_to_bf16_exact(np.array(e["values"], np.float32))
    assert np.array_equal(cache, expect)


def test_single_nonzero_normalises_to_plus_minus_sqrt_r():
    c = workloads.make_cache_write("closed", 91, [37, 5], [3, 130], 64, 16, 16)
    c.gamma = np.ones(64, np.float32)
    c.epsilon = 0.0
    lat = np.zeros((c.total_rows, 80), np.float32)
    g = np.random.default_rng(3)
    cols = g.integers(0, 64, c.total_rows)
    vals = g.choice([-3.0, -0.5, 0.25, 2.0, 7.0], c.total_rows)
    lat[np.arange(c.total_rows), cols] = vals
    lat[:, 64:] = 1.0
    c.latent = f32_to_bf16_exact(lat)
    st, cache = run(c)
    d = dests(c)
    flat = cache[c.layer_idx].reshape(-1)
    for r in range(c.total_rows):
        row = bf16_to_f64(flat[d[r]: d[r] + 64])
        want = np.zeros(64)
        want[cols[r]] = 8.0 * np.sign(vals[r])  # x / sqrt(x^2 / 64) = +-8
        assert np.array_equal(row, want)


def test_rotations_identity_and_quarter_turn_are_exact_and_norm_preserved():
    c = workloads.make_cache_write("rot", 92, [20, 33], [0, 7], 64, 32, 8, max_seq_len=64)
    x = bf16_to_f64(c.latent[:, 64:])
    d = dests(c)
    for mode in ("identity", "quarter", "random"):
        if mode == "identity":
            c.freqs_cis = np.tile(np.array([1.0, 0.0], np.float32), (64, 16))
        elif mode == "quarter":
            c.freqs_cis = np.tile(np.array([0.0, 1.0], np.float32), (64, 16))
        st, cache = run(c)
        flat = cache[c.layer_idx].reshape(-1)
        rope = np.stack([flat[d[r] + 64: d[r] + 96] for r in range(c.total_rows)])
        if mode == "identity":
            assert np.array_equal(rope, c.latent[:, 64:])
        elif mode == "quarter":
            want = np.empty_like(x)
            want[:, 0::2], want[:, 1::2] = -x[:, 1::2], x[:, 0::2]
            assert np.array_equal(bf16_to_f64(rope), want)
        else:
            got = bf16_to_f64(rope)
            pair_in = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
            pair_out = got[:, 0::2] ** 2 + got[:, 1::2] ** 2
            assert np.allclose(pair_out, pair_in, rtol=2e-2, atol=1e-6)
            # against numpy's complex multiply with the positions of the rows
            pos = np.concatenate([np.arange(c.cache_lengths[b], c.cache_lengths[b] + n)
                                  for b, n in enumerate(np.diff(c.input_row_offsets))])
            f = c.freqs_cis[pos].astype(np.float64)
            z = (x[:, 0::2] + 1j * x[:, 1::2]) * (f[:, 0::2] + 1j * f[:, 1::2])
            exact = np.empty_like(x)
            exact[:, 0::2], exact[:, 1::2] = z.real, z.imag
            assert_correctly_rounded_bf16(rope, exact)


def test_normalisation_matches_numpy_and_is_scale_invariant():
    c = workloads.make_cache_write("norm", 93, [50, 1, 17], [5, 0, 300], 128, 64, 32, epsilon=0.0)
    st, cache = run(c)
    d = dests(c)
    x = bf16_to_f64(c.latent[:, :128])
    exact = x / np.sqrt((x * x).mean(axis=1, keepdims=True)) * c.gamma.astype(np.float64)
    flat = cache[c.layer_idx].reshape(-1)
    got = np.stack([flat[d[r]: d[r] + 128] for r in range(c.total_rows)])
    assert_correctly_rounded_bf16(got, exact)
    c2 = workloads.CacheWriteInputs(**{**c.__dict__})
    c2.latent = c.latent.copy()
    c2.latent[:, :128] = f32_to_bf16_exact(bf16_to_f64(c.latent[:, :128]).astype(np.float32) * 4.0)
    st2, cache2 = run(c2)
    got2 = np.stack([cache2[c.layer_idx].reshape(-1)[d[r]: d[r] + 128] for r in range(c.total_rows)])
    assert np.array_equal(got, got2)


def test_writes_exactly_the_kv_matmul_slots_and_skips_out_of_range_rows():
    c = workloads.make_cache_write("slots", 94, [9, 0, 40, 3], [2, 5, 120, 0], 64, 16, 16,
                                   num_layers=3, layer_idx=2, extra_pages=2)
    st, cache = run(c)
    assert st == 0
    d = dests(c)
    changed = np.argwhere((cache != SENT).any(axis=-1))
    got = sorted((int(l), int(p), int(s)) for l, p, s in changed)
    ls, ps, ss = c.strides
    want = sorted((c.layer_idx, int(off) // ps, (int(off) % ps) // ss) for off in d)
    assert got == want
    # a row past max_seq_len and a row on a page id past the cache: status 4, nothing written
    c.freqs_cis = c.freqs_cis[:int(c.cache_lengths[2]) + 40 - 1]
    c.page_table = c.page_table.copy()
    c.page_table[0, 0] = c.num_pages + 7
    st, cache3 = run(c)
    assert st == 4
    written = int((cache3 != SENT).any(axis=-1).sum())
    # request 0's 9 rows (positions 2..10) all sit on its first page; 1 row past max_seq_len
    assert written == c.total_rows - 9 - 1
