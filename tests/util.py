"""Helpers shared by the tests: views of workload arrays for the oracle, bf16 bit tricks,
and the rounding-error bound used to pin the oracle against library products."""
from __future__ import annotations

import numpy as np

import oracle
from workloads import CacheWriteInputs, DecompressInputs, KvMatmulInputs, bf16_bits_to_float


def f32_to_bf16_exact(a) -> np.ndarray:
    """float values that are exactly representable in bf16 -> uint16 bit patterns."""
    a = np.asarray(a, np.float32)
    bits = a.view(np.uint32)
    assert not np.any(bits & 0xFFFF), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


def bf16_to_f64(a) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_half_ulp(exact: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |exact| (8 significant bits, subnormal quantum
    2^-133)."""
    a = np.abs(exact)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = np.exp2(np.maximum(e - 7, -133))
    return 0.5 * np.where(a > 0, q, 2.0 ** -133)


def assert_correctly_rounded_bf16(out_bits, exact, rel_slack=1e-9):
    """out_bits must be a round-to-nearest bf16 of `exact` (fp64), up to rel_slack of the
    exact value for the summation-order noise of the fp64 reference."""
    y = bf16_to_f64(out_bits)
    err = np.abs(y - exact)
    bound = bf16_half_ulp(exact) * (1 + 1e-12) + rel_slack * np.abs(exact) + 1e-300
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} elements not correctly rounded; first at "
                           f"{np.argwhere(bad)[0]}: got {y[bad][0]}, exact {exact[bad][0]}")


def cache_view(d: DecompressInputs) -> oracle.PagedCacheView:
    ls, ps, ss = d.strides
    return oracle.PagedCacheView(d.cache, ls, ps, ss, d.num_pages, d.page_size, d.page_table,
                                 d.page_table.shape[1])


def kv_cache_view(k: KvMatmulInputs, data=None) -> oracle.PagedCacheView:
    ls, ps, ss, kvs = k.strides
    return oracle.PagedCacheView(k.cache if data is None else data, ls, ps, ss, k.num_pages,
                                 k.page_size, k.page_table, k.page_table.shape[1], kv_stride=kvs)


def oracle_decompress(d: DecompressInputs, k_latent=None, k_buffer=None):
    return oracle.decompress_k(cache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets,
                               d.batch, d.buffer_length, d.kv_lora_rank, d.rope_dim, d.w_k,
                               k_latent=k_latent, k_buffer=k_buffer)


def oracle_decompress_fp8(d: DecompressInputs, k_latent=None, k_buffer=None):
    return oracle.decompress_k_fp8(cache_view(d), d.layer_idx, d.buffer_row_offsets,
                                   d.cache_offsets, d.batch, d.buffer_length, d.kv_lora_rank,
                                   d.rope_dim, d.w_k_e4m3, d.w_k_scale, k_latent=k_latent,
                                   k_buffer=k_buffer)


def oracle_kv_matmul(k: KvMatmulInputs):
    """Runs the oracle on a copy of the cache; returns (status, cache_after)."""
    view = kv_cache_view(k, data=k.cache.copy())
    st = oracle.kv_matmul(k.hidden_state, k.input_row_offsets, k.batch, k.total_rows, k.weight,
                          view, k.head_elems, k.cache_lengths, k.layer_idx)
    return st, view.data.reshape(k.cache.shape)


def oracle_cache_write(c: CacheWriteInputs):
    """Runs the cache-write oracle on a copy of the cache; returns (status, cache_after)."""
    ls, ps, ss = c.strides
    view = oracle.PagedCacheView(c.cache.copy(), ls, ps, ss, c.num_pages, c.page_size,
                                 c.page_table, c.page_table.shape[1])
    st = oracle.cache_write(c.latent, c.input_row_offsets, c.batch, c.total_rows, c.kv_lora_rank,
                            c.rope_dim, c.gamma, c.epsilon, c.freqs_cis, view, c.cache_lengths,
                            c.layer_idx)
    return st, view.data.reshape(c.cache.shape)


def qcache_view(d, data=None) -> oracle.QuantCacheView:
    """Oracle view of a quantised cache (DecompressInputs or CacheWriteInputs)."""
    ls, ps, ss = d.strides
    return oracle.QuantCacheView(d.cache if data is None else data, ls, ps, ss, d.num_pages,
                                 d.page_size, d.page_table, d.page_table.shape[1])


def oracle_decompress_qcache(d: DecompressInputs):
    return oracle.decompress_k_qcache_fp8(qcache_view(d), d.layer_idx, d.buffer_row_offsets,
                                          d.cache_offsets, d.batch, d.buffer_length,
                                          d.kv_lora_rank, d.rope_dim, d.w_k_e4m3, d.w_k_scale)


def oracle_cache_write_q(c: CacheWriteInputs):
    """Runs the quantised cache-write oracle on a copy of the cache; returns (status,
    cache_after)."""
    view = qcache_view(c, c.cache.copy())
    st = oracle.cache_write_q(c.latent, c.input_row_offsets, c.batch, c.total_rows,
                              c.kv_lora_rank, c.rope_dim, c.gamma, c.epsilon, c.freqs_cis, view,
                              c.cache_lengths, c.layer_idx)
    return st, view.data.reshape(c.cache.shape)


def oracle_kv_matmul_fp8(k: KvMatmulInputs):
    """Runs the FP8 kv_matmul oracle on a copy of the cache; returns (status, cache_after,
    q, s)."""
    view = kv_cache_view(k, data=k.cache.copy())
    st, q, s = oracle.kv_matmul_fp8(k.hidden_state, k.input_row_offsets, k.batch, k.total_rows,
                                    k.w_e4m3, k.w_scale, view, k.head_elems, k.cache_lengths,
                                    k.layer_idx)
    return st, view.data.reshape(k.cache.shape), q, s


def e4m3_decode_table() -> np.ndarray:
    return np.array([oracle.e4m3_to_double(c) for c in range(256)], np.float64)


def e4m3_midpoint_bf16_values():
    """e4m3 rounding midpoints (normal and subnormal range) and their bf16 neighbours, as
    multiples of the block scale."""
    mids = [(1 + (2 * j + 1) / 16) * 2.0 ** e for e in range(-6, 9) for j in range(8)
            if (1 + (2 * j + 1) / 16) * 2.0 ** e < 448]
    mids += [(2 * i + 1) * 2.0 ** -10 for i in range(7)]
    bits = [bf16_bits_to_float(np.array([oracle.double_to_bf16(m)], np.uint16))[0]
            for m in mids]
    assert all(float(b) == m for b, m in zip(bits, mids))
    out = []
    for m in mids:
        h = oracle.double_to_bf16(m)
        out += [h, h + 1, h - 1]          # the midpoint and one bf16 step either side
    return np.array(out, np.uint16)
