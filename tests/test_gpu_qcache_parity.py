"""GPU parity of the quantised paged latent cache (e4m3 codes, bf16 rope and fp32 block
scales per slot), through the C ABI, against the CPU oracle on the same seeded inputs.

Decompress from a quantised cache: the quantised operands (codes and scales, taken from the
slots as they are) and the dequantised k_latent_buffer are compared bit for bit; k_buffer
within the FP8 tolerance (3e-2 |oracle| + 5e-3).  Cache write into a quantised cache: the
codes are an integer decision made from the bf16-rounded row, so they are checked bit for
bit against the oracle's quantisation of the row the GPU's bf16 cache write produces (itself
parity-checked against the oracle), and the set of bytes written against the oracle's."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import FP8_TOL, DeviceCacheWrite, DeviceDecompress, assert_close_bf16
from util import (e4m3_midpoint_bf16_values, oracle_cache_write_q, oracle_decompress_qcache,
                  qcache_view)

pytestmark = pytest.mark.gpu
SQ = workloads.SENTINEL_QBYTE


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_mla_gb300  # noqa: F401  (raises if the library is missing)


def check_decompress(d, expect_status=0, with_latent=True):
    g = DeviceDecompress(d, with_latent=with_latent)
    g.run()
    lat, kb, status = g.results()
    q, s = g.fp8_workspace()
    st, olat, okb, oq, os_, written = oracle_decompress_qcache(d)
    assert status == expect_status and st == expect_status
    w = written
    assert np.array_equal(q[:d.buffer_length][w], oq[w]) and np.array_equal(s[:d.buffer_length][w], os_[w])
    if with_latent:
        assert np.array_equal(lat[w], olat[w])
        assert (lat[~w] == workloads.SENTINEL_OUT).all()
    else:
        assert (lat == workloads.SENTINEL_OUT).all()
    assert (kb[~w] == workloads.SENTINEL_OUT).all()
    assert_close_bf16(kb[w], okb[w], FP8_TOL, "qcache k_buffer")
    return kb


@pytest.mark.parametrize("lengths,co,ps,R,P,n_out,pad", [
    ([37, 300, 5, 129], [0, 17, 5, 64], 16, 512, 64, 256, 0),   # DeepSeek-V3 slot, ragged
    ([260, 40], [3, 0], 128, 512, 64, 384, 16),                 # padded slots, 3 n tiles
    ([100, 7, 64], [0, 0, 1], 8, 256, 32, 128, 0),
    ([90], [11], 32, 128, 8, 256, 0),                           # smallest R
])
def test_qcache_decompress_mid(lengths, co, ps, R, P, n_out, pad):
    d = workloads.make_qcache_decompress("qmid", 900 + R + ps, lengths, co, ps, R, P, n_out,
                                         num_layers=2, layer_idx=1, extra_pages=3, slot_pad=pad)
    check_decompress(d)


def test_qcache_decompress_without_latent_buffer():
    d = workloads.make_qcache_decompress("qnolat", 911, [200, 33], [4, 0], 16, 512, 64, 256)
    kb1 = check_decompress(d, with_latent=False)
    kb2 = check_decompress(d, with_latent=True)
    assert np.array_equal(kb1, kb2)


def test_qcache_decompress_out_of_range():
    d = workloads.make_qcache_decompress("qoor", 913, [40, 70], [0, 5], 16, 256, 32, 128,
                                         extra_pages=2)
    d.page_table = d.page_table.copy()
    d.page_table[1, 2] = d.num_pages + 5           # tokens 32..47 of request 1
    check_decompress(d, expect_status=4)


def test_qcache_decompress_full_size_sampled():
    """DeepSeek-V3 FP8 decompress over a quantised cache (26 737 rows): codes and scales of
    every row against the slots they come from, k_latent and k_buffer of sampled rows
    against the oracle's row form."""
    d = workloads.WORKLOADS["deepseek_v3_fp8_qcache_decompress"]()
    g = DeviceDecompress(d)
    g.run()
    lat, kb, status = g.results()
    q, s = g.fp8_workspace()
    assert status == 0
    R, P = d.kv_lora_rank, d.rope_dim
    bro = d.buffer_row_offsets.astype(np.int64)
    slots = []
    for b in range(d.batch):
        t = np.arange(int(d.cache_offsets[b]), int(d.lengths[b]))
        pages = d.page_table[b, t // d.page_size]
        slots.append(d.cache[d.layer_idx, pages, t % d.page_size])
    slots = np.concatenate(slots)
    assert slots.shape[0] == bro[-1] == d.buffer_length
    assert np.array_equal(q[:d.buffer_length], slots[:, :R])
    assert np.array_equal(s[:d.buffer_length].view(np.uint8),
                          slots[:, R + 2 * P:R + 2 * P + 4 * (R // 128)].reshape(-1, 4 * (R // 128)))
    assert np.array_equal(lat[:, R:], slots[:, R:R + 2 * P].copy().view(np.uint16))
    rng = np.random.default_rng(5)
    for r in sorted(set(rng.integers(0, d.buffer_length, 48).tolist()) | {0, d.buffer_length - 1}):
        st, l1, k1, q1, s1 = oracle.decompress_k_qcache_fp8_row(
            qcache_view(d), d.layer_idx, d.buffer_row_offsets, d.cache_offsets, d.batch,
            d.buffer_length, R, P, d.w_k_e4m3, d.w_k_scale, r)
        assert st == 0
        assert np.array_equal(lat[r], l1)
        assert_close_bf16(kb[r], k1, FP8_TOL, f"row {r}")


def _written_slots(cache):
    return (cache != SQ).any(-1) if cache.dtype == np.uint8 else (cache != workloads.SENTINEL_CACHE).any(-1)


def check_cache_write_q(cq, cb, expect_status=0):
    """cq and cb: the same problem with a quantised and a bf16 cache."""
    gq = DeviceCacheWrite(cq)
    gq.run()
    outq, stq = gq.results()
    gb = DeviceCacheWrite(cb)
    gb.run()
    outb, stb = gb.results()
    st, refq = oracle_cache_write_q(cq)
    assert stq == st == stb == expect_status
    assert np.array_equal(outq != cq.cache, refq != cq.cache), "written bytes differ"
    R, P = cq.kv_lora_rank, cq.rope_dim
    wq = _written_slots(outq)
    assert np.array_equal(wq, _written_slots(outb))
    for idx in zip(*np.nonzero(wq)):
        q, s = oracle.quantize_row_e4m3(outb[idx], R)
        slot = outq[idx]
        assert np.array_equal(slot[:R], q), idx
        assert np.array_equal(slot[R + 2 * P:R + 2 * P + 4 * (R // 128)].view(np.float32), s), idx
        assert np.array_equal(slot[R:R + 2 * P].view(np.uint16), outb[idx][R:]), idx
    return outq, outb


@pytest.mark.parametrize("new,lens,R,P,ps", [
    ([7, 1, 300, 0, 45], [5, 0, 17, 3, 128], 512, 64, 16),
    ([64, 11, 3], [1, 2, 127], 128, 32, 32),
    ([40], [9], 1024, 256, 8),
    ([17, 9], [3, 60], 384, 0, 16),
])
def test_qcache_write_mid(new, lens, R, P, ps):
    kw = dict(num_layers=2, layer_idx=1, extra_pages=3)
    cq = workloads.make_cache_write("cwq", 800 + R + P, new, lens, R, P, ps, quantised=True, **kw)
    cb = workloads.make_cache_write("cwb", 800 + R + P, new, lens, R, P, ps, **kw)
    check_cache_write_q(cq, cb)


def test_qcache_write_out_of_range_and_padding():
    kw = dict(extra_pages=2, max_seq_len=60)
    cq = workloads.make_cache_write("cwqo", 821, [20, 33], [0, 40], 256, 32, 16, quantised=True,
                                    slot_pad=32, **kw)
    cb = workloads.make_cache_write("cwbo", 821, [20, 33], [0, 40], 256, 32, 16, **kw)
    outq, _ = check_cache_write_q(cq, cb, expect_status=4)
    assert (outq[..., workloads.qslot_payload_bytes(256, 32):] == SQ).all()


def test_qcache_write_then_decompress_matches_the_bf16_fp8_path():
    """GPU end to end: rows written into a quantised cache and decompressed give the k_buffer
    the bf16 cache write followed by the FP8 decompress gives, bit for bit (same codes and
    scales into the same product)."""
    kw = dict(num_layers=1, layer_idx=0)
    new, lens = [300, 41, 129], [0, 0, 0]
    cq = workloads.make_cache_write("e2eq", 833, new, lens, 512, 64, 16, quantised=True, **kw)
    cb = workloads.make_cache_write("e2eb", 833, new, lens, 512, 64, 16, **kw)
    gq = DeviceCacheWrite(cq)
    gq.run()
    gb = DeviceCacheWrite(cb)
    gb.run()
    outq, _ = gq.results()
    outb, _ = gb.results()
    lengths = np.array(new)
    kb = {}
    for name, cache in [("q", outq), ("b", outb)]:
        d = workloads.make_decompress("e2e", 835, lengths, [0, 0, 0], 16, 512, 64, 256, fp8=True,
                                      page_table=cq.page_table, num_pages=cq.num_pages)
        d.cache = cache
        g = DeviceDecompress(d, fp8=True)
        g.run()
        _, k, status = g.results()
        assert status == 0
        kb[name] = k
    assert np.array_equal(kb["q"], kb["b"])


def test_qcache_write_full_size():
    """DeepSeek-V3 prefill write into a quantised cache (~80k rows, 656-byte slots)."""
    cq = workloads.WORKLOADS["cache_write_q_path"]()
    cb = workloads.cache_write_path()
    gq = DeviceCacheWrite(cq)
    gq.run()
    outq, stq = gq.results()
    gb = DeviceCacheWrite(cb)
    gb.run()
    outb, stb = gb.results()
    assert stq == stb == 0
    st, refq = oracle_cache_write_q(cq)
    assert np.array_equal(outq != cq.cache, refq != cq.cache)
    R, P = 512, 64
    wq = _written_slots(outq)
    idx = np.argwhere(wq)
    rng = np.random.default_rng(9)
    for i in rng.choice(len(idx), 400, replace=False):
        k = tuple(idx[i])
        q, s = oracle.quantize_row_e4m3(outb[k], R)
        assert np.array_equal(outq[k][:R], q)
        assert np.array_equal(outq[k][R + 2 * P:R + 2 * P + 16].view(np.float32), s)
        assert np.array_equal(outq[k][R:R + 2 * P].view(np.uint16), outb[k][R:])


def test_fp8_quantisation_at_e4m3_midpoints_bit_exact():
    """Blocks whose scale is a power of two (amax = 448 * 2^k) and whose other values sit on
    e4m3 rounding midpoints (ties to even) or one bf16 step beside them, in the normal and
    subnormal e4m3 range: the GPU's codes and scales must equal the oracle's bit for bit."""
    d = workloads.make_decompress("mid", 951, [64, 64], [0, 0], 16, 512, 64, 128, fp8=True)
    vals = e4m3_midpoint_bf16_values()
    rng = np.random.default_rng(951)
    cache = d.cache.copy()
    L, Pg, S, C = cache.shape
    rows = cache.reshape(-1, C)
    for i in range(rows.shape[0]):
        for kb in range(4):
            k = int(rng.integers(-4, 3))
            blk = rng.choice(vals, 128).astype(np.float64)
            blk = workloads.bf16_bits_to_float(blk.astype(np.uint16)).astype(np.float64)
            blk *= np.where(rng.random(128) < 0.5, -1.0, 1.0) * 2.0 ** k
            blk[int(rng.integers(0, 128))] = 448.0 * 2.0 ** k
            rows[i, kb * 128:(kb + 1) * 128] = [oracle.double_to_bf16(v) for v in blk]
    d.cache = rows.reshape(cache.shape)
    g = DeviceDecompress(d, fp8=True)
    g.run()
    _, _, status = g.results()
    q, s = g.fp8_workspace()
    from util import oracle_decompress_fp8
    st, _, _, oq, os_, written = oracle_decompress_fp8(d)
    assert status == 0 and st == 0 and written.all()
    assert np.array_equal(q[:d.buffer_length], oq) and np.array_equal(s[:d.buffer_length], os_)


def test_qcache_write_at_e4m3_midpoints_bit_exact():
    """x = +-1 and epsilon = 0 make the normalised row y = +-gamma once rounded to bf16; gamma
    holds a block maximum 56 (scale 1/8) and values on e4m3 midpoints (times 1/8) or one bf16
    step beside them, so the quantisation sees ties; rotations by multiples of 90 degrees
    keep the rope exact: the quantised slots must equal the oracle's bit for bit."""
    c = workloads.make_cache_write("cwmid", 953, [70, 33], [0, 5], 512, 64, 16, quantised=True)
    rng = np.random.default_rng(953)
    vals = workloads.bf16_bits_to_float(e4m3_midpoint_bf16_values()).astype(np.float64)
    vals = vals[vals * 8 < 448] / 8
    gamma = rng.choice(vals, 512)
    gamma[::128] = 56.0
    c.gamma = gamma.astype(np.float32)
    c.epsilon = 0.0
    qt = rng.integers(0, 4, size=(c.freqs_cis.shape[0], 32))   # exact rotations for the rope
    c.freqs_cis = np.stack([np.choose(qt, [1.0, 0.0, -1.0, 0.0]), np.choose(qt, [0.0, 1.0, 0.0, -1.0])],
                           -1).reshape(c.freqs_cis.shape).astype(np.float32)
    M, C = c.latent.shape
    sign = np.where(rng.random((M, 512)) < 0.5, 0xBF80, 0x3F80).astype(np.uint16)
    c.latent = c.latent.copy()
    c.latent[:, :512] = sign
    g = DeviceCacheWrite(c)
    g.run()
    out, status = g.results()
    st, ref = oracle_cache_write_q(c)
    assert status == 0 and st == 0
    assert np.array_equal(out, ref)
