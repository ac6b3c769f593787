"""Pins of the oracle's quantised paged latent cache (e4m3 codes, bf16 rope and fp32 block
scales per slot; written by the cache-write side, read by the FP8 decompress) against what
the pages and the mathematics fix: a hand-derived worked example (tests/golden), the
equivalence with quantising the bf16 cache row (so a quantised cache feeds the
block-scaled product the very operands the FP8 decompress makes), the e4m3 rounding bound
of the dequantised values, the fp32 dequantisation against numpy, and the slot layout
(padding, untouched slots, out-of-range rows).  No GPU."""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SQ = workloads.SENTINEL_QBYTE


def qview(c, data=None):
    ls, ps, ss = c.strides
    return oracle.QuantCacheView(c.cache.copy() if data is None else data, ls, ps, ss,
                                 c.num_pages, c.page_size, c.page_table, c.page_table.shape[1])


def bview(c, data):
    ls, ps, ss = c.strides
    return oracle.PagedCacheView(data, ls, ps, ss, c.num_pages, c.page_size, c.page_table,
                                 c.page_table.shape[1])


def write_q(c):
    v = qview(c)
    st = oracle.cache_write_q(c.latent, c.input_row_offsets, c.batch, c.total_rows, c.kv_lora_rank,
                              c.rope_dim, c.gamma, c.epsilon, c.freqs_cis, v, c.cache_lengths,
                              c.layer_idx)
    return st, v.data.reshape(c.cache.shape)


def bf16(x):
    return int(oracle.double_to_bf16(float(x)))


def test_qcache_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "qcache_worked_example.json")))
    R, P, S = g["kv_lora_rank"], g["rope_dim"], g["slot_bytes"]
    k = np.arange(R)
    nope = [np.where(k < 65, 1.0, -1.0), np.where(k % 2 == 0, 2.0, -2.0)]
    latent = np.zeros((2, R + P), np.uint16)
    for r in range(2):
        latent[r, :R] = [bf16(v) for v in nope[r]]
        latent[r, R:] = [bf16(v) for v in g["latent_rope"][r]]
    cache = np.full((1, g["num_pages"], g["page_size"], S), SQ, np.uint8)
    c = workloads.CacheWriteInputs(
        name="golden", latent=latent, input_row_offsets=np.array(g["input_row_offsets"], np.uint32),
        cache_lengths=np.array(g["cache_lengths"], np.uint32),
        page_table=np.array(g["page_table"], np.uint32), cache=cache,
        gamma=np.ones(R, np.float32), epsilon=g["epsilon"],
        freqs_cis=np.array(g["freqs_cis"], np.float32), kv_lora_rank=R, rope_dim=P, layer_idx=0)
    st, out = write_q(c)
    assert st == 0
    flat = out.reshape(-1)
    s = np.float32(1.0) / np.float32(448.0)
    codes = [np.where(k < 65, 0x7E, 0xFE), np.where(k % 2 == 0, 0x7E, 0xFE)]
    touched = np.zeros(flat.size, bool)
    for r, off in enumerate(g["expected_slot_offsets"]):
        slot = flat[off:off + S]
        assert np.array_equal(slot[:R], codes[r])
        rope = slot[R:R + 2 * P].view(np.uint16)
        assert [f"0x{v:04X}" for v in rope] == g["expected_rope_bf16"][r]
        assert slot[R + 2 * P:R + 2 * P + 4].view(np.float32)[0] == s
        touched[off:off + R + 2 * P + 4] = True
    assert (flat[~touched] == SQ).all()          # nothing else in the cache changed

    dc = g["decompress"]
    d = workloads.DecompressInputs(
        name="golden", cache=out, page_table=c.page_table,
        buffer_row_offsets=np.array(dc["buffer_row_offsets"], np.uint32),
        cache_offsets=np.array(dc["cache_offsets"] + [0], np.uint32),
        buffer_length=dc["buffer_length"], kv_lora_rank=R, rope_dim=P, n_out=dc["n_out"],
        layer_idx=0)
    w = np.full((dc["n_out"], R), int(dc["w_k_code"], 16), np.uint8)
    ws = np.full((dc["n_out"] // 128, R // 128), dc["w_k_scale"], np.float32)
    st, lat, kb, q, qs, written = oracle.decompress_k_qcache_fp8(
        qview(d, out.copy()), 0, d.buffer_row_offsets, d.cache_offsets, d.batch, d.buffer_length,
        R, P, w, ws)
    assert st == 0 and written.all()
    assert [f"0x{v:04X}" for v in kb[:, 0]] == g["expected_k_buffer_bf16"]
    assert (kb == kb[:, :1]).all()
    assert np.array_equal(q[0], codes[0]) and np.array_equal(q[1], codes[1])
    assert (qs == s).all()
    assert np.array_equal(lat[0, :R], np.where(k < 65, 0x3F80, 0xBF80))
    assert np.array_equal(lat[1, :R], np.where(k % 2 == 0, 0x3F80, 0xBF80))
    assert [f"0x{v:04X}" for v in lat[0, R:]] == g["expected_rope_bf16"][0]


def test_quantised_cache_holds_the_fp8_path_operands():
    """Writing the same rows into a bf16 cache and into a quantised one: every quantised slot
    holds the codes and scales the FP8 decompress's quantisation makes of the bf16 slot and
    the same rope bits, and decompressing both gives bit-identical k_buffer, codes and
    scales."""
    kw = dict(num_layers=2, layer_idx=1, extra_pages=2)
    new, lens = [37, 5, 90], [3, 70, 0]
    cb = workloads.make_cache_write("eqb", 4242, new, lens, 256, 32, 16, **kw)
    cq = workloads.make_cache_write("eqq", 4242, new, lens, 256, 32, 16, quantised=True, **kw)
    assert np.array_equal(cb.latent, cq.latent) and np.array_equal(cb.page_table, cq.page_table)
    vb = bview(cb, cb.cache.copy())
    assert oracle.cache_write(cb.latent, cb.input_row_offsets, cb.batch, cb.total_rows, 256, 32,
                              cb.gamma, cb.epsilon, cb.freqs_cis, vb, cb.cache_lengths, 1) == 0
    bcache = vb.data.reshape(cb.cache.shape)
    st, qcache = write_q(cq)
    assert st == 0
    R, P = 256, 32
    written = (bcache[1] != workloads.SENTINEL_CACHE).any(-1)
    assert np.array_equal(written, (qcache[1] != SQ).any(-1))
    for page, slot in zip(*np.nonzero(written)):
        q, s = oracle.quantize_row_e4m3(bcache[1, page, slot], R)
        qs = qcache[1, page, slot]
        assert np.array_equal(qs[:R], q)
        assert np.array_equal(qs[R:R + 2 * P].view(np.uint16), bcache[1, page, slot, R:])
        assert np.array_equal(qs[R + 2 * P:R + 2 * P + 4 * (R // 128)].view(np.float32), s)
    # decompress every written token of every request from both caches
    iro = cq.input_row_offsets.astype(np.int64)
    lengths = [int(lens[b] + new[b]) for b in range(3)]
    bro = np.concatenate([[0], np.cumsum(lengths)]).astype(np.uint32)
    co = np.zeros(4, np.uint32)
    g = workloads._gen(77)
    import torch
    w = torch.randn(256, R, generator=g) / 16
    we, wsc = workloads.quantize_weight_e4m3(w)
    sb = oracle.decompress_k_fp8(bview(cb, bcache.copy()), 1, bro, co, 3, int(bro[-1]), R, P, we, wsc)
    sq = oracle.decompress_k_qcache_fp8(qview(cq, qcache.copy()), 1, bro, co, 3, int(bro[-1]), R, P,
                                        we, wsc)
    # tokens before cache_lengths were never written: both report them as sentinel data only
    # through the same slots, so compare rows whose token was written
    tok_written = np.concatenate([np.arange(lengths[b]) >= lens[b] for b in range(3)])
    assert sb[0] == sq[0] == 0
    for a, b in [(sb[2], sq[2]), (sb[3], sq[3]), (sb[4], sq[4])]:
        assert np.array_equal(a[tok_written], b[tok_written])
    assert iro[-1] == tok_written.sum()


def test_dequantised_latent_within_the_e4m3_bound():
    c = workloads.make_cache_write("bnd", 99, [300], [7], 512, 64, 32, quantised=True)
    cb = workloads.make_cache_write("bnd", 99, [300], [7], 512, 64, 32)
    st, qcache = write_q(c)
    vb = bview(cb, cb.cache.copy())
    oracle.cache_write(cb.latent, cb.input_row_offsets, 1, 300, 512, 64, cb.gamma, cb.epsilon,
                       cb.freqs_cis, vb, cb.cache_lengths, 0)
    bcache = vb.data.reshape(cb.cache.shape)
    bro = np.array([0, 300], np.uint32)
    co = np.array([7, 0], np.uint32)
    we = np.full((128, 512), 0x38, np.uint8)
    ws = np.ones((1, 4), np.float32)
    st, lat, kb, q, qs, written = oracle.decompress_k_qcache_fp8(qview(c, qcache), 0, bro, co, 1,
                                                                 300, 512, 64, we, ws)
    assert st == 0 and written.all()
    st, ref, _ = oracle.gather_latent(bview(cb, bcache), 0, bro, co, 1, 300, 576)
    y = workloads.bf16_bits_to_float(ref[:, :512]).astype(np.float64)
    x = workloads.bf16_bits_to_float(lat[:, :512]).astype(np.float64)
    s = np.repeat(qs, 128, axis=1).astype(np.float64)
    # e4m3 keeps 4 significant bits (relative error <= 2^-4) down to 2^-6, then steps of
    # 2^-9; the bf16 rounding of the dequantised value adds 2^-8 relative
    assert (np.abs(x - y) <= (2.0 ** -4 + 2.0 ** -8) * np.abs(y) + s * 2.0 ** -10 + 1e-30).all()
    assert np.array_equal(lat[:, 512:], ref[:, 512:])      # rope bits unchanged


def test_dequantisation_is_one_fp32_product_rounded_to_bf16():
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    for scale in [np.float32(1) / np.float32(448), np.float32(0.0123), np.float32(3.75e-5),
                  np.float32(1.0), np.float32(2.0) ** -20]:
        for code in codes:
            p = np.float32(oracle.e4m3_to_double(code)) * scale      # numpy fp32 multiply
            assert oracle.dequant_bf16(code, scale) == oracle.double_to_bf16(float(p))


def test_slot_padding_untouched_slots_and_out_of_range_rows():
    c = workloads.make_cache_write("pad", 5150, [20, 33], [0, 40], 128, 16, 16, quantised=True,
                                   slot_pad=32, extra_pages=2, max_seq_len=60)
    payload = workloads.qslot_payload_bytes(128, 16)
    st, out = write_q(c)
    assert st == 4                                   # request 1 runs past max_seq_len
    written = (out != SQ).any(-1)
    assert (out[..., payload:] == SQ).all()          # padding after the payload never written
    # exactly request 0's 20 positions and request 1's positions 40..59 were written
    assert written.sum() == 20 + 20
    d = workloads.make_qcache_decompress("pad", 61, [9, 30], [0, 4], 16, 128, 16, 128, slot_pad=32,
                                         extra_pages=1)
    d.page_table = d.page_table.copy()
    d.page_table[1, 1] = d.num_pages + 3             # tokens 16..29 of request 1
    st, lat, kb, q, qs, wr = oracle.decompress_k_qcache_fp8(
        qview(d), 0, d.buffer_row_offsets, d.cache_offsets, d.batch, d.buffer_length, 128, 16,
        d.w_k_e4m3, d.w_k_scale)
    assert st == 4 and wr.sum() == 9 + 12


def test_row_form_matches_full_form():
    d = workloads.make_qcache_decompress("rows", 71, [50, 19], [5, 0], 16, 256, 32, 256,
                                         num_layers=2, layer_idx=1)
    st, lat, kb, q, qs, wr = oracle.decompress_k_qcache_fp8(
        qview(d), 1, d.buffer_row_offsets, d.cache_offsets, d.batch, d.buffer_length, 256, 32,
        d.w_k_e4m3, d.w_k_scale)
    assert st == 0 and wr.all()
    for r in [0, 7, 44, 45, 63]:
        st, l1, k1, q1, s1 = oracle.decompress_k_qcache_fp8_row(
            qview(d), 1, d.buffer_row_offsets, d.cache_offsets, d.batch, d.buffer_length, 256, 32,
            d.w_k_e4m3, d.w_k_scale, r)
        assert st == 0
        assert np.array_equal(l1, lat[r]) and np.array_equal(k1, kb[r])
        assert np.array_equal(q1, q[r]) and np.array_equal(s1, qs[r])
