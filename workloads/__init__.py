"""Seeded synthetic inputs for the paged-KV MLA hot path.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic (no gather, no product, no rounding of results).  Both the CUDA path's tests /
benchmark and the CPU oracle consume the arrays it returns, so the two sides always see
the same bytes.

bf16 tensors are returned as uint16 bit patterns, e4m3 tensors as uint8 codes, metadata
as uint32, scales as float32.  All generation uses a torch CPU ``Generator`` seeded per
workload, so every array is reproducible on any host.

Workload shapes (the MLA decompress of DeepSeek-V3-shaped latent caches and the
kv_matmul write path):
  * tiny decompress: 2 requests (5 and 11 cached tokens), page_size 4, 8 pages assigned by a
    seeded permutation, kv_lora_rank 64 + rope 16, W_k [64, 64].
  * DeepSeek-V3-shaped decompress: 16 requests, lengths ~U[512, 4096], cache_offsets
    ~U[0, len/4] with the copied range running to the end of the history, page_size 128,
    shuffled pages, kv_lora_rank 512 + rope 64, W_k [16384, 512] ~N(0, 1/sqrt(512)).
  * the same shapes with an e4m3 W_k and fp32 scales per 128x128 block.
  * long-context decompress: 4 requests x 32768 tokens, 1024 shuffled pages.
  * kv_matmul: 32 requests, new tokens ~U[1, 512], cache lengths ~U[0, 2048],
    hidden_state [sum(new), 4096] ~N(0,1), weight [4096, 2048] ~N(0, 1/64), K/V planes of
    8 kv heads x 128, page_size 128, cache pre-filled with sentinels.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

PAGE_TABLE_PAD = 0xFFFFFFFF  # unused page-table entries (never read by a correct walk)
SENTINEL_K = 0x7FA1          # bf16 NaN patterns no finite product can produce
SENTINEL_V = 0x7FA2
SENTINEL_OUT = 0x7FA3
SENTINEL_CACHE = 0x7FA4      # latent-cache slots a cache write must leave alone


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, std: float, g: torch.Generator) -> np.ndarray:
    """N(0, std^2) samples rounded to bf16 by torch, returned as uint16 bit patterns."""
    t = torch.randn(*shape, generator=g, dtype=torch.float32) * float(std)
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_small_ints(shape, lo: int, hi: int, g: torch.Generator) -> np.ndarray:
    """Integers in [lo, hi] stored as bf16 bit patterns (exact)."""
    t = torch.randint(lo, hi + 1, shape, generator=g).to(torch.float32)
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_float(a: np.ndarray) -> np.ndarray:
    """Widen uint16 bf16 patterns to float32 (a bit shift; exact)."""
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantize_weight_e4m3(w: torch.Tensor, block: int = 128):
    """Input preparation for the FP8 workloads: per 128x128 block of an fp32 weight,
    scale = amax / 448 (1 for an all-zero block) and codes = torch's float8_e4m3fn cast of
    w / scale.  The kernel under test receives these codes and scales as given."""
    n, k = w.shape
    wb = w.reshape(n // block, block, k // block, block)
    amax = wb.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (wb / scale[:, None, :, None]).reshape(n, k).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy().copy(), scale.to(torch.float32).numpy().copy()


SENTINEL_QBYTE = 0xA5   # unused bytes of a quantised slot, and untouched quantised slots


def qslot_payload_bytes(kv_lora_rank: int, rope_dim: int) -> int:
    """Bytes a quantised slot holds: R e4m3 codes, P bf16 rope values, R/128 fp32 scales."""
    return kv_lora_rank + 2 * rope_dim + 4 * (kv_lora_rank // 128)


def quantized_latent_slots(shape, kv_lora_rank, rope_dim, slot_bytes, g):
    """Input preparation for a quantised latent cache of `shape` (layers, pages, page_size)
    slots: nope values ~N(0, 1) drawn in fp32, per 128-column block scale = amax / 448 and
    codes = torch's float8_e4m3fn cast of x / scale (as the FP8 weights are prepared), rope
    ~N(0, 1) bf16; bytes past the payload hold SENTINEL_QBYTE."""
    R, P = kv_lora_rank, rope_dim
    x = torch.randn(*shape, R // 128, 128, generator=g, dtype=torch.float32)
    amax = x.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (x / scale[..., None]).reshape(*shape, R).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    rope = bf16_normal((*shape, P), 1.0, g)
    out = np.full((*shape, slot_bytes), SENTINEL_QBYTE, np.uint8)
    out[..., :R] = codes
    out[..., R:R + 2 * P] = rope.view(np.uint8).reshape(*shape, 2 * P)
    out[..., R + 2 * P:R + 2 * P + 4 * (R // 128)] = (
        scale.to(torch.float32).numpy().view(np.uint8).reshape(*shape, 4 * (R // 128)))
    return out


@dataclass
class DecompressInputs:
    """One decompress problem.  cache is [num_layers, num_pages, page_size, slot_elems]."""
    name: str
    cache: np.ndarray
    page_table: np.ndarray          # uint32 [batch, max_pages_per_seq]
    buffer_row_offsets: np.ndarray  # uint32 [batch + 1]
    cache_offsets: np.ndarray       # uint32 [batch + 1] (last entry unused)
    buffer_length: int
    kv_lora_rank: int
    rope_dim: int
    n_out: int
    layer_idx: int
    w_k: Optional[np.ndarray] = None        # uint16 bf16 [n_out, kv_lora_rank]
    w_k_e4m3: Optional[np.ndarray] = None   # uint8 [n_out, kv_lora_rank]
    w_k_scale: Optional[np.ndarray] = None  # float32 [n_out/128, kv_lora_rank/128]
    w_uv: Optional[np.ndarray] = None       # uint16 bf16 [num_heads, v_head_dim, kv_lora_rank]
    w_uv_e4m3: Optional[np.ndarray] = None  # uint8 [num_heads, v_head_dim, kv_lora_rank]
    w_uv_scale: Optional[np.ndarray] = None  # float32 [num_heads*v_head_dim/128, kv_lora_rank/128]
    lengths: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def quantised(self) -> bool:
        """cache holds quantised slots (uint8 bytes; strides then count bytes)."""
        return self.cache.dtype == np.uint8

    @property
    def batch(self) -> int:
        return int(self.page_table.shape[0])

    @property
    def latent_cols(self) -> int:
        return self.kv_lora_rank + self.rope_dim

    @property
    def num_layers(self) -> int:
        return int(self.cache.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.cache.shape[1])

    @property
    def page_size(self) -> int:
        return int(self.cache.shape[2])

    @property
    def slot_elems(self) -> int:
        return int(self.cache.shape[3])

    @property
    def strides(self):
        """(layer_stride, page_stride, slot_stride) in elements of `cache` (bytes for a
        quantised cache)."""
        _, P, S, E = self.cache.shape
        return P * S * E, S * E, E

    @property
    def flops(self) -> int:
        """K up-projection, plus the V one when the problem carries a w_uv."""
        rows = min(int(self.buffer_row_offsets[-1]), self.buffer_length)
        return 2 * rows * self.kv_lora_rank * (self.n_out + self.n_out_v)

    @property
    def n_out_v(self) -> int:
        wv = self.w_uv if self.w_uv is not None else self.w_uv_e4m3
        return 0 if wv is None else int(wv.shape[0] * wv.shape[1])


def _assign_pages(pages_needed, total_pages, g):
    perm = torch.randperm(total_pages, generator=g).numpy().astype(np.uint32)
    maxp = max(1, max(pages_needed) if len(pages_needed) else 1)
    pt = np.full((len(pages_needed), maxp), PAGE_TABLE_PAD, np.uint32)
    nxt = 0
    for b, n in enumerate(pages_needed):
        pt[b, :n] = perm[nxt:nxt + n]
        nxt += n
    return pt


def make_decompress(name, seed, lengths, cache_offsets, page_size, kv_lora_rank, rope_dim, n_out,
                    num_layers=1, layer_idx=0, extra_pages=0, w_std=None, fp8=False,
                    int_values=False, slot_pad=0, page_table=None, num_pages=None,
                    buffer_length=None) -> DecompressInputs:
    """General seeded decompress problem.  Request b copies cache tokens
    [cache_offsets[b], lengths[b]) into rows [bro[b], bro[b+1]) of the ragged buffer."""
    g = _gen(seed)
    lengths = np.asarray(lengths, np.int64)
    co = np.asarray(cache_offsets, np.int64)
    B = len(lengths)
    rows = lengths - co
    assert (rows >= 0).all()
    bro = np.zeros(B + 1, np.uint32)
    bro[1:] = np.cumsum(rows)
    C = kv_lora_rank + rope_dim
    pages_needed = [int(math.ceil(l / page_size)) for l in lengths]
    if page_table is None:
        total_pages = sum(pages_needed) + extra_pages
        pt = _assign_pages(pages_needed, total_pages, g)
    else:
        pt = np.asarray(page_table, np.uint32)
        total_pages = int(num_pages)
    slot_elems = C + slot_pad
    shape = (num_layers, total_pages, page_size, slot_elems)
    if int_values:
        cache = bf16_small_ints(shape, -8, 8, g)
    else:
        cache = bf16_normal(shape, 1.0, g)
    L = int(bro[-1]) if buffer_length is None else int(buffer_length)
    d = DecompressInputs(name=name, cache=cache, page_table=pt, buffer_row_offsets=bro,
                         cache_offsets=np.concatenate([co, [0]]).astype(np.uint32), buffer_length=L,
                         kv_lora_rank=kv_lora_rank, rope_dim=rope_dim, n_out=n_out,
                         layer_idx=layer_idx, lengths=lengths)
    std = w_std if w_std is not None else 1.0 / math.sqrt(kv_lora_rank)
    if fp8:
        w = torch.randn(n_out, kv_lora_rank, generator=g, dtype=torch.float32) * std
        d.w_k_e4m3, d.w_k_scale = quantize_weight_e4m3(w)
    elif int_values:
        d.w_k = bf16_small_ints((n_out, kv_lora_rank), -2, 2, g)
    else:
        d.w_k = bf16_normal((n_out, kv_lora_rank), std, g)
    return d


def make_qcache_decompress(name, seed, lengths, cache_offsets, page_size, kv_lora_rank, rope_dim,
                           n_out, num_layers=1, layer_idx=0, extra_pages=0, slot_pad=0,
                           page_table=None, num_pages=None, buffer_length=None) -> DecompressInputs:
    """The FP8 decompress problem of make_decompress (same rows, pages and e4m3 weight) over
    a quantised latent cache: slots of qslot_payload_bytes rounded up to 16 (+ slot_pad)
    bytes from quantized_latent_slots, drawn from their own generator (seed + 7919)."""
    d = make_decompress(name, seed, lengths, cache_offsets, page_size, kv_lora_rank, rope_dim,
                        n_out, num_layers=num_layers, layer_idx=layer_idx,
                        extra_pages=extra_pages, fp8=True, page_table=page_table,
                        num_pages=num_pages, buffer_length=buffer_length)
    slot_bytes = (qslot_payload_bytes(kv_lora_rank, rope_dim) + 15) // 16 * 16 + slot_pad
    d.cache = quantized_latent_slots(d.cache.shape[:3], kv_lora_rank, rope_dim, slot_bytes,
                                     _gen(seed + 7919))
    return d


def add_v_weight(d: DecompressInputs, num_heads, v_head_dim, seed, w_std=None, fp8=False,
                 int_values=False) -> DecompressInputs:
    """Adds a w_uv [num_heads, v_head_dim, kv_lora_rank] drawn from its own seeded generator
    (bf16 ~N(0, std^2), or e4m3 codes + 128x128 block scales quantised like W_k, or small
    integers), so the rest of the problem is the same as without it."""
    g = _gen(seed)
    R = d.kv_lora_rank
    std = w_std if w_std is not None else 1.0 / math.sqrt(R)
    if fp8:
        w = torch.randn(num_heads * v_head_dim, R, generator=g, dtype=torch.float32) * std
        q, sc = quantize_weight_e4m3(w)
        d.w_uv_e4m3 = q.reshape(num_heads, v_head_dim, R)
        d.w_uv_scale = sc
    elif int_values:
        d.w_uv = bf16_small_ints((num_heads, v_head_dim, R), -2, 2, g)
    else:
        d.w_uv = bf16_normal((num_heads, v_head_dim, R), std, g)
    return d


def deepseek_decompress_kv(seed=1001, fp8=False) -> DecompressInputs:
    """The DeepSeek-V3-shaped decompress with the V up-projection as well: w_uv [128 heads,
    v_head_dim 128, 512] ~N(0, 1/512) (bf16, or e4m3 with 128x128 block scales), seed 1006."""
    d = deepseek_decompress(seed, fp8=fp8)
    d.name = d.name + "_kv"
    return add_v_weight(d, 128, 128, 1006, fp8=fp8)


def tiny_decompress(seed=1000) -> DecompressInputs:
    """2 requests of 5 and 11 cached tokens, cache_offsets 0, page_size 4, 8 pages given by a
    seeded permutation reshaped to the [2, 4] page table, latent 64 + 16, W_k [64, 64]."""
    g = _gen(seed)
    pt = torch.randperm(8, generator=g).numpy().astype(np.uint32).reshape(2, 4)
    return make_decompress("tiny_decompress", seed + 1, [5, 11], [0, 0], 4, 64, 16, 64,
                           w_std=1.0 / math.sqrt(64), page_table=pt, num_pages=8)


def deepseek_lengths(seed, batch=16, lo=512, hi=4096):
    g = _gen(seed)
    lengths = torch.randint(lo, hi + 1, (batch,), generator=g).numpy().astype(np.int64)
    co = np.array([int(torch.randint(0, l // 4 + 1, (1,), generator=g)) for l in lengths], np.int64)
    return lengths, co


def deepseek_decompress(seed=1001, fp8=False) -> DecompressInputs:
    """16 requests, len ~U[512,4096], cache_offsets ~U[0,len/4], page_size 128, shuffled
    pages, latent 512 + 64, W_k [16384, 512]."""
    lengths, co = deepseek_lengths(seed)
    return make_decompress("deepseek_v3_fp8_decompress" if fp8 else "deepseek_v3_bf16_decompress",
                           seed + 1, lengths, co, 128, 512, 64, 16384, fp8=fp8)


def deepseek_qcache_decompress(seed=1001) -> DecompressInputs:
    """The DeepSeek-V3 FP8 decompress (same 16 requests, rows, pages and W_k) over a
    quantised latent cache (656-byte slots: 512 e4m3 codes, 64 bf16 rope, 4 fp32 scales)."""
    lengths, co = deepseek_lengths(seed)
    return make_qcache_decompress("deepseek_v3_fp8_qcache_decompress", seed + 1, lengths, co, 128,
                                  512, 64, 16384)


def long_context_decompress(seed=1003) -> DecompressInputs:
    """4 requests x 32768 cached tokens (buffer_length 131072), 1024 shuffled pages."""
    return make_decompress("long_context_decompress", seed, [32768] * 4, [0] * 4, 128, 512, 64,
                           16384)


@dataclass
class CacheWriteInputs:
    """New latent rows [total_rows, R + P] to be normalised, rotated and stored into a paged
    latent cache [num_layers, num_pages, page_size, R + P] after each request's cached
    tokens."""
    name: str
    latent: np.ndarray             # uint16 bf16 [total_rows, R + P]
    input_row_offsets: np.ndarray  # uint32 [batch + 1]
    cache_lengths: np.ndarray      # uint32 [batch]
    page_table: np.ndarray         # uint32 [batch, max_pages_per_seq]
    cache: np.ndarray              # uint16 bf16 pre-filled with SENTINEL_CACHE, or (quantised
                                   # cache) uint8 slots pre-filled with SENTINEL_QBYTE
    gamma: np.ndarray              # float32 [R]
    epsilon: float
    freqs_cis: np.ndarray          # float32 [max_seq_len, P]: P/2 (cos, sin) pairs per position
    kv_lora_rank: int
    rope_dim: int
    layer_idx: int

    @property
    def batch(self) -> int:
        return int(self.page_table.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.latent.shape[0])

    @property
    def row_elems(self) -> int:
        return self.kv_lora_rank + self.rope_dim

    @property
    def num_pages(self) -> int:
        return int(self.cache.shape[1])

    @property
    def page_size(self) -> int:
        return int(self.cache.shape[2])

    @property
    def strides(self):
        L, Pg, S, E = self.cache.shape
        return Pg * S * E, S * E, E

    @property
    def quantised(self) -> bool:
        return self.cache.dtype == np.uint8

    @property
    def bytes_moved(self) -> int:
        """Algorithmic HBM bytes: read every new row and write it into the cache (a bf16 row,
        or a quantised slot's payload), read gamma and the freqs_cis table once."""
        rows = int(self.input_row_offsets[-1])
        out = (qslot_payload_bytes(self.kv_lora_rank, self.rope_dim) if self.quantised
               else 2 * self.row_elems)
        return rows * (2 * self.row_elems + out) + self.gamma.nbytes + self.freqs_cis.nbytes


def make_cache_write(name, seed, new_tokens, cache_lengths, kv_lora_rank, rope_dim, page_size,
                     num_layers=1, layer_idx=0, extra_pages=0, epsilon=1e-6, max_seq_len=None,
                     latent_std=1.0, quantised=False, slot_pad=0) -> CacheWriteInputs:
    """Seeded cache-write problem: latent ~N(0, latent_std^2) bf16, gamma ~1 + N(0, 0.1^2)
    fp32, freqs_cis = (cos phi, sin phi) for phi ~U[0, 2 pi) drawn per position and pair
    (any unit complex numbers are valid RoPE factors), pages assigned in one seeded
    shuffle, the cache filled with SENTINEL_CACHE."""
    g = _gen(seed)
    new_tokens = np.asarray(new_tokens, np.int64)
    cl = np.asarray(cache_lengths, np.int64)
    B = len(new_tokens)
    iro = np.zeros(B + 1, np.uint32)
    iro[1:] = np.cumsum(new_tokens)
    C = kv_lora_rank + rope_dim
    pages_needed = [int(math.ceil((cl[b] + new_tokens[b]) / page_size)) for b in range(B)]
    total_pages = sum(pages_needed) + extra_pages
    pt = _assign_pages(pages_needed, total_pages, g)
    M = int(iro[-1])
    latent = bf16_normal((M, C), latent_std, g)
    gamma = (1.0 + 0.1 * torch.randn(kv_lora_rank, generator=g, dtype=torch.float64)).to(torch.float32)
    if max_seq_len is None:
        max_seq_len = int((cl + new_tokens).max()) + 1
    phi = torch.rand(max_seq_len, rope_dim // 2, generator=g, dtype=torch.float64) * (2 * math.pi)
    freqs = torch.stack([torch.cos(phi), torch.sin(phi)], dim=-1).reshape(max_seq_len, rope_dim)
    if quantised:
        slot_bytes = (qslot_payload_bytes(kv_lora_rank, rope_dim) + 15) // 16 * 16 + slot_pad
        cache = np.full((num_layers, total_pages, page_size, slot_bytes), SENTINEL_QBYTE, np.uint8)
    else:
        cache = np.full((num_layers, total_pages, page_size, C + slot_pad), SENTINEL_CACHE, np.uint16)
    return CacheWriteInputs(name=name, latent=latent, input_row_offsets=iro,
                            cache_lengths=cl.astype(np.uint32), page_table=pt, cache=cache,
                            gamma=gamma.numpy().copy(), epsilon=float(epsilon),
                            freqs_cis=freqs.to(torch.float32).numpy().copy(),
                            kv_lora_rank=kv_lora_rank, rope_dim=rope_dim, layer_idx=layer_idx)


def cache_write_path(seed=1007, quantised=False) -> CacheWriteInputs:
    """DeepSeek-V3 latent cache write of a prefill batch: 32 requests, new ~U[1024, 4096]
    tokens after cache_len ~U[0, 2048], latent 512 + 64, page_size 128, 2 layers (layer 1
    written); bf16 slots, or quantised 656-byte slots."""
    g = _gen(seed)
    new = torch.randint(1024, 4097, (32,), generator=g).numpy()
    cl = torch.randint(0, 2049, (32,), generator=g).numpy()
    return make_cache_write("cache_write_q_path" if quantised else "cache_write_path", seed + 1,
                            new, cl, 512, 64, 128, num_layers=2, layer_idx=1, quantised=quantised)


@dataclass
class KvMatmulInputs:
    """One kv_matmul problem.  cache is [num_layers, 2 (K, V), num_pages, page_size,
    head_elems]; hidden_state [total_rows, k_in]; weight [k_in, n_out] (n_out contiguous)."""
    name: str
    hidden_state: np.ndarray
    input_row_offsets: np.ndarray
    weight: np.ndarray
    cache: np.ndarray
    page_table: np.ndarray
    cache_lengths: np.ndarray
    head_elems: int
    layer_idx: int
    new_tokens: Optional[np.ndarray] = None
    w_e4m3: Optional[np.ndarray] = None   # FP8 form: uint8 [n_out, k_in] (weight is then None)
    w_scale: Optional[np.ndarray] = None  # float32 [n_out/128, k_in/128]

    @property
    def fp8(self) -> bool:
        return self.w_e4m3 is not None

    @property
    def batch(self) -> int:
        return int(self.cache_lengths.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.hidden_state.shape[0])

    @property
    def k_in(self) -> int:
        return int(self.w_e4m3.shape[1] if self.fp8 else self.weight.shape[0])

    @property
    def n_out(self) -> int:
        return int(self.w_e4m3.shape[0] if self.fp8 else self.weight.shape[1])

    @property
    def num_pages(self) -> int:
        return int(self.cache.shape[2])

    @property
    def page_size(self) -> int:
        return int(self.cache.shape[3])

    @property
    def strides(self):
        """(layer_stride, page_stride, slot_stride, kv_stride) in elements."""
        _, two, P, S, E = self.cache.shape
        return two * P * S * E, S * E, E, P * S * E

    @property
    def flops(self) -> int:
        return 2 * self.total_rows * self.k_in * self.n_out

    @property
    def bytes_moved(self) -> int:
        """Algorithmic HBM bytes: read hidden_state and weight once, write every output; the
        FP8 form also writes and reads back the quantised rows (k_in + k_in/32 bytes a row)
        and reads an e4m3 weight with its scales."""
        if self.fp8:
            q = self.total_rows * (self.k_in + self.k_in // 32)
            return (2 * self.total_rows * self.k_in + 2 * q + self.w_e4m3.nbytes +
                    self.w_scale.nbytes + 2 * self.total_rows * self.n_out)
        return 2 * (self.total_rows * self.k_in + self.k_in * self.n_out +
                    self.total_rows * self.n_out)


def make_kv_matmul(name, seed, new_tokens, cache_lengths, k_in, num_kv_heads, head_dim,
                   page_size, num_layers=1, layer_idx=0, k_only=False, extra_pages=0,
                   int_values=False, w_std=None, fp8=False) -> KvMatmulInputs:
    g = _gen(seed)
    new_tokens = np.asarray(new_tokens, np.int64)
    cache_lengths = np.asarray(cache_lengths, np.int64)
    B = len(new_tokens)
    iro = np.zeros(B + 1, np.uint32)
    iro[1:] = np.cumsum(new_tokens)
    M = int(iro[-1])
    HD = num_kv_heads * head_dim
    n_out = HD if k_only else 2 * HD
    pages_needed = [int(math.ceil((c + n) / page_size)) for c, n in zip(cache_lengths, new_tokens)]
    total_pages = sum(pages_needed) + extra_pages
    pt = _assign_pages(pages_needed, total_pages, g)
    if int_values:
        hidden = bf16_small_ints((M, k_in), -4, 4, g)
        weight = bf16_small_ints((k_in, n_out), -2, 2, g)
    else:
        hidden = bf16_normal((M, k_in), 1.0, g)
        weight = bf16_normal((k_in, n_out), w_std if w_std is not None else 1.0 / math.sqrt(k_in), g)
    cache = np.empty((num_layers, 2, total_pages, page_size, HD), np.uint16)
    cache[:, 0] = SENTINEL_K
    cache[:, 1] = SENTINEL_V
    k = KvMatmulInputs(name=name, hidden_state=hidden, input_row_offsets=iro, weight=weight,
                       cache=cache, page_table=pt, cache_lengths=cache_lengths.astype(np.uint32),
                       head_elems=HD, layer_idx=layer_idx, new_tokens=new_tokens)
    if fp8:
        # the FP8 form: a weight drawn in fp32 as [n_out, k_in] and quantised per 128 x 128
        # block like the FP8 decompress weights (its own generator: the rest is unchanged)
        gw = _gen(seed + 7717)
        std = w_std if w_std is not None else 1.0 / math.sqrt(k_in)
        w = torch.randn(n_out, k_in, generator=gw, dtype=torch.float32) * std
        k.w_e4m3, k.w_scale = quantize_weight_e4m3(w)
        k.weight = None
    return k


def kv_matmul_write_path(seed=1004, fp8=False) -> KvMatmulInputs:
    """32 requests, new ~U[1,512], cache_len ~U[0,2048], hidden [sum(new), 4096] ~N(0,1),
    weight [4096, 2048] ~N(0, 1/64), 8 kv heads x 128 (K then V), page_size 128; the FP8
    form has an e4m3 weight [2048, 4096] with 128 x 128 fp32 block scales."""
    g = _gen(seed)
    new = torch.randint(1, 513, (32,), generator=g).numpy()
    cl = torch.randint(0, 2049, (32,), generator=g).numpy()
    return make_kv_matmul("kv_matmul_fp8_write_path" if fp8 else "kv_matmul_write_path",
                          seed + 1, new, cl, 4096, 8, 128, 128, w_std=1.0 / 64, fp8=fp8)


# Names used by tests and the benchmark.
WORKLOADS = {
    "tiny_decompress": tiny_decompress,
    "deepseek_v3_bf16_decompress": lambda: deepseek_decompress(1001, fp8=False),
    "deepseek_v3_fp8_decompress": lambda: deepseek_decompress(1001, fp8=True),
    "long_context_decompress": long_context_decompress,
    "deepseek_v3_bf16_decompress_kv": lambda: deepseek_decompress_kv(1001, fp8=False),
    "deepseek_v3_fp8_decompress_kv": lambda: deepseek_decompress_kv(1001, fp8=True),
    "kv_matmul_write_path": kv_matmul_write_path,
    "kv_matmul_fp8_write_path": lambda: kv_matmul_write_path(1004, fp8=True),
    "cache_write_path": cache_write_path,
    "cache_write_q_path": lambda: cache_write_path(1007, quantised=True),
    "deepseek_v3_fp8_qcache_decompress": deepseek_qcache_decompress,
}
