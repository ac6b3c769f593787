"""CPU oracle for the paged-KV MLA hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product library never calls it, and it shares no code
with the CUDA path.  The arithmetic lives in ``pkm_oracle.c`` (plain C, fp64
accumulation); this module compiles it with gcc and wraps it with numpy arrays.

Each wrapper follows the passage cited in the C source:
  * generic_flare_mla_decompress_k_cache_ragged_paged -- description and Args
  * mla_prefill_decode_graph_fp8 -- Parameters (scale granularities), Args (w_k, w_k_scale,
    w_uv, w_uv_scale)
  * mla_prefill_decode_graph_fp8 -- Args kv_input_fn, kv_norm_gamma, epsilon, freqs_cis
    (the cache-write side)
  * PagedKVCacheCollection[..., scale_dtype_, quantization_granularity_] -- the quantised
    paged latent cache (written by the cache-write side, read by the FP8 decompress)
  * kv_matmul_ragged_paged -- Args (hidden_state, input_row_offsets, weight, kv_collection),
    and its FP8 form with the scale-granularity parameters of mla_prefill_decode_graph_fp8
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libpkm_oracle.so")
_lock = threading.Lock()
_lib = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_i64, _i32, _u32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32


def build(force: bool = False) -> str:
    """Compile pkm_oracle.c into a shared library (plain gcc, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            L.oracle_double_to_bf16.restype = ctypes.c_uint16
            L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_double.restype = ctypes.c_double
            L.oracle_float_to_e4m3_satfinite.argtypes = [ctypes.c_float]
            L.oracle_float_to_e4m3_satfinite.restype = ctypes.c_uint8
            cache_args = [_u16p, _i64, _i64, _i64, _i32, _i32, _u32p, _i32, _u32, _u32p, _u32p,
                          _i32, _i32]
            L.oracle_gather_latent.argtypes = cache_args + [_i32, _u16p, _u8p]
            L.oracle_gather_latent.restype = ctypes.c_int
            L.oracle_up_project_bf16.argtypes = [_u16p, _i32, _u8p, _i32, _u16p, _i32, _i32, _u16p]
            L.oracle_up_project_bf16.restype = None
            L.oracle_decompress_k.argtypes = cache_args + [_i32, _i32, _u16p, _i32, _u16p, _u16p, _u8p]
            L.oracle_decompress_k.restype = ctypes.c_int
            L.oracle_decompress_k_row.argtypes = cache_args + [_i32, _i32, _u16p, _i32, _i64, _u16p,
                                                               _u16p]
            L.oracle_decompress_k_row.restype = ctypes.c_int
            L.oracle_quantize_row_e4m3.argtypes = [_u16p, _i32, _u8p, _f32p]
            L.oracle_quantize_row_e4m3.restype = None
            L.oracle_decompress_k_fp8.argtypes = cache_args + [_i32, _i32, _u8p, _f32p, _i32, _u16p,
                                                               _u16p, _u8p, _f32p, _u8p]
            L.oracle_decompress_k_fp8.restype = ctypes.c_int
            L.oracle_decompress_k_fp8_row.argtypes = cache_args + [_i32, _i32, _u8p, _f32p, _i32,
                                                                   _i64, _u16p, _u16p, _u8p, _f32p]
            L.oracle_decompress_k_fp8_row.restype = ctypes.c_int
            L.oracle_up_project_v_bf16.argtypes = [_u16p, _i32, _u8p, _i32, _u16p, _i32, _i32, _i32,
                                                    _u16p]
            L.oracle_up_project_v_bf16.restype = None
            L.oracle_decompress_kv.argtypes = cache_args + [_i32, _i32, _u16p, _i32, _u16p, _i32, _i32,
                                                            _u16p, _u16p, _u16p, _u8p]
            L.oracle_decompress_kv.restype = ctypes.c_int
            L.oracle_decompress_kv_fp8.argtypes = cache_args + [_i32, _i32, _u8p, _f32p, _i32, _u8p,
                                                                _f32p, _i32, _i32, _u16p, _u16p,
                                                                _u16p, _u8p, _f32p, _u8p]
            L.oracle_decompress_kv_fp8.restype = ctypes.c_int
            L.oracle_decompress_kv_row.argtypes = cache_args + [_i32, _i32, _u16p, _i32, _u16p, _i32,
                                                                _i32, _i64, _u16p, _u16p, _u16p]
            L.oracle_decompress_kv_row.restype = ctypes.c_int
            L.oracle_decompress_kv_fp8_row.argtypes = cache_args + [_i32, _i32, _u8p, _f32p, _i32,
                                                                    _u8p, _f32p, _i32, _i32, _i64,
                                                                    _u16p, _u16p, _u16p, _u8p, _f32p]
            L.oracle_decompress_kv_fp8_row.restype = ctypes.c_int
            L.oracle_cache_write.argtypes = [_u16p, _u32p, _i32, _i32, _i32, _i32, _f32p, ctypes.c_float,
                                             _f32p, _i32, _u16p, _i64, _i64, _i64, _i32, _i32, _u32p,
                                             _i32, _u32p, _u32]
            L.oracle_cache_write.restype = ctypes.c_int
            qcache_args = [_u8p, _i64, _i64, _i64, _i32, _i32, _u32p, _i32, _u32, _u32p, _u32p,
                           _i32, _i32]
            L.oracle_dequant_bf16.argtypes = [ctypes.c_uint8, ctypes.c_float]
            L.oracle_dequant_bf16.restype = ctypes.c_uint16
            L.oracle_qslot_bytes.argtypes = [_i32, _i32]
            L.oracle_qslot_bytes.restype = ctypes.c_int64
            L.oracle_cache_write_q.argtypes = [_u16p, _u32p, _i32, _i32, _i32, _i32, _f32p,
                                               ctypes.c_float, _f32p, _i32, _u8p, _i64, _i64, _i64,
                                               _i32, _i32, _u32p, _i32, _u32p, _u32]
            L.oracle_cache_write_q.restype = ctypes.c_int
            L.oracle_decompress_k_qcache_fp8.argtypes = qcache_args + [_i32, _i32, _u8p, _f32p, _i32,
                                                                       _u16p, _u16p, _u8p, _f32p, _u8p]
            L.oracle_decompress_k_qcache_fp8.restype = ctypes.c_int
            L.oracle_decompress_k_qcache_fp8_row.argtypes = qcache_args + [_i32, _i32, _u8p, _f32p,
                                                                           _i32, _i64, _u16p, _u16p,
                                                                           _u8p, _f32p]
            L.oracle_decompress_k_qcache_fp8_row.restype = ctypes.c_int
            L.oracle_kv_matmul.argtypes = [_u16p, _u32p, _i32, _i32, _i32, _u16p, _i32, _u16p, _i64,
                                           _i64, _i64, _i64, _i32, _i32, _i32, _u32p, _i32, _u32p,
                                           _u32]
            L.oracle_kv_matmul.restype = ctypes.c_int
            L.oracle_kv_matmul_fp8.argtypes = [_u16p, _u32p, _i32, _i32, _i32, _u8p, _f32p, _i32,
                                               _u16p, _i64, _i64, _i64, _i64, _i32, _i32, _i32,
                                               _u32p, _i32, _u32p, _u32, _u8p, _f32p]
            L.oracle_kv_matmul_fp8.restype = ctypes.c_int
            _i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
            L.oracle_kv_row_dest.argtypes = [_u32p, _i32, _i32, _u32p, _u32p, _i32, _i32, _i32, _i64,
                                             _i64, _i64p]
            L.oracle_kv_row_dest.restype = None
            _lib = L
    return _lib


# ---------------------------------------------------------------------------------------
# scalar codecs
# ---------------------------------------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits) & 0xFFFF)


def double_to_bf16(x: float) -> int:
    return int(lib().oracle_double_to_bf16(float(x)))


def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code) & 0xFF)


def float_to_e4m3(x: float) -> int:
    return int(lib().oracle_float_to_e4m3_satfinite(float(np.float32(x))))


# ---------------------------------------------------------------------------------------
# array wrappers (all arrays are numpy; bf16 tensors travel as uint16 bit patterns)
# ---------------------------------------------------------------------------------------

def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class PagedCacheView:
    """Host view of one paged cache: flat uint16 storage plus element strides."""

    def __init__(self, data, layer_stride, page_stride, slot_stride, num_pages, page_size,
                 page_table, max_pages_per_seq, kv_stride=0):
        self.data = _c(np.asarray(data).reshape(-1), np.uint16)
        self.layer_stride = int(layer_stride)
        self.page_stride = int(page_stride)
        self.slot_stride = int(slot_stride)
        self.kv_stride = int(kv_stride)
        self.num_pages = int(num_pages)
        self.page_size = int(page_size)
        self.page_table = _c(np.asarray(page_table).reshape(-1), np.uint32)
        self.max_pages_per_seq = int(max_pages_per_seq)

    def args(self, layer_idx, bro, co, batch, buffer_length):
        return [self.data, self.layer_stride, self.page_stride, self.slot_stride, self.num_pages,
                self.page_size, self.page_table, self.max_pages_per_seq, int(layer_idx),
                _c(bro, np.uint32), _c(co, np.uint32), int(batch), int(buffer_length)]


def decompress_k(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length, kv_lora_rank,
                 rope_dim, w_k, k_latent=None, k_buffer=None):
    """bf16 decompress.  Returns (status, k_latent, k_buffer, row_written).

    k_latent / k_buffer may be passed pre-filled (e.g. with a sentinel) to check that
    untouched rows stay untouched; they are modified in place."""
    w_k = _c(w_k, np.uint16)
    n_out = w_k.shape[0]
    C = kv_lora_rank + rope_dim
    if k_latent is None:
        k_latent = np.zeros((buffer_length, C), np.uint16)
    if k_buffer is None:
        k_buffer = np.zeros((buffer_length, n_out), np.uint16)
    written = np.zeros(max(buffer_length, 1), np.uint8)
    st = lib().oracle_decompress_k(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                   kv_lora_rank, rope_dim, w_k.reshape(-1), n_out,
                                   k_latent.reshape(-1) if buffer_length else np.zeros(1, np.uint16),
                                   k_buffer.reshape(-1) if buffer_length else np.zeros(1, np.uint16),
                                   written)
    return st, k_latent, k_buffer, written[:buffer_length].astype(bool)


def gather_latent(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length, latent_cols,
                  k_latent=None):
    if k_latent is None:
        k_latent = np.zeros((buffer_length, latent_cols), np.uint16)
    written = np.zeros(max(buffer_length, 1), np.uint8)
    st = lib().oracle_gather_latent(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                    latent_cols, k_latent.reshape(-1), written)
    return st, k_latent, written[:buffer_length].astype(bool)


def up_project_bf16(k_latent, latent_cols, w_k, kv_lora_rank, row_written=None):
    k_latent = _c(k_latent, np.uint16)
    w_k = _c(w_k, np.uint16)
    L = k_latent.shape[0]
    n_out = w_k.shape[0]
    out = np.zeros((L, n_out), np.uint16)
    rw = np.ones(L, np.uint8) if row_written is None else _c(row_written, np.uint8)
    lib().oracle_up_project_bf16(k_latent.reshape(-1), latent_cols, rw, L, w_k.reshape(-1),
                                 kv_lora_rank, n_out, out.reshape(-1))
    return out


def decompress_k_row(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length,
                     kv_lora_rank, rope_dim, w_k, r):
    """One row of the bf16 decompress.  Returns (status, latent_row, k_row)."""
    w_k = _c(w_k, np.uint16)
    n_out = w_k.shape[0]
    lat = np.zeros(kv_lora_rank + rope_dim, np.uint16)
    k = np.zeros(n_out, np.uint16)
    st = lib().oracle_decompress_k_row(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                       kv_lora_rank, rope_dim, w_k.reshape(-1), n_out, int(r),
                                       lat, k)
    return st, lat, k


def quantize_row_e4m3(latent_row, kv_lora_rank):
    q = np.zeros(kv_lora_rank, np.uint8)
    s = np.zeros(kv_lora_rank // 128, np.float32)
    lib().oracle_quantize_row_e4m3(_c(latent_row, np.uint16), kv_lora_rank, q, s)
    return q, s


def decompress_k_fp8(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length,
                     kv_lora_rank, rope_dim, w_e4m3, w_scale, k_latent=None, k_buffer=None):
    """FP8 decompress.  Returns (status, k_latent, k_buffer, q_latent, q_scale, row_written)."""
    w_e4m3 = _c(w_e4m3, np.uint8)
    w_scale = _c(w_scale, np.float32)
    n_out = w_e4m3.shape[0]
    C = kv_lora_rank + rope_dim
    L1 = max(buffer_length, 1)
    if k_latent is None:
        k_latent = np.zeros((L1, C), np.uint16)
    if k_buffer is None:
        k_buffer = np.zeros((L1, n_out), np.uint16)
    q = np.zeros((L1, kv_lora_rank), np.uint8)
    qs = np.zeros((L1, kv_lora_rank // 128), np.float32)
    written = np.zeros(L1, np.uint8)
    st = lib().oracle_decompress_k_fp8(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                       kv_lora_rank, rope_dim, w_e4m3.reshape(-1),
                                       w_scale.reshape(-1), n_out, k_latent.reshape(-1),
                                       k_buffer.reshape(-1), q.reshape(-1), qs.reshape(-1), written)
    return (st, k_latent[:buffer_length], k_buffer[:buffer_length], q[:buffer_length],
            qs[:buffer_length], written[:buffer_length].astype(bool))


def decompress_k_fp8_row(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length,
                         kv_lora_rank, rope_dim, w_e4m3, w_scale, r):
    """One row of the FP8 decompress.  Returns (status, latent_row, k_row, q_row, scale_row)."""
    w_e4m3 = _c(w_e4m3, np.uint8)
    n_out = w_e4m3.shape[0]
    lat = np.zeros(kv_lora_rank + rope_dim, np.uint16)
    k = np.zeros(n_out, np.uint16)
    q = np.zeros(kv_lora_rank, np.uint8)
    s = np.zeros(kv_lora_rank // 128, np.float32)
    st = lib().oracle_decompress_k_fp8_row(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                           kv_lora_rank, rope_dim, w_e4m3.reshape(-1),
                                           _c(w_scale, np.float32).reshape(-1), n_out, int(r), lat,
                                           k, q, s)
    return st, lat, k, q, s


def up_project_v_bf16(k_latent, latent_cols, w_uv, kv_lora_rank, row_written=None):
    """V = latent x w_uv per head: w_uv [num_heads, v_head_dim, R]; returns [L, H, Dv]."""
    k_latent = _c(k_latent, np.uint16)
    w_uv = _c(w_uv, np.uint16)
    L = k_latent.shape[0]
    H, Dv = w_uv.shape[0], w_uv.shape[1]
    out = np.zeros((L, H, Dv), np.uint16)
    rw = np.ones(L, np.uint8) if row_written is None else _c(row_written, np.uint8)
    lib().oracle_up_project_v_bf16(k_latent.reshape(-1), latent_cols, rw, L, w_uv.reshape(-1), H,
                                   Dv, kv_lora_rank, out.reshape(-1))
    return out


def decompress_kv(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length, kv_lora_rank,
                  rope_dim, w_k, w_uv, k_latent=None, k_buffer=None, v_buffer=None):
    """bf16 K and V decompress (w_uv [H, Dv, R]).  Returns (status, k_latent, k_buffer,
    v_buffer [L, H, Dv], row_written); pre-filled outputs are modified in place."""
    w_k = _c(w_k, np.uint16)
    w_uv = _c(w_uv, np.uint16)
    n_out = w_k.shape[0]
    H, Dv = w_uv.shape[0], w_uv.shape[1]
    C = kv_lora_rank + rope_dim
    L1 = max(buffer_length, 1)
    if k_latent is None:
        k_latent = np.zeros((L1, C), np.uint16)
    if k_buffer is None:
        k_buffer = np.zeros((L1, n_out), np.uint16)
    if v_buffer is None:
        v_buffer = np.zeros((L1, H, Dv), np.uint16)
    written = np.zeros(L1, np.uint8)
    st = lib().oracle_decompress_kv(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                    kv_lora_rank, rope_dim, w_k.reshape(-1), n_out,
                                    w_uv.reshape(-1), H, Dv, k_latent.reshape(-1),
                                    k_buffer.reshape(-1), v_buffer.reshape(-1), written)
    return (st, k_latent[:buffer_length], k_buffer[:buffer_length], v_buffer[:buffer_length],
            written[:buffer_length].astype(bool))


def decompress_kv_fp8(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length,
                      kv_lora_rank, rope_dim, w_e4m3, w_scale, w_uv_e4m3, w_uv_scale):
    """FP8 K and V decompress.  Returns (status, k_latent, k_buffer, v_buffer, q_latent,
    q_scale, row_written)."""
    w_e4m3 = _c(w_e4m3, np.uint8)
    w_uv_e4m3 = _c(w_uv_e4m3, np.uint8)
    n_out = w_e4m3.shape[0]
    H, Dv = w_uv_e4m3.shape[0], w_uv_e4m3.shape[1]
    C = kv_lora_rank + rope_dim
    L1 = max(buffer_length, 1)
    k_latent = np.zeros((L1, C), np.uint16)
    k_buffer = np.zeros((L1, n_out), np.uint16)
    v_buffer = np.zeros((L1, H, Dv), np.uint16)
    q = np.zeros((L1, kv_lora_rank), np.uint8)
    qs = np.zeros((L1, kv_lora_rank // 128), np.float32)
    written = np.zeros(L1, np.uint8)
    st = lib().oracle_decompress_kv_fp8(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                        kv_lora_rank, rope_dim, w_e4m3.reshape(-1),
                                        _c(w_scale, np.float32).reshape(-1), n_out,
                                        w_uv_e4m3.reshape(-1), _c(w_uv_scale, np.float32).reshape(-1),
                                        H, Dv, k_latent.reshape(-1), k_buffer.reshape(-1),
                                        v_buffer.reshape(-1), q.reshape(-1), qs.reshape(-1), written)
    return (st, k_latent[:buffer_length], k_buffer[:buffer_length], v_buffer[:buffer_length],
            q[:buffer_length], qs[:buffer_length], written[:buffer_length].astype(bool))


def decompress_kv_row(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length,
                      kv_lora_rank, rope_dim, w_k, w_uv, r):
    """One row of the bf16 K and V decompress.  Returns (status, latent_row, k_row, v_row)."""
    w_k = _c(w_k, np.uint16)
    w_uv = _c(w_uv, np.uint16)
    n_out = w_k.shape[0]
    H, Dv = w_uv.shape[0], w_uv.shape[1]
    lat = np.zeros(kv_lora_rank + rope_dim, np.uint16)
    k = np.zeros(n_out, np.uint16)
    v = np.zeros(H * Dv, np.uint16)
    st = lib().oracle_decompress_kv_row(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                        kv_lora_rank, rope_dim, w_k.reshape(-1), n_out,
                                        w_uv.reshape(-1), H, Dv, int(r), lat, k, v)
    return st, lat, k, v.reshape(H, Dv)


def decompress_kv_fp8_row(cache: PagedCacheView, layer_idx, bro, co, batch, buffer_length,
                          kv_lora_rank, rope_dim, w_e4m3, w_scale, w_uv_e4m3, w_uv_scale, r):
    """One row of the FP8 K and V decompress.  Returns (status, latent_row, k_row, v_row,
    q_row, scale_row)."""
    w_e4m3 = _c(w_e4m3, np.uint8)
    w_uv_e4m3 = _c(w_uv_e4m3, np.uint8)
    n_out = w_e4m3.shape[0]
    H, Dv = w_uv_e4m3.shape[0], w_uv_e4m3.shape[1]
    lat = np.zeros(kv_lora_rank + rope_dim, np.uint16)
    k = np.zeros(n_out, np.uint16)
    v = np.zeros(H * Dv, np.uint16)
    q = np.zeros(kv_lora_rank, np.uint8)
    s = np.zeros(kv_lora_rank // 128, np.float32)
    st = lib().oracle_decompress_kv_fp8_row(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                            kv_lora_rank, rope_dim, w_e4m3.reshape(-1),
                                            _c(w_scale, np.float32).reshape(-1), n_out,
                                            w_uv_e4m3.reshape(-1),
                                            _c(w_uv_scale, np.float32).reshape(-1), H, Dv, int(r),
                                            lat, k, v, q, s)
    return st, lat, k, v.reshape(H, Dv), q, s


def cache_write(latent, input_row_offsets, batch, total_rows, kv_lora_rank, rope_dim, gamma,
                epsilon, freqs_cis, cache: PagedCacheView, cache_lengths, layer_idx):
    """RMSNorm + RoPE of new latent rows into the paged cache; cache.data is modified in
    place.  Returns the status."""
    freqs_cis = _c(freqs_cis, np.float32)
    return lib().oracle_cache_write(_c(latent, np.uint16).reshape(-1), _c(input_row_offsets, np.uint32),
                                    int(batch), int(total_rows), int(kv_lora_rank), int(rope_dim),
                                    _c(gamma, np.float32), float(epsilon), freqs_cis.reshape(-1),
                                    int(freqs_cis.shape[0]), cache.data, cache.layer_stride,
                                    cache.page_stride, cache.slot_stride, cache.num_pages,
                                    cache.page_size, cache.page_table, cache.max_pages_per_seq,
                                    _c(cache_lengths, np.uint32), int(layer_idx))


class QuantCacheView:
    """Host view of one quantised paged latent cache: flat bytes plus byte strides (slot
    layout in pkm_oracle.c: codes, rope bf16, fp32 block scales)."""

    def __init__(self, data, layer_stride, page_stride, slot_stride, num_pages, page_size,
                 page_table, max_pages_per_seq):
        self.data = _c(np.asarray(data).reshape(-1), np.uint8)
        self.layer_stride = int(layer_stride)
        self.page_stride = int(page_stride)
        self.slot_stride = int(slot_stride)
        self.num_pages = int(num_pages)
        self.page_size = int(page_size)
        self.page_table = _c(np.asarray(page_table).reshape(-1), np.uint32)
        self.max_pages_per_seq = int(max_pages_per_seq)

    def args(self, layer_idx, bro, co, batch, buffer_length):
        return [self.data, self.layer_stride, self.page_stride, self.slot_stride, self.num_pages,
                self.page_size, self.page_table, self.max_pages_per_seq, int(layer_idx),
                _c(bro, np.uint32), _c(co, np.uint32), int(batch), int(buffer_length)]


def dequant_bf16(code: int, scale: float) -> int:
    return int(lib().oracle_dequant_bf16(int(code), float(np.float32(scale))))


def qslot_bytes(kv_lora_rank, rope_dim) -> int:
    return int(lib().oracle_qslot_bytes(int(kv_lora_rank), int(rope_dim)))


def cache_write_q(latent, input_row_offsets, batch, total_rows, kv_lora_rank, rope_dim, gamma,
                  epsilon, freqs_cis, cache: QuantCacheView, cache_lengths, layer_idx):
    """RMSNorm + RoPE of new latent rows, quantised into the paged cache's slots; cache.data
    is modified in place.  Returns the status."""
    freqs_cis = _c(freqs_cis, np.float32)
    return lib().oracle_cache_write_q(_c(latent, np.uint16).reshape(-1), _c(input_row_offsets, np.uint32),
                                      int(batch), int(total_rows), int(kv_lora_rank), int(rope_dim),
                                      _c(gamma, np.float32), float(epsilon), freqs_cis.reshape(-1),
                                      int(freqs_cis.shape[0]), cache.data, cache.layer_stride,
                                      cache.page_stride, cache.slot_stride, cache.num_pages,
                                      cache.page_size, cache.page_table, cache.max_pages_per_seq,
                                      _c(cache_lengths, np.uint32), int(layer_idx))


def decompress_k_qcache_fp8(cache: QuantCacheView, layer_idx, bro, co, batch, buffer_length,
                            kv_lora_rank, rope_dim, w_e4m3, w_scale, k_latent=None, k_buffer=None):
    """FP8 decompress from a quantised cache.  Returns (status, k_latent, k_buffer, q_latent,
    q_scale, row_written)."""
    w_e4m3 = _c(w_e4m3, np.uint8)
    w_scale = _c(w_scale, np.float32)
    n_out = w_e4m3.shape[0]
    C = kv_lora_rank + rope_dim
    L1 = max(buffer_length, 1)
    if k_latent is None:
        k_latent = np.zeros((L1, C), np.uint16)
    if k_buffer is None:
        k_buffer = np.zeros((L1, n_out), np.uint16)
    q = np.zeros((L1, kv_lora_rank), np.uint8)
    qs = np.zeros((L1, kv_lora_rank // 128), np.float32)
    written = np.zeros(L1, np.uint8)
    st = lib().oracle_decompress_k_qcache_fp8(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                              kv_lora_rank, rope_dim, w_e4m3.reshape(-1),
                                              w_scale.reshape(-1), n_out, k_latent.reshape(-1),
                                              k_buffer.reshape(-1), q.reshape(-1), qs.reshape(-1),
                                              written)
    L = buffer_length
    return st, k_latent[:L], k_buffer[:L], q[:L], qs[:L], written[:L].astype(bool)


def decompress_k_qcache_fp8_row(cache: QuantCacheView, layer_idx, bro, co, batch, buffer_length,
                                kv_lora_rank, rope_dim, w_e4m3, w_scale, r):
    """One row of the quantised-cache FP8 decompress.  Returns (status, latent_row, k_row,
    q_row, scale_row)."""
    w_e4m3 = _c(w_e4m3, np.uint8)
    n_out = w_e4m3.shape[0]
    lat = np.zeros(kv_lora_rank + rope_dim, np.uint16)
    k = np.zeros(n_out, np.uint16)
    q = np.zeros(kv_lora_rank, np.uint8)
    s = np.zeros(kv_lora_rank // 128, np.float32)
    st = lib().oracle_decompress_k_qcache_fp8_row(*cache.args(layer_idx, bro, co, batch, buffer_length),
                                                  kv_lora_rank, rope_dim, w_e4m3.reshape(-1),
                                                  _c(w_scale, np.float32).reshape(-1), n_out, int(r),
                                                  lat, k, q, s)
    return st, lat, k, q, s


def kv_matmul(hidden_state, input_row_offsets, batch, total_rows, weight, cache: PagedCacheView,
              head_elems, cache_lengths, layer_idx):
    """kv_matmul into the paged cache; cache.data is modified in place.  Returns status."""
    hidden_state = _c(hidden_state, np.uint16)
    weight = _c(weight, np.uint16)
    k_in = weight.shape[0]
    n_out = weight.shape[1]
    return lib().oracle_kv_matmul(hidden_state.reshape(-1) if total_rows else np.zeros(1, np.uint16),
                                  _c(input_row_offsets, np.uint32), int(batch), int(total_rows),
                                  k_in, weight.reshape(-1), n_out, cache.data, cache.layer_stride,
                                  cache.page_stride, cache.slot_stride, cache.kv_stride,
                                  cache.num_pages, cache.page_size, int(head_elems),
                                  cache.page_table, cache.max_pages_per_seq,
                                  _c(cache_lengths, np.uint32), int(layer_idx))


def kv_matmul_fp8(hidden_state, input_row_offsets, batch, total_rows, w_e4m3, w_scale,
                  cache: PagedCacheView, head_elems, cache_lengths, layer_idx):
    """FP8 kv_matmul into the paged cache (cache.data modified in place).  Returns (status,
    q [total_rows, k_in], s [total_rows, k_in/128]) with the quantised rows that were
    written (zeros elsewhere)."""
    hidden_state = _c(hidden_state, np.uint16)
    w_e4m3 = _c(w_e4m3, np.uint8)
    n_out, k_in = w_e4m3.shape
    M1 = max(int(total_rows), 1)
    q = np.zeros((M1, k_in), np.uint8)
    s = np.zeros((M1, k_in // 128), np.float32)
    st = lib().oracle_kv_matmul_fp8(hidden_state.reshape(-1) if total_rows else np.zeros(1, np.uint16),
                                    _c(input_row_offsets, np.uint32), int(batch), int(total_rows),
                                    k_in, w_e4m3.reshape(-1), _c(w_scale, np.float32).reshape(-1),
                                    n_out, cache.data, cache.layer_stride, cache.page_stride,
                                    cache.slot_stride, cache.kv_stride, cache.num_pages,
                                    cache.page_size, int(head_elems), cache.page_table,
                                    cache.max_pages_per_seq, _c(cache_lengths, np.uint32),
                                    int(layer_idx), q.reshape(-1), s.reshape(-1))
    return st, q[:total_rows], s[:total_rows]


def kv_row_dest(input_row_offsets, batch, total_rows, cache_lengths, cache: PagedCacheView):
    """Addressing step of kv_matmul alone: per-row element offset of the receiving slot inside
    the layer's K plane (-1 uncovered, -2 out of range)."""
    dest = np.zeros(max(int(total_rows), 1), np.int64)
    lib().oracle_kv_row_dest(_c(input_row_offsets, np.uint32), int(batch), int(total_rows),
                             _c(cache_lengths, np.uint32), cache.page_table,
                             cache.max_pages_per_seq, cache.num_pages, cache.page_size,
                             cache.page_stride, cache.slot_stride, dest)
    return dest[: int(total_rows)]
