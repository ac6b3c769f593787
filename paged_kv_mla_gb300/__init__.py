"""Python binding of the GB300 paged-KV MLA library (libpaged_kv_mla.so).

Argument marshalling only: torch tensors are turned into device pointers and the current
torch CUDA stream is passed as the cudaStream_t; every step of the computation runs in the
library's sm_103a kernels.  There is no CPU path: if the shared library is missing this
module refuses to import, and every call raises on a non-OK status.

Entry points (same names as the C ABI in include/paged_kv_mla.h):
  mla_decompress_k_paged              generic_flare_mla_decompress_k_cache_ragged_paged (bf16)
  mla_decompress_kv_paged             the same gather feeding the K and the V (w_uv) projections
  mla_decompress_k_paged_fp8          the K-decompress stage of mla_prefill_decode_graph_fp8
                                      (+ mla_decompress_k_paged_fp8_workspace_size)
  mla_decompress_kv_paged_fp8         its K and V form
  mla_decompress_k_paged_fp8_noalloc  the FP8 decompress with a fixed in-library workspace
  mla_decompress_k_paged_fp8_qcache   the FP8 decompress reading a quantised paged cache
  mla_cache_write_paged               RMSNorm + RoPE of new latent rows into the paged cache
  mla_cache_write_paged_qcache        the same into a quantised paged cache
  kv_matmul_paged                     kv_matmul_ragged_paged (bf16)
  kv_matmul_paged_fp8                 its FP8 block-scaled form (+ kv_matmul_paged_fp8_workspace_size)
  pkm_check_wait_timeout              the bounded-wait self-check
  pkm_validate_row_offsets            the opt-in check that an offset array is non-decreasing
  status_string, last_cuda_error      pkm_status_string, pkm_last_cuda_error
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpaged_kv_mla.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python paged_kv_mla_gb300/build.py, or __graft_entry__.build()).")

_lib = ctypes.CDLL(LIB_PATH)

PKM_OK = 0
PKM_ERR_INVALID_ARG = 1
PKM_ERR_UNSUPPORTED = 2
PKM_ERR_CUDA = 3
PKM_ERR_OUT_OF_RANGE = 4
PKM_ERR_TIMEOUT = 5


class PkmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {status_string(code)} ({code})"
        if code == PKM_ERR_CUDA:
            msg += f": {last_cuda_error()}"
        super().__init__(msg)


class _CCache(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("layer_stride", ctypes.c_int64),
                ("page_stride", ctypes.c_int64), ("slot_stride", ctypes.c_int64),
                ("kv_stride", ctypes.c_int64), ("num_layers", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("row_elems", ctypes.c_int32), ("page_table", ctypes.c_void_p),
                ("max_pages_per_seq", ctypes.c_int32), ("cache_lengths", ctypes.c_void_p)]


class _CQuantCache(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("layer_stride", ctypes.c_int64),
                ("page_stride", ctypes.c_int64), ("slot_stride", ctypes.c_int64),
                ("num_layers", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("kv_lora_rank", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("page_table", ctypes.c_void_p),
                ("max_pages_per_seq", ctypes.c_int32), ("cache_lengths", ctypes.c_void_p)]


_vp, _i32, _u32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
_lib.pkm_status_string.argtypes = [ctypes.c_int]
_lib.pkm_status_string.restype = ctypes.c_char_p
_lib.pkm_last_cuda_error.argtypes = []
_lib.pkm_last_cuda_error.restype = ctypes.c_char_p
_lib.mla_decompress_k_paged.argtypes = [ctypes.POINTER(_CCache), _u32, _vp, _vp, _i32, _i32, _i32,
                                        _i32, _vp, _i32, _vp, _vp, _vp, _vp]
_lib.mla_decompress_k_paged.restype = ctypes.c_int
_lib.mla_decompress_k_paged_fp8_workspace_size.argtypes = [_i32, _i32]
_lib.mla_decompress_k_paged_fp8_workspace_size.restype = _sz
_lib.mla_decompress_k_paged_fp8.argtypes = [ctypes.POINTER(_CCache), _u32, _vp, _vp, _i32, _i32,
                                            _i32, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp,
                                            _vp]
_lib.mla_decompress_k_paged_fp8.restype = ctypes.c_int
_lib.mla_decompress_k_paged_fp8_qcache.argtypes = [ctypes.POINTER(_CQuantCache), _u32, _vp, _vp,
                                                   _i32, _i32, _vp, _vp, _i32, _vp, _vp, _vp,
                                                   _sz, _vp, _vp]
_lib.mla_decompress_k_paged_fp8_qcache.restype = ctypes.c_int
_lib.mla_cache_write_paged_qcache.argtypes = [_vp, _vp, _i32, _i32, _vp, ctypes.c_float, _vp,
                                              _i32, ctypes.POINTER(_CQuantCache), _u32, _vp, _vp]
_lib.mla_cache_write_paged_qcache.restype = ctypes.c_int
_lib.mla_decompress_kv_paged.argtypes = [ctypes.POINTER(_CCache), _u32, _vp, _vp, _i32, _i32, _i32,
                                         _i32, _vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp]
_lib.mla_decompress_kv_paged.restype = ctypes.c_int
_lib.mla_decompress_kv_paged_fp8.argtypes = [ctypes.POINTER(_CCache), _u32, _vp, _vp, _i32, _i32,
                                             _i32, _i32, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _vp,
                                             _vp, _vp, _vp, _sz, _vp, _vp]
_lib.mla_decompress_kv_paged_fp8.restype = ctypes.c_int
_lib.mla_cache_write_paged.argtypes = [_vp, _vp, _i32, _i32, _i32, _i32, _vp, ctypes.c_float, _vp,
                                       _i32, ctypes.POINTER(_CCache), _u32, _vp, _vp]
_lib.mla_cache_write_paged.restype = ctypes.c_int
_lib.kv_matmul_paged_fp8_workspace_size.argtypes = [_i32, _i32]
_lib.kv_matmul_paged_fp8_workspace_size.restype = _sz
_lib.kv_matmul_paged_fp8.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32,
                                     ctypes.POINTER(_CCache), _u32, _vp, _sz, _vp, _vp]
_lib.kv_matmul_paged_fp8.restype = ctypes.c_int
_lib.kv_matmul_paged.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _i32, ctypes.POINTER(_CCache),
                                 _u32, _vp, _vp]
_lib.kv_matmul_paged.restype = ctypes.c_int
_lib.mla_decompress_k_paged_fp8_noalloc.argtypes = [ctypes.POINTER(_CCache), _u32, _vp, _vp, _i32,
                                                    _i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp,
                                                    _vp, _vp]
_lib.mla_decompress_k_paged_fp8_noalloc.restype = ctypes.c_int
FP8_NOALLOC_SCRATCH_BYTES = 16 << 20
_lib.pkm_check_wait_timeout.argtypes = [_vp, _u32, _vp]
_lib.pkm_check_wait_timeout.restype = ctypes.c_int
_lib.pkm_validate_row_offsets.argtypes = [_vp, _i32, _vp, _vp]
_lib.pkm_validate_row_offsets.restype = ctypes.c_int


def status_string(code: int) -> str:
    return _lib.pkm_status_string(int(code)).decode()


def last_cuda_error() -> str:
    """What lies behind the last PKM_ERR_CUDA the library returned on this thread."""
    return _lib.pkm_last_cuda_error().decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return int(t)
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


@dataclass
class PagedCache:
    """A paged cache (all layers) described by element strides; see pkm_paged_cache.

    data: bf16 storage (any shape; only its base pointer is used).
    page_table: uint32/int32 [batch, max_pages_per_seq].
    cache_lengths: uint32/int32 [batch] (kv_matmul_paged only).
    """
    data: torch.Tensor
    page_table: torch.Tensor
    layer_stride: int
    page_stride: int
    slot_stride: int
    num_layers: int
    num_pages: int
    page_size: int
    row_elems: int
    kv_stride: int = 0
    cache_lengths: Optional[torch.Tensor] = None

    def c_struct(self) -> _CCache:
        return _CCache(self.data.data_ptr(), int(self.layer_stride), int(self.page_stride),
                       int(self.slot_stride), int(self.kv_stride), int(self.num_layers),
                       int(self.num_pages), int(self.page_size), int(self.row_elems),
                       self.page_table.data_ptr(), int(self.page_table.shape[-1]),
                       _ptr(self.cache_lengths))


@dataclass
class QuantCache:
    """A quantised paged latent cache described by byte strides; see pkm_quant_cache.

    data: storage of the slots (any dtype and shape; only its base pointer is used).  A slot
    holds kv_lora_rank e4m3 codes, rope_dim bf16 values and kv_lora_rank/128 fp32 scales.
    """
    data: torch.Tensor
    page_table: torch.Tensor
    layer_stride: int
    page_stride: int
    slot_stride: int
    num_layers: int
    num_pages: int
    page_size: int
    kv_lora_rank: int
    rope_dim: int
    cache_lengths: Optional[torch.Tensor] = None

    def c_struct(self) -> _CQuantCache:
        return _CQuantCache(self.data.data_ptr(), int(self.layer_stride), int(self.page_stride),
                            int(self.slot_stride), int(self.num_layers), int(self.num_pages),
                            int(self.page_size), int(self.kv_lora_rank), int(self.rope_dim),
                            self.page_table.data_ptr(), int(self.page_table.shape[-1]),
                            _ptr(self.cache_lengths))


def _check(code: int, where: str, check: bool) -> int:
    if check and code != PKM_OK:
        raise PkmError(code, where)
    return code


def mla_decompress_k_paged(cache: PagedCache, layer_idx: int, buffer_row_offsets: torch.Tensor,
                           cache_offsets: torch.Tensor, buffer_length: int, kv_lora_rank: int,
                           rope_dim: int, w_k: torch.Tensor, k_latent_buffer: torch.Tensor,
                           k_buffer: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                           stream=None, check: bool = True) -> int:
    c = cache.c_struct()
    batch = int(buffer_row_offsets.shape[0]) - 1
    code = _lib.mla_decompress_k_paged(ctypes.byref(c), int(layer_idx), _ptr(buffer_row_offsets),
                                       _ptr(cache_offsets), batch, int(buffer_length),
                                       int(kv_lora_rank), int(rope_dim), _ptr(w_k),
                                       int(w_k.shape[0]), _ptr(k_latent_buffer), _ptr(k_buffer),
                                       _ptr(dev_status), _stream(stream))
    return _check(code, "mla_decompress_k_paged", check)


def mla_decompress_kv_paged(cache: PagedCache, layer_idx: int, buffer_row_offsets: torch.Tensor,
                            cache_offsets: torch.Tensor, buffer_length: int, kv_lora_rank: int,
                            rope_dim: int, w_k: torch.Tensor, w_uv: torch.Tensor,
                            k_latent_buffer: torch.Tensor, k_buffer: torch.Tensor,
                            v_buffer: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                            stream=None, check: bool = True) -> int:
    """K and V from one gather; w_uv is [num_heads, v_head_dim, kv_lora_rank]."""
    c = cache.c_struct()
    batch = int(buffer_row_offsets.shape[0]) - 1
    code = _lib.mla_decompress_kv_paged(ctypes.byref(c), int(layer_idx), _ptr(buffer_row_offsets),
                                        _ptr(cache_offsets), batch, int(buffer_length),
                                        int(kv_lora_rank), int(rope_dim), _ptr(w_k),
                                        int(w_k.shape[0]), _ptr(w_uv), int(w_uv.shape[0]),
                                        int(w_uv.shape[1]), _ptr(k_latent_buffer), _ptr(k_buffer),
                                        _ptr(v_buffer), _ptr(dev_status), _stream(stream))
    return _check(code, "mla_decompress_kv_paged", check)


def mla_decompress_k_paged_fp8_workspace_size(buffer_length: int, kv_lora_rank: int) -> int:
    return int(_lib.mla_decompress_k_paged_fp8_workspace_size(int(buffer_length), int(kv_lora_rank)))


def fp8_workspace_views(workspace: torch.Tensor, buffer_length: int, kv_lora_rank: int):
    """(q_latent [L, R] uint8, q_scale [L, R/128] float32) views of an FP8 workspace."""
    L, R = int(buffer_length), int(kv_lora_rank)
    q = workspace[: L * R].view(L, R)
    off = (L * R + 255) // 256 * 256
    s = workspace[off: off + L * (R // 128) * 4].view(torch.float32).view(L, R // 128)
    return q, s


def mla_decompress_k_paged_fp8(cache: PagedCache, layer_idx: int,
                               buffer_row_offsets: torch.Tensor, cache_offsets: torch.Tensor,
                               buffer_length: int, kv_lora_rank: int, rope_dim: int,
                               w_k_e4m3: torch.Tensor, w_k_scale: torch.Tensor,
                               k_latent_buffer: torch.Tensor, k_buffer: torch.Tensor,
                               workspace: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                               stream=None, check: bool = True) -> int:
    c = cache.c_struct()
    batch = int(buffer_row_offsets.shape[0]) - 1
    code = _lib.mla_decompress_k_paged_fp8(
        ctypes.byref(c), int(layer_idx), _ptr(buffer_row_offsets), _ptr(cache_offsets), batch,
        int(buffer_length), int(kv_lora_rank), int(rope_dim), _ptr(w_k_e4m3), _ptr(w_k_scale),
        int(w_k_e4m3.shape[0]), _ptr(k_latent_buffer), _ptr(k_buffer), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    return _check(code, "mla_decompress_k_paged_fp8", check)


def mla_decompress_k_paged_fp8_qcache(cache: QuantCache, layer_idx: int,
                                      buffer_row_offsets: torch.Tensor, cache_offsets: torch.Tensor,
                                      buffer_length: int, w_k_e4m3: torch.Tensor,
                                      w_k_scale: torch.Tensor, k_latent_buffer: Optional[torch.Tensor],
                                      k_buffer: torch.Tensor, workspace: torch.Tensor,
                                      dev_status: Optional[torch.Tensor] = None, stream=None,
                                      check: bool = True) -> int:
    """FP8 decompress reading codes and scales straight from a quantised cache;
    k_latent_buffer (dequantised bf16 rows) may be None."""
    c = cache.c_struct()
    batch = int(buffer_row_offsets.shape[0]) - 1
    code = _lib.mla_decompress_k_paged_fp8_qcache(
        ctypes.byref(c), int(layer_idx), _ptr(buffer_row_offsets), _ptr(cache_offsets), batch,
        int(buffer_length), _ptr(w_k_e4m3), _ptr(w_k_scale), int(w_k_e4m3.shape[0]),
        _ptr(k_latent_buffer), _ptr(k_buffer), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    return _check(code, "mla_decompress_k_paged_fp8_qcache", check)


def mla_cache_write_paged_qcache(latent: torch.Tensor, input_row_offsets: torch.Tensor,
                                 kv_norm_gamma: torch.Tensor, epsilon: float,
                                 freqs_cis: torch.Tensor, cache: QuantCache, layer_idx: int,
                                 dev_status: Optional[torch.Tensor] = None, stream=None,
                                 check: bool = True) -> int:
    """RMSNorm + RoPE of new latent rows, quantised into a quantised cache's slots."""
    c = cache.c_struct()
    batch = int(input_row_offsets.shape[0]) - 1
    code = _lib.mla_cache_write_paged_qcache(_ptr(latent), _ptr(input_row_offsets), batch,
                                             int(latent.shape[0]), _ptr(kv_norm_gamma),
                                             float(epsilon), _ptr(freqs_cis),
                                             int(freqs_cis.shape[0]), ctypes.byref(c),
                                             int(layer_idx), _ptr(dev_status), _stream(stream))
    return _check(code, "mla_cache_write_paged_qcache", check)


def mla_decompress_kv_paged_fp8(cache: PagedCache, layer_idx: int,
                                buffer_row_offsets: torch.Tensor, cache_offsets: torch.Tensor,
                                buffer_length: int, kv_lora_rank: int, rope_dim: int,
                                w_k_e4m3: torch.Tensor, w_k_scale: torch.Tensor,
                                w_uv_e4m3: torch.Tensor, w_uv_scale: torch.Tensor,
                                k_latent_buffer: torch.Tensor, k_buffer: torch.Tensor,
                                v_buffer: torch.Tensor, workspace: torch.Tensor,
                                dev_status: Optional[torch.Tensor] = None, stream=None,
                                check: bool = True) -> int:
    """FP8 K and V from one gather and one activation quantisation."""
    c = cache.c_struct()
    batch = int(buffer_row_offsets.shape[0]) - 1
    code = _lib.mla_decompress_kv_paged_fp8(
        ctypes.byref(c), int(layer_idx), _ptr(buffer_row_offsets), _ptr(cache_offsets), batch,
        int(buffer_length), int(kv_lora_rank), int(rope_dim), _ptr(w_k_e4m3), _ptr(w_k_scale),
        int(w_k_e4m3.shape[0]), _ptr(w_uv_e4m3), _ptr(w_uv_scale), int(w_uv_e4m3.shape[0]),
        int(w_uv_e4m3.shape[1]), _ptr(k_latent_buffer), _ptr(k_buffer), _ptr(v_buffer),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status),
        _stream(stream))
    return _check(code, "mla_decompress_kv_paged_fp8", check)


def mla_cache_write_paged(latent: torch.Tensor, input_row_offsets: torch.Tensor,
                          kv_norm_gamma: torch.Tensor, epsilon: float, freqs_cis: torch.Tensor,
                          cache: PagedCache, layer_idx: int, kv_lora_rank: int, rope_dim: int,
                          dev_status: Optional[torch.Tensor] = None, stream=None,
                          check: bool = True) -> int:
    """RMSNorm + RoPE of new latent rows [total_rows, R + P] into the paged latent cache."""
    c = cache.c_struct()
    batch = int(input_row_offsets.shape[0]) - 1
    code = _lib.mla_cache_write_paged(_ptr(latent), _ptr(input_row_offsets), batch,
                                      int(latent.shape[0]), int(kv_lora_rank), int(rope_dim),
                                      _ptr(kv_norm_gamma), float(epsilon), _ptr(freqs_cis),
                                      int(freqs_cis.shape[0]), ctypes.byref(c), int(layer_idx),
                                      _ptr(dev_status), _stream(stream))
    return _check(code, "mla_cache_write_paged", check)


def kv_matmul_paged_fp8_workspace_size(total_rows: int, k_in: int) -> int:
    return int(_lib.kv_matmul_paged_fp8_workspace_size(int(total_rows), int(k_in)))


def kv_matmul_paged_fp8(hidden_state: torch.Tensor, input_row_offsets: torch.Tensor,
                        w_e4m3: torch.Tensor, w_scale: torch.Tensor, kv_cache: PagedCache,
                        layer_idx: int, workspace: torch.Tensor,
                        dev_status: Optional[torch.Tensor] = None, stream=None,
                        check: bool = True) -> int:
    """FP8 kv_matmul: hidden_state bf16 [M, k_in], w_e4m3 [n_out, k_in] with fp32 block scales
    [n_out/128, k_in/128]; the quantised rows land in `workspace`."""
    c = kv_cache.c_struct()
    batch = int(input_row_offsets.shape[0]) - 1
    code = _lib.kv_matmul_paged_fp8(_ptr(hidden_state), _ptr(input_row_offsets), batch,
                                    int(hidden_state.shape[0]), int(hidden_state.shape[1]),
                                    _ptr(w_e4m3), _ptr(w_scale), int(w_e4m3.shape[0]),
                                    ctypes.byref(c), int(layer_idx), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _ptr(dev_status), _stream(stream))
    return _check(code, "kv_matmul_paged_fp8", check)


def mla_decompress_k_paged_fp8_noalloc(cache: PagedCache, layer_idx: int,
                                       buffer_row_offsets: torch.Tensor,
                                       cache_offsets: torch.Tensor, buffer_length: int,
                                       kv_lora_rank: int, rope_dim: int, w_k_e4m3: torch.Tensor,
                                       w_k_scale: torch.Tensor, k_latent_buffer: torch.Tensor,
                                       k_buffer: torch.Tensor,
                                       dev_status: Optional[torch.Tensor] = None, stream=None,
                                       check: bool = True) -> int:
    """The FP8 decompress without a caller workspace, for callers that cannot allocate
    device memory: the library's fixed 16 MiB device array holds the quantised latent."""
    c = cache.c_struct()
    batch = int(buffer_row_offsets.shape[0]) - 1
    code = _lib.mla_decompress_k_paged_fp8_noalloc(
        ctypes.byref(c), int(layer_idx), _ptr(buffer_row_offsets), _ptr(cache_offsets), batch,
        int(buffer_length), int(kv_lora_rank), int(rope_dim), _ptr(w_k_e4m3), _ptr(w_k_scale),
        int(w_k_e4m3.shape[0]), _ptr(k_latent_buffer), _ptr(k_buffer), _ptr(dev_status),
        _stream(stream))
    return _check(code, "mla_decompress_k_paged_fp8_noalloc", check)


def kv_matmul_paged(hidden_state: torch.Tensor, input_row_offsets: torch.Tensor,
                    weight: torch.Tensor, kv_cache: PagedCache, layer_idx: int,
                    dev_status: Optional[torch.Tensor] = None, stream=None,
                    check: bool = True) -> int:
    c = kv_cache.c_struct()
    batch = int(input_row_offsets.shape[0]) - 1
    code = _lib.kv_matmul_paged(_ptr(hidden_state), _ptr(input_row_offsets), batch,
                                int(hidden_state.shape[0]), int(hidden_state.shape[1]),
                                _ptr(weight), int(weight.shape[1]), ctypes.byref(c),
                                int(layer_idx), _ptr(dev_status), _stream(stream))
    return _check(code, "kv_matmul_paged", check)


def pkm_check_wait_timeout(dev_status: torch.Tensor, timeout_ms: int, stream=None,
                           check: bool = True) -> int:
    code = _lib.pkm_check_wait_timeout(_ptr(dev_status), int(timeout_ms), _stream(stream))
    return _check(code, "pkm_check_wait_timeout", check)


__all__ = ["pkm_check_wait_timeout", "mla_decompress_k_paged_fp8_noalloc",
           "FP8_NOALLOC_SCRATCH_BYTES", "PagedCache", "PkmError", "mla_decompress_k_paged", "mla_decompress_k_paged_fp8",
           "mla_decompress_k_paged_fp8_workspace_size", "fp8_workspace_views", "kv_matmul_paged",
           "status_string", "LIB_PATH", "PKM_OK", "PKM_ERR_INVALID_ARG", "PKM_ERR_UNSUPPORTED",
           "PKM_ERR_CUDA", "PKM_ERR_OUT_OF_RANGE", "PKM_ERR_TIMEOUT"]


def pkm_validate_row_offsets(offsets: torch.Tensor, dev_status: torch.Tensor, stream=None,
                             check: bool = True) -> int:
    """Merges PKM_ERR_INVALID_ARG into dev_status when the offset array (batch + 1 entries)
    decreases somewhere; writes nothing else."""
    code = _lib.pkm_validate_row_offsets(_ptr(offsets), int(offsets.shape[0]) - 1,
                                         _ptr(dev_status), _stream(stream))
    return _check(code, "pkm_validate_row_offsets", check)
