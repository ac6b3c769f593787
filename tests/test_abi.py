"""The C-ABI library builds, loads without a GPU, exports every function include/*.h
declares, and rejects invalid calls on the host (before any CUDA call).  No GPU."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_mla_gb300
    return ctypes.CDLL(paged_kv_mla_gb300.LIB_PATH)


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["mla_decompress_k_paged", "mla_decompress_k_paged_fp8", "mla_decompress_kv_paged",
              "mla_decompress_kv_paged_fp8", "mla_cache_write_paged",
              "mla_decompress_k_paged_fp8_qcache", "mla_cache_write_paged_qcache",
              "kv_matmul_paged_fp8", "kv_matmul_paged_fp8_workspace_size",
              "mla_decompress_k_paged_fp8_workspace_size", "kv_matmul_paged", "pkm_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings(lib):
    lib.pkm_status_string.restype = ctypes.c_char_p
    assert lib.pkm_status_string(0) == b"PKM_OK"
    assert lib.pkm_status_string(4) == b"PKM_ERR_OUT_OF_RANGE"
    assert lib.pkm_status_string(99) == b"PKM_ERR_UNKNOWN"
    lib.pkm_last_cuda_error.restype = ctypes.c_char_p
    assert lib.pkm_last_cuda_error() == b"no CUDA failure recorded"


def test_workspace_size(lib):
    f = lib.mla_decompress_k_paged_fp8_workspace_size
    f.restype = ctypes.c_size_t
    assert f(1000, 512) == 512000 + (1000 * 4 * 4 + 255) // 256 * 256
    assert f(1000, 500) == 0 and f(-1, 512) == 0
    assert f(0, 512) == 0


def _cache(pkm, **kw):
    import torch
    base = dict(data=torch.zeros(4096, dtype=torch.int16), page_table=torch.zeros(8, dtype=torch.int32),
                layer_stride=2048, page_stride=16 * 80, slot_stride=80, num_layers=1, num_pages=1,
                page_size=16, row_elems=80)
    base.update(kw)
    return pkm.PagedCache(**base)


def test_invalid_calls_return_status_without_a_gpu(lib):
    import torch
    import paged_kv_mla_gb300 as pkm
    t16 = torch.zeros(1024, dtype=torch.int16)
    bro = torch.tensor([0, 4], dtype=torch.int32)
    co = torch.zeros(2, dtype=torch.int32)
    w = torch.zeros(64 * 64, dtype=torch.int16).view(64, 64)

    def call(cache, L=4, R=64, P=16, w=w, lat=t16, kb=t16, bro=bro):
        return pkm.mla_decompress_k_paged(cache, 0, bro, co, L, R, P, w, lat, kb, stream=0,
                                          check=False)

    good = _cache(pkm)
    assert call(good, R=60, P=20) == pkm.PKM_ERR_UNSUPPORTED          # R not a multiple of 64
    assert call(good, R=576, P=0) != pkm.PKM_OK                        # row_elems mismatch
    assert call(_cache(pkm, row_elems=81), P=17) == pkm.PKM_ERR_UNSUPPORTED  # 81*2 B rows
    assert call(_cache(pkm, slot_stride=81)) == pkm.PKM_ERR_INVALID_ARG  # 16-byte rule
    assert call(_cache(pkm, num_pages=0)) == pkm.PKM_ERR_INVALID_ARG
    assert call(good, L=-1) == pkm.PKM_ERR_INVALID_ARG
    assert call(good, L=0) == pkm.PKM_OK                               # nothing to do
    assert call(good, lat=t16[1:]) == pkm.PKM_ERR_INVALID_ARG          # misaligned output
    r = pkm.kv_matmul_paged(torch.zeros(4, 100, dtype=torch.int16), bro, torch.zeros(100, 128, dtype=torch.int16),
                            _cache(pkm, row_elems=128, cache_lengths=co), 0, stream=0, check=False)
    assert r == pkm.PKM_ERR_UNSUPPORTED                                # k_in not a multiple of 64
    r = pkm.kv_matmul_paged(torch.zeros(4, 128, dtype=torch.int16), bro, torch.zeros(128, 96, dtype=torch.int16),
                            _cache(pkm, row_elems=128, cache_lengths=co), 0, stream=0, check=False)
    assert r == pkm.PKM_ERR_INVALID_ARG                                # n_out not HD or 2 HD
    r = pkm.kv_matmul_paged(torch.zeros(4, 128, dtype=torch.int16), bro, torch.zeros(128, 128, dtype=torch.int16),
                            _cache(pkm, row_elems=128), 0, stream=0, check=False)
    assert r == pkm.PKM_ERR_INVALID_ARG                                # cache_lengths missing
    with pytest.raises(pkm.PkmError):
        pkm.mla_decompress_k_paged(good, 0, bro, co, 4, 60, 20, w, t16, t16, stream=0)
    # K and V: the V operands are checked before anything launches
    wv = torch.zeros(3 * 20 * 64, dtype=torch.int16).view(3, 20, 64)  # 3 x 20 = 60 columns

    def call_kv(w_uv, L=4, v=t16):
        return pkm.mla_decompress_kv_paged(good, 0, bro, co, L, 64, 16, w, w_uv, t16, t16, v,
                                           stream=0, check=False)
    assert call_kv(wv) == pkm.PKM_ERR_UNSUPPORTED                      # H * Dv not a multiple of 64
    assert call_kv(torch.zeros(1, 64, 64, dtype=torch.int16), v=t16[1:]) == pkm.PKM_ERR_INVALID_ARG  # misaligned v
    assert call_kv(wv, L=0) == pkm.PKM_OK                              # nothing to do
    # cache write: shapes, alignment and the cache descriptor are checked before any launch
    lat = torch.zeros(4, 80, dtype=torch.int16)
    gamma = torch.ones(64, dtype=torch.float32)
    freqs = torch.zeros(32, 16, dtype=torch.float32)
    cw_cache = _cache(pkm, cache_lengths=co)

    def call_cw(cache=cw_cache, lat=lat, R=64, P=16, gamma=gamma, freqs=freqs, iro=bro):
        return pkm.mla_cache_write_paged(lat, iro, gamma, 1e-6, freqs, cache, 0, R, P, stream=0,
                                         check=False)
    assert call_cw(R=60, P=20) == pkm.PKM_ERR_UNSUPPORTED               # R not a multiple of 8
    assert call_cw(R=1032, P=16) == pkm.PKM_ERR_UNSUPPORTED             # R above 1024
    assert call_cw(R=56, P=16) == pkm.PKM_ERR_INVALID_ARG               # row_elems != R + P
    assert call_cw(cache=_cache(pkm)) == pkm.PKM_ERR_INVALID_ARG        # cache_lengths missing
    assert call_cw(gamma=torch.ones(65, dtype=torch.float32)[1:]) == pkm.PKM_ERR_INVALID_ARG  # misaligned gamma
    assert call_cw(cache=_cache(pkm, cache_lengths=co, slot_stride=81)) == pkm.PKM_ERR_INVALID_ARG
    assert call_cw(lat=lat[:0]) == pkm.PKM_OK                           # no new rows
    # quantised cache: byte strides, payload and R rules are checked on the host
    def qc(**kw):
        base = dict(data=torch.zeros(4096, dtype=torch.uint8), page_table=torch.zeros(8, dtype=torch.int32),
                    layer_stride=16 * 160, page_stride=16 * 160, slot_stride=160, num_layers=1,
                    num_pages=1, page_size=16, kv_lora_rank=128, rope_dim=8, cache_lengths=co)
        base.update(kw)
        return pkm.QuantCache(**base)
    w8 = torch.zeros(128 * 128, dtype=torch.uint8).view(128, 128)
    ws = torch.ones(1, dtype=torch.float32)
    wraw = torch.zeros((1 << 16) + 256, dtype=torch.uint8)
    wsp = wraw[(-wraw.data_ptr()) % 256:][:1 << 16]                       # 256-byte aligned

    def call_qd(cache, w=w8, kl=None, L=4):
        return pkm.mla_decompress_k_paged_fp8_qcache(cache, 0, bro, co, L, w, ws, kl, t16, wsp,
                                                     stream=0, check=False)
    assert call_qd(qc(slot_stride=144)) == pkm.PKM_ERR_INVALID_ARG      # below the 148-byte payload
    assert call_qd(qc(slot_stride=168)) == pkm.PKM_ERR_INVALID_ARG      # not a multiple of 16
    assert call_qd(qc(kv_lora_rank=64, slot_stride=96)) == pkm.PKM_ERR_UNSUPPORTED
    assert call_qd(qc(), kl=t16[1:]) == pkm.PKM_ERR_INVALID_ARG          # misaligned k_latent
    assert call_qd(qc(), L=0) == pkm.PKM_OK
    lq = torch.zeros(4, 136, dtype=torch.int16)
    fq = torch.zeros(32, 8, dtype=torch.float32)
    g128 = torch.ones(128, dtype=torch.float32)

    def call_qw(cache):
        return pkm.mla_cache_write_paged_qcache(lq, bro, g128, 1e-6, fq, cache, 0, stream=0,
                                                check=False)
    assert call_qw(qc(kv_lora_rank=256, slot_stride=272)) == pkm.PKM_ERR_INVALID_ARG  # payload 280
    assert call_qw(qc(kv_lora_rank=192, slot_stride=224)) == pkm.PKM_ERR_UNSUPPORTED  # R % 128
    assert call_qw(qc(cache_lengths=None)) == pkm.PKM_ERR_INVALID_ARG
    # FP8 kv_matmul
    assert pkm.kv_matmul_paged_fp8_workspace_size(10, 256) == 2560 + 256   # 2560 codes, 80 B scales
    assert pkm.kv_matmul_paged_fp8_workspace_size(10, 200) == 0
    kvc = _cache(pkm, row_elems=128, cache_lengths=co)
    hid = torch.zeros(4, 256, dtype=torch.int16)

    def call_kf(n_out=256, h=hid, w=None, ws_=wsp):
        w = torch.zeros(n_out, h.shape[1], dtype=torch.uint8) if w is None else w
        return pkm.kv_matmul_paged_fp8(h, bro, w, ws, kvc, 0, ws_, stream=0, check=False)
    assert call_kf(n_out=192) == pkm.PKM_ERR_INVALID_ARG                # not HD or 2 HD
    assert call_kf(h=torch.zeros(4, 192, dtype=torch.int16)) == pkm.PKM_ERR_UNSUPPORTED  # k_in % 128
    assert call_kf(ws_=wsp[:100]) == pkm.PKM_ERR_INVALID_ARG            # workspace too small
    assert call_kf(ws_=wsp[64:]) == pkm.PKM_ERR_INVALID_ARG             # workspace misaligned
    assert call_kf(h=hid[:0]) == pkm.PKM_OK                             # no rows


def test_oracle_and_product_share_no_code():
    """The oracle is test infrastructure: the CUDA sources never include or name it, and it
    never includes the library's headers."""
    for f in glob.glob(os.path.join(ROOT, "paged_kv_mla_gb300", "**", "*"), recursive=True):
        if f.endswith((".cu", ".cuh", ".h", ".py")):
            assert "oracle" not in open(f).read().lower(), f
    src = open(os.path.join(ROOT, "oracle", "pkm_oracle.c")).read()
    assert "#include \"" not in src and "paged_kv_mla" not in src


def test_noalloc_status_codes_match_the_workspace_entry_point_without_a_gpu(lib):
    """Argument errors of the allocation-free FP8 call return what mla_decompress_k_paged_fp8
    returns for the same arguments (it checks sizes first, then does nothing for an empty
    call, then checks pointers and the rank); none of these calls touches the GPU."""
    import torch
    import paged_kv_mla_gb300 as pkm
    t16 = torch.zeros(1024, dtype=torch.int16)
    raw = torch.zeros(1 << 16, dtype=torch.uint8)
    off = (-raw.data_ptr()) % 256
    ws = raw[off:off + (1 << 15)]                  # a 256-byte-aligned host stand-in
    ws_scale = torch.ones(4, dtype=torch.float32)
    co = torch.zeros(2, dtype=torch.int32)

    def both(cache, bro, L, R, P, n_out, lat=t16, kb=t16):
        w = torch.zeros(max(n_out, 0) * max(R, 1), dtype=torch.uint8).view(max(n_out, 0), max(R, 1))
        a = pkm.mla_decompress_k_paged_fp8(cache, 0, bro, co, L, R, P, w, ws_scale, lat, kb, ws,
                                           stream=0, check=False)
        b = pkm.mla_decompress_k_paged_fp8_noalloc(cache, 0, bro, co, L, R, P, w, ws_scale, lat,
                                                   kb, stream=0, check=False)
        return a, b

    one = torch.tensor([0, 4], dtype=torch.int32)
    none = torch.tensor([0], dtype=torch.int32)     # batch 0
    good = _cache(pkm)                             # row_elems 80 = 64 + 16
    cases = [
        (good, none, 4, 64, 16, 0, pkm.PKM_ERR_INVALID_ARG),    # n_out 0, nothing to do
        (good, one, 0, 0, 16, 128, pkm.PKM_ERR_INVALID_ARG),    # rank 0, no rows
        (good, one, 0, 64, -1, 128, pkm.PKM_ERR_INVALID_ARG),   # negative rope_dim
        (good, one, -1, 64, 16, 128, pkm.PKM_ERR_INVALID_ARG),  # negative length
        (good, none, 4, 64, 16, 128, pkm.PKM_OK),               # no requests
        (good, one, 0, 64, 16, 128, pkm.PKM_OK),                # no rows
        (good, one, 4, 64, 16, 128, pkm.PKM_ERR_UNSUPPORTED),   # rank not a multiple of 128
        (_cache(pkm, num_pages=0), one, 4, 64, 16, 128, pkm.PKM_ERR_INVALID_ARG),
    ]
    for cache, bro, L, R, P, n_out, want in cases:
        assert both(cache, bro, L, R, P, n_out) == (want, want), (L, R, P, n_out)
    a, b = both(good, one, 4, 64, 16, 128, kb=t16[1:])     # misaligned output
    assert a == b == pkm.PKM_ERR_INVALID_ARG


def test_offset_check_arguments_without_a_gpu(lib):
    import torch
    import paged_kv_mla_gb300 as pkm
    st = torch.zeros(1, dtype=torch.int32)
    assert pkm.pkm_validate_row_offsets(torch.zeros(1, dtype=torch.int32), st, stream=0,
                                        check=False) == pkm.PKM_OK        # batch 0
    assert lib.pkm_validate_row_offsets(None, 3, st.data_ptr(), None) == pkm.PKM_ERR_INVALID_ARG
    assert lib.pkm_validate_row_offsets(st.data_ptr(), 3, None, None) == pkm.PKM_ERR_INVALID_ARG
    assert lib.pkm_validate_row_offsets(st.data_ptr(), -1, st.data_ptr(), None) == pkm.PKM_ERR_INVALID_ARG

