"""Device-side helpers for the GPU tests: move a workload to cuda:0, call the library
through its Python binding (which calls the C ABI), and bring results back as numpy bit
patterns for comparison with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from workloads import SENTINEL_OUT, CacheWriteInputs, DecompressInputs, KvMatmulInputs

BF16_TOL = (1e-2, 2e-3)   # |gpu - ref| <= rtol * |ref| + atol, bf16 in / fp32 accumulate
FP8_TOL = (3e-2, 5e-3)    # same form, FP8 path against the dequantised-value oracle


def _i16(v: int) -> int:
    return v - 65536 if v >= 32768 else v


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy array -> device tensor with the same bytes (uint16 travels as int16, uint32 as
    int32)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(device)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def bf16_f64(a) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close_bf16(got_bits, ref_bits, tol, what=""):
    g = bf16_f64(got_bits)
    r = bf16_f64(ref_bits)
    rtol, atol = tol
    err = np.abs(g - r)
    bad = ~(err <= rtol * np.abs(r) + atol)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements outside tolerance; "
                             f"first at {tuple(idx)}: gpu {g[tuple(idx)]} oracle {r[tuple(idx)]}")


class DeviceDecompress:
    """A DecompressInputs problem resident on the GPU, with sentinel-filled outputs."""

    def __init__(self, d: DecompressInputs, fp8: bool = False, with_latent: bool = True):
        import paged_kv_mla_gb300 as pkm
        self.d = d
        self.cache = dev(d.cache)
        self.pt = dev(d.page_table)
        self.bro = dev(d.buffer_row_offsets)
        self.co = dev(d.cache_offsets)
        ls, ps, ss = d.strides
        self.with_latent = with_latent
        if d.quantised:     # a quantised cache is only read by the FP8 path
            fp8 = True
            self.qc = pkm.QuantCache(data=self.cache, page_table=self.pt, layer_stride=ls,
                                     page_stride=ps, slot_stride=ss, num_layers=d.num_layers,
                                     num_pages=d.num_pages, page_size=d.page_size,
                                     kv_lora_rank=d.kv_lora_rank, rope_dim=d.rope_dim)
        else:
            self.pc = pkm.PagedCache(data=self.cache, page_table=self.pt, layer_stride=ls,
                                     page_stride=ps, slot_stride=ss, num_layers=d.num_layers,
                                     num_pages=d.num_pages, page_size=d.page_size,
                                     row_elems=d.latent_cols)
        L = max(d.buffer_length, 1)
        self.k_latent = torch.full((L, d.latent_cols), _i16(SENTINEL_OUT), dtype=torch.int16,
                                   device="cuda")
        self.k_buffer = torch.full((L, d.n_out), _i16(SENTINEL_OUT), dtype=torch.int16,
                                   device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.fp8 = fp8
        # the V up-projection rides along when the problem carries a w_uv
        wv = d.w_uv_e4m3 if fp8 else d.w_uv
        self.w_uv = dev(wv) if wv is not None else None
        self.w_uv_scale = dev(d.w_uv_scale) if (fp8 and wv is not None) else None
        self.v_buffer = None
        if wv is not None:
            self.v_buffer = torch.full((L, wv.shape[0], wv.shape[1]), _i16(SENTINEL_OUT),
                                       dtype=torch.int16, device="cuda")
        if fp8:
            self.w = dev(d.w_k_e4m3)
            self.w_scale = dev(d.w_k_scale)
            nbytes = pkm.mla_decompress_k_paged_fp8_workspace_size(d.buffer_length, d.kv_lora_rank)
            self.workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        else:
            self.w = dev(d.w_k)

    def run(self, stream=None, check=True):
        import paged_kv_mla_gb300 as pkm
        d = self.d
        if d.quantised:
            return pkm.mla_decompress_k_paged_fp8_qcache(
                self.qc, d.layer_idx, self.bro, self.co, d.buffer_length, self.w, self.w_scale,
                self.k_latent if self.with_latent else None, self.k_buffer, self.workspace,
                dev_status=self.status, stream=stream, check=check)
        if self.w_uv is not None and self.fp8:
            return pkm.mla_decompress_kv_paged_fp8(
                self.pc, d.layer_idx, self.bro, self.co, d.buffer_length, d.kv_lora_rank,
                d.rope_dim, self.w, self.w_scale, self.w_uv, self.w_uv_scale, self.k_latent,
                self.k_buffer, self.v_buffer, self.workspace, dev_status=self.status,
                stream=stream, check=check)
        if self.w_uv is not None:
            return pkm.mla_decompress_kv_paged(
                self.pc, d.layer_idx, self.bro, self.co, d.buffer_length, d.kv_lora_rank,
                d.rope_dim, self.w, self.w_uv, self.k_latent, self.k_buffer, self.v_buffer,
                dev_status=self.status, stream=stream, check=check)
        if self.fp8:
            return pkm.mla_decompress_k_paged_fp8(
                self.pc, d.layer_idx, self.bro, self.co, d.buffer_length, d.kv_lora_rank,
                d.rope_dim, self.w, self.w_scale, self.k_latent, self.k_buffer, self.workspace,
                dev_status=self.status, stream=stream, check=check)
        return pkm.mla_decompress_k_paged(self.pc, d.layer_idx, self.bro, self.co, d.buffer_length,
                                          d.kv_lora_rank, d.rope_dim, self.w, self.k_latent,
                                          self.k_buffer, dev_status=self.status, stream=stream,
                                          check=check)

    def results(self):
        torch.cuda.synchronize()
        L = self.d.buffer_length
        return (host_u16(self.k_latent)[:L], host_u16(self.k_buffer)[:L],
                int(self.status.item()))

    def v_results(self):
        torch.cuda.synchronize()
        return host_u16(self.v_buffer)[:self.d.buffer_length]

    def fp8_workspace(self):
        import paged_kv_mla_gb300 as pkm
        q, s = pkm.fp8_workspace_views(self.workspace, self.d.buffer_length, self.d.kv_lora_rank)
        return q.cpu().numpy(), s.cpu().numpy()


class DeviceKvMatmul:
    def __init__(self, k: KvMatmulInputs):
        import paged_kv_mla_gb300 as pkm
        self.k = k
        self.hidden = dev(k.hidden_state)
        self.iro = dev(k.input_row_offsets)
        if k.fp8:
            self.weight = dev(k.w_e4m3)
            self.w_scale = dev(k.w_scale)
            nbytes = pkm.kv_matmul_paged_fp8_workspace_size(k.total_rows, k.k_in)
            self.workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        else:
            self.weight = dev(k.weight)
        self.cache = dev(k.cache)
        self.pt = dev(k.page_table)
        self.cl = dev(k.cache_lengths)
        ls, ps, ss, kvs = k.strides
        self.pc = pkm.PagedCache(data=self.cache, page_table=self.pt, layer_stride=ls,
                                 page_stride=ps, slot_stride=ss, num_layers=k.cache.shape[0],
                                 num_pages=k.num_pages, page_size=k.page_size,
                                 row_elems=k.head_elems, kv_stride=kvs, cache_lengths=self.cl)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self, stream=None, check=True):
        import paged_kv_mla_gb300 as pkm
        if self.k.fp8:
            return pkm.kv_matmul_paged_fp8(self.hidden, self.iro, self.weight, self.w_scale, self.pc,
                                           self.k.layer_idx, self.workspace,
                                           dev_status=self.status, stream=stream, check=check)
        return pkm.kv_matmul_paged(self.hidden, self.iro, self.weight, self.pc, self.k.layer_idx,
                                   dev_status=self.status, stream=stream, check=check)

    def quantised_rows(self):
        """(codes [M, k_in], scales [M, k_in/128]) from the FP8 workspace (which holds the
        scales k-block-major)."""
        torch.cuda.synchronize()
        M, K = self.k.total_rows, self.k.k_in
        ws = self.workspace.cpu().numpy()
        q = ws[:M * K].reshape(M, K)
        off = (M * K + 255) // 256 * 256
        s = ws[off:off + M * (K // 128) * 4].view(np.float32).reshape(K // 128, M).T.copy()
        return q, s

    def results(self):
        torch.cuda.synchronize()
        return host_u16(self.cache).reshape(self.k.cache.shape), int(self.status.item())


class DeviceCacheWrite:
    def __init__(self, c: CacheWriteInputs):
        import paged_kv_mla_gb300 as pkm
        self.c = c
        self.latent = dev(c.latent)
        self.iro = dev(c.input_row_offsets)
        self.gamma = torch.from_numpy(c.gamma).cuda()
        self.freqs = torch.from_numpy(np.ascontiguousarray(c.freqs_cis)).cuda()
        self.cache = dev(c.cache)
        self.pt = dev(c.page_table)
        self.cl = dev(c.cache_lengths)
        ls, ps, ss = c.strides
        if c.quantised:
            self.qc = pkm.QuantCache(data=self.cache, page_table=self.pt, layer_stride=ls,
                                     page_stride=ps, slot_stride=ss, num_layers=c.cache.shape[0],
                                     num_pages=c.num_pages, page_size=c.page_size,
                                     kv_lora_rank=c.kv_lora_rank, rope_dim=c.rope_dim,
                                     cache_lengths=self.cl)
        else:
            self.pc = pkm.PagedCache(data=self.cache, page_table=self.pt, layer_stride=ls,
                                     page_stride=ps, slot_stride=ss, num_layers=c.cache.shape[0],
                                     num_pages=c.num_pages, page_size=c.page_size,
                                     row_elems=c.row_elems, cache_lengths=self.cl)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self, stream=None, check=True):
        import paged_kv_mla_gb300 as pkm
        c = self.c
        if c.quantised:
            return pkm.mla_cache_write_paged_qcache(self.latent, self.iro, self.gamma, c.epsilon,
                                                    self.freqs, self.qc, c.layer_idx,
                                                    dev_status=self.status, stream=stream,
                                                    check=check)
        return pkm.mla_cache_write_paged(self.latent, self.iro, self.gamma, c.epsilon, self.freqs,
                                         self.pc, c.layer_idx, c.kv_lora_rank, c.rope_dim,
                                         dev_status=self.status, stream=stream, check=check)

    def results(self):
        torch.cuda.synchronize()
        out = self.cache.cpu().numpy() if self.c.quantised else host_u16(self.cache)
        return out.reshape(self.c.cache.shape), int(self.status.item())
