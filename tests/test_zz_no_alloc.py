"""The allocation-free FP8 decompress (mla_decompress_k_paged_fp8_noalloc) against the
regular FP8 entry point.

The no-alloc call is for callers that cannot allocate device memory (an engine plug-in that
only receives pre-planned buffers, a serving loop that must not call cudaMalloc); it keeps
its quantised latent in a fixed device array inside the library.  Both calls run the same
deterministic kernels on the same inputs, so its outputs must equal those of
mla_decompress_k_paged_fp8 with a caller workspace bit for bit, on two calls in a row (the
second call reuses the array the first one left behind); once, they are also checked against
the CPU oracle.  This file is collected last so a stop-at-first-failure run has already run
every other test; it also passes alone in a fresh process."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from gpu_util import FP8_TOL, DeviceDecompress, _i16, assert_close_bf16, host_u16
from util import oracle_decompress_fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_mla_gb300  # noqa: F401


def _noalloc_run(g: DeviceDecompress):
    import paged_kv_mla_gb300 as pkm
    d = g.d
    lat = torch.full_like(g.k_latent, _i16(workloads.SENTINEL_OUT))
    kb = torch.full_like(g.k_buffer, _i16(workloads.SENTINEL_OUT))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = pkm.mla_decompress_k_paged_fp8_noalloc(g.pc, d.layer_idx, g.bro, g.co, d.buffer_length,
                                                  d.kv_lora_rank, d.rope_dim, g.w, g.w_scale, lat,
                                                  kb, dev_status=st, check=False)
    torch.cuda.synchronize()
    L = d.buffer_length
    return code, host_u16(lat)[:L], host_u16(kb)[:L], int(st.item())


@pytest.mark.parametrize("seed,lengths,offsets,R,N", [
    (701, [300, 0, 517, 64, 129], [7, 0, 100, 0, 1], 512, 1024),
    (702, [700, 77, 41], [31, 5, 0], 256, 512),
])
def test_noalloc_matches_the_workspace_entry_point_twice(seed, lengths, offsets, R, N):
    import paged_kv_mla_gb300 as pkm
    d = workloads.make_decompress("noalloc", seed, lengths, offsets, 16, R, 64, N, fp8=True,
                                  num_layers=2, layer_idx=1, extra_pages=3)
    g = DeviceDecompress(d, fp8=True)
    g.run()
    ref_lat, ref_kb, ref_st = g.results()
    assert ref_st == 0
    for _ in range(2):
        code, lat, kb, st = _noalloc_run(g)
        assert code == pkm.PKM_OK and st == 0
        assert np.array_equal(lat, ref_lat)
        assert np.array_equal(kb, ref_kb), "no-alloc k_buffer differs from the workspace call"
    if seed == 701:  # and once against the oracle (dequantised-value fp64 product)
        ost, olat, ok, oq, os_, written = oracle_decompress_fp8(d)
        assert ost == 0
        assert np.array_equal(lat[written], olat[written])
        assert_close_bf16(kb[written], ok[written], FP8_TOL, "no-alloc k_buffer vs oracle")
        assert (kb[~written] == workloads.SENTINEL_OUT).all()


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    import paged_kv_mla_gb300 as pkm
    d = workloads.make_decompress("noalloc_big", 703, [31776], [0], 128, 512, 64, 128, fp8=True)
    assert pkm.mla_decompress_k_paged_fp8_workspace_size(31776, 512) > pkm.FP8_NOALLOC_SCRATCH_BYTES
    assert pkm.mla_decompress_k_paged_fp8_workspace_size(31775, 512) <= pkm.FP8_NOALLOC_SCRATCH_BYTES
    g = DeviceDecompress(d, fp8=True)
    code, lat, kb, st = _noalloc_run(g)
    assert code == pkm.PKM_ERR_UNSUPPORTED and st == 0
    assert (kb == workloads.SENTINEL_OUT).all() and (lat == workloads.SENTINEL_OUT).all()
