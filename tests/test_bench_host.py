"""Host logic of bench.py's CPU legs (no GPU): the all-cores oracle splits a workload into
windows of consecutive rows, each a sub-problem of its own (buffer_row_offsets clipped and
shifted, cache_offsets advanced).  Those windows must reproduce, bit for bit, the rows one
oracle call over the whole buffer computes, and the process pool must cover every row it is
given exactly once."""
from __future__ import annotations

import os
import sys

import numpy as np

import workloads
from util import oracle_decompress

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    # imported by name: the pool's spawned workers import the same module to find their
    # entry points
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    return bench


def _problem():
    # five requests, one of them empty, rows starting mid-page, pages shuffled
    return workloads.make_decompress("windows", 1201, [40, 0, 75, 9, 66], [3, 0, 10, 0, 1], 16,
                                     64, 16, 128)


def test_row_windows_reproduce_the_whole_buffer():
    import oracle
    from util import cache_view
    bench = _bench()
    d = _problem()
    L = d.buffer_length
    st, lat, kb, written = oracle_decompress(d)
    assert st == 0 and written.all()
    for start, rows in [(0, 7), (7, 30), (37, 60), (97, L - 97), (L - 5, 5), (20, 1)]:
        sub_bro, sub_co = bench._sub_problem(d, start, rows)
        s2, lat2, kb2, w2 = oracle.decompress_k(cache_view(d), d.layer_idx, sub_bro, sub_co,
                                                d.batch, rows, d.kv_lora_rank, d.rope_dim, d.w_k)
        assert s2 == 0 and w2.all()
        assert np.array_equal(lat2, lat[start:start + rows])
        assert np.array_equal(kb2, kb[start:start + rows])


def test_oracle_pool_covers_each_row_once():
    bench = _bench()
    d = _problem()
    pool = bench.OraclePool(d, workers=2)
    try:
        rows, wall, busy = pool.run(0, d.buffer_length // 2)
        assert rows == 2 * (d.buffer_length // 2)
        rows, _, _ = pool.run(d.buffer_length - 4, 2)
        assert rows == 4
    finally:
        pool.close()


def test_roofline_rows_recompute_from_their_own_fields():
    """Each bench row's roofline object is recomputable from the fields it carries: the
    bound is the slower of FLOPs at the tensor peak and algorithmic bytes at the HBM peak,
    `achieved` is that unit's rate over the row's device time and `frac` = achieved / peak."""
    import bench
    peaks = {"hbm_gbs": 6775.3}
    # a tensor-bound row (the bf16 decompress shape) and an HBM-bound row (a cache write)
    for flop, nbytes, t in [(4.486e14, 9.545e8, 2.64e-4), (0.0, 1.456e8, 4.1e-5),
                            (4.486e14, 9.47e8, 2.65e-4)]:
        r = bench.roofline_row(["k"], t, flop, nbytes, peaks, 1933.3, "measured burst")
        t_tensor = flop / (1933.3e12) if flop else 0.0
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
        assert r["bound"] == ("tensor" if t_tensor >= t_hbm else "hbm")
        rate = flop / r["ms"] * 1e3 / 1e12 if r["bound"] == "tensor" else nbytes / r["ms"] * 1e3 / 1e9
        assert abs(r["achieved"] - rate) <= 1e-9 * rate
        assert abs(r["frac"] - r["achieved"] / r["peak"]) <= 1e-12
        assert r["unit"] == ("TFLOP/s" if r["bound"] == "tensor" else "GB/s")
        assert abs(r["hbm_frac"] - nbytes / t / 1e9 / peaks["hbm_gbs"]) <= 1e-12
