#!/usr/bin/env python3
"""Runs one hot-path entry point a few times on a named seeded workload, for profiler
captures (ncu) of a single kernel on a known case.  Exits 0 when every call returned
PKM_OK and the device status word stayed 0.

  python tests/profile_case.py --workload deepseek_v3_bf16_decompress --launches 4
"""
from __future__ import annotations

import argparse
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)


def main():
    import torch
    import workloads
    from gpu_util import DeviceCacheWrite, DeviceDecompress, DeviceKvMatmul

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="deepseek_v3_bf16_decompress",
                    choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--launches", type=int, default=4)
    args = ap.parse_args()
    w = workloads.WORKLOADS[args.workload]()
    if args.workload.startswith("kv_matmul"):
        g = DeviceKvMatmul(w)
    elif args.workload.startswith("cache_write"):
        g = DeviceCacheWrite(w)
    else:
        g = DeviceDecompress(w, fp8=w.w_k_e4m3 is not None)
    for _ in range(args.launches):
        g.run()
    torch.cuda.synchronize()
    status = int(g.status.item())
    print(f"{args.workload}: {args.launches} calls, device status {status}")
    sys.exit(0 if status == 0 else 1)


if __name__ == "__main__":
    main()
