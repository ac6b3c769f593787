"""The quantisers' scales and e4m3 codes (E4m3Block: the scale by a corrected constant
reciprocal, the quotients by an approximate reciprocal per 128-value block and one remainder
correction, correctly rounded division for blocks below 2^-100) against CUDA's correctly
rounded fp32 division, exhaustively over the inputs they see: every bf16 x with |x| <= amax,
every positive finite bf16 amax.  The scales must equal RN(amax / 448) and the codes those of
RN(x / s) for every pair, so every quantised output equals what the method and the oracle
state; the corrected quotient itself may miss RN(x / s) by an ulp where that changes no
code."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_division_matches_the_correctly_rounded_quotient_for_every_bf16_input(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    so = str(tmp_path / "div_check.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "paged_kv_mla_gb300", "csrc"),
                    os.path.join(HERE, "native", "div_check.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    counts = (ctypes.c_ulonglong * 4)()
    first = (ctypes.c_uint32 * 5)()
    assert lib.pkm_div_check(counts, first) == 0
    pairs, off_q, bad_code, bad_scale = counts[0], counts[1], counts[2], counts[3]
    assert pairs > 5e8
    assert off_q < pairs // 20           # the corrected quotient is an ulp off rarely
    assert bad_scale == 0, f"{bad_scale} scales differ from RN(amax / 448)"
    assert bad_code == 0, (
        f"{bad_code} code mismatches; first at amax bits "
        f"{first[1]:#06x}, x bits {first[2]:#06x}; amax bits of mismatches in "
        f"[{first[3]:#06x}, {first[4]:#06x}]")
