// Exhaustive check of the quantisers' scales and e4m3 codes (E4m3Block, pkm_device.cuh)
// against CUDA's correctly rounded fp32 division, on every input the quantisers can see:
// x any bf16 value with |x| <= amax, amax any positive finite bf16 value.  Counts scales
// that differ from RN(amax / 448) and codes that differ from those of RN(x / s) (both must
// be none) and, for information, the quotients of div_by_scale that differ from RN(x / s).
// Built and run by tests/test_gpu_quant_division.py; not part of the library.
#include <cstdint>
#include <cuda_runtime.h>
#include "pkm_device.cuh"

namespace {

__global__ void div_check_kernel(unsigned long long* counts, uint32_t* first_bad) {
    // blockIdx.x walks amax codes; threads walk x codes up to amax, both signs
    const uint32_t amax_bits = blockIdx.x + 1;  // 0x0001 .. 0x7F7F
    const float amax = __uint_as_float(amax_bits << 16);
    const pkm::E4m3Block qb(amax);
    const float s = qb.s;
    if (threadIdx.x == 0 && __float_as_uint(s) != __float_as_uint(__fdiv_rn(amax, 448.0f)))
        atomicAdd(&counts[3], 1ull);
    unsigned long long bad_q = 0, bad_code = 0, n = 0;
    for (uint32_t xb = threadIdx.x; xb <= amax_bits; xb += blockDim.x) {
        for (int neg = 0; neg < 2; ++neg) {
            const float x = __uint_as_float((xb | (neg ? 0x8000u : 0u)) << 16);
            const float q_ref = __fdiv_rn(x, s);
            const float q = pkm::div_by_scale(x, s, -qb.yn);
            ++n;
            const bool dq = __float_as_uint(q_ref) != __float_as_uint(q);
            const uint32_t ref = pkm::e4m3x2(q_ref, 0.0f) & 0xFFu;  // one code, in all four bytes
            const bool dc = ref * 0x01010101u != qb.codes4(x, x, x, x);
            bad_q += dq;
            bad_code += dc;
            if (dc) {
                if (atomicCAS(first_bad, 0u, 1u) == 0u) {
                    first_bad[1] = amax_bits;
                    first_bad[2] = xb | (neg ? 0x8000u : 0u);
                }
                atomicMin(&first_bad[3], amax_bits);
                atomicMax(&first_bad[4], amax_bits);
            }
        }
    }
    atomicAdd(&counts[0], n);
    atomicAdd(&counts[1], bad_q);
    atomicAdd(&counts[2], bad_code);
}

}  // namespace

// counts (host): pairs checked, div_by_scale quotients off RN(x / s), code mismatches,
// scale mismatches;
// first_bad (host): flag, amax bits and x bits of the first code mismatch, smallest and
// largest amax bits of any.  Returns a cudaError_t.
extern "C" int pkm_div_check(unsigned long long* counts, uint32_t* first_bad) {
    unsigned long long* dc = nullptr;
    uint32_t* df = nullptr;
    cudaError_t e = cudaMalloc(&dc, 4 * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMalloc(&df, 5 * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(dc, 0, 4 * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(df, 0, 3 * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(df + 3, 0xFF, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(df + 4, 0, sizeof(uint32_t));
    if (e == cudaSuccess) {
        div_check_kernel<<<0x7F7F, 256>>>(dc, df);
        e = cudaDeviceSynchronize();
    }
    if (e == cudaSuccess) e = cudaMemcpy(counts, dc, 4 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(first_bad, df, 5 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
    cudaFree(dc);
    cudaFree(df);
    return static_cast<int>(e);
}
