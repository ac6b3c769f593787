// decompress_fp8.cu -- FP8 block-scaled latent-K decompress.
//
// The K-decompress stage of mla_prefill_decode_graph_fp8 (Modular MAX,
// attention/gpu/mla_graph): Parameters fp8_dtype / fp8_scale_dtype and
// m/n/k_scale_granularity, Args buffer_row_offsets, cache_offsets, buffer_length, w_k
// ([num_heads * qk_nope_head_dim, kv_latent_dim], e4m3) and w_k_scale.  Granularities
// m = 1, n = k = 128.
//
// Two kernels:
//   1. fp8_gather_quantize_kernel: one warp per output row resolves the row through the
//      page table, copies the bf16 latent row to k_latent_buffer with 16-byte vector
//      loads/stores, and quantises its first kv_lora_rank columns per 128-column block
//      (s = amax / 448, q = e4m3_rne_satfinite(x / s), fp32) into the workspace.  Every
//      row is quantised exactly once, however many n tiles later consume it.
//   2. decompress_fp8_gemm_kernel: persistent CTAs over 128 x 128 output tiles (one n
//      tile = one weight-scale block).  TMA brings the quantised A tile (resident for the
//      CTA's range segment) and W_k blocks of 128 x 128 e4m3 through an 8-stage ring;
//      tcgen05.mma kind::f8f6f4 accumulates each 128-wide k-block into its own TMEM
//      accumulator (4 x 128 columns), and 8 epilogue warps combine them in registers as
//      sum_kb (s_a[row, kb] * s_w[n_tile, kb]) * acc_kb before rounding to bf16 and
//      TMA-storing k_buffer.  An accumulator is released as soon as the epilogue has read
//      it, so the next tile's MMAs overlap the rest of the epilogue.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

// ------------------------------------------------------------------------------------
// 1. gather + quantise
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;  // lo in the low byte
}

__global__ void __launch_bounds__(256)
    fp8_gather_quantize_kernel(const DecompressArgs a, const Fp8Extra x) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t row_end = decompress_row_end(a);
    const int R = a.kv_lora_rank;
    const int C = a.latent_cols;
    const int nope_chunks = R / 8;
    const int all_chunks = C / 8;
    const int kblocks = R / 128;
    for (int64_t r = warp_id; r < row_end; r += nwarps) {
        const int64_t off = decompress_row_source(a, r, row_end);
        if (off < 0) {
            if (off == -2 && lane == 0) report(a.status, PKM_ERR_OUT_OF_RANGE);
            continue;
        }
        const uint16_t* src = a.cache_layer + off;
        uint16_t* lat = a.k_latent + r * C;
        uint8_t* qrow = x.q_latent + r * R;
        for (int base = 0; base < nope_chunks; base += 32) {
            const int c = base + lane;
            const bool active = c < nope_chunks;
            const uint4 v = active ? ld_nc_v4(src + c * 8) : make_uint4(0u, 0u, 0u, 0u);
            if (active) st_v4(lat + c * 8, v);
            float f[8];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
            // one 128-column block = 16 chunks = one half-warp
#pragma unroll
            for (int sh = 8; sh >= 1; sh >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
            const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
            if (active) {
                uint32_t lo = e4m3x2(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s)) |
                              (e4m3x2(__fdiv_rn(f[2], s), __fdiv_rn(f[3], s)) << 16);
                uint32_t hi = e4m3x2(__fdiv_rn(f[4], s), __fdiv_rn(f[5], s)) |
                              (e4m3x2(__fdiv_rn(f[6], s), __fdiv_rn(f[7], s)) << 16);
                *reinterpret_cast<uint2*>(qrow + c * 8) = make_uint2(lo, hi);
                if ((lane & 15) == 0) x.q_scale[r * kblocks + c / 16] = s;
            }
        }
        for (int c = nope_chunks + lane; c < all_chunks; c += 32)
            st_v4(lat + c * 8, ld_nc_v4(src + c * 8));
    }
}

// ------------------------------------------------------------------------------------
// 2. block-scaled GEMM
// ------------------------------------------------------------------------------------

constexpr int kThreads = 320;                 // producer, MMA, 8 epilogue warps
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kKBMax = 4;                     // kv_lora_rank <= 512
constexpr int kABlockBytes = kBM * 128;       // 128 rows x 128 e4m3
constexpr int kStages = 8;
constexpr int kBStageBytes = kBN * 128;
constexpr int kEpiWarps = 8;
constexpr int kOutBufBytes = 32 * 128;
constexpr uint32_t kTmemCols = 512;           // kKBMax accumulators x 128 columns

struct Bars {
    uint64_t b_full[kStages];
    uint64_t b_empty[kStages];
    uint64_t a_full;
    uint64_t a_empty;
    uint64_t t_full[kKBMax];
    uint64_t t_empty[kKBMax];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kOffA = 0;
constexpr size_t kOffB = kOffA + size_t(kKBMax) * kABlockBytes;
constexpr size_t kOffOut = kOffB + size_t(kStages) * kBStageBytes;
constexpr size_t kOffBars = kOffOut + size_t(kEpiWarps) * kOutBufBytes;
constexpr size_t kSmemBytes = kOffBars + sizeof(Bars) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103a CTA");

__global__ void __launch_bounds__(kThreads, 1)
    decompress_fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_q,
                               const __grid_constant__ CUtensorMap tm_w,
                               const __grid_constant__ CUtensorMap tm_kbuf,
                               const DecompressArgs a, const Fp8Extra x) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem + kOffA;
    uint8_t* sB = smem + kOffB;
    uint8_t* sOut = smem + kOffOut;
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int KB = a.kv_lora_rank / 128;
    const int64_t T = a.total_tiles;
    const int64_t G = gridDim.x;
    const int64_t t_begin = T * blockIdx.x / G;
    const int64_t t_end = T * (blockIdx.x + 1) / G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->b_full[s], 1);
            mbar_init(&bars->b_empty[s], 1);
        }
        mbar_init(&bars->a_full, 1);
        mbar_init(&bars->a_empty, 1);
        for (int i = 0; i < kKBMax; ++i) {
            mbar_init(&bars->t_full[i], 1);
            mbar_init(&bars->t_empty[i], kEpiWarps);
        }
        mbar_init(&bars->mma_done, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_w);
        tma_prefetch_map(&tm_kbuf);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const WaitCtl wc{&bars->abort_flag, a.status, a.timeout_ns};
    const int64_t row_end = decompress_row_end(a);

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t keep = policy_evict_last();
            uint32_t it = 0, seg = 0;
            int64_t cur_m = -1;
            bool issued[kStages] = {};
            uint32_t last_phase[kStages] = {};
            bool a_issued = false;
            uint32_t a_phase = 0;
            bool ok = true;
            for (int64_t t = t_begin; t < t_end && ok; ++t) {
                const int64_t m = t / a.n_tiles;
                const int n = static_cast<int>(t % a.n_tiles);
                if (m != cur_m) {
                    cur_m = m;
                    if (seg > 0 && !mbar_wait(&bars->a_empty, (seg - 1) & 1, wc)) break;
                    mbar_arrive_expect_tx(&bars->a_full,
                                          static_cast<uint32_t>(KB) * kABlockBytes);
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load_2d(sA + kb * kABlockBytes, &tm_q, &bars->a_full, kb * 128,
                                    static_cast<int32_t>(m * kBM));
                    a_issued = true;
                    a_phase = seg & 1;
                    ++seg;
                }
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1;
                    if (!mbar_wait(&bars->b_empty[s], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->b_full[s], kBStageBytes);
                    tma_load_2d_hint(sB + s * kBStageBytes, &tm_w, &bars->b_full[s], kb * 128,
                                     n * kBN, keep);
                    issued[s] = true;
                    last_phase[s] = ph;
                    ++it;
                }
            }
            if (bars->abort_flag) {
                for (int s = 0; s < kStages; ++s)
                    if (issued[s]) mbar_wait(&bars->b_full[s], last_phase[s], wc, false);
                if (a_issued) mbar_wait(&bars->a_full, a_phase, wc, false);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3(128, kBN);
            uint32_t it = 0, tile_i = 0, seg = 0;
            int64_t cur_m = -1;
            bool ok = true;
            for (int64_t t = t_begin; t < t_end && ok; ++t) {
                const int64_t m = t / a.n_tiles;
                if (m != cur_m) {
                    if (cur_m >= 0) {
                        mma_commit(&bars->a_empty);
                        ++seg;
                    }
                    cur_m = m;
                    if (!mbar_wait(&bars->a_full, seg & 1, wc)) break;
                }
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&bars->t_empty[kb], (tile_i & 1) ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1;
                    if (!mbar_wait(&bars->b_full[s], ph, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + kb * kABlockBytes);
                    const uint32_t b_addr = smem_u32(sB + s * kBStageBytes);
                    const uint32_t d = tmem + static_cast<uint32_t>(kb) * kBN;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_e4m3(d, sdesc_sw128(a_addr + k * 32, 16, 1024),
                                 sdesc_sw128(b_addr + k * 32, 16, 1024), idesc, k != 0 ? 1u : 0u);
                    mma_commit(&bars->b_empty[s]);
                    mma_commit(&bars->t_full[kb]);
                    ++it;
                }
                ++tile_i;
            }
            mma_commit(&bars->mma_done);
            mbar_wait(&bars->mma_done, 0, wc, false);
        }
    } else {
        // 8 epilogue warps: warp w reads TMEM lane quarter w % 4 (32 rows) and one 64-column
        // half of the 128-column tile, so each keeps 64 fp32 partial sums and issues both
        // 32-column TMEM loads of a k-block before waiting once.
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        uint8_t* stage = sOut + (warp - 2) * kOutBufBytes;
        uint32_t tile_i = 0;
        int64_t cur_m = -1, my_row = 0;
        bool slab_full = false, my_valid = false;
        float sa[kKBMax] = {0.f, 0.f, 0.f, 0.f};
        bool ok = true;
        for (int64_t t = t_begin; t < t_end && ok; ++t) {
            const int64_t m = t / a.n_tiles;
            const int n = static_cast<int>(t % a.n_tiles);
            if (m != cur_m) {
                cur_m = m;
                my_row = m * kBM + q * 32 + lane;
                my_valid = decompress_row_source(a, my_row, row_end) >= 0;
                slab_full = __all_sync(0xffffffffu, my_valid);
#pragma unroll
                for (int kb = 0; kb < kKBMax; ++kb)
                    sa[kb] = (my_valid && kb < KB) ? x.q_scale[my_row * KB + kb] : 0.0f;
            }
            float acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
#pragma unroll
            for (int kb = 0; kb < kKBMax; ++kb) {
                if (kb >= KB) break;
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->t_full[kb], tile_i & 1, wc))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float cs = sa[kb] * __ldg(x.w_scale + static_cast<int64_t>(n) * KB + kb);
                const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(kb) * kBN + h * 64;
                uint32_t v0[32], v1[32];
                tmem_ld_x32(tbase, v0);
                tmem_ld_x32(tbase + 32, v1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->t_empty[kb]);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    acc[j] = fmaf(cs, __uint_as_float(v0[j]), acc[j]);
                    acc[32 + j] = fmaf(cs, __uint_as_float(v1[j]), acc[32 + j]);
                }
            }
            if (!ok) break;
            uint32_t p[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) p[j] = pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
            const int col = n * kBN + h * 64;
            if (slab_full) {
                if (lane == 0) bulk_wait_read<0>();  // the previous store read this box
                __syncwarp();
                const uint32_t rowaddr = smem_u32(stage) + lane * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4), p[4 * j], p[4 * j + 1],
                                 p[4 * j + 2], p[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tm_kbuf, stage, col, static_cast<int32_t>(m * kBM + q * 32));
                    bulk_commit();
                }
            } else if (my_valid) {
                uint16_t* dst = a.k_buffer + my_row * a.n_out + col;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_v4(dst + j * 8, make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]));
            }
            ++tile_i;
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_fp8_gather_quantize(DecompressArgs args, Fp8Extra extra, int num_sms,
                                       cudaStream_t stream) {
    const int64_t rows = args.buffer_length;
    int64_t blocks = (rows + 7) / 8;  // 8 warps (rows in flight) per block
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fp8_gather_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(args, extra);
    return cudaGetLastError();
}

cudaError_t launch_decompress_fp8_gemm(const CUtensorMap& tm_q, const CUtensorMap& tm_w,
                                       const CUtensorMap& tm_kbuf, DecompressArgs args,
                                       Fp8Extra extra, int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(decompress_fp8_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t grid = args.total_tiles < num_sms ? args.total_tiles : num_sms;
    decompress_fp8_gemm_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(
        tm_q, tm_w, tm_kbuf, args, extra);
    return cudaGetLastError();
}

}  // namespace pkm
