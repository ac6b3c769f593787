// kv_matmul.cu -- ragged GEMM written into the paged K/V cache, on CTA pairs.
//
// kv_matmul_ragged_paged (Modular MAX, nn/kv_cache_ragged), description and Args: Y =
// hidden_state [sum(seq_lens), num_heads*head_size] x weight [num_heads*head_size,
// num_kv_heads*head_size]; row i of request b is written into the cache of layer
// layer_idx at position cache_lengths[b] + i.  The output columns are split K then V
// (head_elems each).
//
// Clusters of two CTAs compute 256 x bn tiles with tcgen05.mma.cta_group::2 (M = 256):
// each CTA streams its own 128 rows of A (hidden_state, K-major, box 64 x 128) and half of
// the tile's B columns (weight, N contiguous = MN-major, boxes of 64 x 64) with TMA into a
// 6-stage ring whose completion is signalled on the even CTA's barriers; the even CTA
// issues the MMAs.  Each CTA's 4 epilogue warps drain its 128 x bn accumulator (TMEM,
// double-buffered), round to bf16, and scatter each row's 64-column chunk to its
// (page, slot) with 16-byte stores, 4 full rows of 128 bytes per warp instruction.  When
// n_out is an odd multiple of 64, the last n tile is half empty: its missing weight
// columns load as zeros and are not stored.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;                      // rows per CTA (256 per pair)
constexpr int kStages = 6;
constexpr int kAStageBytes = kBM * 128;       // 128 rows x 64 bf16
constexpr int kBStageBytes = 2 * 64 * 128;    // bn/2 <= 128 columns: 2 boxes of 64 k x 64 n
constexpr int kStageBytes = kAStageBytes + kBStageBytes;
constexpr int kEpiWarps = 4;
constexpr int kOutBufBytes = 32 * 128;
constexpr uint32_t kTmemCols = 512;

struct Bars {
    uint64_t full[kStages];     // even CTA: both CTAs' A and B halves of a stage landed
    uint64_t empty[kStages];    // both CTAs: the pair's MMAs are done with a stage
    uint64_t t_full[2];         // both CTAs: accumulator ready
    uint64_t t_empty[2];        // even CTA: both CTAs' epilogues drained an accumulator
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kOffStages = 0;
constexpr size_t kOffOut = kOffStages + size_t(kStages) * kStageBytes;
constexpr size_t kOffBars = kOffOut + size_t(kEpiWarps) * kOutBufBytes;
constexpr size_t kSmemBytes = kOffBars + sizeof(Bars) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103a CTA");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    kv_matmul_kernel(const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_w, const KvMatmulArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sStages = smem + kOffStages;
    uint8_t* sOut = smem + kOffOut;
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int bn = a.bn;          // pair N tile
    const int half = bn / 2;      // B columns this CTA loads
    const int KB = a.k_in / 64;
    const int64_t T = a.total_tiles;  // pair tiles
    const int64_t P = gridDim.x / 2;
    const int64_t pair = blockIdx.x / 2;
    const int64_t t_begin = T * pair / P;
    const int64_t t_end = T * (pair + 1) / P;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->t_full[i], 1);
            mbar_init(&bars->t_empty[i], 2 * kEpiWarps);
        }
        mbar_init(&bars->mma_done, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tm_x);
        tma_prefetch_map(&tm_w);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const WaitCtl wc{&bars->abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        if (lane == 0) {
            // A rows are re-read for every n tile of their block and W by every block: both
            // (tens of MB) are kept in L2 ahead of the scattered cache writes
            const uint64_t keep = policy_evict_last();
            const uint32_t pair_tx = 2 * (kAStageBytes + static_cast<uint32_t>(half) * 128);
            RingPos rp;
            bool issued[kStages] = {};
            uint32_t last_phase[kStages] = {};
            bool ok = true;
            for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid() && ok; w.next()) {
                const int64_t m = w.m * 2 + rank;  // this CTA's 128-row block
                const int n = w.n;
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t s = rp.stage, ph = rp.phase;
                    if (!mbar_wait(&bars->empty[s], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = sStages + s * kStageBytes;
                    const uint32_t full_leader = mapa_shared(smem_u32(&bars->full[s]), 0);
                    if (leader) mbar_arrive_expect_tx(&bars->full[s], pair_tx);
                    tma_load_2d_pair(st, &tm_x, full_leader, kb * 64,
                                     static_cast<int32_t>(m * kBM), keep);
                    for (int j = 0; j < half / 64; ++j)
                        tma_load_2d_pair(st + kAStageBytes + j * 8192, &tm_w, full_leader,
                                         n * bn + static_cast<int>(rank) * half + j * 64,
                                         kb * 64, keep);
                    issued[s] = true;
                    last_phase[s] = ph;
                    rp.next(kStages);
                }
            }
            if (!ok) {
                if (leader) {
                    for (int s = 0; s < kStages; ++s)
                        if (issued[s]) mbar_wait(&bars->full[s], last_phase[s], wc, false);
                } else {
                    spin_ns(50000);
                }
            }
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            const uint32_t idesc = idesc_bf16(256, bn, false, true);
            // operand descriptors built once; each MMA adds its offset (16-byte units)
            const uint64_t a_desc0 = sdesc_sw128(smem_u32(sStages), 16, 1024);
            const uint64_t b_desc0 = sdesc_sw128(smem_u32(sStages + kAStageBytes), 8192, 1024);
            uint32_t tile_i = 0;
            RingPos rp;
            bool ok = true;
            for (int64_t t = t_begin; t < t_end && ok; ++t) {
                const uint32_t acc = tile_i & 1, aph = (tile_i >> 1) & 1;
                if (!mbar_wait(&bars->t_empty[acc], aph ^ 1, wc)) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * static_cast<uint32_t>(bn);
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t s = rp.stage, ph = rp.phase;
                    if (!mbar_wait(&bars->full[s], ph, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_add_bytes(a_desc0, s * kStageBytes);
                    const uint64_t bd = desc_add_bytes(b_desc0, s * kStageBytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // K = 16: 32 bytes of A, 2048 of MN-major B
                        mma_bf16_pair(d, ad + 2 * k, bd + 128 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    mma_commit_pair(&bars->empty[s], 3);
                    rp.next(kStages);
                }
                if (!ok) break;
                mma_commit_pair(&bars->t_full[acc], 3);
                ++tile_i;
            }
            mma_commit_pair(&bars->mma_done, 1);
            mbar_wait(&bars->mma_done, 0, wc, false);
        }
    } else {
        const int q = warp & 3;
        uint8_t* stage = sOut + q * kOutBufBytes;
        const uint32_t stage_addr = smem_u32(stage);
        const uint32_t t_empty_leader = mapa_shared(smem_u32(&bars->t_empty[0]), 0);
        uint32_t tile_i = 0;
        int64_t cur_m = -1, my_dst = -1;
        for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid(); w.next()) {
            const int64_t m = w.m * 2 + rank;
            const int n = w.n;
            if (m != cur_m) {
                cur_m = m;
                my_dst = kv_row_dest(a, m * kBM + q * 32 + lane);
                if (my_dst == -2) report(a.status, PKM_ERR_OUT_OF_RANGE);
            }
            const uint32_t acc = tile_i & 1, ph = (tile_i >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->t_full[acc], ph, wc))) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * static_cast<uint32_t>(bn);
            for (int c = 0; c < bn / 64; ++c) {
                const int col0 = n * bn + c * 64;
                if (col0 >= a.n_out) break;  // padded half of the last n tile
                uint32_t v0[32], v1[32];
                tmem_ld_x32(tbase + c * 64, v0);
                tmem_ld_x32(tbase + c * 64 + 32, v1);
                tmem_ld_wait();
                uint32_t p[32];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    p[j] = pack_bf16x2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1]));
                    p[16 + j] =
                        pack_bf16x2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1]));
                }
                const uint32_t rowaddr = stage_addr + lane * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4), p[4 * j], p[4 * j + 1],
                                 p[4 * j + 2], p[4 * j + 3]);
                __syncwarp();
                // 64 output columns of one chunk lie entirely in the K or the V plane
                const int64_t plane = col0 < a.head_elems ? 0 : a.kv_stride;
                const int colp = (col0 < a.head_elems ? col0 : col0 - a.head_elems) + (lane & 7) * 8;
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int row = it * 4 + (lane >> 3);
                    const int64_t dst = __shfl_sync(0xffffffffu, my_dst, row);
                    const uint4 v = ld_shared_v4(stage_addr + row * 128 + (((lane & 7) ^ (row & 7)) << 4));
                    if (dst >= 0) st_v4(a.cache_layer + plane + dst + colp, v);
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(t_empty_leader + acc * sizeof(uint64_t));
            ++tile_i;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_kv_matmul(const CUtensorMap& tm_x, const CUtensorMap& tm_w, KvMatmulArgs args,
                             int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kv_matmul_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t max_pairs = num_sms / 2;
    const int64_t pairs = args.total_tiles < max_pairs ? args.total_tiles : max_pairs;
    kv_matmul_kernel<<<static_cast<unsigned>(2 * pairs), kThreads, kSmemBytes, stream>>>(
        tm_x, tm_w, args);
    return cudaGetLastError();
}

}  // namespace pkm
