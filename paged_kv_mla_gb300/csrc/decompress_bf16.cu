// decompress_bf16.cu -- fused paged gather + tcgen05 up-projection (bf16), on CTA pairs.
//
// generic_flare_mla_decompress_k_cache_ragged_paged (Modular MAX, nn/kv_cache_ragged),
// description and Args: rows [buffer_row_offsets[b], buffer_row_offsets[b+1]) of the
// ragged buffer receive the latent K rows of cache tokens starting at cache_offsets[b];
// they are copied to k_latent_buffer and their first kv_lora_rank columns are multiplied
// by W_k^T into k_buffer.
//
// The grid is made of clusters of two CTAs on two SMs (a CTA pair).  A pair computes
// 256 x bn output tiles with tcgen05.mma.cta_group::2 (M = 256): each CTA gathers and keeps
// its own 128 latent rows (A) in shared memory and loads one half (bn/2 rows) of each W_k
// tile (B); the even CTA issues the MMAs, which read both CTAs' shared memory and write
// each CTA's 128 x bn accumulator into its own TMEM.  Splitting B halves the W_k bytes each
// SM pulls from L2 per FLOP and halves the shared memory one pipeline stage needs, so each
// CTA keeps five W_k stages in flight next to its resident A tile.
//
// Each pair walks a contiguous range of tile ids (m_pair * n_tiles + n), so consecutive
// tiles reuse the gathered rows.  Warp roles, in both CTAs:
//   warps 0, 8  TMA producers: this CTA's half of W_k [bn/2 x 64] (128-byte swizzle) into a
//               5-stage ring, alternate stages each; completion is signalled on the even
//               CTA's barrier.
//   warp 1      TMEM allocator (pair); in the even CTA also the single MMA-issuing thread.
//   warps 2-3   gatherers: resolve rows through buffer_row_offsets / cache_offsets / the
//               page table, cp.async the nope columns into the swizzled A tile (one group
//               and one barrier arrival per 64-column k-block), copy whole latent rows to
//               k_latent_buffer.
//   warps 4-7   epilogue: tcgen05.ld of this CTA's accumulator (double-buffered), bf16
//               rounding, a swizzled 4 KB staging box per warp, TMA stores of 32 x 64
//               boxes of k_buffer.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

constexpr int kThreads = 288;                // 9 warps: + a second W_k producer
constexpr int kBM = 128;                     // rows per CTA (256 per pair)
constexpr int kKBMax = 8;                    // kv_lora_rank <= 512 = 8 k-blocks of 64
constexpr int kABlockBytes = kBM * 128;      // 16 KB per k-block
constexpr int kStages = 5;
constexpr int kBStageBytes = 128 * 128;      // bn/2 <= 128 rows of 128 bytes
constexpr int kEpiWarps = 4;
constexpr int kOutBufBytes = 32 * 128;       // 32 rows x 64 bf16
constexpr int kGatherThreads = 64;
constexpr uint32_t kTmemCols = 512;

struct Bars {
    uint64_t b_full[kStages];   // even CTA: both halves of a W_k stage landed
    uint64_t b_empty[kStages];  // both CTAs: the pair's MMAs are done with a stage
    uint64_t a_full[kKBMax];    // even CTA: k-block of both CTAs' A gathered
    uint64_t a_empty;           // both CTAs: the MMAs are done with A
    uint64_t t_full[2];         // both CTAs: accumulator ready
    uint64_t t_empty[2];        // even CTA: both CTAs' epilogues drained an accumulator
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int gather_go;
};

constexpr size_t kOffA = 0;
constexpr size_t kOffB = kOffA + size_t(kKBMax) * kABlockBytes;
constexpr size_t kOffOut = kOffB + size_t(kStages) * kBStageBytes;
constexpr size_t kOffRows = kOffOut + size_t(kEpiWarps) * kOutBufBytes;
constexpr size_t kOffBars = kOffRows + kBM * sizeof(int64_t);
constexpr size_t kSmemBytes = kOffBars + sizeof(Bars) + 1024;  // + base alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103a CTA");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decompress_bf16_kernel(const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_kbuf, const DecompressArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem + kOffA;
    uint8_t* sB = smem + kOffB;
    uint8_t* sOut = smem + kOffOut;
    int64_t* s_rows = reinterpret_cast<int64_t*>(smem + kOffRows);
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 = even CTA (issues the MMAs), 1 = odd
    const bool leader = rank == 0;
    const int KB = a.kv_lora_rank / 64;
    const int bn = a.bn;                      // pair N tile
    const int half = bn / 2;                  // W_k rows this CTA loads per tile
    const int64_t T = a.total_tiles;          // pair tiles
    const int64_t P = gridDim.x / 2;
    const int64_t pair = blockIdx.x / 2;
    const int64_t t_begin = T * pair / P;
    const int64_t t_end = T * (pair + 1) / P;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->b_full[s], 1);
            mbar_init(&bars->b_empty[s], 1);
        }
        for (int kb = 0; kb < kKBMax; ++kb) mbar_init(&bars->a_full[kb], 2 * kGatherThreads);
        mbar_init(&bars->a_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->t_full[i], 1);
            mbar_init(&bars->t_empty[i], 2 * kEpiWarps);
        }
        mbar_init(&bars->mma_done, 1);
        bars->abort_flag = 0;
        bars->gather_go = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tm_w);
        tma_prefetch_map(&tm_kbuf);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const WaitCtl wc{&bars->abort_flag, a.status, a.timeout_ns};
    const int64_t row_end = decompress_row_end(a);

    if (warp == 0 || warp == 8) {
        // ---------------- W_k producers (this CTA's half of each tile) ----------------
        // Two threads issue alternate ring iterations: a TMA load costs its issuing thread a
        // roughly fixed time, so one thread could not keep up with the MMAs.
        if (lane == 0) {
            const uint32_t who = warp == 0 ? 0u : 1u;
            const uint64_t keep = policy_evict_last();
            uint32_t it = 0;
            bool issued[kStages] = {};
            uint32_t last_phase[kStages] = {};
            bool ok = true;
            for (int64_t t = t_begin; t < t_end && ok; ++t) {
                const int n = static_cast<int>(t % a.n_tiles);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    if ((it & 1u) != who) continue;
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1;
                    if (!mbar_wait(&bars->b_empty[s], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    if (leader)  // both halves complete on the even CTA's barrier
                        mbar_arrive_expect_tx(&bars->b_full[s], static_cast<uint32_t>(bn) * 128);
                    tma_load_2d_pair(sB + s * kBStageBytes, &tm_w,
                                     mapa_shared(smem_u32(&bars->b_full[s]), 0), kb * 64,
                                     n * bn + static_cast<int>(rank) * half, keep);
                    issued[s] = true;
                    last_phase[s] = ph;
                }
            }
            if (!ok) {  // let loads already in flight land before the CTA retires
                if (leader) {
                    for (int s = 0; s < kStages; ++s)
                        if (issued[s]) mbar_wait(&bars->b_full[s], last_phase[s], wc, false);
                } else {
                    spin_ns(50000);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (even CTA) ----------------
        if (leader && lane == 0) {
            const uint32_t idesc = idesc_bf16(256, bn, false, false);
            uint32_t it = 0, tile_i = 0, seg = 0;
            int64_t cur_m = -1;
            bool ok = true;
            for (int64_t t = t_begin; t < t_end && ok; ++t) {
                const int64_t m = t / a.n_tiles;
                const bool new_seg = (m != cur_m);
                if (new_seg) {
                    if (cur_m >= 0) {
                        mma_commit_pair(&bars->a_empty, 3);  // both A tiles free once retired
                        ++seg;
                    }
                    cur_m = m;
                }
                const uint32_t acc = tile_i & 1, aph = (tile_i >> 1) & 1;
                if (!mbar_wait(&bars->t_empty[acc], aph ^ 1, wc)) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * static_cast<uint32_t>(bn);
                for (int kb = 0; kb < KB; ++kb) {
                    if (new_seg && !mbar_wait_cluster(&bars->a_full[kb], seg & 1, wc)) {
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
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16_pair(d, sdesc_sw128(a_addr + k * 32, 16, 1024),
                                      sdesc_sw128(b_addr + k * 32, 16, 1024), idesc,
                                      (kb | k) != 0 ? 1u : 0u);
                    mma_commit_pair(&bars->b_empty[s], 3);
                    ++it;
                }
                if (!ok) break;
                mma_commit_pair(&bars->t_full[acc], 3);
                ++tile_i;
            }
            mma_commit_pair(&bars->mma_done, 1);
            mbar_wait(&bars->mma_done, 0, wc, false);
        }
    } else if (warp < 4) {
        // ---------------- gatherers (this CTA's 128 rows) ----------------
        const int g = threadIdx.x - 64;
        const int chunk = g & 7;   // 16-byte chunk inside a 128-byte k-block row
        const int rsub = g >> 3;   // row phase 0..7
        const int cchunks = a.latent_cols / 8;
        uint32_t seg = 0;
        int64_t cur_m = -1;
        for (int64_t t = t_begin; t < t_end; ++t) {
            const int64_t m_pair = t / a.n_tiles;
            if (m_pair == cur_m) continue;
            cur_m = m_pair;
            const int64_t m = m_pair * 2 + rank;          // this CTA's 128-row block
            const bool writer = (t % a.n_tiles) == 0;      // this pair owns tile (m_pair, 0)
            for (int i = g; i < kBM; i += kGatherThreads) {
                const int64_t off = decompress_row_source(a, m * kBM + i, row_end);
                if (off == -2) report(a.status, PKM_ERR_OUT_OF_RANGE);
                s_rows[i] = off;
            }
            if (g == 0)
                bars->gather_go =
                    (seg == 0 || mbar_wait(&bars->a_empty, (seg - 1) & 1, wc)) ? 1 : 0;
            named_bar_sync(1, kGatherThreads);
            if (!bars->gather_go) break;
            for (int kb = 0; kb < KB; ++kb) {
                const uint32_t base = smem_u32(sA + kb * kABlockBytes);
#pragma unroll 4
                for (int j = 0; j < kBM / 8; ++j) {
                    const int row = rsub + 8 * j;
                    const int64_t off = s_rows[row];
                    const uint16_t* src =
                        off >= 0 ? a.cache_layer + off + kb * 64 + chunk * 8 : a.cache_layer;
                    cp_async_16(base + row * 128 + ((chunk ^ (row & 7)) << 4), src,
                                off >= 0 ? 16u : 0u);
                }
                cp_async_commit();
            }
            for (int kb = 0; kb < KB; ++kb) {
                cp_async_wait_dyn(KB - 1 - kb);
                fence_proxy_async_smem();
                mbar_arrive_cluster(mapa_shared(smem_u32(&bars->a_full[kb]), 0));
            }
            if (writer) {
                const int total = kBM * cchunks;
                for (int i0 = g; i0 < total; i0 += 4 * kGatherThreads) {
                    uint4 v[4];
                    int64_t dst[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int idx = i0 + u * kGatherThreads;
                        dst[u] = -1;
                        if (idx < total) {
                            const int row = idx / cchunks;
                            const int c = idx - row * cchunks;
                            const int64_t off = s_rows[row];
                            if (off >= 0) {
                                v[u] = ld_nc_v4(a.cache_layer + off + c * 8);
                                dst[u] = (m * kBM + row) * a.latent_cols + c * 8;
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (dst[u] >= 0) st_v4(a.k_latent + dst[u], v[u]);
                }
            }
            named_bar_sync(1, kGatherThreads);
            ++seg;
        }
        cp_async_wait<0>();
    } else if (warp < 8) {
        // ---------------- epilogue (this CTA's 128 rows) ----------------
        const int q = warp & 3;  // TMEM lane quarter == 32-row slab of the CTA's rows
        const uint32_t t_empty_leader = mapa_shared(smem_u32(&bars->t_empty[0]), 0);
        uint32_t tile_i = 0;
        int64_t cur_m = -1, my_row = 0, m = 0;
        bool slab_full = false, my_valid = false;
        for (int64_t t = t_begin; t < t_end; ++t) {
            const int64_t m_pair = t / a.n_tiles;
            const int n = static_cast<int>(t % a.n_tiles);
            if (m_pair != cur_m) {
                cur_m = m_pair;
                m = m_pair * 2 + rank;
                my_row = m * kBM + q * 32 + lane;
                my_valid = decompress_row_source(a, my_row, row_end) >= 0;
                slab_full = __all_sync(0xffffffffu, my_valid);
            }
            const uint32_t acc = tile_i & 1, ph = (tile_i >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->t_full[acc], ph, wc))) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * static_cast<uint32_t>(bn);
            for (int c = 0; c < bn / 64; ++c) {
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
                if (slab_full) {
                    uint8_t* stage = sOut + q * kOutBufBytes;
                    if (lane == 0) bulk_wait_read<0>();  // the previous store read its box
                    __syncwarp();
                    const uint32_t rowaddr = smem_u32(stage) + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4), p[4 * j], p[4 * j + 1],
                                     p[4 * j + 2], p[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_kbuf, stage, n * bn + c * 64,
                                     static_cast<int32_t>(m * kBM + q * 32));
                        bulk_commit();
                    }
                } else if (my_valid) {  // slab with uncovered rows: plain per-row stores
                    uint16_t* dst = a.k_buffer + my_row * a.n_out + n * bn + c * 64;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_v4(dst + j * 8,
                              make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(t_empty_leader + acc * sizeof(uint64_t));
            ++tile_i;
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA of the pair retires while the other may still signal it
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_decompress_bf16(const CUtensorMap& tm_w, const CUtensorMap& tm_kbuf,
                                   DecompressArgs args, int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(decompress_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t max_pairs = num_sms / 2;
    const int64_t pairs = args.total_tiles < max_pairs ? args.total_tiles : max_pairs;
    decompress_bf16_kernel<<<static_cast<unsigned>(2 * pairs), kThreads, kSmemBytes, stream>>>(
        tm_w, tm_kbuf, args);
    return cudaGetLastError();
}

}  // namespace pkm
