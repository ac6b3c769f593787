// decompress_bf16.cu -- fused paged gather + tcgen05 up-projection (bf16), on CTA pairs.
//
// generic_flare_mla_decompress_k_cache_ragged_paged (Modular MAX, nn/kv_cache_ragged),
// description and Args: rows [buffer_row_offsets[b], buffer_row_offsets[b+1]) of the
// ragged buffer receive the latent K rows of cache tokens starting at cache_offsets[b];
// they are copied to k_latent_buffer and their first kv_lora_rank columns are multiplied
// by W_k^T into k_buffer.  With w_uv (mla_prefill_decode_graph_fp8, Args w_uv: "projecting
// latent values to V", [num_heads, v_head_dim, kv_latent_dim]) the same gathered rows are
// also multiplied by w_uv^T into v_buffer: the V tiles follow the K tiles of each 256-row
// block, so the rows are gathered once for both.
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
//               page table (one 256-row block ahead of the MMAs), bring the nope columns
//               into the swizzled A tile -- one 4-D TMA load per 8-row group that is eight
//               consecutive slots of one page, cp.async row by row for the other groups --
//               and copy whole latent rows to k_latent_buffer.
//   warps 4-7   epilogue: tcgen05.ld of this CTA's accumulator (double-buffered), bf16
//               rounding, then per 32 x 64 box a pass through a swizzled 4 KB shared
//               buffer that turns lane-per-row registers into whole 128-byte row segments
//               for coalesced global stores.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

// A row's source inside the cache layer, as kept in shared memory: its element offset / 8
// (every row starts on a 16-byte boundary), or one of two markers.
constexpr uint32_t kSrcOutOfRange = 0xFFFFFFFEu;  // page lookup out of range (reported)
constexpr uint32_t kSrcNone = 0xFFFFFFFFu;        // no request covers the row

// Resolves row i of a 128-row block into src[i]; the first row of each 8-row group also
// leaves its (page, slot) in grp[i / 8], the coordinates of a TMA box starting there.
__device__ __forceinline__ void resolve_row(const DecompressArgs& a, int64_t block_row0, int i,
                                            int64_t row_end, uint32_t* src, uint2* grp) {
    uint32_t page = 0, slot = 0;
    const int64_t off = decompress_row_locate(a, block_row0 + i, row_end, &page, &slot);
    if (off == -2) report(a.status, PKM_ERR_OUT_OF_RANGE);
    src[i] = off >= 0 ? static_cast<uint32_t>(off >> 3) : off == -2 ? kSrcOutOfRange : kSrcNone;
    if ((i & 7) == 0) grp[i >> 3] = make_uint2(page, slot);
}

constexpr int kThreads = 288;                // 9 warps: + a second W_k producer
constexpr int kBM = 128;                     // rows per CTA (256 per pair)
constexpr int kKBMax = 8;                    // kv_lora_rank <= 512 = 8 k-blocks of 64
constexpr int kGroups = kBM / 8;             // 8-row groups of the A tile
constexpr int kStages = 5;
constexpr int kBStageBytes = 128 * 128;      // bn/2 <= 128 rows of 128 bytes
constexpr int kEpiWarps = 4;
constexpr int kOutBufBytes = 32 * 128;       // 32 rows x 64 bf16
constexpr int kGatherThreads = 64;
constexpr uint32_t kTmemCols = 512;

struct Bars {
    uint64_t b_full[kStages];   // even CTA: both halves of a W_k stage landed
    uint64_t b_empty[kStages];  // both CTAs: the pair's MMAs are done with a stage
    uint64_t a_full;            // even CTA: both CTAs' A tiles gathered
    uint64_t a_empty;           // both CTAs: the MMAs are done with A
    uint64_t t_full[2];         // both CTAs: accumulator ready
    uint64_t t_empty[2];        // even CTA: both CTAs' epilogues drained an accumulator
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int gather_go;
    uint32_t gather_mask;       // bit g: 8-row group g of the A tile comes by TMA
};

// The A tile is kept as [8-row group][k-block][8 rows x 128 bytes]: one TMA box (eight
// slots, all k-blocks) fills one group; the MMA steps 8-row groups by KB KB.
constexpr size_t kOffA = 0;
constexpr size_t kOffB = kOffA + size_t(kKBMax) * kBM * 128;
constexpr size_t kOffOut = kOffB + size_t(kStages) * kBStageBytes;
constexpr size_t kOffRows = kOffOut + size_t(kEpiWarps) * kOutBufBytes;
constexpr size_t kOffGrp = kOffRows + 2 * kBM * sizeof(uint32_t);
constexpr size_t kOffBars = kOffGrp + 2 * kGroups * sizeof(uint2);
constexpr size_t kSmemBytes = kOffBars + sizeof(Bars) + 1024;  // + base alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103a CTA");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decompress_bf16_kernel(const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_wv,
                           const __grid_constant__ CUtensorMap tm_cache, const DecompressArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem + kOffA;
    uint8_t* sB = smem + kOffB;
    uint8_t* sOut = smem + kOffOut;
    // sources of this CTA's 128 rows, for the current and the next 256-row block
    uint32_t* s_src = reinterpret_cast<uint32_t*>(smem + kOffRows);
    uint2* s_grp = reinterpret_cast<uint2*>(smem + kOffGrp);
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
        mbar_init(&bars->a_full, 2 * kGatherThreads);
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
        if (a.n_tiles > a.n_tiles_k) tma_prefetch_map(&tm_wv);
        if (a.gather_tma) tma_prefetch_map(&tm_cache);
    }
    // The first block's row sources, one row per thread: each is a chain of dependent
    // loads (row offsets, cache offset, page table), so resolve them all at once.
    if (threadIdx.x < kBM && t_begin < t_end)
        resolve_row(a, ((t_begin / a.n_tiles) * 2 + rank) * kBM, threadIdx.x,
                    decompress_row_end(a), s_src, s_grp);
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
            RingPos rp;
            bool issued[kStages] = {};
            uint32_t last_phase[kStages] = {};
            bool ok = true;
            for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid() && ok; w.next()) {
                // n tiles [0, n_tiles_k) project with W_k, the rest with w_uv
                const bool v_tile = w.n >= a.n_tiles_k;
                const CUtensorMap* wmap = v_tile ? &tm_wv : &tm_w;
                const int n = v_tile ? w.n - a.n_tiles_k : w.n;
                for (int kb = 0; kb < KB; ++kb, ++it, rp.next(kStages)) {
                    if ((it & 1u) != who) continue;
                    const uint32_t s = rp.stage, ph = rp.phase;
                    if (!mbar_wait(&bars->b_empty[s], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    if (leader)  // both halves complete on the even CTA's barrier
                        mbar_arrive_expect_tx(&bars->b_full[s], static_cast<uint32_t>(bn) * 128);
                    tma_load_2d_pair(sB + s * kBStageBytes, wmap,
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
            // operand descriptors built once; each MMA adds its offset (16-byte units): a
            // per-MMA rebuild sits between consecutive MMA issues and leaves the tensor
            // pipe idle
            const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), 16, KB * 1024);
            const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), 16, 1024);
            uint32_t tile_i = 0, seg = 0;
            RingPos rp;
            int64_t cur_m = -1;
            bool ok = true;
            for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid() && ok; w.next()) {
                const int64_t m = w.m;
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
                if (new_seg && !mbar_wait_cluster(&bars->a_full, seg & 1, wc)) break;
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t s = rp.stage, ph = rp.phase;
                    if (!mbar_wait(&bars->b_full[s], ph, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_add_bytes(a_desc0, static_cast<uint32_t>(kb) * 1024);
                    const uint64_t bd = desc_add_bytes(b_desc0, s * kBStageBytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // K = 16 bf16 = 32 bytes a step
                        mma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    mma_commit_pair(&bars->b_empty[s], 3);
                    rp.next(kStages);
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
        // Each 8-row group of the block whose rows are eight consecutive slots of one page
        // comes with one TMA load (all k-blocks); the other groups row by row with cp.async.
        const int g = threadIdx.x - 64;
        const int chunk = g & 7;   // 16-byte chunk inside a 128-byte k-block row
        const int rsub = g >> 3;   // row inside an 8-row group
        const int cchunks = a.latent_cols / 8;
        const uint32_t grp_bytes = static_cast<uint32_t>(KB) * 1024;
        const uint32_t slot_units = static_cast<uint32_t>(a.slot_stride >> 3);
        const uint32_t a_full_leader = mapa_shared(smem_u32(&bars->a_full), 0);
        uint32_t seg = 0;
        for (int64_t m_pair = t_begin / a.n_tiles; m_pair * a.n_tiles < t_end; ++m_pair) {
            const int64_t m = m_pair * 2 + rank;          // this CTA's 128-row block
            // the pair holding the block's middle tile copies its latent rows: it has at
            // least half the block's tiles left to hide the copy behind
            const int64_t t_mid = m_pair * a.n_tiles + a.n_tiles / 2;
            const bool writer = t_mid >= t_begin && t_mid < t_end;
            const uint32_t* src = s_src + (seg & 1) * kBM;  // resolved one block ahead
            const uint2* grp = s_grp + (seg & 1) * kGroups;
            if (warp == 2) {
                bool tma = false;
                if (lane < kGroups && a.gather_tma) {
                    const uint32_t u0 = src[lane * 8];
                    tma = u0 < kSrcOutOfRange &&
                          static_cast<int64_t>(grp[lane].y) + 8 <= a.page_size;
                    for (int i = 1; i < 8; ++i) tma = tma && src[lane * 8 + i] == u0 + i * slot_units;
                }
                const uint32_t mask = __ballot_sync(0xffffffffu, tma);
                if (lane == 0) {
                    bars->gather_mask = mask;
                    bars->gather_go =
                        (seg == 0 || mbar_wait(&bars->a_empty, (seg - 1) & 1, wc)) ? 1 : 0;
                }
            }
            named_bar_sync(1, kGatherThreads);
            if (!bars->gather_go) break;
            const uint32_t mask = bars->gather_mask;
            if (g < kGroups && ((mask >> g) & 1u)) {
                mbar_expect_tx_cluster(a_full_leader, grp_bytes);
                tma_load_4d_pair(sA + g * grp_bytes, &tm_cache, a_full_leader, 0,
                                 static_cast<int32_t>(grp[g].y), static_cast<int32_t>(grp[g].x),
                                 0);
            }
            for (int G = 0; G < kGroups; ++G) {
                if ((mask >> G) & 1u) continue;
                const uint32_t u = src[G * 8 + rsub];
                const bool have = u < kSrcOutOfRange;
                const uint16_t* p = a.cache_layer + (have ? static_cast<int64_t>(u) * 8 + chunk * 8 : 0);
                const uint32_t dst = smem_u32(sA + G * grp_bytes) + rsub * 128 + ((chunk ^ rsub) << 4);
                for (int kb = 0; kb < KB; ++kb)
                    cp_async_16(dst + kb * 1024, p + (have ? kb * 64 : 0), have ? 16u : 0u);
            }
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive_cluster(a_full_leader);
            // While the MMAs run on this block, resolve the rows of the pair's next one.
            if ((m_pair + 1) * a.n_tiles < t_end) {
                uint32_t* nsrc = s_src + ((seg + 1) & 1) * kBM;
                uint2* ngrp = s_grp + ((seg + 1) & 1) * kGroups;
                for (int i = g; i < kBM; i += kGatherThreads)
                    resolve_row(a, ((m_pair + 1) * 2 + rank) * kBM, i, row_end, nsrc, ngrp);
            }
            if (writer) {
                const int total = kBM * cchunks;
                for (int i0 = g; i0 < total; i0 += 8 * kGatherThreads) {
                    uint4 v[8];
                    int64_t dst[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int idx = i0 + u * kGatherThreads;
                        dst[u] = -1;
                        if (idx < total) {
                            const int row = idx / cchunks;
                            const int c = idx - row * cchunks;
                            const uint32_t su = src[row];
                            if (su < kSrcOutOfRange) {
                                v[u] = ld_nc_v4(a.cache_layer + static_cast<int64_t>(su) * 8 + c * 8);
                                dst[u] = (m * kBM + row) * a.latent_cols + c * 8;
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (dst[u] >= 0) st_v4(a.k_latent + dst[u], v[u]);
                }
            }
            named_bar_sync(1, kGatherThreads);
            ++seg;
        }
        if (bars->abort_flag) spin_ns(50000);  // let gather loads in flight land
        cp_async_wait<0>();
    } else if (warp < 8) {
        // ---------------- epilogue (this CTA's 128 rows) ----------------
        const int q = warp & 3;  // TMEM lane quarter == 32-row slab of the CTA's rows
        const uint32_t t_empty_leader = mapa_shared(smem_u32(&bars->t_empty[0]), 0);
        uint32_t tile_i = 0;
        const uint32_t stage = smem_u32(sOut + q * kOutBufBytes);
        int64_t cur_m = -1;
        uint16_t* row0 = a.k_buffer;   // first row of this warp's 32-row slab, in k_buffer
        uint16_t* row0v = a.v_buffer;  // and in v_buffer
        uint32_t valid = 0;            // bit r: slab row r is a buffer row with a source
        for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid(); w.next()) {
            const int64_t m_pair = w.m;
            if (m_pair != cur_m) {
                cur_m = m_pair;
                const int64_t first = (m_pair * 2 + rank) * kBM + q * 32;
                row0 = a.k_buffer + first * a.n_out;
                if (a.v_buffer != nullptr) row0v = a.v_buffer + first * a.n_out_v;
                valid = __ballot_sync(0xffffffffu,
                                      decompress_row_source(a, first + lane, row_end) >= 0);
            }
            const bool v_tile = w.n >= a.n_tiles_k;
            uint16_t* out = v_tile ? row0v + (w.n - a.n_tiles_k) * bn : row0 + w.n * bn;
            const int64_t pitch = v_tile ? a.n_out_v : a.n_out;
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
                warp_store_rows_32x64(stage, p, out + c * 64, pitch, valid, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(t_empty_leader + acc * sizeof(uint64_t));
            ++tile_i;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA of the pair retires while the other may still signal it
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_decompress_bf16(const CUtensorMap& tm_w, const CUtensorMap& tm_wv,
                                   const CUtensorMap& tm_cache, DecompressArgs args, int num_sms,
                                   cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(decompress_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t max_pairs = num_sms / 2;
    const int64_t pairs = args.total_tiles < max_pairs ? args.total_tiles : max_pairs;
    decompress_bf16_kernel<<<static_cast<unsigned>(2 * pairs), kThreads, kSmemBytes, stream>>>(
        tm_w, tm_wv, tm_cache, args);
    return cudaGetLastError();
}

}  // namespace pkm
