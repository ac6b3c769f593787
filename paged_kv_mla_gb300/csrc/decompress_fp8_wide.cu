// decompress_fp8_wide.cu -- the block-scaled FP8 decompress GEMM on 256-wide pair tiles.
//
// The K-decompress stage of mla_prefill_decode_graph_fp8 (Modular MAX,
// attention/gpu/mla_graph): Parameters fp8_dtype / fp8_scale_dtype and
// m/n/k_scale_granularity, Args w_k ([num_heads * qk_nope_head_dim, kv_latent_dim], e4m3)
// and w_k_scale, with granularities m = 1, n = k = 128:
//     k_buffer[r, n] = bf16( sum_kb s_a[r, kb] * s_w[n / 128, kb] * sum_{k in kb} q_a[r, k] q_w[n, k] ).
// The quantised rows q_a / s_a come from the gather + quantise prepass
// (fp8_gather_quantize_kernel or fp8_gather_qcache_kernel); this kernel is launched as its
// programmatic dependent.  With w_uv the V tiles follow the K tiles of each row block.
//
// Clusters of two CTAs (a CTA pair) walk 256 x 256 output tiles: every k-block's
// accumulator has to leave TMEM before its slot is reused, and with N = 256 one such
// hand-off covers twice the output columns it covers with N = 128.
// Each CTA keeps its 128 quantised rows resident (one 16 KB TMA box per 128-wide k-block,
// refilled k-block by k-block when the pair moves to its next row block) and streams its
// 128-row half of each tile's weight slice k-block by k-block through a TMA ring.  Every
// k-block carries its own scales, so each k-block's product needs its own accumulator: the
// even CTA's MMA thread writes k-block j of the pair's walk into TMEM accumulator j % 2
// (two of 256 columns), and 16 epilogue warps per CTA (32 rows x 64 columns each) fold it
// into fp32 running sums, s_a * s_w * partial, handing the accumulator back as soon as it
// is read, so the MMAs of the next k-block run meanwhile.  After a tile's last k-block each
// warp rounds its sums to bf16 into its 128-byte-swizzled 32 x 64 part of a 64 KB shared
// box, and a store thread writes the CTA's whole 128 x 256 tile with one 3-D TMA store
// (rows past buffer_length are clipped by the tensor map); a row block with rows that must
// stay untouched is stored row by row by the epilogue warps instead.  Each warp makes its
// box writes visible to the TMA store (proxy fence, then its arrival) only after it has
// handed back the next tile's first accumulator, so the wait for its stores to land is
// off the MMAs' path.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kFirstEpiWarp = 4;
// warpgroup 0: producer, MMA and two idle warps; warpgroups 1-4: the epilogue.  Registers
// are granted per warpgroup: launched at 96 a thread (the most 640 threads get), warpgroup
// 0 drops to 40 and the epilogue rises to 104 (128 x 40 + 512 x 104 <= 640 x 96).
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
constexpr int kLaunchRegs = 96;
constexpr int kCtlRegs = 40;
constexpr int kEpiRegs = 104;
static_assert(128 * kCtlRegs + 32 * kEpiWarps * kEpiRegs <= kThreads * kLaunchRegs,
              "warpgroup register split exceeds the launch's pool");
constexpr int kBM = 128;                        // rows per CTA (256 per pair)
constexpr int kBN = 256;                        // pair N tile: two weight-scale blocks
constexpr int kKBMax = 4;                       // kv_lora_rank <= 512
constexpr int kKBBytes = 128 * 128;             // 128 rows x one 128-wide k-block of e4m3
constexpr int kBStageKB = 2;                    // k-blocks of weights per ring stage
constexpr int kBStageBytes = kBStageKB * kKBBytes;
constexpr int kBStages = 3;
constexpr int kAcc = 2;
constexpr int kOutBufBytes = 32 * 128;          // a warp's 32 x 64 bf16 box
constexpr uint32_t kTmemCols = kAcc * kBN;

struct Bars {
    uint64_t b_full[kBStages];   // even CTA: both weight halves of a stage landed
    uint64_t b_empty[kBStages];  // both CTAs: the pair's MMAs are done with a stage
    uint64_t a_full[kKBMax];     // even CTA: both CTAs' rows of a k-block landed
    uint64_t a_empty[kKBMax];    // both CTAs: the MMAs are done with a k-block of rows
    uint64_t t_full[kAcc];       // both CTAs: a k-block's accumulator is ready
    uint64_t t_empty[kAcc];      // even CTA: both CTAs' epilogues have read it
    uint64_t staged;             // the 16 epilogue warps staged a tile's rounded results
    uint64_t box_free;           // the store thread's TMA store has read them
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kOffA = 0;
constexpr size_t kOffB = kOffA + size_t(kKBMax) * kKBBytes;
constexpr size_t kOffOut = kOffB + size_t(kBStages) * kBStageBytes;
constexpr size_t kOffBars = kOffOut + size_t(kEpiWarps) * kOutBufBytes;
constexpr size_t kSmemBytes = kOffBars + sizeof(Bars) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103a CTA");
static_assert(kOffOut % 1024 == 0, "128-byte-swizzled boxes start on 1 KB boundaries");

// Whether the CTA's 128-row block starting at row_blk may be stored whole by TMA: every
// row either has a source (it is written) or lies past buffer_length (the tensor map clips
// it).  A row below buffer_length without a source must stay untouched.  Warp-uniform.
__device__ __forceinline__ bool block_tma_ok(const DecompressArgs& a, int row_blk,
                                             int64_t row_end, int lane) {
    bool ok = true;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = row_blk + j * 32 + lane;
        ok = ok && (r >= a.buffer_length || decompress_row_source(a, r, row_end) >= 0);
    }
    return __all_sync(0xffffffffu, ok);
}


__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decompress_fp8_wide_kernel(const __grid_constant__ CUtensorMap tm_q,
                               const __grid_constant__ CUtensorMap tm_w,
                               const __grid_constant__ CUtensorMap tm_wv,
                               const __grid_constant__ CUtensorMap tm_ok,
                               const __grid_constant__ CUtensorMap tm_ov,
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
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int KB = a.kv_lora_rank / 128;
    const int64_t T = a.total_tiles;  // pair tiles
    const int64_t P = gridDim.x / 2;
    const int64_t pair = blockIdx.x / 2;
    const int64_t t_begin = T * pair / P;
    const int64_t t_end = T * (pair + 1) / P;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&bars->b_full[s], 1);
            mbar_init(&bars->b_empty[s], 1);
        }
        for (int kb = 0; kb < kKBMax; ++kb) {
            mbar_init(&bars->a_full[kb], 1);
            mbar_init(&bars->a_empty[kb], 1);
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(&bars->t_full[i], 1);
            mbar_init(&bars->t_empty[i], 2 * kEpiWarps);
        }
        mbar_init(&bars->staged, kEpiWarps);
        mbar_init(&bars->box_free, 1);
        mbar_init(&bars->mma_done, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_w);
        tma_prefetch_map(&tm_ok);
        if (a.n_tiles > a.n_tiles_k) {
            tma_prefetch_map(&tm_wv);
            tma_prefetch_map(&tm_ov);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    griddep_wait();  // the prepass's quantised rows (this kernel is its programmatic dependent)
    const uint32_t tmem = bars->tmem_base;
    const WaitCtl wc{&bars->abort_flag, a.status, a.timeout_ns};
    const int64_t row_end = decompress_row_end(a);

    if (warp < kFirstEpiWarp) {
      warpgroup_reg_dealloc<kCtlRegs>();
      if (warp == 0) {
        // ---------------- TMA producer (this CTA's rows and weight halves) ----------------
        if (lane == 0) {
            const uint64_t keep = policy_evict_last();
            uint32_t blk = 0;  // row blocks begun so far
            RingPos rp;
            int cur_m = -1;
            int m = static_cast<int>(t_begin / a.n_tiles);
            int nn = static_cast<int>(t_begin - static_cast<int64_t>(m) * a.n_tiles);
            bool ok = true;
            for (int t = static_cast<int>(t_begin); t < static_cast<int>(t_end) && ok; ++t) {
                const bool v_tile = nn >= a.n_tiles_k;
                const CUtensorMap* wmap = v_tile ? &tm_wv : &tm_w;
                const int n = v_tile ? nn - a.n_tiles_k : nn;
                const bool new_blk = m != cur_m;
                cur_m = m;
                for (int kb0 = 0; kb0 < KB; kb0 += kBStageKB) {
                    const int nkb = KB - kb0 < kBStageKB ? KB - kb0 : kBStageKB;
                    const uint32_t s = rp.stage, ph = rp.phase;
                    if (!mbar_wait_inl(&bars->b_empty[s], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = mapa_shared(smem_u32(&bars->b_full[s]), 0);
                    if (leader)
                        mbar_arrive_expect_tx(&bars->b_full[s],
                                              2u * static_cast<uint32_t>(nkb) * kKBBytes);
                    for (int i = 0; i < nkb; ++i)
                        tma_load_2d_pair(sB + s * kBStageBytes + i * kKBBytes, wmap, full,
                                         (kb0 + i) * 128,
                                         n * kBN + static_cast<int>(rank) * (kBN / 2), keep);
                    rp.next(kBStages);
                    if (!new_blk) continue;
                    // a k-block of the previous block's rows is free once the MMAs of that
                    // block's last tile have read it
                    for (int kb = kb0; kb < kb0 + nkb; ++kb) {
                        if (blk > 0 && !mbar_wait_inl(&bars->a_empty[kb], (blk - 1) & 1, wc)) {
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(&bars->a_full[kb], 2u * kKBBytes);
                        tma_load_2d_pair(sA + kb * kKBBytes, &tm_q,
                                         mapa_shared(smem_u32(&bars->a_full[kb]), 0), kb * 128,
                                         (m * 2 + static_cast<int>(rank)) * kBM, keep);
                    }
                }
                if (new_blk) ++blk;
                if (++nn == a.n_tiles) {
                    nn = 0;
                    ++m;
                }
            }
            if (bars->abort_flag) spin_ns(50000);  // let loads in flight land before retiring
        }
      } else if (warp == 1) {
        // ---------------- MMA issuer (even CTA) ----------------
        if (leader && lane == 0) {
            const uint32_t idesc = idesc_e4m3(256, kBN);
            const uint64_t a_desc = sdesc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc = sdesc_sw128(smem_u32(sB), 16, 1024);
            uint32_t blk = 0, kbg = 0;  // row blocks begun; k-blocks issued (accumulator kbg % 2)
            RingPos rp;
            int cur_m = -1;
            int m = static_cast<int>(t_begin / a.n_tiles);
            int nn = static_cast<int>(t_begin - static_cast<int64_t>(m) * a.n_tiles);
            bool ok = true;
            for (int t = static_cast<int>(t_begin); t < static_cast<int>(t_end) && ok; ++t) {
                const bool new_blk = m != cur_m;
                cur_m = m;
                // the MMAs of the block's last tile in this pair's range release its rows
                const bool last_of_blk = nn == a.n_tiles - 1 || t + 1 == static_cast<int>(t_end);
                for (int kb0 = 0; kb0 < KB && ok; kb0 += kBStageKB) {
                    const int kb1 = KB - kb0 < kBStageKB ? KB : kb0 + kBStageKB;
                    const uint32_t s = rp.stage;
                    if (!mbar_wait_inl(&bars->b_full[s], rp.phase, wc)) {
                        ok = false;
                        break;
                    }
                    for (int kb = kb0; kb < kb1; ++kb) {
                        const uint32_t acc = kbg & 1u;
                        if ((new_blk && !mbar_wait_inl(&bars->a_full[kb], blk & 1u, wc)) ||
                            !mbar_wait_inl(&bars->t_empty[acc], ((kbg >> 1) & 1u) ^ 1u, wc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = desc_add_bytes(a_desc, static_cast<uint32_t>(kb) * kKBBytes);
                        const uint64_t bd =
                            desc_add_bytes(b_desc, s * kBStageBytes + (kb - kb0) * kKBBytes);
                        const uint32_t d = tmem + acc * kBN;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_e4m3_pair(d, ad + 2 * k, bd + 2 * k, idesc, k != 0 ? 1u : 0u);
                        mma_commit_pair(&bars->t_full[acc], 3);
                        if (last_of_blk) mma_commit_pair(&bars->a_empty[kb], 3);
                        ++kbg;
                    }
                    mma_commit_pair(&bars->b_empty[s], 3);
                    rp.next(kBStages);
                }
                if (new_blk) ++blk;
                if (++nn == a.n_tiles) {
                    nn = 0;
                    ++m;
                }
            }
            mma_commit_pair(&bars->mma_done, 1);
            mbar_wait_inl(&bars->mma_done, 0, wc, false);
        }
      } else if (warp == 2) {
        // ---------------- store thread: one 3-D TMA store per tile ----------------
        // The 16 staged 32 x 64 boxes form [column quarter][128 rows][64 columns], the
        // layout of one {64, 128, 4} box of the output viewed as {64 columns, rows, column
        // blocks of 64}.
        int m = static_cast<int>(t_begin / a.n_tiles);
        int nn = static_cast<int>(t_begin - static_cast<int64_t>(m) * a.n_tiles);
        int cur_m = -1;
        bool blk_ok = false;
        uint32_t tile_i = 0;
        for (int t = static_cast<int>(t_begin); t < static_cast<int>(t_end); ++t) {
            const int row_blk = (m * 2 + static_cast<int>(rank)) * kBM;
            if (m != cur_m) {
                cur_m = m;
                blk_ok = row_blk < a.buffer_length && block_tma_ok(a, row_blk, row_end, lane);
            }
            if (!mbar_wait_inl(&bars->staged, tile_i & 1u, wc)) break;
            if (lane == 0) {
                if (blk_ok) {
                    const bool v_tile = nn >= a.n_tiles_k;
                    const int n = v_tile ? nn - a.n_tiles_k : nn;
                    tma_store_3d(v_tile ? &tm_ov : &tm_ok, smem_u32(sOut), 0, row_blk,
                                 n * (kBN / 64));
                    bulk_commit();
                    bulk_wait_read<0>();
                }
                mbar_arrive(&bars->box_free);
            }
            __syncwarp();
            ++tile_i;
            if (++nn == a.n_tiles) {
                nn = 0;
                ++m;
            }
        }
        if (lane == 0) bulk_wait<0>();  // every store has completed before the CTA retires
      }
    } else {
        warpgroup_reg_alloc<kEpiRegs>();
        // ---------------- 16 epilogue warps ----------------
        // Warp e reads TMEM lane quarter warp % 4 (32 rows) and the 64-column quarter e / 4
        // of each 256-column accumulator, keeping 64 fp32 running sums across a tile's
        // k-blocks.
        const int e = warp - kFirstEpiWarp;
        const int q = warp & 3;
        const int cq = e >> 2;
        const uint32_t stage = smem_u32(sOut + (cq * 4 + q) * kOutBufBytes);
        const uint32_t t_empty_leader = mapa_shared(smem_u32(&bars->t_empty[0]), 0);
        // this warp's lanes and columns of accumulator 0 (accumulator 1 is kBN columns on)
        const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16) + cq * 64;
        // 32-bit tile walk (the host keeps the tile count below 2^31): the epilogue holds 64
        // running sums and 16 loaded values, so its other state has to stay small
        const int n_tiles = a.n_tiles;
        const int t_last = static_cast<int>(t_end);
        int m = static_cast<int>(t_begin / n_tiles);
        int nn = static_cast<int>(t_begin - static_cast<int64_t>(m) * n_tiles);
        uint32_t kbg = 0;
        int cur_m = -1;
        int row0 = 0;          // first row of this warp's 32-row slab
        uint32_t valid = 0;    // bit r: slab row r is a buffer row with a source
        bool blk_ok = false;   // the store thread writes this block's tiles by TMA
        uint32_t tile_i = 0;
        float sa[kKBMax] = {0.f, 0.f, 0.f, 0.f};
        // weight scales of this warp's 128-column scale block in tile n_any; the next
        // tile's are fetched before this tile's rounding and store
        auto load_ws = [&](int n_any, float (&dst)[kKBMax]) {
            const bool vt = n_any >= a.n_tiles_k;
            const int nb = (vt ? n_any - a.n_tiles_k : n_any) * 2 + (cq >> 1);
            const float* src = (vt ? x.w_scale_v : x.w_scale) + nb * KB;
#pragma unroll
            for (int kb = 0; kb < kKBMax; ++kb) dst[kb] = kb < KB ? __ldg(src + kb) : 0.0f;
        };
        float ws[kKBMax];
        if (t_begin < t_end) load_ws(nn, ws);
        bool ok = true;
        bool stage_pending = false;  // the previous tile's box awaits its fence and arrival
        for (int t = static_cast<int>(t_begin); t < t_last && ok; ++t) {
            const bool v_tile = nn >= a.n_tiles_k;
            const int n = v_tile ? nn - a.n_tiles_k : nn;
            if (m != cur_m) {
                cur_m = m;
                row0 = (m * 2 + static_cast<int>(rank)) * kBM + q * 32;
                const int my_row = row0 + lane;
                const bool my_valid = decompress_row_source(a, my_row, row_end) >= 0;
                valid = __ballot_sync(0xffffffffu, my_valid);
                const int row_blk = (m * 2 + static_cast<int>(rank)) * kBM;
                blk_ok = row_blk < a.buffer_length && block_tma_ok(a, row_blk, row_end, lane);
#pragma unroll
                for (int kb = 0; kb < kKBMax; ++kb)
                    sa[kb] = (my_valid && kb < KB)
                                 ? x.q_scale[static_cast<int64_t>(my_row) * KB + kb]
                                 : 0.0f;
            }
            float acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
#pragma unroll
            for (int kb = 0; kb < kKBMax; ++kb) {
                if (kb >= KB) break;
                const uint32_t slot = kbg & 1u, ph = (kbg >> 1) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait_inl(&bars->t_full[slot], ph, wc))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float cs = sa[kb] * ws[kb];
                const uint32_t tbase = tq + slot * kBN;
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    uint32_t v[16];
                    tmem_ld_x16(tbase + part * 16, v);
                    tmem_ld_wait();
                    if (part == 3) {  // the accumulator has been read: back to the MMAs
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive_remote(t_empty_leader + slot * sizeof(uint64_t));
                        if (stage_pending) {
                            // the previous tile's box: its shared-memory writes are made
                            // visible to the TMA store only now, after this hand-off, so
                            // that waiting for them does not delay the MMAs
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bars->staged);
                            stage_pending = false;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; j += 2)
                        fma2(acc[part * 16 + j], acc[part * 16 + j + 1], cs,
                             __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                }
                ++kbg;
            }
            if (!ok) break;
            const int n_next = nn + 1 == n_tiles ? 0 : nn + 1;
            if (t + 1 < t_last) load_ws(n_next, ws);
            // the store thread has read the previous tile's boxes
            if (tile_i > 0 &&
                !__all_sync(0xffffffffu, mbar_wait_inl(&bars->box_free, (tile_i - 1) & 1u, wc))) {
                ok = false;
                break;
            }
            const uint32_t rowaddr = stage + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4),
                             pack_bf16x2(acc[8 * j], acc[8 * j + 1]),
                             pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]),
                             pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]),
                             pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]));
            if (blk_ok) {
                stage_pending = true;  // fence and arrival after the next tile's first hand-off
            } else if (row0 < a.buffer_length) {
                // a block with rows that must stay untouched: this warp writes its valid rows
                __syncwarp();
                const int64_t pitch = v_tile ? a.n_out_v : a.n_out;
                uint16_t* dst =
                    (v_tile ? a.v_buffer : a.k_buffer) + row0 * pitch + n * kBN + cq * 64;
                const int chunk = lane & 7;
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int r = it * 4 + (lane >> 3);
                    const uint4 v = ld_shared_v4(stage + r * 128 + ((chunk ^ (r & 7)) << 4));
                    if ((valid >> r) & 1u) st_v4(dst + r * pitch + chunk * 8, v);
                }
            }
            if (!stage_pending) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->staged);
            }
            ++tile_i;
            nn = n_next;
            if (nn == 0) ++m;
        }
        if (stage_pending) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->staged);
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_decompress_fp8_wide(const CUtensorMap& tm_q, const CUtensorMap& tm_w,
                                       const CUtensorMap& tm_wv, const CUtensorMap& tm_ok,
                                       const CUtensorMap& tm_ov, DecompressArgs args,
                                       Fp8Extra extra, int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(decompress_fp8_wide_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t max_pairs = num_sms / 2;
    const int64_t pairs = args.total_tiles < max_pairs ? args.total_tiles : max_pairs;
    return launch_dependent(decompress_fp8_wide_kernel, static_cast<unsigned>(2 * pairs),
                            kThreads, kSmemBytes, stream, tm_q, tm_w, tm_wv, tm_ok, tm_ov, args,
                            extra);
}

}  // namespace pkm
