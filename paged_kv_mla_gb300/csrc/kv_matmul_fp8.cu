// kv_matmul_fp8.cu -- the ragged GEMM of kv_matmul_ragged_paged in FP8 with block scales,
// written into the paged K/V cache.
//
// kv_matmul_ragged_paged (Modular MAX, nn/kv_cache_ragged), description and Args: Y =
// hidden_state x weight on the ragged rows, row i of request b written at cache position
// cache_lengths[b] + i, columns split K then V.  In FP8 form (the fp8 type and m/n/k scale
// granularities of mla_prefill_decode_graph_fp8): the bf16 hidden rows are quantised per
// token per 128 columns (s = amax / 448, q = e4m3_rne(x / s), fp32), the weight is e4m3
// [n_out, k_in] with fp32 scales per 128 x 128 block, and
//     Y[r, n] = bf16( sum_kb s_x[r, kb] * s_w[n / 128, kb] * sum_{k in kb} q_x[r, k] q_w[n, k] ).
//
// Two kernels:
//   1. fp8_quantize_rows_kernel: warps quantise 512-column slices of the hidden rows into the
//      workspace (codes [M, k_in]; scales k-block-major, [k_in / 128, M], so that the
//      epilogue's per-k-block scale loads of 32 consecutive rows are one 128-byte line).
//   2. kv_matmul_fp8_kernel: clusters of two CTAs over 256 x 256 output tiles (two
//      weight-scale blocks; one accumulator hand-off per k-block then covers 256 output
//      columns, twice as many as with N = 128, and the hand-off, not the MMA rate, bounds
//      this GEMM).  Each CTA streams, per 128-wide k-block, its 128 rows of quantised A and
//      its 128-row half of the weight through a 5-stage TMA ring; the even CTA issues
//      tcgen05.mma.cta_group::2 kind::f8f6f4 (M = 256) into one of two 256-column TMEM
//      accumulators.  Because every k-block carries its own scales, 16 epilogue warps per
//      CTA (32 rows x 64 columns each) fold each k-block's accumulator into fp32 running sums
//      (acc += s_x * s_w * partial, packed fp32x2 FMAs) and hand it back at once, so the
//      MMAs of the next k-block proceed meanwhile.  After a tile's last k-block each warp
//      rounds its sums to bf16 and scatters its rows' 64-column segments to their
//      (page, slot) in the K or V plane through a swizzled shared-memory box.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

// ------------------------------------------------------------------------------------
// 1. quantise the hidden rows
// ------------------------------------------------------------------------------------

// Grid: blockIdx.y = a 512-column slice of the rows (four 128-column blocks, eight lanes a
// block, 16 values = 32 bytes a lane), blockIdx.x and the warp pick rows.  Each warp takes
// four rows at a time and issues their loads before any arithmetic, so that enough bytes
// are in flight to keep HBM busy.
constexpr int kQuantUnroll = 4;

__global__ void __launch_bounds__(256)
    fp8_quantize_rows_kernel(const KvMatmulArgs a, const KvFp8Extra x) {
    griddep_launch_dependents();  // the GEMM may start its prologue; it waits for our writes
    const int lane = threadIdx.x & 31;
    const int64_t warp_x = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nwarps_x = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int K = a.k_in;
    const int col = static_cast<int>(blockIdx.y) * 512 + lane * 16;  // this lane's 16 columns
    const bool act = col < K;  // a last slice of fewer blocks leaves whole 8-lane groups idle
    const int64_t M = a.total_rows;
    for (int64_t r0 = warp_x; r0 < M; r0 += kQuantUnroll * nwarps_x) {
        uint4 v[kQuantUnroll][2];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t r = r0 + u * nwarps_x;
            const bool ld = act && r < M;
            const uint16_t* src = a.hidden + r * K + col;
            v[u][0] = ld ? ld_nc_v4(src) : make_uint4(0u, 0u, 0u, 0u);
            v[u][1] = ld ? ld_nc_v4(src + 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t r = r0 + u * nwarps_x;
            if (r >= M) break;  // warp-uniform
            float f[16];
            const uint32_t w[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                                   v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
#pragma unroll
            for (int i = 0; i < 8; ++i) bf16x2_to_f32(w[i], f[2 * i], f[2 * i + 1]);
            float amax = fmax3_abs(fmax3_abs(f[0], f[1], f[2]), fmax3_abs(f[3], f[4], f[5]),
                                   fmax3_abs(f[6], f[7], f[8]));
            amax = fmax3_abs(amax, fmax3_abs(f[9], f[10], f[11]), fmax3_abs(f[12], f[13], f[14]));
            amax = fmax3_abs(amax, f[15], 0.0f);
#pragma unroll
            for (int sh = 4; sh >= 1; sh >>= 1)  // the eight lanes of one block
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
            const E4m3Block qb(amax);
            const float s = qb.s;
            // one warp-uniform choice of the quotient path (every block in the fast range
            // is the rule); lanes without columns take no part in it
            const bool all_fast = __all_sync(0xffffffffu, qb.fast || !act);
            if (!act) continue;
            uint32_t o[4];
            if (all_fast) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o[i] = qb.codes4_fast(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o[i] = qb.codes4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
            }
            st_v4(x.q + r * K + col, make_uint4(o[0], o[1], o[2], o[3]));
            if ((lane & 7) == 0) x.q_scale[static_cast<int64_t>(col / 128) * M + r] = s;
        }
    }
}

// ------------------------------------------------------------------------------------
// 2. block-scaled GEMM + scatter
// ------------------------------------------------------------------------------------

constexpr int kEpiWarps = 16;
constexpr int kThreads = 32 * (2 + kEpiWarps);  // producer, MMA, 16 epilogue warps
constexpr int kBM = 128;                       // rows per CTA (256 per pair)
constexpr int kBN = 256;                       // pair N tile: two weight-scale blocks
constexpr int kABytes = kBM * 128;             // 128 rows x 128 e4m3
constexpr int kBBytes = (kBN / 2) * 128;       // this CTA's 128 weight rows x 128 e4m3
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStages = 5;
constexpr int kAcc = 2;                        // TMEM accumulators of 256 columns
constexpr int kOutBufBytes = 32 * 128;         // a warp's 32 x 64 bf16 box
constexpr uint32_t kTmemCols = kAcc * kBN;

struct Bars {
    uint64_t full[kStages];     // even CTA: both CTAs' A and B halves of a stage landed
    uint64_t empty[kStages];    // both CTAs: the pair's MMAs are done with a stage
    uint64_t t_full[kAcc];      // both CTAs: a k-block's accumulator is ready
    uint64_t t_empty[kAcc];     // even CTA: both CTAs' epilogues have read it
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
    kv_matmul_fp8_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_w, const KvMatmulArgs a,
                         const KvFp8Extra x) {
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
    const int KB = a.k_in / 128;
    const int NB = a.n_out / 128;     // weight-scale blocks along n
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
        for (int i = 0; i < kAcc; ++i) {
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
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_w);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    griddep_wait();  // the prepass's quantised rows (this kernel is its programmatic dependent)
    const uint32_t tmem = bars->tmem_base;
    const WaitCtl wc{&bars->abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        if (lane == 0) {
            // A rows are re-read for every n tile of their block and the weight by every
            // block: both are kept in L2 ahead of the scattered cache writes
            const uint64_t keep = policy_evict_last();
            RingPos rp;
            bool issued[kStages] = {};
            uint32_t last_phase[kStages] = {};
            bool ok = true;
            for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid() && ok; w.next()) {
                const int64_t m = w.m * 2 + rank;  // this CTA's 128-row block
                const int n = static_cast<int>(w.n);
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t s = rp.stage, ph = rp.phase;
                    if (!mbar_wait(&bars->empty[s], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = sStages + s * kStageBytes;
                    const uint32_t full_leader = mapa_shared(smem_u32(&bars->full[s]), 0);
                    if (leader) mbar_arrive_expect_tx(&bars->full[s], 2u * kStageBytes);
                    tma_load_2d_pair(st, &tm_q, full_leader, kb * 128,
                                     static_cast<int32_t>(m * kBM), keep);
                    // weight rows past n_out (a half tile at the end) load as zeros
                    tma_load_2d_pair(st + kABytes, &tm_w, full_leader, kb * 128,
                                     n * kBN + static_cast<int>(rank) * (kBN / 2), keep);
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
            const uint32_t idesc = idesc_e4m3(256, kBN);
            // operand descriptors built once; each MMA adds its offset (16-byte units)
            const uint64_t a_desc0 = sdesc_sw128(smem_u32(sStages), 16, 1024);
            const uint64_t b_desc0 = sdesc_sw128(smem_u32(sStages + kABytes), 16, 1024);
            RingPos rp;
            uint32_t kbg = 0;  // k-blocks issued so far: accumulator kbg % kAcc
            bool ok = true;
            for (int64_t t = t_begin; t < t_end && ok; ++t) {
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t s = rp.stage, ph = rp.phase;
                    const uint32_t acc = kbg % kAcc, aph = (kbg / kAcc) & 1;
                    if (!mbar_wait(&bars->full[s], ph, wc) ||
                        !mbar_wait(&bars->t_empty[acc], aph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_add_bytes(a_desc0, s * kStageBytes);
                    const uint64_t bd = desc_add_bytes(b_desc0, s * kStageBytes);
                    const uint32_t d = tmem + acc * kBN;
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // K = 32 e4m3 = 32 bytes a step
                        mma_e4m3_pair(d, ad + 2 * k, bd + 2 * k, idesc, k != 0 ? 1u : 0u);
                    mma_commit_pair(&bars->t_full[acc], 3);
                    mma_commit_pair(&bars->empty[s], 3);
                    rp.next(kStages);
                    ++kbg;
                }
            }
            mma_commit_pair(&bars->mma_done, 1);
            mbar_wait(&bars->mma_done, 0, wc, false);
        }
    } else {
        // 16 epilogue warps: warp w reads TMEM lane quarter w % 4 (32 rows) and one 64-column
        // quarter of the tile, keeps 64 fp32 running sums across the tile's k-blocks, and at
        // the end of the tile rounds them and scatters its rows' 64-column segments.
        const int e = warp - 2;
        const int q = warp & 3;
        const int cq = e >> 2;                  // column quarter 0..3
        const uint32_t stage = smem_u32(sOut + e * kOutBufBytes);
        const uint32_t t_empty_leader = mapa_shared(smem_u32(&bars->t_empty[0]), 0);
        uint32_t kbg = 0;
        int64_t cur_m = -1, my_dst = -1, my_row = 0;
        bool ok = true;
        for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid() && ok; w.next()) {
            const int64_t m = w.m * 2 + rank;
            const int n = static_cast<int>(w.n);
            if (m != cur_m) {
                cur_m = m;
                my_row = m * kBM + q * 32 + lane;
                my_dst = kv_row_dest(a, my_row);
                if (my_dst == -2 && cq == 0) report(a.status, PKM_ERR_OUT_OF_RANGE);
            }
            const int nb = n * 2 + (cq >> 1);   // weight-scale block of these columns
            const bool cols_live = nb < NB;     // false in the empty half of a last half tile
            // scales of this row and column block, fetched two k-blocks ahead of their use
            // (the row scales of a k-block are contiguous over rows: one line per warp)
            const float* scol = x.q_scale + my_row;
            const int64_t sstep = a.total_rows;
            const float* wrow = x.w_scale + static_cast<int64_t>(cols_live ? nb : 0) * KB;
            const bool live = my_dst >= 0 && cols_live;
            float sa0 = live ? __ldg(scol) : 0.0f, ws0 = __ldg(wrow);
            float sa1 = (live && KB > 1) ? __ldg(scol + sstep) : 0.0f;
            float ws1 = KB > 1 ? __ldg(wrow + 1) : 0.0f;
            float acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
            for (int kb = 0; kb < KB; ++kb) {
                const float cs = sa0 * ws0;
                sa0 = sa1;
                ws0 = ws1;
                if (kb + 2 < KB) {
                    sa1 = live ? __ldg(scol + (kb + 2) * sstep) : 0.0f;
                    ws1 = __ldg(wrow + kb + 2);
                }
                const uint32_t slot = kbg % kAcc, ph = (kbg / kAcc) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->t_full[slot], ph, wc))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase =
                    tmem + (static_cast<uint32_t>(q * 32) << 16) + slot * kBN + cq * 64;
                // four 16-column quarters: 18 warps leave under 100 registers a thread
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
                    }
#pragma unroll
                    for (int j = 0; j < 16; j += 2)
                        fma2(acc[part * 16 + j], acc[part * 16 + j + 1], cs,
                             __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                }
                ++kbg;
            }
            if (!ok || !cols_live) continue;
            // round, stage the 32 x 64 box (swizzled 128-byte rows), scatter each row's
            // segment to its slot, eight lanes a row; 64 columns lie in one K or V plane
            const uint32_t rowaddr = stage + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4),
                             pack_bf16x2(acc[8 * j], acc[8 * j + 1]),
                             pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]),
                             pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]),
                             pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]));
            __syncwarp();
            const int col0 = n * kBN + cq * 64;
            const int64_t pc = col0 < a.head_elems ? col0 : a.kv_stride + (col0 - a.head_elems);
            const int chunk = lane & 7;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + (lane >> 3);
                const int64_t d = __shfl_sync(0xffffffffu, my_dst, r);
                const uint4 v = ld_shared_v4(stage + r * 128 + ((chunk ^ (r & 7)) << 4));
                if (d >= 0) st_v4(a.cache_layer + pc + d + chunk * 8, v);
            }
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_kv_matmul_fp8(const CUtensorMap& tm_q, const CUtensorMap& tm_w,
                                 KvMatmulArgs args, KvFp8Extra extra, int num_sms,
                                 cudaStream_t stream) {
    const int slices = (args.k_in + 511) / 512;
    int64_t bx = (static_cast<int64_t>(args.total_rows) + 8 * kQuantUnroll - 1) / (8 * kQuantUnroll);
    // one wave: four 256-thread blocks an SM are resident at the kernel's register count
    const int64_t cap = (static_cast<int64_t>(num_sms) * 4 + slices - 1) / slices;
    if (bx > cap) bx = cap;
    if (bx < 1) bx = 1;
    fp8_quantize_rows_kernel<<<dim3(static_cast<unsigned>(bx), static_cast<unsigned>(slices)), 256,
                               0, stream>>>(args, extra);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kv_matmul_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t max_pairs = num_sms / 2;
    const int64_t pairs = args.total_tiles < max_pairs ? args.total_tiles : max_pairs;
    return launch_dependent(kv_matmul_fp8_kernel, static_cast<unsigned>(2 * pairs), kThreads,
                            kSmemBytes, stream, tm_q, tm_w, args, extra);
}

}  // namespace pkm
