// decompress_fp8.cu -- FP8 block-scaled latent-K decompress.
//
// The K-decompress stage of mla_prefill_decode_graph_fp8 (Modular MAX,
// attention/gpu/mla_graph): Parameters fp8_dtype / fp8_scale_dtype and
// m/n/k_scale_granularity, Args buffer_row_offsets, cache_offsets, buffer_length, w_k
// ([num_heads * qk_nope_head_dim, kv_latent_dim], e4m3) and w_k_scale.  Granularities
// m = 1, n = k = 128.
//
// Two kernels:
//   1. fp8_gather_quantize_kernel: one warp per output row (two rows in flight) resolves the
//      row through the page table, copies the bf16 latent row to k_latent_buffer with
//      16-byte vector loads/stores, and quantises its first kv_lora_rank columns per
//      128-column block (s = amax / 448, q = e4m3_rne_satfinite(x / s), fp32) into the
//      workspace.  Every row is quantised exactly once, however many n tiles consume it.
//   2. decompress_fp8_gemm_kernel: clusters of two CTAs (a CTA pair) over 256 x 128 output
//      tiles (one n tile = one weight-scale block; with w_uv the V tiles follow the K tiles
//      and reuse the same quantised rows).  Each CTA brings its 128 rows of the
//      quantised A tile (resident for the pair's range segment) and its 64-row half of the
//      tile's 128 x kv_lora_rank e4m3 W_k slice (one 3-D TMA operation, all k-blocks) into a
//      4-tile ring; the even CTA issues
//      tcgen05.mma.cta_group::2 kind::f8f6f4 (M = 256), accumulating each 128-wide k-block
//      into its own TMEM accumulator (4 x 128 columns per CTA).  8 epilogue warps per CTA
//      read each k-block as soon as its MMAs retire and combine them in registers as
//      sum_kb (s_a[row, kb] * s_w[n_tile, kb]) * acc_kb before rounding to bf16 and storing
//      k_buffer in whole 128-byte row segments (through a swizzled 4 KB shared buffer per
//      warp).  The accumulators go back to the MMAs once per tile, right after the last
//      k-block is read, so the rounding and stores overlap the next tile's MMAs.
#include <cuda_fp16.h>

#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

// ------------------------------------------------------------------------------------
// 1. gather + quantise
// ------------------------------------------------------------------------------------

// Each warp takes a contiguous range of output rows, two at a time, resolving them with a
// forward walk (one binary search per warp, page ids reused along a page): the rows are
// resolved and all their loads issued before any arithmetic.  A lane holds 16 nope values (32 bytes), so a 128-column
// block is eight lanes (kv_lora_rank <= 512 fits one pass); lanes below rope_dim / 8 also
// carry one 16-byte chunk of the rope columns.
constexpr int kGatherRows = 2;

__global__ void __launch_bounds__(256)
    fp8_gather_quantize_kernel(const DecompressArgs a, const Fp8Extra x) {
    griddep_launch_dependents();  // the GEMM may start its prologue; it waits for our writes
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t row_end = decompress_row_end(a);
    const int R = a.kv_lora_rank;
    const int C = a.latent_cols;
    const int kblocks = R / 128;
    const bool nope = lane * 16 < R;
    const bool rope = lane < (C - R) / 8;
    // this warp's rows: a contiguous range, resolved by a forward walk
    const int64_t rb = row_end * warp_id / nwarps;
    const int64_t re = row_end * (warp_id + 1) / nwarps;
    RowSourceWalk walk(a, rb);
    for (int64_t r0 = rb; r0 < re; r0 += kGatherRows) {
        int64_t off[kGatherRows];
        uint4 nv[kGatherRows][2], rv[kGatherRows];
#pragma unroll
        for (int u = 0; u < kGatherRows; ++u) {
            const int64_t r = r0 + u;
            off[u] = r < re ? walk.source(a, r) : -1;
            const uint16_t* src = a.cache_layer + (off[u] >= 0 ? off[u] : 0);
            const bool live = off[u] >= 0;
            nv[u][0] = live && nope ? ld_nc_v4(src + lane * 16) : make_uint4(0u, 0u, 0u, 0u);
            nv[u][1] = live && nope ? ld_nc_v4(src + lane * 16 + 8) : make_uint4(0u, 0u, 0u, 0u);
            rv[u] = live && rope ? ld_nc_v4(src + R + lane * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kGatherRows; ++u) {
            if (off[u] < 0) {  // warp-uniform
                if (off[u] == -2 && lane == 0) report(a.status, PKM_ERR_OUT_OF_RANGE);
                continue;
            }
            const int64_t r = r0 + u;
            uint16_t* lat = a.k_latent + r * C;
            if (nope) {
                st_v4(lat + lane * 16, nv[u][0]);
                st_v4(lat + lane * 16 + 8, nv[u][1]);
            }
            if (rope) st_v4(lat + R + lane * 8, rv[u]);
            float f[16];
            const uint32_t w[8] = {nv[u][0].x, nv[u][0].y, nv[u][0].z, nv[u][0].w,
                                   nv[u][1].x, nv[u][1].y, nv[u][1].z, nv[u][1].w};
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
            const bool all_fast = __all_sync(0xffffffffu, qb.fast || !nope);
            if (!nope) continue;
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
            st_v4(x.q_latent + r * R + lane * 16, make_uint4(o[0], o[1], o[2], o[3]));
            if ((lane & 7) == 0) x.q_scale[r * kblocks + lane / 8] = s;
        }
    }
}

// 1b. gather from a quantised cache: the slot already holds the codes and the block
// scales, so they are copied as they are; k_latent (optional) gets the dequantised nope
// values fl32(e4m3 * scale) rounded to bf16 and the rope columns bit for bit.

// Two e4m3 codes (first in the low byte) to fp32, exactly (e4m3 is a subset of f16).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two, float& lo, float& hi) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two)));
    lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
    hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

__global__ void __launch_bounds__(256)
    fp8_gather_qcache_kernel(const DecompressArgs a, const Fp8Extra x) {
    griddep_launch_dependents();  // the GEMM may start its prologue; it waits for our writes
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t row_end = decompress_row_end(a);
    const int R = a.kv_lora_rank;
    const int C = a.latent_cols;
    const int P = C - R;
    const int code_chunks = R / 16;  // 16 codes per 16-byte chunk
    const int rope_chunks = P / 8;   // 8 bf16 values per 16-byte chunk
    const int kblocks = R / 128;
    for (int64_t r = warp_id; r < row_end; r += nwarps) {
        const int64_t off = decompress_row_source(a, r, row_end);
        if (off < 0) {
            if (off == -2 && lane == 0) report(a.status, PKM_ERR_OUT_OF_RANGE);
            continue;
        }
        const uint8_t* slot = a.qcache_layer + off;
        const float* scales = reinterpret_cast<const float*>(slot + R + 2 * P);
        uint8_t* qrow = x.q_latent + r * R;
        for (int c = lane; c < code_chunks; c += 32) {
            const uint4 v = ld_nc_v4(slot + c * 16);
            st_v4(qrow + c * 16, v);
            if (a.k_latent != nullptr) {
                const float s = __ldg(scales + c / 8);  // 8 chunks = one 128-column block
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float f0, f1, f2, f3;
                    e4m3x2_to_f32(w[i] & 0xFFFFu, f0, f1);
                    e4m3x2_to_f32(w[i] >> 16, f2, f3);
                    o[2 * i] = pack_bf16x2(__fmul_rn(f0, s), __fmul_rn(f1, s));
                    o[2 * i + 1] = pack_bf16x2(__fmul_rn(f2, s), __fmul_rn(f3, s));
                }
                uint16_t* lat = a.k_latent + r * C + c * 16;
                st_v4(lat, make_uint4(o[0], o[1], o[2], o[3]));
                st_v4(lat + 8, make_uint4(o[4], o[5], o[6], o[7]));
            }
        }
        if (lane < kblocks) x.q_scale[r * kblocks + lane] = __ldg(scales + lane);
        if (a.k_latent != nullptr)
            for (int c = lane; c < rope_chunks; c += 32)
                st_v4(a.k_latent + r * C + R + c * 8, ld_nc_v4(slot + R + c * 16));
    }
}

// ------------------------------------------------------------------------------------
// 2. block-scaled GEMM
// ------------------------------------------------------------------------------------

constexpr int kThreads = 448;                 // producer, MMA, 8 epilogue, 4 store warps
constexpr int kBM = 128;                      // rows per CTA (256 per pair)
constexpr int kBN = 128;                      // pair N tile = one weight-scale block
constexpr int kKBMax = 4;                     // kv_lora_rank <= 512
constexpr int kABlockBytes = kBM * 128;       // 128 rows x 128 e4m3
constexpr int kStages = 4;
constexpr int kBKBlockBytes = (kBN / 2) * 128;        // this CTA's 64 weight rows x 128 e4m3
constexpr int kBStageBytes = kKBMax * kBKBlockBytes;  // a tile's weight half: 32 KB
constexpr int kEpiWarps = 8;
constexpr int kStoreWarps = 4;
constexpr int kFirstStoreWarp = 2 + kEpiWarps;
constexpr int kOutBufBytes = 32 * 128;
constexpr uint32_t kTmemCols = 512;           // kKBMax accumulators x 128 columns

struct Bars {
    uint64_t b_full[kStages];   // even CTA: both halves of a W_k stage landed
    uint64_t b_empty[kStages];  // both CTAs: the pair's MMAs are done with a stage
    uint64_t a_full;            // even CTA: both CTAs' A tiles landed
    uint64_t a_empty;           // both CTAs: the MMAs are done with A
    uint64_t t_full[kKBMax];    // both CTAs: k-block accumulator ready
    uint64_t t_drained;         // even CTA: both CTAs' epilogues read all of a tile's
                                // accumulators
    uint64_t st_full;           // the epilogue warps staged a tile's rounded results
    uint64_t st_empty;          // the store warps wrote them out; the staging is free
    struct {
        uint16_t* dst;          // first element of the box in k_buffer / v_buffer
        int64_t pitch;          // row pitch in elements
        uint32_t valid;         // bit r: row r of the box is written
    } box[kEpiWarps];           // where each epilogue warp's staged 32 x 64 box goes
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decompress_fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_q,
                               const __grid_constant__ CUtensorMap tm_w,
                               const __grid_constant__ CUtensorMap tm_wv,
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
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->b_full[s], 1);
            mbar_init(&bars->b_empty[s], 1);
        }
        mbar_init(&bars->a_full, 1);
        mbar_init(&bars->a_empty, 1);
        for (int i = 0; i < kKBMax; ++i) mbar_init(&bars->t_full[i], 1);
        mbar_init(&bars->t_drained, 2 * kEpiWarps);
        mbar_init(&bars->st_full, kEpiWarps);
        mbar_init(&bars->st_empty, kStoreWarps);
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
        if (a.n_tiles > a.n_tiles_k) tma_prefetch_map(&tm_wv);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    griddep_wait();  // the prepass's quantised rows (this kernel is its programmatic dependent)
    const uint32_t tmem = bars->tmem_base;
    const WaitCtl wc{&bars->abort_flag, a.status, a.timeout_ns};
    const int64_t row_end = decompress_row_end(a);

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t keep = policy_evict_last();
            const uint32_t a_full_leader = mapa_shared(smem_u32(&bars->a_full), 0);
            uint32_t seg = 0;
            RingPos rp;
            int64_t cur_m = -1;
            bool ok = true;
            for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid() && ok; w.next()) {
                const int64_t m_pair = w.m;
                // n tiles [0, n_tiles_k) project with W_k, the rest with w_uv
                const bool v_tile = w.n >= a.n_tiles_k;
                const CUtensorMap* wmap = v_tile ? &tm_wv : &tm_w;
                const int n = v_tile ? w.n - a.n_tiles_k : w.n;
                if (m_pair != cur_m) {
                    cur_m = m_pair;
                    if (seg > 0 && !mbar_wait(&bars->a_empty, (seg - 1) & 1, wc)) break;
                    if (leader)
                        mbar_arrive_expect_tx(&bars->a_full,
                                              2u * static_cast<uint32_t>(KB) * kABlockBytes);
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load_2d_pair(sA + kb * kABlockBytes, &tm_q, a_full_leader, kb * 128,
                                         static_cast<int32_t>((m_pair * 2 + rank) * kBM), keep);
                    ++seg;
                }
                {  // one 3-D operation: all k-blocks of this CTA's 64 weight rows
                    const uint32_t s = rp.stage, ph = rp.phase;
                    if (!mbar_wait(&bars->b_empty[s], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    if (leader)
                        mbar_arrive_expect_tx(&bars->b_full[s],
                                              2u * static_cast<uint32_t>(KB) * kBKBlockBytes);
                    tma_load_3d_pair(sB + s * kBStageBytes, wmap,
                                     mapa_shared(smem_u32(&bars->b_full[s]), 0), 0,
                                     n * kBN + static_cast<int>(rank) * (kBN / 2), 0, keep);
                    rp.next(kStages);
                }
            }
            if (bars->abort_flag) spin_ns(50000);  // let loads in flight land before retiring
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            const uint32_t idesc = idesc_e4m3(256, kBN);
            // operand descriptors built once; each MMA adds its offset (16-byte units)
            const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), 16, 1024);
            uint32_t tile_i = 0, seg = 0;
            RingPos rp;
            int64_t cur_m = -1;
            bool ok = true;
            for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid() && ok; w.next()) {
                const int64_t m = w.m;
                if (m != cur_m) {
                    if (cur_m >= 0) {
                        mma_commit_pair(&bars->a_empty, 3);
                        ++seg;
                    }
                    cur_m = m;
                    if (!mbar_wait(&bars->a_full, seg & 1, wc)) break;
                }
                const uint32_t s = rp.stage, ph = rp.phase;
                // the accumulators are handed back once per tile: a wait, a fence and a
                // commit between the MMAs of every k-block left the tensor pipe idle for a
                // third of the time
                if (!mbar_wait(&bars->b_full[s], ph, wc) ||
                    !mbar_wait(&bars->t_drained, (tile_i & 1) ^ 1, wc))
                    break;
                tc_fence_after();
                const uint64_t b_stage = desc_add_bytes(b_desc0, s * kBStageBytes);
                for (int kb = 0; kb < KB; ++kb) {
                    const uint64_t ad = desc_add_bytes(a_desc0, static_cast<uint32_t>(kb) * kABlockBytes);
                    const uint64_t bd = desc_add_bytes(b_stage, static_cast<uint32_t>(kb) * kBKBlockBytes);
                    const uint32_t d = tmem + static_cast<uint32_t>(kb) * kBN;
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // K = 32 e4m3 = 32 bytes a step
                        mma_e4m3_pair(d, ad + 2 * k, bd + 2 * k, idesc, k != 0 ? 1u : 0u);
                    mma_commit_pair(&bars->t_full[kb], 3);
                }
                mma_commit_pair(&bars->b_empty[s], 3);
                rp.next(kStages);
                ++tile_i;
            }
            mma_commit_pair(&bars->mma_done, 1);
            mbar_wait(&bars->mma_done, 0, wc, false);
        }
    } else if (warp < kFirstStoreWarp) {
        // 8 epilogue warps: warp w reads TMEM lane quarter w % 4 (32 rows) and one 64-column
        // half of the 128-column tile and keeps 64 fp32 partial sums.  The rounded results
        // go to shared memory; the store warps write them out while these warps go on to the
        // next tile (one SM moves only ~26 bytes per cycle to global memory, so storing a
        // tile takes about as long as computing it).
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const uint32_t stage = smem_u32(sOut + (warp - 2) * kOutBufBytes);
        const uint32_t t_drained_leader = mapa_shared(smem_u32(&bars->t_drained), 0);
        uint32_t tile_i = 0;
        int64_t cur_m = -1;
        uint16_t* row0 = a.k_buffer;   // first row of this warp's 32-row slab, in k_buffer
        uint16_t* row0v = a.v_buffer;  // and in v_buffer
        uint32_t valid = 0;            // bit r: slab row r is a buffer row with a source
        float sa[kKBMax] = {0.f, 0.f, 0.f, 0.f};
        // weight scales of an n tile (tile id n_any in [0, n_tiles)); the next tile's are
        // fetched before this tile's rounding and stores, off the first k-block's path
        auto load_ws = [&](int n_any, float (&dst)[kKBMax]) {
            const bool vt = n_any >= a.n_tiles_k;
            const float* src = (vt ? x.w_scale_v : x.w_scale) +
                               static_cast<int64_t>(vt ? n_any - a.n_tiles_k : n_any) * KB;
#pragma unroll
            for (int kb = 0; kb < kKBMax; ++kb) dst[kb] = kb < KB ? __ldg(src + kb) : 0.0f;
        };
        float ws[kKBMax];
        if (t_begin < t_end) load_ws(static_cast<int>(t_begin % a.n_tiles), ws);
        bool ok = true;
        for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid() && ok; w.next()) {
            const int64_t m_pair = w.m;
            const bool v_tile = w.n >= a.n_tiles_k;
            const int n = v_tile ? w.n - a.n_tiles_k : w.n;
            if (m_pair != cur_m) {
                cur_m = m_pair;
                const int64_t first = (m_pair * 2 + rank) * kBM + q * 32;
                const int64_t my_row = first + lane;
                const bool my_valid = decompress_row_source(a, my_row, row_end) >= 0;
                row0 = a.k_buffer + first * a.n_out;
                if (a.v_buffer != nullptr) row0v = a.v_buffer + first * a.n_out_v;
                valid = __ballot_sync(0xffffffffu, my_valid);
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
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&bars->t_full[kb], tile_i & 1, wc))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float cs = sa[kb] * ws[kb];
                const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(kb) * kBN + h * 64;
                // two 32-column halves: 14 warps leave 128 registers a thread
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    tmem_ld_x32(tbase + half * 32, v);
                    tmem_ld_wait();
                    if (half == 1 && kb == KB - 1) {  // every accumulator has been read
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote(t_drained_leader);
                    }
                    // packed FMAs: the two epilogue warps on the MMA warp's scheduler slow
                    // its MMA issue in proportion to the instructions they issue
#pragma unroll
                    for (int j = 0; j < 32; j += 2)
                        fma2(acc[half * 32 + j], acc[half * 32 + j + 1], cs,
                             __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                }
            }
            if (!ok) break;
            if (w.t + 1 < t_end) load_ws(w.n + 1 == a.n_tiles ? 0 : w.n + 1, ws);
            // stage the rounded box once the store warps have written out the previous one
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->st_empty, (tile_i & 1) ^ 1, wc))) {
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
            if (lane == 0) {
                auto& b = bars->box[warp - 2];
                b.dst = (v_tile ? row0v : row0) + n * kBN + h * 64;
                b.pitch = v_tile ? a.n_out_v : a.n_out;
                b.valid = valid;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->st_full);
            ++tile_i;
        }
    } else {
        // 4 store warps: store warp s writes out the boxes of epilogue warps 2s and 2s + 1,
        // each as whole 128-byte row segments (eight lanes per row).
        const int s = warp - kFirstStoreWarp;
        const int chunk = lane & 7;
        uint32_t tile_i = 0;
        for (TileWalk w(t_begin, t_end, a.n_tiles); w.valid(); w.next()) {
            if (!mbar_wait(&bars->st_full, tile_i & 1, wc)) break;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int src = 2 * s + e;
                const uint32_t box = smem_u32(sOut + src * kOutBufBytes);
                uint16_t* dst = bars->box[src].dst;
                const int64_t pitch = bars->box[src].pitch;
                const uint32_t valid = bars->box[src].valid;
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int r = it * 4 + (lane >> 3);
                    const uint4 v = ld_shared_v4(box + r * 128 + ((chunk ^ (r & 7)) << 4));
                    if ((valid >> r) & 1u) st_v4(dst + r * pitch + chunk * 8, v);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->st_empty);
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

cudaError_t launch_fp8_gather_quantize(DecompressArgs args, Fp8Extra extra, int num_sms,
                                       cudaStream_t stream) {
    const int64_t rows = args.buffer_length;
    int64_t blocks = (rows + 8 * kGatherRows - 1) / (8 * kGatherRows);  // 8 warps per block
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fp8_gather_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(args, extra);
    return cudaGetLastError();
}

cudaError_t launch_fp8_gather_qcache(DecompressArgs args, Fp8Extra extra, int num_sms,
                                     cudaStream_t stream) {
    const int64_t rows = args.buffer_length;
    int64_t blocks = (rows + 7) / 8;  // 8 warps (rows in flight) per block
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fp8_gather_qcache_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(args, extra);
    return cudaGetLastError();
}

cudaError_t launch_decompress_fp8_gemm(const CUtensorMap& tm_q, const CUtensorMap& tm_w,
                                       const CUtensorMap& tm_wv, DecompressArgs args,
                                       Fp8Extra extra, int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(decompress_fp8_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t max_pairs = num_sms / 2;
    const int64_t pairs = args.total_tiles < max_pairs ? args.total_tiles : max_pairs;
    return launch_dependent(decompress_fp8_gemm_kernel, static_cast<unsigned>(2 * pairs), kThreads,
                            kSmemBytes, stream, tm_q, tm_w, tm_wv, args, extra);
}

}  // namespace pkm
