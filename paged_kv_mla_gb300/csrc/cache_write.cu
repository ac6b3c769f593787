// cache_write.cu -- the cache-write side of MLA: new latent rows are RMS-normalised and
// rotated, then stored into the paged latent cache.
//
// mla_prefill_decode_graph_fp8 (Modular MAX, attention/gpu/mla_graph), Args kv_input_fn
// (the new latent rows, [tot_seq_len, cache_head_dim]), kv_norm_gamma (the RMSNorm scale
// vector, [kv_lora_rank]), epsilon, freqs_cis (rotary factors per position, [max_seq_len,
// qk_rope_head_dim]), input_row_offsets, kv_collection and layer_idx.  Row i of request b is token position cache_lengths[b] + i
// (the position kv_matmul_ragged_paged gives new tokens); its first R columns become
// x_k * gamma_k / sqrt(mean_k x_k^2 + epsilon), its last P columns are rotated pair by pair
// by the (cos, sin) pairs of freqs_cis[position], and the row is stored, rounded to bf16,
// into that position's slot of the layer.
//
// A streaming kernel, HBM-bound (2 x 1152 bytes a row for DeepSeek-V3 shapes).  One
// persistent CTA per SM owns a contiguous range of rows, taken 30 at a time (a chunk)
// through a ring of shared-memory stages.  In the producer warp lane i < 30 resolves row i's
// position (its request only moves forward, so the offsets and cache lengths are re-read
// once per request) and loads its page id while the stage is still in use; once the stage
// is free the lanes write slots and page ids into it, each run of rows of one request
// bulk-copies its (consecutive) freqs_cis rows, lane 0 bulk-copies the chunk's rows, and
// all of it completes on the stage's barrier.  Each of 15
// consumer warps then takes two rows of the chunk out of shared memory, frees the stage,
// reduces the sum of squares across the warp and writes the normalised and rotated rows
// (fp32 arithmetic, rounded to bf16) straight into their slots with 16-byte stores.
// Nothing else in the cache is written.
//
// Into a quantised cache (PagedKVCacheCollection's scale_dtype_ / quantization_granularity_)
// the rounded bf16 values of each 128-column block are quantised on the spot, the block
// being the 16 chunks of one half-warp: s = amax / 448 (fp32), codes e4m3_rne_satfinite(y / s)
// with the codes of the correctly rounded fp32 quotient; the slot gets the codes, the bf16
// rope columns and the scales.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

constexpr int kConsumerWarps = 15;
constexpr int kRowsPerWarp = 2;
constexpr int kChunkRows = kConsumerWarps * kRowsPerWarp;  // 30 rows a stage
constexpr int kThreads = 32 * (1 + kConsumerWarps);        // warp 0: producer
constexpr int kMaxStages = 12;
constexpr int kSmemBudget = 220 * 1024;
constexpr int32_t kSlotNone = -1;        // no request covers the row
constexpr int32_t kSlotOutOfRange = -2;  // position past freqs_cis or the page-table row

// Byte offsets inside one stage: the chunk's rows, their freqs_cis rows, page ids, slots.
struct StageLayout {
    uint32_t freqs, page, slot, bytes;
};

struct Bars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int abort_flag;
};

// The request a lane's rows belong to.  A lane visits its rows in increasing order, so after
// one binary search the request only ever moves forward.
struct RowCursor {
    int b;
    uint32_t lo, hi, cl;  // input_row_offsets[b], input_row_offsets[b + 1], cache_lengths[b]

    __device__ __forceinline__ void init(const CacheWriteArgs& a, int64_t r) {
        const uint32_t* iro = a.row_offsets;
        int l = 0, h = a.batch;  // largest b with iro[b] <= r (0 when r < iro[0])
        while (h - l > 1) {
            const int mid = (l + h) >> 1;
            if (static_cast<int64_t>(__ldg(iro + mid)) <= r) l = mid;
            else h = mid;
        }
        b = l;
        lo = __ldg(iro + l);
        hi = __ldg(iro + l + 1);
        cl = __ldg(a.cache_lengths + l);
    }

    // Moves to the request covering r (r never decreases); false when none does.
    __device__ __forceinline__ bool seek(const CacheWriteArgs& a, int64_t r) {
        while (r >= static_cast<int64_t>(hi) && b + 1 < a.batch) {
            ++b;
            lo = hi;
            hi = __ldg(a.row_offsets + b + 1);
            cl = __ldg(a.cache_lengths + b);
        }
        return r >= static_cast<int64_t>(lo) && r < static_cast<int64_t>(hi);
    }
};

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        bf16x2_to_f32(w[i], f[2 * i], f[2 * i + 1]);
    }
}

// Bytes of latent rows in the chunk starting at row r0.
__device__ __forceinline__ uint32_t rows_bytes_of(int64_t r0, int64_t total_rows, int C) {
    const int64_t rows = min(static_cast<int64_t>(kChunkRows), total_rows - r0);
    return static_cast<uint32_t>(rows * C * 2);
}

// NC = 16-byte chunks of the normalised part per lane (ceil(R / 256)).  QUANT: the
// destination is a quantised cache (codes, bf16 rope, fp32 block scales per slot).
template <int NC, bool QUANT>
__global__ void __launch_bounds__(kThreads, 1)
    cache_write_kernel(const CacheWriteArgs a, int32_t stages, StageLayout L) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Bars bars;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int R = a.kv_lora_rank, P = a.rope_dim, C = R + P;
    const int64_t n_chunks = (static_cast<int64_t>(a.total_rows) + kChunkRows - 1) / kChunkRows;
    const int64_t c_begin = n_chunks * blockIdx.x / gridDim.x;
    const int64_t c_end = n_chunks * (blockIdx.x + 1) / gridDim.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&bars.full[s], 1);  // producer lane 0, with the stage's byte count
            mbar_init(&bars.empty[s], kConsumerWarps);
        }
        bars.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl wc{&bars.abort_flag, a.status, a.timeout_ns};
    RingPos p;

    if (warp == 0) {
        const int64_t covered = min(static_cast<int64_t>(a.total_rows),
                                    static_cast<int64_t>(__ldg(a.row_offsets + a.batch)));
        RowCursor q;
        q.init(a, c_begin * kChunkRows + lane);
        for (int64_t k = c_begin; k < c_end; ++k) {
            // lane i < 30: row i of the chunk -> slot and page id (loaded before the stage is
            // free, so that the load overlaps the wait)
            const int64_t r0 = k * kChunkRows;
            const int64_t r = r0 + lane;
            int32_t slot = kSlotNone, req = -1;
            uint32_t page = 0;
            uint64_t pos = 0;
            if (lane < kChunkRows && r < covered && q.seek(a, r)) {
                pos = static_cast<uint64_t>(q.cl) + static_cast<uint64_t>(r - q.lo);
                const uint64_t lp = pos / static_cast<uint64_t>(a.page_size);
                if (pos >= static_cast<uint64_t>(a.max_seq_len) ||
                    lp >= static_cast<uint64_t>(a.max_pages)) {
                    slot = kSlotOutOfRange;
                } else {
                    slot = static_cast<int32_t>(pos % static_cast<uint64_t>(a.page_size));
                    page = __ldg(a.page_table + static_cast<int64_t>(q.b) * a.max_pages + lp);
                    req = q.b;
                }
            }
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&bars.empty[p.stage], p.phase ^ 1u, wc);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            __syncwarp();  // the consumers' reads of this stage precede every lane's writes
            uint8_t* stage = smem + p.stage * L.bytes;
            uint64_t* full = &bars.full[p.stage];
            if (lane < kChunkRows) {
                reinterpret_cast<int32_t*>(stage + L.slot)[lane] = slot;
                reinterpret_cast<uint32_t*>(stage + L.page)[lane] = page;
            }
            // freqs_cis rows: one bulk copy per run of rows of one request (consecutive
            // positions, so consecutive freqs_cis rows)
            const bool live = slot >= 0;
            const int prev_live = __shfl_up_sync(0xffffffffu, live ? 1 : 0, 1);
            const int prev_req = __shfl_up_sync(0xffffffffu, req, 1);
            const bool run_start = live && (lane == 0 || !prev_live || prev_req != req);
            const uint32_t live_mask = __ballot_sync(0xffffffffu, live);
            const uint32_t bound = __ballot_sync(0xffffffffu, !live || run_start);
            if (run_start && P > 0) {
                const uint32_t after = bound & ~((2u << lane) - 1u);  // lane < 30 here
                const int len = __ffs(after) - 1 - lane;
                bulk_load_1d(stage + L.freqs + lane * P * 4, a.freqs + pos * P,
                             static_cast<uint32_t>(len * P * 4), full);
            }
            if (lane == 0)
                bulk_load_1d(stage, a.latent + r0 * C, rows_bytes_of(r0, a.total_rows, C), full);
            __syncwarp();  // slots and page ids are written before lane 0 releases them
            if (lane == 0)
                mbar_arrive_expect_tx(full, rows_bytes_of(r0, a.total_rows, C) +
                                                static_cast<uint32_t>(__popc(live_mask) * P * 4));
            p.next(stages);
        }
    } else {
        constexpr int U = kRowsPerWarp;
        const int nope_chunks = R / 8;
        const bool has_rope = lane < P / 8;
        const int j0 = (warp - 1) * U;  // this warp's first row inside a chunk
        // this lane's gamma values (its normalised chunks never change) and 1 / R
        float gr[NC][8];
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const int c = lane + 32 * j;
            float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
            if (c < nope_chunks) {
                g0 = __ldg(reinterpret_cast<const float4*>(a.gamma + c * 8));
                g1 = __ldg(reinterpret_cast<const float4*>(a.gamma + c * 8 + 4));
            }
            gr[j][0] = g0.x; gr[j][1] = g0.y; gr[j][2] = g0.z; gr[j][3] = g0.w;
            gr[j][4] = g1.x; gr[j][5] = g1.y; gr[j][6] = g1.z; gr[j][7] = g1.w;
        }
        const float inv_r = 1.0f / static_cast<float>(R);
        for (int64_t k = c_begin; k < c_end; ++k) {
            if (!mbar_wait(&bars.full[p.stage], p.phase, wc)) break;
            const uint8_t* stage = smem + p.stage * L.bytes;
            const uint32_t base = smem_u32(stage);
            int32_t slot[U];
            uint32_t page[U];
            uint4 nv[U][NC], rv[U], fq[U][2];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                slot[u] = reinterpret_cast<const int32_t*>(stage + L.slot)[j0 + u];
                page[u] = slot[u] >= 0 ? reinterpret_cast<const uint32_t*>(stage + L.page)[j0 + u]
                                       : 0u;
                const bool live = slot[u] >= 0;
                const uint32_t row = base + static_cast<uint32_t>((j0 + u) * C * 2);
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    const int c = lane + 32 * j;
                    nv[u][j] = live && c < nope_chunks ? ld_shared_v4(row + c * 16)
                                                       : make_uint4(0u, 0u, 0u, 0u);
                }
                const bool rope = live && has_rope;
                const uint32_t fr = base + L.freqs + static_cast<uint32_t>((j0 + u) * P * 4 + lane * 32);
                rv[u] = rope ? ld_shared_v4(row + (R + lane * 8) * 2) : make_uint4(0u, 0u, 0u, 0u);
                fq[u][0] = rope ? ld_shared_v4(fr) : make_uint4(0u, 0u, 0u, 0u);
                fq[u][1] = rope ? ld_shared_v4(fr + 16) : make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.empty[p.stage]);
            p.next(stages);
            bool ok[U];
            int64_t doff[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                ok[u] = slot[u] >= 0 && page[u] < static_cast<uint32_t>(a.num_pages);
                if (!ok[u] && (slot[u] == kSlotOutOfRange || slot[u] >= 0) && lane == 0)
                    report(a.status, PKM_ERR_OUT_OF_RANGE);
                doff[u] = static_cast<int64_t>(page[u]) * a.page_stride +
                          static_cast<int64_t>(max(slot[u], 0)) * a.slot_stride;
            }
            // RMSNorm factor of each row (rows that are not stored compute on zeros); the
            // rows go through every step side by side, so that their latencies overlap.  The
            // nope values are unpacked to fp32 once and kept for the normalisation.
            float f[U][NC][8];
            float inv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    unpack8(nv[u][j], f[u][j]);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        fma2v(s0, s1, f[u][j][2 * i], f[u][j][2 * i + 1], f[u][j][2 * i],
                              f[u][j][2 * i + 1]);
                }
                inv[u] = s0 + s1;
            }
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1)
#pragma unroll
                for (int u = 0; u < U; ++u) inv[u] += __shfl_xor_sync(0xffffffffu, inv[u], sh);
#pragma unroll
            for (int u = 0; u < U; ++u) inv[u] = rsqrtf(fmaf(inv[u], inv_r, a.epsilon));
            if constexpr (QUANT) {
                // round to bf16 as the bf16 cache would, then quantise each 128-column block
                // (16 chunks = one half-warp): s = amax / 448, q = e4m3(y / s).  Each step is
                // taken for every block of both rows before the next, so that the latencies of
                // the reductions and reciprocals overlap.  The two half-warps' block maxima
                // come from two whole-warp reductions in which the other half contributes zero.
                float y[U][NC][8];
                uint32_t mlo[U][NC], mhi[U][NC];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int j = 0; j < NC; ++j) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float g0, g1, y0, y1;
                            mul2(g0, g1, gr[j][2 * i], gr[j][2 * i + 1], inv[u], inv[u]);
                            mul2(y0, y1, f[u][j][2 * i], f[u][j][2 * i + 1], g0, g1);
                            const uint32_t pk = pack_bf16x2(y0, y1);
                            bf16x2_to_f32(pk, y[u][j][2 * i], y[u][j][2 * i + 1]);
                        }
                        const float m = fmax3_abs(fmax3_abs(y[u][j][0], y[u][j][1], y[u][j][2]),
                                                  fmax3_abs(y[u][j][3], y[u][j][4], y[u][j][5]),
                                                  fmax3_abs(y[u][j][6], y[u][j][7], 0.0f));
                        const uint32_t mb = __float_as_uint(m);
                        mlo[u][j] = lane < 16 ? mb : 0u;
                        mhi[u][j] = lane < 16 ? 0u : mb;
                    }
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int j = 0; j < NC; ++j) {
                        mlo[u][j] = warp_max_u32(mlo[u][j]);
                        mhi[u][j] = warp_max_u32(mhi[u][j]);
                    }
                E4m3Block qb[U][NC];
                bool fast = true;
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int j = 0; j < NC; ++j) {
                        qb[u][j] = E4m3Block(__uint_as_float(lane < 16 ? mlo[u][j] : mhi[u][j]));
                        fast = fast && qb[u][j].fast;
                    }
                // one warp-uniform choice: every block in the fast range (the rule) or not
                uint32_t lo[U][NC], hi[U][NC];
                if (__all_sync(0xffffffffu, fast)) {
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int j = 0; j < NC; ++j) {
                            const float* v = y[u][j];
                            lo[u][j] = qb[u][j].codes4_fast(v[0], v[1], v[2], v[3]);
                            hi[u][j] = qb[u][j].codes4_fast(v[4], v[5], v[6], v[7]);
                        }
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int j = 0; j < NC; ++j) {
                            const float* v = y[u][j];
                            lo[u][j] = qb[u][j].codes4(v[0], v[1], v[2], v[3]);
                            hi[u][j] = qb[u][j].codes4(v[4], v[5], v[6], v[7]);
                        }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (!ok[u]) continue;
                    uint8_t* dstq = a.qcache_layer + doff[u];
#pragma unroll
                    for (int j = 0; j < NC; ++j) {
                        const int c = lane + 32 * j;
                        if (c >= nope_chunks) break;
                        *reinterpret_cast<uint2*>(dstq + c * 8) = make_uint2(lo[u][j], hi[u][j]);
                        if ((lane & 15) == 0)
                            *reinterpret_cast<float*>(dstq + R + 2 * P + 4 * (c / 16)) = qb[u][j].s;
                    }
                }
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (!ok[u]) continue;
                    uint16_t* dst = a.cache_layer + doff[u];
#pragma unroll
                    for (int j = 0; j < NC; ++j) {
                        const int c = lane + 32 * j;
                        if (c >= nope_chunks) break;
                        uint32_t o[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float g0, g1, y0, y1;
                            mul2(g0, g1, gr[j][2 * i], gr[j][2 * i + 1], inv[u], inv[u]);
                            mul2(y0, y1, f[u][j][2 * i], f[u][j][2 * i + 1], g0, g1);
                            o[i] = pack_bf16x2(y0, y1);
                        }
                        st_v4(dst + c * 8, make_uint4(o[0], o[1], o[2], o[3]));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!ok[u] || !has_rope) continue;
                float f[8];
                unpack8(rv[u], f);
                const float cs[8] = {__uint_as_float(fq[u][0].x), __uint_as_float(fq[u][0].y),
                                     __uint_as_float(fq[u][0].z), __uint_as_float(fq[u][0].w),
                                     __uint_as_float(fq[u][1].x), __uint_as_float(fq[u][1].y),
                                     __uint_as_float(fq[u][1].z), __uint_as_float(fq[u][1].w)};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {  // pair i: (x0, x1) by (cos, sin)
                    const float x0 = f[2 * i], x1 = f[2 * i + 1];
                    const float c = cs[2 * i], s = cs[2 * i + 1];
                    o[i] = pack_bf16x2(fmaf(x0, c, -x1 * s), fmaf(x0, s, x1 * c));
                }
                if constexpr (QUANT)
                    st_v4(a.qcache_layer + doff[u] + R + lane * 16, make_uint4(o[0], o[1], o[2], o[3]));
                else
                    st_v4(a.cache_layer + doff[u] + R + lane * 8, make_uint4(o[0], o[1], o[2], o[3]));
            }
        }
    }
    __syncthreads();
    // After an abort, copies may still be landing in the ring: wait (bounded) for the last
    // phase the producer started in every stage before the CTA exits.
    if (threadIdx.x == 0 && bars.abort_flag) {
        const int64_t issued = c_end - c_begin;
        for (int s = 0; s < stages && s < issued; ++s) {
            const int64_t last = s + ((issued - 1 - s) / stages) * stages;  // last chunk in s
            const uint32_t parity = static_cast<uint32_t>((last / stages) & 1);
            mbar_wait(&bars.full[s], parity, wc, false);
        }
    }
}

uint32_t round16(uint32_t v) { return (v + 15u) & ~15u; }

template <int NC, bool QUANT>
cudaError_t launch_nc(const CacheWriteArgs& args, int num_sms, cudaStream_t stream) {
    const uint32_t C = static_cast<uint32_t>(args.kv_lora_rank + args.rope_dim);
    StageLayout L;
    L.freqs = round16(kChunkRows * C * 2);
    L.page = L.freqs + round16(kChunkRows * static_cast<uint32_t>(args.rope_dim) * 4);
    L.slot = L.page + round16(kChunkRows * 4);
    L.bytes = (L.slot + round16(kChunkRows * 4) + 127u) & ~127u;
    int stages = static_cast<int>(kSmemBudget / L.bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) stages = 2;
    const size_t smem = static_cast<size_t>(stages) * L.bytes;
    cudaError_t e = cudaFuncSetAttribute(cache_write_kernel<NC, QUANT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t n_chunks = (static_cast<int64_t>(args.total_rows) + kChunkRows - 1) / kChunkRows;
    int64_t blocks = n_chunks < num_sms ? n_chunks : num_sms;
    if (blocks < 1) blocks = 1;
    cache_write_kernel<NC, QUANT><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(
        args, stages, L);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cache_write(CacheWriteArgs args, int num_sms, cudaStream_t stream) {
    const bool q = args.qcache_layer != nullptr;
    switch ((args.kv_lora_rank / 8 + 31) / 32) {
        case 1: return q ? launch_nc<1, true>(args, num_sms, stream)
                         : launch_nc<1, false>(args, num_sms, stream);
        case 2: return q ? launch_nc<2, true>(args, num_sms, stream)
                         : launch_nc<2, false>(args, num_sms, stream);
        case 3: return q ? launch_nc<3, true>(args, num_sms, stream)
                         : launch_nc<3, false>(args, num_sms, stream);
        default: return q ? launch_nc<4, true>(args, num_sms, stream)
                          : launch_nc<4, false>(args, num_sms, stream);
    }
}

}  // namespace pkm
