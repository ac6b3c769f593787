// pkm_internal.h -- argument blocks passed from the C entry points (api.cu) to the kernel
// launchers (decompress_bf16.cu, decompress_fp8.cu, kv_matmul.cu).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <utility>

namespace pkm {

// One decompress problem, already validated on the host.  Pointers are device memory.
struct DecompressArgs {
    const uint16_t* cache_layer;   // cache data + layer_idx * layer_stride (bf16)
    const uint8_t* qcache_layer;   // or: a quantised cache's layer (strides then in bytes)
    int64_t page_stride;           // elements (bytes for a quantised cache)
    int64_t slot_stride;           // elements (bytes for a quantised cache)
    int32_t num_pages;
    int32_t page_size;
    int32_t max_pages;             // page-table row length
    const uint32_t* page_table;    // [batch, max_pages]
    const uint32_t* row_offsets;   // buffer_row_offsets [batch + 1]
    const uint32_t* cache_offsets; // [>= batch]
    int32_t batch;
    int32_t buffer_length;         // rows of the outputs
    int32_t kv_lora_rank;          // R
    int32_t latent_cols;           // C = R + rope
    int32_t n_out;                 // N
    uint16_t* k_latent;            // [L, C] bf16
    uint16_t* k_buffer;            // [L, N] bf16
    uint16_t* v_buffer;            // [L, N_v] bf16, or null (no V up-projection)
    int32_t n_out_v;               // N_v = num_heads * v_head_dim (0 without V)
    int32_t* status;               // nullable
    uint64_t timeout_ns;
    // tiling, filled by the launcher
    int32_t bn;                    // N tile
    int32_t n_tiles;               // (N + N_v) / bn: K tiles first, then V tiles
    int32_t n_tiles_k;             // N / bn
    int32_t m_tiles;               // ceil(L / rows per tile)
    int64_t total_tiles;           // m_tiles * n_tiles
    int32_t gather_tma;            // bf16 kernel: the cache gather map is valid (page_size >= 8)
};

struct Fp8Extra {
    uint8_t* q_latent;             // [L, R] e4m3 (workspace)
    float* q_scale;                // [L, R/128] (workspace)
    const float* w_scale;          // [N/128, R/128]
    const float* w_scale_v;        // [N_v/128, R/128], or null
};

// One cache write (new latent rows -> RMSNorm / RoPE -> paged latent cache), validated.
struct CacheWriteArgs {
    const uint16_t* latent;        // [total_rows, R + P] bf16
    const uint32_t* row_offsets;   // input_row_offsets [batch + 1]
    int32_t batch;
    int32_t total_rows;
    int32_t kv_lora_rank;          // R, multiple of 8, <= 1024
    int32_t rope_dim;              // P, multiple of 8, <= 256
    const float* gamma;            // [R]
    float epsilon;
    const float* freqs;            // [max_seq_len, P]
    int32_t max_seq_len;
    uint16_t* cache_layer;         // cache data + layer_idx * layer_stride
    int64_t page_stride, slot_stride;
    int32_t num_pages, page_size, max_pages;
    const uint32_t* page_table;
    const uint32_t* cache_lengths;
    int32_t* status;
    uint64_t timeout_ns;
    uint8_t* qcache_layer;         // quantised destination (byte strides), or null
};

// One kv_matmul problem, already validated.
struct KvMatmulArgs {
    const uint16_t* hidden;        // [M, K] bf16
    const uint32_t* row_offsets;   // input_row_offsets [batch + 1]
    int32_t batch;
    int32_t total_rows;            // M
    int32_t k_in;                  // K
    int32_t n_out;                 // N = HD or 2 HD
    int32_t head_elems;            // HD
    uint16_t* cache_layer;         // cache data + layer_idx * layer_stride
    int64_t page_stride, slot_stride, kv_stride;
    int32_t num_pages, page_size, max_pages;
    const uint32_t* page_table;
    const uint32_t* cache_lengths;
    int32_t* status;
    uint64_t timeout_ns;
    int32_t bn, n_tiles, m_tiles;
    int64_t total_tiles;
};

// FP8 kv_matmul operands: the quantised hidden rows (workspace) and the weight scales.
struct KvFp8Extra {
    uint8_t* q;                    // [M, k_in] e4m3 (workspace)
    float* q_scale;                // [M, k_in/128] (workspace)
    const float* w_scale;          // [n_out/128, k_in/128]
};

// Launches `kernel` as a programmatic dependent of the work before it on `stream`: it may
// start while the previous kernel (a prepass that triggers its dependents) still runs, and
// waits for that kernel's writes with griddepcontrol.wait before reading them.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                             size_t smem, cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers (return a CUDA error code; 0 = success).  Tensor maps are encoded by the
// caller.
cudaError_t launch_decompress_bf16(const CUtensorMap& tm_w, const CUtensorMap& tm_wv,
                                   const CUtensorMap& tm_cache, DecompressArgs args, int num_sms,
                                   cudaStream_t stream);
cudaError_t launch_fp8_gather_quantize(DecompressArgs args, Fp8Extra extra, int num_sms,
                                       cudaStream_t stream);
cudaError_t launch_fp8_gather_qcache(DecompressArgs args, Fp8Extra extra, int num_sms,
                                     cudaStream_t stream);
cudaError_t launch_decompress_fp8_gemm(const CUtensorMap& tm_q, const CUtensorMap& tm_w,
                                       const CUtensorMap& tm_wv, DecompressArgs args,
                                       Fp8Extra extra, int num_sms, cudaStream_t stream);
cudaError_t launch_decompress_fp8_wide(const CUtensorMap& tm_q, const CUtensorMap& tm_w,
                                       const CUtensorMap& tm_wv, const CUtensorMap& tm_ok,
                                       const CUtensorMap& tm_ov, DecompressArgs args,
                                       Fp8Extra extra, int num_sms, cudaStream_t stream);
cudaError_t launch_kv_matmul(const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                             KvMatmulArgs args, int num_sms, cudaStream_t stream);
cudaError_t launch_kv_matmul_fp8(const CUtensorMap& tm_q, const CUtensorMap& tm_w,
                                 KvMatmulArgs args, KvFp8Extra extra, int num_sms,
                                 cudaStream_t stream);
cudaError_t launch_cache_write(CacheWriteArgs args, int num_sms, cudaStream_t stream);
cudaError_t launch_wait_timeout_check(int32_t* status, uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_validate_offsets(const uint32_t* offsets, int32_t batch, int32_t* status,
                                    cudaStream_t stream);

// Row bookkeeping shared by the decompress kernels: element offset (inside the layer) of
// the cache slot that feeds output row r, -1 when no request covers r (or r >= row_end),
// -2 when the token resolves past the page-table row or to a page id >= num_pages.
// The request of r is the largest b with row_offsets[b] <= r (row_offsets non-decreasing,
// so empty requests are skipped); its token is cache_offsets[b] + r - row_offsets[b].
__device__ __forceinline__ int64_t decompress_row_locate(const DecompressArgs& a, int64_t r,
                                                         int64_t row_end, uint32_t* page_out,
                                                         uint32_t* slot_out) {
    if (r >= row_end) return -1;
    const uint32_t* bro = a.row_offsets;
    if (static_cast<uint64_t>(r) < static_cast<uint64_t>(__ldg(bro))) return -1;
    int lo = 0, hi = a.batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<uint64_t>(__ldg(bro + mid)) <= static_cast<uint64_t>(r)) lo = mid;
        else hi = mid;
    }
    const uint64_t i = static_cast<uint64_t>(r) - __ldg(bro + lo);
    const uint64_t t = static_cast<uint64_t>(__ldg(a.cache_offsets + lo)) + i;
    const uint64_t lp = t / static_cast<uint64_t>(a.page_size);
    if (lp >= static_cast<uint64_t>(a.max_pages)) return -2;
    const uint32_t page = __ldg(a.page_table + static_cast<int64_t>(lo) * a.max_pages + lp);
    if (page >= static_cast<uint32_t>(a.num_pages)) return -2;
    const uint32_t slot = static_cast<uint32_t>(t % static_cast<uint64_t>(a.page_size));
    *page_out = page;
    *slot_out = slot;
    return static_cast<int64_t>(page) * a.page_stride + static_cast<int64_t>(slot) * a.slot_stride;
}

__device__ __forceinline__ int64_t decompress_row_source(const DecompressArgs& a, int64_t r,
                                                         int64_t row_end) {
    uint32_t page, slot;
    return decompress_row_locate(a, r, row_end, &page, &slot);
}

// decompress_row_source for a run of increasing rows: one binary search for the first row,
// then the request only moves forward and the page id of the last logical page is reused,
// so a row costs no chain of dependent loads.  Same results as decompress_row_source.
struct RowSourceWalk {
    int b;
    int64_t lo, hi;        // request b covers rows [lo, hi)
    uint64_t co;           // cache_offsets[b]
    uint64_t page_key;     // (b, logical page) whose id is in page
    uint32_t page;

    __device__ __forceinline__ RowSourceWalk(const DecompressArgs& a, int64_t r) {
        const uint32_t* bro = a.row_offsets;
        int l = 0, h = a.batch;  // largest b with bro[b] <= r (0 when r < bro[0])
        while (h - l > 1) {
            const int mid = (l + h) >> 1;
            if (static_cast<int64_t>(__ldg(bro + mid)) <= r) l = mid;
            else h = mid;
        }
        b = l;
        lo = __ldg(bro + l);
        hi = __ldg(bro + l + 1);
        co = __ldg(a.cache_offsets + l);
        page_key = ~0ull;
        page = 0;
    }

    // Rows must come in non-decreasing order.
    __device__ __forceinline__ int64_t source(const DecompressArgs& a, int64_t r) {
        while (r >= hi && b + 1 < a.batch) {
            ++b;
            lo = hi;
            hi = __ldg(a.row_offsets + b + 1);
            co = __ldg(a.cache_offsets + b);
        }
        if (r < lo || r >= hi) return -1;
        const uint64_t t = co + static_cast<uint64_t>(r - lo);
        const uint64_t lp = t / static_cast<uint64_t>(a.page_size);
        if (lp >= static_cast<uint64_t>(a.max_pages)) return -2;
        const uint64_t key = (static_cast<uint64_t>(b) << 32) | lp;
        if (key != page_key) {
            page = __ldg(a.page_table + static_cast<int64_t>(b) * a.max_pages + lp);
            page_key = key;
        }
        if (page >= static_cast<uint32_t>(a.num_pages)) return -2;
        const uint64_t slot = t - lp * static_cast<uint64_t>(a.page_size);
        return static_cast<int64_t>(page) * a.page_stride +
               static_cast<int64_t>(slot) * a.slot_stride;
    }
};

// min(buffer_length, row_offsets[batch]): rows at or past it are not written.
__device__ __forceinline__ int64_t decompress_row_end(const DecompressArgs& a) {
    const int64_t covered = static_cast<int64_t>(__ldg(a.row_offsets + a.batch));
    return covered < a.buffer_length ? covered : a.buffer_length;
}

// kv_matmul rows: element offset (inside the layer's K plane) of the slot that receives
// row r, -1 when no request covers r, -2 when the position resolves past the page table or
// the cache.  Row i of request b (the largest b with row_offsets[b] <= r) is position
// cache_lengths[b] + i.
__device__ __forceinline__ int64_t kv_row_dest(const KvMatmulArgs& a, int64_t r) {
    const uint32_t* iro = a.row_offsets;
    const int64_t covered = static_cast<int64_t>(__ldg(iro + a.batch));
    if (r >= a.total_rows || r >= covered) return -1;
    if (static_cast<uint64_t>(r) < static_cast<uint64_t>(__ldg(iro))) return -1;
    int lo = 0, hi = a.batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<uint64_t>(__ldg(iro + mid)) <= static_cast<uint64_t>(r)) lo = mid;
        else hi = mid;
    }
    const uint64_t pos = static_cast<uint64_t>(__ldg(a.cache_lengths + lo)) +
                         (static_cast<uint64_t>(r) - __ldg(iro + lo));
    const uint64_t lp = pos / static_cast<uint64_t>(a.page_size);
    if (lp >= static_cast<uint64_t>(a.max_pages)) return -2;
    const uint32_t page = __ldg(a.page_table + static_cast<int64_t>(lo) * a.max_pages + lp);
    if (page >= static_cast<uint32_t>(a.num_pages)) return -2;
    return static_cast<int64_t>(page) * a.page_stride +
           static_cast<int64_t>(pos % static_cast<uint64_t>(a.page_size)) * a.slot_stride;
}

}  // namespace pkm
