// api.cu -- the C entry points declared in include/paged_kv_mla.h: host-side argument
// checks, tensor-map encoding, tile selection and kernel launches.  Every check that can
// be made without touching the GPU is made before the first CUDA call, so invalid calls
// return a status and launch nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "paged_kv_mla.h"
#include "pkm_internal.h"

namespace {

using pkm::DecompressArgs;
using pkm::Fp8Extra;
using pkm::CacheWriteArgs;
using pkm::KvMatmulArgs;
using pkm::KvFp8Extra;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool mult8(int64_t v) { return v >= 0 && (v % 8) == 0; }

uint64_t wait_timeout_ns() {
    static uint64_t ns = [] {
        const char* s = std::getenv("PKM_WAIT_TIMEOUT_MS");
        long ms = s ? std::strtol(s, nullptr, 10) : 1000;
        if (ms <= 0) ms = 1000;
        return static_cast<uint64_t>(ms) * 1000000ull;
    }();
    return ns;
}

// Streaming multiprocessors of the current device, cached per device id.  Threads may race
// to fill an entry; they all store the same value, and the atomics make that well defined.
cudaError_t current_sm_count(int* out) {
    static std::atomic<int> counts[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        counts[dev].store(n, std::memory_order_relaxed);
    }
    *out = n;
    return cudaSuccess;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D row-major tensor [outer, inner] with a row pitch in bytes, boxes of
// [box_outer, box_inner] elements, 128-byte swizzle, zero fill out of bounds.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// A row-major matrix [rows, K] viewed as k-blocks: 3-D tensor {inner = K elements of one
// k-block, rows, k-blocks} with strides {row pitch, k-block pitch} (the k-block dimension
// steps inside a row), boxes of {inner, box_rows, box_kblocks}.  One box lands in shared
// memory as box_kblocks consecutive [box_rows x inner] tiles, each 128-byte swizzled.
bool encode_kblocks_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                       uint64_t inner, uint64_t rows, uint64_t kblocks, uint64_t row_pitch_bytes,
                       uint64_t kblock_pitch_bytes, uint32_t box_rows, uint32_t box_kblocks) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {inner, rows, kblocks};
    const cuuint64_t strides[2] = {row_pitch_bytes, kblock_pitch_bytes};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(inner), box_rows, box_kblocks};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// One layer of the paged latent cache as a 4-D tensor {64 columns of a k-block, slot, page,
// k-block} (strides slot_stride, page_stride and 128 bytes), boxes of {64, 8 slots, 1 page,
// kblocks}: one box is eight consecutive slots of one page with all their k-blocks, landing
// as kblocks 1 KB tiles of [8 rows x 128 bytes], 128-byte swizzled.
bool encode_cache_gather(CUtensorMap* map, const void* layer, int32_t page_size,
                         int32_t num_pages, int32_t kblocks, int64_t slot_stride,
                         int64_t page_stride) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(page_size),
                                static_cast<cuuint64_t>(num_pages),
                                static_cast<cuuint64_t>(kblocks)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(slot_stride) * 2,
                                   static_cast<cuuint64_t>(page_stride) * 2, 128};
    const cuuint32_t box[4] = {64, 8, 1, static_cast<cuuint32_t>(kblocks)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(layer), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Checks shared by both decompress entry points.  Returns PKM_OK or the error.
pkm_status check_decompress(const pkm_paged_cache* cache, uint32_t layer_idx, const uint32_t* bro,
                            const uint32_t* co, int32_t batch, int32_t buffer_length,
                            int32_t kv_lora_rank, int32_t rope_dim, const void* w, int32_t n_out,
                            void* k_latent, void* k_buffer) {
    if (cache == nullptr || bro == nullptr || co == nullptr || w == nullptr ||
        k_latent == nullptr || k_buffer == nullptr || cache->data == nullptr ||
        cache->page_table == nullptr)
        return PKM_ERR_INVALID_ARG;
    if (cache->num_layers <= 0 || layer_idx >= static_cast<uint32_t>(cache->num_layers) ||
        cache->num_pages <= 0 || cache->page_size <= 0 || cache->max_pages_per_seq <= 0)
        return PKM_ERR_INVALID_ARG;
    if (cache->row_elems != kv_lora_rank + rope_dim) return PKM_ERR_INVALID_ARG;
    if (!mult8(cache->layer_stride) || !mult8(cache->page_stride) || !mult8(cache->slot_stride))
        return PKM_ERR_INVALID_ARG;
    if (!aligned16(cache->data) || !aligned16(w) || !aligned16(k_latent) || !aligned16(k_buffer))
        return PKM_ERR_INVALID_ARG;
    if ((kv_lora_rank + rope_dim) % 8 != 0) return PKM_ERR_UNSUPPORTED;
    return PKM_OK;
}

// Size checks that come before any pointer check: a call with nothing to do (no rows or no
// requests) succeeds whatever its pointers are.
pkm_status check_decompress_sizes(int32_t batch, int32_t buffer_length, int32_t kv_lora_rank,
                                  int32_t rope_dim, int32_t n_out, bool* empty) {
    if (batch < 0 || buffer_length < 0 || rope_dim < 0 || n_out <= 0 || kv_lora_rank <= 0)
        return PKM_ERR_INVALID_ARG;
    *empty = (buffer_length == 0 || batch == 0);
    return PKM_OK;
}

DecompressArgs make_decompress_args(const pkm_paged_cache* cache, uint32_t layer_idx,
                                    const uint32_t* bro, const uint32_t* co, int32_t batch,
                                    int32_t buffer_length, int32_t kv_lora_rank, int32_t rope_dim,
                                    int32_t n_out, void* k_latent, void* k_buffer,
                                    int32_t* dev_status, int bn) {
    DecompressArgs a{};
    a.cache_layer = static_cast<const uint16_t*>(cache->data) +
                    static_cast<int64_t>(layer_idx) * cache->layer_stride;
    a.page_stride = cache->page_stride;
    a.slot_stride = cache->slot_stride;
    a.num_pages = cache->num_pages;
    a.page_size = cache->page_size;
    a.max_pages = cache->max_pages_per_seq;
    a.page_table = cache->page_table;
    a.row_offsets = bro;
    a.cache_offsets = co;
    a.batch = batch;
    a.buffer_length = buffer_length;
    a.kv_lora_rank = kv_lora_rank;
    a.latent_cols = kv_lora_rank + rope_dim;
    a.n_out = n_out;
    a.k_latent = static_cast<uint16_t*>(k_latent);
    a.k_buffer = static_cast<uint16_t*>(k_buffer);
    a.status = dev_status;
    a.timeout_ns = wait_timeout_ns();
    a.bn = bn;
    a.n_tiles = n_out / bn;
    a.m_tiles = (buffer_length + 127) / 128;
    a.total_tiles = static_cast<int64_t>(a.m_tiles) * a.n_tiles;
    return a;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// What lies behind the last PKM_ERR_CUDA this thread returned (pkm_last_cuda_error).
thread_local const char* g_last_cuda_error = "no CUDA failure recorded";

pkm_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return PKM_OK;
    g_last_cuda_error = cudaGetErrorString(e);
    return PKM_ERR_CUDA;
}

pkm_status encode_failed() {
    g_last_cuda_error = "cuTensorMapEncodeTiled rejected a tensor map";
    return PKM_ERR_CUDA;
}

// PKM_DEBUG_VALIDATE=1: every entry point checks its offset array on the device first
// (pkm_validate_row_offsets into its status word, when it has one).
bool debug_validate_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("PKM_DEBUG_VALIDATE");
        return v != nullptr && v[0] == '1';
    }();
    return on;
}

cudaError_t debug_validate(const uint32_t* offsets, int32_t batch, int32_t* dev_status,
                           void* stream) {
    if (!debug_validate_enabled() || dev_status == nullptr || batch <= 0) return cudaSuccess;
    return pkm::launch_validate_offsets(offsets, batch, dev_status,
                                        static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

const char* pkm_last_cuda_error(void) { return g_last_cuda_error; }

const char* pkm_status_string(pkm_status status) {
    switch (status) {
        case PKM_OK: return "PKM_OK";
        case PKM_ERR_INVALID_ARG: return "PKM_ERR_INVALID_ARG";
        case PKM_ERR_UNSUPPORTED: return "PKM_ERR_UNSUPPORTED";
        case PKM_ERR_CUDA: return "PKM_ERR_CUDA";
        case PKM_ERR_OUT_OF_RANGE: return "PKM_ERR_OUT_OF_RANGE";
        case PKM_ERR_TIMEOUT: return "PKM_ERR_TIMEOUT";
    }
    return "PKM_ERR_UNKNOWN";
}

}  // extern "C"

namespace {

// V operands of the K-and-V entry points (all null / zero for the K-only ones).
struct VOperands {
    const void* w_uv = nullptr;   // [num_heads, v_head_dim, R], bf16 or e4m3
    const float* w_uv_scale = nullptr;
    int32_t n_v = 0;              // num_heads * v_head_dim
    void* v_buffer = nullptr;     // [buffer_length, n_v] bf16
};

pkm_status check_v(const VOperands& v, int32_t num_heads, int32_t v_head_dim, int multiple) {
    if (v.w_uv == nullptr || v.v_buffer == nullptr) return PKM_ERR_INVALID_ARG;
    if (num_heads <= 0 || v_head_dim <= 0) return PKM_ERR_INVALID_ARG;
    if (!aligned16(v.w_uv) || !aligned16(v.v_buffer)) return PKM_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_heads) * v_head_dim > (static_cast<int64_t>(1) << 30))
        return PKM_ERR_UNSUPPORTED;
    if ((static_cast<int64_t>(num_heads) * v_head_dim) % multiple != 0) return PKM_ERR_UNSUPPORTED;
    return PKM_OK;
}

// Body of the bf16 entry points: K alone (v.w_uv == nullptr) or K and V from one gather.
pkm_status decompress_bf16(const pkm_paged_cache* cache, uint32_t layer_idx,
                           const uint32_t* buffer_row_offsets, const uint32_t* cache_offsets,
                           int32_t batch, int32_t buffer_length, int32_t kv_lora_rank,
                           int32_t rope_dim, const void* w_k, int32_t n_out,
                           const VOperands& v, void* k_latent_buffer, void* k_buffer,
                           int32_t* dev_status, void* stream) {
    bool empty = false;
    pkm_status st = check_decompress_sizes(batch, buffer_length, kv_lora_rank, rope_dim, n_out,
                                           &empty);
    if (st != PKM_OK || empty) return st;
    st = check_decompress(cache, layer_idx, buffer_row_offsets, cache_offsets, batch,
                                     buffer_length, kv_lora_rank, rope_dim, w_k, n_out,
                                     k_latent_buffer, k_buffer);
    if (st != PKM_OK) return st;
    if (kv_lora_rank % 64 != 0 || kv_lora_rank > 512 || n_out % 64 != 0) return PKM_ERR_UNSUPPORTED;
    // the kernel keeps each row's offset in the layer as a 32-bit count of 16-byte units
    const int64_t layer_span = static_cast<int64_t>(cache->num_pages) * cache->page_stride +
                               static_cast<int64_t>(cache->page_size) * cache->slot_stride;
    if (layer_span >= (static_cast<int64_t>(1) << 35) - 64) return PKM_ERR_UNSUPPORTED;
    // CTA-pair tiles of 256 rows x bn columns (the widest of 256 / 128 / 64 dividing
    // n_out, and n_v with V); each CTA loads bn/2 weight rows per k-block
    const int32_t nv = v.w_uv != nullptr ? v.n_v : 0;
    const int32_t both = nv > 0 ? (n_out | nv) : n_out;
    const int bn = (both % 256 == 0) ? 256 : (both % 128 == 0) ? 128 : 64;
    DecompressArgs a = make_decompress_args(cache, layer_idx, buffer_row_offsets, cache_offsets,
                                            batch, buffer_length, kv_lora_rank, rope_dim, n_out,
                                            k_latent_buffer, k_buffer, dev_status, bn);
    a.n_tiles_k = a.n_tiles;
    if (nv > 0) {
        a.v_buffer = static_cast<uint16_t*>(v.v_buffer);
        a.n_out_v = nv;
        a.n_tiles += nv / bn;
    }
    int sms = 0;
    if (const cudaError_t e = current_sm_count(&sms)) return cuda_status(e);
    a.m_tiles = (buffer_length + 255) / 256;
    a.total_tiles = static_cast<int64_t>(a.m_tiles) * a.n_tiles;
    alignas(64) CUtensorMap tm_w;
    alignas(64) CUtensorMap tm_wv;
    alignas(64) CUtensorMap tm_c = {};
    if (!encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_k, kv_lora_rank, n_out,
                   static_cast<uint64_t>(kv_lora_rank) * 2, 64, bn / 2))
        return encode_failed();
    if (nv > 0) {
        if (!encode_2d(&tm_wv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v.w_uv, kv_lora_rank, nv,
                       static_cast<uint64_t>(kv_lora_rank) * 2, 64, bn / 2))
            return encode_failed();
    } else {
        tm_wv = tm_w;
    }
    // Rows arriving as runs of eight slots of one page come by TMA; that needs pages of at
    // least eight slots.  Otherwise every row takes the per-row path.
    a.gather_tma = cache->page_size >= 8 ? 1 : 0;
    if (a.gather_tma &&
        !encode_cache_gather(&tm_c, a.cache_layer, cache->page_size, cache->num_pages,
                             kv_lora_rank / 64, cache->slot_stride, cache->page_stride))
        return encode_failed();
    if (const cudaError_t e = debug_validate(buffer_row_offsets, batch, dev_status, stream))
        return cuda_status(e);
    return cuda_status(pkm::launch_decompress_bf16(tm_w, tm_wv, tm_c, a, sms,
                                       static_cast<cudaStream_t>(stream)));
}

// Body of the FP8 entry points: K alone (v.w_uv == nullptr) or K and V, the activations
// quantised once for both.
// Checks of a quantised cache for the decompress (the bf16 cache's check_decompress).
pkm_status check_qdecompress(const pkm_quant_cache* cache, uint32_t layer_idx, const uint32_t* bro,
                             const uint32_t* co, const void* w, void* k_latent, void* k_buffer) {
    if (cache == nullptr || bro == nullptr || co == nullptr || w == nullptr ||
        k_buffer == nullptr || cache->data == nullptr || cache->page_table == nullptr)
        return PKM_ERR_INVALID_ARG;
    if (cache->num_layers <= 0 || layer_idx >= static_cast<uint32_t>(cache->num_layers) ||
        cache->num_pages <= 0 || cache->page_size <= 0 || cache->max_pages_per_seq <= 0)
        return PKM_ERR_INVALID_ARG;
    const int64_t payload = static_cast<int64_t>(cache->kv_lora_rank) + 2 * cache->rope_dim +
                            4 * (cache->kv_lora_rank / 128);
    if (cache->layer_stride < 0 || cache->layer_stride % 16 != 0 || cache->page_stride < 0 ||
        cache->page_stride % 16 != 0 || cache->slot_stride % 16 != 0 ||
        cache->slot_stride < payload)
        return PKM_ERR_INVALID_ARG;
    if (!aligned16(cache->data) || !aligned16(w) || !aligned16(k_buffer) ||
        (k_latent != nullptr && !aligned16(k_latent)))
        return PKM_ERR_INVALID_ARG;
    return PKM_OK;
}

pkm_status decompress_fp8(const pkm_paged_cache* cache, uint32_t layer_idx,
                          const uint32_t* buffer_row_offsets, const uint32_t* cache_offsets,
                          int32_t batch, int32_t buffer_length, int32_t kv_lora_rank,
                          int32_t rope_dim, const void* w_k_e4m3, const float* w_k_scale,
                          int32_t n_out, const VOperands& v, void* k_latent_buffer,
                          void* k_buffer, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream,
                          const pkm_quant_cache* qcache = nullptr) {
    bool empty = false;
    pkm_status st = check_decompress_sizes(batch, buffer_length, kv_lora_rank, rope_dim, n_out,
                                           &empty);
    if (st != PKM_OK || empty) return st;
    if (qcache != nullptr) {
        if (rope_dim % 8 != 0 || rope_dim > 256) return PKM_ERR_UNSUPPORTED;
        st = check_qdecompress(qcache, layer_idx, buffer_row_offsets, cache_offsets, w_k_e4m3,
                               k_latent_buffer, k_buffer);
    } else {
        st = check_decompress(cache, layer_idx, buffer_row_offsets, cache_offsets, batch,
                              buffer_length, kv_lora_rank, rope_dim, w_k_e4m3, n_out,
                              k_latent_buffer, k_buffer);
    }
    if (st != PKM_OK) return st;
    if (w_k_scale == nullptr || workspace == nullptr) return PKM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKM_ERR_INVALID_ARG;
    if (kv_lora_rank % 128 != 0 || kv_lora_rank > 512 || n_out % 128 != 0)
        return PKM_ERR_UNSUPPORTED;
    if (workspace_bytes < mla_decompress_k_paged_fp8_workspace_size(buffer_length, kv_lora_rank))
        return PKM_ERR_INVALID_ARG;
    const int32_t nv = v.w_uv != nullptr ? v.n_v : 0;
    // 256-wide pair tiles (full-rate e4m3 MMAs) when every projection splits into them,
    // else 128-wide ones
    const bool wide = n_out % 256 == 0 && nv % 256 == 0;
    const int bn = wide ? 256 : 128;
    DecompressArgs a{};
    if (qcache != nullptr) {
        // the same problem over byte strides: the page walk is unit-agnostic
        pkm_paged_cache view{};
        view.data = qcache->data;
        view.page_stride = qcache->page_stride;
        view.slot_stride = qcache->slot_stride;
        view.num_pages = qcache->num_pages;
        view.page_size = qcache->page_size;
        view.page_table = qcache->page_table;
        view.max_pages_per_seq = qcache->max_pages_per_seq;
        a = make_decompress_args(&view, 0, buffer_row_offsets, cache_offsets, batch,
                                 buffer_length, kv_lora_rank, rope_dim, n_out, k_latent_buffer,
                                 k_buffer, dev_status, bn);
        a.cache_layer = nullptr;
        a.qcache_layer = static_cast<const uint8_t*>(qcache->data) +
                         static_cast<int64_t>(layer_idx) * qcache->layer_stride;
    } else {
        a = make_decompress_args(cache, layer_idx, buffer_row_offsets, cache_offsets, batch,
                                 buffer_length, kv_lora_rank, rope_dim, n_out, k_latent_buffer,
                                 k_buffer, dev_status, bn);
    }
    a.n_tiles_k = a.n_tiles;
    if (nv > 0) {
        a.v_buffer = static_cast<uint16_t*>(v.v_buffer);
        a.n_out_v = nv;
        a.n_tiles += nv / bn;
    }
    a.m_tiles = (buffer_length + 255) / 256;  // CTA-pair tiles of 256 rows
    a.total_tiles = static_cast<int64_t>(a.m_tiles) * a.n_tiles;
    if (a.total_tiles > INT32_MAX) return PKM_ERR_UNSUPPORTED;  // 32-bit tile walk
    Fp8Extra x{};
    x.q_latent = static_cast<uint8_t*>(workspace);
    x.q_scale = reinterpret_cast<float*>(
        static_cast<uint8_t*>(workspace) +
        align256(static_cast<size_t>(buffer_length) * static_cast<size_t>(kv_lora_rank)));
    x.w_scale = w_k_scale;
    x.w_scale_v = nv > 0 ? v.w_uv_scale : nullptr;
    int sms = 0;
    if (const cudaError_t e = current_sm_count(&sms)) return cuda_status(e);
    alignas(64) CUtensorMap tm_q, tm_w, tm_wv;
    if (!encode_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, x.q_latent, kv_lora_rank, buffer_length,
                   static_cast<uint64_t>(kv_lora_rank), 128, 128))
        return encode_failed();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (wide) {
        // weights by 128 x 128 boxes (one k-block of a CTA's half tile); outputs viewed as
        // {64 columns, rows, column blocks of 64} and stored by {64, 128, 4} boxes (a CTA's
        // 128 rows x 256 columns of one tile)
        alignas(64) CUtensorMap tm_ok, tm_ov;
        if (!encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_k_e4m3, kv_lora_rank, n_out,
                       static_cast<uint64_t>(kv_lora_rank), 128, 128) ||
            !encode_kblocks_3d(&tm_ok, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_buffer, 64,
                               buffer_length, n_out / 64, static_cast<uint64_t>(n_out) * 2, 128,
                               128, 4))
            return encode_failed();
        if (nv > 0) {
            if (!encode_2d(&tm_wv, CU_TENSOR_MAP_DATA_TYPE_UINT8, v.w_uv, kv_lora_rank, nv,
                           static_cast<uint64_t>(kv_lora_rank), 128, 128) ||
                !encode_kblocks_3d(&tm_ov, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v.v_buffer, 64,
                                   buffer_length, nv / 64, static_cast<uint64_t>(nv) * 2, 128,
                                   128, 4))
                return encode_failed();
        } else {
            tm_wv = tm_w;
            tm_ov = tm_ok;
        }
        if (const cudaError_t e = debug_validate(buffer_row_offsets, batch, dev_status, stream))
            return cuda_status(e);
        const cudaError_t ge = qcache != nullptr ? pkm::launch_fp8_gather_qcache(a, x, sms, s)
                                                 : pkm::launch_fp8_gather_quantize(a, x, sms, s);
        if (ge != cudaSuccess) return cuda_status(ge);
        return cuda_status(pkm::launch_decompress_fp8_wide(tm_q, tm_w, tm_wv, tm_ok, tm_ov, a, x, sms, s));
    }
    if (!encode_kblocks_3d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_k_e4m3, 128, n_out,
                           kv_lora_rank / 128, static_cast<uint64_t>(kv_lora_rank), 128, 64,
                           kv_lora_rank / 128))
        return encode_failed();
    if (nv > 0) {
        if (!encode_kblocks_3d(&tm_wv, CU_TENSOR_MAP_DATA_TYPE_UINT8, v.w_uv, 128, nv,
                               kv_lora_rank / 128, static_cast<uint64_t>(kv_lora_rank), 128, 64,
                               kv_lora_rank / 128))
            return encode_failed();
    } else {
        tm_wv = tm_w;
    }
    if (const cudaError_t e = debug_validate(buffer_row_offsets, batch, dev_status, stream))
        return cuda_status(e);
    const cudaError_t ge = qcache != nullptr ? pkm::launch_fp8_gather_qcache(a, x, sms, s)
                                             : pkm::launch_fp8_gather_quantize(a, x, sms, s);
    if (ge != cudaSuccess) return cuda_status(ge);
    return cuda_status(pkm::launch_decompress_fp8_gemm(tm_q, tm_w, tm_wv, a, x, sms, s));
}

}  // namespace

extern "C" {

pkm_status mla_decompress_k_paged(const pkm_paged_cache* cache, uint32_t layer_idx,
                                  const uint32_t* buffer_row_offsets,
                                  const uint32_t* cache_offsets, int32_t batch,
                                  int32_t buffer_length, int32_t kv_lora_rank, int32_t rope_dim,
                                  const void* w_k, int32_t n_out, void* k_latent_buffer,
                                  void* k_buffer, int32_t* dev_status, void* stream) {
    return decompress_bf16(cache, layer_idx, buffer_row_offsets, cache_offsets, batch,
                           buffer_length, kv_lora_rank, rope_dim, w_k, n_out, VOperands{},
                           k_latent_buffer, k_buffer, dev_status, stream);
}

pkm_status mla_decompress_kv_paged(const pkm_paged_cache* cache, uint32_t layer_idx,
                                   const uint32_t* buffer_row_offsets,
                                   const uint32_t* cache_offsets, int32_t batch,
                                   int32_t buffer_length, int32_t kv_lora_rank, int32_t rope_dim,
                                   const void* w_k, int32_t n_out, const void* w_uv,
                                   int32_t num_heads, int32_t v_head_dim, void* k_latent_buffer,
                                   void* k_buffer, void* v_buffer, int32_t* dev_status,
                                   void* stream) {
    bool empty = false;
    pkm_status st = check_decompress_sizes(batch, buffer_length, kv_lora_rank, rope_dim, n_out,
                                           &empty);
    if (st != PKM_OK || empty) return st;
    VOperands v{w_uv, nullptr, 0, v_buffer};
    st = check_v(v, num_heads, v_head_dim, 64);
    if (st != PKM_OK) return st;
    v.n_v = num_heads * v_head_dim;
    return decompress_bf16(cache, layer_idx, buffer_row_offsets, cache_offsets, batch,
                           buffer_length, kv_lora_rank, rope_dim, w_k, n_out, v,
                           k_latent_buffer, k_buffer, dev_status, stream);
}

size_t mla_decompress_k_paged_fp8_workspace_size(int32_t buffer_length, int32_t kv_lora_rank) {
    if (buffer_length < 0 || kv_lora_rank <= 0 || kv_lora_rank % 128 != 0) return 0;
    const size_t L = static_cast<size_t>(buffer_length);
    const size_t R = static_cast<size_t>(kv_lora_rank);
    return align256(L * R) + align256(L * (R / 128) * sizeof(float));
}

pkm_status mla_decompress_k_paged_fp8(const pkm_paged_cache* cache, uint32_t layer_idx,
                                      const uint32_t* buffer_row_offsets,
                                      const uint32_t* cache_offsets, int32_t batch,
                                      int32_t buffer_length, int32_t kv_lora_rank,
                                      int32_t rope_dim, const void* w_k_e4m3,
                                      const float* w_k_scale, int32_t n_out,
                                      void* k_latent_buffer, void* k_buffer, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return decompress_fp8(cache, layer_idx, buffer_row_offsets, cache_offsets, batch,
                          buffer_length, kv_lora_rank, rope_dim, w_k_e4m3, w_k_scale, n_out,
                          VOperands{}, k_latent_buffer, k_buffer, workspace, workspace_bytes,
                          dev_status, stream);
}

pkm_status mla_decompress_kv_paged_fp8(const pkm_paged_cache* cache, uint32_t layer_idx,
                                       const uint32_t* buffer_row_offsets,
                                       const uint32_t* cache_offsets, int32_t batch,
                                       int32_t buffer_length, int32_t kv_lora_rank,
                                       int32_t rope_dim, const void* w_k_e4m3,
                                       const float* w_k_scale, int32_t n_out,
                                       const void* w_uv_e4m3, const float* w_uv_scale,
                                       int32_t num_heads, int32_t v_head_dim,
                                       void* k_latent_buffer, void* k_buffer, void* v_buffer,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* dev_status, void* stream) {
    bool empty = false;
    pkm_status st = check_decompress_sizes(batch, buffer_length, kv_lora_rank, rope_dim, n_out,
                                           &empty);
    if (st != PKM_OK || empty) return st;
    VOperands v{w_uv_e4m3, w_uv_scale, 0, v_buffer};
    st = check_v(v, num_heads, v_head_dim, 128);
    if (st != PKM_OK) return st;
    if (w_uv_scale == nullptr) return PKM_ERR_INVALID_ARG;
    v.n_v = num_heads * v_head_dim;
    return decompress_fp8(cache, layer_idx, buffer_row_offsets, cache_offsets, batch,
                          buffer_length, kv_lora_rank, rope_dim, w_k_e4m3, w_k_scale, n_out, v,
                          k_latent_buffer, k_buffer, workspace, workspace_bytes, dev_status,
                          stream);
}

pkm_status mla_decompress_k_paged_fp8_qcache(const pkm_quant_cache* cache, uint32_t layer_idx,
                                             const uint32_t* buffer_row_offsets,
                                             const uint32_t* cache_offsets, int32_t batch,
                                             int32_t buffer_length, const void* w_k_e4m3,
                                             const float* w_k_scale, int32_t n_out,
                                             void* k_latent_buffer, void* k_buffer,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, void* stream) {
    if (cache == nullptr) return PKM_ERR_INVALID_ARG;
    return decompress_fp8(nullptr, layer_idx, buffer_row_offsets, cache_offsets, batch,
                          buffer_length, cache->kv_lora_rank, cache->rope_dim, w_k_e4m3,
                          w_k_scale, n_out, VOperands{}, k_latent_buffer, k_buffer, workspace,
                          workspace_bytes, dev_status, stream, cache);
}

}  // extern "C"

namespace {

// Body of both cache-write entry points: a bf16 cache, or (qcache) a quantised one.
pkm_status cache_write(const void* latent, const uint32_t* input_row_offsets, int32_t batch,
                       int32_t total_rows, int32_t kv_lora_rank, int32_t rope_dim,
                       const float* kv_norm_gamma, float epsilon, const float* freqs_cis,
                       int32_t max_seq_len, const pkm_paged_cache* cache,
                       const pkm_quant_cache* qcache, uint32_t layer_idx, int32_t* dev_status,
                       void* stream) {
    if (batch < 0 || total_rows < 0 || kv_lora_rank <= 0 || rope_dim < 0 || max_seq_len <= 0)
        return PKM_ERR_INVALID_ARG;
    if (batch == 0 || total_rows == 0) return PKM_OK;
    if (latent == nullptr || input_row_offsets == nullptr || kv_norm_gamma == nullptr ||
        (freqs_cis == nullptr && rope_dim > 0))
        return PKM_ERR_INVALID_ARG;
    if (kv_lora_rank % 8 != 0 || kv_lora_rank > 1024 || rope_dim % 8 != 0 || rope_dim > 256)
        return PKM_ERR_UNSUPPORTED;
    if (!aligned16(latent) || !aligned16(kv_norm_gamma) || !aligned16(freqs_cis))
        return PKM_ERR_INVALID_ARG;
    CacheWriteArgs a{};
    if (qcache != nullptr) {
        if (qcache->data == nullptr || qcache->page_table == nullptr ||
            qcache->cache_lengths == nullptr)
            return PKM_ERR_INVALID_ARG;
        if (qcache->num_layers <= 0 || layer_idx >= static_cast<uint32_t>(qcache->num_layers) ||
            qcache->num_pages <= 0 || qcache->page_size <= 0 || qcache->max_pages_per_seq <= 0)
            return PKM_ERR_INVALID_ARG;
        if (kv_lora_rank % 128 != 0) return PKM_ERR_UNSUPPORTED;
        const int64_t payload = static_cast<int64_t>(kv_lora_rank) + 2 * rope_dim +
                                4 * (kv_lora_rank / 128);
        if (qcache->layer_stride < 0 || qcache->layer_stride % 16 != 0 ||
            qcache->page_stride < 0 || qcache->page_stride % 16 != 0 ||
            qcache->slot_stride % 16 != 0 || qcache->slot_stride < payload ||
            !aligned16(qcache->data))
            return PKM_ERR_INVALID_ARG;
        a.qcache_layer = static_cast<uint8_t*>(qcache->data) +
                         static_cast<int64_t>(layer_idx) * qcache->layer_stride;
        a.page_stride = qcache->page_stride;
        a.slot_stride = qcache->slot_stride;
        a.num_pages = qcache->num_pages;
        a.page_size = qcache->page_size;
        a.max_pages = qcache->max_pages_per_seq;
        a.page_table = qcache->page_table;
        a.cache_lengths = qcache->cache_lengths;
    } else {
        if (cache == nullptr || cache->data == nullptr || cache->page_table == nullptr ||
            cache->cache_lengths == nullptr)
            return PKM_ERR_INVALID_ARG;
        if (cache->num_layers <= 0 || layer_idx >= static_cast<uint32_t>(cache->num_layers) ||
            cache->num_pages <= 0 || cache->page_size <= 0 || cache->max_pages_per_seq <= 0)
            return PKM_ERR_INVALID_ARG;
        if (cache->row_elems != kv_lora_rank + rope_dim) return PKM_ERR_INVALID_ARG;
        if (!mult8(cache->layer_stride) || !mult8(cache->page_stride) ||
            !mult8(cache->slot_stride) || !aligned16(cache->data))
            return PKM_ERR_INVALID_ARG;
        a.cache_layer = static_cast<uint16_t*>(cache->data) +
                        static_cast<int64_t>(layer_idx) * cache->layer_stride;
        a.page_stride = cache->page_stride;
        a.slot_stride = cache->slot_stride;
        a.num_pages = cache->num_pages;
        a.page_size = cache->page_size;
        a.max_pages = cache->max_pages_per_seq;
        a.page_table = cache->page_table;
        a.cache_lengths = cache->cache_lengths;
    }
    a.latent = static_cast<const uint16_t*>(latent);
    a.row_offsets = input_row_offsets;
    a.batch = batch;
    a.total_rows = total_rows;
    a.kv_lora_rank = kv_lora_rank;
    a.rope_dim = rope_dim;
    a.gamma = kv_norm_gamma;
    a.epsilon = epsilon;
    a.freqs = freqs_cis;
    a.max_seq_len = max_seq_len;
    a.status = dev_status;
    a.timeout_ns = wait_timeout_ns();
    int sms = 0;
    if (const cudaError_t e = current_sm_count(&sms)) return cuda_status(e);
    if (const cudaError_t e = debug_validate(a.row_offsets, batch, dev_status, stream))
        return cuda_status(e);
    return cuda_status(pkm::launch_cache_write(a, sms, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

pkm_status mla_cache_write_paged(const void* latent, const uint32_t* input_row_offsets,
                                 int32_t batch, int32_t total_rows, int32_t kv_lora_rank,
                                 int32_t rope_dim, const float* kv_norm_gamma, float epsilon,
                                 const float* freqs_cis, int32_t max_seq_len,
                                 const pkm_paged_cache* cache, uint32_t layer_idx,
                                 int32_t* dev_status, void* stream) {
    return cache_write(latent, input_row_offsets, batch, total_rows, kv_lora_rank, rope_dim,
                       kv_norm_gamma, epsilon, freqs_cis, max_seq_len, cache, nullptr,
                       layer_idx, dev_status, stream);
}

pkm_status mla_cache_write_paged_qcache(const void* latent, const uint32_t* input_row_offsets,
                                        int32_t batch, int32_t total_rows,
                                        const float* kv_norm_gamma, float epsilon,
                                        const float* freqs_cis, int32_t max_seq_len,
                                        const pkm_quant_cache* cache, uint32_t layer_idx,
                                        int32_t* dev_status, void* stream) {
    if (cache == nullptr) return PKM_ERR_INVALID_ARG;
    return cache_write(latent, input_row_offsets, batch, total_rows, cache->kv_lora_rank,
                       cache->rope_dim, kv_norm_gamma, epsilon, freqs_cis, max_seq_len, nullptr,
                       cache, layer_idx, dev_status, stream);
}

pkm_status kv_matmul_paged(const void* hidden_state, const uint32_t* input_row_offsets,
                           int32_t batch, int32_t total_rows, int32_t k_in, const void* weight,
                           int32_t n_out, const pkm_paged_cache* kv_cache, uint32_t layer_idx,
                           int32_t* dev_status, void* stream) {
    if (batch < 0 || total_rows < 0 || k_in <= 0 || n_out <= 0) return PKM_ERR_INVALID_ARG;
    if (total_rows == 0 || batch == 0) return PKM_OK;
    if (hidden_state == nullptr || input_row_offsets == nullptr || weight == nullptr ||
        kv_cache == nullptr || kv_cache->data == nullptr || kv_cache->page_table == nullptr ||
        kv_cache->cache_lengths == nullptr)
        return PKM_ERR_INVALID_ARG;
    if (kv_cache->num_layers <= 0 || layer_idx >= static_cast<uint32_t>(kv_cache->num_layers) ||
        kv_cache->num_pages <= 0 || kv_cache->page_size <= 0 ||
        kv_cache->max_pages_per_seq <= 0 || kv_cache->row_elems <= 0)
        return PKM_ERR_INVALID_ARG;
    const int32_t hd = kv_cache->row_elems;
    if (n_out != hd && n_out != 2 * hd) return PKM_ERR_INVALID_ARG;
    if (!mult8(kv_cache->layer_stride) || !mult8(kv_cache->page_stride) ||
        !mult8(kv_cache->slot_stride) || !mult8(kv_cache->kv_stride))
        return PKM_ERR_INVALID_ARG;
    if (!aligned16(hidden_state) || !aligned16(weight) || !aligned16(kv_cache->data))
        return PKM_ERR_INVALID_ARG;
    if (k_in % 64 != 0 || hd % 64 != 0) return PKM_ERR_UNSUPPORTED;
    KvMatmulArgs a{};
    a.hidden = static_cast<const uint16_t*>(hidden_state);
    a.row_offsets = input_row_offsets;
    a.batch = batch;
    a.total_rows = total_rows;
    a.k_in = k_in;
    a.n_out = n_out;
    a.head_elems = hd;
    a.cache_layer = static_cast<uint16_t*>(kv_cache->data) +
                    static_cast<int64_t>(layer_idx) * kv_cache->layer_stride;
    a.page_stride = kv_cache->page_stride;
    a.slot_stride = kv_cache->slot_stride;
    a.kv_stride = kv_cache->kv_stride;
    a.num_pages = kv_cache->num_pages;
    a.page_size = kv_cache->page_size;
    a.max_pages = kv_cache->max_pages_per_seq;
    a.page_table = kv_cache->page_table;
    a.cache_lengths = kv_cache->cache_lengths;
    a.status = dev_status;
    a.timeout_ns = wait_timeout_ns();
    // CTA-pair tiles: 256 rows (128 per CTA) x bn columns, bn = 256 or 128; when n_out is an
    // odd multiple of 64 the last 128-wide tile is half padding
    a.bn = (n_out % 256 == 0) ? 256 : 128;
    a.n_tiles = (n_out + a.bn - 1) / a.bn;
    a.m_tiles = (total_rows + 255) / 256;
    a.total_tiles = static_cast<int64_t>(a.m_tiles) * a.n_tiles;
    int sms = 0;
    if (const cudaError_t e = current_sm_count(&sms)) return cuda_status(e);
    alignas(64) CUtensorMap tm_x, tm_w;
    if (!encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, hidden_state, k_in, total_rows,
                   static_cast<uint64_t>(k_in) * 2, 64, 128) ||
        !encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, weight, n_out, k_in,
                   static_cast<uint64_t>(n_out) * 2, 64, 64))
        return encode_failed();
    if (const cudaError_t e = debug_validate(a.row_offsets, a.batch, a.status, stream))
        return cuda_status(e);
    return cuda_status(pkm::launch_kv_matmul(tm_x, tm_w, a, sms, static_cast<cudaStream_t>(stream)));
}

size_t kv_matmul_paged_fp8_workspace_size(int32_t total_rows, int32_t k_in) {
    if (total_rows < 0 || k_in <= 0 || k_in % 128 != 0) return 0;
    const size_t M = static_cast<size_t>(total_rows), K = static_cast<size_t>(k_in);
    return align256(M * K) + align256(M * (K / 128) * sizeof(float));
}

pkm_status kv_matmul_paged_fp8(const void* hidden_state, const uint32_t* input_row_offsets,
                               int32_t batch, int32_t total_rows, int32_t k_in,
                               const void* w_e4m3, const float* w_scale, int32_t n_out,
                               const pkm_paged_cache* kv_cache, uint32_t layer_idx,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               void* stream) {
    if (batch < 0 || total_rows < 0 || k_in <= 0 || n_out <= 0) return PKM_ERR_INVALID_ARG;
    if (total_rows == 0 || batch == 0) return PKM_OK;
    if (hidden_state == nullptr || input_row_offsets == nullptr || w_e4m3 == nullptr ||
        w_scale == nullptr || workspace == nullptr || kv_cache == nullptr ||
        kv_cache->data == nullptr || kv_cache->page_table == nullptr ||
        kv_cache->cache_lengths == nullptr)
        return PKM_ERR_INVALID_ARG;
    if (kv_cache->num_layers <= 0 || layer_idx >= static_cast<uint32_t>(kv_cache->num_layers) ||
        kv_cache->num_pages <= 0 || kv_cache->page_size <= 0 ||
        kv_cache->max_pages_per_seq <= 0 || kv_cache->row_elems <= 0)
        return PKM_ERR_INVALID_ARG;
    const int32_t hd = kv_cache->row_elems;
    if (n_out != hd && n_out != 2 * hd) return PKM_ERR_INVALID_ARG;
    if (!mult8(kv_cache->layer_stride) || !mult8(kv_cache->page_stride) ||
        !mult8(kv_cache->slot_stride) || !mult8(kv_cache->kv_stride))
        return PKM_ERR_INVALID_ARG;
    if (!aligned16(hidden_state) || !aligned16(w_e4m3) || !aligned16(kv_cache->data) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return PKM_ERR_INVALID_ARG;
    if (k_in % 128 != 0 || hd % 64 != 0 || n_out % 128 != 0) return PKM_ERR_UNSUPPORTED;
    if (workspace_bytes < kv_matmul_paged_fp8_workspace_size(total_rows, k_in))
        return PKM_ERR_INVALID_ARG;
    KvMatmulArgs a{};
    a.hidden = static_cast<const uint16_t*>(hidden_state);
    a.row_offsets = input_row_offsets;
    a.batch = batch;
    a.total_rows = total_rows;
    a.k_in = k_in;
    a.n_out = n_out;
    a.head_elems = hd;
    a.cache_layer = static_cast<uint16_t*>(kv_cache->data) +
                    static_cast<int64_t>(layer_idx) * kv_cache->layer_stride;
    a.page_stride = kv_cache->page_stride;
    a.slot_stride = kv_cache->slot_stride;
    a.kv_stride = kv_cache->kv_stride;
    a.num_pages = kv_cache->num_pages;
    a.page_size = kv_cache->page_size;
    a.max_pages = kv_cache->max_pages_per_seq;
    a.page_table = kv_cache->page_table;
    a.cache_lengths = kv_cache->cache_lengths;
    a.status = dev_status;
    a.timeout_ns = wait_timeout_ns();
    a.bn = 256;  // pair tiles of 256 rows x two 128-column weight-scale blocks
    a.n_tiles = (n_out + 255) / 256;  // an odd number of blocks leaves a half tile
    a.m_tiles = (total_rows + 255) / 256;
    a.total_tiles = static_cast<int64_t>(a.m_tiles) * a.n_tiles;
    KvFp8Extra x{};
    x.q = static_cast<uint8_t*>(workspace);
    x.q_scale = reinterpret_cast<float*>(
        static_cast<uint8_t*>(workspace) +
        align256(static_cast<size_t>(total_rows) * static_cast<size_t>(k_in)));
    x.w_scale = w_scale;
    int sms = 0;
    if (const cudaError_t e = current_sm_count(&sms)) return cuda_status(e);
    alignas(64) CUtensorMap tm_q, tm_w;
    if (!encode_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, x.q, k_in, total_rows,
                   static_cast<uint64_t>(k_in), 128, 128) ||
        !encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_e4m3, k_in, n_out,
                   static_cast<uint64_t>(k_in), 128, 128))
        return encode_failed();
    if (const cudaError_t e = debug_validate(a.row_offsets, a.batch, a.status, stream))
        return cuda_status(e);
    return cuda_status(pkm::launch_kv_matmul_fp8(tm_q, tm_w, a, x, sms, static_cast<cudaStream_t>(stream)));
}

pkm_status pkm_validate_row_offsets(const uint32_t* offsets, int32_t batch, int32_t* dev_status,
                                    void* stream) {
    if (offsets == nullptr || dev_status == nullptr || batch < 0) return PKM_ERR_INVALID_ARG;
    if (batch == 0) return PKM_OK;
    return cuda_status(pkm::launch_validate_offsets(offsets, batch, dev_status,
                                                    static_cast<cudaStream_t>(stream)));
}

pkm_status pkm_check_wait_timeout(int32_t* dev_status, uint32_t timeout_ms, void* stream) {
    if (dev_status == nullptr || timeout_ms == 0 || timeout_ms > 5000) return PKM_ERR_INVALID_ARG;
    return cuda_status(pkm::launch_wait_timeout_check(dev_status, static_cast<uint64_t>(timeout_ms) * 1000000ull,
                                          static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
