// decompress_fp8_noalloc.cu -- the FP8 decompress for callers that cannot allocate device
// memory.
//
// mla_decompress_k_paged_fp8 needs a workspace for the quantised latent (e4m3 codes and
// fp32 block scales) that the caller allocates.  Some callers have no way to do that: a
// plug-in running inside an engine that owns every device allocation up front, or a
// latency-critical serving loop that must not call cudaMalloc (which can synchronise the
// whole device).  This entry point takes its workspace from a fixed array in device global
// memory that belongs to this library instead.  The array is a file-scope __device__
// variable, so it is created when this file's device code is loaded on a GPU and lives until
// the process exits; no call allocates or frees anything.
//
// Host code cannot use the array's name as a device pointer (on the host it names a
// stand-in object).  The device address is looked up with cudaGetSymbolAddress once per
// device, on the first call made while that device is current, and cached; it is not
// looked up again, so the device's context must outlive the calls (no cudaDeviceReset
// after the first one).
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "paged_kv_mla.h"

namespace {

constexpr size_t kScratchBytes = PKM_FP8_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_fp8_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_fp8_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fp8_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

pkm_status mla_decompress_k_paged_fp8_noalloc(const pkm_paged_cache* cache, uint32_t layer_idx,
                                              const uint32_t* buffer_row_offsets,
                                              const uint32_t* cache_offsets, int32_t batch,
                                              int32_t buffer_length, int32_t kv_lora_rank,
                                              int32_t rope_dim, const void* w_k_e4m3,
                                              const float* w_k_scale, int32_t n_out,
                                              void* k_latent_buffer, void* k_buffer,
                                              int32_t* dev_status, void* stream) {
    // The status codes follow mla_decompress_k_paged_fp8's order of checks: invalid sizes,
    // then calls with nothing to do, then everything else.  Those first two never touch
    // the workspace, so they go to that entry point without one.
    const bool bad_sizes = batch < 0 || buffer_length < 0 || rope_dim < 0 || n_out <= 0 ||
                           kv_lora_rank <= 0;
    if (bad_sizes || batch == 0 || buffer_length == 0)
        return mla_decompress_k_paged_fp8(cache, layer_idx, buffer_row_offsets, cache_offsets,
                                          batch, buffer_length, kv_lora_rank, rope_dim, w_k_e4m3,
                                          w_k_scale, n_out, k_latent_buffer, k_buffer, nullptr, 0,
                                          dev_status, stream);
    const size_t need = mla_decompress_k_paged_fp8_workspace_size(buffer_length, kv_lora_rank);
    if (need == 0) {
        // kv_lora_rank is not a multiple of 128: the regular entry point rejects the call
        // (pointer checks first, then the unsupported rank) before it would touch a
        // workspace, so a stand-in that is never dereferenced takes the workspace's place
        alignas(256) static unsigned char stand_in[256];
        return mla_decompress_k_paged_fp8(cache, layer_idx, buffer_row_offsets, cache_offsets,
                                          batch, buffer_length, kv_lora_rank, rope_dim, w_k_e4m3,
                                          w_k_scale, n_out, k_latent_buffer, k_buffer, stand_in,
                                          sizeof(stand_in), dev_status, stream);
    }
    if (need > kScratchBytes) return PKM_ERR_UNSUPPORTED;  // more rows than the fixed scratch holds
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return PKM_ERR_CUDA;
    // Nothing in the scratch has to start at zero: every code and scale a kept output row
    // depends on is written by this call before it is read.
    return mla_decompress_k_paged_fp8(cache, layer_idx, buffer_row_offsets, cache_offsets, batch,
                                      buffer_length, kv_lora_rank, rope_dim, w_k_e4m3, w_k_scale,
                                      n_out, k_latent_buffer, k_buffer, scratch, kScratchBytes,
                                      dev_status, stream);
}

}  // extern "C"
