// validate.cu -- opt-in device check of a request offset array (buffer_row_offsets of the
// decompress, input_row_offsets of kv_matmul and the cache write).
//
// generic_flare_mla_decompress_k_cache_ragged_paged (Args buffer_row_offsets_1d) and
// kv_matmul_ragged_paged (Args input_row_offsets) give these arrays as prefix offsets: the
// rows of request b are [offsets[b], offsets[b+1]).  The kernels rely on that order (they
// find a row's request by binary search), so an array that decreases somewhere gives other
// rows than a per-request loop would.  Such an array cannot make a kernel read or write out
// of bounds -- every lookup is range-checked -- but it goes unreported.  This check reads
// the array on the device (where the caller's array lives) and merges PKM_ERR_INVALID_ARG
// into the status word when offsets[b] > offsets[b+1] for some b; it writes nothing else.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

__global__ void __launch_bounds__(256)
    validate_offsets_kernel(const uint32_t* offsets, int32_t batch, int32_t* status) {
    bool bad = false;
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < batch;
         b += static_cast<int64_t>(gridDim.x) * blockDim.x)
        bad = bad || __ldg(offsets + b) > __ldg(offsets + b + 1);
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) report(status, PKM_ERR_INVALID_ARG);
}

}  // namespace

cudaError_t launch_validate_offsets(const uint32_t* offsets, int32_t batch, int32_t* status,
                                    cudaStream_t stream) {
    int64_t blocks = (static_cast<int64_t>(batch) + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) blocks = 1;
    validate_offsets_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(offsets, batch,
                                                                               status);
    return cudaGetLastError();
}

}  // namespace pkm
