/*
 * paged_kv_mla.h -- C ABI of the GB300 (sm_103a) paged-KV MLA hot path.
 *
 * The operations, after the Modular MAX kernel pages that define them:
 *
 *   mla_decompress_k_paged      generic_flare_mla_decompress_k_cache_ragged_paged
 *                               (nn/kv_cache_ragged; signature, description and Args):
 *                               gather each request's latent K rows out of a paged cache
 *                               into k_latent_buffer, then k_buffer = latent[:, :R] . W_k^T.
 *   mla_decompress_kv_paged     the same gather feeding the K and the V (w_uv) up-projection.
 *   mla_decompress_k_paged_fp8  the same decompress as the K-decompress stage of
 *                               mla_prefill_decode_graph_fp8 (attention/gpu/mla_graph;
 *                               Parameters m/n/k_scale_granularity, Args w_k, w_k_scale,
 *                               buffer_row_offsets, cache_offsets, buffer_length), with an
 *                               e4m3 W_k carrying 128x128 fp32 block scales and the latent
 *                               quantised per token per 128-column block
 *                               (+ _kv_ with w_uv / w_uv_scale, + _noalloc).
 *   mla_decompress_k_paged_fp8_qcache  the FP8 decompress reading a quantised paged cache.
 *   mla_cache_write_paged[_qcache]     the cache-write side of mla_prefill_decode_graph_fp8
 *                               (kv_norm_gamma, epsilon, freqs_cis): RMSNorm and RoPE of new
 *                               latent rows stored into a bf16 or a quantised paged cache.
 *   kv_matmul_paged[_fp8]       kv_matmul_ragged_paged (nn/kv_cache_ragged; description and
 *                               Args): Y = hidden_state . weight on the ragged rows, with
 *                               row i of request b written into the paged K/V cache at
 *                               position cache_lengths[b] + i (bf16, or FP8 block-scaled).
 *
 * Conventions shared by every entry point
 *   - Every tensor argument is DEVICE memory on the current CUDA device, allocated and
 *     owned by the caller.  Shape scalars are host values.  The library keeps no pointer
 *     after a call returns and allocates no device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous on it; outputs are valid once the stream has reached the call.
 *   - The return value reports what the host can check before launching: a NULL
 *     required pointer, misaligned pointer or stride (16-byte rules below), a size the
 *     kernels do not support, or a failed CUDA launch.  Nothing is launched when it is
 *     not PKM_OK.  A call with nothing to do (no rows or no requests) returns PKM_OK
 *     after checking only its sizes, and launches nothing.
 *   - `dev_status` (nullable, device int32) receives errors found on the device, merged
 *     with atomicMax: PKM_ERR_OUT_OF_RANGE when a token resolves past the page table row
 *     or to a page id >= num_pages (that row is then neither read nor written), and
 *     PKM_ERR_TIMEOUT when an internal pipeline wait exceeded its limit (about one
 *     second, PKM_WAIT_TIMEOUT_MS overrides) and the kernel stopped early.  The caller
 *     zeroes it and reads it after synchronising.
 *   - The kernels never trap and never write outside the rows / cache slots the
 *     operation defines.
 *   - bf16 values are IEEE binary32 truncated to 16 bits; products accumulate in fp32 on
 *     the tensor cores and are rounded to bf16 with round-to-nearest-even.
 */
#ifndef PAGED_KV_MLA_H
#define PAGED_KV_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKM_OK = 0,
    PKM_ERR_INVALID_ARG = 1,   /* NULL / misaligned pointer, negative or inconsistent size */
    PKM_ERR_UNSUPPORTED = 2,   /* a size outside what the kernels implement */
    PKM_ERR_CUDA = 3,          /* a CUDA runtime / driver call failed */
    PKM_ERR_OUT_OF_RANGE = 4,  /* device: a token resolved outside the page table / cache */
    PKM_ERR_TIMEOUT = 5        /* device: a pipeline wait timed out, the kernel stopped */
} pkm_status;

/*
 * One paged cache (the PagedKVCacheCollection of the pages, for all layers), described by
 * element strides so that any row-contiguous layout can be addressed.  The slot of token t
 * of request b in layer l is
 *     data + l*layer_stride + page_table[b*max_pages_per_seq + t/page_size]*page_stride
 *          + (t % page_size)*slot_stride            (+ kv_stride for the V plane)
 * and holds row_elems contiguous bf16 values.
 *   data              device, bf16, 16-byte aligned.
 *   *_stride          in elements; layer/page/slot/kv strides must be multiples of 8
 *                     (16 bytes).
 *   num_layers        layers in `data`; layer_idx must be below it.
 *   num_pages         physical pages per layer; page ids >= num_pages are out of range.
 *   page_size         tokens per page (> 0).
 *   row_elems         values per slot that the operation reads or writes: the latent width
 *                     kv_lora_rank + qk_rope_head_dim for the decompress entry points,
 *                     num_kv_heads*head_size for kv_matmul_paged (per plane).
 *   page_table        device uint32 [batch, max_pages_per_seq], row-major.
 *   cache_lengths     device uint32 [batch]: tokens already in the cache per request.  Read
 *                     by kv_matmul_paged only (and never updated by it); may be NULL for
 *                     the decompress entry points.
 *   kv_stride         offset of the V plane from the K plane; kv_matmul_paged only.
 */
typedef struct {
    void* data;
    int64_t layer_stride;
    int64_t page_stride;
    int64_t slot_stride;
    int64_t kv_stride;
    int32_t num_layers;
    int32_t num_pages;
    int32_t page_size;
    int32_t row_elems;
    const uint32_t* page_table;
    int32_t max_pages_per_seq;
    const uint32_t* cache_lengths;
} pkm_paged_cache;

/*
 * A quantised paged latent cache (PagedKVCacheCollection's type parameters scale_dtype_ and
 * quantization_granularity_; the pages give no layout).  One token's slot is a byte string:
 *     bytes [0, R)                     e4m3 codes of the R = kv_lora_rank nope columns
 *     bytes [R, R + 2P)                the P = rope_dim rope columns, bf16
 *     bytes [R + 2P, R + 2P + 4R/128)  fp32 scales, one per 128 columns (scale_dtype_ =
 *                                      float32, quantization_granularity_ = 128)
 * A nope value is fl32(e4m3(code) * scale).  The codes and scales are those the FP8
 * decompress's quantisation (s = amax/448 per 128-column block, q = e4m3_rne(x / s)) makes
 * of the bf16 row a bf16 cache would hold, so the quantised cache (656 bytes a token for
 * DeepSeek-V3 against 1152) feeds the FP8 product the same operands.
 *
 *   data             device bytes, 16-byte aligned.
 *   layer_stride, page_stride, slot_stride   bytes, multiples of 16; slot_stride >= the
 *                    payload R + 2P + 4R/128.
 *   kv_lora_rank     R: a multiple of 128, 128..512 (1024 for the cache write).
 *   rope_dim         P: a multiple of 8, at most 256.
 *   cache_lengths    [batch] existing lengths (the cache write only).
 */
typedef struct {
    void* data;
    int64_t layer_stride;
    int64_t page_stride;
    int64_t slot_stride;
    int32_t num_layers;
    int32_t num_pages;
    int32_t page_size;
    int32_t kv_lora_rank;
    int32_t rope_dim;
    const uint32_t* page_table;
    int32_t max_pages_per_seq;
    const uint32_t* cache_lengths;
} pkm_quant_cache;

/*
 * bf16 latent-K decompress.
 * Source: generic_flare_mla_decompress_k_cache_ragged_paged -- signature, description
 * (latent K rows gathered into k_latent_buffer as buffer_row_offsets and cache_offsets
 * direct, then multiplied by the weight), Args buffer_row_offsets_1d, cache_offsets_1d,
 * buffer_length, weight, kv_collection, layer_idx, k_latent_buffer, k_buffer.
 *
 * For every request b < batch and i < buffer_row_offsets[b+1] - buffer_row_offsets[b]:
 *     r = buffer_row_offsets[b] + i          (skipped when r >= buffer_length)
 *     t = cache_offsets[b] + i               (cache token, resolved through the page table)
 *     k_latent_buffer[r, 0:C] = cache slot of t, bit for bit, C = kv_lora_rank + rope_dim
 *     k_buffer[r, n] = bf16( sum_{k < kv_lora_rank} k_latent_buffer[r, k] * w_k[n, k] )
 * Rows of the outputs that no request covers (r >= buffer_row_offsets[batch], or
 * r < buffer_row_offsets[0]) are left untouched.
 *
 *   cache                host struct; cache->row_elems must equal C.
 *   buffer_row_offsets   device uint32 [batch+1], non-decreasing (not checked here;
 *                        pkm_validate_row_offsets checks it on request).
 *   cache_offsets        device uint32 [>= batch]; entries past batch-1 are not read.
 *   buffer_length        rows of k_latent_buffer and k_buffer (>= 0; 0 launches nothing).
 *   kv_lora_rank         R: multiple of 64, 64..512.
 *   rope_dim             P: C = R + P must be a multiple of 8.
 *   w_k                  device bf16 [n_out, R], R contiguous, 16-byte aligned.
 *   n_out                num_heads * qk_nope_head_dim: a multiple of 64.
 *   k_latent_buffer      device bf16 [buffer_length, C], row-major, 16-byte aligned.
 *   k_buffer             device bf16 [buffer_length, n_out], row-major, 16-byte aligned.
 *
 * Returns PKM_ERR_UNSUPPORTED (launching nothing) when one layer of the cache spans
 * 2^35 - 64 elements (about 64 GiB) or more: the kernel keeps row addresses as 32-bit
 * counts of 16-byte units inside the layer.
 */
pkm_status mla_decompress_k_paged(const pkm_paged_cache* cache, uint32_t layer_idx,
                                  const uint32_t* buffer_row_offsets,
                                  const uint32_t* cache_offsets, int32_t batch,
                                  int32_t buffer_length, int32_t kv_lora_rank,
                                  int32_t rope_dim, const void* w_k, int32_t n_out,
                                  void* k_latent_buffer, void* k_buffer, int32_t* dev_status,
                                  void* stream);

/*
 * bf16 latent-K and V decompress: one gather for both up-projections.
 * Source: generic_flare_mla_decompress_k_cache_ragged_paged (the gather and K, as for
 * mla_decompress_k_paged) and mla_prefill_decode_graph_fp8 -- Args w_uv (the weight that
 * maps latent rows to V, [num_heads, v_head_dim, kv_latent_dim]).
 *
 * Computes exactly what mla_decompress_k_paged computes (k_latent_buffer, k_buffer) and,
 * for every written row r, head h and d < v_head_dim:
 *     v_buffer[r, h, d] = bf16( sum_{k < kv_lora_rank} k_latent_buffer[r, k] * w_uv[h, d, k] )
 * (fp32 accumulation, round to nearest even).  Rows of v_buffer that no request covers
 * are left untouched, like those of the other outputs.
 *
 *   w_uv                 device bf16 [num_heads, v_head_dim, kv_lora_rank], 16-byte aligned.
 *   num_heads, v_head_dim  > 0, num_heads * v_head_dim a multiple of 64.
 *   v_buffer             device bf16 [buffer_length, num_heads, v_head_dim], row-major,
 *                        16-byte aligned.
 *   other arguments      as for mla_decompress_k_paged (same errors).
 */
pkm_status mla_decompress_kv_paged(const pkm_paged_cache* cache, uint32_t layer_idx,
                                   const uint32_t* buffer_row_offsets,
                                   const uint32_t* cache_offsets, int32_t batch,
                                   int32_t buffer_length, int32_t kv_lora_rank,
                                   int32_t rope_dim, const void* w_k, int32_t n_out,
                                   const void* w_uv, int32_t num_heads, int32_t v_head_dim,
                                   void* k_latent_buffer, void* k_buffer, void* v_buffer,
                                   int32_t* dev_status, void* stream);

/*
 * Bytes of device workspace mla_decompress_k_paged_fp8 needs for buffer_length rows of
 * kv_lora_rank latent columns (0 for invalid sizes).  Layout, for a caller that wants to
 * read the quantised activations back:
 *     offset 0                                 e4m3 codes [buffer_length, kv_lora_rank]
 *     offset align256(buffer_length*R)         fp32 scales [buffer_length, kv_lora_rank/128]
 */
size_t mla_decompress_k_paged_fp8_workspace_size(int32_t buffer_length, int32_t kv_lora_rank);

/*
 * FP8 block-scaled latent-K decompress.
 * Source: mla_prefill_decode_graph_fp8 -- Parameters fp8_dtype, fp8_scale_dtype,
 * m_scale_granularity, n_scale_granularity, k_scale_granularity; Args buffer_row_offsets,
 * cache_offsets, buffer_length, w_k (lifts the latent cache to the full K,
 * [num_heads * qk_nope_head_dim, kv_latent_dim]) and w_k_scale.  Granularities are fixed
 * at m = 1, n = 128, k = 128.
 *
 * Same rows and the same k_latent_buffer copy as mla_decompress_k_paged (bf16, all C
 * columns).  Then, per written row r and per 128-column block kb of its first R columns:
 *     s[r, kb] = amax_k |x[r, k]| / 448 in fp32 (1 when the block is all zeros)
 *     q[r, k]  = e4m3_rne_satfinite(x[r, k] / s[r, kb]), the division in fp32
 *     k_buffer[r, n] = bf16( sum_kb s[r, kb] * w_k_scale[n/128, kb]
 *                              * sum_{k in kb} q[r, k] * w_k_e4m3[n, k] )
 *
 *   kv_lora_rank         R: multiple of 128, 128..512.
 *   w_k_e4m3             device e4m3 [n_out, R], R contiguous, 16-byte aligned.
 *   w_k_scale            device fp32 [n_out/128, R/128], row-major.
 *   n_out                multiple of 128.
 *   workspace            device, >= mla_decompress_k_paged_fp8_workspace_size(...) bytes,
 *                        256-byte aligned; receives q and s (layout above).
 *   workspace_bytes      its size.
 *   other arguments      as for mla_decompress_k_paged.
 */
pkm_status mla_decompress_k_paged_fp8(const pkm_paged_cache* cache, uint32_t layer_idx,
                                      const uint32_t* buffer_row_offsets,
                                      const uint32_t* cache_offsets, int32_t batch,
                                      int32_t buffer_length, int32_t kv_lora_rank,
                                      int32_t rope_dim, const void* w_k_e4m3,
                                      const float* w_k_scale, int32_t n_out,
                                      void* k_latent_buffer, void* k_buffer, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status,
                                      void* stream);

/*
 * FP8 block-scaled latent-K and V decompress: one gather and one activation quantisation
 * for both up-projections.
 * Source: mla_prefill_decode_graph_fp8 -- Args w_k, w_k_scale, w_uv (latent-to-V weight,
 * [num_heads, v_head_dim, kv_latent_dim]), w_uv_scale (its scales; no shape is given).
 *
 * Computes exactly what mla_decompress_k_paged_fp8 computes (k_latent_buffer, k_buffer,
 * the workspace) and, with the same quantised row q[r, :] and scales s[r, kb]:
 *     v_buffer[r, h, d] = bf16( sum_kb s[r, kb] * w_uv_scale[j/128, kb]
 *                               * sum_{k in kb} q[r, k] * w_uv_e4m3[h, d, k] ),  j = h*v_head_dim + d
 * i.e. w_uv_scale has w_k_scale's 128 x 128 granularity over w_uv read as a
 * [num_heads * v_head_dim, kv_lora_rank] matrix (the page gives no layout for it).
 *
 *   w_uv_e4m3            device e4m3 [num_heads, v_head_dim, kv_lora_rank], 16-byte aligned.
 *   w_uv_scale           device fp32 [num_heads*v_head_dim/128, kv_lora_rank/128].
 *   num_heads, v_head_dim  > 0, num_heads * v_head_dim a multiple of 128.
 *   v_buffer             device bf16 [buffer_length, num_heads, v_head_dim], 16-byte aligned.
 *   other arguments      as for mla_decompress_k_paged_fp8 (same workspace size).
 */
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
                                       int32_t* dev_status, void* stream);

/*
 * The cache-write side of MLA: new latent rows are RMS-normalised and rotated, then
 * stored into the paged latent cache.
 * Source: mla_prefill_decode_graph_fp8 -- Args kv_input_fn (supplies the new latent rows,
 * [tot_seq_len, cache_head_dim]), kv_norm_gamma (the RMSNorm scale vector applied before
 * caching, [kv_lora_rank]), epsilon (the RMSNorm stabilising term), freqs_cis (rotary
 * factors per position, [max_seq_len, qk_rope_head_dim]), input_row_offsets,
 * kv_collection, layer_idx.
 *
 * For every request b and i < input_row_offsets[b+1] - input_row_offsets[b], with
 * r = input_row_offsets[b] + i (r < total_rows) and position pos = cache_lengths[b] + i:
 *     ms  = (sum_{k < R} x[r, k]^2) / R
 *     slot(pos)[k]         = bf16( x[r, k] * kv_norm_gamma[k] / sqrt(ms + epsilon) ),  k < R
 *     slot(pos)[R+2j, R+2j+1] = bf16( (x0 c - x1 s, x0 s + x1 c) ),  j < P/2,
 *         (x0, x1) = x[r, R+2j .. R+2j+1],  (c, s) = freqs_cis[pos, 2j .. 2j+1]
 * where slot(pos) is the cache row of layer_idx at page page_table[b][pos / page_size],
 * slot pos % page_size.  fp32 arithmetic, round to nearest even.  No other cache element
 * is written; cache_lengths are read, not updated.
 *
 *   latent          device bf16 [total_rows, R + P], row-major, 16-byte aligned.
 *   input_row_offsets  device uint32 [batch+1], non-decreasing (pkm_validate_row_offsets).
 *   kv_lora_rank    R: a multiple of 8, at most 1024.
 *   rope_dim        P: a multiple of 8, at most 256.
 *   kv_norm_gamma   device fp32 [R], 16-byte aligned.
 *   freqs_cis       device fp32 [max_seq_len, P], 16-byte aligned: P/2 (cos, sin) pairs
 *                   per position (may be null when P = 0).
 *   cache           row_elems = R + P; cache_lengths required.
 * Errors: PKM_ERR_INVALID_ARG / PKM_ERR_UNSUPPORTED before any launch; a position past
 * max_seq_len, the page-table row or the cache sets PKM_ERR_OUT_OF_RANGE in dev_status and
 * leaves that row unwritten.
 */
pkm_status mla_cache_write_paged(const void* latent, const uint32_t* input_row_offsets,
                                 int32_t batch, int32_t total_rows, int32_t kv_lora_rank,
                                 int32_t rope_dim, const float* kv_norm_gamma, float epsilon,
                                 const float* freqs_cis, int32_t max_seq_len,
                                 const pkm_paged_cache* cache, uint32_t layer_idx,
                                 int32_t* dev_status, void* stream);

/*
 * FP8 latent-K decompress from a quantised paged cache.
 * Source: generic_flare_mla_decompress_k_cache_ragged_paged (rows, tokens, page walk) with
 * the FP8 product of mla_prefill_decode_graph_fp8 (Args w_k, w_k_scale) over a
 * PagedKVCacheCollection with scale_dtype_ / quantization_granularity_ (layout above).
 *
 * The rows and cache tokens of mla_decompress_k_paged.  Every written row r takes its
 * slot's codes and scales as they are (workspace: codes [L, R] at 0, scales [L, R/128] at
 * align256(L*R), the layout of mla_decompress_k_paged_fp8), and
 *     k_latent_buffer[r, k]     = bf16_rne(fl32(e4m3(code_k) * scale_{k/128})),  k < R
 *     k_latent_buffer[r, R + j] = the slot's rope value j, bit for bit
 *     k_buffer[r, n] = bf16( sum_kb scale[kb] * w_k_scale[n/128, kb]
 *                              * sum_{k in kb} code_k * w_k_e4m3[n, k] )
 * (no quantisation step: the cache already holds the operands).
 *
 *   cache             host struct (kv_lora_rank 128..512, a multiple of 128).
 *   k_latent_buffer   device bf16 [buffer_length, R + P], 16-byte aligned, or null to skip.
 *   workspace         >= mla_decompress_k_paged_fp8_workspace_size(buffer_length, R) bytes,
 *                     256-byte aligned.
 *   other arguments   as for mla_decompress_k_paged_fp8.
 */
pkm_status mla_decompress_k_paged_fp8_qcache(const pkm_quant_cache* cache, uint32_t layer_idx,
                                             const uint32_t* buffer_row_offsets,
                                             const uint32_t* cache_offsets, int32_t batch,
                                             int32_t buffer_length, const void* w_k_e4m3,
                                             const float* w_k_scale, int32_t n_out,
                                             void* k_latent_buffer, void* k_buffer,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, void* stream);

/*
 * Cache write into a quantised paged cache: the rows mla_cache_write_paged would store
 * (RMSNorm with kv_norm_gamma, RoPE with freqs_cis, rounded to bf16), quantised per
 * 128-column block into the slot layout above (s = amax/448 in fp32, 1 for an all-zero
 * block; q = e4m3_rne_satfinite(y / s) with the division in fp32).  Only the slot's payload
 * bytes are written.  Arguments as for mla_cache_write_paged, with R and P taken from the
 * descriptor (R a multiple of 128, at most 1024).
 */
pkm_status mla_cache_write_paged_qcache(const void* latent, const uint32_t* input_row_offsets,
                                        int32_t batch, int32_t total_rows,
                                        const float* kv_norm_gamma, float epsilon,
                                        const float* freqs_cis, int32_t max_seq_len,
                                        const pkm_quant_cache* cache, uint32_t layer_idx,
                                        int32_t* dev_status, void* stream);

/*
 * FP8 decompress for callers that cannot allocate device memory.  The API pages have no
 * counterpart: this entry point exists for users of this library, not for the method.
 *
 * Some callers cannot call cudaMalloc or an allocator of their own: a plug-in inside an
 * engine that hands out only the buffers it planned up front, or a latency-critical serving
 * loop where an allocation (which may synchronise the whole device) is not acceptable.
 * This call computes exactly what mla_decompress_k_paged_fp8 computes, with the same
 * arguments minus the workspace: the quantised latent goes to a fixed array of
 * PKM_FP8_NOALLOC_SCRATCH_BYTES (16 MiB) that the library keeps in device memory.  Every
 * GPU on which the library's device code is loaded holds that array until the process
 * exits.  No call allocates or frees memory.
 *
 *   - Size limit: mla_decompress_k_paged_fp8_workspace_size(buffer_length, kv_lora_rank)
 *     must not exceed PKM_FP8_NOALLOC_SCRATCH_BYTES (for kv_lora_rank 512: at most 31 775
 *     rows); larger calls return PKM_ERR_UNSUPPORTED and launch nothing.
 *   - Set-up: the first call on a device (with that device current) looks up the array's
 *     device address and caches it; make that first call before any stream capture.  The
 *     cached address belongs to the device's current primary context: resetting the device
 *     (cudaDeviceReset) after the first call is not supported, since later calls would
 *     still pass the old address.
 *   - Status codes: the same as mla_decompress_k_paged_fp8's for the same arguments, plus
 *     PKM_ERR_UNSUPPORTED for a call larger than the array.
 *   - Sharing: every call on a device uses the same array and leaves its contents behind.
 *     Nothing in it needs to start at zero.  Calls whose kernels overlap on the GPU (other
 *     streams, other threads) race on the array: order them on one stream or serialise them.
 *   - The quantised codes and scales are not returned; use mla_decompress_k_paged_fp8 with
 *     your own workspace to read them.
 */
#define PKM_FP8_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
pkm_status mla_decompress_k_paged_fp8_noalloc(const pkm_paged_cache* cache, uint32_t layer_idx,
                                              const uint32_t* buffer_row_offsets,
                                              const uint32_t* cache_offsets, int32_t batch,
                                              int32_t buffer_length, int32_t kv_lora_rank,
                                              int32_t rope_dim, const void* w_k_e4m3,
                                              const float* w_k_scale, int32_t n_out,
                                              void* k_latent_buffer, void* k_buffer,
                                              int32_t* dev_status, void* stream);

/*
 * Ragged GEMM written into the paged K/V cache.
 * Source: kv_matmul_ragged_paged -- description (a matmul whose output lands in the KV
 * cache collection) and Args hidden_state (sum(seq_lens), num_heads * head_size),
 * input_row_offsets (batch_size + 1), weight (num_heads * head_size,
 * num_kv_heads * head_size), kv_collection (the K and V cache), layer_idx.
 *
 * For every request b < batch and i < input_row_offsets[b+1] - input_row_offsets[b]:
 *     r = input_row_offsets[b] + i              (skipped when r >= total_rows)
 *     pos = cache->cache_lengths[b] + i          (resolved through the page table)
 *     Y[r, :] = bf16( hidden_state[r, :] . weight )
 *     K plane slot of pos (layer layer_idx)  <- Y[r, 0 : HD]
 *     V plane slot of pos                    <- Y[r, HD : 2 HD]     (when n_out == 2 HD)
 * with HD = cache->row_elems.  No other cache element is written.
 *
 *   hidden_state         device bf16 [total_rows, k_in], row-major, 16-byte aligned.
 *   input_row_offsets    device uint32 [batch+1], non-decreasing (pkm_validate_row_offsets).
 *   total_rows           rows of hidden_state (>= 0; 0 launches nothing).
 *   k_in                 num_heads * head_size: a multiple of 64.
 *   weight               device bf16 [k_in, n_out], n_out contiguous, 16-byte aligned.
 *   n_out                HD (K only) or 2*HD (K then V); HD a multiple of 64.
 *   kv_cache             host struct; cache_lengths required, kv_stride used for V.
 */
pkm_status kv_matmul_paged(const void* hidden_state, const uint32_t* input_row_offsets,
                           int32_t batch, int32_t total_rows, int32_t k_in,
                           const void* weight, int32_t n_out, const pkm_paged_cache* kv_cache,
                           uint32_t layer_idx, int32_t* dev_status, void* stream);

/*
 * Bytes of device workspace kv_matmul_paged_fp8 needs for total_rows hidden rows of k_in
 * columns (0 for invalid sizes).  Layout:
 *     offset 0                                e4m3 codes [total_rows, k_in]
 *     offset align256(total_rows * k_in)      fp32 scales [k_in / 128, total_rows]
 *                                             (k-block-major: scale of row r, block kb at
 *                                             kb * total_rows + r)
 */
size_t kv_matmul_paged_fp8_workspace_size(int32_t total_rows, int32_t k_in);

/*
 * FP8 ragged GEMM with block scales, written into the paged K/V cache.
 * Source: kv_matmul_ragged_paged (as for kv_matmul_paged) with the fp8 type and the
 * m/n/k scale-granularity parameters of mla_prefill_decode_graph_fp8 (Parameters fp8_dtype,
 * fp8_scale_dtype, m_scale_granularity, n_scale_granularity, k_scale_granularity), taken
 * as m = 1, n = k = 128.
 *
 * The rows and positions of kv_matmul_paged.  Each hidden row is quantised per 128-column
 * block like the FP8 decompress's latent (s = amax / 448 in fp32, 1 for an all-zero block;
 * q = e4m3_rne_satfinite(x / s), the division in fp32), then
 *     Y[r, n] = bf16( sum_kb s[r, kb] * w_scale[n / 128, kb]
 *                      * sum_{k in kb} q[r, k] * w_e4m3[n, k] )
 * goes to the K plane (n < HD) or the V plane (n >= HD) of position pos's slot.
 *
 *   hidden_state   device bf16 [total_rows, k_in], 16-byte aligned.
 *   k_in           a multiple of 128.
 *   w_e4m3         device e4m3 [n_out, k_in], k_in contiguous (the bf16 weight's
 *                  transpose), 16-byte aligned.
 *   w_scale        device fp32 [n_out / 128, k_in / 128], row-major.
 *   n_out          HD or 2*HD, a multiple of 128; HD a multiple of 64.
 *   workspace      device, >= kv_matmul_paged_fp8_workspace_size(total_rows, k_in) bytes,
 *                  256-byte aligned; receives the quantised rows (layout above).
 *   other arguments and errors as for kv_matmul_paged.
 */
pkm_status kv_matmul_paged_fp8(const void* hidden_state, const uint32_t* input_row_offsets,
                               int32_t batch, int32_t total_rows, int32_t k_in,
                               const void* w_e4m3, const float* w_scale, int32_t n_out,
                               const pkm_paged_cache* kv_cache, uint32_t layer_idx,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               void* stream);

/*
 * Failure-detection self check (no counterpart on the pages).  Launches one CTA that waits,
 * with the same bounded mbarrier wait every kernel above uses, on a barrier phase that
 * nothing completes.  After timeout_ms (1..5000) the wait gives up and PKM_ERR_TIMEOUT is
 * merged into *dev_status (device int32, required); the kernel then returns normally and
 * the CUDA context stays usable.  Returns PKM_ERR_INVALID_ARG for a NULL status or a limit
 * out of range.
 */
pkm_status pkm_check_wait_timeout(int32_t* dev_status, uint32_t timeout_ms, void* stream);

/*
 * Opt-in check of a request offset array (buffer_row_offsets, input_row_offsets).
 * Source: generic_flare_mla_decompress_k_cache_ragged_paged -- Args buffer_row_offsets_1d,
 * and kv_matmul_ragged_paged -- Args input_row_offsets: prefix offsets, the rows of request
 * b being [offsets[b], offsets[b+1]).
 *
 * Every entry point above requires its offset array to be non-decreasing.  The kernels find
 * a row's request by binary search, so an array that decreases somewhere yields other rows
 * than the per-request definition; it cannot make a kernel access memory out of bounds (every
 * lookup is range-checked), but nothing reports it.  This call launches a small kernel on
 * `stream` that reads offsets[0 .. batch] and merges PKM_ERR_INVALID_ARG into *dev_status
 * (device int32, required) when offsets[b] > offsets[b+1] for some b; it writes nothing else.
 * With the environment variable PKM_DEBUG_VALIDATE=1 every entry point runs it on its own
 * offsets (into its dev_status, when one is given) before its kernels.
 *
 *   offsets     device uint32 [batch + 1].
 *   batch       >= 0 (0 launches nothing).
 * Returns PKM_ERR_INVALID_ARG for a NULL pointer or a negative batch.
 */
pkm_status pkm_validate_row_offsets(const uint32_t* offsets, int32_t batch, int32_t* dev_status,
                                    void* stream);

/* Static, human-readable name of a status code. */
const char* pkm_status_string(pkm_status status);

/* The cause of the last PKM_ERR_CUDA an entry point returned on the calling thread: the
 * CUDA runtime's text for the failed call (a launch, an attribute, a device query), or a
 * note that a tensor map was rejected.  A static string owned by the library, valid until
 * the thread's next failing call; "no CUDA failure recorded" before any.  Not a part of the
 * pages' interface: a diagnostic of this library. */
const char* pkm_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_MLA_H */
