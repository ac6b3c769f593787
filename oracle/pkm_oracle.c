/*
 * pkm_oracle.c -- plain, slow, single-threaded CPU oracle for the paged-KV MLA hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or calls
 * this file; only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes, and from which passage:
 *   - generic_flare_mla_decompress_k_cache_ragged_paged (Modular MAX kernels,
 *     nn/kv_cache_ragged), description and Args: for every request b, the rows
 *     [buffer_row_offsets[b], buffer_row_offsets[b+1]) of the ragged buffer receive the
 *     latent K vectors of cache tokens starting at cache_offsets[b]; the gathered rows go
 *     to k_latent_buffer, and k_buffer = latent[:, :kv_lora_rank] x weight^T.
 *   - mla_prefill_decode_graph_fp8 (Modular MAX kernels, attention/gpu/mla_graph),
 *     Parameters (m/n/k_scale_granularity) and Args (w_k, w_k_scale,
 *     buffer_row_offsets, cache_offsets, buffer_length): the same decompress with an
 *     e4m3 weight carrying block scales; the activations are quantised per token per
 *     128-column block (the reading of the silent points is stated at each function).
 *   - mla_prefill_decode_graph_fp8, Args w_uv / w_uv_scale: the V up-projection of the same
 *     gathered latent rows (bf16 and block-scaled FP8).
 *   - mla_prefill_decode_graph_fp8, Args kv_input_fn, kv_norm_gamma, epsilon, freqs_cis: the
 *     cache-write side (RMSNorm and RoPE of new latent rows, stored into the paged cache).
 *   - PagedKVCacheCollection's type parameters scale_dtype_ and quantization_granularity_
 *     (generic_flare_mla_decompress_k_cache_ragged_paged, signature): a quantised paged
 *     latent cache, written by the cache-write side and read by the FP8 decompress.
 *   - kv_matmul_ragged_paged (Modular MAX kernels, nn/kv_cache_ragged), Args: a GEMM on
 *     the ragged hidden_state whose rows are written into the paged cache of one layer,
 *     after each request's existing cache length.  Its FP8 form takes the fp8
 *     type and m/n/k scale granularities of mla_prefill_decode_graph_fp8.
 *
 * Arithmetic: fp64 accumulation; the only roundings are the final fp64 -> bf16
 * round-to-nearest-even, and (FP8 path) the activation quantisation, which is taken in
 * fp32 exactly as the GPU takes it (a quantised code is an integer decision, so both
 * sides decide it in the same precision).
 *
 * Number formats are written from their definitions:
 *   bf16  = 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits (IEEE-754 binary32
 *           truncated to its upper 16 bits);
 *   e4m3  = the OCP FP8 "E4M3" format: 1 sign, 4 exponent bits (bias 7), 3 fraction bits,
 *           no infinities, S.1111.111 is NaN, largest finite 448, smallest subnormal 2^-9.
 *
 * Every pointer is host memory owned by the caller.  Functions return 0 on success and a
 * positive code when the metadata points outside the cache (see each function).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* bf16                                                                                  */
/* ------------------------------------------------------------------------------------ */

/* Exact value of a bf16 bit pattern (every bf16 is a float whose low 16 bits are zero). */
double oracle_bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round-half-to-even of a non-negative double k to an integer-valued double. */
static double rne_integer(double k) {
    double fl = floor(k);
    double frac = k - fl; /* exact: k and fl share the exponent range */
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* fp64 -> bf16, round to nearest, ties to even, overflow to infinity, directly from the
 * double (no intermediate float rounding).  bf16 keeps 8 significant bits; its smallest
 * normal is 2^-126 and its subnormal quantum is 2^-133. */
uint16_t oracle_double_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    int qexp = e - 8;             /* 8 significant bits */
    if (qexp < -133) qexp = -133; /* subnormal quantum */
    double quantum = ldexp(1.0, qexp);
    double r = rne_integer(a / quantum) * quantum; /* a / quantum is exact */
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits and is in range */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------------------ */
/* e4m3 (OCP FP8 E4M3, "fn" variant: finite values and NaN only)                         */
/* ------------------------------------------------------------------------------------ */

double oracle_e4m3_to_double(uint8_t q) {
    int s = (q >> 7) & 1;
    int e = (q >> 3) & 0xF;
    int m = q & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);            /* subnormal: 0.m x 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);   /* normal: 1.m x 2^(e-7) */
    return s ? -v : v;
}

/* float -> e4m3 with round-to-nearest-even and saturation to the largest finite value
 * (448).  NaN maps to the positive NaN code 0x7F.  The sign of zero is kept.  The result
 * is found by rounding |x| on the e4m3 grid (4 significant bits, subnormal quantum 2^-9)
 * and looking the rounded value up among the 127 finite non-negative codes. */
uint8_t oracle_float_to_e4m3_satfinite(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E; /* saturate (also covers +-inf) */
    double r = 0.0;
    if (a != 0.0) {
        int e;
        frexp(a, &e);              /* a = m * 2^e, m in [0.5, 1) */
        int qexp = e - 4;          /* 4 significant bits */
        if (qexp < -9) qexp = -9;  /* subnormal quantum */
        double quantum = ldexp(1.0, qexp);
        r = rne_integer(a / quantum) * quantum;
    }
    /* r <= 448 here: the largest value below 448 rounds at most up to 448 */
    for (int code = 0; code <= 0x7E; ++code)
        if (oracle_e4m3_to_double((uint8_t)code) == r) return sign | (uint8_t)code;
    return 0x7F; /* unreachable for finite input */
}

/* ------------------------------------------------------------------------------------ */
/* Paged-cache addressing                                                                */
/* ------------------------------------------------------------------------------------ */

/* Element offset (from the start of `layer`'s cache) of token t of request b:
 * logical page t / page_size through the page table, slot t % page_size.
 * Returns -1 if the logical page is past the table row or the physical page is past the
 * cache. */
static int64_t token_offset(const uint32_t* page_table, int32_t max_pages_per_seq,
                            int32_t num_pages, int32_t page_size, int64_t page_stride,
                            int64_t slot_stride, int32_t b, uint64_t t) {
    uint64_t logical_page = t / (uint64_t)page_size;
    uint64_t slot = t % (uint64_t)page_size;
    if (logical_page >= (uint64_t)max_pages_per_seq) return -1;
    uint32_t page = page_table[(int64_t)b * max_pages_per_seq + (int64_t)logical_page];
    if (page >= (uint32_t)num_pages) return -1;
    return (int64_t)page * page_stride + (int64_t)slot * slot_stride;
}

/* ------------------------------------------------------------------------------------ */
/* generic_flare_mla_decompress_k_cache_ragged_paged (bf16)                              */
/* ------------------------------------------------------------------------------------ */

/*
 * Step 1 (gather), the explicit loop of the description: for each request b and each
 * i in [0, bro[b+1] - bro[b]): row r = bro[b] + i, cache token t = co[b] + i;
 * k_latent[r, 0:C] = cache[layer][page(b, t)][slot(t)][0:C], copied bit for bit.
 * Rows r >= buffer_length are not written (buffer_length is the row count of the
 * outputs); rows not covered by any request are not written either.
 * row_written[r] (optional, length buffer_length) is set to 1 for every written row.
 * Returns 0, or 4 if some token resolved outside the page table / the cache (that row is
 * then skipped).
 */
int oracle_gather_latent(const uint16_t* cache, int64_t layer_stride, int64_t page_stride,
                         int64_t slot_stride, int32_t num_pages, int32_t page_size,
                         const uint32_t* page_table, int32_t max_pages_per_seq,
                         uint32_t layer_idx, const uint32_t* buffer_row_offsets,
                         const uint32_t* cache_offsets, int32_t batch,
                         int32_t buffer_length, int32_t latent_cols, uint16_t* k_latent,
                         uint8_t* row_written) {
    int status = 0;
    const uint16_t* layer = cache + (int64_t)layer_idx * layer_stride;
    for (int32_t b = 0; b < batch; ++b) {
        uint32_t begin = buffer_row_offsets[b];
        uint32_t end = buffer_row_offsets[b + 1];
        for (uint32_t i = 0; begin + i < end; ++i) {
            uint64_t r = (uint64_t)begin + i;
            if (r >= (uint64_t)buffer_length) break;
            uint64_t t = (uint64_t)cache_offsets[b] + i;
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, t);
            if (off < 0) {
                status = 4;
                continue;
            }
            memcpy(k_latent + r * (uint64_t)latent_cols, layer + off,
                   sizeof(uint16_t) * (size_t)latent_cols);
            if (row_written) row_written[r] = 1;
        }
    }
    return status;
}

/*
 * Step 2 (up-projection), the triple loop: for every written row r and output column n,
 * k[r, n] = bf16_rne( sum_{k < R} latent[r, k] * W[n, k] ), summed in fp64 in order of k.
 * W is [n_out, R] with R contiguous (weight "[num_heads * qk_nope_head_dim,
 * kv_latent_dim]"); only the first R columns of a latent row are multiplied.
 */
void oracle_up_project_bf16(const uint16_t* k_latent, int32_t latent_cols,
                            const uint8_t* row_written, int32_t buffer_length,
                            const uint16_t* w, int32_t kv_lora_rank, int32_t n_out,
                            uint16_t* k_buffer) {
    for (int64_t r = 0; r < buffer_length; ++r) {
        if (row_written && !row_written[r]) continue;
        const uint16_t* a = k_latent + r * latent_cols;
        for (int64_t n = 0; n < n_out; ++n) {
            const uint16_t* wn = w + n * kv_lora_rank;
            double acc = 0.0;
            for (int64_t k = 0; k < kv_lora_rank; ++k)
                acc += oracle_bf16_to_double(a[k]) * oracle_bf16_to_double(wn[k]);
            k_buffer[r * n_out + n] = oracle_double_to_bf16(acc);
        }
    }
}

/* Whole bf16 decompress = step 1 then step 2.  Returns step 1's status. */
int oracle_decompress_k(const uint16_t* cache, int64_t layer_stride, int64_t page_stride,
                        int64_t slot_stride, int32_t num_pages, int32_t page_size,
                        const uint32_t* page_table, int32_t max_pages_per_seq,
                        uint32_t layer_idx, const uint32_t* buffer_row_offsets,
                        const uint32_t* cache_offsets, int32_t batch, int32_t buffer_length,
                        int32_t kv_lora_rank, int32_t rope_dim, const uint16_t* w,
                        int32_t n_out, uint16_t* k_latent, uint16_t* k_buffer,
                        uint8_t* row_written) {
    int32_t latent_cols = kv_lora_rank + rope_dim;
    int st = oracle_gather_latent(cache, layer_stride, page_stride, slot_stride, num_pages,
                                  page_size, page_table, max_pages_per_seq, layer_idx,
                                  buffer_row_offsets, cache_offsets, batch, buffer_length,
                                  latent_cols, k_latent, row_written);
    oracle_up_project_bf16(k_latent, latent_cols, row_written, buffer_length, w,
                           kv_lora_rank, n_out, k_buffer);
    return st;
}

/*
 * Single-row form for sampled checks at full size: computes row `r` alone by finding the
 * request whose range [bro[b], bro[b+1]) holds r (a linear scan), then the same copy and
 * dot products.  Returns 0 when the row is written, 1 when no request covers it or
 * r >= buffer_length, 4 when its token resolves outside the page table / cache.
 */
int oracle_decompress_k_row(const uint16_t* cache, int64_t layer_stride,
                            int64_t page_stride, int64_t slot_stride, int32_t num_pages,
                            int32_t page_size, const uint32_t* page_table,
                            int32_t max_pages_per_seq, uint32_t layer_idx,
                            const uint32_t* buffer_row_offsets,
                            const uint32_t* cache_offsets, int32_t batch,
                            int32_t buffer_length, int32_t kv_lora_rank, int32_t rope_dim,
                            const uint16_t* w, int32_t n_out, int64_t r,
                            uint16_t* latent_row, uint16_t* k_row) {
    if (r < 0 || r >= buffer_length) return 1;
    int32_t latent_cols = kv_lora_rank + rope_dim;
    for (int32_t b = 0; b < batch; ++b) {
        if ((uint64_t)buffer_row_offsets[b] <= (uint64_t)r &&
            (uint64_t)r < (uint64_t)buffer_row_offsets[b + 1]) {
            uint64_t t = (uint64_t)cache_offsets[b] + ((uint64_t)r - buffer_row_offsets[b]);
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, t);
            if (off < 0) return 4;
            const uint16_t* src = cache + (int64_t)layer_idx * layer_stride + off;
            memcpy(latent_row, src, sizeof(uint16_t) * (size_t)latent_cols);
            for (int64_t n = 0; n < n_out; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < kv_lora_rank; ++k)
                    acc += oracle_bf16_to_double(latent_row[k]) *
                           oracle_bf16_to_double(w[n * kv_lora_rank + k]);
                k_row[n] = oracle_double_to_bf16(acc);
            }
            return 0;
        }
    }
    return 1;
}

/* ------------------------------------------------------------------------------------ */
/* FP8 block-scaled decompress (the decompress stage of mla_prefill_decode_graph_fp8)     */
/* ------------------------------------------------------------------------------------ */

/*
 * Activation quantisation of one latent row, 1 x 128 blocks over the first R columns
 * (m_scale_granularity = 1, k_scale_granularity = 128).  Reading of the silent points:
 * the block scale is s = amax / 448 in fp32 (448 = largest finite e4m3), or 1 when the
 * block is all zeros; each element is q = e4m3_rne_satfinite(x / s) with the division
 * in fp32, correctly rounded.  Writes R codes and R/128 scales.
 */
void oracle_quantize_row_e4m3(const uint16_t* latent_row, int32_t kv_lora_rank,
                              uint8_t* q_row, float* scale_row) {
    for (int32_t kb = 0; kb < kv_lora_rank / 128; ++kb) {
        float amax = 0.0f;
        for (int32_t k = kb * 128; k < kb * 128 + 128; ++k) {
            float v = fabsf((float)oracle_bf16_to_double(latent_row[k]));
            if (v > amax) amax = v;
        }
        float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        scale_row[kb] = s;
        for (int32_t k = kb * 128; k < kb * 128 + 128; ++k) {
            float x = (float)oracle_bf16_to_double(latent_row[k]);
            float y = x / s;
            q_row[k] = oracle_float_to_e4m3_satfinite(y);
        }
    }
}

/*
 * Block-scaled product of one quantised row with the e4m3 weight:
 *   k[n] = bf16_rne( sum_kb  sa[kb] * sw[n/128, kb] * sum_{k in kb} dq(q[k]) * dq(qw[n, k]) )
 * in fp64 on the dequantised values.  qw is [n_out, R] (R contiguous); sw is
 * [n_out/128, R/128] (n_scale_granularity = k_scale_granularity = 128).
 */
static void fp8_row_product(const uint8_t* q_row, const float* sa_row, const uint8_t* qw,
                            const float* sw, int32_t kv_lora_rank, int32_t n_out,
                            uint16_t* k_row) {
    int32_t kblocks = kv_lora_rank / 128;
    for (int64_t n = 0; n < n_out; ++n) {
        double total = 0.0;
        for (int32_t kb = 0; kb < kblocks; ++kb) {
            double part = 0.0;
            for (int64_t k = (int64_t)kb * 128; k < (int64_t)kb * 128 + 128; ++k)
                part += oracle_e4m3_to_double(q_row[k]) *
                        oracle_e4m3_to_double(qw[n * kv_lora_rank + k]);
            total += (double)sa_row[kb] * (double)sw[(n / 128) * kblocks + kb] * part;
        }
        k_row[n] = oracle_double_to_bf16(total);
    }
}

/*
 * Whole FP8 decompress: gather (bit copy, as in the bf16 path; k_latent keeps all C bf16
 * columns, rope included), quantise every written row, then the block-scaled product.
 * q_latent [buffer_length, R] and q_scale [buffer_length, R/128] receive the quantised
 * activations of the written rows.  Returns the gather's status.
 */
int oracle_decompress_k_fp8(const uint16_t* cache, int64_t layer_stride, int64_t page_stride,
                            int64_t slot_stride, int32_t num_pages, int32_t page_size,
                            const uint32_t* page_table, int32_t max_pages_per_seq,
                            uint32_t layer_idx, const uint32_t* buffer_row_offsets,
                            const uint32_t* cache_offsets, int32_t batch,
                            int32_t buffer_length, int32_t kv_lora_rank, int32_t rope_dim,
                            const uint8_t* w_e4m3, const float* w_scale, int32_t n_out,
                            uint16_t* k_latent, uint16_t* k_buffer, uint8_t* q_latent,
                            float* q_scale, uint8_t* row_written) {
    int32_t latent_cols = kv_lora_rank + rope_dim;
    int st = oracle_gather_latent(cache, layer_stride, page_stride, slot_stride, num_pages,
                                  page_size, page_table, max_pages_per_seq, layer_idx,
                                  buffer_row_offsets, cache_offsets, batch, buffer_length,
                                  latent_cols, k_latent, row_written);
    int32_t kblocks = kv_lora_rank / 128;
    for (int64_t r = 0; r < buffer_length; ++r) {
        if (!row_written[r]) continue;
        oracle_quantize_row_e4m3(k_latent + r * latent_cols, kv_lora_rank,
                                 q_latent + r * kv_lora_rank, q_scale + r * kblocks);
        fp8_row_product(q_latent + r * kv_lora_rank, q_scale + r * kblocks, w_e4m3, w_scale,
                        kv_lora_rank, n_out, k_buffer + r * n_out);
    }
    return st;
}

/* Single-row FP8 form (same return codes as oracle_decompress_k_row). */
int oracle_decompress_k_fp8_row(const uint16_t* cache, int64_t layer_stride,
                                int64_t page_stride, int64_t slot_stride, int32_t num_pages,
                                int32_t page_size, const uint32_t* page_table,
                                int32_t max_pages_per_seq, uint32_t layer_idx,
                                const uint32_t* buffer_row_offsets,
                                const uint32_t* cache_offsets, int32_t batch,
                                int32_t buffer_length, int32_t kv_lora_rank,
                                int32_t rope_dim, const uint8_t* w_e4m3,
                                const float* w_scale, int32_t n_out, int64_t r,
                                uint16_t* latent_row, uint16_t* k_row, uint8_t* q_row,
                                float* scale_row) {
    if (r < 0 || r >= buffer_length) return 1;
    int32_t latent_cols = kv_lora_rank + rope_dim;
    for (int32_t b = 0; b < batch; ++b) {
        if ((uint64_t)buffer_row_offsets[b] <= (uint64_t)r &&
            (uint64_t)r < (uint64_t)buffer_row_offsets[b + 1]) {
            uint64_t t = (uint64_t)cache_offsets[b] + ((uint64_t)r - buffer_row_offsets[b]);
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, t);
            if (off < 0) return 4;
            memcpy(latent_row, cache + (int64_t)layer_idx * layer_stride + off,
                   sizeof(uint16_t) * (size_t)latent_cols);
            oracle_quantize_row_e4m3(latent_row, kv_lora_rank, q_row, scale_row);
            fp8_row_product(q_row, scale_row, w_e4m3, w_scale, kv_lora_rank, n_out, k_row);
            return 0;
        }
    }
    return 1;
}

/* ------------------------------------------------------------------------------------ */
/* V up-projection with w_uv (mla_prefill_decode_graph_fp8, Args w_uv / w_uv_scale)      */
/* ------------------------------------------------------------------------------------ */

/*
 * w_uv maps latent rows to V, shape [num_heads, v_head_dim, kv_latent_dim].  For every written row r (the rows step 1 of the
 * decompress gathered), head h and d < v_head_dim:
 *   v[r, h, d] = bf16_rne( sum_{k < R} latent[r, k] * w_uv[h, d, k] ),
 * summed in fp64 in order of k, over the first R = kv_lora_rank latent columns (the
 * latent "values" are the same gathered rows the K up-projection reads; the rope columns
 * take no part).  v_buffer is [buffer_length, num_heads, v_head_dim] row-major.
 */
void oracle_up_project_v_bf16(const uint16_t* k_latent, int32_t latent_cols,
                              const uint8_t* row_written, int32_t buffer_length,
                              const uint16_t* w_uv, int32_t num_heads, int32_t v_head_dim,
                              int32_t kv_lora_rank, uint16_t* v_buffer) {
    for (int64_t r = 0; r < buffer_length; ++r) {
        if (row_written && !row_written[r]) continue;
        const uint16_t* a = k_latent + r * latent_cols;
        for (int64_t h = 0; h < num_heads; ++h) {
            for (int64_t d = 0; d < v_head_dim; ++d) {
                const uint16_t* w = w_uv + (h * v_head_dim + d) * kv_lora_rank;
                double acc = 0.0;
                for (int64_t k = 0; k < kv_lora_rank; ++k)
                    acc += oracle_bf16_to_double(a[k]) * oracle_bf16_to_double(w[k]);
                v_buffer[(r * num_heads + h) * v_head_dim + d] = oracle_double_to_bf16(acc);
            }
        }
    }
}

/*
 * K and V from one gather: step 1 (gather), step 2 with w_k into k_buffer, and the V
 * up-projection with w_uv into v_buffer.  Returns the gather's status.
 */
int oracle_decompress_kv(const uint16_t* cache, int64_t layer_stride, int64_t page_stride,
                         int64_t slot_stride, int32_t num_pages, int32_t page_size,
                         const uint32_t* page_table, int32_t max_pages_per_seq,
                         uint32_t layer_idx, const uint32_t* buffer_row_offsets,
                         const uint32_t* cache_offsets, int32_t batch, int32_t buffer_length,
                         int32_t kv_lora_rank, int32_t rope_dim, const uint16_t* w_k,
                         int32_t n_out, const uint16_t* w_uv, int32_t num_heads,
                         int32_t v_head_dim, uint16_t* k_latent, uint16_t* k_buffer,
                         uint16_t* v_buffer, uint8_t* row_written) {
    int32_t latent_cols = kv_lora_rank + rope_dim;
    int st = oracle_gather_latent(cache, layer_stride, page_stride, slot_stride, num_pages,
                                  page_size, page_table, max_pages_per_seq, layer_idx,
                                  buffer_row_offsets, cache_offsets, batch, buffer_length,
                                  latent_cols, k_latent, row_written);
    oracle_up_project_bf16(k_latent, latent_cols, row_written, buffer_length, w_k,
                           kv_lora_rank, n_out, k_buffer);
    oracle_up_project_v_bf16(k_latent, latent_cols, row_written, buffer_length, w_uv,
                             num_heads, v_head_dim, kv_lora_rank, v_buffer);
    return st;
}

/*
 * Block-scaled V product of one quantised row with the e4m3 w_uv.  Reading of the silent
 * point: w_uv_scale has the same 128 x 128 block granularity as w_k_scale over w_uv seen
 * as a [num_heads * v_head_dim, R] matrix, i.e. w_uv_scale[(h * v_head_dim + d) / 128,
 * k / 128]:
 *   v[h, d] = bf16_rne( sum_kb sa[kb] * sv[(h*Dv + d)/128, kb]
 *                        * sum_{k in kb} dq(q[k]) * dq(w_uv[h, d, k]) )  in fp64.
 */
static void fp8_row_product_v(const uint8_t* q_row, const float* sa_row, const uint8_t* qv,
                              const float* sv, int32_t num_heads, int32_t v_head_dim,
                              int32_t kv_lora_rank, uint16_t* v_row) {
    int32_t kblocks = kv_lora_rank / 128;
    for (int64_t h = 0; h < num_heads; ++h) {
        for (int64_t d = 0; d < v_head_dim; ++d) {
            const int64_t j = h * v_head_dim + d;
            double total = 0.0;
            for (int32_t kb = 0; kb < kblocks; ++kb) {
                double part = 0.0;
                for (int64_t k = (int64_t)kb * 128; k < (int64_t)kb * 128 + 128; ++k)
                    part += oracle_e4m3_to_double(q_row[k]) *
                            oracle_e4m3_to_double(qv[j * kv_lora_rank + k]);
                total += (double)sa_row[kb] * (double)sv[(j / 128) * kblocks + kb] * part;
            }
            v_row[j] = oracle_double_to_bf16(total);
        }
    }
}

/*
 * FP8 K and V from one gather and one activation quantisation: the rows are gathered and
 * quantised exactly as in oracle_decompress_k_fp8, then multiplied by w_k (into
 * k_buffer) and by w_uv (into v_buffer [buffer_length, num_heads, v_head_dim]).
 */
int oracle_decompress_kv_fp8(const uint16_t* cache, int64_t layer_stride, int64_t page_stride,
                             int64_t slot_stride, int32_t num_pages, int32_t page_size,
                             const uint32_t* page_table, int32_t max_pages_per_seq,
                             uint32_t layer_idx, const uint32_t* buffer_row_offsets,
                             const uint32_t* cache_offsets, int32_t batch,
                             int32_t buffer_length, int32_t kv_lora_rank, int32_t rope_dim,
                             const uint8_t* w_e4m3, const float* w_scale, int32_t n_out,
                             const uint8_t* w_uv_e4m3, const float* w_uv_scale,
                             int32_t num_heads, int32_t v_head_dim, uint16_t* k_latent,
                             uint16_t* k_buffer, uint16_t* v_buffer, uint8_t* q_latent,
                             float* q_scale, uint8_t* row_written) {
    int st = oracle_decompress_k_fp8(cache, layer_stride, page_stride, slot_stride, num_pages,
                                     page_size, page_table, max_pages_per_seq, layer_idx,
                                     buffer_row_offsets, cache_offsets, batch, buffer_length,
                                     kv_lora_rank, rope_dim, w_e4m3, w_scale, n_out, k_latent,
                                     k_buffer, q_latent, q_scale, row_written);
    int32_t kblocks = kv_lora_rank / 128;
    int64_t nv = (int64_t)num_heads * v_head_dim;
    for (int64_t r = 0; r < buffer_length; ++r) {
        if (!row_written[r]) continue;
        fp8_row_product_v(q_latent + r * kv_lora_rank, q_scale + r * kblocks, w_uv_e4m3,
                          w_uv_scale, num_heads, v_head_dim, kv_lora_rank, v_buffer + r * nv);
    }
    return st;
}

/*
 * Single-row forms for sampled checks at full size (same return codes as
 * oracle_decompress_k_row).  The FP8 form also returns the quantised row.
 */
int oracle_decompress_kv_row(const uint16_t* cache, int64_t layer_stride,
                             int64_t page_stride, int64_t slot_stride, int32_t num_pages,
                             int32_t page_size, const uint32_t* page_table,
                             int32_t max_pages_per_seq, uint32_t layer_idx,
                             const uint32_t* buffer_row_offsets,
                             const uint32_t* cache_offsets, int32_t batch,
                             int32_t buffer_length, int32_t kv_lora_rank, int32_t rope_dim,
                             const uint16_t* w_k, int32_t n_out, const uint16_t* w_uv,
                             int32_t num_heads, int32_t v_head_dim, int64_t r,
                             uint16_t* latent_row, uint16_t* k_row, uint16_t* v_row) {
    int st = oracle_decompress_k_row(cache, layer_stride, page_stride, slot_stride, num_pages,
                                     page_size, page_table, max_pages_per_seq, layer_idx,
                                     buffer_row_offsets, cache_offsets, batch, buffer_length,
                                     kv_lora_rank, rope_dim, w_k, n_out, r, latent_row, k_row);
    if (st != 0) return st;
    const uint8_t one = 1;
    oracle_up_project_v_bf16(latent_row, kv_lora_rank + rope_dim, &one, 1, w_uv, num_heads,
                             v_head_dim, kv_lora_rank, v_row);
    return 0;
}

int oracle_decompress_kv_fp8_row(const uint16_t* cache, int64_t layer_stride,
                                 int64_t page_stride, int64_t slot_stride, int32_t num_pages,
                                 int32_t page_size, const uint32_t* page_table,
                                 int32_t max_pages_per_seq, uint32_t layer_idx,
                                 const uint32_t* buffer_row_offsets,
                                 const uint32_t* cache_offsets, int32_t batch,
                                 int32_t buffer_length, int32_t kv_lora_rank,
                                 int32_t rope_dim, const uint8_t* w_e4m3,
                                 const float* w_scale, int32_t n_out,
                                 const uint8_t* w_uv_e4m3, const float* w_uv_scale,
                                 int32_t num_heads, int32_t v_head_dim, int64_t r,
                                 uint16_t* latent_row, uint16_t* k_row, uint16_t* v_row,
                                 uint8_t* q_row, float* scale_row) {
    int st = oracle_decompress_k_fp8_row(cache, layer_stride, page_stride, slot_stride,
                                         num_pages, page_size, page_table, max_pages_per_seq,
                                         layer_idx, buffer_row_offsets, cache_offsets, batch,
                                         buffer_length, kv_lora_rank, rope_dim, w_e4m3,
                                         w_scale, n_out, r, latent_row, k_row, q_row,
                                         scale_row);
    if (st != 0) return st;
    fp8_row_product_v(q_row, scale_row, w_uv_e4m3, w_uv_scale, num_heads, v_head_dim,
                      kv_lora_rank, v_row);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Cache-write side of mla_prefill_decode_graph_fp8 (kv_norm_gamma, epsilon, freqs_cis)  */
/* ------------------------------------------------------------------------------------ */

/*
 * The graph's Args: kv_input_fn supplies the new latent rows, shape [tot_seq_len,
 * cache_head_dim]; kv_norm_gamma is the RMSNorm scale vector, [kv_lora_rank]; epsilon is
 * the RMSNorm constant; freqs_cis holds the rotary factors of each position,
 * [max_seq_len, qk_rope_head_dim]; input_row_offsets delimits each request's rows;
 * kv_collection / layer_idx name the cache.
 *
 * Readings of the silent points:
 *   - row r = iro[b] + i of the new latent values is token position pos = cache_lengths[b]
 *     + i of request b (the position rule kv_matmul_ragged_paged uses for new tokens) and
 *     goes to that position's cache slot: logical page pos / page_size through the page
 *     table, slot pos % page_size;
 *   - the first R = kv_lora_rank columns are RMS-normalised:
 *         y_k = x_k * gamma_k / sqrt( (sum_{k<R} x_k^2) / R + epsilon ),
 *   - the last P = qk_rope_head_dim columns are rotated by freqs_cis[pos], read as P/2
 *     complex numbers (cos, sin) applied to the interleaved pairs (x_2j, x_2j+1):
 *         (x_2j, x_2j+1) -> (x_2j * cos - x_2j+1 * sin, x_2j * sin + x_2j+1 * cos),
 *   - gamma and freqs_cis are fp32; the arithmetic is fp64 here and every result is
 *     rounded once to bf16.
 * Nothing else in the cache is written.  Returns 0, or 4 if a row's position resolves
 * outside the page table / the cache or past max_seq_len (that row is skipped).
 */
/* One row: x (R + P bf16 values) -> y, with f = freqs_cis[pos]. */
static void cache_write_row(const uint16_t* x, int32_t kv_lora_rank, int32_t rope_dim,
                            const float* gamma, float epsilon, const float* f, uint16_t* y) {
    double sumsq = 0.0;
    for (int32_t k = 0; k < kv_lora_rank; ++k) {
        double v = oracle_bf16_to_double(x[k]);
        sumsq += v * v;
    }
    double inv = 1.0 / sqrt(sumsq / (double)kv_lora_rank + (double)epsilon);
    for (int32_t k = 0; k < kv_lora_rank; ++k)
        y[k] = oracle_double_to_bf16(oracle_bf16_to_double(x[k]) * inv * (double)gamma[k]);
    for (int32_t j = 0; j < rope_dim / 2; ++j) {
        double x0 = oracle_bf16_to_double(x[kv_lora_rank + 2 * j]);
        double x1 = oracle_bf16_to_double(x[kv_lora_rank + 2 * j + 1]);
        double c = (double)f[2 * j], sn = (double)f[2 * j + 1];
        y[kv_lora_rank + 2 * j] = oracle_double_to_bf16(x0 * c - x1 * sn);
        y[kv_lora_rank + 2 * j + 1] = oracle_double_to_bf16(x0 * sn + x1 * c);
    }
}

int oracle_cache_write(const uint16_t* latent, const uint32_t* input_row_offsets,
                       int32_t batch, int32_t total_rows, int32_t kv_lora_rank,
                       int32_t rope_dim, const float* gamma, float epsilon,
                       const float* freqs_cis, int32_t max_seq_len, uint16_t* cache,
                       int64_t layer_stride, int64_t page_stride, int64_t slot_stride,
                       int32_t num_pages, int32_t page_size, const uint32_t* page_table,
                       int32_t max_pages_per_seq, const uint32_t* cache_lengths,
                       uint32_t layer_idx) {
    int status = 0;
    const int32_t C = kv_lora_rank + rope_dim;
    uint16_t* layer = cache + (int64_t)layer_idx * layer_stride;
    for (int32_t b = 0; b < batch; ++b) {
        uint32_t begin = input_row_offsets[b];
        uint32_t end = input_row_offsets[b + 1];
        for (uint32_t i = 0; begin + i < end; ++i) {
            uint64_t r = (uint64_t)begin + i;
            if (r >= (uint64_t)total_rows) break;
            uint64_t pos = (uint64_t)cache_lengths[b] + i;
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, pos);
            if (off < 0 || pos >= (uint64_t)max_seq_len) {
                status = 4;
                continue;
            }
            cache_write_row(latent + r * (uint64_t)C, kv_lora_rank, rope_dim, gamma, epsilon,
                            freqs_cis + pos * (uint64_t)rope_dim, layer + off);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------------------ */
/* Quantised paged latent cache (PagedKVCacheCollection scale_dtype_,                    */
/* quantization_granularity_)                                                            */
/* ------------------------------------------------------------------------------------ */

/*
 * The collection's type parameters scale_dtype_ and quantization_granularity_ say that a
 * paged cache may hold quantised values with scales; the pages give no layout and no rule.
 * Readings:
 *   - one token's slot is a byte string:
 *         [0, R)                     e4m3 codes of the R nope columns,
 *         [R, R + 2P)                the P rope columns in bf16 (not quantised),
 *         [R + 2P, R + 2P + 4R/128)  fp32 scales, one per 128-column block
 *     (scale_dtype_ = float32, quantization_granularity_ = 128 columns of one token);
 *   - the codes and scales are exactly what the FP8 decompress's activation quantisation
 *     (oracle_quantize_row_e4m3) makes of the bf16 row the bf16 cache would hold, so a
 *     quantised cache feeds the block-scaled product the same operands;
 *   - a nope value reads back as fl32(dq(code) * scale) rounded to bf16: the dequantisation
 *     is taken in the scale's dtype.
 * Strides of a quantised cache are in bytes.
 */

uint16_t oracle_dequant_bf16(uint8_t code, float scale) {
    volatile float p = (float)oracle_e4m3_to_double(code) * scale;  /* one fp32 rounding */
    return oracle_double_to_bf16((double)p);
}

/* Stores the bf16 row y (R + P values) into a quantised slot. */
static void qslot_store(const uint16_t* y, int32_t kv_lora_rank, int32_t rope_dim,
                        uint8_t* slot) {
    float scales[8];
    oracle_quantize_row_e4m3(y, kv_lora_rank, slot, scales);
    memcpy(slot + kv_lora_rank, y + kv_lora_rank, sizeof(uint16_t) * (size_t)rope_dim);
    memcpy(slot + kv_lora_rank + 2 * rope_dim, scales, sizeof(float) * (size_t)(kv_lora_rank / 128));
}

/* Bytes of a quantised slot's payload (its stride may be larger). */
int64_t oracle_qslot_bytes(int32_t kv_lora_rank, int32_t rope_dim) {
    return (int64_t)kv_lora_rank + 2 * (int64_t)rope_dim + 4 * (int64_t)(kv_lora_rank / 128);
}

/*
 * Cache write into a quantised cache: the row oracle_cache_write would store (RMSNorm,
 * RoPE, bf16), quantised into the slot as above.  R is a multiple of 128, at most 1024;
 * P at most 256.  Same positions, same status as oracle_cache_write.
 */
int oracle_cache_write_q(const uint16_t* latent, const uint32_t* input_row_offsets,
                         int32_t batch, int32_t total_rows, int32_t kv_lora_rank,
                         int32_t rope_dim, const float* gamma, float epsilon,
                         const float* freqs_cis, int32_t max_seq_len, uint8_t* cache,
                         int64_t layer_stride, int64_t page_stride, int64_t slot_stride,
                         int32_t num_pages, int32_t page_size, const uint32_t* page_table,
                         int32_t max_pages_per_seq, const uint32_t* cache_lengths,
                         uint32_t layer_idx) {
    int status = 0;
    const int32_t C = kv_lora_rank + rope_dim;
    uint16_t y[1280];
    uint8_t* layer = cache + (int64_t)layer_idx * layer_stride;
    for (int32_t b = 0; b < batch; ++b) {
        uint32_t begin = input_row_offsets[b];
        uint32_t end = input_row_offsets[b + 1];
        for (uint32_t i = 0; begin + i < end; ++i) {
            uint64_t r = (uint64_t)begin + i;
            if (r >= (uint64_t)total_rows) break;
            uint64_t pos = (uint64_t)cache_lengths[b] + i;
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, pos);
            if (off < 0 || pos >= (uint64_t)max_seq_len) {
                status = 4;
                continue;
            }
            cache_write_row(latent + r * (uint64_t)C, kv_lora_rank, rope_dim, gamma, epsilon,
                            freqs_cis + pos * (uint64_t)rope_dim, y);
            qslot_store(y, kv_lora_rank, rope_dim, layer + off);
        }
    }
    return status;
}

/* Reads one quantised slot: codes and scales as stored, the bf16 latent row dequantised. */
static void qslot_load(const uint8_t* slot, int32_t kv_lora_rank, int32_t rope_dim,
                       uint16_t* latent_row, uint8_t* q_row, float* scale_row) {
    memcpy(q_row, slot, (size_t)kv_lora_rank);
    memcpy(scale_row, slot + kv_lora_rank + 2 * rope_dim,
           sizeof(float) * (size_t)(kv_lora_rank / 128));
    for (int32_t k = 0; k < kv_lora_rank; ++k)
        latent_row[k] = oracle_dequant_bf16(q_row[k], scale_row[k / 128]);
    memcpy(latent_row + kv_lora_rank, slot + kv_lora_rank, sizeof(uint16_t) * (size_t)rope_dim);
}

/*
 * FP8 decompress from a quantised cache: the rows and tokens of the decompress; each
 * written row takes its slot's codes and scales as they are (q_latent, q_scale), its
 * dequantised bf16 row (k_latent, C = R + P columns) and the block-scaled product with
 * the e4m3 weight (k_buffer).  Returns 0, or 4 as the gather does.
 */
int oracle_decompress_k_qcache_fp8(const uint8_t* cache, int64_t layer_stride,
                                   int64_t page_stride, int64_t slot_stride, int32_t num_pages,
                                   int32_t page_size, const uint32_t* page_table,
                                   int32_t max_pages_per_seq, uint32_t layer_idx,
                                   const uint32_t* buffer_row_offsets,
                                   const uint32_t* cache_offsets, int32_t batch,
                                   int32_t buffer_length, int32_t kv_lora_rank,
                                   int32_t rope_dim, const uint8_t* w_e4m3,
                                   const float* w_scale, int32_t n_out, uint16_t* k_latent,
                                   uint16_t* k_buffer, uint8_t* q_latent, float* q_scale,
                                   uint8_t* row_written) {
    int status = 0;
    const int32_t C = kv_lora_rank + rope_dim;
    const int32_t kblocks = kv_lora_rank / 128;
    const uint8_t* layer = cache + (int64_t)layer_idx * layer_stride;
    for (int32_t b = 0; b < batch; ++b) {
        uint32_t begin = buffer_row_offsets[b];
        uint32_t end = buffer_row_offsets[b + 1];
        for (uint32_t i = 0; begin + i < end; ++i) {
            uint64_t r = (uint64_t)begin + i;
            if (r >= (uint64_t)buffer_length) break;
            uint64_t t = (uint64_t)cache_offsets[b] + i;
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, t);
            if (off < 0) {
                status = 4;
                continue;
            }
            qslot_load(layer + off, kv_lora_rank, rope_dim, k_latent + r * (uint64_t)C,
                       q_latent + r * (uint64_t)kv_lora_rank, q_scale + r * (uint64_t)kblocks);
            fp8_row_product(q_latent + r * (uint64_t)kv_lora_rank, q_scale + r * (uint64_t)kblocks,
                            w_e4m3, w_scale, kv_lora_rank, n_out, k_buffer + r * (uint64_t)n_out);
            if (row_written) row_written[r] = 1;
        }
    }
    return status;
}

/* Single-row form of oracle_decompress_k_qcache_fp8 (returns 1 if no request covers r). */
int oracle_decompress_k_qcache_fp8_row(const uint8_t* cache, int64_t layer_stride,
                                       int64_t page_stride, int64_t slot_stride,
                                       int32_t num_pages, int32_t page_size,
                                       const uint32_t* page_table, int32_t max_pages_per_seq,
                                       uint32_t layer_idx, const uint32_t* buffer_row_offsets,
                                       const uint32_t* cache_offsets, int32_t batch,
                                       int32_t buffer_length, int32_t kv_lora_rank,
                                       int32_t rope_dim, const uint8_t* w_e4m3,
                                       const float* w_scale, int32_t n_out, int64_t r,
                                       uint16_t* latent_row, uint16_t* k_row, uint8_t* q_row,
                                       float* scale_row) {
    if (r < 0 || r >= buffer_length) return 1;
    for (int32_t b = 0; b < batch; ++b) {
        if ((uint64_t)buffer_row_offsets[b] <= (uint64_t)r &&
            (uint64_t)r < (uint64_t)buffer_row_offsets[b + 1]) {
            uint64_t t = (uint64_t)cache_offsets[b] + ((uint64_t)r - buffer_row_offsets[b]);
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, t);
            if (off < 0) return 4;
            qslot_load(cache + (int64_t)layer_idx * layer_stride + off, kv_lora_rank, rope_dim,
                       latent_row, q_row, scale_row);
            fp8_row_product(q_row, scale_row, w_e4m3, w_scale, kv_lora_rank, n_out, k_row);
            return 0;
        }
    }
    return 1;
}

/* ------------------------------------------------------------------------------------ */
/* kv_matmul_ragged_paged                                                                */
/* ------------------------------------------------------------------------------------ */

/*
 * Y = hidden_state x weight, hidden_state [total_rows, k_in] (k_in contiguous), weight
 * [k_in, n_out] (n_out contiguous), summed in fp64 in order of k, rounded to bf16.
 * Row r of request b (i = r - iro[b]) lands at cache position pos = cache_lengths[b] + i:
 * page = page_table[b][pos / page_size], slot = pos % page_size.  Columns
 * [0, head_elems) go to the K plane of `layer`, columns [head_elems, 2*head_elems) to the
 * V plane (kv_stride elements further); n_out is head_elems (K only) or 2*head_elems.
 * Nothing else in the cache is written.  Returns 0, or 4 if some row resolved outside the
 * page table / cache (that row is skipped).
 */
int oracle_kv_matmul(const uint16_t* hidden_state, const uint32_t* input_row_offsets,
                     int32_t batch, int32_t total_rows, int32_t k_in, const uint16_t* weight,
                     int32_t n_out, uint16_t* cache, int64_t layer_stride,
                     int64_t page_stride, int64_t slot_stride, int64_t kv_stride,
                     int32_t num_pages, int32_t page_size, int32_t head_elems,
                     const uint32_t* page_table, int32_t max_pages_per_seq,
                     const uint32_t* cache_lengths, uint32_t layer_idx) {
    int status = 0;
    uint16_t* layer = cache + (int64_t)layer_idx * layer_stride;
    for (int32_t b = 0; b < batch; ++b) {
        uint32_t begin = input_row_offsets[b];
        uint32_t end = input_row_offsets[b + 1];
        for (uint32_t i = 0; begin + i < end; ++i) {
            uint64_t r = (uint64_t)begin + i;
            if (r >= (uint64_t)total_rows) break;
            uint64_t pos = (uint64_t)cache_lengths[b] + i;
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, pos);
            if (off < 0) {
                status = 4;
                continue;
            }
            for (int64_t n = 0; n < n_out; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < k_in; ++k)
                    acc += oracle_bf16_to_double(hidden_state[r * k_in + k]) *
                           oracle_bf16_to_double(weight[k * n_out + n]);
                int64_t plane = (n < head_elems) ? 0 : kv_stride;
                layer[plane + off + (n % head_elems)] = oracle_double_to_bf16(acc);
            }
        }
    }
    return status;
}

/*
 * FP8 kv_matmul with block scales (kv_matmul_ragged_paged's GEMM and scatter, with the FP8
 * type and scale-granularity parameters of mla_prefill_decode_graph_fp8: fp8_dtype,
 * fp8_scale_dtype, m/n/k_scale_granularity).  Readings: the hidden state still arrives in
 * bf16 and is quantised per token per 128-column block exactly as the FP8 decompress
 * quantises the latent (oracle_quantize_row_e4m3: s = amax/448, q = e4m3_rne(x / s));
 * the weight is given quantised, e4m3 [n_out, k_in] (k_in contiguous, the transpose of the
 * bf16 weight's [k_in, n_out]) with fp32 scales [n_out/128, k_in/128];
 *   Y[r, n] = bf16( sum_kb sx[r, kb] * sw[n/128, kb] * sum_{k in kb} qx[r, k] * qw[n, k] )
 * in fp64 on the dequantised values (fp8_row_product), stored like oracle_kv_matmul.
 * q_out [total_rows, k_in] and s_out [total_rows, k_in/128] (optional) receive the
 * quantised rows that were written.  Returns 0 or 4 as oracle_kv_matmul does.
 */
int oracle_kv_matmul_fp8(const uint16_t* hidden_state, const uint32_t* input_row_offsets,
                         int32_t batch, int32_t total_rows, int32_t k_in, const uint8_t* w_e4m3,
                         const float* w_scale, int32_t n_out, uint16_t* cache,
                         int64_t layer_stride, int64_t page_stride, int64_t slot_stride,
                         int64_t kv_stride, int32_t num_pages, int32_t page_size,
                         int32_t head_elems, const uint32_t* page_table,
                         int32_t max_pages_per_seq, const uint32_t* cache_lengths,
                         uint32_t layer_idx, uint8_t* q_out, float* s_out) {
    int status = 0;
    uint16_t* layer = cache + (int64_t)layer_idx * layer_stride;
    uint8_t q[8192];
    float sx[64];
    uint16_t y[8192];
    if (k_in > 8192 || n_out > 8192) return 1;
    for (int32_t b = 0; b < batch; ++b) {
        uint32_t begin = input_row_offsets[b];
        uint32_t end = input_row_offsets[b + 1];
        for (uint32_t i = 0; begin + i < end; ++i) {
            uint64_t r = (uint64_t)begin + i;
            if (r >= (uint64_t)total_rows) break;
            uint64_t pos = (uint64_t)cache_lengths[b] + i;
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, pos);
            if (off < 0) {
                status = 4;
                continue;
            }
            oracle_quantize_row_e4m3(hidden_state + r * (uint64_t)k_in, k_in, q, sx);
            if (q_out) memcpy(q_out + r * (uint64_t)k_in, q, (size_t)k_in);
            if (s_out) memcpy(s_out + r * (uint64_t)(k_in / 128), sx, sizeof(float) * (size_t)(k_in / 128));
            fp8_row_product(q, sx, w_e4m3, w_scale, k_in, n_out, y);
            for (int64_t n = 0; n < n_out; ++n) {
                int64_t plane = (n < head_elems) ? 0 : kv_stride;
                layer[plane + off + (n % head_elems)] = y[n];
            }
        }
    }
    return status;
}

/*
 * The addressing step of kv_matmul_ragged_paged alone, for checks at sizes where the
 * oracle's GEMM is too slow: dest[r] (r < total_rows) = element offset, inside the K plane
 * of the layer, of the slot that receives row r (same walk as oracle_kv_matmul), -1 when no
 * request covers r, -2 when the position resolves outside the page table / cache.
 */
void oracle_kv_row_dest(const uint32_t* input_row_offsets, int32_t batch, int32_t total_rows,
                        const uint32_t* cache_lengths, const uint32_t* page_table,
                        int32_t max_pages_per_seq, int32_t num_pages, int32_t page_size,
                        int64_t page_stride, int64_t slot_stride, int64_t* dest) {
    for (int64_t r = 0; r < total_rows; ++r) dest[r] = -1;
    for (int32_t b = 0; b < batch; ++b) {
        uint32_t begin = input_row_offsets[b];
        uint32_t end = input_row_offsets[b + 1];
        for (uint32_t i = 0; begin + i < end; ++i) {
            uint64_t r = (uint64_t)begin + i;
            if (r >= (uint64_t)total_rows) break;
            uint64_t pos = (uint64_t)cache_lengths[b] + i;
            int64_t off = token_offset(page_table, max_pages_per_seq, num_pages, page_size,
                                       page_stride, slot_stride, b, pos);
            dest[r] = off < 0 ? -2 : off;
        }
    }
}
