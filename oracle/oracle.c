/* CPU oracle for paged, quantized KV-cache decode attention and the
 * quantize-on-write.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may call it.  It shares no code with the
 * CUDA library and must never be used as a fallback for it.
 *
 * Sources (web pages on PagedAttention and KV-cache quantization):
 *  - "Reducing LLM Inference Latency: KV Cache Quantization and
 *    PagedAttention in vLLM" (mohashari.github.io): KV-size formula and its
 *    snippet-1; block manager and address translation, snippet-3; block-wise
 *    FP8 E4M3 scale = amax / 448 clamped at 1e-12 and the cast, snippet-4;
 *    E4M3 = 1 sign, 4 exponent, 3 mantissa bits, max 448.
 *  - "Optimizing KV-Cache Memory Footprint in High-Throughput LLM Serving"
 *    (publishertech.pages.dev): section 2 formula 2*L*H*D*S*B*P; section 4
 *    INT4 group-wise quantization with per-group scales.
 *  - "KV Cache Compression & Paged Attention" deep dive
 *    (www.myaihardware.com), "Implementation Details": the kernel's inputs
 *    (query, page table, pool of pages, token count) and its loop over
 *    logical blocks -> physical blocks -> K, V -> scores -> softmax ->
 *    weighted sum.
 *  - "KV Cache Optimization: 3x Faster LLM Inference on 24GB VRAM"
 *    (tildalice.io): softmax(Q K^T / sqrt(d_k)) V per head, GQA groups of
 *    query heads sharing one KV pair, ceil(n/p) pages.
 *
 * Readings where the pages leave a step open (each is stated where used):
 *  R1  pool layout per KV tensor [num_blocks, num_kv_heads, block_size, row].
 *  R2  GQA: query head h reads KV head h / (Hq / Hkv).
 *  R3  the page loop runs over ceil(ctx / bs) blocks; tokens >= ctx masked.
 *  R4  FP8 scale per (block, kv-head), separately for K and V.  A call
 *      that writes the token at offset 0 of a block opens that block: its
 *      scale is max(amax / 448, 1e-12) with amax over every token that the
 *      same call writes into the block ("Block-Wise Scaling Factors",
 *      snippet-4: one scale from the absolute maximum of the block).  Tokens
 *      that a later call appends to the block reuse that scale and saturate
 *      at +-448 (the tokens to come are not known when the block opens).
 *  R5  FP8 code = E4M3 round-to-nearest-even with saturation to +-448 of
 *      the fp32 quotient x / scale (one IEEE fp32 division).
 *  R6  INT4: per (token, kv-head, 32 consecutive d), asymmetric:
 *      scale = fp16(fp32(max - min + 0) / 15), zero = fp16(min + 0) (the
 *      "+ 0" makes a signed-zero min or range +0),
 *      code = clamp(rint((x - zero) / scale), 0, 15) in fp32 (0 if scale is
 *      0); element 2i in the low nibble of byte i, 2i+1 in the high nibble.
 *  R7  context_len == 0 gives out = 0; slot -1 means "skip this token".
 *  R8  FP8 E5M2 (1 sign, 5 exponent, 2 mantissa bits; the pages name E4M3
 *      only): the same block-wise recipe as R4/R5 with 57344, E5M2's
 *      largest finite value, in place of 448.
 *  R18 chunked prefill: query j of a chunk of n over a context of c tokens
 *      sits at position c - n + j and sees tokens 0 .. c - n + j (causal).
 *  R9  INT8 (the pages give one byte per element and no format): the same
 *      block-wise recipe with 127: scale = max(amax / 127, 1e-12), code =
 *      clamp(rint(x / scale), -127, 127) of the fp32 quotient, round half to
 *      even, stored as a two's complement byte; dequantized = code * scale.
 *
 * Build with -ffp-contract=off: the encoders must round each fp32 step.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { DT_F16 = 0, DT_BF16 = 1, DT_FP8 = 2, DT_INT4 = 3, DT_E5M2 = 4, DT_INT8 = 5 };

/* one byte per element, one fp32 scale per (block, KV head): FP8 and INT8 */
static int is_blk8(int kv_dtype) {
    return kv_dtype == DT_FP8 || kv_dtype == DT_E5M2 || kv_dtype == DT_INT8;
}

/* ------------------------------------------------------------ codecs */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1F;
    int f = bits & 0x3FF;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp(1.0 + f / 1024.0, e - 15);
    return sign ? -mag : mag;
}

/* bfloat16: the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 7) & 0xFF;
    int f = bits & 0x7F;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -133);                /* subnormal: f/128 * 2^-126 */
    else if (e == 255)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp(1.0 + f / 128.0, e - 127);
    return sign ? -mag : mag;
}

static double half_word_to_double(uint16_t bits, int dtype) {
    return dtype == DT_F16 ? oracle_f16_to_double(bits) : oracle_bf16_to_double(bits);
}

/* fp32 -> binary16, round to nearest, ties to even.  Works on the exact
 * value in double: scale into an integer significand grid and rint(). */
uint16_t oracle_f32_to_f16_rne(float xf) {
    double x = (double)xf;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7E00;
    if (a >= 65520.0) return sign | 0x7C00;          /* rounds past 65504 -> inf */
    if (a < ldexp(1.0, -14)) {
        /* subnormal grid of 2^-24; a result of 1024 is the smallest normal */
        double m = rint(a * ldexp(1.0, 24));
        return sign | (uint16_t)m;
    }
    int ex;
    frexp(a, &ex);                                   /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                                  /* a in [2^e, 2^(e+1)) */
    double m = rint((a / ldexp(1.0, e) - 1.0) * 1024.0);   /* 0..1024 */
    /* m == 1024 carries into the exponent field through the addition */
    return sign | (uint16_t)(((e + 15) << 10) + (int)m);
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * no infinities; S.1111.111 is NaN; largest finite 448 = 0x7E;
 * subnormals m/8 * 2^-6. */
double oracle_e4m3_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 15 && m == 7)
        mag = NAN;
    else if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* E4M3, round to nearest even, saturating to +-448 (R5).  The sign of the
 * input is kept, so -0 and negative values that round to 0 give 0x80. */
uint8_t oracle_e4m3_encode(float yf) {
    double y = (double)yf;
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0;
    double a = fabs(y);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        double m = rint(a * ldexp(1.0, 9));          /* subnormal grid 2^-9; 8 = min normal */
        return sign | (uint8_t)m;
    }
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    double m = rint((a / ldexp(1.0, e) - 1.0) * 8.0);       /* 0..8 */
    int code = ((e + 7) << 3) + (int)m;
    if (code > 0x7E) code = 0x7E;                    /* 464 <= a < 480 would round to 480 */
    return sign | (uint8_t)code;
}

/* OCP FP8 E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits, IEEE-like:
 * S.11111.00 is infinity, S.11111.xx (xx != 0) NaN; largest finite
 * 1.75 * 2^15 = 57344 = 0x7B; subnormals m/4 * 2^-14. */
double oracle_e5m2_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 2) & 0x1F;
    int m = code & 0x3;
    double mag;
    if (e == 31)
        mag = m ? NAN : INFINITY;
    else if (e == 0)
        mag = ldexp((double)m, -16);
    else
        mag = ldexp(1.0 + m / 4.0, e - 15);
    return sign ? -mag : mag;
}

/* E5M2, round to nearest even, saturating to +-57344 (R8); sign kept as in
 * the E4M3 encoder; NaN gives 0x7F. */
uint8_t oracle_e5m2_encode(float yf) {
    double y = (double)yf;
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0;
    double a = fabs(y);
    if (a >= 57344.0) return sign | 0x7B;
    if (a < ldexp(1.0, -14)) {
        double m = rint(a * ldexp(1.0, 16));         /* subnormal grid 2^-16; 4 = min normal */
        return sign | (uint8_t)m;
    }
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    double m = rint((a / ldexp(1.0, e) - 1.0) * 4.0);       /* 0..4 */
    int code = ((e + 15) << 2) + (int)m;
    if (code > 0x7B) code = 0x7B;
    return sign | (uint8_t)code;
}

/* INT8 code of the fp32 quotient y (R9): round half to even, clamp to
 * [-127, 127] (NaN gives 0). */
int8_t oracle_int8_encode(float yf) {
    double y = (double)yf;
    if (isnan(y)) return 0;
    double r = rint(y);                  /* the default rounding mode: half to even */
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int8_t)r;
}

/* ------------------------------------------------------------ formulas */

/* KV bytes = 2 (K and V) * layers * heads * head_dim * seq_len * batch * bytes. */
double oracle_kv_cache_bytes(double layers, double heads, double head_dim, double seq_len,
                             double batch, double bytes_per_elem) {
    return 2.0 * layers * heads * head_dim * seq_len * batch * bytes_per_elem;
}

/* ceil(tokens / page_size) pages. */
int64_t oracle_num_pages(int64_t tokens, int64_t page_size) {
    return (tokens + page_size - 1) / page_size;
}

/* logical block = t / bs, offset = t % bs, physical = table[logical]. */
int oracle_physical_address(const int32_t* table_row, int num_entries, int block_size,
                            int64_t token_index, int32_t* physical_block, int32_t* offset) {
    if (token_index < 0 || block_size <= 0) return -1;
    int64_t logical = token_index / block_size;
    if (logical >= num_entries) return -1;
    *physical_block = table_row[logical];
    *offset = (int32_t)(token_index % block_size);
    return 0;
}

/* ------------------------------------------------------------ layouts */

/* bytes of one token row of one head in the cache (R1) */
static int64_t row_bytes(int kv_dtype, int head_dim) {
    switch (kv_dtype) {
    case DT_F16: case DT_BF16: return 2 * (int64_t)head_dim;
    case DT_FP8: case DT_E5M2: case DT_INT8: return head_dim;
    case DT_INT4: return head_dim / 2;
    }
    return -1;
}

static int64_t row_index(int32_t block, int kv_head, int offset,
                         int num_kv_heads, int block_size) {
    return ((int64_t)block * num_kv_heads + kv_head) * block_size + offset;
}

/* FP8 scales: f32 [2][num_blocks][num_kv_heads] */
static float* fp8_scale_ptr(void* scales, int which_kv, int32_t block, int kv_head,
                            int num_blocks, int num_kv_heads) {
    return (float*)scales +
           ((int64_t)which_kv * num_blocks + block) * num_kv_heads + kv_head;
}

/* INT4 scale/zero pairs: f16 [2][num_blocks][num_kv_heads][block_size][D/32][2] */
static uint16_t* int4_pair_ptr(void* scales, int which_kv, int32_t block, int kv_head,
                               int offset, int group, int num_blocks, int num_kv_heads,
                               int block_size, int head_dim) {
    int64_t r = ((int64_t)which_kv * num_blocks + block) * num_kv_heads + kv_head;
    r = (r * block_size + offset) * (head_dim / 32) + group;
    return (uint16_t*)scales + 2 * r;
}

int oracle_dequant_row(const void* cache, const void* scales, int which_kv, int kv_dtype,
                       int num_blocks, int num_kv_heads, int head_dim, int block_size,
                       int32_t block, int kv_head, int offset, double* row) {
    if (block < 0 || block >= num_blocks) return -1;
    int64_t rb = row_bytes(kv_dtype, head_dim);
    const uint8_t* base = (const uint8_t*)cache +
                          row_index(block, kv_head, offset, num_kv_heads, block_size) * rb;
    switch (kv_dtype) {
    case DT_F16: case DT_BF16: {
        const uint16_t* h = (const uint16_t*)base;
        for (int d = 0; d < head_dim; ++d) row[d] = half_word_to_double(h[d], kv_dtype);
        return 0;
    }
    case DT_FP8: case DT_E5M2: {
        /* snippet-4's dequantize: code value times the block's scale */
        double s = *fp8_scale_ptr((void*)scales, which_kv, block, kv_head, num_blocks,
                                  num_kv_heads);
        for (int d = 0; d < head_dim; ++d)
            row[d] = (kv_dtype == DT_FP8 ? oracle_e4m3_to_double(base[d])
                                         : oracle_e5m2_to_double(base[d])) * s;
        return 0;
    }
    case DT_INT8: {
        double s = *fp8_scale_ptr((void*)scales, which_kv, block, kv_head, num_blocks,
                                  num_kv_heads);
        for (int d = 0; d < head_dim; ++d) row[d] = (double)(int8_t)base[d] * s;   /* R9 */
        return 0;
    }
    case DT_INT4: {
        for (int d = 0; d < head_dim; ++d) {
            int code = (d & 1) ? (base[d / 2] >> 4) & 0xF : base[d / 2] & 0xF;
            const uint16_t* sz = int4_pair_ptr((void*)scales, which_kv, block, kv_head, offset,
                                               d / 32, num_blocks, num_kv_heads, block_size,
                                               head_dim);
            row[d] = code * oracle_f16_to_double(sz[0]) + oracle_f16_to_double(sz[1]);
        }
        return 0;
    }
    }
    return -1;
}

/* ------------------------------------------------------------ the write */

static int check_geometry(int kv_dtype, int num_blocks, int num_kv_heads, int head_dim,
                          int block_size) {
    if (kv_dtype < DT_F16 || kv_dtype > DT_INT8) return -1;
    if (num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return -1;
    if (kv_dtype == DT_INT4 && head_dim % 32) return -1;
    return 0;
}

/* ------------------------------------------------------------ block copies */

/* Copy-on-write / beam fork ("KV Cache Compression & Paged Attention Deep
 * Dive", sections "PagedAttention: Operating System-Inspired Memory
 * Management for LLMs" and "Implementation Details"): for each (src, dst)
 * pair in order, every K and V row of every head of block dst, and the
 * scales that belong to those rows, become those of block src.  Pairs with
 * an id outside [0, num_blocks) are skipped; the return value counts them
 * (negative on a bad argument). */
int oracle_copy_blocks(void* k_cache, void* v_cache, void* scales, int kv_dtype,
                       const int32_t* pairs, int num_pairs, int num_blocks, int num_kv_heads,
                       int head_dim, int block_size) {
    if (check_geometry(kv_dtype, num_blocks, num_kv_heads, head_dim, block_size)) return -1;
    if (num_pairs < 0) return -1;
    int64_t rb = row_bytes(kv_dtype, head_dim);
    int skipped = 0;
    for (int i = 0; i < num_pairs; ++i) {
        int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            ++skipped;
            continue;
        }
        for (int which = 0; which < 2; ++which) {
            uint8_t* cache = (uint8_t*)(which ? v_cache : k_cache);
            for (int h = 0; h < num_kv_heads; ++h) {
                for (int o = 0; o < block_size; ++o)
                    memmove(cache + row_index(dst, h, o, num_kv_heads, block_size) * rb,
                            cache + row_index(src, h, o, num_kv_heads, block_size) * rb,
                            (size_t)rb);
                if (is_blk8(kv_dtype))
                    *fp8_scale_ptr(scales, which, dst, h, num_blocks, num_kv_heads) =
                        *fp8_scale_ptr(scales, which, src, h, num_blocks, num_kv_heads);
                if (kv_dtype == DT_INT4)
                    for (int o = 0; o < block_size; ++o)
                        for (int g = 0; g < head_dim / 32; ++g) {
                            uint16_t* d = int4_pair_ptr(scales, which, dst, h, o, g, num_blocks,
                                                        num_kv_heads, block_size, head_dim);
                            const uint16_t* sp = int4_pair_ptr(scales, which, src, h, o, g,
                                                               num_blocks, num_kv_heads,
                                                               block_size, head_dim);
                            d[0] = sp[0];
                            d[1] = sp[1];
                        }
            }
        }
    }
    return skipped;
}


/* largest finite code value of a one-byte format: E4M3 448 (snippet-4),
 * E5M2 57344 (R8), INT8 127 (R9) */
static float blk8_max(int kv_dtype) {
    return kv_dtype == DT_FP8 ? 448.0f : kv_dtype == DT_E5M2 ? 57344.0f : 127.0f;
}

/* max |x_d| of one row in fp32; a NaN element is passed over */
static float row_amax(const float* x, int head_dim) {
    float amax = 0.0f;
    for (int d = 0; d < head_dim; ++d) {
        float a = fabsf(x[d]);
        if (a > amax) amax = a;
    }
    return amax;
}

/* Encode one token row of one head (R4-R6).  x: the row as fp32 values;
 * one-byte formats use the block's scale, already set (*fp8_scale). */
static void encode_row(const float* x, int head_dim, int kv_dtype, uint8_t* dst,
                       const float* fp8_scale, uint16_t* int4_pairs) {
    if (is_blk8(kv_dtype)) {
        float s = *fp8_scale;
        for (int d = 0; d < head_dim; ++d) {
            if (kv_dtype == DT_INT8)
                dst[d] = (uint8_t)oracle_int8_encode(x[d] / s);
            else
                dst[d] = kv_dtype == DT_FP8 ? oracle_e4m3_encode(x[d] / s)
                                            : oracle_e5m2_encode(x[d] / s);
        }
        return;
    }
    /* INT4, R6 */
    for (int g = 0; g < head_dim / 32; ++g) {
        const float* xg = x + 32 * g;
        float mn = xg[0], mx = xg[0];
        for (int i = 1; i < 32; ++i) {
            if (xg[i] < mn) mn = xg[i];
            if (xg[i] > mx) mx = xg[i];
        }
        /* "+ 0.0f" turns a -0 minimum or range into +0, so the stored bits do
         * not depend on which of two signed zeros a min/max search meets first */
        float range = (mx - mn) + 0.0f;
        uint16_t sh = oracle_f32_to_f16_rne(range / 15.0f);
        uint16_t zh = oracle_f32_to_f16_rne(mn + 0.0f);
        float sf = (float)oracle_f16_to_double(sh);
        float zf = (float)oracle_f16_to_double(zh);
        int4_pairs[2 * g] = sh;
        int4_pairs[2 * g + 1] = zh;
        for (int i = 0; i < 32; ++i) {
            int code = 0;
            if (sf != 0.0f) {
                float t = (xg[i] - zf) / sf;
                float r = rintf(t);
                if (r < 0.0f) r = 0.0f;
                if (r > 15.0f) r = 15.0f;
                code = (int)r;
            }
            int d = 32 * g + i;
            uint8_t* byte = dst + d / 2;
            if (d & 1)
                *byte = (uint8_t)((*byte & 0x0F) | (code << 4));
            else
                *byte = (uint8_t)((*byte & 0xF0) | code);
        }
    }
}

static void row_to_f32(const uint16_t* srow, int new_dtype, int head_dim, float* x) {
    for (int d = 0; d < head_dim; ++d) x[d] = (float)half_word_to_double(srow[d], new_dtype);
}

/* The quantize-on-write of one call (R4-R9), in four plain steps:
 *  1. the blocks this call opens: those whose offset-0 slot it writes;
 *  2. for each opened block, KV head and K/V: amax over every token of the
 *     call that lands in the block (snippet-4's block-wide absolute max);
 *  3. the opened blocks' scales: max(amax / max_finite, 1e-12) in fp32;
 *  4. every token row encoded with its block's scale (set in step 3, or by
 *     an earlier call).
 * Steps 1-3 concern the one-byte formats only.  Slots of -1 (and any slot
 * outside the pool) are skipped. */
int oracle_kv_write(const uint16_t* k_new, const uint16_t* v_new, int new_dtype,
                    const int64_t* slot_mapping, int64_t num_tokens,
                    void* k_cache, void* v_cache, void* scales, int kv_dtype,
                    int num_blocks, int num_kv_heads, int head_dim, int block_size) {
    if (check_geometry(kv_dtype, num_blocks, num_kv_heads, head_dim, block_size)) return -1;
    if (new_dtype != DT_F16 && new_dtype != DT_BF16) return -1;
    if ((kv_dtype == DT_F16 || kv_dtype == DT_BF16) && new_dtype != kv_dtype) return -1;
    int64_t nslots = (int64_t)num_blocks * block_size;
    int64_t rb = row_bytes(kv_dtype, head_dim);
    float* x = (float*)malloc(sizeof(float) * head_dim);
    if (!x) return -2;

    if (is_blk8(kv_dtype)) {
        int64_t nscale = 2 * (int64_t)num_blocks * num_kv_heads;
        uint8_t* opened = (uint8_t*)calloc((size_t)num_blocks, 1);
        float* amax = (float*)calloc((size_t)nscale, sizeof(float));
        if (!opened || !amax) {
            free(opened);
            free(amax);
            free(x);
            return -2;
        }
        for (int64_t i = 0; i < num_tokens; ++i) {                       /* step 1 */
            int64_t slot = slot_mapping[i];
            if (slot >= 0 && slot < nslots && slot % block_size == 0)
                opened[slot / block_size] = 1;
        }
        for (int64_t i = 0; i < num_tokens; ++i) {                       /* step 2 */
            int64_t slot = slot_mapping[i];
            if (slot < 0 || slot >= nslots || !opened[slot / block_size]) continue;
            int32_t block = (int32_t)(slot / block_size);
            for (int which = 0; which < 2; ++which)
                for (int h = 0; h < num_kv_heads; ++h) {
                    const uint16_t* src = which ? v_new : k_new;
                    row_to_f32(src + (i * num_kv_heads + h) * (int64_t)head_dim, new_dtype,
                               head_dim, x);
                    float a = row_amax(x, head_dim);
                    float* m = &amax[((int64_t)which * num_blocks + block) * num_kv_heads + h];
                    if (a > *m) *m = a;
                }
        }
        for (int32_t b = 0; b < num_blocks; ++b) {                       /* step 3 */
            if (!opened[b]) continue;
            for (int which = 0; which < 2; ++which)
                for (int h = 0; h < num_kv_heads; ++h) {
                    float s = amax[((int64_t)which * num_blocks + b) * num_kv_heads + h] /
                              blk8_max(kv_dtype);
                    if (s < 1e-12f) s = 1e-12f;
                    *fp8_scale_ptr(scales, which, b, h, num_blocks, num_kv_heads) = s;
                }
        }
        free(opened);
        free(amax);
    }

    for (int64_t i = 0; i < num_tokens; ++i) {                           /* step 4 */
        int64_t slot = slot_mapping[i];
        if (slot < 0 || slot >= nslots) continue;                        /* -1: skip (R7) */
        int32_t block = (int32_t)(slot / block_size);
        int offset = (int)(slot % block_size);
        for (int which = 0; which < 2; ++which) {
            const uint16_t* src = which ? v_new : k_new;
            uint8_t* cache = (uint8_t*)(which ? v_cache : k_cache);
            for (int h = 0; h < num_kv_heads; ++h) {
                const uint16_t* srow = src + (i * num_kv_heads + h) * (int64_t)head_dim;
                uint8_t* dst = cache + row_index(block, h, offset, num_kv_heads,
                                                 block_size) * rb;
                if (kv_dtype == DT_F16 || kv_dtype == DT_BF16) {
                    memcpy(dst, srow, (size_t)rb);
                    continue;
                }
                row_to_f32(srow, new_dtype, head_dim, x);
                const float* s8 = is_blk8(kv_dtype)
                                      ? fp8_scale_ptr(scales, which, block, h, num_blocks,
                                                      num_kv_heads)
                                      : NULL;
                uint16_t* p4 = kv_dtype == DT_INT4
                                   ? int4_pair_ptr(scales, which, block, h, offset, 0,
                                                   num_blocks, num_kv_heads, block_size,
                                                   head_dim)
                                   : NULL;
                encode_row(x, head_dim, kv_dtype, dst, s8, p4);
            }
        }
    }
    free(x);
    return 0;
}

/* ------------------------------------------------------------ attention */

/* One (sequence, query head): out = sum_t e^(s_t - max) V_t / sum_t e^(s_t - max),
 * s_t = softmax_scale * q . K_t, all in fp64 over dequantized K/V. */
static int attend_one(const uint16_t* q, int q_dtype, const void* k_cache,
                      const void* v_cache, const int32_t* table_row, int max_blocks_per_seq,
                      int ctx, const void* scales, int kv_dtype, int num_blocks, double* out,
                      double softmax_scale, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int seq, int head, double* scratch) {
    int group = num_q_heads / num_kv_heads;
    int kv_head = head / group;                          /* R2 */
    double* qd = scratch;
    double* row = scratch + head_dim;
    double* scores = scratch + 2 * head_dim;
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (ctx <= 0) return 0;                              /* R7 */
    const uint16_t* qrow = q + ((int64_t)seq * num_q_heads + head) * head_dim;
    for (int d = 0; d < head_dim; ++d) qd[d] = half_word_to_double(qrow[d], q_dtype);
    double mx = -INFINITY;
    for (int t = 0; t < ctx; ++t) {
        int32_t phys, off;
        if (oracle_physical_address(table_row, max_blocks_per_seq, block_size, t, &phys, &off))
            return -1;
        if (oracle_dequant_row(k_cache, scales, 0, kv_dtype, num_blocks, num_kv_heads,
                               head_dim, block_size, phys, kv_head, off, row))
            return -1;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += qd[d] * row[d];
        scores[t] = softmax_scale * dot;
        if (scores[t] > mx) mx = scores[t];
    }
    double denom = 0.0;
    for (int t = 0; t < ctx; ++t) {
        int32_t phys, off;
        if (oracle_physical_address(table_row, max_blocks_per_seq, block_size, t, &phys, &off))
            return -1;
        if (oracle_dequant_row(v_cache, scales, 1, kv_dtype, num_blocks, num_kv_heads, head_dim,
                               block_size, phys, kv_head, off, row))
            return -1;
        double w = exp(scores[t] - mx);
        denom += w;
        for (int d = 0; d < head_dim; ++d) out[d] += w * row[d];
    }
    for (int d = 0; d < head_dim; ++d) out[d] /= denom;
    return 0;
}

static int check_attn(int q_dtype, int kv_dtype, int num_blocks, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, int num_seqs) {
    if (q_dtype != DT_F16 && q_dtype != DT_BF16) return -1;
    if (check_geometry(kv_dtype, num_blocks, num_kv_heads, head_dim, block_size)) return -1;
    if (num_q_heads <= 0 || num_q_heads % num_kv_heads || num_seqs < 0) return -1;
    return 0;
}

int oracle_decode_attention_pairs(const uint16_t* q, int q_dtype,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int num_seqs,
                                  const void* scales, int kv_dtype, int num_blocks,
                                  double* out, double softmax_scale,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, const int32_t* pair_seq,
                                  const int32_t* pair_head, int n_pairs, int num_threads) {
    if (check_attn(q_dtype, kv_dtype, num_blocks, num_q_heads, num_kv_heads, head_dim,
                   block_size, num_seqs))
        return -1;
    int max_ctx = 0;
    for (int b = 0; b < num_seqs; ++b)
        if (context_lens[b] > max_ctx) max_ctx = context_lens[b];
    int err = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads) reduction(| : err)
#endif
    {
        double* scratch = (double*)malloc(sizeof(double) * (2 * (size_t)head_dim + max_ctx + 1));
        if (!scratch) {
            err |= 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int i = 0; i < n_pairs; ++i) {
                int b = pair_seq[i], h = pair_head[i];
                if (b < 0 || b >= num_seqs || h < 0 || h >= num_q_heads) {
                    err |= 1;
                    continue;
                }
                if (attend_one(q, q_dtype, k_cache, v_cache,
                               block_tables + (int64_t)b * max_blocks_per_seq,
                               max_blocks_per_seq, context_lens[b], scales, kv_dtype,
                               num_blocks, out + (int64_t)i * head_dim, softmax_scale,
                               num_q_heads, num_kv_heads, head_dim, block_size, b, h, scratch))
                    err |= 1;
            }
            free(scratch);
        }
    }
    (void)num_threads;
    return err ? -1 : 0;
}

int oracle_decode_attention(const uint16_t* q, int q_dtype,
                            const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs,
                            const void* scales, int kv_dtype, int num_blocks,
                            double* out, double softmax_scale,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int num_threads) {
    int n = num_seqs * num_q_heads;
    int32_t* ps = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n + 1));
    int32_t* ph = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n + 1));
    if (!ps || !ph) {
        free(ps);
        free(ph);
        return -2;
    }
    for (int i = 0; i < n; ++i) {
        ps[i] = i / num_q_heads;
        ph[i] = i % num_q_heads;
    }
    int r = oracle_decode_attention_pairs(q, q_dtype, k_cache, v_cache, block_tables,
                                          max_blocks_per_seq, context_lens, num_seqs, scales,
                                          kv_dtype, num_blocks, out, softmax_scale,
                                          num_q_heads, num_kv_heads, head_dim, block_size, ps,
                                          ph, n, num_threads);
    free(ps);
    free(ph);
    return r;
}

/* Chunked prefill (R18): sequence b's queries are rows q_start[b] ..
 * q_start[b+1] - 1 of q; query j sits at position pos = ctx_b - n_b + j and
 * attends to tokens 0 .. pos (the plain softmax definition over them, as
 * attend_one); a query at a negative position gives zeros.  out: fp64
 * [q_start[num_seqs]][num_q_heads][head_dim]. */
int oracle_prefill_attention(const uint16_t* q, int q_dtype, const int32_t* q_start,
                             const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, int num_seqs, const void* scales,
                             int kv_dtype, int num_blocks, double* out, double softmax_scale,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_threads) {
    if (check_attn(q_dtype, kv_dtype, num_blocks, num_q_heads, num_kv_heads, head_dim,
                   block_size, num_seqs))
        return -1;
    int rows = num_seqs > 0 ? q_start[num_seqs] : 0;
    int max_ctx = 0;
    for (int b = 0; b < num_seqs; ++b) {
        if (q_start[b + 1] < q_start[b]) return -1;
        if (context_lens[b] > max_ctx) max_ctx = context_lens[b];
    }
    int32_t* seq_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(rows + 1));
    if (!seq_of) return -2;
    for (int b = 0; b < num_seqs; ++b)
        for (int r = q_start[b]; r < q_start[b + 1]; ++r) seq_of[r] = b;
    int err = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads) reduction(| : err)
#endif
    {
        double* scratch = (double*)malloc(sizeof(double) * (2 * (size_t)head_dim + max_ctx + 1));
        if (!scratch) {
            err |= 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int i = 0; i < rows * num_q_heads; ++i) {
                int r = i / num_q_heads, h = i % num_q_heads, b = seq_of[r];
                int n = q_start[b + 1] - q_start[b];
                int pos = context_lens[b] - n + (r - q_start[b]);
                double* o = out + (int64_t)i * head_dim;
                /* attend_one reads row r of q (its `seq` argument) over pos + 1 tokens */
                if (attend_one(q, q_dtype, k_cache, v_cache,
                               block_tables + (int64_t)b * max_blocks_per_seq, max_blocks_per_seq,
                               pos + 1, scales, kv_dtype, num_blocks, o, softmax_scale,
                               num_q_heads, num_kv_heads, head_dim, block_size, r, h, scratch))
                    err |= 1;
            }
            free(scratch);
        }
    }
    free(seq_of);
    (void)num_threads;
    return err ? -1 : 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
