/* CPU oracle for paged, quantized KV-cache decode attention and the
 * quantize-on-write.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg are the only callers.  It shares no
 * code with the CUDA library.
 *
 * Plain, slow and obviously correct: fp64 attention by the softmax
 * definition over K/V dequantized with the formats' definitions; the write
 * follows the stated encoding rules step by step in fp32 where the rule
 * says so (the precision the encoded integer is decided in).
 *
 * dtype tags: 0 = f16, 1 = bf16, 2 = FP8 E4M3 (per-(block, kv-head) fp32
 * scale), 3 = INT4 group-32 (fp16 scale + zero per token, head and group),
 * 4 = FP8 E5M2 (scaled like E4M3), 5 = INT8 (symmetric codes, scaled like
 * E4M3 with 127 in place of 448).
 * Layouts are those of the library (documented in oracle.c).
 */
#ifndef PKV_ORACLE_H
#define PKV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* format codecs */
double oracle_f16_to_double(uint16_t bits);
double oracle_bf16_to_double(uint16_t bits);
uint16_t oracle_f32_to_f16_rne(float x);
double oracle_e4m3_to_double(uint8_t code);
uint8_t oracle_e4m3_encode(float y);
double oracle_e5m2_to_double(uint8_t code);
uint8_t oracle_e5m2_encode(float y);
int8_t oracle_int8_encode(float y);

/* sizing formulas */
double oracle_kv_cache_bytes(double layers, double heads, double head_dim, double seq_len,
                             double batch, double bytes_per_elem);
int64_t oracle_num_pages(int64_t tokens, int64_t page_size);
int oracle_physical_address(const int32_t* table_row, int num_entries, int block_size,
                            int64_t token_index, int32_t* physical_block, int32_t* offset);

/* the write: 0 on success, negative on a bad argument */
int oracle_kv_write(const uint16_t* k_new, const uint16_t* v_new, int new_dtype,
                    const int64_t* slot_mapping, int64_t num_tokens,
                    void* k_cache, void* v_cache, void* scales, int kv_dtype,
                    int num_blocks, int num_kv_heads, int head_dim, int block_size);

/* whole-block copies (src, dst) pairs [num_pairs][2]: the number of pairs
 * skipped for an out-of-range id, negative on a bad argument */
int oracle_copy_blocks(void* k_cache, void* v_cache, void* scales, int kv_dtype,
                       const int32_t* pairs, int num_pairs, int num_blocks, int num_kv_heads,
                       int head_dim, int block_size);

/* decode attention into fp64 out [num_seqs, num_q_heads, head_dim] */
int oracle_decode_attention(const uint16_t* q, int q_dtype,
                            const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs,
                            const void* scales, int kv_dtype, int num_blocks,
                            double* out, double softmax_scale,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int num_threads);

/* the same over a subset of (sequence, q-head) pairs; out [n_pairs, head_dim] */
int oracle_decode_attention_pairs(const uint16_t* q, int q_dtype,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int num_seqs,
                                  const void* scales, int kv_dtype, int num_blocks,
                                  double* out, double softmax_scale,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, const int32_t* pair_seq,
                                  const int32_t* pair_head, int n_pairs, int num_threads);

/* chunked prefill: out fp64 [q_start[num_seqs], num_q_heads, head_dim] */
int oracle_prefill_attention(const uint16_t* q, int q_dtype, const int32_t* q_start,
                             const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, int num_seqs, const void* scales,
                             int kv_dtype, int num_blocks, double* out, double softmax_scale,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_threads);

/* dequantized K or V row of one token/head (fp64) */
int oracle_dequant_row(const void* cache, const void* scales, int which_kv, int kv_dtype,
                       int num_blocks, int num_kv_heads, int head_dim, int block_size,
                       int32_t block, int kv_head, int offset, double* row);

int oracle_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
