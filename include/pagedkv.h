/* pagedkv — paged, quantized KV cache for decode on GB300 (sm_103a).
 *
 * Two operations, as the PagedAttention pages state the problem:
 *   paged_kv_write          store each step's new K/V rows into their physical
 *                           block slots, quantizing on the way in;
 *   paged_decode_attention  one decode step of attention for every sequence,
 *                           reading K/V through a block table.
 *
 * Sources: "Reducing LLM Inference Latency: KV Cache Quantization and
 * PagedAttention in vLLM" (mohashari.github.io) — block pool, block table,
 * address translation (snippet-3), block-wise FP8 E4M3 scale and cast
 * (snippet-4); "KV Cache Compression & Paged Attention" (myaihardware.com),
 * "Implementation Details" — the kernel's inputs and its loop over logical
 * blocks; "Optimizing KV-Cache Memory Footprint" (publishertech.pages.dev),
 * section 4 — INT4 group-wise quantization; "KV Cache Optimization: 3x
 * Faster LLM Inference" (tildalice.io) — softmax(q K^T / sqrt(d)) V and GQA.
 *
 * Conventions shared by every call:
 *  - Every buffer is caller-owned DEVICE memory, 16-byte aligned.  The
 *    library allocates nothing and keeps no state between calls.
 *  - Calls are asynchronous on `stream` (a cudaStream_t, NULL = the legacy
 *    default stream) and never synchronize.  Host-visible argument errors
 *    return a nonzero pkv_status before anything is launched.
 *  - `dev_status` (optional, may be NULL) is one int in device memory.  A
 *    kernel that meets a block id or slot outside the pool ORs
 *    PKV_ERR_DEVICE_BOUNDS into it and skips that block or token; it never
 *    traps.  The caller reads it back whenever it likes.
 *  - Cache layout per KV tensor (K and V are separate buffers):
 *      [num_blocks][num_kv_heads][block_size][row], where a row holds one
 *      token of one head: head_dim 16-bit values (F16/BF16), head_dim FP8
 *      bytes (E4M3, E5M2) or int8 codes (INT8), or head_dim/2 bytes of 4-bit
 *      codes (INT4: element 2i in the low nibble of byte i, 2i+1 in the high
 *      nibble).
 *  - `scales` layout (index 0 of the leading 2 is K, 1 is V):
 *      FP8 (E4M3, E5M2) and INT8:  float [2][num_blocks][num_kv_heads] — one
 *            scale per block and KV head;
 *      INT4: half  [2][num_blocks][num_kv_heads][block_size][head_dim/32][2]
 *            — (scale, zero) per token, head and group of 32 elements;
 *      F16/BF16: unused (may be NULL).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_F16 = 0,       /* IEEE half */
    PKV_BF16 = 1,      /* bfloat16 */
    PKV_FP8_E4M3 = 2,  /* OCP E4M3 ("e4m3fn"), per-(block, kv-head) fp32 scale */
    PKV_INT4_G32 = 3,  /* asymmetric 4-bit, groups of 32 along head_dim, fp16 scale+zero */
    PKV_FP8_E5M2 = 4,  /* OCP E5M2, per-(block, kv-head) fp32 scale */
    PKV_INT8 = 5       /* symmetric int8 codes, per-(block, kv-head) fp32 scale */
} pkv_dtype;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,    /* NULL, negative size, misaligned pointer, Hq % Hkv != 0 */
    PKV_ERR_UNSUPPORTED = 2,    /* a shape or dtype combination this build has no kernel for */
    PKV_ERR_CUDA = 3,           /* a CUDA launch failed (see cudaGetLastError) */
    PKV_ERR_DEVICE_BOUNDS = 4,  /* written to *dev_status by a kernel, never returned */
    PKV_ERR_WORKSPACE = 5,      /* workspace missing or smaller than required */
    PKV_ERR_DEVICE_TIMEOUT = 8  /* ORed into *dev_status by a kernel whose wait for its own
                                   asynchronous work ran out (the launch then stops early
                                   and its outputs are undefined); never returned */
} pkv_status;

/* paged_kv_write — quantize-on-write of new K/V rows into their slots.
 *
 * k_new, v_new   [num_tokens][num_kv_heads][head_dim] in new_dtype (F16 or BF16).
 * slot_mapping   int64 [num_tokens]; slot = physical_block * block_size + offset
 *                (the block manager's address translation, snippet-3 of the
 *                mohashari page).  -1 skips the token; any other value outside
 *                [0, num_blocks * block_size) is skipped and flagged in dev_status.
 * k_cache, v_cache, scales   the pool, layouts above, updated in place.
 * kv_dtype       F16/BF16: a plain copy (new_dtype must equal kv_dtype).
 *                FP8_E4M3: one scale per block, KV head and K/V from the
 *                block's absolute maximum ("Block-Wise Scaling Factors",
 *                snippet-4 of the mohashari page).  A call that writes the
 *                slot at offset 0 of a block opens the block: its scales
 *                become max(amax / 448, 1e-12) in fp32, amax taken over every
 *                token this call writes into the block (a whole prefilled
 *                block is scaled by its own maximum).  A call that writes
 *                into a block without its offset-0 slot reuses the stored
 *                scales, and values beyond them saturate (the tokens still to
 *                come are unknown when a block opens).  code = E4M3 round-to-
 *                nearest-even with saturation to +-448 of the fp32 quotient
 *                x / scale.  The result does not depend on the order of the
 *                tokens within the call.  Stored scales must be non-negative
 *                (zeroed, or written by this library): the write uses the
 *                sign bit of an opened block's scale as a mark while it runs,
 *                as three launches (open, grow the maximum, encode).
 *                FP8_E5M2: the same with 57344 (the largest finite E5M2) in
 *                place of 448, codes rounded to nearest even and saturated.
 *                INT8: the same block-wise rule with 127: scale =
 *                max(amax / 127, 1e-12), code = clamp(rint(x / scale), -127,
 *                127) (fp32 quotient, round half to even), two's complement.
 *                INT4_G32: per token, head and 32-element group,
 *                scale = fp16(fp32(max - min) / 15), zero = fp16(min),
 *                code = clamp(rint((x - zero) / scale), 0, 15) in fp32 (0 when
 *                scale is 0).  head_dim must be a multiple of 32.
 * Supported: head_dim in {64, 128}, block_size a multiple of 16 up to 256.
 * Two tokens of one call must not target the same slot (the result would
 * depend on the order the GPU runs them in).
 */
int paged_kv_write(const void* k_new, const void* v_new, int new_dtype,
                   const int64_t* slot_mapping, int64_t num_tokens,
                   void* k_cache, void* v_cache, void* scales, int kv_dtype,
                   int num_blocks, int num_kv_heads, int head_dim, int block_size,
                   int* dev_status, void* stream);

/* paged_kv_copy_blocks — copy whole physical blocks within the pool
 * (copy-on-write and beam-search forks: "KV Cache Compression & Paged
 * Attention Deep Dive", myaihardware page, sections "PagedAttention:
 * Operating System-Inspired Memory Management for LLMs" and "Implementation
 * Details: PagedAttention Kernel and Page Table").  The block manager keeps
 * the reference counts and picks the pairs; this call moves the bytes.
 *
 * block_pairs    int32 [num_pairs][2] (src, dst), device memory.  For each
 *                pair, block dst of k_cache and v_cache (all KV heads) and its
 *                scales (FP8: the per-head K and V scales; INT4: every
 *                (scale, zero) pair of the block) become byte copies of block
 *                src's, so dst dequantizes to exactly what src did.  src == dst
 *                is a no-op; an id outside [0, num_blocks) skips the pair and
 *                flags PKV_ERR_DEVICE_BOUNDS in dev_status.  No block may be
 *                both a source and a destination in one call, and destinations
 *                must be distinct (otherwise the result depends on the order
 *                the GPU runs the pairs in).
 * k_cache, v_cache, scales, kv_dtype, num_blocks, num_kv_heads, head_dim,
 * block_size     the pool, as for paged_kv_write.
 * Host-visible errors as for paged_kv_write; 0 pairs is a no-op.
 */
int paged_kv_copy_blocks(void* k_cache, void* v_cache, void* scales, int kv_dtype,
                         const int32_t* block_pairs, int num_pairs, int num_blocks,
                         int num_kv_heads, int head_dim, int block_size, int* dev_status,
                         void* stream);

/* paged_decode_attention — one decode step over a paged, optionally
 * quantized KV cache (the PagedAttention kernel of the myaihardware page,
 * "Implementation Details": per head, walk the logical blocks, translate
 * each to its physical block, load K and V, score, softmax, weighted sum).
 *
 * q              [num_seqs][num_q_heads][head_dim] in q_dtype (F16 or BF16).
 * block_tables   int32 [num_seqs][max_blocks_per_seq]; entry j of row b is
 *                the physical block holding tokens [j*bs, (j+1)*bs) of b.
 * context_lens   int32 [num_seqs]; tokens to attend over, the new token
 *                included (write first, then attend).  0 gives out = 0.
 * out            [num_seqs][num_q_heads][head_dim] in q_dtype:
 *                out = sum_t softmax_t(softmax_scale * q.K_t) V_t, fp32
 *                accumulation, over K/V dequantized in registers.
 * GQA            query head h reads KV head h / (num_q_heads / num_kv_heads).
 * partition_size tokens per split-KV partition (multiple of 16), or 0 for
 *                the library's choice.  With more than one partition each
 *                partition writes a partial (max, sum, output) to `workspace`
 *                and a second kernel merges them by log-sum-exp.
 * workspace      device scratch of at least paged_decode_workspace_bytes(...)
 *                bytes (may be NULL when that is 0).
 * Work split: the library picks between CTAs whose warps share a partition
 * (merging their states), warps that each own a (partition, KV head) unit,
 * and the balanced split, in which one resident wave of warps takes equal
 * shares of all (sequence, KV head) pairs' tiles and the merge combines the
 * pieces (chosen where warp-owned units would be, for up to 512 sequences).
 * The environment variable PKV_DECODE_MODE=shared|warp|balanced, read on each
 * call, forces one (for testing; results agree to rounding).  The test
 * build of the library (libpagedkv_test.so, used by the tests only) also
 * takes PKV_DECODE_MODE=simt, a CUDA-core comparator of the same computation
 * (16-bit, FP8 and INT8 caches; kept to measure what the tensor cores buy),
 * and PKV_DECODE_MODE=tc, a comparator on the tcgen05 tensor cores with
 * tensor-memory accumulators (FP8 and INT8 caches with head_dim 128; slower
 * than the default kernel).  The product library holds neither.
 * Supported: head_dim in {64, 128}; num_q_heads / num_kv_heads <= 8;
 * block_size a multiple of 16 up to 256; F16/BF16 caches need q_dtype equal
 * to kv_dtype; FP8/INT4 caches take F16 or BF16 q; num_blocks * num_kv_heads
 * below 2^27 (PKV_ERR_UNSUPPORTED otherwise).
 */
int paged_decode_attention(const void* q, int q_dtype,
                           const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs,
                           const void* scales, int kv_dtype, int num_blocks,
                           void* out, float softmax_scale,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int partition_size, void* workspace, size_t workspace_bytes,
                           int* dev_status, void* stream);

/* paged_decode_attention_with_write — paged_kv_write of each sequence's new
 * token and paged_decode_attention in one launch (the quantize-on-write step
 * of the mohashari page's snippet-4 and the attention of the myaihardware
 * page's "Implementation Details", fused: the write launch and its re-read
 * disappear from the decode step).
 *
 * k_new, v_new   [num_seqs][num_kv_heads][head_dim] in q_dtype: the new token
 *                of each sequence (for F16/BF16 caches q_dtype must equal
 *                kv_dtype, as for paged_kv_write).
 * slot_mapping   int64 [num_seqs]: -1 (sequence b writes nothing), or the slot
 *                of position context_lens[b] - 1 of sequence b, i.e.
 *                block_tables[b][(ctx-1)/bs] * bs + (ctx-1) % bs.  Any other
 *                value is flagged (PKV_ERR_DEVICE_BOUNDS) and not written:
 *                only that position's row is read by the same CTA that
 *                writes it, which is what makes the fusion race-free.
 * Everything else as for paged_decode_attention; the cache and scales are
 * updated exactly as paged_kv_write would (encodings and FP8 scale rule
 * included) and the attention sees the written token.  Results are those of
 * paged_kv_write followed by paged_decode_attention with the same arguments.
 */
int paged_decode_attention_with_write(const void* q, int q_dtype, const void* k_new,
                                      const void* v_new, const int64_t* slot_mapping,
                                      void* k_cache, void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int num_seqs, void* scales,
                                      int kv_dtype, int num_blocks, void* out,
                                      float softmax_scale, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int partition_size,
                                      void* workspace, size_t workspace_bytes, int* dev_status,
                                      void* stream);

/* paged_prefill_attention — chunked-prefill attention over the paged cache:
 * each sequence brings a chunk of new query tokens whose K/V are already in
 * the cache (written with paged_kv_write), and each query attends causally
 * to every cached token up to its own position.  The pages pair
 * PagedAttention with chunked prefill (publishertech page, section 5,
 * "Production Benchmarks & Implementation"); the causal rule is the usual
 * prefill one.
 *
 * q              [q_start[num_seqs]][num_q_heads][head_dim] in q_dtype: the
 *                chunks of all sequences, back to back.
 * q_start        int32 [num_seqs + 1], device: sequence b's queries are rows
 *                q_start[b] .. q_start[b+1] - 1 (a chunk of n_b tokens).
 * max_query_len  sizes the grid; normally the largest n_b.  Queries
 *                j >= max_query_len of a chunk are not computed and their
 *                output rows are left untouched (positions still count from
 *                the whole chunk of n_b).
 * context_lens   int32 [num_seqs]: tokens in the cache, the chunk included.
 *                Query j of sequence b sits at position ctx_b - n_b + j and
 *                attends to tokens 0 .. ctx_b - n_b + j.  A chunk longer than
 *                its context is flagged (PKV_ERR_DEVICE_BOUNDS); its queries
 *                at negative positions give zeros.
 * out            [q_start[num_seqs]][num_q_heads][head_dim] in q_dtype.
 * Everything else as for paged_decode_attention (no workspace: no split-KV).
 * Supported: as paged_decode_attention, with num_q_heads / num_kv_heads in
 * {1, 2, 4, 8}.
 * Every cache dtype (head_dim 64 or 128) runs on the tcgen05 tensor cores
 * (accumulators in tensor memory; INT4 caches dequantized into hi + lo
 * operand pairs in the query's type, so with f16 queries their values must
 * lie in the f16 range); the waits on the tensor cores are bounded, and one
 * that runs out sets PKV_ERR_DEVICE_TIMEOUT in dev_status and leaves the
 * affected output rows zero.  The environment variable PKV_PREFILL_MODE=mma
 * (read on each call) selects the mma.sync kernel instead.  Both compute the
 * same definition.
 */
int paged_prefill_attention(const void* q, int q_dtype, const int32_t* q_start,
                            int max_query_len, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, const void* scales,
                            int kv_dtype, int num_blocks, void* out, float softmax_scale,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int* dev_status, void* stream);

/* paged_decode_attention_noalloc — paged_decode_attention without a
 * caller-supplied workspace, for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a convenience of this library.
 *
 * Some callers cannot call cudaMalloc at all: code running inside a custom
 * allocator's callbacks, processes whose device memory is one fixed pool
 * handed out up front, runtimes that forbid allocation on their hot path,
 * or plain C callers with no allocator at hand.  For them this variant takes
 * the split-KV scratch (the per-partition partial results) from one static
 * device array inside the library: 64 MiB on every GPU that loads the
 * library, held until the process exits.
 *
 * Arguments, layouts and results are those of paged_decode_attention, minus
 * workspace/workspace_bytes.  Requests whose scratch
 * (paged_decode_workspace_bytes(...)) exceeds 64 MiB return
 * PKV_ERR_WORKSPACE before anything is launched.  Each call looks up the
 * array's address (cudaGetSymbolAddress) in the current device's context;
 * the first call on a device also loads the library's module there, so make
 * that first call before any stream capture.  Every
 * call shares the one array, so calls that overlap on the GPU (other
 * streams, other host threads) race on it: serialize them.
 */
int paged_decode_attention_noalloc(const void* q, int q_dtype,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs,
                                   const void* scales, int kv_dtype, int num_blocks,
                                   void* out, float softmax_scale,
                                   int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int partition_size,
                                   int* dev_status, void* stream);

/* Partition size paged_decode_attention will use for these arguments
 * (resolves partition_size == 0); 0 if the arguments are invalid. */
int paged_decode_partition_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                int max_blocks_per_seq, int block_size, int partition_size);

/* Workspace bytes paged_decode_attention needs for these arguments (0 when
 * every sequence fits one partition, and 0 for arguments the calls reject,
 * e.g. more than 2^40 split-KV partial rows). */
size_t paged_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int max_blocks_per_seq, int block_size,
                                    int partition_size);

/* Human-readable name of a pkv_status value. */
const char* paged_kv_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int paged_kv_version(void);

#ifdef __cplusplus
}
#endif
#endif
