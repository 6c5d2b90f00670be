// Chunked-prefill attention on the tcgen05 tensor cores, with warp roles,
// for 16-bit caches (F16, BF16), one-byte caches (FP8 E4M3 / E5M2, INT8; one
// fp32 scale per block and KV head) and INT4 caches (groups of 32 along
// head_dim with an fp16 scale and zero point per token).  Chunked prefill is a dense
// contraction (every cached token meets a whole chunk of queries), unlike the
// decode step, so it runs where the dense tensor throughput is: "Optimizing
// KV-Cache Memory Footprint in High-Throughput LLM Serving", section 5, pairs
// PagedAttention with GQA and chunked prefill; query j of a chunk of n over c
// cached tokens sits at position c - n + j and sees tokens 0 .. c - n + j.
//
// One CTA per SM (320 threads, 384 for one-byte and INT4 caches; all 512
// tensor-memory columns) takes two adjacent Q tiles of 128 query rows each --
// 128/G query tokens of one sequence times the G query heads of one KV head
// per tile -- and walks that KV head's cache in 128-token tiles (INT4: 64),
// K and V of a tile shared by both Q tiles:
//  * load warp (warp 9, 16-bit caches): looks up the tile's eight 16-token
//    pieces in the block table and brings K and V into rings of two (head_dim
//    64: three) stages with TMA tensor copies (a 16 x 64 box per piece and
//    128-byte column block, 128-byte swizzle), signalled on mbarriers by byte
//    count.  The piece that straddles the end of the range has its V rows
//    copied by the warp's lanes instead, with the rows past the end
//    zero-filled, so that P = 0 never meets a non-finite value from an
//    unwritten slot; a piece in an out-of-range block reads as zeros and is
//    flagged (the softmax leaves it out);
//  * load warps (warps 9-11, one-byte caches): bring the codes with 16-byte
//    loads through the block table and convert them exactly to f16 operands
//    in the same layouts (E4M3 / E5M2 by cvt, INT8 as 1024 + (x + 128) -
//    1152), zeros past the range or in an out-of-range block;
//  * load warps (warps 9-11, INT4 caches, 64-token tiles): dequantize each
//    element once, x = scale n + zero in fp32, into a hi + lo pair of the
//    query's 16-bit type, written to a hi and a lo operand tile; S sums the
//    products with both, O takes P_hi V_hi + P_lo V_hi + P_hi V_lo;
//  * MMA warp (warp 8, one lane): S_A = Q_A K^T, then O_B += P_B V of the
//    previous tile, then S_B = Q_B K^T, then O_A += P_A V, so that each
//    softmax warpgroup works while the tensor cores serve the other tile;
//    each batch is committed to an mbarrier.  Products of N = 128 (S over
//    128 tokens, O over head_dim 128) keep the tensor cores' work per
//    instruction large;
//  * softmax warpgroups (warps 0-3: tile A, 4-7: tile B): thread r reads row
//    r of S from tensor memory, applies the causal mask and the online
//    softmax (the row max over a tree of three-input max instructions; the
//    running max raised lazily, by more than 2^8 only, O rescaled in tensor
//    memory when it is), writes row r of P as a 16-bit hi + lo pair
//    over S's own columns and signals the MMA warp.  The tensor cores run a
//    thread's products in issue order, so S(t + 1), issued after P V(t),
//    overwrites P(t) only after that product has read it.
// One-byte caches also: bf16 queries enter as f16 times a power of two per
// row (exact for every value above 2^-28 of the row's largest), taken off in
// the softmax multiplier; each token's K block scale multiplies its score
// column; its V block scale enters P as vs / vu, vu the largest V scale of the
// CTA's blocks (found by the softmax threads while tile 0 loads), so
// P'' = p vs / vu <= p and the output is O / l times vu.
// Shared-memory operands use the canonical 128-byte-swizzle layouts: Q and K
// K-major (rows of 128 bytes, 8-row atoms 1024 bytes apart, the second half
// of head_dim 128 in its own region), V MN-major (token rows of 128 bytes, 8
// tokens per atom, the two 64-value halves of head_dim 128 one region apart).
// Every wait is bounded and also ends when another role has given up: the
// launch then ORs PKV_ERR_DEVICE_TIMEOUT into dev_status, waits (bounded) for
// its own copies and products in flight, writes zeros and frees its tensor
// memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>

#include "pagedkv.h"
#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {
using namespace tc;

constexpr int kWsRows = 128;                         // query rows per Q tile (the MMA M)
constexpr int kWsPiece = 16;                         // tokens per TMA box
constexpr int kWsMmaWarp = 8;
constexpr int kWsLoadWarp = 9;                       // the first load warp

// The warps of a cache dtype: 0-7 softmax, 8 MMA, then the load warps: one
// issuing TMA copies for 16-bit caches, three that load and convert the codes
// for one-byte and INT4 caches (12 warps still leave 168 registers per
// thread).  INT4 caches dequantize into hi + lo operand pairs, which double
// the K and V tiles, so they walk the cache in 64-token tiles.
template <int KV> struct WsRoles {
  static constexpr bool kB8 = is_blk8(KV);
  static constexpr bool kI4 = KV == PKV_INT4_G32;
  static constexpr bool kConvert = kB8 || kI4;     // load warps convert the codes
  static constexpr int kLoadWarps = kConvert ? 3 : 1;
  static constexpr int kThreads = (kWsLoadWarp + kLoadWarps) * kWarp;
  static constexpr int kTok = kI4 ? 64 : 128;       // KV tokens per tile
  static constexpr int kPieces = kTok / kWsPiece;
  static constexpr int kParts = kI4 ? 2 : 1;        // operand tiles per K or V stage (hi, lo)
};
constexpr float kWsTau = 8.f;                        // lazy rescale threshold (log2 units)
constexpr int kWsBoxBytes = kWsPiece * 128;          // one box: 16 rows of 128 bytes

// Shared memory (operand regions 1024-byte aligned; V first, so that every
// operand address stays low in the CTA's window) and tensor memory: Q tile i
// owns columns [256 i, 256 i + 256): S [0, 128), overwritten by P (tokens
// 32c .. 32c + 31: hi at columns 32c .. 32c + 15, lo at 32c + 16 .. 32c + 31),
// and O [128, 128 + D).
template <int D, int KV> struct WsPlan {
  using R = WsRoles<KV>;
  static constexpr int kHalves = D / 64;             // 128-byte column blocks per row
  static_assert(kHalves == 1 || kHalves == 2, "head_dim 64 or 128");
  static constexpr int kStages = D == 128 ? 2 : 3;
  static constexpr int kTileBytes = R::kTok * D * 2;  // one K or V operand tile
  static constexpr int kStageBytes = R::kParts * kTileBytes;
  static constexpr int kKvHalf = R::kTok * 128;      // one column block of an operand tile
  static constexpr int kQBytes = kWsRows * D * 2;
  static constexpr int kQHalf = kWsRows * 128;
  static constexpr int kOffV = 0;
  static constexpr int kOffK = kOffV + kStages * kStageBytes;
  static constexpr int kOffQ = kOffK + kStages * kStageBytes;
  static constexpr int kOffBar = kOffQ + 2 * kQBytes;
  // mbarriers: k_full, v_full, k_empty, v_empty per stage; q_full; s_full,
  // p_full, o_done per Q tile; final.  Then the tensor-memory address and the
  // abort flag.
  static constexpr int kBarKFull = 0, kBarVFull = kStages, kBarKEmpty = 2 * kStages;
  static constexpr int kBarVEmpty = 3 * kStages;
  static constexpr int kBarQ = 4 * kStages, kBarSFull = kBarQ + 1;
  static constexpr int kBarPFull = kBarSFull + 2, kBarODone = kBarPFull + 2;
  static constexpr int kBarFinal = kBarODone + 2, kNumBars = kBarFinal + 1;
  static constexpr int kOffSlot = kOffBar + 8 * kNumBars;
  // one-byte caches: each softmax warp's largest V scale over the CTA's blocks
  static constexpr int kOffVu = kOffSlot + 16;
  static constexpr int kSmem = kOffVu + 8 * 4;
  // one CTA per SM: it takes all of tensor memory, so the request is at least
  // half of shared memory
  static constexpr int kSmemRequest = kSmem > 120 * 1024 ? kSmem : 120 * 1024;
  static_assert(kSmemRequest <= 232448, "shared memory");
  static constexpr uint32_t kTmemCols = 512;
};

struct WsParams {
  CUtensorMap tmap_k;          // 16-bit caches: [num_blocks * Hkv][block_size][D] values
  CUtensorMap tmap_v;
  const uint16_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* scales;         // one-byte caches: fp32 [2][num_blocks][num_kv_heads]
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* q_start;
  void* out;
  int* dev_status;
  int max_query_len;
  int max_blocks_per_seq;
  int num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int block_size;
  float softmax_scale;
#ifdef PKV_TEST_HOOKS
  int test_drop_commit;        // test of the bounded waits: tile A's first S is not committed
#endif
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// an arrival once this thread's earlier cp.async copies have landed (the
// barrier's expected count includes it)
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// one box of a 3-D tensor map into shared memory, completing bytes on `bar`
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Shared-memory descriptor of a 128-byte-swizzled operand: start address,
// leading byte offset (MN-major: the next 64-value column block; unused for
// K-major), stride byte offset 1024 (the next 8-row atom), version bit 46,
// layout type 2 (128-byte swizzle) at bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// OR of `pred` over the eight softmax warps (named barrier 1, 256 threads);
// the barrier also orders their shared-memory stores before it.
__device__ __forceinline__ bool softmax_bar_or(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out) : "r"(pred ? 1u : 0u) : "memory");
  return out != 0;
}

// Bounded wait for phase `parity` that also ends when another role has set
// the abort flag; a wait that runs out flags the timeout and sets the flag.
__device__ __forceinline__ bool ws_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        int* dev_status) {
  const long long start = clock64();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 15) == 15 && *abort_flag) return false;
    if (clock64() - start > kWaitCycles) {
      flag_status(dev_status, PKV_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}
// Bounded wait that ignores the abort flag (the clean-up waits for work in
// flight); running out flags the timeout and the abort.
__device__ __forceinline__ void ws_drain(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* dev_status) {
  if (!mbar_wait(bar, parity)) {
    flag_status(dev_status, PKV_ERR_DEVICE_TIMEOUT);
    *abort_flag = 1;
  }
}

// 128 consecutive fp32 columns of this thread's tensor-memory lane in one
// load, and its wait (the registers are defined only after both)
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
        "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
        "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
        "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
        "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
        "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns, likewise
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
template <int N>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, float (&v)[N]) {
  if constexpr (N == 128) tmem_ld128(taddr, v);
  else tmem_ld64(taddr, v);
}

// Scores of the 16-token pieces flagged in `bad` (bit j: piece j; the same
// for the whole warp) set to -inf.
template <int N>
__device__ __forceinline__ void mask_pieces(float (&s)[N], uint32_t bad) {
  if (bad == 0) return;
#pragma unroll
  for (int j = 0; j < N / kWsPiece; ++j)
    if ((bad >> j) & 1u) {
#pragma unroll
      for (int c = 0; c < kWsPiece; ++c) s[kWsPiece * j + c] = -INFINITY;
    }
}

// Three-input max and min (sm_100 and later): a row's 128 values reduce in
// 65 instructions over a tree of depth 5 instead of 127 over depth 7.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
template <bool kMin, int N>
__device__ __forceinline__ float tree_reduce3(const float (&v)[N]) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    constexpr int M = (N + 2) / 3;
    float w[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
      if (3 * i + 2 < N)
        w[i] = kMin ? fmin3(v[3 * i], v[3 * i + 1], v[3 * i + 2]) : fmax3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
      else if (3 * i + 1 < N)
        w[i] = kMin ? fminf(v[3 * i], v[3 * i + 1]) : fmaxf(v[3 * i], v[3 * i + 1]);
      else
        w[i] = v[3 * i];
    }
    return tree_reduce3<kMin, M>(w);
  }
}
// The largest of a row's N scores, and the largest of their negations, as
// trees of three-input instructions (log3 N dependent steps instead of N)
template <int N>
__device__ __forceinline__ float row_max(const float (&s)[N]) {
  return tree_reduce3<false, N>(s);
}
template <int N>
__device__ __forceinline__ float row_max_neg(const float (&s)[N]) {
  return -tree_reduce3<true, N>(s);
}

// KV: the cache dtype; QT: the query dtype; the operands of the products are
// QT for 16-bit caches and f16 for one-byte caches (codes converted exactly,
// bf16 q as f16 times a power of two per row).
template <int KV, int QT, int D>
__global__ void __launch_bounds__(WsRoles<KV>::kThreads, 1)
prefill_ws_kernel(const __grid_constant__ WsParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using PL = WsPlan<D, KV>;
  using R = WsRoles<KV>;
  constexpr bool kB8 = R::kB8, kI4 = R::kI4;
  constexpr int kWsKv = R::kTok, kWsPieces = R::kPieces;
  constexpr int OT = kB8 ? PKV_F16 : QT;               // operand type of the products
  constexpr int S = PL::kStages;
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int group = p.num_q_heads / p.num_kv_heads;
  const int qpb = kWsRows / group;                     // query tokens per Q tile
  const int nq = p.q_start[b + 1] - p.q_start[b];
  const int nqc = min(nq, p.max_query_len);            // queries computed
  const int j0 = static_cast<int>(blockIdx.x) * 2 * qpb;   // tile A's first query, B's: j0 + qpb
  if (j0 >= nqc) return;                                // whole CTA: no query here
  const int cap = p.max_blocks_per_seq * p.block_size;
  int ctx = p.context_lens[b];
  if (ctx > cap) {
    if (tid == 0 && blockIdx.x == 0 && kvh == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
    ctx = cap;
  }
  const int pos0 = ctx - nq;                           // position of query 0 of the chunk
  if (pos0 < 0 && j0 == 0 && tid == 0 && kvh == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
  const int last_j = min(j0 + 2 * qpb, nqc) - 1;
  const int kv_end = max(0, min(ctx, pos0 + last_j + 1));  // tokens any row of the CTA sees
  const int nt = (kv_end + kWsKv - 1) / kWsKv;

  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + PL::kOffBar + 8 * i; };
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + PL::kOffSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + PL::kOffSlot + 4);

  if (warp == kWsMmaWarp) {
    tmem_alloc(sb + PL::kOffSlot, PL::kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      // 16-bit: the TMA bytes (and, for V, the load warp's lanes); one-byte:
      // one arrival per load warp
      mbar_init(bar(PL::kBarKFull + s), R::kConvert ? R::kLoadWarps : 1);
      mbar_init(bar(PL::kBarVFull + s), R::kConvert ? R::kLoadWarps : 1 + kWarp);
      mbar_init(bar(PL::kBarKEmpty + s), 1);
      mbar_init(bar(PL::kBarVEmpty + s), 1);
    }
    mbar_init(bar(PL::kBarQ), 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(PL::kBarSFull + i), 1);
      mbar_init(bar(PL::kBarPFull + i), 4);
      mbar_init(bar(PL::kBarODone + i), 1);
    }
    mbar_init(bar(PL::kBarFinal), 1);
    mbar_init_fence();
    *abort_flag = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int64_t per_kv = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads;

  // softmax rows: warpgroup i = warp / 4 owns Q tile i, thread r its row r =
  // query token ji + r / G, head r % G
  const int qt = warp >> 2, r = tid & 127;
  const int ji = j0 + qt * qpb;
  const int jj = r / group, g = r % group;
  const bool row_q = warp < 8 && ji + jj < nqc;
  const int pos = pos0 + ji + jj;
  const bool row_ok = row_q && pos >= 0;
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  const uint32_t t_s = tmem + lane_base + 256 * qt;    // S and P; O at + 128
  float l = 0.f;
  float vu = 1.f;                                      // one-byte caches: the V scale unit

  if (warp < 8) {
    // ------------------------------------------------------------ softmax
    float qexp = 1.f;                                    // one-byte caches: q's row scale undone
    {
      // Q row r of tile qt (128-byte swizzle; zeros for rows without a query)
      const uint16_t* qrow =
          p.q + ((static_cast<int64_t>(p.q_start[b]) + ji + (row_q ? jj : 0)) * p.num_q_heads +
                 kvh * group + g) * D;
      const uint32_t qbase = sb + PL::kOffQ + qt * PL::kQBytes + r * 128;
      if constexpr (!kB8) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint32_t dst = qbase + (c >> 3) * PL::kQHalf + (((c & 7) ^ (r & 7)) << 4);
          if (row_ok) cp_async_16(dst, qrow + 8 * c);
          else st_shared_v4(dst, make_uint4(0, 0, 0, 0));
        }
        cp_async_wait_all();
      } else {
        // f16 operands: a bf16 row enters as f16 times 2^e, e putting its
        // largest magnitude in [2^13, 2^14) (exact for every value above 2^-28
        // of it); qexp = 2^-e goes into the softmax multiplier
        uint4 w[D / 8];
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
          w[c] = row_ok ? __ldg(reinterpret_cast<const uint4*>(qrow) + c) : make_uint4(0, 0, 0, 0);
        float scale = 1.f;
        if constexpr (QT == PKV_BF16) {
          float qmax = 0.f;
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            const uint32_t ww[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = Half16<PKV_BF16>::unpack(ww[k]);
              qmax = fmaxf(qmax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
          if (qmax > 0.f) {
            int ex;
            frexpf(qmax, &ex);                            // qmax in [2^(ex-1), 2^ex)
            scale = ldexpf(1.f, 14 - ex);
            qexp = ldexpf(1.f, ex - 14);
          }
        }
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          uint4 h = w[c];
          if constexpr (QT == PKV_BF16) {
            const uint32_t ww[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
            uint32_t hh[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = Half16<PKV_BF16>::unpack(ww[k]);
              hh[k] = Half16<PKV_F16>::pack_rn(f.x * scale, f.y * scale);
            }
            h = make_uint4(hh[0], hh[1], hh[2], hh[3]);
          }
          st_shared_v4(qbase + (c >> 3) * PL::kQHalf + (((c & 7) ^ (r & 7)) << 4), h);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(PL::kBarQ));
    }
    const float mult = p.softmax_scale * 1.4426950408889634f * qexp;
    const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
    // While tile 0's loads and S product run, the 256 softmax threads scan the
    // CTA's blocks: whether any is out of the pool (then each tile's pieces are
    // looked up; a table of valid ids costs the tiles nothing) and, for
    // one-byte caches, the largest V scale vu (V scales enter P as vs / vu <= 1;
    // a range without written V blocks: vu 1).
    bool any_bad;
    {
      const int nblk = (kv_end + p.block_size - 1) / p.block_size;
      bool bad_here = false;
      float vmax = 0.f;
      for (int i = tid; i < nblk; i += 256) {
        const int phys = __ldg(trow + i);
        const bool bad = phys < 0 || phys >= p.num_blocks;
        bad_here |= bad;
        if (kB8 && !bad)
          vmax = fmaxf(vmax, __ldg(p.scales + per_kv + static_cast<int64_t>(phys) * p.num_kv_heads + kvh));
      }
      if constexpr (kB8) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        if (lane == 0) reinterpret_cast<float*>(smem + PL::kOffVu)[warp] = vmax;
      }
      any_bad = softmax_bar_or(bad_here);
      if constexpr (kB8) {
        vmax = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) vmax = fmaxf(vmax, reinterpret_cast<const float*>(smem + PL::kOffVu)[w]);
        if (vmax > 0.f) vu = vmax;
      }
    }
    const float inv_vu = 1.f / vu;
    float m = -INFINITY;
#pragma unroll 1
    for (int t = 0; t < nt; ++t) {
      const int t0 = t * kWsKv;
      // the tile's 16-token pieces in an out-of-range block (bit j: piece j),
      // which take no part (the load warp reads them as zeros and flags them)
      // One-byte caches: lane j < 8 also takes piece j's K scale and V scale / vu.
      uint32_t bad = 0;
      float pk = 0.f, pv = 0.f;
      if (kB8 || any_bad) {
        const int tok = t0 + lane * kWsPiece;
        bool bb = false;
        if (lane < kWsPieces && tok < kv_end) {
          const int phys = __ldg(trow + tok / p.block_size);
          bb = phys < 0 || phys >= p.num_blocks;
          if (kB8 && !bb) {
            const int64_t idx = static_cast<int64_t>(phys) * p.num_kv_heads + kvh;
            pk = __ldg(p.scales + idx);
            pv = __ldg(p.scales + per_kv + idx) * inv_vu;
          }
        }
        bad = __ballot_sync(0xffffffffu, bb);
      }
      // 1. row r of S_qt(t)
      bool ok = ws_wait(bar(PL::kBarSFull + qt), t & 1, abort_flag, p.dev_status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      // 2. row r of S in registers (one load of all 128 columns), scaled to
      //    log2 units and masked where needed (tiles below the range end and
      //    below every row's causal limit need no mask; the scale then goes
      //    into the exponent's fma), and its largest value
      float sv[kWsKv];
      tmem_ld_row<kWsKv>(t_s, sv);
      const bool full = t0 + kWsKv <= kv_end && t0 + kWsKv - 1 <= pos0 + ji && bad == 0;
      float tmax, pmul;
      if constexpr (kB8) {
        // each piece's column of scores times its K scale and this row's
        // multiplier
#pragma unroll
        for (int j = 0; j < kWsPieces; ++j) {
          const float kj = __shfl_sync(0xffffffffu, pk, j) * mult;
          const uint64_t k2 = f2_pack(kj, kj);
#pragma unroll
          for (int c = 0; c < kWsPiece; c += 2) {
            const float2 x = f2_unpack(f2_mul(f2_pack(sv[kWsPiece * j + c], sv[kWsPiece * j + c + 1]), k2));
            sv[kWsPiece * j + c] = x.x;
            sv[kWsPiece * j + c + 1] = x.y;
          }
        }
        if (!full) {
#pragma unroll
          for (int c = 0; c < kWsKv; ++c) {
            const int abs_t = t0 + c;
            const bool valid = abs_t < kv_end && (!row_ok || abs_t <= pos);
            if (!valid) sv[c] = -INFINITY;
          }
          mask_pieces(sv, bad);
        }
        tmax = row_max(sv);
        pmul = 1.f;
      } else if (full) {
        // (a negative scale turns the row's smallest score into its largest)
        tmax = (mult >= 0.f ? row_max(sv) : -row_max_neg(sv)) * mult;
        pmul = mult;
      } else {
#pragma unroll
        for (int c = 0; c < kWsKv; ++c) {
          const int abs_t = t0 + c;
          const bool valid = abs_t < kv_end && (!row_ok || abs_t <= pos);
          sv[c] = valid ? sv[c] * mult : -INFINITY;
        }
        mask_pieces(sv, bad);
        tmax = row_max(sv);
        pmul = 1.f;
      }
      // 3. online softmax; the running max moves only past m + tau
      const bool raise = tmax > m + kWsTau;
      float alpha = 1.f;
      if (raise) {
        const float mn = fmaxf(m, tmax);
        alpha = ex2_ftz(m - mn);
        m = mn;
        l *= alpha;
      }
      // 4. P = 2^(s - m) as a 16-bit hi + lo pair over row r's S columns
      //    (two tokens per 32-bit column; tokens 32c .. 32c + 31: hi at
      //    columns 32c .. 32c + 15, lo at 32c + 16 .. 32c + 31); exponent
      //    arguments, the lo parts and the row sum on packed fp32 pairs, the
      //    sum in two interleaved chains
      //    One-byte caches: the pair is of P'' = p vs / vu (the token's V
      //    scale over the range's largest), and the row sum stays in p.
      const uint64_t pm2 = f2_pack(pmul, pmul), nm2 = f2_pack(-m, -m);
      uint64_t lsum[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int c8 = 0; c8 < kWsKv / 8; ++c8) {
        uint32_t hw[4], lw[4];
        const float vr = kB8 ? __shfl_sync(0xffffffffu, pv, c8 >> 1) : 1.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = 8 * c8 + 2 * k;
          const float2 x = f2_unpack(f2_fma(f2_pack(sv[i], sv[i + 1]), pm2, nm2));
          uint64_t pp = f2_pack(ex2_ftz(x.x), ex2_ftz(x.y));
          lsum[k & 1] = f2_add(lsum[k & 1], pp);
          if constexpr (kB8) pp = f2_mul(pp, f2_pack(vr, vr));
          const float2 pf = f2_unpack(pp);
          hw[k] = Half16<OT>::pack_rn(pf.x, pf.y);
          const float2 f = Half16<OT>::unpack(hw[k]);
          const float2 d = f2_unpack(f2_sub(pp, f2_pack(f.x, f.y)));
          lw[k] = Half16<OT>::pack_rn(d.x, d.y);
        }
        // tokens 8 c8 .. 8 c8 + 7: chunk c8 / 4 of 32 tokens, its 4-column group c8 % 4
        const uint32_t col = 32 * (c8 >> 2) + 4 * (c8 & 3);
        tmem_st4(t_s + col, hw[0], hw[1], hw[2], hw[3]);
        tmem_st4(t_s + col + 16, lw[0], lw[1], lw[2], lw[3]);
      }
      {
        const float2 a = f2_unpack(lsum[0]), c = f2_unpack(lsum[1]);
        l += (a.x + a.y) + (c.x + c.y);
      }
      // 5. O rescaled when the max rose, once the previous P V of this tile
      //    has finished with it (S(t) was computed after it, so it has)
      if (t > 0) {
        ok = ws_wait(bar(PL::kBarODone + qt), (t - 1) & 1, abort_flag, p.dev_status);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, raise)) {           // warp-collective
#pragma unroll
          for (int k = 0; k < D / 32; ++k) {
            float o[32];
            tmem_ld32(t_s + 128 + 32 * k, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(t_s + 128 + 32 * k, o);
          }
        }
      }
      tmem_store_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(PL::kBarPFull + qt));
    }
    // the last P V
    if (nt > 0) ws_wait(bar(PL::kBarODone + qt), (nt - 1) & 1, abort_flag, p.dev_status);
  } else if (warp == kWsMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr bool kBf = OT == PKV_BF16;
      constexpr uint32_t kIdescS = umma_idesc(kBf, kWsRows, kWsKv, false);
      constexpr uint32_t kIdescO = umma_idesc(kBf, kWsRows, D, true);
      // S_i = Q_i K^T over head_dim in steps of 16 (32 bytes inside a
      // 128-byte swizzle row; the second column block in its own region)
      // (INT4: K as its hi and then its lo operand tile, one sum)
      auto issue_s = [&](int i, int st) {
        const uint32_t qb = sb + PL::kOffQ + i * PL::kQBytes;
#pragma unroll
        for (int part = 0; part < R::kParts; ++part) {
          const uint32_t kb = sb + PL::kOffK + st * PL::kStageBytes + part * PL::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk & 3) * 32;
            umma(tmem + 256 * i, sw128_desc(qb + (kk >> 2) * PL::kQHalf + off, 16),
                 sw128_desc(kb + (kk >> 2) * PL::kKvHalf + off, 16), kIdescS, part > 0 || kk > 0);
          }
        }
      };
      // O_i += P_i V: 16 tokens per product (two 8-token atoms of V, 8
      // tensor-memory columns of P: tokens 16kk .. sit at column
      // 32 (kk / 2) + 8 (kk % 2), their lo parts 16 columns on), the hi part
      // and then the lo part
      // (INT4: P hi V hi, P lo V hi, P hi V lo)
      auto issue_pv = [&](int i, int st, bool acc) {
        const uint32_t vb = sb + PL::kOffV + st * PL::kStageBytes;
        const uint32_t o = tmem + 256 * i + 128;
#pragma unroll
        for (int kk = 0; kk < kWsKv / 16; ++kk)
          umma_ts(o, tmem + 256 * i + 32 * (kk >> 1) + 8 * (kk & 1),
                  sw128_desc(vb + kk * 2048, PL::kKvHalf), kIdescO, acc || kk > 0);
#pragma unroll
        for (int kk = 0; kk < kWsKv / 16; ++kk)
          umma_ts(o, tmem + 256 * i + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                  sw128_desc(vb + kk * 2048, PL::kKvHalf), kIdescO, 1u);
        if constexpr (kI4) {
#pragma unroll
          for (int kk = 0; kk < kWsKv / 16; ++kk)
            umma_ts(o, tmem + 256 * i + 32 * (kk >> 1) + 8 * (kk & 1),
                    sw128_desc(vb + PL::kTileBytes + kk * 2048, PL::kKvHalf), kIdescO, 1u);
        }
      };
      bool ok = nt == 0 || ws_wait(bar(PL::kBarQ), 0, abort_flag, p.dev_status);
#pragma unroll 1
      for (int t = 0; ok && t < nt; ++t) {
        const int st = t % S;
        const uint32_t ph = (t / S) & 1;
        const int prev = (t + S - 1) % S;
        // S_A(t) (over P_A(t - 1), whose product was issued before)
        if (!ws_wait(bar(PL::kBarKFull + st), ph, abort_flag, p.dev_status)) break;
        tc_fence_after();
        issue_s(0, st);
#ifdef PKV_TEST_HOOKS
        // (the test build's check of the bounded waits leaves the first S_A
        // uncommitted: tile A's wait for it runs out)
        if (!(p.test_drop_commit && t == 0)) umma_commit(bar(PL::kBarSFull + 0));
#else
        umma_commit(bar(PL::kBarSFull + 0));
#endif
        // O_B += P_B V(t - 1); then V of tile t - 1 is free
        if (t > 0) {
          if (!ws_wait(bar(PL::kBarPFull + 1), (t - 1) & 1, abort_flag, p.dev_status)) break;
          tc_fence_after();
          issue_pv(1, prev, t > 1);
          umma_commit(bar(PL::kBarODone + 1));
          umma_commit(bar(PL::kBarVEmpty + prev));
        }
        // S_B(t) (over P_B(t - 1)); then K of tile t is free
        issue_s(1, st);
        umma_commit(bar(PL::kBarSFull + 1));
        umma_commit(bar(PL::kBarKEmpty + st));
        // O_A += P_A V(t) (rows the load warp wrote itself: visible to the
        // tensor cores after the proxy fence)
        if (!ws_wait(bar(PL::kBarVFull + st), ph, abort_flag, p.dev_status)) break;
        fence_proxy_async_smem();
        if (!ws_wait(bar(PL::kBarPFull + 0), t & 1, abort_flag, p.dev_status)) break;
        tc_fence_after();
        issue_pv(0, st, t > 0);
        umma_commit(bar(PL::kBarODone + 0));
        if (t == nt - 1) {
          if (!ws_wait(bar(PL::kBarPFull + 1), t & 1, abort_flag, p.dev_status)) break;
          tc_fence_after();
          issue_pv(1, st, t > 0);
          umma_commit(bar(PL::kBarODone + 1));
        }
      }
      // every product issued has finished before the tensor memory is read or freed
      umma_commit(bar(PL::kBarFinal));
      ws_drain(bar(PL::kBarFinal), 0, abort_flag, p.dev_status);
    }
    __syncwarp();
  } else if (warp >= kWsLoadWarp) {
    if constexpr (!R::kConvert) {
      // ------------------------------------------------------------ loads
      const int nbh = p.num_blocks * p.num_kv_heads;      // the maps' outer extent
      const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
      int k_issued = 0, v_issued = 0;                     // tiles whose K / V copies were issued
  #pragma unroll 1
      for (int t = 0; t < nt; ++t) {
        const int st = t % S;
        // K of tile t - S has been used by both S products
        if (t >= S) {
          const bool ok = ws_wait(bar(PL::kBarKEmpty + st), ((t / S) - 1) & 1, abort_flag, p.dev_status);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        // lane j < 8 locates piece j (tokens t0 + 16 j ..): z = physical block *
        // Hkv + kvh, y = offset in the block; past the range or in an
        // out-of-range block, z = nbh, which the copies read as zeros
        int z = nbh, y = 0, strad = 0;
        if (lane < kWsPieces) {
          const int tok = t * kWsKv + lane * kWsPiece;
          if (tok < kv_end) {
            const int logical = tok / p.block_size;
            const int phys = __ldg(trow + logical);
            if (phys >= 0 && phys < p.num_blocks) {
              z = phys * p.num_kv_heads + kvh;
              y = tok - logical * p.block_size;
              strad = tok + kWsPiece > kv_end;
            } else {
              flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
            }
          }
        }
        int pz[kWsPieces], py[kWsPieces], ps[kWsPieces], nstrad = 0;
  #pragma unroll
        for (int j = 0; j < kWsPieces; ++j) {
          pz[j] = __shfl_sync(0xffffffffu, z, j);
          py[j] = __shfl_sync(0xffffffffu, y, j);
          ps[j] = __shfl_sync(0xffffffffu, strad, j);
          nstrad += ps[j];
        }
        const uint32_t kst = sb + PL::kOffK + st * PL::kStageBytes;
        const uint32_t vst = sb + PL::kOffV + st * PL::kStageBytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(PL::kBarKFull + st), kWsPieces * PL::kHalves * kWsBoxBytes);
  #pragma unroll
          for (int j = 0; j < kWsPieces; ++j)
  #pragma unroll
            for (int h = 0; h < PL::kHalves; ++h)
              tma_load_3d(kst + h * PL::kKvHalf + j * kWsBoxBytes, &p.tmap_k, 64 * h, py[j], pz[j],
                          bar(PL::kBarKFull + st));
        }
        k_issued = t + 1;
        // V of tile t - S has been used by both P V products
        if (t >= S) {
          const bool ok = ws_wait(bar(PL::kBarVEmpty + st), ((t / S) - 1) & 1, abort_flag, p.dev_status);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(PL::kBarVFull + st),
                                (kWsPieces - nstrad) * PL::kHalves * kWsBoxBytes);
  #pragma unroll
          for (int j = 0; j < kWsPieces; ++j)
            if (!ps[j])
  #pragma unroll
              for (int h = 0; h < PL::kHalves; ++h)
                tma_load_3d(vst + h * PL::kKvHalf + j * kWsBoxBytes, &p.tmap_v, 64 * h, py[j], pz[j],
                            bar(PL::kBarVFull + st));
        }
        // the straddling piece's V rows, copied by the lanes in the same
        // swizzled layout, rows past the range end zero-filled
  #pragma unroll
        for (int j = 0; j < kWsPieces; ++j) {
          if (!ps[j]) continue;
          const int tok0 = t * kWsKv + j * kWsPiece;
          const uint8_t* src0 =
              p.v_cache + (static_cast<int64_t>(pz[j]) * p.block_size + py[j]) * (D * 2);
          for (int idx = lane; idx < kWsPiece * (D / 8); idx += kWarp) {
            const int rr = idx / (D / 8), c = idx % (D / 8);
            const int row = j * kWsPiece + rr;
            const uint32_t dst = vst + (c >> 3) * PL::kKvHalf + row * 128 + (((c & 7) ^ (row & 7)) << 4);
            const bool valid = tok0 + rr < kv_end;
            cp_async_16_zfill(dst, valid ? src0 + rr * (D * 2) + c * 16 : p.v_cache, valid ? 16u : 0u);
          }
        }
        cp_async_arrive_noinc(bar(PL::kBarVFull + st));
        v_issued = t + 1;
      }
      // the copies still in flight land before the CTA ends: the last fill of each stage
      cp_async_wait_all();
      if (lane == 0) {
        for (int st = 0; st < S; ++st) {
          const int kf = k_issued > st ? (k_issued - st + S - 1) / S : 0;
          const int vf = v_issued > st ? (v_issued - st + S - 1) / S : 0;
          if (kf > 0) ws_drain(bar(PL::kBarKFull + st), (kf - 1) & 1, abort_flag, p.dev_status);
          if (vf > 0) ws_drain(bar(PL::kBarVFull + st), (vf - 1) & 1, abort_flag, p.dev_status);
        }
      }
      __syncwarp();

    } else {
      // ---------------------------------------------------------- code loads
      // One-byte caches: the three load warps bring each tile's K and V codes
      // with 16-byte loads through the block table and convert them exactly to
      // f16 (E4M3 / E5M2 by cvt, INT8 as 1024 + (x + 128) - 1152) into the
      // same swizzled operand layouts, zeros past the range or in an
      // out-of-range block; each warp then fences its stores for the tensor
      // cores and arrives once.
      // INT4 caches: an item is one 32-element group of a token (16 bytes of
      // codes and its fp16 scale and zero point); each element x = scale n +
      // zero (one rounding in fp32) becomes a hi + lo pair in the query's
      // 16-bit type, hi = x rounded, lo = (x - hi) rounded, into the stage's hi
      // and lo operand tiles.
      const int lt = (warp - kWsLoadWarp) * kWarp + lane;       // 0 .. 95
      constexpr int kLoaders = R::kLoadWarps * kWarp;
      constexpr int kItemCols = kI4 ? 32 : 16;                  // elements per item
      constexpr int kItems = kWsKv * (D / kItemCols);
      constexpr int kPer = (kItems + kLoaders - 1) / kLoaders;
      const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
      const int64_t rows_total = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads * p.block_size;
      auto convert_tile = [&](const uint8_t* cache, int which, uint32_t dst, int t) {
        // lane j < pieces: the first cache row of piece j, or -1
        int64_t base = -1;
        if (lane < kWsPieces) {
          const int tok = t * kWsKv + lane * kWsPiece;
          if (tok < kv_end) {
            const int logical = tok / p.block_size;
            const int phys = __ldg(trow + logical);
            if (phys >= 0 && phys < p.num_blocks)
              base = (static_cast<int64_t>(phys) * p.num_kv_heads + kvh) * p.block_size +
                     (tok - logical * p.block_size);
            else
              flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
          }
        }
        constexpr int kRowBytes = kI4 ? D / 2 : D;              // code bytes per cache row
        uint4 raw[kPer];
        uint32_t szp[kPer];                                     // INT4: fp16 scale | zero << 16
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int idx = lt + k * kLoaders;
          const int rr = idx / (D / kItemCols), cc = idx % (D / kItemCols);
          const int64_t rb = __shfl_sync(0xffffffffu, base, (rr / kWsPiece) & 7);
          raw[k] = make_uint4(0, 0, 0, 0);
          szp[k] = 0;
          if (idx < kItems && rb >= 0 && t * kWsKv + rr < kv_end) {
            const int64_t row = rb + rr % kWsPiece;
            raw[k] = ld_global_nc_v4(cache + row * kRowBytes + cc * 16);
            if constexpr (kI4)
              szp[k] = __ldg(reinterpret_cast<const uint32_t*>(p.scales) +
                             (which * rows_total + row) * (D / 32) + cc);
          }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int idx = lt + k * kLoaders;
          if (idx < kItems) {
            const int rr = idx / (D / kItemCols), cc = idx % (D / kItemCols);
            const uint32_t row = dst + rr * 128;
            if constexpr (kI4) {
              // f16 chunks 4 cc .. 4 cc + 3 of row rr, in the hi and the lo tile
              const float sc = __half2float(__ushort_as_half(static_cast<uint16_t>(szp[k] & 0xFFFFu)));
              const float zp = __half2float(__ushort_as_half(static_cast<uint16_t>(szp[k] >> 16)));
              const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const uint32_t byte = (w[q4] >> (8 * e)) & 0xFFu;
                  const float x0 = __fmaf_rn(sc, static_cast<float>(byte & 15u), zp);
                  const float x1 = __fmaf_rn(sc, static_cast<float>(byte >> 4), zp);
                  hw[e] = Half16<QT>::pack_rn(x0, x1);
                  const float2 f = Half16<QT>::unpack(hw[e]);
                  lw[e] = Half16<QT>::pack_rn(x0 - f.x, x1 - f.y);
                }
                const int c = 4 * cc + q4;
                const uint32_t at = row + (c >> 3) * PL::kKvHalf + (((c & 7) ^ (rr & 7)) << 4);
                st_shared_v4(at, make_uint4(hw[0], hw[1], hw[2], hw[3]));
                st_shared_v4(at + PL::kTileBytes, make_uint4(lw[0], lw[1], lw[2], lw[3]));
              }
            } else {
              uint4 lo, hi;
              codes16_to_f16<KV>(raw[k], lo, hi);
              const int c0 = 2 * cc;                     // f16 chunks c0, c0 + 1 of row rr
              st_shared_v4(row + (c0 >> 3) * PL::kKvHalf + (((c0 & 7) ^ (rr & 7)) << 4), lo);
              st_shared_v4(row + ((c0 + 1) >> 3) * PL::kKvHalf + ((((c0 + 1) & 7) ^ (rr & 7)) << 4), hi);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
      };
#pragma unroll 1
      for (int t = 0; t < nt; ++t) {
        const int st = t % S;
        if (t >= S) {
          const bool ok = ws_wait(bar(PL::kBarKEmpty + st), ((t / S) - 1) & 1, abort_flag, p.dev_status);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        convert_tile(p.k_cache, 0, sb + PL::kOffK + st * PL::kStageBytes, t);
        if (lane == 0) mbar_arrive(bar(PL::kBarKFull + st));
        if (t >= S) {
          const bool ok = ws_wait(bar(PL::kBarVEmpty + st), ((t / S) - 1) & 1, abort_flag, p.dev_status);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        convert_tile(p.v_cache, 1, sb + PL::kOffV + st * PL::kStageBytes, t);
        if (lane == 0) mbar_arrive(bar(PL::kBarVFull + st));
      }
    }
  }

  // ------------------------------------------------------------ output
  __syncthreads();
  const bool all_ok = *abort_flag == 0;
  if (warp < 8) {
    tmem_store_wait();                                   // (a launch that gave up mid-tile)
    tc_fence_after();
    uint16_t* orow = static_cast<uint16_t*>(p.out) +
                     ((static_cast<int64_t>(p.q_start[b]) + ji + jj) * p.num_q_heads +
                      kvh * group + g) * D;
    if (all_ok && nt > 0) {
      // (one-byte caches: O is in units of vu)
      const float inv = (row_ok && l > 0.f) ? vu / l : 0.f;
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        float o[32];
        tmem_ld32(t_s + 128 + 32 * k, o);                // warp-collective: every row
        if (row_q) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 w;
            w.x = Half16<QT>::pack_rn(o[8 * c] * inv, o[8 * c + 1] * inv);
            w.y = Half16<QT>::pack_rn(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
            w.z = Half16<QT>::pack_rn(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
            w.w = Half16<QT>::pack_rn(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
            reinterpret_cast<uint4*>(orow + 32 * k)[c] = w;
          }
        }
      }
    } else if (row_q) {
      for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWsMmaWarp) tmem_dealloc(tmem, PL::kTmemCols);
  pdl_launch_dependents();
}

// ---------------------------------------------------------------- host side
using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

// cuTensorMapEncodeTiled, taken from the driver once
EncodeTiled encode_tiled() {
  static std::atomic<EncodeTiled> fn{nullptr};
  EncodeTiled f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && ptr != nullptr) {
      f = reinterpret_cast<EncodeTiled>(ptr);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

// The cache [num_blocks][Hkv][block_size][D] of 16-bit values as a 3-D tensor
// (D, block_size, num_blocks * Hkv), read in boxes of 64 values x 16 rows with
// the 128-byte swizzle; boxes outside it read as zeros.
bool cache_map(CUtensorMap* map, const void* cache, int num_blocks, int num_kv_heads,
               int block_size, int head_dim) {
  const EncodeTiled enc = encode_tiled();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(block_size),
                              static_cast<cuuint64_t>(num_blocks) * num_kv_heads};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(block_size) * head_dim * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kWsPiece), 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(cache), dims, strides, box,
             elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KV, int QT, int D>
cudaError_t launch_ws_t(const PrefillArgs& a, cudaStream_t st) {
  using PL = WsPlan<D, KV>;
  using R = WsRoles<KV>;
  WsParams p;
  if (!R::kConvert &&
      (!cache_map(&p.tmap_k, a.k_cache, a.num_blocks, a.num_kv_heads, a.block_size, D) ||
       !cache_map(&p.tmap_v, a.v_cache, a.num_blocks, a.num_kv_heads, a.block_size, D)))
    return cudaErrorInvalidValue;
  p.q = static_cast<const uint16_t*>(a.q);
  p.k_cache = static_cast<const uint8_t*>(a.k_cache);
  p.v_cache = static_cast<const uint8_t*>(a.v_cache);
  p.scales = static_cast<const float*>(a.scales);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.q_start = a.q_start;
  p.out = a.out;
  p.dev_status = a.dev_status;
  p.max_query_len = a.max_query_len;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.softmax_scale = a.softmax_scale;
#ifdef PKV_TEST_HOOKS
  p.test_drop_commit = getenv("PKV_TEST_DROP_COMMIT") != nullptr;
#endif
  auto kern = prefill_ws_kernel<KV, QT, D>;
  static std::atomic<int> attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PL::kSmemRequest);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(1, std::memory_order_relaxed);
  }
  const int group = a.num_q_heads / a.num_kv_heads;
  const int rows = 2 * (kWsRows / group);               // query tokens per CTA
  const dim3 grid(static_cast<unsigned>((a.max_query_len + rows - 1) / rows),
                  static_cast<unsigned>(a.num_kv_heads), static_cast<unsigned>(a.num_seqs));
  return launch_pdl(kern, grid, dim3(R::kThreads), PL::kSmemRequest, st, p);
}

template <int KV, int D>
cudaError_t launch_ws_q(const PrefillArgs& a, cudaStream_t st) {
  if constexpr (KV == PKV_F16 || KV == PKV_BF16) {
    return launch_ws_t<KV, KV, D>(a, st);
  } else {
    return a.q_dtype == PKV_F16 ? launch_ws_t<KV, PKV_F16, D>(a, st)
                                : launch_ws_t<KV, PKV_BF16, D>(a, st);
  }
}

template <int D>
cudaError_t launch_ws_d(const PrefillArgs& a, cudaStream_t st) {
  switch (a.kv_dtype) {
    case PKV_F16: return launch_ws_q<PKV_F16, D>(a, st);
    case PKV_BF16: return launch_ws_q<PKV_BF16, D>(a, st);
    case PKV_FP8_E4M3: return launch_ws_q<PKV_FP8_E4M3, D>(a, st);
    case PKV_FP8_E5M2: return launch_ws_q<PKV_FP8_E5M2, D>(a, st);
    case PKV_INT8: return launch_ws_q<PKV_INT8, D>(a, st);
    case PKV_INT4_G32: return launch_ws_q<PKV_INT4_G32, D>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool prefill_ws_supported(const PrefillArgs& a) {
  return (a.kv_dtype == PKV_F16 || a.kv_dtype == PKV_BF16 || is_blk8(a.kv_dtype) ||
          a.kv_dtype == PKV_INT4_G32) &&
         (a.head_dim == 64 || a.head_dim == 128);
}

cudaError_t launch_prefill_ws(const PrefillArgs& a, cudaStream_t st) {
  if (a.num_seqs == 0 || a.max_query_len == 0) return cudaSuccess;
  return a.head_dim == 64 ? launch_ws_d<64>(a, st) : launch_ws_d<128>(a, st);
}

}  // namespace pkv
