// paged_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits — inside a
// custom allocator's own callbacks, in a process whose memory pool is fixed
// and fully handed out up front, under a runtime that forbids allocation on
// its hot path, or in plain C callers that have no allocator to ask for
// scratch.  Long contexts need split-KV scratch for the per-partition
// partial results; this entry point takes that scratch from one static
// device array compiled into the library instead of from the caller.
//
// The array holds kNoAllocScratchBytes (64 MiB) on every GPU that loads the
// library, for the life of the process.  Requests whose partial results need
// more are rejected with PKV_ERR_WORKSPACE before anything is launched.
//
// Sharing: every call uses the same array.  Nothing in it has to start at
// zero (each partition writes its partial result before the merge reads it,
// and the merge reads only partitions written by the same call), but two
// calls that overlap on the GPU — on different streams, or from different
// host threads — race on it and may return wrong results.  Serialize them.
//
// Set-up: every call looks up the array's device address with
// cudaGetSymbolAddress, with the caller's device current.  The address is
// not cached: after cudaDeviceReset, or when a context is destroyed and
// created again, the library's module is loaded anew and the array can sit
// at another address, so a cached pointer could point at freed memory.  The
// first call on a device loads the module there (CUDA loads modules lazily);
// make that first call before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"
#include "pkv_internal.h"

#define PKV_NOALLOC_SCRATCH_BYTES (size_t(64) << 20)

// The scratch itself.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;

// Device address of the scratch array in the current device's context.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" int paged_decode_attention_noalloc(
    const void* q, int q_dtype, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, const void* scales, int kv_dtype, int num_blocks, void* out,
    float softmax_scale, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int partition_size, int* dev_status, void* stream) {
  // the scratch this request needs (0 when every sequence fits one partition)
  const size_t need = paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                   head_dim, max_blocks_per_seq, block_size,
                                                   partition_size);
  if (need > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0 && scratch_address(&scratch) != cudaSuccess) return PKV_ERR_CUDA;
  // the regular entry point does the validation and the launches; it is
  // handed the static scratch as its workspace
  return paged_decode_attention(q, q_dtype, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, scales, kv_dtype, num_blocks, out,
                                softmax_scale, num_q_heads, num_kv_heads, head_dim, block_size,
                                partition_size, scratch, need > 0 ? kNoAllocScratchBytes : 0,
                                dev_status, stream);
}
