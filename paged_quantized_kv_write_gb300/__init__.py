"""Python binding of libpagedkv (paged, quantized KV-cache decode for GB300).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory and
streams); each call passes raw device pointers and sizes to the C ABI
declared in include/pagedkv.h, on the current torch stream unless a stream
is given.  There is no CPU fallback: importing this package loads
libpagedkv.so and fails loudly when it is missing.

Calls (same names as the C ABI):
    paged_kv_write(k_new, v_new, slot_mapping, k_cache, v_cache, scales, kv_dtype, ...)
    paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scales, out,
                           softmax_scale, num_kv_heads, kv_dtype, block_size, ...)
    paged_decode_attention_with_write(q, k_new, v_new, slot_mapping, k_cache, v_cache, ...)
    paged_kv_copy_blocks(k_cache, v_cache, scales, kv_dtype, block_pairs, ...)
    paged_prefill_attention(q, q_start, k_cache, v_cache, block_tables, context_lens, ...)
    paged_decode_workspace_bytes(...), paged_decode_partition_size(...)
"""

from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

PKV_F16, PKV_BF16, PKV_FP8_E4M3, PKV_INT4_G32, PKV_FP8_E5M2, PKV_INT8 = 0, 1, 2, 3, 4, 5
(PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_DEVICE_BOUNDS,
 PKV_ERR_WORKSPACE, PKV_ERR_DEVICE_TIMEOUT) = 0, 1, 2, 3, 4, 5, 8

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpagedkv.so")
# the test build: the same library plus the decode comparators and the switch
# that exercises the bounded waits (see build.py); only the tests load it
TEST_LIB_PATH = os.path.join(_HERE, "_lib", "libpagedkv_test.so")


def _load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{os.path.basename(path)} not found at {path}; build it with "
            "`python paged_quantized_kv_write_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(path)
    P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                        ctypes.c_size_t)
    lib.paged_kv_write.argtypes = [P, P, I, P, I64, P, P, P, I, I, I, I, I, P, P]
    lib.paged_kv_write.restype = I
    lib.paged_decode_attention_with_write.argtypes = [P, I, P, P, P, P, P, P, I, P, I, P, I, I,
                                                      P, F, I, I, I, I, I, P, SZ, P, P]
    lib.paged_decode_attention_with_write.restype = I
    lib.paged_prefill_attention.argtypes = [P, I, P, I, P, P, P, I, P, I, P, I, I, P, F, I, I, I,
                                            I, P, P]
    lib.paged_prefill_attention.restype = I
    lib.paged_kv_copy_blocks.argtypes = [P, P, P, I, P, I, I, I, I, I, P, P]
    lib.paged_kv_copy_blocks.restype = I
    lib.paged_decode_attention.argtypes = [P, I, P, P, P, I, P, I, P, I, I, P, F, I, I, I, I, I,
                                           P, SZ, P, P]
    lib.paged_decode_attention.restype = I
    lib.paged_decode_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.paged_decode_workspace_bytes.restype = SZ
    lib.paged_decode_partition_size.argtypes = [I, I, I, I, I, I]
    lib.paged_decode_partition_size.restype = I
    lib.paged_kv_status_string.argtypes = [I]
    lib.paged_kv_status_string.restype = ctypes.c_char_p
    lib.paged_kv_version.argtypes = []
    lib.paged_kv_version.restype = I
    return lib


_lib = _load()
_loaded = {"product": _lib}


@contextlib.contextmanager
def library(kind: str):
    """Route the calls of this module through the product library ("product")
    or the test build ("test") inside a with-block; both share torch's device
    memory and streams."""
    global _lib
    if kind not in _loaded:
        if kind != "test":
            raise ValueError(f"unknown library {kind!r}")
        _loaded[kind] = _load(TEST_LIB_PATH)
    prev = _lib
    _lib = _loaded[kind]
    try:
        yield _lib
    finally:
        _lib = prev


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib.paged_kv_status_string(status).decode()} ({status})")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PKV_F16
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"expected a float16 or bfloat16 tensor, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("pagedkv takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("pagedkv takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream if hasattr(s, "cuda_stream") else int(s))


def row_bytes(kv_dtype: int, head_dim: int) -> int:
    return {PKV_F16: 2 * head_dim, PKV_BF16: 2 * head_dim, PKV_FP8_E4M3: head_dim,
            PKV_FP8_E5M2: head_dim, PKV_INT8: head_dim, PKV_INT4_G32: head_dim // 2}[kv_dtype]


def alloc_cache(kv_dtype: int, num_blocks: int, num_kv_heads: int, head_dim: int,
                block_size: int, device="cuda"):
    """Zeroed k_cache, v_cache and scales in the library's layout."""
    if kv_dtype in (PKV_F16, PKV_BF16):
        dt = torch.float16 if kv_dtype == PKV_F16 else torch.bfloat16
        k = torch.zeros((num_blocks, num_kv_heads, block_size, head_dim), dtype=dt, device=device)
        return k, torch.zeros_like(k), None
    k = torch.zeros((num_blocks, num_kv_heads, block_size, row_bytes(kv_dtype, head_dim)),
                    dtype=torch.uint8, device=device)
    if kv_dtype in (PKV_FP8_E4M3, PKV_FP8_E5M2, PKV_INT8):
        s = torch.zeros((2, num_blocks, num_kv_heads), dtype=torch.float32, device=device)
    else:
        s = torch.zeros((2, num_blocks, num_kv_heads, block_size, head_dim // 32, 2),
                        dtype=torch.float16, device=device)
    return k, torch.zeros_like(k), s


def paged_kv_write(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, scales: Optional[torch.Tensor],
                   kv_dtype: int, block_size: int, head_dim: int,
                   dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """k_new/v_new [T, Hkv, D]; slot_mapping int64 [T]; caches [NB, Hkv, bs, row]."""
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    num_tokens = slot_mapping.numel()
    num_kv_heads = k_cache.shape[1]
    r = _lib.paged_kv_write(_ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(slot_mapping),
                            num_tokens, _ptr(k_cache), _ptr(v_cache), _ptr(scales), kv_dtype,
                            k_cache.shape[0], num_kv_heads, head_dim, block_size,
                            _ptr(dev_status), _stream(stream))
    if r != PKV_OK:
        raise PagedKVError(r, "paged_kv_write")


def paged_kv_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor,
                         scales: Optional[torch.Tensor], kv_dtype: int, block_pairs: torch.Tensor,
                         block_size: int, head_dim: int, dev_status: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    """block_pairs int32 [n, 2] (src, dst): block dst becomes a byte copy of block src."""
    if block_pairs.dtype != torch.int32 or block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise TypeError("block_pairs must be int32 [n, 2]")
    if not block_pairs.is_contiguous():
        raise ValueError("block_pairs must be contiguous")
    r = _lib.paged_kv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(scales), kv_dtype,
                                  _ptr(block_pairs), block_pairs.shape[0], k_cache.shape[0],
                                  k_cache.shape[1], head_dim, block_size, _ptr(dev_status),
                                  _stream(stream))
    if r != PKV_OK:
        raise PagedKVError(r, "paged_kv_copy_blocks")


def paged_decode_partition_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                max_blocks_per_seq: int, block_size: int,
                                partition_size: int = 0) -> int:
    return _lib.paged_decode_partition_size(num_seqs, num_q_heads, num_kv_heads,
                                            max_blocks_per_seq, block_size, partition_size)


def paged_decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                 head_dim: int, max_blocks_per_seq: int, block_size: int,
                                 partition_size: int = 0) -> int:
    return _lib.paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, partition_size)


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           scales: Optional[torch.Tensor], out: torch.Tensor,
                           softmax_scale: float, num_kv_heads: int, kv_dtype: int,
                           block_size: int, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None,
                           dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q/out [B, Hq, D]; block_tables int32 [B, MB]; context_lens int32 [B]."""
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    b, hq, d = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    r = _lib.paged_decode_attention(_ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_tables), block_tables.shape[1],
                                    _ptr(context_lens), b, _ptr(scales), kv_dtype,
                                    k_cache.shape[0], _ptr(out), float(softmax_scale), hq,
                                    num_kv_heads, d, block_size, partition_size,
                                    _ptr(workspace), ws_bytes, _ptr(dev_status),
                                    _stream(stream))
    if r != PKV_OK:
        raise PagedKVError(r, "paged_decode_attention")


def paged_decode_attention_with_write(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                      slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                                      context_lens: torch.Tensor, scales: Optional[torch.Tensor],
                                      out: torch.Tensor, softmax_scale: float, kv_dtype: int,
                                      block_size: int, partition_size: int = 0,
                                      workspace: Optional[torch.Tensor] = None,
                                      dev_status: Optional[torch.Tensor] = None,
                                      stream=None) -> None:
    """Write each sequence's new token (k_new/v_new [B, Hkv, D], slot_mapping int64 [B])
    and attend, in one launch."""
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    b, hq, d = q.shape
    num_kv_heads = k_new.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    r = _lib.paged_decode_attention_with_write(
        _ptr(q), _dtype_code(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), b,
        _ptr(scales), kv_dtype, k_cache.shape[0], _ptr(out), float(softmax_scale), hq,
        num_kv_heads, d, block_size, partition_size, _ptr(workspace), ws_bytes,
        _ptr(dev_status), _stream(stream))
    if r != PKV_OK:
        raise PagedKVError(r, "paged_decode_attention_with_write")


def paged_prefill_attention(q: torch.Tensor, q_start: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, scales: Optional[torch.Tensor],
                            out: torch.Tensor, softmax_scale: float, num_kv_heads: int,
                            kv_dtype: int, block_size: int, max_query_len: int,
                            dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Chunked prefill: q/out [T, Hq, D] (sequence b's chunk = rows q_start[b]..q_start[b+1]-1),
    q_start int32 [B + 1]; each query attends causally up to its own position."""
    if q_start.dtype != torch.int32 or block_tables.dtype != torch.int32 or \
            context_lens.dtype != torch.int32:
        raise TypeError("q_start, block_tables and context_lens must be int32")
    t, hq, d = q.shape
    r = _lib.paged_prefill_attention(
        _ptr(q), _dtype_code(q), _ptr(q_start), int(max_query_len), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), context_lens.numel(),
        _ptr(scales), kv_dtype, k_cache.shape[0], _ptr(out), float(softmax_scale), hq,
        num_kv_heads, d, block_size, _ptr(dev_status), _stream(stream))
    if r != PKV_OK:
        raise PagedKVError(r, "paged_prefill_attention")


def make_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   max_blocks_per_seq: int, block_size: int, partition_size: int = 0,
                   device="cuda") -> Optional[torch.Tensor]:
    n = paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                     max_blocks_per_seq, block_size, partition_size)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device)


def version() -> int:
    return _lib.paged_kv_version()


lib = _lib
