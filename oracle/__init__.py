"""ctypes binding of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only importers.  The CUDA library never
imports it, and nothing here falls back to it.

Arrays are numpy host arrays; 16-bit floats are passed as raw uint16 bits.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

_lib: Optional[ctypes.CDLL] = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
D = ctypes.c_double


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_double.restype = D
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = D
        L.oracle_f32_to_f16_rne.argtypes = [ctypes.c_float]
        L.oracle_f32_to_f16_rne.restype = ctypes.c_uint16
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_double.restype = D
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e5m2_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e5m2_to_double.restype = D
        L.oracle_e5m2_encode.argtypes = [ctypes.c_float]
        L.oracle_e5m2_encode.restype = ctypes.c_uint8
        L.oracle_int8_encode.argtypes = [ctypes.c_float]
        L.oracle_int8_encode.restype = ctypes.c_int8
        L.oracle_kv_cache_bytes.argtypes = [D] * 6
        L.oracle_kv_cache_bytes.restype = D
        L.oracle_num_pages.argtypes = [I64, I64]
        L.oracle_num_pages.restype = I64
        L.oracle_physical_address.argtypes = [P, I32, I32, I64, P, P]
        L.oracle_physical_address.restype = I32
        L.oracle_kv_write.argtypes = [P, P, I32, P, I64, P, P, P, I32, I32, I32, I32, I32]
        L.oracle_kv_write.restype = I32
        L.oracle_decode_attention.argtypes = [P, I32, P, P, P, I32, P, I32, P, I32, I32, P, D,
                                              I32, I32, I32, I32, I32]
        L.oracle_decode_attention.restype = I32
        L.oracle_decode_attention_pairs.argtypes = [P, I32, P, P, P, I32, P, I32, P, I32, I32,
                                                    P, D, I32, I32, I32, I32, P, P, I32, I32]
        L.oracle_decode_attention_pairs.restype = I32
        L.oracle_dequant_row.argtypes = [P, P, I32, I32, I32, I32, I32, I32, I32, I32, I32, P]
        L.oracle_dequant_row.restype = I32
        L.oracle_prefill_attention.argtypes = [P, I32, P, P, P, P, I32, P, I32, P, I32, I32, P, D,
                                                I32, I32, I32, I32, I32]
        L.oracle_prefill_attention.restype = I32
        L.oracle_copy_blocks.argtypes = [P, P, P, I32, P, I32, I32, I32, I32, I32]
        L.oracle_copy_blocks.restype = I32
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = I32
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- codecs
def f16_to_double(bits: int) -> float:
    return lib().oracle_f16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def f32_to_f16_rne(x: float) -> int:
    return lib().oracle_f32_to_f16_rne(float(np.float32(x)))


def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code))


def e4m3_encode(y: float) -> int:
    return lib().oracle_e4m3_encode(float(np.float32(y)))


def e5m2_to_double(code: int) -> float:
    return lib().oracle_e5m2_to_double(int(code))


def e5m2_encode(y: float) -> int:
    return lib().oracle_e5m2_encode(float(np.float32(y)))


def int8_encode(y: float) -> int:
    return lib().oracle_int8_encode(float(np.float32(y)))


# ---------------------------------------------------------------- formulas
def kv_cache_bytes(layers, heads, head_dim, seq_len, batch, bytes_per_elem) -> float:
    return lib().oracle_kv_cache_bytes(layers, heads, head_dim, seq_len, batch, bytes_per_elem)


def num_pages(tokens: int, page_size: int) -> int:
    return lib().oracle_num_pages(tokens, page_size)


def physical_address(table_row, block_size: int, token_index: int):
    row = np.ascontiguousarray(table_row, dtype=np.int32)
    pb, off = I32(), I32()
    r = lib().oracle_physical_address(_ptr(row), len(row), block_size, token_index,
                                      ctypes.byref(pb), ctypes.byref(off))
    if r:
        raise IndexError("token outside the block table")
    return pb.value, off.value


# ---------------------------------------------------------------- cache
def alloc_cache(kv_dtype: int, num_blocks: int, num_kv_heads: int, head_dim: int,
                block_size: int):
    """Zeroed host k_cache, v_cache, scales in the library's layout."""
    if kv_dtype in (0, 1):
        k = np.zeros((num_blocks, num_kv_heads, block_size, head_dim), np.uint16)
        return k, k.copy(), None
    if kv_dtype in (2, 4, 5):
        k = np.zeros((num_blocks, num_kv_heads, block_size, head_dim), np.uint8)
        return k, k.copy(), np.zeros((2, num_blocks, num_kv_heads), np.float32)
    if kv_dtype == 3:
        k = np.zeros((num_blocks, num_kv_heads, block_size, head_dim // 2), np.uint8)
        s = np.zeros((2, num_blocks, num_kv_heads, block_size, head_dim // 32, 2), np.uint16)
        return k, k.copy(), s
    raise ValueError(kv_dtype)


def kv_write(k_new, v_new, new_dtype, slot_mapping, k_cache, v_cache, scales, kv_dtype,
             num_blocks, num_kv_heads, head_dim, block_size) -> None:
    k_new = np.ascontiguousarray(k_new, np.uint16)
    v_new = np.ascontiguousarray(v_new, np.uint16)
    slots = np.ascontiguousarray(slot_mapping, np.int64)
    r = lib().oracle_kv_write(_ptr(k_new), _ptr(v_new), new_dtype, _ptr(slots), len(slots),
                              _ptr(k_cache), _ptr(v_cache), _ptr(scales), kv_dtype, num_blocks,
                              num_kv_heads, head_dim, block_size)
    if r:
        raise ValueError(f"oracle_kv_write rejected its arguments ({r})")


def copy_blocks(k_cache, v_cache, scales, kv_dtype, pairs, num_blocks, num_kv_heads, head_dim,
                block_size) -> int:
    """Block dst of each (src, dst) pair becomes a copy of block src; returns the
    number of pairs skipped for an out-of-range id."""
    pr = np.ascontiguousarray(pairs, np.int32).reshape(-1, 2)
    r = lib().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(scales), kv_dtype, _ptr(pr),
                                 len(pr), num_blocks, num_kv_heads, head_dim, block_size)
    if r < 0:
        raise ValueError("oracle_copy_blocks rejected its arguments")
    return r


def decode_attention(q, q_dtype, k_cache, v_cache, block_tables, context_lens, scales,
                     kv_dtype, num_blocks, softmax_scale, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_threads: int = 0) -> np.ndarray:
    q = np.ascontiguousarray(q, np.uint16)
    bt = np.ascontiguousarray(block_tables, np.int32)
    cl = np.ascontiguousarray(context_lens, np.int32)
    b = len(cl)
    out = np.zeros((b, num_q_heads, head_dim), np.float64)
    r = lib().oracle_decode_attention(_ptr(q), q_dtype, _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                      bt.shape[1], _ptr(cl), b, _ptr(scales), kv_dtype,
                                      num_blocks, _ptr(out), softmax_scale, num_q_heads,
                                      num_kv_heads, head_dim, block_size, num_threads)
    if r:
        raise ValueError(f"oracle_decode_attention failed ({r})")
    return out


def prefill_attention(q, q_dtype, q_start, k_cache, v_cache, block_tables, context_lens, scales,
                      kv_dtype, num_blocks, softmax_scale, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_threads: int = 0) -> np.ndarray:
    """Chunked prefill: rows q_start[b]..q_start[b+1]-1 of q are sequence b's chunk."""
    q = np.ascontiguousarray(q, np.uint16)
    qs = np.ascontiguousarray(q_start, np.int32)
    bt = np.ascontiguousarray(block_tables, np.int32)
    cl = np.ascontiguousarray(context_lens, np.int32)
    out = np.zeros((int(qs[-1]), num_q_heads, head_dim), np.float64)
    r = lib().oracle_prefill_attention(_ptr(q), q_dtype, _ptr(qs), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(bt), bt.shape[1], _ptr(cl), len(cl), _ptr(scales),
                                       kv_dtype, num_blocks, _ptr(out), softmax_scale,
                                       num_q_heads, num_kv_heads, head_dim, block_size,
                                       num_threads)
    if r:
        raise ValueError(f"oracle_prefill_attention failed ({r})")
    return out


def decode_attention_pairs(q, q_dtype, k_cache, v_cache, block_tables, context_lens, scales,
                           kv_dtype, num_blocks, softmax_scale, num_q_heads, num_kv_heads,
                           head_dim, block_size, pair_seq, pair_head,
                           num_threads: int = 0) -> np.ndarray:
    q = np.ascontiguousarray(q, np.uint16)
    bt = np.ascontiguousarray(block_tables, np.int32)
    cl = np.ascontiguousarray(context_lens, np.int32)
    ps = np.ascontiguousarray(pair_seq, np.int32)
    ph = np.ascontiguousarray(pair_head, np.int32)
    out = np.zeros((len(ps), head_dim), np.float64)
    r = lib().oracle_decode_attention_pairs(_ptr(q), q_dtype, _ptr(k_cache), _ptr(v_cache),
                                            _ptr(bt), bt.shape[1], _ptr(cl), len(cl),
                                            _ptr(scales), kv_dtype, num_blocks, _ptr(out),
                                            softmax_scale, num_q_heads, num_kv_heads, head_dim,
                                            block_size, _ptr(ps), _ptr(ph), len(ps),
                                            num_threads)
    if r:
        raise ValueError(f"oracle_decode_attention_pairs failed ({r})")
    return out


def dequant_row(cache, scales, which_kv, kv_dtype, num_blocks, num_kv_heads, head_dim,
                block_size, block, kv_head, offset) -> np.ndarray:
    row = np.zeros(head_dim, np.float64)
    r = lib().oracle_dequant_row(_ptr(cache), _ptr(scales), which_kv, kv_dtype, num_blocks,
                                 num_kv_heads, head_dim, block_size, block, kv_head, offset,
                                 _ptr(row))
    if r:
        raise ValueError("oracle_dequant_row failed")
    return row


def max_threads() -> int:
    return lib().oracle_max_threads()


# ---------------------------------------------------------------- helpers
def prefill_case(case):
    """The case's context written by the oracle's own write: (k_cache, v_cache, scales)."""
    w = case.w
    k, v, s = alloc_cache(w.kv_dtype, case.num_blocks, w.num_kv_heads, w.head_dim,
                          w.block_size)
    kv_write(case.prefill_k, case.prefill_v, w.q_dtype, case.prefill_slots, k, v, s,
             w.kv_dtype, case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    return k, v, s


def step_case(case, k, v, s, num_threads: int = 0) -> np.ndarray:
    """One decode step on the oracle: write the new token, then attend (fp64 out)."""
    w = case.w
    kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
             case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    return decode_attention(case.q, w.q_dtype, k, v, case.block_tables, case.context_lens, s,
                            w.kv_dtype, case.num_blocks, w.softmax_scale, w.num_q_heads,
                            w.num_kv_heads, w.head_dim, w.block_size, num_threads)


os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")
