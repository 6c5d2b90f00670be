"""Shared helpers for the GPU parity tests: upload a case, run the library,
compare with the oracle under the stated tolerances."""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads as W

# max-abs tolerances on the attention output (the benchmark spec): 2e-3 for 16-bit
# KV, 5e-3 for FP8/INT4 against the oracle on the same dequantized values.
TOL = {W.F16: 2e-3, W.BF16: 2e-3, W.FP8_E4M3: 5e-3, W.INT4_G32: 5e-3, W.FP8_E5M2: 5e-3,
       W.INT8: 5e-3}


def torch_dtype(code: int):
    return torch.float16 if code == W.F16 else torch.bfloat16


def bits_to_tensor(bits: np.ndarray, code: int, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch_dtype(code)).to(device)


def tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def cache_to_device(k: np.ndarray, v: np.ndarray, s, kv_dtype: int, device="cuda"):
    if kv_dtype in (W.F16, W.BF16):
        kt = bits_to_tensor(k, kv_dtype, device)
        vt = bits_to_tensor(v, kv_dtype, device)
    else:
        kt = torch.from_numpy(np.ascontiguousarray(k)).to(device)
        vt = torch.from_numpy(np.ascontiguousarray(v)).to(device)
    st = None
    if s is not None:
        if kv_dtype in W.BLK8_TYPES:
            st = torch.from_numpy(np.ascontiguousarray(s)).to(device)
        else:
            st = torch.from_numpy(np.ascontiguousarray(s).view(np.int16)).view(torch.float16).to(device)
    return kt, vt, st


def cache_to_host(kt, vt, st, kv_dtype: int):
    def raw(t):
        if t is None:
            return None
        if t.dtype in (torch.float16, torch.bfloat16):
            return t.view(torch.int16).cpu().numpy().view(np.uint16)
        return t.cpu().numpy()
    return raw(kt), raw(vt), raw(st)


def half_ulp(x: np.ndarray, code: int) -> np.ndarray:
    """Half a unit in the last place of |x| in the output dtype (the final rounding)."""
    mant = 10 if code == W.F16 else 7
    a = np.maximum(np.abs(x), 2.0 ** -14 if code == W.F16 else 2.0 ** -126)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - mant - 1)


def round_to(x: np.ndarray, code: int) -> np.ndarray:
    """fp64 values rounded (nearest even) to the 16-bit output dtype, back as fp64."""
    if code == W.F16:
        return x.astype(np.float16).astype(np.float64)
    return W.bits_to_f32(W.f32_to_bf16_bits(x.astype(np.float32)), W.BF16).astype(np.float64)


def check_close(gpu: np.ndarray, ref: np.ndarray, kv_dtype: int, out_dtype: int, what=""):
    """Assert |gpu - oracle| <= tol + half an ulp of the output dtype at |oracle|.

    Returns (max |gpu - oracle|, max |gpu - oracle rounded to the output dtype|,
    max error / bound)."""
    err = np.abs(gpu - ref)
    bound = TOL[kv_dtype] + half_ulp(ref, out_dtype)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} outputs exceed tolerance; worst at {i}: "
            f"gpu {gpu[i]!r} oracle {ref[i]!r} err {err[i]:.3g} bound {bound[i]:.3g}")
    if not err.size:
        return 0.0, 0.0, 0.0
    err_r = np.abs(gpu - round_to(ref, out_dtype))
    return float(err.max()), float(err_r.max()), float((err / bound).max())


class GpuCase:
    """A workload's inputs on the GPU, with an oracle-written cache uploaded."""

    def __init__(self, case: W.Case, k, v, s, partition_size: int = 0, device_cache=None):
        """device_cache: (k, v, scales) tensors already on the GPU, used instead of
        uploading k, v, s."""
        import paged_quantized_kv_write_gb300 as pkv
        w = case.w
        self.case, self.w, self.pkv = case, w, pkv
        self.q = bits_to_tensor(case.q, w.q_dtype)
        if device_cache is not None:
            self.k, self.v, self.s = device_cache
        else:
            self.k, self.v, self.s = cache_to_device(k, v, s, w.kv_dtype)
        self.tables = torch.from_numpy(case.block_tables).cuda()
        self.ctx = torch.from_numpy(case.context_lens).cuda()
        self.out = torch.empty_like(self.q)
        self.partition_size = partition_size
        self.ws = pkv.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                     case.max_blocks_per_seq, w.block_size, partition_size)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def attend(self, ctx=None, tables=None):
        w = self.w
        self.pkv.paged_decode_attention(
            self.q, self.k, self.v, self.tables if tables is None else tables,
            self.ctx if ctx is None else ctx, self.s, self.out, w.softmax_scale,
            w.num_kv_heads, w.kv_dtype, w.block_size, self.partition_size, self.ws, self.status)
        torch.cuda.synchronize()
        return tensor_to_f64(self.out)


def oracle_attention(case: W.Case, k, v, s, ctx=None, tables=None) -> np.ndarray:
    w = case.w
    return oracle.decode_attention(case.q, w.q_dtype, k, v,
                                   case.block_tables if tables is None else tables,
                                   case.context_lens if ctx is None else ctx, s, w.kv_dtype,
                                   case.num_blocks, w.softmax_scale, w.num_q_heads,
                                   w.num_kv_heads, w.head_dim, w.block_size)


def workload(cfg):
    """A benchmark workload by number; "3-e5m2" / "3-int8" are workload 3 with an E5M2 /
    INT8 cache."""
    if cfg == "3-e5m2":
        return W.CONFIGS[3].scaled(kv_dtype=W.FP8_E5M2, name="FP8 E5M2 KV with quantize-on-write")
    if cfg == "3-int8":
        return W.CONFIGS[3].scaled(kv_dtype=W.INT8, name="INT8 KV with quantize-on-write")
    return W.CONFIGS[cfg]


def seed_of(cfg) -> int:
    """A fixed small integer per workload name (for seeding its scaled variants)."""
    return cfg if isinstance(cfg, int) else {"3-e5m2": 6, "3-int8": 8}[cfg]
