"""Shared helpers for the GPU parity tests: upload a case, run the library,
compare with the oracle under the stated tolerances."""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads as W

# max-abs tolerances on the attention output: 2e-3 for 16-bit KV, 5e-3 for
# FP8/INT4 against the oracle on the same dequantized values.
TOL = {W.F16: 2e-3, W.BF16: 2e-3, W.FP8_E4M3: 5e-3, W.INT4_G32: 5e-3, W.FP8_E5M2: 5e-3,
       W.INT8: 5e-3}


def library_for(decode_mode: str):
    """The library build a decode mode runs in: the comparators ("simt", "tc") are in
    the test build only; everything else runs the product library."""
    import paged_quantized_kv_write_gb300 as pkv
    return pkv.library("test" if decode_mode in ("simt", "tc") else "product")


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


def _ulp(x: np.ndarray, code: int) -> np.ndarray:
    """Spacing of the 16-bit output dtype in the binade of |x| (subnormal spacing
    below the smallest normal)."""
    mant, emin = (10, -14) if code == W.F16 else (7, -126)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, emin), emin)
    return 2.0 ** (e - mant)


def round_down(x: np.ndarray, code: int) -> np.ndarray:
    """x rounded toward -inf to the 16-bit output dtype (as fp64).  Multiples of the
    binade's spacing, and the binade's ends, are all representable."""
    u = _ulp(x, code)
    return np.floor(x / u) * u


def round_up(x: np.ndarray, code: int) -> np.ndarray:
    """x rounded toward +inf to the 16-bit output dtype (as fp64)."""
    u = _ulp(x, code)
    return np.ceil(x / u) * u


def round_to(x: np.ndarray, code: int) -> np.ndarray:
    """fp64 values rounded (nearest even) to the 16-bit output dtype, back as fp64."""
    if code == W.F16:
        return x.astype(np.float16).astype(np.float64)
    return W.bits_to_f32(W.f32_to_bf16_bits(x.astype(np.float32)), W.BF16).astype(np.float64)


def check_close(gpu: np.ndarray, ref: np.ndarray, kv_dtype: int, out_dtype: int, what=""):
    """Assert that each output is within the tolerance of the oracle before its
    final rounding: gpu in [round_down(oracle - tol), round_up(oracle + tol)], both
    ends rounded in the output dtype (tol: 2e-3 for 16-bit KV, 5e-3 for FP8/INT4).
    A result computed within tol of the oracle lands there whatever its magnitude,
    and nothing farther does.

    Returns (max |gpu - oracle|, max |gpu - oracle rounded to the output dtype|,
    the share of tol the worst output needs: the smallest t / tol for which
    gpu lies in [round_down(oracle - t), round_up(oracle + t)], <= 1)."""
    tol = TOL[kv_dtype]
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    lo = round_down(ref - tol, out_dtype)
    hi = round_up(ref + tol, out_dtype)
    bad = ~((gpu >= lo) & (gpu <= hi))
    if bad.any():
        over = np.where(gpu > hi, gpu - hi, np.where(gpu < lo, lo - gpu, 0.0))
        over = np.where(np.isnan(gpu), np.inf, over)
        i = np.unravel_index(np.argmax(over), over.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {gpu.size} outputs outside the tolerance; worst at "
            f"{i}: gpu {gpu[i]!r} oracle {ref[i]!r} err {abs(gpu[i] - ref[i]):.3g} allowed "
            f"[{lo[i]!r}, {hi[i]!r}]")
    if not gpu.size:
        return 0.0, 0.0, 0.0
    err = np.abs(gpu - ref)
    # an output above the oracle needs t past the representable value just below it
    # (below the oracle: past the one just above it); one equal to the oracle's own
    # rounding needs nothing
    below = round_down(np.nextafter(gpu, -np.inf), out_dtype)
    above = round_up(np.nextafter(gpu, np.inf), out_dtype)
    need = np.where(gpu > ref, np.maximum(0.0, below - ref),
                    np.where(gpu < ref, np.maximum(0.0, ref - above), 0.0))
    err_r = np.abs(gpu - round_to(ref, out_dtype))
    return float(err.max()), float(err_r.max()), float(need.max() / tol)


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

    def attend(self, ctx=None, tables=None, scale=None):
        w = self.w
        self.pkv.paged_decode_attention(
            self.q, self.k, self.v, self.tables if tables is None else tables,
            self.ctx if ctx is None else ctx, self.s, self.out,
            w.softmax_scale if scale is None else scale,
            w.num_kv_heads, w.kv_dtype, w.block_size, self.partition_size, self.ws, self.status)
        torch.cuda.synchronize()
        return tensor_to_f64(self.out)


def oracle_attention(case: W.Case, k, v, s, ctx=None, tables=None, scale=None) -> np.ndarray:
    w = case.w
    return oracle.decode_attention(case.q, w.q_dtype, k, v,
                                   case.block_tables if tables is None else tables,
                                   case.context_lens if ctx is None else ctx, s, w.kv_dtype,
                                   case.num_blocks, w.softmax_scale if scale is None else scale,
                                   w.num_q_heads,
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
