"""Seeded synthetic inputs for paged, quantized KV-cache decode.

This module stands in for the block manager and the model that feed the
kernels.  It draws random queries, keys and values, picks context lengths,
lays out a physical block pool with shuffled block tables and derives the
slot mapping of every token that must be written.  It holds none of the
method's arithmetic: no quantisation, no dequantisation, no attention.  Both
the CUDA path and the CPU oracle consume what it produces.

Address translation used for slot mappings is the block manager's job
("Reducing LLM Inference Latency ... PagedAttention in vLLM", snippet-3,
``get_physical_address``): ``slot = table[t // bs] * bs + t % bs``.

Workloads (shapes, dtypes and distributions of the pages' Llama-3-8B/70B
decode layers, plus a tiny case):

1. tiny: B=4, 8 q heads, 2 KV heads, D=64, bs=16, f16, ctx ~ U[1,128],
   pool of 64 blocks.
2. Llama-3-8B-shaped layer, bf16 KV: B=64, 32/8 heads, D=128, bs=16,
   every ctx 4096, pool = needed blocks + 10%.
3. FP8 E4M3 KV with quantize-on-write: B=128, 32/8, D=128, bs=16, ctx
   log-normal (median 2048, sigma 0.5) clipped to [256, 8192], 1% of K/V
   elements scaled by 20.
4. Llama-3-70B-shaped layer, INT4 KV: B=128, 64/8, D=128, bs=32, ctx ~
   U[1024, 8192]; the first 1024 tokens of every sequence live in the same
   32 physical blocks (shared prefix).
5. Long-context split-KV, FP8 KV: B=16, 64/8, D=128, bs=16, every ctx
   32768, partitions of 512 tokens.

Every workload is one decode step: the context holds ``ctx_b - 1`` tokens
written beforehand ("prefill"), the step writes token ``ctx_b - 1`` (the
new token) and then attends over all ``ctx_b`` tokens.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np

# dtype tags shared by the C ABI and the oracle (plain integers).
F16, BF16, FP8_E4M3, INT4_G32, FP8_E5M2, INT8 = 0, 1, 2, 3, 4, 5
DTYPE_NAMES = {F16: "f16", BF16: "bf16", FP8_E4M3: "fp8_e4m3", INT4_G32: "int4_g32",
               FP8_E5M2: "fp8_e5m2", INT8: "int8"}
FP8_TYPES = (FP8_E4M3, FP8_E5M2)
BLK8_TYPES = (FP8_E4M3, FP8_E5M2, INT8)      # one byte per element, one fp32 scale per block


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: int
    q_dtype: int                   # also the dtype of k_new/v_new and out
    ctx_kind: str                  # "uniform" | "fixed" | "lognormal"
    ctx_lo: int
    ctx_hi: int
    ctx_median: int = 0
    ctx_sigma: float = 0.0
    outlier_prob: float = 0.0
    outlier_scale: float = 1.0
    shared_prefix_tokens: int = 0
    pool_blocks: int = 0           # 0 -> needed blocks + 10% spare
    partition_size: int = 0        # 0 -> library heuristic
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def scaled(self, batch: Optional[int] = None, ctx_cap: Optional[int] = None,
               seed: Optional[int] = None, **kw) -> "Workload":
        """A smaller variant with the same heads, head_dim, block size and dtypes.

        ``ctx_cap`` caps the context-length distribution (and the shared prefix).
        """
        upd = dict(kw)
        if batch is not None:
            upd["batch"] = batch
        if seed is not None:
            upd["seed"] = seed
        if ctx_cap is not None:
            lo = min(self.ctx_lo, ctx_cap)
            upd.update(ctx_lo=max(1, lo), ctx_hi=min(self.ctx_hi, ctx_cap),
                       ctx_median=min(self.ctx_median, ctx_cap))
            if self.shared_prefix_tokens:
                bs = self.block_size
                sp = min(self.shared_prefix_tokens, (max(1, lo) // bs) * bs)
                upd["shared_prefix_tokens"] = sp
        if self.pool_blocks and "pool_blocks" not in upd and (batch or ctx_cap):
            upd["pool_blocks"] = 0
        return dataclasses.replace(self, **upd)


CONFIGS: Dict[int, Workload] = {
    1: Workload("tiny paged decode", 4, 8, 2, 64, 16, F16, F16, "uniform", 1, 128,
                pool_blocks=64, seed=1001),
    2: Workload("Llama-3-8B-shaped decode, bf16 KV", 64, 32, 8, 128, 16, BF16, BF16,
                "fixed", 4096, 4096, seed=1002),
    3: Workload("FP8 E4M3 KV with quantize-on-write", 128, 32, 8, 128, 16, FP8_E4M3, BF16,
                "lognormal", 256, 8192, ctx_median=2048, ctx_sigma=0.5,
                outlier_prob=0.01, outlier_scale=20.0, seed=1003),
    4: Workload("Llama-3-70B-shaped decode, INT4 KV, shared prefix", 128, 64, 8, 128, 32,
                INT4_G32, BF16, "uniform", 1024, 8192, shared_prefix_tokens=1024, seed=1004),
    5: Workload("long-context split-KV decode, FP8 KV", 16, 64, 8, 128, 16, FP8_E4M3, BF16,
                "fixed", 32768, 32768, partition_size=512, seed=1005),
}


# ---------------------------------------------------------------- dtype casts
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 values to the 16-bit dtype ``dtype`` and return raw uint16 bits."""
    if dtype == F16:
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)
    if dtype == BF16:
        return f32_to_bf16_bits(x)
    raise ValueError(f"not a 16-bit float dtype: {dtype}")


def bits_to_f32(b: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F16:
        return b.view(np.float16).astype(np.float32)
    if dtype == BF16:
        return bf16_bits_to_f32(b)
    raise ValueError(f"not a 16-bit float dtype: {dtype}")


# ---------------------------------------------------------- pool geometry
def cache_shapes(w: Workload, num_blocks: int):
    """Shapes (numpy dtype, shape) of k_cache/v_cache and of the scales buffer.

    Layout per KV tensor: [num_blocks, num_kv_heads, block_size, row] where a
    row is D 16-bit values, D bytes (FP8) or D/2 bytes (INT4, two codes per
    byte).  Scales: FP8 f32 [2, num_blocks, num_kv_heads]; INT4 f16
    [2, num_blocks, num_kv_heads, block_size, D/32, 2] (scale, zero); none for
    16-bit caches.  Index 0 of the leading 2 is K, 1 is V.
    """
    nb, h, bs, d = num_blocks, w.num_kv_heads, w.block_size, w.head_dim
    if w.kv_dtype in (F16, BF16):
        return (np.uint16, (nb, h, bs, d)), None
    if w.kv_dtype in BLK8_TYPES:
        return (np.uint8, (nb, h, bs, d)), (np.float32, (2, nb, h))
    if w.kv_dtype == INT4_G32:
        return (np.uint8, (nb, h, bs, d // 2)), (np.uint16, (2, nb, h, bs, d // 32, 2))
    raise ValueError(w.kv_dtype)


def slots_for(table_row: np.ndarray, positions: np.ndarray, block_size: int) -> np.ndarray:
    """Block-manager address translation: token position -> flat slot index."""
    positions = np.asarray(positions, dtype=np.int64)
    return table_row[positions // block_size].astype(np.int64) * block_size + positions % block_size


def draw_context_lens(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.ctx_kind == "fixed":
        return np.full(w.batch, w.ctx_hi, dtype=np.int32)
    if w.ctx_kind == "uniform":
        return rng.integers(w.ctx_lo, w.ctx_hi + 1, size=w.batch).astype(np.int32)
    if w.ctx_kind == "lognormal":
        x = np.exp(rng.normal(math.log(w.ctx_median), w.ctx_sigma, size=w.batch))
        return np.clip(np.rint(x), w.ctx_lo, w.ctx_hi).astype(np.int32)
    raise ValueError(w.ctx_kind)


def build_tables(w: Workload, ctx: np.ndarray, rng: np.random.Generator,
                 identity: bool = False, max_blocks_per_seq: Optional[int] = None):
    """Block tables over a shuffled pool; unused entries are -1.

    With a shared prefix, logical blocks [0, prefix/bs) of every sequence map
    to the same physical blocks.  ``identity`` lays every sequence out in
    consecutive physical blocks (the contiguous-cache comparator).
    """
    bs = w.block_size
    nblk = (ctx.astype(np.int64) + bs - 1) // bs
    shared = w.shared_prefix_tokens // bs
    needed = int(shared + np.maximum(nblk - shared, 0).sum())
    num_blocks = w.pool_blocks if w.pool_blocks else int(math.ceil(1.1 * needed))
    if num_blocks < needed:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {needed}")
    mb = int(nblk.max()) if max_blocks_per_seq is None else max_blocks_per_seq
    perm = rng.permutation(num_blocks)          # drawn in both cases: same stream after
    order = np.arange(num_blocks, dtype=np.int64) if identity else perm
    tables = np.full((w.batch, max(mb, 1)), -1, dtype=np.int32)
    nxt = 0
    shared_ids = order[:shared]
    nxt = shared
    for b in range(w.batch):
        n = int(nblk[b])
        s = min(shared, n)
        tables[b, :s] = shared_ids[:s]
        own = n - s
        tables[b, s:n] = order[nxt:nxt + own]
        nxt += own
    return tables, num_blocks


@dataclasses.dataclass
class Case:
    """One decode step's inputs (host numpy arrays, raw bits for 16-bit floats)."""
    w: Workload
    context_lens: np.ndarray       # int32 [B] (includes the new token)
    block_tables: np.ndarray       # int32 [B, max_blocks_per_seq]
    num_blocks: int
    q: np.ndarray                  # uint16 [B, Hq, D] in q_dtype
    # prefill tokens: every context token but the last of each sequence
    prefill_slots: np.ndarray      # int64 [T]
    prefill_k: np.ndarray          # uint16 [T, Hkv, D] in q_dtype
    prefill_v: np.ndarray
    # the step's new token (position ctx-1) per sequence; slot -1 = already present
    new_slots: np.ndarray          # int64 [B]
    k_new: np.ndarray              # uint16 [B, Hkv, D]
    v_new: np.ndarray

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_tables.shape[1]


def _kv_values(w: Workload, rng: np.random.Generator, n: int) -> np.ndarray:
    x = rng.standard_normal((n, w.num_kv_heads, w.head_dim), dtype=np.float32)
    if w.outlier_prob > 0:
        mask = rng.random(x.shape, dtype=np.float32) < w.outlier_prob
        x[mask] *= np.float32(w.outlier_scale)
    return to_bits(x, w.q_dtype)


def make_case(w: Workload, identity_tables: bool = False,
              max_blocks_per_seq: Optional[int] = None, prefill_values: bool = True) -> Case:
    """Draw one decode step for workload ``w`` (deterministic in ``w.seed``).

    ``prefill_values=False`` leaves ``prefill_k``/``prefill_v`` as None (a
    caller that draws them on the device with ``draw_kv_device``); everything
    else is drawn as usual, though k_new/v_new then take other values of the
    same distribution (the host stream skips the prefill draws)."""
    rng = np.random.default_rng(w.seed)
    ctx = draw_context_lens(w, rng)
    tables, num_blocks = build_tables(w, ctx, rng, identity_tables, max_blocks_per_seq)
    q = to_bits(rng.standard_normal((w.batch, w.num_q_heads, w.head_dim), dtype=np.float32),
                w.q_dtype)
    bs = w.block_size
    sp = w.shared_prefix_tokens
    slot_parts = []
    # shared prefix tokens are written once (their values are common to all sequences)
    if sp:
        first = int(np.argmax(ctx >= 1))
        slot_parts.append(slots_for(tables[first], np.arange(sp), bs))
    for b in range(w.batch):
        lo = sp if sp else 0
        hi = int(ctx[b]) - 1
        if hi > lo:
            slot_parts.append(slots_for(tables[b], np.arange(lo, hi), bs))
    prefill_slots = (np.concatenate(slot_parts) if slot_parts
                     else np.zeros(0, dtype=np.int64)).astype(np.int64)
    prefill_k = _kv_values(w, rng, len(prefill_slots)) if prefill_values else None
    prefill_v = _kv_values(w, rng, len(prefill_slots)) if prefill_values else None
    new_pos = ctx.astype(np.int64) - 1
    new_slots = np.full(w.batch, -1, dtype=np.int64)
    for b in range(w.batch):
        if ctx[b] >= 1 and new_pos[b] >= sp:
            new_slots[b] = slots_for(tables[b], new_pos[b:b + 1], bs)[0]
    k_new = _kv_values(w, rng, w.batch)
    v_new = _kv_values(w, rng, w.batch)
    return Case(w, ctx, tables, num_blocks, q, prefill_slots, prefill_k, prefill_v,
                new_slots, k_new, v_new)


def draw_kv_device(w: Workload, n: int, seed: int, device, chunk: int = 1 << 18):
    """K or V rows of ``n`` tokens drawn on a CUDA device with the workload's
    distribution (N(0,1), each element times ``outlier_scale`` with probability
    ``outlier_prob``, rounded to the 16-bit dtype): the same recipe as the host
    draws, from torch's seeded generator, for benchmarks whose host draws would
    take longer than the measurement.  Returns a [n, Hkv, D] tensor of w.q_dtype."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.float16 if w.q_dtype == F16 else torch.bfloat16
    out = torch.empty((n, w.num_kv_heads, w.head_dim), dtype=dt, device=device)
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        x = torch.randn((m, w.num_kv_heads, w.head_dim), generator=g, device=device,
                        dtype=torch.float32)
        if w.outlier_prob > 0:
            mask = torch.rand(x.shape, generator=g, device=device) < w.outlier_prob
            x = torch.where(mask, x * w.outlier_scale, x)
        out[i:i + m] = x.to(dt)
    return out


def prefill_chunk(case: Case, chunk_lens, seed: int = 0):
    """Queries for a chunked-prefill step over ``case``'s cache.

    ``chunk_lens[b]`` new query tokens per sequence (their K/V are the last
    ``chunk_lens[b]`` context tokens, already in the case's cache once the
    decode step's new token is written).  Returns (q bits [sum n, Hq, D] in
    the query dtype, q_start int32 [B + 1]).
    """
    w = case.w
    n = np.asarray(chunk_lens, dtype=np.int64)
    q_start = np.zeros(w.batch + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(n)
    rng = np.random.default_rng(10_000 + w.seed * 7 + seed)
    q = to_bits(rng.standard_normal((int(q_start[-1]), w.num_q_heads, w.head_dim),
                                    dtype=np.float32), w.q_dtype)
    return q, q_start


def prefill_workload():
    """Chunked-prefill benchmark workload: workload 2's Llama-3-8B-shaped bf16 layer
    (32/8 heads, D 128, bs 16, 4096-token contexts) for 8 sequences, each of which
    brings a chunk of its last 512 tokens.  Returns (workload, chunk length)."""
    return CONFIGS[2].scaled(batch=8, seed=2002), 512


def prefill_flops(context_lens, chunk_lens, num_q_heads: int, head_dim: int) -> int:
    """Multiply-adds x 2 of a chunked-prefill step: QK^T and PV over each query's
    causal range (query j of a chunk of n over c tokens sees c - n + j + 1)."""
    total = 0
    for c, n in zip(np.asarray(context_lens, np.int64), np.asarray(chunk_lens, np.int64)):
        first = max(0, int(c) - int(n))
        seen = int(n) * (first + 1) + int(n) * (int(n) - 1) // 2      # sum over j of first + j + 1
        total += seen
    return 4 * total * num_q_heads * head_dim


def algorithmic_bytes(case: Case, unique: bool = True) -> int:
    """Bytes one decode step must move at minimum (attention + the write).

    KV codes of every context token (shared-prefix blocks once if ``unique``),
    their scales, q, the block-table entries in use, context_lens, out, and
    the write's new K/V in, slot_mapping in and codes (+ scales) out.
    """
    w = case.w
    h, d, bs = w.num_kv_heads, w.head_dim, w.block_size
    ctx = case.context_lens.astype(np.int64)
    tokens = int(ctx.sum())
    if unique and w.shared_prefix_tokens:
        sp = w.shared_prefix_tokens
        tokens = tokens - int(np.minimum(ctx, sp).sum()) + int(min(sp, ctx.max()))
    if w.kv_dtype in (F16, BF16):
        per_tok_head = 2 * d
        scale_bytes = 0
    elif w.kv_dtype in BLK8_TYPES:
        per_tok_head = d
        nblk = (ctx + bs - 1) // bs
        if unique and w.shared_prefix_tokens:
            s = w.shared_prefix_tokens // bs
            blocks = int(nblk.sum() - np.minimum(nblk, s).sum() + s)
        else:
            blocks = int(nblk.sum())
        scale_bytes = blocks * h * 2 * 4
    else:
        per_tok_head = d // 2 + (d // 32) * 4
        scale_bytes = 0
    kv = 2 * tokens * h * per_tok_head + scale_bytes
    qb = w.batch * w.num_q_heads * d * 2
    table = int(((ctx + bs - 1) // bs).sum()) * 4
    out = qb
    nwrite = int((case.new_slots >= 0).sum())
    write_in = 2 * nwrite * h * d * 2 + w.batch * 8
    if w.kv_dtype in (F16, BF16):
        write_out = 2 * nwrite * h * d * 2
    elif w.kv_dtype in BLK8_TYPES:
        write_out = 2 * nwrite * h * d + 2 * nwrite * h * 4
    else:
        write_out = 2 * nwrite * h * (d // 2 + (d // 32) * 4)
    return kv + qb + table + w.batch * 4 + out + write_in + write_out


def attention_bytes(case: Case, unique: bool = True) -> int:
    """Algorithmic bytes of the attention call alone (no write)."""
    w = case.w
    total = algorithmic_bytes(case, unique)
    h, d = w.num_kv_heads, w.head_dim
    nwrite = int((case.new_slots >= 0).sum())
    write_in = 2 * nwrite * h * d * 2 + w.batch * 8
    if w.kv_dtype in (F16, BF16):
        write_out = 2 * nwrite * h * d * 2
    elif w.kv_dtype in BLK8_TYPES:
        write_out = 2 * nwrite * h * d + 2 * nwrite * h * 4
    else:
        write_out = 2 * nwrite * h * (d // 2 + (d // 32) * 4)
    return total - write_in - write_out
