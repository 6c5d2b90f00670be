"""Seeded random cases across the whole parameter space, every kernel path,
against the oracle: decode (every work split and comparator, with and without
the fused write, split or whole partitions) and chunked prefill (tcgen05 and
mma.sync).  Each case draws its dtype, GQA group, head_dim, block size
(including ones that are not powers of two), batch, context mix, partition
size and outliers from a fixed seed, so a failure names a reproducible case."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu

KV_TYPES = [W.F16, W.BF16, W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32]
DECODE_MODES = ["default", "shared", "warp", "balanced", "simt", "tc"]


def _draw(seed: int, max_ctx=(17, 100, 700, 2000)):
    rng = np.random.default_rng(70_000 + seed)
    kv = KV_TYPES[rng.integers(len(KV_TYPES))]
    qd = kv if kv in (W.F16, W.BF16) else (W.F16 if rng.random() < 0.3 else W.BF16)
    head_dim = int(rng.choice([64, 128]))
    group = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    block_size = int(rng.choice([16, 32, 48, 64, 128, 256]))
    batch = int(rng.integers(1, 7))
    hi = int(rng.choice(max_ctx))
    outliers = rng.random() < 0.5
    w = W.Workload(f"fuzz{seed}", batch, group * hkv, hkv, head_dim, block_size, kv, qd,
                   "uniform", 1, hi, outlier_prob=0.01 if outliers else 0.0,
                   outlier_scale=20.0, seed=seed)
    partition = int(rng.choice([0, 16, 64, 256]))
    return w, partition, rng


@pytest.mark.parametrize("seed", range(100))
def test_fuzz_decode(seed, monkeypatch):
    import paged_quantized_kv_write_gb300 as pkv
    w, partition, rng = _draw(seed)
    mode = DECODE_MODES[seed % len(DECODE_MODES)]
    fused = bool(rng.random() < 0.5)
    if mode != "default":
        monkeypatch.setenv("PKV_DECODE_MODE", mode)
    else:
        monkeypatch.delenv("PKV_DECODE_MODE", raising=False)
    with H.library_for(mode):                   # the comparators are in the test build
        _fuzz_decode_case(pkv, seed, w, partition, mode, fused)


def _fuzz_decode_case(pkv, seed, w, partition, mode, fused):
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    g = H.GpuCase(case, k, v, s, partition)
    if fused:
        pkv.paged_decode_attention_with_write(
            g.q, H.bits_to_tensor(case.k_new, w.q_dtype), H.bits_to_tensor(case.v_new, w.q_dtype),
            torch.from_numpy(case.new_slots).cuda(), g.k, g.v, g.tables, g.ctx, g.s, g.out,
            w.softmax_scale, w.kv_dtype, w.block_size, partition, g.ws, g.status)
    else:
        pkv.paged_kv_write(H.bits_to_tensor(case.k_new, w.q_dtype),
                           H.bits_to_tensor(case.v_new, w.q_dtype),
                           torch.from_numpy(case.new_slots).cuda(), g.k, g.v, g.s, w.kv_dtype,
                           w.block_size, w.head_dim, g.status)
        g.attend()
    torch.cuda.synchronize()
    out = H.tensor_to_f64(g.out)
    ref = oracle.step_case(case, k, v, s)
    gk, gv, gs = H.cache_to_host(g.k, g.v, g.s, w.kv_dtype)
    what = (f"seed {seed}: kv {W.DTYPE_NAMES[w.kv_dtype]} q {W.DTYPE_NAMES[w.q_dtype]} "
            f"D {w.head_dim} {w.num_q_heads}/{w.num_kv_heads} bs {w.block_size} B {w.batch} "
            f"partition {partition} mode {mode} fused {fused}")
    assert np.array_equal(gk, k) and np.array_equal(gv, v), f"{what}: cache bytes differ"
    if s is not None:
        assert np.array_equal(gs.view(np.uint8), s.view(np.uint8)), f"{what}: scales differ"
    assert g.status.item() == 0, what
    H.check_close(out, ref, w.kv_dtype, w.q_dtype, what)


@pytest.mark.parametrize("seed", range(48))
def test_fuzz_prefill(seed, monkeypatch):
    import paged_quantized_kv_write_gb300 as pkv
    w, _, rng = _draw(1000 + seed, max_ctx=(40, 300, 900))
    mode = "mma" if seed % 3 == 2 else "default"
    if mode == "mma":
        monkeypatch.setenv("PKV_PREFILL_MODE", "mma")
    else:
        monkeypatch.delenv("PKV_PREFILL_MODE", raising=False)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    # chunk of each sequence: anything from one token to the whole context
    chunk = [int(rng.integers(1, int(c) + 1)) for c in case.context_lens]
    q, q_start = W.prefill_chunk(case, chunk, seed)
    kd, vd, sd = H.cache_to_device(k, v, s, w.kv_dtype)
    qt = H.bits_to_tensor(q, w.q_dtype)
    out = torch.full_like(qt, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_prefill_attention(qt, torch.from_numpy(q_start).cuda(), kd, vd,
                                torch.from_numpy(case.block_tables).cuda(),
                                torch.from_numpy(case.context_lens).cuda(), sd, out,
                                w.softmax_scale, w.num_kv_heads, w.kv_dtype, w.block_size,
                                max(chunk), status)
    torch.cuda.synchronize()
    ref = oracle.prefill_attention(q, w.q_dtype, q_start, k, v, case.block_tables,
                                   case.context_lens, s, w.kv_dtype, case.num_blocks,
                                   w.softmax_scale, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                   w.block_size)
    what = (f"seed {seed}: kv {W.DTYPE_NAMES[w.kv_dtype]} q {W.DTYPE_NAMES[w.q_dtype]} "
            f"D {w.head_dim} {w.num_q_heads}/{w.num_kv_heads} bs {w.block_size} B {w.batch} "
            f"chunks {chunk} mode {mode}")
    assert status.item() == 0, what
    H.check_close(H.tensor_to_f64(out), ref, w.kv_dtype, w.q_dtype, what)
