"""GPU parity of paged_prefill_attention (chunked prefill over the paged cache)
against the fp64 oracle: every query attends causally up to its position."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _pkv():
    import paged_quantized_kv_write_gb300 as pkv
    return pkv


def _full_cache(case):
    w = case.w
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    return k, v, s


def _run(case, chunk, max_query_len=None, seed=0, ctx=None, tables=None, oracle_ref=True,
         scale=None):
    """GPU and oracle prefill for the given chunk lengths; returns (gpu, ref, status, q_start)
    (ref None without oracle_ref).  `tables` replaces the case's block tables on the GPU;
    `scale` replaces the softmax scale 1/sqrt(head_dim) on both sides."""
    pkv = _pkv()
    w = case.w
    scale = w.softmax_scale if scale is None else scale
    k, v, s = _full_cache(case)
    q, q_start = W.prefill_chunk(case, chunk, seed)
    ctx = case.context_lens if ctx is None else ctx
    kd, vd, sd = H.cache_to_device(k, v, s, w.kv_dtype)
    qt = H.bits_to_tensor(q, w.q_dtype)
    out = torch.full_like(qt, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mql = int(max(chunk)) if max_query_len is None else max_query_len
    pkv.paged_prefill_attention(qt, torch.from_numpy(q_start).cuda(), kd, vd,
                                torch.from_numpy(case.block_tables if tables is None
                                                 else tables).cuda(),
                                torch.from_numpy(np.ascontiguousarray(ctx, np.int32)).cuda(),
                                sd, out, scale, w.num_kv_heads, w.kv_dtype,
                                w.block_size, mql, status)
    torch.cuda.synchronize()
    ref = None
    if oracle_ref:
        ref = oracle.prefill_attention(q, w.q_dtype, q_start, k, v, case.block_tables, ctx, s,
                                       w.kv_dtype, case.num_blocks, scale,
                                       w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size)
    return H.tensor_to_f64(out), ref, status.item(), q_start


@pytest.fixture(params=["default", "mma"])
def pf_mode(request, monkeypatch):
    """default: the warp-role tcgen05 kernel for every cache dtype; mma: the
    mma.sync kernel for every call."""
    if request.param == "mma":
        monkeypatch.setenv("PKV_PREFILL_MODE", "mma")
    else:
        monkeypatch.delenv("PKV_PREFILL_MODE", raising=False)
    return request.param


@pytest.mark.parametrize("kv", [W.F16, W.BF16, W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (16, 2)])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_prefill_dtypes_groups_dims(kv, hq, hkv, head_dim, pf_mode):
    qd = W.F16 if kv == W.F16 else W.BF16
    w = W.Workload("pf", 4, hq, hkv, head_dim, 16, kv, qd, "uniform", 40, 260,
                   outlier_prob=0.01, outlier_scale=20.0, seed=hq + hkv + head_dim + 3 * kv)
    case = W.make_case(w)
    chunk = [int(min(c, n)) for c, n in zip(case.context_lens, [1, 17, 40, 130])]
    gpu, ref, st, _ = _run(case, chunk)
    assert st == 0
    H.check_close(gpu, ref, kv, qd, f"prefill kv {kv} {hq}/{hkv} D {head_dim}")


@pytest.mark.parametrize("kv", [W.F16, W.BF16, W.FP8_E4M3, W.INT4_G32])
def test_prefill_negative_softmax_scale(kv, pf_mode):
    """A negative softmax scale makes each row's smallest score its largest
    scaled one: tiles below every causal limit take the row's minimum, the
    masked tiles their scaled maximum."""
    qd = W.F16 if kv == W.F16 else W.BF16
    w = W.Workload("pfneg", 3, 32, 8, 128, 16, kv, qd, "uniform", 200, 700,
                   outlier_prob=0.01, outlier_scale=20.0, seed=77 + kv)
    case = W.make_case(w)
    chunk = [int(min(c, n)) for c, n in zip(case.context_lens, [1, 150, 300])]
    gpu, ref, st, _ = _run(case, chunk, scale=-w.softmax_scale)
    assert st == 0
    H.check_close(gpu, ref, kv, qd, f"prefill negative scale, kv {kv}")


@pytest.mark.parametrize("kv", [W.FP8_E4M3, W.FP8_E5M2, W.INT8])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 8), (64, 8)])
def test_prefill_one_byte_cache_with_f16_queries(kv, hq, hkv, pf_mode):
    """f16 queries over one-byte caches (the bf16-query cases are above), with
    ragged chunks that leave partial tiles and whole-context chunks."""
    w = W.Workload("pf16", 3, hq, hkv, 128, 16, kv, W.F16, "uniform", 60, 330,
                   outlier_prob=0.01, outlier_scale=20.0, seed=31 + hq + 7 * kv)
    case = W.make_case(w)
    chunk = [int(min(c, n)) for c, n in zip(case.context_lens, [5, 64, 400])]
    gpu, ref, st, _ = _run(case, chunk)
    assert st == 0
    H.check_close(gpu, ref, kv, W.F16, f"prefill f16 q, kv {kv} {hq}/{hkv}")


@pytest.mark.parametrize("kv", [W.BF16, W.FP8_E4M3, W.INT4_G32])
@pytest.mark.parametrize("block_size", [16, 32, 64, 128])
def test_prefill_block_sizes_and_whole_context_chunks(kv, block_size):
    """Chunks covering the whole context (a full prefill) and ragged ones."""
    w = W.Workload("pf", 3, 32, 8, 128, block_size, kv, W.BF16, "uniform", 1, 700,
                   seed=block_size + kv)
    case = W.make_case(w)
    chunk = [int(case.context_lens[0]), max(1, int(case.context_lens[1]) // 3), 1]
    gpu, ref, st, _ = _run(case, chunk)
    assert st == 0
    H.check_close(gpu, ref, kv, W.BF16, f"prefill bs {block_size}")


def test_prefill_chunk_of_one_matches_decode():
    pkv = _pkv()
    w = W.CONFIGS[3].scaled(batch=6, ctx_cap=400, seed=321)
    case = W.make_case(w)
    gpu, ref, st, _ = _run(case, [1] * w.batch)
    assert st == 0
    H.check_close(gpu, ref, w.kv_dtype, w.q_dtype, "chunk of one")
    # against the decode kernel on the same queries
    k, v, s = _full_cache(case)
    q, _ = W.prefill_chunk(case, [1] * w.batch)
    dcase = W.Case(**{**case.__dict__})
    dcase.q = q
    g = H.GpuCase(dcase, k, v, s, 0)
    dec = g.attend()
    H.check_close(gpu, dec, w.kv_dtype, w.q_dtype, "prefill vs decode")


EDGE_KERNELS = [(W.BF16, 64), (W.BF16, 128), (W.FP8_E4M3, 128), (W.INT8, 128)]


@pytest.mark.parametrize("kv,head_dim", EDGE_KERNELS)
def test_prefill_chunk_longer_than_context_is_flagged_and_zero(kv, head_dim):
    pkv = _pkv()
    w = W.Workload("pf", 2, 8, 2, head_dim, 16, kv, W.BF16, "fixed", 6, 6, seed=4)
    case = W.make_case(w)
    gpu, ref, st, _ = _run(case, [9, 3])
    assert st == pkv.PKV_ERR_DEVICE_BOUNDS
    assert not gpu[:3].any()                       # queries at positions -3..-1
    H.check_close(gpu, ref, kv, W.BF16, "long chunk")


@pytest.mark.parametrize("kv,head_dim", EDGE_KERNELS)
def test_prefill_max_query_len_bounds_the_grid(kv, head_dim):
    w = W.Workload("pf", 2, 8, 2, head_dim, 16, kv, W.BF16, "fixed", 100, 100, seed=5)
    case = W.make_case(w)
    gpu, ref, st, q_start = _run(case, [40, 10], max_query_len=16)
    assert st == 0
    computed = np.r_[0:16, 40:50]
    H.check_close(gpu[computed], ref[computed], kv, W.BF16, "bounded")
    assert np.isnan(gpu[16:40]).all()              # beyond max_query_len: not written


@pytest.mark.parametrize("kv,head_dim", EDGE_KERNELS + [(W.INT4_G32, 128)])
def test_prefill_bad_block_id_is_flagged_and_skipped(kv, head_dim, monkeypatch):
    """A block id outside the pool in one sequence's table (tokens 32..47 of
    sequence 1): the call flags PKV_ERR_DEVICE_BOUNDS, the other sequences
    match the oracle, and sequence 1 matches the mma.sync path, which leaves
    that block's tokens out in the same way."""
    pkv = _pkv()
    w = W.Workload("pfbad", 3, 8, 2, head_dim, 16, kv, W.BF16, "fixed", 200, 200, seed=8)
    case = W.make_case(w)
    bad = case.block_tables.copy()
    bad[1, 2] = case.num_blocks + 7
    chunk = [16, 40, 24]
    monkeypatch.delenv("PKV_PREFILL_MODE", raising=False)
    gpu, _, st, q_start = _run(case, chunk, tables=bad, oracle_ref=False)
    assert st == pkv.PKV_ERR_DEVICE_BOUNDS
    _, ref, _, _ = _run(case, chunk)
    others = np.r_[q_start[0]:q_start[1], q_start[2]:q_start[3]]
    H.check_close(gpu[others], ref[others], kv, W.BF16, "other sequences")
    monkeypatch.setenv("PKV_PREFILL_MODE", "mma")
    mma, _, st_mma, _ = _run(case, chunk, tables=bad, oracle_ref=False)
    assert st_mma == pkv.PKV_ERR_DEVICE_BOUNDS
    rows = np.r_[q_start[1]:q_start[2]]
    assert np.isfinite(gpu[rows]).all()
    H.check_close(gpu[rows], mma[rows], kv, W.BF16, "sequence with the bad block")


@pytest.mark.slow
def test_prefill_benchmark_workload_sampled():
    """The benchmark's chunked-prefill workload at full size; the oracle computes
    sampled query rows, each as a chunk of one at its own position."""
    pkv = _pkv()
    w, n = W.prefill_workload()
    case = W.make_case(w)
    chunk = [n] * w.batch
    k, v, s = _full_cache(case)
    q, q_start = W.prefill_chunk(case, chunk)
    kd, vd, sd = H.cache_to_device(k, v, s, w.kv_dtype)
    qt = H.bits_to_tensor(q, w.q_dtype)
    out = torch.empty_like(qt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_prefill_attention(qt, torch.from_numpy(q_start).cuda(), kd, vd,
                                torch.from_numpy(case.block_tables).cuda(),
                                torch.from_numpy(case.context_lens).cuda(), sd, out,
                                w.softmax_scale, w.num_kv_heads, w.kv_dtype, w.block_size, n,
                                status)
    torch.cuda.synchronize()
    assert status.item() == 0
    gpu = H.tensor_to_f64(out)
    rng = np.random.default_rng(1)
    for r in np.sort(rng.choice(len(q), 24, replace=False)):
        b = int(np.searchsorted(q_start, r, side="right") - 1)
        ctx = case.context_lens.copy()
        ctx[b] = case.context_lens[b] - n + (r - q_start[b]) + 1    # the row's position + 1
        one = np.zeros(w.batch + 1, np.int32)
        one[b + 1:] = 1
        ref = oracle.prefill_attention(q[r:r + 1], w.q_dtype, one, k, v, case.block_tables, ctx,
                                       s, w.kv_dtype, case.num_blocks, w.softmax_scale,
                                       w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size)
        H.check_close(gpu[r:r + 1], ref, w.kv_dtype, w.q_dtype, f"row {r}")


def test_prefill_tc_bounded_wait_reports_a_timeout(monkeypatch):
    """The 16-bit tcgen05 prefill (warp roles) with its first S batch left
    uncommitted (PKV_TEST_DROP_COMMIT): the softmax's bounded wait on it runs out
    (about 2 s), every other role's wait ends on the abort, the call
    reports PKV_ERR_DEVICE_TIMEOUT through dev_status and zeros in its rows, and
    the next call on the same context is exact again."""
    pkv = _pkv()
    monkeypatch.delenv("PKV_PREFILL_MODE", raising=False)
    w = W.Workload("timeout", 1, 8, 2, 128, 16, W.BF16, W.BF16, "fixed", 40, 40, seed=9)
    case = W.make_case(w)
    monkeypatch.setenv("PKV_TEST_DROP_COMMIT", "1")
    with pkv.library("test"):                    # the switch exists in the test build only
        gpu, _, st, _ = _run(case, [8])
        assert st & pkv.PKV_ERR_DEVICE_TIMEOUT
        assert not gpu.any()
        monkeypatch.delenv("PKV_TEST_DROP_COMMIT")
        gpu, ref, st, _ = _run(case, [8])
    assert st == 0
    H.check_close(gpu, ref, W.BF16, W.BF16, "after a timed-out launch")
