"""GPU parity of paged_kv_write: cache bytes and scales bit-exact to the oracle."""

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


def _gpu_write(case, k_dev, v_dev, s_dev, slots, kvals, vvals, status):
    pkv = _pkv()
    w = case.w
    pkv.paged_kv_write(H.bits_to_tensor(kvals, w.q_dtype), H.bits_to_tensor(vvals, w.q_dtype),
                       torch.from_numpy(np.ascontiguousarray(slots, np.int64)).cuda(), k_dev,
                       v_dev, s_dev, w.kv_dtype, w.block_size, w.head_dim, status)


def _prefill_both(case):
    """Prefill with the oracle and with the GPU from zeroed pools; return both."""
    pkv = _pkv()
    w = case.w
    k, v, s = oracle.prefill_case(case)
    kd, vd, sd = pkv.alloc_cache(w.kv_dtype, case.num_blocks, w.num_kv_heads, w.head_dim,
                                 w.block_size)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _gpu_write(case, kd, vd, sd, case.prefill_slots, case.prefill_k, case.prefill_v, status)
    torch.cuda.synchronize()
    return (k, v, s), (kd, vd, sd), status


def _assert_same(case, host, dev):
    k, v, s = host
    gk, gv, gs = H.cache_to_host(*dev, case.w.kv_dtype)
    assert np.array_equal(gk, k), f"K cache differs at {np.argwhere(gk != k)[:5]}"
    assert np.array_equal(gv, v), f"V cache differs at {np.argwhere(gv != v)[:5]}"
    if s is not None:
        diff = gs.view(np.uint8) != s.view(np.uint8)
        assert not diff.any(), f"scales differ at {np.argwhere(diff)[:5]}"


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, "3-e5m2", "3-int8"])
def test_prefill_and_step_write_bit_exact(cfg):
    w = H.workload(cfg).scaled(batch=6, ctx_cap=200, seed=500 + H.seed_of(cfg))
    case = W.make_case(w)
    host, dev, status = _prefill_both(case)
    _assert_same(case, host, dev)
    # the decode step's new token
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, *host, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    _gpu_write(case, *dev, case.new_slots, case.k_new, case.v_new, status)
    torch.cuda.synchronize()
    _assert_same(case, host, dev)
    assert status.item() == 0


@pytest.mark.parametrize("kv", [W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32, W.BF16, W.F16])
@pytest.mark.parametrize("head_dim,block_size", [(64, 16), (128, 32), (64, 64), (128, 256)])
def test_write_shapes(kv, head_dim, block_size):
    qd = W.F16 if kv == W.F16 else W.BF16
    w = W.Workload("shapes", 5, 8, 4, head_dim, block_size, kv, qd, "uniform", 1, 300,
                   outlier_prob=0.02, outlier_scale=30.0, seed=head_dim + block_size + kv)
    case = W.make_case(w)
    host, dev, status = _prefill_both(case)
    _assert_same(case, host, dev)
    assert status.item() == 0


@pytest.mark.parametrize("kv", W.BLK8_TYPES)
def test_fp8_offset_zero_tokens_apply_first_in_one_call(kv):
    w = W.Workload("order", 3, 4, 2, 128, 16, kv, W.BF16, "fixed", 40, 40, seed=77)
    case = W.make_case(w)
    rev = W.Case(**{**case.__dict__})
    order = np.arange(len(case.prefill_slots))[::-1].copy()     # offset-0 tokens last
    rev.prefill_slots = case.prefill_slots[order]
    rev.prefill_k = case.prefill_k[order]
    rev.prefill_v = case.prefill_v[order]
    host, dev, _ = _prefill_both(rev)
    _assert_same(rev, host, dev)
    host2, _, _ = _prefill_both(case)
    for a, b in zip(host, host2):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("kv", W.BLK8_TYPES)
def test_block_scale_over_the_opening_call_then_kept(kv):
    """The context written in two calls, split at a point inside blocks: the first
    call opens blocks (scale = amax over its rows in them, "Block-Wise Scaling
    Factors"), the second appends to those partial blocks (kept scale, saturating)
    and opens new ones, in one launch set.  Bit-exact to the oracle after each call,
    with x20 outliers so that appended rows do saturate."""
    pkv = _pkv()
    w = W.Workload("two calls", 5, 8, 2, 128, 16, kv, W.BF16, "uniform", 20, 260,
                   outlier_prob=0.02, outlier_scale=20.0, seed=91 + kv)
    case = W.make_case(w)
    k, v, s = oracle.alloc_cache(kv, case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    kd, vd, sd = pkv.alloc_cache(kv, case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # sequence b's prefill rows are its positions 0 .. ctx_b - 2, in order; the first
    # call takes positions below a random cut of each sequence, the second the rest,
    # each call in a shuffled token order
    rng = np.random.default_rng(7)
    first, second, base = [], [], 0
    for c in case.context_lens:
        n = int(c) - 1
        cut = int(rng.integers(0, n + 1))
        first += range(base, base + cut)
        second += range(base + cut, base + n)
        base += n
    for part in (rng.permutation(np.array(first, np.int64)),
                 rng.permutation(np.array(second, np.int64))):
        slots = np.ascontiguousarray(case.prefill_slots[part])
        kx = np.ascontiguousarray(case.prefill_k[part])
        vx = np.ascontiguousarray(case.prefill_v[part])
        oracle.kv_write(kx, vx, w.q_dtype, slots, k, v, s, kv, case.num_blocks,
                        w.num_kv_heads, w.head_dim, w.block_size)
        _gpu_write(case, kd, vd, sd, slots, kx, vx, status)
        torch.cuda.synchronize()
        _assert_same(case, (k, v, s), (kd, vd, sd))
    assert status.item() == 0
    # more codes at the format's largest value than opened (block, head) scales: the
    # appended rows did saturate, so the case tests the kept scale
    def n_top(c):
        if kv == W.INT8:
            return int((np.abs(c.view(np.int8).astype(np.int32)) == 127).sum())
        return int(((c & 0x7F) == (0x7E if kv == W.FP8_E4M3 else 0x7B)).sum())
    assert n_top(k) + n_top(v) > int((s > 0).sum())


def test_write_skips_minus_one_and_flags_out_of_range():
    pkv = _pkv()
    w = W.Workload("bounds", 2, 4, 2, 64, 16, W.INT4_G32, W.BF16, "fixed", 20, 20, seed=5)
    case = W.make_case(w)
    host, dev, status = _prefill_both(case)
    before = H.cache_to_host(*dev, w.kv_dtype)
    slots = np.array([-1, case.num_blocks * 16 + 3], np.int64)   # skip, out of range
    _gpu_write(case, *dev, slots, case.k_new, case.v_new, status)
    torch.cuda.synchronize()
    after = H.cache_to_host(*dev, w.kv_dtype)
    for a, b in zip(before, after):
        assert np.array_equal(a, b)
    assert status.item() == pkv.PKV_ERR_DEVICE_BOUNDS
    status.zero_()
    _gpu_write(case, *dev, np.array([-7, -1], np.int64), case.k_new, case.v_new, status)
    torch.cuda.synchronize()
    assert status.item() == pkv.PKV_ERR_DEVICE_BOUNDS


def test_write_special_values():
    """Zero rows (FP8 eps scale), signed zeros, saturating outliers, constant INT4 groups."""
    for kv in (W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32):
        w = W.Workload("special", 4, 4, 2, 128, 16, kv, W.BF16, "fixed", 17, 17, seed=9)
        case = W.make_case(w)
        rows = case.prefill_k.copy()
        rows[0] = 0                                     # all-zero offset-0 row
        rows[1] = 0x8000                                # all -0
        rows[2, :, :64] = W.to_bits(np.full((2, 64), 3.0, np.float32), W.BF16)  # constant groups
        rows[3] = W.to_bits(np.full((2, 128), 1e4, np.float32), W.BF16)          # saturation
        case.prefill_k = rows
        host, dev, status = _prefill_both(case)
        _assert_same(case, host, dev)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [2, 3, 4, 5, "3-e5m2", "3-int8"])
def test_full_size_prefill_bit_exact(cfg):
    case = W.make_case(H.workload(cfg))
    host, dev, status = _prefill_both(case)
    _assert_same(case, host, dev)
    assert status.item() == 0
