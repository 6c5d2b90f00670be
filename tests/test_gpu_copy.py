"""GPU parity of paged_kv_copy_blocks: byte-exact against the oracle's copy, and
the copy-on-write invariant through the decode kernel."""

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


def _pool(kv, head_dim=128, block_size=16, seed=0, pool_blocks=0):
    qd = W.F16 if kv == W.F16 else W.BF16
    w = W.Workload("copy", 6, 16, 4, head_dim, block_size, kv, qd, "uniform", 1, 300,
                   outlier_prob=0.01, outlier_scale=20.0, pool_blocks=pool_blocks, seed=seed)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    return w, case, k, v, s


def _free_blocks(case):
    used = set(case.block_tables[case.block_tables >= 0].ravel().tolist())
    return [b for b in range(case.num_blocks) if b not in used]


def _copy_both(w, case, k, v, s, pairs):
    pkv = _pkv()
    kd, vd, sd = H.cache_to_device(k, v, s, w.kv_dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pt = torch.from_numpy(np.ascontiguousarray(pairs, np.int32).reshape(-1, 2)).cuda()
    pkv.paged_kv_copy_blocks(kd, vd, sd, w.kv_dtype, pt, w.block_size, w.head_dim, status)
    torch.cuda.synchronize()
    oracle.copy_blocks(k, v, s, w.kv_dtype, pairs, case.num_blocks, w.num_kv_heads, w.head_dim,
                       w.block_size)
    return H.cache_to_host(kd, vd, sd, w.kv_dtype), status.item()


def _assert_same(host, dev):
    for a, b in zip(host, dev):
        if a is None:
            assert b is None
            continue
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), np.argwhere(a != b)[:5]


@pytest.mark.parametrize("kv", [W.F16, W.BF16, W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32])
@pytest.mark.parametrize("head_dim,block_size", [(128, 16), (64, 32), (128, 256)])
def test_copy_blocks_bit_exact(kv, head_dim, block_size):
    w, case, k, v, s = _pool(kv, head_dim, block_size, seed=kv * 7 + block_size,
                             pool_blocks=0)
    rng = np.random.default_rng(block_size + kv)
    used = np.unique(case.block_tables[case.block_tables >= 0])
    free = np.array(_free_blocks(case))
    n = min(len(free), len(used), 9)
    assert n > 0
    pairs = np.stack([rng.choice(used, n, replace=False), rng.choice(free, n, replace=False)], 1)
    pairs = np.concatenate([pairs, [[used[0], used[0]]]])          # src == dst: a no-op
    dev, st = _copy_both(w, case, k, v, s, pairs)
    _assert_same((k, v, s), dev)
    assert st == 0


def test_copy_blocks_flags_and_skips_out_of_range_ids():
    pkv = _pkv()
    w, case, k, v, s = _pool(W.INT4_G32, seed=5)
    free = _free_blocks(case)
    pairs = np.array([[-1, free[0]], [0, case.num_blocks], [case.block_tables[0, 0], free[1]]],
                     np.int32)
    dev, st = _copy_both(w, case, k, v, s, pairs)
    _assert_same((k, v, s), dev)                                   # the good pair still lands
    assert st == pkv.PKV_ERR_DEVICE_BOUNDS


def test_copy_zero_pairs_is_a_no_op():
    pkv = _pkv()
    w, case, k, v, s = _pool(W.BF16, seed=6)
    kd, vd, sd = H.cache_to_device(k, v, s, w.kv_dtype)
    pkv.paged_kv_copy_blocks(kd, vd, sd, w.kv_dtype,
                             torch.zeros((0, 2), dtype=torch.int32, device="cuda"),
                             w.block_size, w.head_dim)
    torch.cuda.synchronize()
    _assert_same((k, v, s), H.cache_to_host(kd, vd, sd, w.kv_dtype))


@pytest.mark.parametrize("kv", [W.FP8_E4M3, W.INT4_G32, W.BF16])
def test_copy_on_write_fork_then_write_and_attend(kv):
    """Fork: each sequence's last (partly filled) block is copied into a fresh
    one and its table remapped, the new token is written into the copy, and
    attention through the new tables matches the oracle doing the same steps."""
    pkv = _pkv()
    base = W.Workload("fork", 4, 64, 8, 128, 16, kv, W.BF16, "uniform", 20, 150,
                      pool_blocks=64, seed=91)
    case = W.make_case(base)
    w = case.w
    k, v, s = oracle.prefill_case(case)
    free = _free_blocks(case)
    tables = case.block_tables.copy()
    slots = case.new_slots.copy()
    pairs = []
    for b in range(w.batch):
        last = (int(case.context_lens[b]) - 1) // w.block_size
        src, dst = int(tables[b, last]), free.pop()
        pairs.append([src, dst])
        tables[b, last] = dst
        slots[b] = W.slots_for(tables[b], np.array([case.context_lens[b] - 1]), w.block_size)[0]
    pairs = np.array(pairs, np.int32)
    # GPU: copy, write the new token into the copies, attend through the new tables
    kd, vd, sd = H.cache_to_device(k, v, s, w.kv_dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_copy_blocks(kd, vd, sd, kv, torch.from_numpy(pairs).cuda(), w.block_size,
                             w.head_dim, status)
    pkv.paged_kv_write(H.bits_to_tensor(case.k_new, w.q_dtype), H.bits_to_tensor(case.v_new, w.q_dtype),
                       torch.from_numpy(slots).cuda(), kd, vd, sd, kv, w.block_size, w.head_dim,
                       status)
    fork = W.Case(**{**case.__dict__})
    fork.block_tables = tables
    fork.new_slots = slots
    g = H.GpuCase(fork, None, None, None, 0, device_cache=(kd, vd, sd))
    out = g.attend()
    assert status.item() == 0 and g.status.item() == 0
    # oracle: the same three steps
    oracle.copy_blocks(k, v, s, kv, pairs, case.num_blocks, w.num_kv_heads, w.head_dim,
                       w.block_size)
    ref = oracle.step_case(fork, k, v, s)
    _assert_same((k, v, s), H.cache_to_host(kd, vd, sd, kv))
    H.check_close(out, ref, kv, w.q_dtype, f"fork kv {kv}")
