"""GPU parity of paged_decode_attention_with_write (the write of each sequence's
new token fused into the decode launch): the cache must end up byte-identical
to the oracle's write, the output must match the oracle's attention, and both
must equal the unfused paged_kv_write + paged_decode_attention."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["shared", "warp", "balanced", "tc"])
def mode(request, monkeypatch):
    monkeypatch.setenv("PKV_DECODE_MODE", request.param)
    with H.library_for(request.param):
        yield request.param


def _pkv():
    import paged_quantized_kv_write_gb300 as pkv
    return pkv


def _fused(g: H.GpuCase, slots: np.ndarray):
    pkv = _pkv()
    case, w = g.case, g.w
    pkv.paged_decode_attention_with_write(
        g.q, H.bits_to_tensor(case.k_new, w.q_dtype), H.bits_to_tensor(case.v_new, w.q_dtype),
        torch.from_numpy(np.ascontiguousarray(slots, np.int64)).cuda(), g.k, g.v, g.tables,
        g.ctx, g.s, g.out, w.softmax_scale, w.kv_dtype, w.block_size, g.partition_size, g.ws,
        g.status)
    torch.cuda.synchronize()
    return H.tensor_to_f64(g.out)


def _check(w, partition_size=0, slots=None, case=None):
    case = case or W.make_case(w)
    slots = case.new_slots if slots is None else slots
    k, v, s = oracle.prefill_case(case)
    g = H.GpuCase(case, k, v, s, partition_size)
    out = _fused(g, slots)
    # oracle: the write, then the attention
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    ref = H.oracle_attention(case, k, v, s)
    gk, gv, gs = H.cache_to_host(g.k, g.v, g.s, w.kv_dtype)
    assert np.array_equal(gk, k) and np.array_equal(gv, v), "cache bytes differ"
    if s is not None:
        assert np.array_equal(gs.view(np.uint8), s.view(np.uint8)), "scales differ"
    H.check_close(out, ref, w.kv_dtype, w.q_dtype, f"fused {w.name}")
    return case, g, out, (k, v, s)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, "3-e5m2", "3-int8"])
@pytest.mark.parametrize("partition_size", [0, 32])
def test_fused_matches_oracle_and_unfused(cfg, partition_size, mode):
    pkv = _pkv()
    w = H.workload(cfg).scaled(batch=5, ctx_cap=300, seed=900 + H.seed_of(cfg))
    case, g, out, _ = _check(w, partition_size)
    assert g.status.item() == 0
    # unfused on a fresh upload of the same prefill: identical output bits
    k, v, s = oracle.prefill_case(case)
    g2 = H.GpuCase(case, k, v, s, partition_size)
    pkv.paged_kv_write(H.bits_to_tensor(case.k_new, w.q_dtype), H.bits_to_tensor(case.v_new, w.q_dtype),
                       torch.from_numpy(case.new_slots).cuda(), g2.k, g2.v, g2.s, w.kv_dtype,
                       w.block_size, w.head_dim, g2.status)
    out2 = g2.attend()
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("kv", [W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32, W.BF16])
def test_fused_new_token_opens_a_block(kv, mode):
    """ctx = 16 m + 1: the new token sits at offset 0 of a fresh block, so for
    FP8 it sets that block's scales inside the fused launch."""
    qd = W.BF16
    w = W.Workload("open", 6, 32, 8, 128, 16, kv, qd, "fixed", 145, 145, seed=77 + kv)
    _check(w, partition_size=64)


def test_fused_skips_minus_one_and_flags_a_foreign_slot(mode):
    pkv = _pkv()
    w = W.Workload("slots", 4, 16, 4, 128, 16, W.FP8_E4M3, W.BF16, "uniform", 20, 200, seed=12)
    case = W.make_case(w)
    slots = case.new_slots.copy()
    slots[1] = -1                                   # nothing to write for sequence 1
    k, v, s = oracle.prefill_case(case)
    g = H.GpuCase(case, k, v, s, 0)
    bad = slots.copy()
    bad[2] = slots[0]                               # sequence 2 aims at sequence 0's slot
    out = _fused(g, bad)
    assert g.status.item() == pkv.PKV_ERR_DEVICE_BOUNDS
    # oracle: sequences 0 and 3 written, 1 and 2 not
    ok = slots.copy()
    ok[2] = -1
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, ok, k, v, s, w.kv_dtype, case.num_blocks,
                    w.num_kv_heads, w.head_dim, w.block_size)
    gk, gv, gs = H.cache_to_host(g.k, g.v, g.s, w.kv_dtype)
    assert np.array_equal(gk, k) and np.array_equal(gv, v) and np.array_equal(gs, s)
    H.check_close(out, H.oracle_attention(case, k, v, s), w.kv_dtype, w.q_dtype, "foreign slot")


def test_fused_requires_a_slot_mapping():
    pkv = _pkv()
    w = W.Workload("args", 2, 8, 2, 64, 16, W.BF16, W.BF16, "fixed", 20, 20, seed=1)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    g = H.GpuCase(case, k, v, s, 0)
    import ctypes
    P = ctypes.c_void_p
    r = pkv.lib.paged_decode_attention_with_write(
        P(g.q.data_ptr()), w.q_dtype, P(g.q.data_ptr()), P(g.q.data_ptr()), None,
        P(g.k.data_ptr()), P(g.v.data_ptr()), P(g.tables.data_ptr()), case.max_blocks_per_seq,
        P(g.ctx.data_ptr()), w.batch, None, w.kv_dtype, case.num_blocks, P(g.out.data_ptr()),
        w.softmax_scale, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, 0, None, 0,
        None, None)
    assert r == pkv.PKV_ERR_INVALID_ARG


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_fused_full_size_sampled(cfg):
    """The benchmark's workloads at full size through the fused call: cache
    bit-exact everywhere, attention on sampled (sequence, head) outputs."""
    w = H.workload(cfg)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    g = H.GpuCase(case, k, v, s, w.partition_size)
    out = _fused(g, case.new_slots)
    assert g.status.item() == 0
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    gk, gv, gs = H.cache_to_host(g.k, g.v, g.s, w.kv_dtype)
    assert np.array_equal(gk, k) and np.array_equal(gv, v)
    if s is not None:
        assert np.array_equal(gs.view(np.uint8), s.view(np.uint8))
    rng = np.random.default_rng(cfg)
    ps = rng.integers(0, w.batch, 64)
    ph = rng.integers(0, w.num_q_heads, 64)
    ref = oracle.decode_attention_pairs(case.q, w.q_dtype, k, v, case.block_tables,
                                        case.context_lens, s, w.kv_dtype, case.num_blocks,
                                        w.softmax_scale, w.num_q_heads, w.num_kv_heads,
                                        w.head_dim, w.block_size, ps, ph)
    H.check_close(out[ps, ph], ref, w.kv_dtype, w.q_dtype, f"fused full config {cfg}")
