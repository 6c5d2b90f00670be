"""GPU parity of paged_decode_attention against the fp64 oracle.

The GPU reads the oracle-written cache (so both sides see the same bytes);
each output must lie within the stated max-abs tolerance (2e-3 for 16-bit KV,
5e-3 for FP8/INT4) of the oracle before its final rounding to the output
dtype (tests/helpers.py, check_close).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["shared", "warp", "balanced", "simt", "tc"])
def mode(request, monkeypatch):
    """Run a test under the decode kernel's work splits (shared partitions,
    warp-owned partitions, the balanced split of all tiles over one wave of
    warps), under the SIMT
    comparator (which takes 16-bit, FP8 and INT8 caches; INT4 stays on the
    tensor path), and under the tcgen05 kernel (one-byte caches with head_dim
    128; other calls keep the mma.sync kernel).  The comparators live in the
    test build of the library only."""
    monkeypatch.setenv("PKV_DECODE_MODE", request.param)
    with H.library_for(request.param):
        yield request.param


def _run(w, partition_size=0, identity=False, max_blocks_per_seq=None):
    case = W.make_case(w, identity_tables=identity, max_blocks_per_seq=max_blocks_per_seq)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    g = H.GpuCase(case, k, v, s, partition_size)
    out = g.attend()
    ref = H.oracle_attention(case, k, v, s)
    assert g.status.item() == 0
    return case, g, out, ref, (k, v, s)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, "3-e5m2", "3-int8"])
@pytest.mark.parametrize("partition_size", [0, 32, 64])
def test_configs_small(cfg, partition_size, mode):
    w = H.workload(cfg).scaled(batch=5, ctx_cap=300, seed=700 + H.seed_of(cfg))
    case, g, out, ref, _ = _run(w, partition_size)
    H.check_close(out, ref, w.kv_dtype, w.q_dtype, f"config {cfg} P={partition_size}")


def test_config1_exact_shape():
    w = W.CONFIGS[1]
    case, g, out, ref, _ = _run(w)
    H.check_close(out, ref, w.kv_dtype, w.q_dtype, "config 1")


@pytest.mark.parametrize("kv", [W.F16, W.BF16, W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (16, 2), (4, 1)])
def test_heads_dims_dtypes(kv, head_dim, hq, hkv, mode):
    qd = W.F16 if kv == W.F16 else W.BF16
    w = W.Workload("grid", 3, hq, hkv, head_dim, 16, kv, qd, "uniform", 1, 200, seed=hq * 7 + hkv + head_dim + kv)
    case, g, out, ref, _ = _run(w, partition_size=64)
    H.check_close(out, ref, kv, qd, f"kv {kv} D {head_dim} {hq}/{hkv}")


@pytest.mark.parametrize("kv", [W.F16, W.BF16, W.FP8_E4M3, W.INT8, W.INT4_G32])
def test_negative_softmax_scale(kv, mode):
    """A negative softmax scale: each head's largest scaled score is its
    smallest raw one."""
    qd = W.F16 if kv == W.F16 else W.BF16
    w = W.Workload("neg", 4, 32, 8, 128, 16, kv, qd, "uniform", 50, 600,
                   outlier_prob=0.01, outlier_scale=20.0, seed=91 + kv)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    g = H.GpuCase(case, k, v, s, 128)
    out = g.attend(scale=-w.softmax_scale)
    assert g.status.item() == 0
    ref = H.oracle_attention(case, k, v, s, scale=-w.softmax_scale)
    H.check_close(out, ref, kv, qd, f"negative scale, kv {kv}")


@pytest.mark.parametrize("kv", [W.BF16, W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32])
@pytest.mark.parametrize("block_size", [16, 32, 64, 128])
def test_block_sizes(kv, block_size, mode):
    w = W.Workload("bs", 4, 8, 2, 128, block_size, kv, W.BF16, "uniform", 1, 400, seed=block_size + kv)
    case, g, out, ref, _ = _run(w, partition_size=96)
    H.check_close(out, ref, kv, W.BF16, f"bs {block_size}")


@pytest.mark.parametrize("kv", [W.F16, W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32])
def test_context_length_edges(kv, mode):
    """ctx in {0, 1, 15, 16, 17, P-1, P, P+1, 2P+1} with P = 64."""
    qd = W.F16 if kv == W.F16 else W.BF16
    lens = [0, 1, 15, 16, 17, 63, 64, 65, 129]
    w = W.Workload("edges", len(lens), 8, 2, 64, 16, kv, qd, "fixed", 129, 129, seed=31 + kv)
    case = W.make_case(w)
    case.context_lens = np.array(lens, np.int32)
    k, v, s = oracle.prefill_case(case)
    for P in (0, 64):
        g = H.GpuCase(case, k, v, s, P)
        out = g.attend()
        ref = H.oracle_attention(case, k, v, s)
        H.check_close(out, ref, kv, qd, f"edges P={P}")
        assert not out[0].any(), "context_len 0 must give zeros"
        # ctx == 1: the V row of token 0, rounded to the output dtype
        p0 = case.block_tables[1, 0]
        vrow = oracle.dequant_row(v, s, 1, kv, case.num_blocks, 2, 64, 16, p0, 0, 0)
        assert np.allclose(out[1, 0], vrow, atol=H.TOL[kv], rtol=2 ** -8)


@pytest.mark.parametrize("cfg", [1, 3, 4])
def test_block_permutation_is_bit_exact(cfg, mode):
    w = W.CONFIGS[cfg].scaled(batch=4, ctx_cap=250, seed=900 + cfg)
    case, g, out, ref, (k, v, s) = _run(w, partition_size=64)
    rng = np.random.default_rng(3)
    perm = rng.permutation(case.num_blocks)
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm], v2[perm] = k, v
    s2 = None
    if s is not None:
        s2 = np.empty_like(s)
        s2[:, perm] = s
    bt = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1).astype(np.int32)
    case2 = W.Case(**{**case.__dict__, "block_tables": bt})
    g2 = H.GpuCase(case2, k2, v2, s2, 64)
    out2 = g2.attend()
    assert np.array_equal(out, out2)


def test_identity_tables_match_shuffled():
    w = W.CONFIGS[2].scaled(batch=4, ctx_cap=256, seed=55)
    _, _, out_a, ref_a, _ = _run(w)
    _, _, out_b, ref_b, _ = _run(w, identity=True)
    assert np.array_equal(ref_a, ref_b)
    assert np.array_equal(out_a, out_b)


@pytest.mark.parametrize("kv", [W.BF16, W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32])
def test_split_matches_unsplit(kv, mode):
    w = W.Workload("split", 3, 16, 2, 128, 16, kv, W.BF16, "fixed", 1000, 1000, seed=kv + 101)
    _, _, out_1, ref, _ = _run(w, partition_size=1008)
    _, _, out_n, _, _ = _run(w, partition_size=48)
    H.check_close(out_1, ref, kv, W.BF16, "unsplit")
    H.check_close(out_n, ref, kv, W.BF16, "split")
    assert np.max(np.abs(out_1 - out_n)) <= 2 * H.TOL[kv]


def test_constant_keys_give_mean_of_values():
    w = W.Workload("constk", 2, 8, 2, 128, 16, W.BF16, W.BF16, "fixed", 300, 300, seed=3)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, 2, 128, 16)
    k[:] = W.to_bits(np.float32([0.25]), W.BF16)[0]
    g = H.GpuCase(case, k, v, s, 64)
    out = g.attend()
    for b in range(2):
        n = case.context_lens[b]
        rows = np.stack([v[case.block_tables[b, t // 16], :, t % 16] for t in range(n)])
        mean = W.bits_to_f32(rows, W.BF16).astype(np.float64).mean(0)       # [Hkv, D]
        H.check_close(out[b], np.repeat(mean, 4, 0), W.BF16, W.BF16, "constant K")


@pytest.mark.parametrize("kv", [W.FP8_E4M3, W.FP8_E5M2, W.INT8, W.INT4_G32, W.BF16])
def test_unwritten_last_token_matches_oracle(kv, mode):
    """Attend over a context whose last token was never written (zeroed pool):
    an FP8 block with scale 0 and INT4 rows with scale 0 dequantize to 0, so the
    output stays finite and equal to the oracle's."""
    w = W.Workload("unwritten", 8, 16, 2, 128, 16, kv, W.BF16, "fixed", 33, 33, seed=61 + kv)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)          # the new token (offset 0 of block 2) stays 0
    g = H.GpuCase(case, k, v, s, 16)
    out = g.attend()
    ref = H.oracle_attention(case, k, v, s)
    assert np.isfinite(out).all()
    H.check_close(out, ref, kv, W.BF16, "unwritten last token")


@pytest.mark.parametrize("kv,head_dim", [(W.BF16, 64), (W.FP8_E4M3, 128)])
def test_bad_block_id_is_flagged_and_skipped(kv, head_dim, mode):
    import paged_quantized_kv_write_gb300 as pkv
    w = W.Workload("badid", 3, 8, 2, head_dim, 16, kv, W.BF16, "fixed", 40, 40, seed=4)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    bt = case.block_tables.copy()
    bt[1, 1] = case.num_blocks + 5                     # tokens 16..31 of sequence 1
    g = H.GpuCase(case, k, v, s, 0)
    out = g.attend(tables=torch.from_numpy(bt).cuda())
    assert g.status.item() == pkv.PKV_ERR_DEVICE_BOUNDS
    # the other sequences are untouched
    ref = H.oracle_attention(case, k, v, s)
    H.check_close(out[[0, 2]], ref[[0, 2]], kv, W.BF16, "other sequences")


def test_argument_errors_return_status():
    import paged_quantized_kv_write_gb300 as pkv
    w = W.Workload("args", 2, 8, 2, 64, 16, W.BF16, W.BF16, "fixed", 40, 40, seed=4)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    g = H.GpuCase(case, k, v, s, 0)
    with pytest.raises(pkv.PagedKVError):   # Hq not a multiple of Hkv
        pkv.paged_decode_attention(g.q, g.k, g.v, g.tables, g.ctx, None, g.out, 0.1, 3,
                                   W.BF16, 16)
    with pytest.raises(pkv.PagedKVError):   # split without a workspace
        pkv.paged_decode_attention(g.q, g.k, g.v, g.tables, g.ctx, None, g.out, 0.1, 2,
                                   W.BF16, 16, partition_size=16)


# ----------------------------------------------------------------- full size
@pytest.mark.slow
@pytest.mark.parametrize("cfg", [2, 3, 4, 5, "3-e5m2", "3-int8"])
def test_full_size_sampled(cfg):
    """The benchmark's workloads at full size, in the launch configuration the
    benchmark times (partition_size from the workload, else the library's
    choice); the oracle computes a sample of (sequence, head) outputs."""
    w = H.workload(cfg)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    g = H.GpuCase(case, k, v, s, w.partition_size)
    out = g.attend()
    assert g.status.item() == 0
    rng = np.random.default_rng(H.seed_of(cfg))
    n = 96
    ps = np.concatenate([rng.integers(0, w.batch, n), np.zeros(w.num_q_heads, int)])
    ph = np.concatenate([rng.integers(0, w.num_q_heads, n), np.arange(w.num_q_heads)])
    ref = oracle.decode_attention_pairs(case.q, w.q_dtype, k, v, case.block_tables,
                                        case.context_lens, s, w.kv_dtype, case.num_blocks,
                                        w.softmax_scale, w.num_q_heads, w.num_kv_heads,
                                        w.head_dim, w.block_size, ps, ph)
    H.check_close(out[ps, ph], ref, w.kv_dtype, w.q_dtype, f"full config {cfg}")
    assert np.isfinite(out).all()
