"""Host-side checks of the seeded input generator (block tables, slots, sizes)."""

import json
import os

import numpy as np
import pytest

import workloads as W

FACTS = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


@pytest.mark.parametrize("cfg", [1, 3, 4])
def test_tables_are_a_valid_paging(cfg):
    w = W.CONFIGS[cfg].scaled(batch=16, ctx_cap=600, seed=5) if cfg != 1 else W.CONFIGS[1]
    case = W.make_case(w)
    bs = w.block_size
    ctx = case.context_lens
    owners = {}
    sp_blocks = w.shared_prefix_tokens // bs
    for b in range(w.batch):
        n = -(-int(ctx[b]) // bs)
        row = case.block_tables[b]
        assert np.all(row[:n] >= 0) and np.all(row[:n] < case.num_blocks)
        assert np.all(row[n:] == -1)
        for j in range(n):
            if j < sp_blocks:
                assert row[j] == case.block_tables[0, j]
                continue
            assert row[j] not in owners, "a private block is mapped twice"
            owners[row[j]] = b
        # waste: the unused tail of the last block is at most bs - 1 tokens
        assert n * bs - int(ctx[b]) <= bs - 1


def test_waste_bound_matches_page_fact():
    f = FACTS["max_waste_tokens_block_16"]
    w = W.CONFIGS[3].scaled(batch=64, ctx_cap=300, seed=8)
    case = W.make_case(w)
    n = -(-case.context_lens.astype(np.int64) // f["block_size"])
    waste = n * f["block_size"] - case.context_lens
    assert waste.max() <= f["max_waste_tokens"]


def test_config2_pool_is_needed_plus_ten_percent():
    rng = np.random.default_rng(0)
    w = W.CONFIGS[2]
    ctx = W.draw_context_lens(w, rng)
    tables, nb = W.build_tables(w, ctx, rng)
    assert nb == 18023 and tables.shape == (64, 256)


def test_slots_cover_every_context_token_once():
    w = W.CONFIGS[3].scaled(batch=8, ctx_cap=200, seed=12)
    case = W.make_case(w)
    all_slots = np.concatenate([case.prefill_slots, case.new_slots[case.new_slots >= 0]])
    assert len(np.unique(all_slots)) == len(all_slots) == int(case.context_lens.sum())


def test_shared_prefix_written_once_and_new_token_skipped_when_shared():
    w = W.CONFIGS[4].scaled(batch=6, ctx_cap=64, seed=2)
    case = W.make_case(w)
    sp = w.shared_prefix_tokens
    assert sp == 64 // w.block_size * w.block_size
    uniq = len(np.unique(case.prefill_slots))
    assert uniq == len(case.prefill_slots)
    for b in range(w.batch):
        if case.context_lens[b] <= sp:
            assert case.new_slots[b] == -1


def test_slot_mapping_snippet3_example():
    f = FACTS["snippet3_address"]
    table = np.arange(3, dtype=np.int32)
    assert W.slots_for(table, np.array([f["token_index"]]), f["block_size"])[0] == \
        f["physical_block"] * f["block_size"] + f["offset"]


def test_lognormal_lengths_are_clipped_and_centred():
    w = W.CONFIGS[3].scaled(batch=4000, seed=77)
    ctx = W.draw_context_lens(w, np.random.default_rng(77))
    assert ctx.min() >= 256 and ctx.max() <= 8192
    assert 1900 < np.median(ctx) < 2200


def test_bf16_rounding_matches_torch_cast():
    import torch
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(10000) * 100,
                        np.float32([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.f32_to_bf16_bits(x), ref)
    assert W.bf16_bits_to_f32(W.f32_to_bf16_bits(np.float32([1.00390625])))[0] == 1.0  # tie -> even


def test_algorithmic_bytes_config2():
    case = W.make_case(W.CONFIGS[2].scaled(batch=2, seed=3))
    kv = 2 * int(case.context_lens.sum()) * 8 * 128 * 2
    got = W.attention_bytes(case)
    assert got == kv + 2 * 2 * 32 * 128 * 2 + 2 * 256 * 4 + 2 * 4


def test_prefill_flops_closed_form_matches_brute_force():
    """The prefill FLOP count behind the TFLOP/s figures: QK^T and PV over each
    query's causal range (query j of a chunk of n over c tokens sees c - n + j + 1
    tokens), 2 flops per multiply-add, counted query by query."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        b = int(rng.integers(1, 5))
        ctx = rng.integers(1, 300, size=b)
        chunk = [int(rng.integers(1, c + 1)) for c in ctx]
        hq, d = int(rng.choice([4, 32])), int(rng.choice([64, 128]))
        brute = 0
        for c, n in zip(ctx, chunk):
            for j in range(n):
                seen = int(c) - n + j + 1
                brute += 2 * 2 * seen * d * hq          # QK^T and PV, 2 flops per multiply-add
        assert W.prefill_flops(ctx, chunk, hq, d) == brute
    # the benchmark's workload: 8 chunks of 512 over 4096-token contexts, 32 heads, D 128
    w, n = W.prefill_workload()
    assert W.prefill_flops([4096] * 8, [n] * 8, w.num_q_heads, w.head_dim) == 257_731_592_192
