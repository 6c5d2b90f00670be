"""Pins of the CPU oracle to things other than itself.

Each test checks the oracle against a library routine on a special case, a
closed form, a brute-force search, an invariant, or a value the pages print
(tests/golden/page_facts.json, each entry with its citation).  They are
chosen so that a plausible slip in the oracle (a dropped term, a wrong sign
or index, a transposed operand, a wrong GQA mapping, a missing mask) fails
at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")
FACTS = json.load(open(GOLDEN))


# ------------------------------------------------------------------ formulas
def test_kv_size_formula_160_gib():
    f = FACTS["kv_bytes_70b_example"]
    b = oracle.kv_cache_bytes(f["layers"], f["heads"], f["head_dim"], f["seq_len"], f["batch"],
                              f["bytes_per_elem"])
    assert b / 2**30 == f["gib"]


def test_kv_size_formula_13b_per_token():
    f = FACTS["llama2_13b_bytes_per_token"]
    b = oracle.kv_cache_bytes(f["layers"], f["heads"], f["head_dim"], f["seq_len"], f["batch"],
                              f["bytes_per_elem"])
    assert b == 819200
    assert b / 1024 == f["approx_kilobytes"]
    g = FACTS["llama2_13b_4000_tokens_over_gb"]
    assert b * g["tokens"] > g["at_least_bytes"]


@pytest.mark.parametrize("key", ["pages_512_tokens_page_16", "pages_2048_tokens_page_16"])
def test_num_pages(key):
    f = FACTS[key]
    assert oracle.num_pages(f["tokens"], f["page_size"]) == f["pages"]
    # ceil, not floor: one token more needs one more page
    assert oracle.num_pages(f["tokens"] + 1, f["page_size"]) == f["pages"] + 1


def test_snippet3_address_translation():
    f = FACTS["snippet3_address"]
    free = list(range(f["pool_blocks"]))
    needed = -(-f["allocated_tokens"] // f["block_size"])
    table = [free.pop(0) for _ in range(needed)]
    phys, off = oracle.physical_address(table, f["block_size"], f["token_index"])
    assert (phys, off) == (f["physical_block"], f["offset"])
    with pytest.raises(IndexError):
        oracle.physical_address(table, f["block_size"], needed * f["block_size"])


# ------------------------------------------------------------------ 16-bit decoders
def test_f16_decode_all_codes_vs_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_decode_all_codes_vs_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def _dense_f32_sweep(rng, n=40000, lo=-30, hi=18):
    mags = np.exp2(rng.uniform(lo, hi, n)).astype(np.float32)
    signs = np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    return np.concatenate([mags * signs, np.float32([0.0, -0.0, 65504, 65519.99, 65520,
                                                     -65520, 6.1035156e-05, 5.9604645e-08,
                                                     2.9802322e-08, 2.9802326e-08])])


def test_f32_to_f16_rne_vs_numpy():
    rng = np.random.default_rng(7)
    x = _dense_f32_sweep(rng)
    # every f16 midpoint, exactly: ties must go to the even code
    f16 = np.arange(0, 0x7BFF, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = ((f16[:-1] + f16[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ E4M3
def _finite_e4m3_table():
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    return codes, np.array([oracle.e4m3_to_double(c) for c in codes])


def test_e4m3_decode_all_codes_vs_torch():
    f = FACTS["e4m3_format"]
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.nanmax(got) == f["max_finite"] == oracle.e4m3_to_double(0x7E)
    assert oracle.e4m3_to_double(0x08) == 2.0**-6
    assert oracle.e4m3_to_double(0x01) == 2.0**-9
    # 1/4/3 bits: 2^3 mantissa steps per binade, 15 usable exponents
    assert oracle.e4m3_to_double(0x39) - oracle.e4m3_to_double(0x38) == 2.0**-3


def _brute_force_e4m3(y: float, codes, vals) -> int:
    """Nearest finite E4M3 value, ties to the even code; saturate at +-448."""
    a = abs(y)
    if a >= 448.0:
        return 0xFE if math.copysign(1, y) < 0 else 0x7E
    best, bestd = None, None
    for c, v in zip(codes, vals):
        if c & 0x80:
            continue
        d = abs(a - v)
        if bestd is None or d < bestd or (d == bestd and (c & 1) == 0):
            best, bestd = c, d
    return best | (0x80 if math.copysign(1, y) < 0 else 0)


def test_e4m3_encode_vs_brute_force_nearest_even():
    codes, vals = _finite_e4m3_table()
    pos = sorted(set(v for c, v in zip(codes, vals) if not c & 0x80))
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    rng = np.random.default_rng(11)
    xs = list(np.float32(pos)) + list(np.float32(mids))
    xs += [np.nextafter(np.float32(m), np.float32(np.inf)) for m in mids]
    xs += [np.nextafter(np.float32(m), np.float32(-np.inf)) for m in mids]
    xs += list(np.exp2(rng.uniform(-14, 10, 3000)).astype(np.float32))
    xs += [np.float32(v) for v in (448.0, 449.0, 463.9, 464.0, 479.0, 480.0, 1e6, 1e-30)]
    for x in xs:
        for y in (float(x), -float(x)):
            assert oracle.e4m3_encode(y) == _brute_force_e4m3(y, codes, vals), y


def test_e4m3_encode_vs_torch_cast_in_range():
    rng = np.random.default_rng(12)
    y = np.concatenate([rng.standard_normal(20000) * 60,
                        np.exp2(rng.uniform(-12, 8.7, 20000)) * rng.choice([-1, 1], 20000)])
    y = np.clip(y, -447.9, 447.9).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in y], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturation_and_signed_zero():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-9) == 0x80
    assert oracle.e4m3_encode(float("nan")) == 0x7F


# ------------------------------------------------------------------ E5M2
def _finite_e5m2_table():
    codes = [c for c in range(256) if (c >> 2) & 0x1F != 0x1F]
    return codes, np.array([oracle.e5m2_to_double(c) for c in codes])


def test_e5m2_decode_all_codes_vs_torch():
    f = FACTS["e5m2_format"]
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).double().numpy()
    got = np.array([oracle.e5m2_to_double(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert oracle.e5m2_to_double(0x7C) == math.inf and oracle.e5m2_to_double(0xFC) == -math.inf
    # 1/5/2 bits with FP16's exponent range: same smallest normal and top binade
    assert f["exponent_bits"] == 5 and f["mantissa_bits"] == 2
    f16_min_normal = float(np.array([0x0400], np.uint16).view(np.float16)[0])
    f16_max = float(np.finfo(np.float16).max)
    assert oracle.e5m2_to_double(0x04) == f16_min_normal == 2.0**-14
    assert math.frexp(oracle.e5m2_to_double(0x7B))[1] == math.frexp(f16_max)[1]
    assert oracle.e5m2_to_double(0x7B) == 57344.0
    assert oracle.e5m2_to_double(0x01) == 2.0**-16
    assert oracle.e5m2_to_double(0x3D) - oracle.e5m2_to_double(0x3C) == 2.0**-2


def _brute_force_e5m2(y: float, codes, vals) -> int:
    """Nearest finite E5M2 value, ties to the even code; saturate at +-57344."""
    a = abs(y)
    neg = math.copysign(1, y) < 0
    if a >= 57344.0:
        return 0xFB if neg else 0x7B
    best, bestd = None, None
    for c, v in zip(codes, vals):
        if c & 0x80:
            continue
        d = abs(a - v)
        if bestd is None or d < bestd or (d == bestd and (c & 1) == 0):
            best, bestd = c, d
    return best | (0x80 if neg else 0)


def test_e5m2_encode_vs_brute_force_nearest_even():
    codes, vals = _finite_e5m2_table()
    pos = sorted(set(v for c, v in zip(codes, vals) if not c & 0x80))
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    rng = np.random.default_rng(13)
    xs = list(np.float32(pos)) + list(np.float32(mids))
    xs += [np.nextafter(np.float32(m), np.float32(np.inf)) for m in mids]
    xs += [np.nextafter(np.float32(m), np.float32(-np.inf)) for m in mids]
    xs += list(np.exp2(rng.uniform(-18, 16, 3000)).astype(np.float32))
    xs += [np.float32(v) for v in (57344.0, 57345.0, 61439.0, 61440.0, 65536.0, 1e9, 1e-30)]
    for x in xs:
        for y in (float(x), -float(x)):
            assert oracle.e5m2_encode(y) == _brute_force_e5m2(y, codes, vals), y


def test_e5m2_encode_vs_torch_cast_in_range():
    rng = np.random.default_rng(14)
    y = np.concatenate([rng.standard_normal(20000) * 3000,
                        np.exp2(rng.uniform(-16, 15.8, 20000)) * rng.choice([-1, 1], 20000)])
    y = np.clip(y, -57343.0, 57343.0).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e5m2).view(torch.uint8).numpy()
    got = np.array([oracle.e5m2_encode(float(v)) for v in y], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e5m2_encode_saturation_and_signed_zero():
    assert oracle.e5m2_encode(57344.0) == 0x7B
    assert oracle.e5m2_encode(61440.0) == 0x7B      # would round up to 2^16 = infinity
    assert oracle.e5m2_encode(-1e9) == 0xFB
    assert oracle.e5m2_encode(float("inf")) == 0x7B
    assert oracle.e5m2_encode(-0.0) == 0x80
    assert oracle.e5m2_encode(float("nan")) == 0x7F


# ------------------------------------------------------------------ INT8
def test_int8_encode_is_numpy_rint_half_even_clamped():
    """code = clamp(rint(y), -127, 127): numpy's rint rounds half to even."""
    rng = np.random.default_rng(15)
    halves = np.arange(-140, 140.5, 0.5)                # every tie and integer in range
    y = np.concatenate([halves, rng.uniform(-200, 200, 5000),
                        np.nextafter(halves, np.inf), np.nextafter(halves, -np.inf)])
    y = y.astype(np.float32)
    ref = np.clip(np.rint(y.astype(np.float64)), -127, 127).astype(np.int8)
    got = np.array([oracle.int8_encode(float(v)) for v in y], dtype=np.int8)
    assert np.array_equal(got, ref)
    assert oracle.int8_encode(2.5) == 2 and oracle.int8_encode(3.5) == 4
    assert oracle.int8_encode(-2.5) == -2 and oracle.int8_encode(-0.5) == 0
    assert oracle.int8_encode(1e9) == 127 and oracle.int8_encode(-1e9) == -127   # never -128
    assert oracle.int8_encode(float("nan")) == 0


def test_write_int8_scale_is_amax_over_127():
    rng = np.random.default_rng(16)
    row = (rng.standard_normal(64) * 2).astype(np.float32)
    row[9] = -7.25
    k, v, s, x = _one_block_write(W.INT8, row[None], [0])
    xr = W.bits_to_f32(x[0, 0], W.BF16)
    assert s[0, 1, 0] == np.float32(np.float32(7.25) / np.float32(127.0))
    codes = k[1, 0, 0].view(np.int8)
    assert codes[9] == -127
    # dequantized within half a step of the input
    deq = codes.astype(np.float64) * float(s[0, 1, 0])
    assert np.all(np.abs(deq - xr) <= 0.5 * float(s[0, 1, 0]) * (1 + 1e-6))
    # one call writing both tokens: the block's scale comes from both (amax 3 * 7.25)
    k2, _, s2, _ = _one_block_write(W.INT8, np.stack([row, row * 3]), [0, 1])
    assert s2[0, 1, 0] == np.float32(np.float32(21.75) / np.float32(127.0))
    assert k2[1, 0, 1].view(np.int8)[9] == -127
    # a larger token that a later call appends saturates at +-127 under the kept scale
    nb, bs = 3, 16
    x3 = W.to_bits((row * 3)[None, None, :], W.BF16)
    oracle.kv_write(x3, x3, W.BF16, np.array([1 * bs + 1]), k, v, s, W.INT8, nb, 1, 64, bs)
    assert s[0, 1, 0] == np.float32(np.float32(7.25) / np.float32(127.0))
    big = np.abs(row * 3) > 7.25 * 1.01
    assert np.all(np.abs(k[1, 0, 1].view(np.int8)[big]) == 127)


# ------------------------------------------------------------------ the write
def _one_block_write(kv_dtype, rows, offsets, head_dim=64, block_size=16, dtype=W.BF16,
                     num_kv_heads=1):
    """Write `rows` (float32 [n, D]) at `offsets` of physical block 1; return cache."""
    nb = 3
    k, v, s = oracle.alloc_cache(kv_dtype, nb, num_kv_heads, head_dim, block_size)
    x = W.to_bits(np.repeat(np.asarray(rows, np.float32)[:, None, :], num_kv_heads, 1), dtype)
    slots = np.array([1 * block_size + o for o in offsets], np.int64)
    oracle.kv_write(x, x, dtype, slots, k, v, s, kv_dtype, nb, num_kv_heads, head_dim,
                    block_size)
    return k, v, s, x


def test_write_16bit_is_a_copy_at_the_translated_slot():
    rng = np.random.default_rng(3)
    rows = rng.standard_normal((3, 64)).astype(np.float32)
    k, v, s, x = _one_block_write(W.BF16, rows, [5, 0, 15])
    for i, o in enumerate([5, 0, 15]):
        assert np.array_equal(k[1, 0, o], x[i, 0])
        assert np.array_equal(v[1, 0, o], x[i, 0])
    assert not k[0].any() and not k[2].any()


def test_write_fp8_scale_is_amax_over_448():
    f = FACTS["fp8_scale_rule"]
    rng = np.random.default_rng(4)
    row = (rng.standard_normal(64) * 3).astype(np.float32)
    row[17] = -9.5
    k, v, s, x = _one_block_write(W.FP8_E4M3, row[None], [0])
    xr = W.bits_to_f32(x[0, 0], W.BF16)
    amax = np.float32(np.abs(xr).max())
    assert s[0, 1, 0] == np.float32(amax / np.float32(f["fp8_max"]))
    assert s[1, 1, 0] == s[0, 1, 0]
    # the largest magnitude lands on the largest code, with its sign
    assert k[1, 0, 0, 17] == 0xFE
    # round trip within half an E4M3 step (2^-4 relative for normals)
    deq = np.array([oracle.e4m3_to_double(c) for c in k[1, 0, 0]]) * float(s[0, 1, 0])
    err = np.abs(deq - xr)
    assert np.all(err <= np.maximum(np.abs(xr) * 2.0**-4, 2.0**-10 * float(s[0, 1, 0])) + 1e-12)


def test_write_e5m2_scale_is_amax_over_its_largest_finite():
    rng = np.random.default_rng(6)
    row = (rng.standard_normal(64) * 3).astype(np.float32)
    row[5] = 11.0
    k, v, s, x = _one_block_write(W.FP8_E5M2, row[None], [0])
    xr = W.bits_to_f32(x[0, 0], W.BF16)
    assert s[0, 1, 0] == np.float32(np.float32(11.0) / np.float32(57344.0))
    assert k[1, 0, 0, 5] == 0x7B
    deq = np.array([oracle.e5m2_to_double(c) for c in k[1, 0, 0]]) * float(s[0, 1, 0])
    # half an E5M2 step: 2^-3 relative for normals
    assert np.all(np.abs(deq - xr) <= np.abs(xr) * 2.0**-3 + 2.0**-17 * float(s[0, 1, 0]))


def test_write_fp8_zero_row_uses_eps_scale():
    f = FACTS["fp8_scale_rule"]
    k, v, s, x = _one_block_write(W.FP8_E4M3, np.zeros((1, 64)), [0])
    assert s[0, 1, 0] == np.float32(f["eps"])
    assert not k[1, 0, 0].any()


def test_write_fp8_block_scale_is_the_amax_of_every_token_the_call_writes():
    """"Block-Wise Scaling Factors" (snippet-4): one scale per block from the absolute
    maximum over the whole block.  A 16-token block written in one call with a x20
    outlier at offset 9: scale = |outlier| / 448, the outlier takes the largest code
    with its sign, and no other code saturates."""
    f = FACTS["fp8_scale_rule"]
    rng = np.random.default_rng(21)
    rows = rng.standard_normal((16, 64)).astype(np.float32)
    rows[9, 40] = -20.0 * 1.375                       # the block's largest magnitude
    k, v, s, x = _one_block_write(W.FP8_E4M3, rows, list(range(16)))
    xr = W.bits_to_f32(x[:, 0], W.BF16)
    assert s[0, 1, 0] == np.float32(np.float32(27.5) / np.float32(f["fp8_max"]))
    assert s[1, 1, 0] == s[0, 1, 0]
    assert k[1, 0, 9, 40] == 0xFE
    mag = k[1, 0] & 0x7F
    assert (mag == 0x7E).sum() == 1 and not (mag == 0x7F).any()
    # every code within half an E4M3 step of x / scale (nothing clipped)
    deq = np.vectorize(oracle.e4m3_to_double)(k[1, 0]) * float(s[0, 1, 0])
    step = np.maximum(np.abs(xr) * 2.0**-4, 2.0**-10 * float(s[0, 1, 0]))
    assert np.all(np.abs(deq - xr) <= step + 1e-12)
    # the order of the tokens within the call does not matter
    kb, _, sb, _ = _one_block_write(W.FP8_E4M3, rows[::-1].copy(), list(range(15, -1, -1)))
    assert np.array_equal(k, kb) and np.array_equal(s, sb)


def test_write_fp8_whole_block_equals_snippet4_through_torch():
    """snippet-4 run by torch on one block (fp32 tensor, one KV head): scale =
    clamp(max|x| / 448, 1e-12), codes = (x / scale).to(float8_e4m3fn).  The
    oracle's one-call write of the same 16 tokens gives the same scale and bytes."""
    rng = np.random.default_rng(22)
    rows = (rng.standard_normal((16, 128)) * 5.0).astype(np.float32)
    rows[rng.random((16, 128)) < 0.01] *= 20.0
    k, v, s, x = _one_block_write(W.FP8_E4M3, rows, list(range(16)), head_dim=128)
    blk = torch.from_numpy(W.bits_to_f32(x[:, 0], W.BF16).astype(np.float32))
    scale = (torch.max(torch.abs(blk)) / 448.0).clamp(min=1e-12)
    codes = (blk / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert s[0, 1, 0] == np.float32(scale.item())
    assert np.array_equal(k[1, 0], codes)


def test_write_fp8_scale_kept_for_tokens_a_later_call_appends():
    """A block opened by one call keeps its scale; a later call's tokens (no
    offset-0 token among them) reuse it and saturate at +-448."""
    rng = np.random.default_rng(5)
    r0 = rng.standard_normal((4, 64)).astype(np.float32)
    k, v, s, x = _one_block_write(W.FP8_E4M3, r0, [0, 1, 2, 3])
    s_open = s.copy()
    amax = np.abs(W.bits_to_f32(x[:, 0], W.BF16)).max()
    assert s[0, 1, 0] == np.float32(np.float32(amax) / np.float32(448.0))
    nb, bs = 3, 16
    big = (r0[0] * 50).astype(np.float32)
    xb = W.to_bits(np.stack([big, r0[1] * 0.5])[:, None, :], W.BF16)
    oracle.kv_write(xb, xb, W.BF16, np.array([1 * bs + 4, 1 * bs + 5]), k, v, s, W.FP8_E4M3,
                    nb, 1, 64, bs)
    assert np.array_equal(s, s_open)
    sat = np.abs(W.bits_to_f32(xb[0, 0], W.BF16)) >= amax * 1.04
    assert sat.any() and np.all((k[1, 0, 4][sat] & 0x7F) == 0x7E)
    # a call that writes offset 0 again opens the block afresh from its own tokens
    oracle.kv_write(xb[1:], xb[1:], W.BF16, np.array([1 * bs]), k, v, s, W.FP8_E4M3, nb, 1, 64,
                    bs)
    a2 = np.abs(W.bits_to_f32(xb[1, 0], W.BF16)).max()
    assert s[0, 1, 0] == np.float32(np.float32(a2) / np.float32(448.0))


def test_write_fp8_scales_are_per_block_and_per_head():
    """Two blocks and two KV heads written in one call: each (block, head) scale is
    the amax of that head's rows in that block only; K and V are scaled apart."""
    rng = np.random.default_rng(23)
    nb, bs, hkv, d = 4, 16, 2, 64
    kx = rng.standard_normal((20, hkv, d)).astype(np.float32)
    vx = (rng.standard_normal((20, hkv, d)) * 0.1).astype(np.float32)
    kx[3, 1, 7] = 40.0                                   # block 2, head 1
    kx[17, 0, 2] = -33.0                                 # block 0, head 0
    slots = np.array([2 * bs + i for i in range(16)] + [0, 1, 2, 3], np.int64)
    k, v, s = oracle.alloc_cache(W.FP8_E4M3, nb, hkv, d, bs)
    kb, vb = W.to_bits(kx, W.BF16), W.to_bits(vx, W.BF16)
    oracle.kv_write(kb, vb, W.BF16, slots, k, v, s, W.FP8_E4M3, nb, hkv, d, bs)
    kf, vf = W.bits_to_f32(kb, W.BF16), W.bits_to_f32(vb, W.BF16)
    for which, arr in ((0, kf), (1, vf)):
        for blk, sel in ((2, slice(0, 16)), (0, slice(16, 20))):
            for h in range(hkv):
                want = max(np.float32(np.abs(arr[sel, h]).max()) / np.float32(448.0),
                           np.float32(1e-12))
                assert s[which, blk, h] == np.float32(want), (which, blk, h)
    assert s[0, 2, 1] == np.float32(np.float32(40.0) / np.float32(448.0))
    assert s[0, 0, 0] == np.float32(np.float32(33.0) / np.float32(448.0))
    assert not s[:, 1].any() and not s[:, 3].any()       # untouched blocks


def test_write_int4_round_trip_bound_and_extremes():
    rng = np.random.default_rng(6)
    rows = (rng.standard_normal((4, 64)) * np.array([[1], [10], [0.01], [300]])).astype(np.float32)
    k, v, s, x = _one_block_write(W.INT4_G32, rows, [0, 1, 2, 3])
    for i in range(4):
        xr = W.bits_to_f32(x[i, 0], W.BF16).astype(np.float64)
        codes = np.empty(64, np.int64)
        codes[0::2] = k[1, 0, i] & 0xF
        codes[1::2] = k[1, 0, i] >> 4
        for g in range(2):
            sc = np.float16(s[0, 1, 0, i, g, 0].view(np.float16)).astype(np.float64)
            z = np.float16(s[0, 1, 0, i, g, 1].view(np.float16)).astype(np.float64)
            seg = xr[32 * g:32 * (g + 1)]
            c = codes[32 * g:32 * (g + 1)]
            assert c.min() >= 0 and c.max() <= 15
            assert c[np.argmin(seg)] == 0 and c[np.argmax(seg)] == 15
            rec = c * sc + z
            # half a step, plus the fp16 rounding of the zero point
            assert np.all(np.abs(rec - seg) <= sc / 2 + abs(z - seg.min()) + 1e-6 * np.abs(seg).max())
            # the dequantizer reads the same layout
            row = oracle.dequant_row(k, s, 0, W.INT4_G32, 3, 1, 64, 16, 1, 0, i)
            assert np.allclose(row[32 * g:32 * (g + 1)], rec, rtol=0, atol=1e-12)


def test_write_int4_worked_example():
    # one group holding 0..31: min 0, max 31 -> scale fp16(31/15) = 2.06640625, zero 0
    row = np.concatenate([np.arange(32), np.full(32, 7.0)]).astype(np.float32)
    k, v, s, x = _one_block_write(W.INT4_G32, row[None], [0])
    assert s[0, 1, 0, 0, 0, 0].view(np.float16) == np.float16(2.06640625)
    assert s[0, 1, 0, 0, 0, 1].view(np.float16) == 0
    codes = np.empty(64, np.int64)
    codes[0::2] = k[1, 0, 0] & 0xF
    codes[1::2] = k[1, 0, 0] >> 4
    # i / 2.0664 rounded: 0,0,1,1,2,2,3,3,4,4,5,5,6,6,7,7,8,8,9,9,10,10,11,11,12,12,13,13,14,14,15,15
    assert list(codes[:32]) == [i // 2 for i in range(32)]
    # a constant group: range 0 -> scale 0 -> every code 0, zero = the value
    assert s[0, 1, 0, 0, 1, 0].view(np.float16) == 0
    assert s[0, 1, 0, 0, 1, 1].view(np.float16) == np.float16(7.0)
    assert not codes[32:].any()


def test_write_skips_negative_slots():
    k, v, s, x = _one_block_write(W.F16, np.ones((1, 64)), [0], dtype=W.F16)
    k2 = k.copy()
    oracle.kv_write(x, x, W.F16, np.array([-1], np.int64), k2, v, s, W.F16, 3, 1, 64, 16)
    assert np.array_equal(k, k2)


# ------------------------------------------------------------------ attention
def _dense_reference(q, kd, vd, scale, group):
    """torch SDPA (fp64) on contiguous K/V: q [Hq, D], kd/vd [Hkv, T, D]."""
    qt = torch.from_numpy(q)[None, :, None, :]                       # [1, Hq, 1, D]
    kt = torch.from_numpy(kd).repeat_interleave(group, 0)[None]      # [1, Hq, T, D]
    vt = torch.from_numpy(vd).repeat_interleave(group, 0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, :, 0, :].numpy()


def _gathered(case, k, v, s, b):
    """Dequantize sequence b's K/V by an independent route (library decoders)."""
    w = case.w
    n = int(case.context_lens[b])
    bs, h, d = w.block_size, w.num_kv_heads, w.head_dim
    kd = np.zeros((h, n, d))
    vd = np.zeros((h, n, d))
    for t in range(n):
        p = case.block_tables[b, t // bs]
        o = t % bs
        for j, (cache, out) in enumerate(((k, kd), (v, vd))):
            raw = cache[p, :, o]
            if w.kv_dtype == W.F16:
                out[:, t] = raw.view(np.float16).astype(np.float64)
            elif w.kv_dtype == W.BF16:
                out[:, t] = torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16).double().numpy()
            elif w.kv_dtype in W.FP8_TYPES:
                fmt = torch.float8_e4m3fn if w.kv_dtype == W.FP8_E4M3 else torch.float8_e5m2
                dec = torch.from_numpy(np.ascontiguousarray(raw)).view(fmt).double().numpy()
                out[:, t] = dec * s[j, p, :, None].astype(np.float64)
            elif w.kv_dtype == W.INT8:
                out[:, t] = raw.view(np.int8).astype(np.float64) * s[j, p, :, None].astype(np.float64)
            else:
                lo = (raw & 0xF).astype(np.float64)
                hi = (raw >> 4).astype(np.float64)
                codes = np.stack([lo, hi], -1).reshape(h, d)
                sz = s[j, p, :, o].view(np.float16).astype(np.float64)   # [h, D/32, 2]
                out[:, t] = codes * np.repeat(sz[..., 0], 32, 1) + np.repeat(sz[..., 1], 32, 1)
    return kd, vd


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, "3-e5m2", "3-int8"])
def test_attention_matches_sdpa_on_gathered_kv(cfg):
    if cfg == "3-e5m2":
        w = W.CONFIGS[3].scaled(batch=3, ctx_cap=70, seed=106, kv_dtype=W.FP8_E5M2)
    elif cfg == "3-int8":
        w = W.CONFIGS[3].scaled(batch=3, ctx_cap=70, seed=107, kv_dtype=W.INT8)
    else:
        w = W.CONFIGS[cfg].scaled(batch=3, ctx_cap=70, seed=100 + cfg)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    out = oracle.step_case(case, k, v, s)
    for b in range(w.batch):
        q = W.bits_to_f32(case.q[b], w.q_dtype).astype(np.float64)
        kd, vd = _gathered(case, k, v, s, b)
        ref = _dense_reference(q, kd, vd, w.softmax_scale, w.group)
        assert np.allclose(out[b], ref, rtol=0, atol=1e-12), (cfg, b)


def _tiny_case(cfg=1, **kw):
    w = W.CONFIGS[cfg].scaled(**kw)
    return W.make_case(w)


def test_attention_gqa_mapping_uses_contiguous_groups():
    w = W.Workload("gqa", 1, 8, 4, 64, 16, W.F16, W.F16, "fixed", 20, 20, pool_blocks=4, seed=9)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, 4, 64, 16)
    for h in range(4):
        v[:, h] = np.float16(h + 1).view(np.uint16)
    out = oracle.decode_attention(case.q, w.q_dtype, k, v, case.block_tables, case.context_lens,
                                  s, w.kv_dtype, case.num_blocks, w.softmax_scale, 8, 4, 64, 16)
    for h in range(8):
        assert np.allclose(out[0, h], h // 2 + 1, atol=1e-12)


def test_attention_context_one_returns_v():
    case = _tiny_case(batch=4, ctx_cap=1, seed=21)
    k, v, s = oracle.prefill_case(case)
    out = oracle.step_case(case, k, v, s)
    for b in range(4):
        p = case.block_tables[b, 0]
        vrow = v[p, :, 0].view(np.float16).astype(np.float64)         # [Hkv, D]
        assert np.array_equal(out[b], np.repeat(vrow, 4, 0))


def test_attention_constant_keys_give_mean_of_values():
    case = _tiny_case(batch=2, seed=22)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, 0, case.new_slots, k, v, s, 0, case.num_blocks, 2,
                    64, 16)
    k[:] = np.float16(0.37).view(np.uint16)
    out = oracle.decode_attention(case.q, 0, k, v, case.block_tables, case.context_lens, s, 0,
                                  case.num_blocks, 0.125, 8, 2, 64, 16)
    for b in range(2):
        n = case.context_lens[b]
        rows = np.stack([v[case.block_tables[b, t // 16], :, t % 16] for t in range(n)])
        mean = rows.view(np.float16).astype(np.float64).mean(0)
        assert np.allclose(out[b], np.repeat(mean, 4, 0), atol=1e-12)


def test_attention_two_token_closed_form():
    # q = e0, K0 = 0, K1 = ln(3)/scale * e0: weights exactly 1/4 and 3/4
    w = W.Workload("two", 1, 1, 1, 64, 16, W.BF16, W.BF16, "fixed", 2, 2, pool_blocks=2, seed=1)
    case = W.make_case(w)
    k, v, s = oracle.alloc_cache(W.BF16, 2, 1, 64, 16)
    q = np.zeros((1, 1, 64), np.float32); q[0, 0, 0] = 1.0
    p = case.block_tables[0, 0]
    kk = np.zeros((2, 64), np.float64)
    kk[1, 0] = math.log(3.0) * 8.0
    vv = np.zeros((2, 64), np.float64); vv[0] = 1.0; vv[1] = -1.0
    # use values exactly representable in bf16 by picking the scale from the stored key
    kbits = W.to_bits(kk.astype(np.float32), W.BF16)
    k[p, 0, :2] = kbits
    v[p, 0, :2] = W.to_bits(vv.astype(np.float32), W.BF16)
    stored = float(W.bits_to_f32(kbits[1:2, :1], W.BF16)[0, 0])
    scale = math.log(3.0) / stored
    out = oracle.decode_attention(W.to_bits(q, W.BF16), W.BF16, k, v, case.block_tables,
                                  case.context_lens, None, W.BF16, 2, scale, 1, 1, 64, 16)
    assert np.allclose(out[0, 0], 0.25 * 1 + 0.75 * -1, atol=1e-14)


def test_attention_context_zero_gives_zeros():
    case = _tiny_case(batch=2, seed=23)
    k, v, s = oracle.prefill_case(case)
    cl = case.context_lens.copy(); cl[1] = 0
    out = oracle.decode_attention(case.q, 0, k, v, case.block_tables, cl, s, 0, case.num_blocks,
                                  0.125, 8, 2, 64, 16)
    assert not out[1].any() and out[0].any()


def test_attention_masks_tokens_past_context():
    case = _tiny_case(batch=3, seed=24)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, 0, case.new_slots, k, v, s, 0, case.num_blocks, 2,
                    64, 16)
    args = (case.block_tables, case.context_lens, s, 0, case.num_blocks, 0.125, 8, 2, 64, 16)
    out = oracle.decode_attention(case.q, 0, k, v, *args)
    k2, v2 = k.copy(), v.copy()
    for b in range(3):
        n = case.context_lens[b]
        last = case.block_tables[b, (n - 1) // 16]
        k2[last, :, (n - 1) % 16 + 1:] = np.float16(300.0).view(np.uint16)
        v2[last, :, (n - 1) % 16 + 1:] = np.float16(-300.0).view(np.uint16)
    out2 = oracle.decode_attention(case.q, 0, k2, v2, *args)
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("cfg", [1, 3, 4])
def test_attention_invariant_under_block_permutation(cfg):
    w = W.CONFIGS[cfg].scaled(batch=3, ctx_cap=90, seed=30 + cfg)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    out = oracle.step_case(case, k, v, s)
    rng = np.random.default_rng(1)
    perm = rng.permutation(case.num_blocks)                # new id of old block i = perm[i]
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm], v2[perm] = k, v
    s2 = None
    if s is not None:
        s2 = np.empty_like(s)
        s2[:, perm] = s
    bt = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1).astype(np.int32)
    out2 = oracle.decode_attention(case.q, w.q_dtype, k2, v2, bt, case.context_lens, s2,
                                   w.kv_dtype, case.num_blocks, w.softmax_scale, w.num_q_heads,
                                   w.num_kv_heads, w.head_dim, w.block_size)
    assert np.array_equal(out, out2)


def test_attention_paged_equals_contiguous_layout():
    w = W.CONFIGS[2].scaled(batch=2, ctx_cap=100, seed=41)
    a = W.make_case(w)
    b = W.make_case(w, identity_tables=True)
    assert np.array_equal(a.prefill_k, b.prefill_k)
    ka, va, sa = oracle.prefill_case(a)
    kb, vb, sb = oracle.prefill_case(b)
    oa = oracle.step_case(a, ka, va, sa)
    ob = oracle.step_case(b, kb, vb, sb)
    assert np.array_equal(oa, ob)


def test_attention_pairs_match_full():
    w = W.CONFIGS[3].scaled(batch=4, ctx_cap=64, seed=51)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    full = oracle.step_case(case, k, v, s)
    ps = np.array([0, 3, 2, 1]); ph = np.array([5, 0, 31, 17])
    sub = oracle.decode_attention_pairs(case.q, w.q_dtype, k, v, case.block_tables,
                                        case.context_lens, s, w.kv_dtype, case.num_blocks,
                                        w.softmax_scale, w.num_q_heads, w.num_kv_heads,
                                        w.head_dim, w.block_size, ps, ph)
    assert np.array_equal(sub, full[ps, ph])


# ------------------------------------------------------------------ block copies
@pytest.mark.parametrize("kv", [W.F16, W.BF16, W.FP8_E4M3, W.FP8_E5M2, W.INT4_G32])
def test_copy_blocks_equals_numpy_block_assignment(kv):
    """Block dst of [NB, Hkv, bs, row] (and its scales) becomes block src."""
    qd = W.F16 if kv == W.F16 else W.BF16
    w = W.Workload("copy", 4, 8, 2, 64, 16, kv, qd, "uniform", 20, 60, seed=31 + kv)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    pairs = np.array([[case.block_tables[0, 0], 3], [case.block_tables[1, 1], 5],
                      [7, 7]], np.int32)
    ek, ev = k.copy(), v.copy()
    es = None if s is None else s.copy()
    for src, dst in pairs:
        ek[dst] = ek[src]
        ev[dst] = ev[src]
        if es is not None:
            es[:, dst] = es[:, src]         # FP8 [2, NB, Hkv]; INT4 [2, NB, Hkv, bs, D/32, 2]
    skipped = oracle.copy_blocks(k, v, s, kv, pairs, case.num_blocks, w.num_kv_heads,
                                 w.head_dim, w.block_size)
    assert skipped == 0
    assert np.array_equal(k, ek) and np.array_equal(v, ev)
    if s is not None:
        assert np.array_equal(s.view(np.uint8), es.view(np.uint8))


def test_copy_blocks_skips_out_of_range_ids():
    w = W.Workload("copy", 2, 4, 1, 64, 16, W.FP8_E4M3, W.BF16, "fixed", 20, 20, seed=3)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    before = (k.copy(), v.copy(), s.copy())
    pairs = np.array([[-1, 2], [1, case.num_blocks], [case.num_blocks + 5, 0]], np.int32)
    assert oracle.copy_blocks(k, v, s, w.kv_dtype, pairs, case.num_blocks, 1, 64, 16) == 3
    for a, b in zip(before, (k, v, s)):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("kv", [W.FP8_E4M3, W.INT4_G32, W.BF16])
def test_copy_on_write_fork_attends_like_the_shared_block(kv):
    """A sequence whose table points at a copied block attends exactly as it did
    through the original (the copy-on-write invariant)."""
    w = W.CONFIGS[4].scaled(batch=3, ctx_cap=200, seed=55, kv_dtype=kv,
                            q_dtype=W.BF16, pool_blocks=64)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    ref = oracle.step_case(case, k, v, s)
    used = set(case.block_tables[case.block_tables >= 0].ravel().tolist())
    free = [b for b in range(case.num_blocks) if b not in used]
    tables = case.block_tables.copy()
    pairs = []
    for b in range(w.batch):                     # fork each sequence's first block
        src = tables[b, 0]
        dst = free.pop()
        pairs.append([src, dst])
        tables[b, 0] = dst
    assert oracle.copy_blocks(k, v, s, kv, np.array(pairs, np.int32), case.num_blocks,
                              w.num_kv_heads, w.head_dim, w.block_size) == 0
    out = oracle.decode_attention(case.q, w.q_dtype, k, v, tables, case.context_lens, s, kv,
                                  case.num_blocks, w.softmax_scale, w.num_q_heads,
                                  w.num_kv_heads, w.head_dim, w.block_size)
    assert np.array_equal(out, ref)


# ------------------------------------------------------------------ chunked prefill
def _full_cache(case):
    """The case's cache with every context token written (the new one included)."""
    w = case.w
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    return k, v, s


def _prefill(case, k, v, s, q, q_start, ctx=None):
    w = case.w
    return oracle.prefill_attention(q, w.q_dtype, q_start, k, v, case.block_tables,
                                    case.context_lens if ctx is None else ctx, s, w.kv_dtype,
                                    case.num_blocks, w.softmax_scale, w.num_q_heads,
                                    w.num_kv_heads, w.head_dim, w.block_size)


@pytest.mark.parametrize("kv", [W.BF16, W.FP8_E4M3, W.INT8, W.INT4_G32])
def test_prefill_matches_causal_sdpa_on_gathered_kv(kv):
    w = W.Workload("pf", 3, 8, 2, 64, 16, kv, W.BF16, "uniform", 20, 60, seed=40 + kv)
    case = W.make_case(w)
    k, v, s = _full_cache(case)
    n = [5, 1, 17]
    q, q_start = W.prefill_chunk(case, n)
    out = _prefill(case, k, v, s, q, q_start)
    for b in range(w.batch):
        kd, vd = _gathered(case, k, v, s, b)                  # [Hkv, ctx, D], torch decoders
        c = int(case.context_lens[b])
        rows = slice(q_start[b], q_start[b + 1])
        qb = W.bits_to_f32(q[rows], w.q_dtype).astype(np.float64)      # [n, Hq, D]
        pos = c - n[b] + np.arange(n[b])
        mask = torch.from_numpy(np.arange(c)[None, :] <= pos[:, None])  # [n, ctx]
        kt = torch.from_numpy(np.repeat(kd, w.group, 0))[None]          # [1, Hq, ctx, D]
        vt = torch.from_numpy(np.repeat(vd, w.group, 0))[None]
        qt = torch.from_numpy(qb.transpose(1, 0, 2).copy())[None]       # [1, Hq, n, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                               scale=w.softmax_scale)
        assert np.allclose(out[rows], ref[0].numpy().transpose(1, 0, 2), rtol=0, atol=1e-12), b


def test_prefill_chunk_split_invariance_and_decode_limit():
    w = W.Workload("pf", 2, 8, 4, 64, 16, W.FP8_E4M3, W.BF16, "fixed", 50, 50, seed=9)
    case = W.make_case(w)
    k, v, s = _full_cache(case)
    q, q_start = W.prefill_chunk(case, [12, 12])
    whole = _prefill(case, k, v, s, q, q_start)
    # the same queries as two chunks: the first 7 over a context 5 shorter, then the last 5
    first = np.concatenate([q[0:7], q[12:19]])
    out_a = _prefill(case, k, v, s, first, np.array([0, 7, 14], np.int32),
                     ctx=case.context_lens - 5)
    second = np.concatenate([q[7:12], q[19:24]])
    out_b = _prefill(case, k, v, s, second, np.array([0, 5, 10], np.int32))
    assert np.array_equal(whole[0:7], out_a[0:7]) and np.array_equal(whole[12:19], out_a[7:14])
    assert np.array_equal(whole[7:12], out_b[0:5]) and np.array_equal(whole[19:24], out_b[5:10])
    # a chunk of one is a decode step with that query
    one = _prefill(case, k, v, s, case.q, np.array([0, 1, 2], np.int32))
    dec = oracle.decode_attention(case.q, w.q_dtype, k, v, case.block_tables, case.context_lens,
                                  s, w.kv_dtype, case.num_blocks, w.softmax_scale,
                                  w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size)
    assert np.array_equal(one, dec)


def test_prefill_negative_positions_give_zeros():
    w = W.Workload("pf", 1, 4, 2, 64, 16, W.BF16, W.BF16, "fixed", 6, 6, seed=3)
    case = W.make_case(w)
    k, v, s = _full_cache(case)
    q, q_start = W.prefill_chunk(case, [9])               # 9 queries over 6 tokens
    out = _prefill(case, k, v, s, q, q_start)
    assert not out[:3].any()                              # positions -3, -2, -1
    assert np.abs(out[3:]).sum() > 0
