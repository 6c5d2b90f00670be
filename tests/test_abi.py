"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching the GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(paged_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import paged_quantized_kv_write_gb300 as pkv
    return pkv


def test_header_declares_the_two_calls():
    names = _declared()
    assert "paged_kv_write" in names and "paged_decode_attention" in names


def test_every_declared_symbol_is_exported(lib):
    dll = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared():
        assert hasattr(dll, name), name


def test_product_library_holds_no_comparators(lib):
    """The decode comparators (CUDA-core and tcgen05) and the bounded-wait test switch
    are compiled into the test build only; both builds export the same C ABI."""
    import subprocess
    test_path = os.path.join(os.path.dirname(lib.LIB_PATH), "libpagedkv_test.so")
    test_dll = ctypes.CDLL(test_path)
    for name in _declared():
        assert hasattr(test_dll, name), name

    def symbols(path):
        r = subprocess.run(["nm", "-C", path], capture_output=True, text=True, check=True)
        return r.stdout

    prod, test = symbols(lib.LIB_PATH), symbols(test_path)
    for marker in ("simt_decode_kernel", "decode_tc_kernel", "launch_simt", "launch_decode_tc"):
        assert marker not in prod, marker
        assert marker in test, marker


def test_version_and_status_strings(lib):
    assert lib.version() == 100
    assert lib.lib.paged_kv_status_string(0) == b"ok"
    assert b"outside" in lib.lib.paged_kv_status_string(4)
    assert b"timed out" in lib.lib.paged_kv_status_string(8)
    assert lib.lib.paged_kv_status_string(99) == b"unknown status"


def test_binding_constants_match_the_header(lib):
    """Every enumerator of the header's dtype and status enums has the same value
    in the Python binding."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    enums = dict((n, int(v)) for n, v in re.findall(r"\b(PKV_[A-Z0-9_]+)\s*=\s*(\d+)", src))
    assert "PKV_ERR_DEVICE_TIMEOUT" in enums and "PKV_INT8" in enums
    for name, value in enums.items():
        assert getattr(lib, name) == value, name


def test_host_validation_without_gpu(lib):
    L = lib.lib
    V = ctypes.c_void_p
    fake = V(0x10000)          # never dereferenced: validation fails first
    # num_q_heads not a multiple of num_kv_heads
    assert L.paged_decode_attention(fake, 1, fake, fake, fake, 4, fake, 2, None, 1, 10, fake,
                                    0.1, 6, 4, 128, 16, 0, None, 0, None, None) == 1
    # unsupported head_dim
    assert L.paged_decode_attention(fake, 1, fake, fake, fake, 4, fake, 2, None, 1, 10, fake,
                                    0.1, 8, 2, 96, 16, 0, None, 0, None, None) == 2
    # 16-bit cache with a different q dtype
    assert L.paged_decode_attention(fake, 0, fake, fake, fake, 4, fake, 2, None, 1, 10, fake,
                                    0.1, 8, 2, 128, 16, 0, None, 0, None, None) == 2
    # group larger than 8
    assert L.paged_decode_attention(fake, 1, fake, fake, fake, 4, fake, 2, None, 1, 10, fake,
                                    0.1, 32, 2, 128, 16, 0, None, 0, None, None) == 2
    # FP8 without scales
    assert L.paged_decode_attention(fake, 1, fake, fake, fake, 4, fake, 2, None, 2, 10, fake,
                                    0.1, 8, 2, 128, 16, 0, None, 0, None, None) == 1
    # misaligned q
    assert L.paged_decode_attention(V(0x10002), 1, fake, fake, fake, 4, fake, 2, None, 1, 10,
                                    fake, 0.1, 8, 2, 128, 16, 0, None, 0, None, None) == 1
    # a pool of 2^27 (block, KV head) pairs or more
    assert L.paged_decode_attention(fake, 1, fake, fake, fake, 4, fake, 2, None, 1, 1 << 24, fake,
                                    0.1, 64, 8, 128, 16, 0, None, 0, None, None) == 2
    # split-KV without workspace
    assert L.paged_decode_attention(fake, 1, fake, fake, fake, 400, fake, 2, None, 1, 10, fake,
                                    0.1, 8, 2, 128, 16, 64, None, 0, None, None) == 5
    # more (sequence, q head) pairs than a 1-D grid holds: 65535 x 65535*8 heads
    assert L.paged_decode_attention(fake, 1, fake, fake, fake, 4, fake, 65535, None, 1, 10,
                                    fake, 0.1, 8 * 65535, 65535, 128, 16, 0, None, 0, None,
                                    None) == 2
    # split-KV partial rows beyond 2^40 (65535 seqs x 32768 heads x 2^24 partitions of 16):
    # refused up front, and the size query answers 0 rather than a wrapped count
    assert L.paged_decode_attention(fake, 1, fake, fake, fake, (1 << 31) // 16 - 1, fake, 65535,
                                    None, 1, 10, fake, 0.1, 32768, 4096, 128, 16, 16, None, 0,
                                    None, None) == 2
    assert lib.paged_decode_workspace_bytes(65535, 32768, 4096, 128, (1 << 31) // 16 - 1, 16,
                                            16) == 0
    # a partition request near INT_MAX is clamped, not wrapped
    assert lib.paged_decode_partition_size(4, 8, 2, 8, 16, 0x7FFFFFFF) > 0
    # bad block size, bad dtype, NULL buffers on the write
    assert L.paged_kv_write(fake, fake, 1, fake, 4, fake, fake, None, 1, 10, 2, 128, 24,
                            None, None) == 2
    assert L.paged_kv_write(fake, fake, 1, fake, 4, fake, fake, None, 7, 10, 2, 128, 16,
                            None, None) == 2
    assert L.paged_kv_write(None, fake, 1, fake, 4, fake, fake, None, 1, 10, 2, 128, 16,
                            None, None) == 1
    assert L.paged_kv_write(fake, fake, 1, fake, 4, fake, fake, None, 3, 10, 2, 128, 16,
                            None, None) == 1
    # a token count whose warp count would overflow the grid
    assert L.paged_kv_write(fake, fake, 1, fake, 1 << 40, fake, fake, None, 1, 10, 2, 128, 16,
                            None, None) == 2
    # zero tokens / zero sequences are no-ops
    assert L.paged_kv_write(None, None, 1, None, 0, None, None, None, 1, 10, 2, 128, 16,
                            None, None) == 0


def test_workspace_and_partition_queries(lib):
    # short contexts: one partition, no workspace
    assert lib.paged_decode_workspace_bytes(4, 8, 2, 64, 8, 16) == 0
    assert lib.paged_decode_partition_size(4, 8, 2, 8, 16) == 128
    # explicit partition: B * Hq * NP * (D + 2) floats (+ alignment)
    n = lib.paged_decode_workspace_bytes(16, 64, 8, 128, 2048, 16, 512)
    assert n >= 16 * 64 * 64 * 130 * 4
    assert lib.paged_decode_partition_size(16, 64, 8, 2048, 16, 500) == 512


@pytest.mark.parametrize("cfg,expected", [(2, 1024), (3, 512), (4, 512), (5, 512)])
def test_partition_heuristic_and_workspace_for_the_benchmark_workloads(lib, cfg, expected):
    """The library's own partition choice for each benchmark workload (the one the
    block-size / partition sweep found best or within 1.5% of it), and the
    workspace it needs: one fp32 row of head_dim per (sequence, q head,
    partition), 256-byte aligned, then (max, sum) per partition."""
    import workloads as W
    w = W.CONFIGS[cfg]
    mb = -(-w.ctx_hi // w.block_size)            # the table width of the longest context
    part = lib.lib.paged_decode_partition_size(w.batch, w.num_q_heads, w.num_kv_heads, mb,
                                               w.block_size, 0)
    assert part == expected and part % 16 == 0
    np_ = -(-mb * w.block_size // part)
    heads = w.batch * w.num_q_heads
    out_bytes = heads * np_ * w.head_dim * 4
    want = (-(-out_bytes // 256)) * 256 + heads * np_ * 2 * 4
    # ... or the balanced split's layout when that is larger and the call may take
    # it: (2432 warp slots + one per (sequence, KV head)) x G rows of head_dim
    # floats, then (max, sum) per row from a 256-byte boundary
    tiles = -(-mb * w.block_size // 16)
    if np_ > 1 and w.batch <= 512 and w.batch * w.num_kv_heads * tiles < 2**30:
        rows = (2432 + w.batch * w.num_kv_heads) * (w.num_q_heads // w.num_kv_heads)
        want = max(want, -(-(rows * w.head_dim * 4) // 256) * 256 + rows * 2 * 4)
    got = lib.lib.paged_decode_workspace_bytes(w.batch, w.num_q_heads, w.num_kv_heads,
                                               w.head_dim, mb, w.block_size, 0)
    assert got == want
    # an explicit request is rounded up to a multiple of 16 tokens
    assert lib.lib.paged_decode_partition_size(w.batch, w.num_q_heads, w.num_kv_heads, mb,
                                               w.block_size, 100) == 112
