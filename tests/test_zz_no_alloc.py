"""paged_decode_attention_noalloc — decode attention for callers that cannot allocate.

Some callers cannot call cudaMalloc: code inside a custom allocator's own
callbacks, processes whose device memory is one fixed pool handed out up
front, runtimes that forbid allocation on their hot path, plain C callers
with no allocator.  For them the library takes the split-KV scratch from a
static device array of its own (64 MiB per GPU).  This file checks, through
the C ABI, that the allocation-free entry point returns what the regular
entry point returns with a caller-supplied workspace, on two calls in a row
(the second call must not be disturbed by what the first left in the shared
array), and that a request too large for the array is refused up front.

It is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu

P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float


def _entry():
    import paged_quantized_kv_write_gb300 as pkv
    f = pkv.lib.paged_decode_attention_noalloc
    f.argtypes = [P, I, P, P, P, I, P, I, P, I, I, P, F, I, I, I, I, I, P, P]
    f.restype = I
    return f


def _call_noalloc(g: H.GpuCase, out: torch.Tensor) -> int:
    w = g.w
    ptr = lambda t: None if t is None else P(t.data_ptr())     # noqa: E731
    r = _entry()(ptr(g.q), w.q_dtype, ptr(g.k), ptr(g.v), ptr(g.tables),
                 g.case.max_blocks_per_seq, ptr(g.ctx), w.batch, ptr(g.s), w.kv_dtype,
                 g.case.num_blocks, ptr(out), w.softmax_scale, w.num_q_heads, w.num_kv_heads,
                 w.head_dim, w.block_size, g.partition_size, ptr(g.status),
                 P(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return r


def _gpu_case(kv, seed):
    w = W.Workload("noalloc", 6, 16, 2, 128, 16, kv, W.BF16, "uniform", 1, 700, seed=seed)
    case = W.make_case(w)
    k, v, s = oracle.prefill_case(case)
    oracle.kv_write(case.k_new, case.v_new, w.q_dtype, case.new_slots, k, v, s, w.kv_dtype,
                    case.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
    return H.GpuCase(case, k, v, s, partition_size=64), (k, v, s)


@pytest.mark.parametrize("kv", [W.BF16, W.FP8_E4M3, W.INT4_G32])
def test_noalloc_matches_regular_entry_point_twice(kv):
    for seed in (11, 12):                       # two calls in a row, different inputs
        g, (k, v, s) = _gpu_case(kv, seed + kv)
        ref = g.attend()                        # regular entry point, torch workspace
        assert g.status.item() == 0
        g.status.zero_()
        out = torch.full_like(g.q, float("nan"))
        assert _call_noalloc(g, out) == 0
        got = H.tensor_to_f64(out)
        assert g.status.item() == 0
        # the same kernels with the same partitions: the same bits, whatever the
        # previous call left in the shared array
        assert np.array_equal(got, ref)
        H.check_close(got, H.oracle_attention(g.case, k, v, s), kv, W.BF16, "noalloc")


def test_noalloc_refuses_requests_beyond_its_scratch():
    fake = P(0x10000)                           # never dereferenced: refused before launch
    # 4096 sequences x 64 heads x 16 partitions x 130 floats is far beyond 64 MiB
    r = _entry()(fake, W.BF16, fake, fake, fake, 8192 // 16, fake, 4096, None, W.BF16, 10,
                 fake, 0.1, 64, 8, 128, 16, 512, None, None)
    assert r == 5                               # PKV_ERR_WORKSPACE
