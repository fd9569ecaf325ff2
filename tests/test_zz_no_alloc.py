"""pa_decode_static_ws: the decode entry point that allocates nothing.

Callers that cannot call cudaMalloc (a plugin whose host program owns all
device memory, a serving loop that may not synchronise the device) use the
scratch built into the library instead of a workspace of their own.  These
tests call it through the C ABI and check that its output is bit for bit
pa_decode's at the same partition (the same kernels on the same inputs) and
within the decode tolerance of the oracle, on two calls in a row that need the
split-K scratch, with different inputs, so that the second call runs over
what the first left in the shared array.  With partition_size 0 the call
resolves the automatic partition before checking the size, so a request that
fits the scratch at that partition is accepted.  The file is collected last on
purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status
from paged_kv_cache_75_gb300 import workloads as W
from paged_kv_cache_75_gb300 import build as pkg_build

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH = 16 * 1024 * 1024


def _call_static(lib, out, q, cache, bt, lens, max_len, scale, P, st):
    cs = cache.c_struct()
    B, H, _ = q.shape
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pa_decode_static_ws(C.c_void_p(out.data_ptr()), C.c_void_p(q.data_ptr()),
                                   pk.torch_dtype_code(q.dtype), C.byref(cs), C.c_void_p(bt.data_ptr()),
                                   bt.shape[1], C.c_void_p(lens.data_ptr()), B, max_len, H, scale, P,
                                   C.c_void_p(st.data_ptr()), stream)


def _reference(case, q, cache, bt, lens, max_len, P):
    out = torch.empty_like(q)
    ws = torch.empty(max(pk.pa_decode_workspace_size(q.shape[0], q.shape[1], q.shape[2], max_len,
                                                     case.block_size, P), 16), dtype=torch.uint8, device=DEV)
    st = dev_status()
    pk.pa_decode(out, q, cache, bt, lens, max_len, case.scale, P, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out


def _oracle(case):
    _, ref, rc = oracle.decode(W.as_bits(case.q), case.q_dtype, W.as_bits(case.k_cache), W.as_bits(case.v_cache),
                               case.kv_dtype, case.block_table.numpy(), case.seq_lens.numpy(), case.scale,
                               case.k_scale, case.v_scale)
    assert rc == 0
    return ref


def _check_twice(lib, cases, max_len, P):
    """Both cases in a row through the scratch; each bit-identical to
    pa_decode at the partition the call resolves to, and within tolerance of
    the oracle."""
    for case in cases:
        B, H, D = case.q.shape
        Peff = P or pk.pa_decode_partition_size(B, H, case.num_kv_heads, max_len)
        need = pk.pa_decode_workspace_size(B, H, D, max_len, case.block_size, Peff)
        assert 0 < need <= SCRATCH  # the split-K scratch is in use
        q = case.q.to(DEV)
        cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV), case.k_scale, case.v_scale)
        bt = case.block_table.to(DEV)
        sl = case.seq_lens.to(DEV)
        out = torch.full_like(q, float("nan"))
        st = dev_status()
        assert _call_static(lib, out, q, cache, bt, sl, max_len, case.scale, P, st) == 0
        torch.cuda.synchronize()
        assert st.item() == 0
        ref = _reference(case, q, cache, bt, sl, max_len, Peff)
        assert np.array_equal(W.as_bits(out), W.as_bits(ref)), "static scratch differs from pa_decode"
        assert_close(W.as_bits(out), _oracle(case), case.q_dtype, case.kv_dtype, "static scratch vs oracle")


@pytest.mark.parametrize("qd,kd", [(W.F16, W.F16), (W.BF16, W.E4M3)])
def test_static_scratch_decode_matches_pa_decode_twice(qd, kd):
    pkg_build.build()
    lib = pk.library()
    cases = []
    for seed, lens in ((1, [1, 130, 900, 2047, 64, 513]), (2, [2047, 3, 700, 1500, 257, 129])):
        case = W.make_decode_case(seed, lens, 16, 4, 128, 16, 800, qd, kd)
        if kd == W.E4M3:
            case.k_scale, case.v_scale = 0.5, 1.25
        cases.append(case)
    _check_twice(lib, cases, 2048, 128)


def test_static_scratch_automatic_partition_twice():
    # partition_size 0: four query heads per KV head, a few sequences over
    # 1024 tokens, so the automatic partition splits them and the partials
    # land in the scratch
    pkg_build.build()
    lib = pk.library()
    cases = [W.make_decode_case(seed, lens, 32, 8, 128, 16, 1200, W.BF16, W.BF16)
             for seed, lens in ((3, [1500, 4000, 1025, 17]), (4, [4096, 2, 3000, 1100]))]
    _check_twice(lib, cases, 4096, 0)


def test_static_scratch_long_context_shape_is_accepted():
    # the long-context shape (8 sequences, 64 query / 8 KV heads, up to 131072
    # tokens, E4M3, block size 32) needs about 8.4 MB of partials at the
    # automatic partition (4096 tokens): the call is accepted and runs; the
    # lengths attended here are short so that the oracle stays quick
    pkg_build.build()
    lib = pk.library()
    max_len = 131072
    assert pk.pa_decode_workspace_size(8, 64, 128, max_len, 32, 0) > SCRATCH  # sized at 512 it would not fit
    lens = [9000, 4097, 100, 1, 8192, 300, 5000, 64]
    case = W.make_decode_case(5, lens, 64, 8, 128, 32, sum(W.pages_for(x, 32) for x in lens) + 2, W.BF16, W.E4M3,
                              max_blocks=W.pages_for(max_len, 32))
    _check_twice(lib, [case], max_len, 0)


def test_static_scratch_rejects_oversized_requests():
    pkg_build.build()
    lib = pk.library()
    case = W.make_decode_case(3, [40, 40], 8, 8, 128, 16, 10, W.F16, W.F16)
    q = case.q.to(DEV)
    cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    out = torch.empty_like(q)
    # 2 seqs x 8 heads x 2^20 / 16 partitions x 129 floats: far beyond 16 MiB
    big = 1 << 20
    assert pk.pa_decode_workspace_size(2, 8, 128, big, 16, 16) > SCRATCH
    st = dev_status()
    rc = _call_static(lib, out, q, cache, case.block_table.to(DEV), case.seq_lens.to(DEV), big, case.scale, 16, st)
    assert rc == 2  # PA_ERR_UNSUPPORTED, nothing launched
