"""pa_decode_static_ws: the decode entry point that allocates nothing.

Callers that cannot call cudaMalloc (a plugin whose host program owns all
device memory, a serving loop that may not synchronise the device) use the
scratch built into the library instead of a workspace of their own.  This
test calls it through the C ABI and compares its output with pa_decode's
(same tolerance as the other decode tests), on two calls in a row that need
the split-K scratch, with different inputs, so that the second call runs over
what the first left in the shared array.  It is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status, values
from paged_kv_cache_75_gb300 import workloads as W
from paged_kv_cache_75_gb300 import build as pkg_build

pytestmark = pytest.mark.gpu
DEV = "cuda"


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


@pytest.mark.parametrize("qd,kd", [(W.F16, W.F16), (W.BF16, W.E4M3)])
def test_static_scratch_decode_matches_pa_decode_twice(qd, kd):
    pkg_build.build()
    lib = pk.library()
    P = 128
    for seed, lens in ((1, [1, 130, 900, 2047, 64, 513]), (2, [2047, 3, 700, 1500, 257, 129])):
        case = W.make_decode_case(seed, lens, 16, 4, 128, 16, 800, qd, kd)
        if kd == W.E4M3:
            case.k_scale, case.v_scale = 0.5, 1.25
        need = pk.pa_decode_workspace_size(len(lens), 16, 128, 2048, 16, P)
        assert 0 < need <= 16 * 1024 * 1024  # the split-K scratch is in use
        q = case.q.to(DEV)
        cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV), case.k_scale, case.v_scale)
        bt = case.block_table.to(DEV)
        sl = case.seq_lens.to(DEV)
        out = torch.full_like(q, float("nan"))
        st = dev_status()
        assert _call_static(lib, out, q, cache, bt, sl, 2048, case.scale, P, st) == 0
        torch.cuda.synchronize()
        assert st.item() == 0
        ref = _reference(case, q, cache, bt, sl, 2048, P)
        # same tolerance as the decode parity tests, against pa_decode's result
        assert_close(W.as_bits(out), values(W.as_bits(ref), qd), qd, kd, "static scratch vs pa_decode")


def test_static_scratch_rejects_oversized_requests():
    pkg_build.build()
    lib = pk.library()
    case = W.make_decode_case(3, [40, 40], 8, 8, 128, 16, 10, W.F16, W.F16)
    q = case.q.to(DEV)
    cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    out = torch.empty_like(q)
    # 2 seqs x 8 heads x 2^20 / 16 partitions x 129 floats: far beyond 16 MiB
    big = 1 << 20
    assert pk.pa_decode_workspace_size(2, 8, 128, big, 16, 16) > 16 * 1024 * 1024
    st = dev_status()
    rc = _call_static(lib, out, q, cache, case.block_table.to(DEV), case.seq_lens.to(DEV), big, case.scale, 16, st)
    assert rc == 2  # PA_ERR_UNSUPPORTED, nothing launched
