"""A decode whose waits run out ends with PA_ERR_TIMEOUT and leaves the GPU
usable.

Every mbarrier wait in the library's kernels is bounded (2 s), so that a copy
that never lands ends in an error status instead of a hung GPU.  The test hook
pa_decode_test_wait_timeout launches the decode with a producer warp that
issues no copy at all: the consumers' waits for the query and the first pages
run out with nothing in flight, the kernel writes PA_ERR_TIMEOUT (5) to the
status word and returns.  A plain pa_decode on the same stream afterwards must
still match the oracle.  Both consumers are covered (one query head per KV
head on CUDA cores, four on tensor cores), with and without split-K.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("G,P", [(1, 0), (4, 0), (4, 128)])
def test_decode_wait_runs_out_then_decode_still_correct(G, P):
    lens = [100, 700, 33, 1]
    case = W.make_decode_case(21 + G, lens, 4 * G, 4, 128, 16, 80, W.BF16, W.BF16)
    q = case.q.to(DEV)
    cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    bt, sl = case.block_table.to(DEV), case.seq_lens.to(DEV)
    max_len = max(lens)
    ws = torch.empty(max(16, pk.pa_decode_workspace_size(4, 4 * G, 128, max_len, 16, P)), dtype=torch.uint8,
                     device=DEV)
    out = torch.zeros_like(q)
    st = dev_status()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    pk.pa_decode_test_wait_timeout(out, q, cache, bt, sl, max_len, case.scale, P, ws, st)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert int(st.item()) == 5  # PA_ERR_TIMEOUT
    assert 1.0 < waited < 60.0  # the wait limit ran out, then the kernel returned
    # the context is intact: a normal decode on the same stream is correct
    st2 = dev_status()
    out2 = torch.empty_like(q)
    pk.pa_decode(out2, q, cache, bt, sl, max_len, case.scale, P, ws, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    _, ref, rc = oracle.decode(W.as_bits(case.q), W.BF16, W.as_bits(case.k_cache), W.as_bits(case.v_cache), W.BF16,
                               case.block_table.numpy(), np.asarray(lens, np.int32), case.scale)
    assert rc == 0
    assert_close(W.as_bits(out2), ref, W.BF16, W.BF16, "after the timeout")
