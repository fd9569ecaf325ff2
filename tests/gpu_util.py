"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

from paged_kv_cache_75_gb300 import workloads as W

RTOL = {W.F16: 1e-2, W.BF16: 1e-2, W.E4M3: 3e-2}  # relative part, by KV dtype
ATOL = 2e-3


def values(bits, dtype):
    bits = np.ascontiguousarray(bits)
    if dtype == W.E4M3:
        t = torch.from_numpy(bits.view(np.uint8)).view(torch.float8_e4m3fn)
    else:
        t = torch.from_numpy(bits.view(np.int16)).view(torch.float16 if dtype == W.F16 else torch.bfloat16)
    return t.to(torch.float64).numpy()


def assert_close(gpu_bits, ref64, out_dtype, kv_dtype, what=""):
    """|gpu - ref| <= 2e-3 + rel * |ref| element by element (rel = 1e-2 for
    16-bit caches, 3e-2 for an E4M3 cache); ref is the oracle's fp64 value."""
    g = values(gpu_bits, out_dtype)
    ref = np.asarray(ref64)
    assert np.all(np.isfinite(g)), "non-finite GPU output %s" % what
    err = np.abs(g - ref)
    lim = ATOL + RTOL[kv_dtype] * np.abs(ref)
    bad = err > lim
    if bad.any():
        i = np.unravel_index(np.argmax(err - lim), err.shape)
        raise AssertionError("%s: %d/%d elements off; worst at %s gpu=%r ref=%r (max abs err %.3g)"
                             % (what, int(bad.sum()), bad.size, i, g[i], ref[i], err.max()))
    return float(err.max())


def dev_status(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)
