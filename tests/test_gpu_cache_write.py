"""GPU parity of pa_kv_cache_write / pa_copy_blocks: bit-exact against the
oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import dev_status
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
TD = W.TORCH_DTYPE


def _setup(seed, nb, hkv, bs, d, kv_dtype):
    g = torch.Generator().manual_seed(seed)
    kc = W.random_values(g, (nb, hkv, bs, d), kv_dtype)
    vc = W.random_values(g, (nb, hkv, bs, d), kv_dtype)
    return kc, vc


@pytest.mark.parametrize("kv_dtype,in_dtype", [(W.F16, W.F16), (W.BF16, W.BF16), (W.E4M3, W.F16),
                                                (W.E4M3, W.BF16)])
@pytest.mark.parametrize("T,stride_pad,hkv,d", [(1, 0, 4, 64), (37, 0, 8, 128), (1000, 3 * 128 * 8, 8, 128),
                                                (5, 7, 2, 64)])
def test_cache_write_bit_exact(kv_dtype, in_dtype, T, stride_pad, hkv, d):
    bs, nb = 16, 200
    kc, vc = _setup(1, nb, hkv, bs, d, kv_dtype)
    g = torch.Generator().manual_seed(2)
    row = hkv * d + stride_pad
    kin = W.random_values(g, (T, row), in_dtype) * 40  # reaches E4M3 saturation
    vin = W.random_values(g, (T, row), in_dtype)
    rng = np.random.default_rng(3)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[rng.random(T) < 0.1] = -1
    ks, vs = (0.5, 1.75) if kv_dtype == W.E4M3 else (1.0, 1.0)
    cache = pk.KVCache(kc.to(DEV), vc.to(DEV), ks, vs)
    st = dev_status()
    kd, vd = kin.to(DEV), vin.to(DEV)
    pk.pa_kv_cache_write(cache, kd[:, :hkv * d] if stride_pad else kd.view(T, hkv, d),
                         vd[:, :hkv * d] if stride_pad else vd.view(T, hkv, d), torch.from_numpy(slots).to(DEV), st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kref, vref = W.as_bits(kc), W.as_bits(vc)
    assert oracle.cache_write(kref, vref, kv_dtype, W.as_bits(kin), W.as_bits(vin), in_dtype, slots, ks, vs,
                              token_stride=row) == 0
    assert np.array_equal(W.as_bits(cache.k_cache), kref)
    assert np.array_equal(W.as_bits(cache.v_cache), vref)


def test_e4m3_quantize_all_f16_codes():
    """Every finite fp16 value through the fp8 write, against the oracle's codec."""
    codes = np.arange(65536, dtype=np.uint16)
    finite = (codes & 0x7c00) != 0x7c00
    codes = codes[finite]
    T = codes.size // 64
    codes = codes[:T * 64]
    kin = torch.from_numpy(codes.view(np.int16).reshape(T, 1, 64)).view(torch.float16)
    nb, bs = (T + 15) // 16, 16
    kc = torch.zeros((nb, 1, bs, 64), dtype=torch.float8_e4m3fn)
    cache = pk.KVCache(kc.to(DEV), kc.clone().to(DEV), 1.0, 3.0)
    slots = np.arange(T, dtype=np.int64)
    pk.pa_kv_cache_write(cache, kin.to(DEV), kin.to(DEV), torch.from_numpy(slots).to(DEV))
    torch.cuda.synchronize()
    kref = W.as_bits(kc)
    vref = kref.copy()
    oracle.cache_write(kref, vref, W.E4M3, codes.reshape(T, 1, 64), codes.reshape(T, 1, 64), W.F16, slots, 1.0, 3.0)
    assert np.array_equal(W.as_bits(cache.k_cache), kref)
    assert np.array_equal(W.as_bits(cache.v_cache), vref)


def test_bad_slot_is_reported_and_skipped():
    kc, vc = _setup(4, 4, 2, 16, 64, W.F16)
    cache = pk.KVCache(kc.to(DEV), vc.to(DEV))
    g = torch.Generator().manual_seed(5)
    kin = W.random_values(g, (3, 2, 64), W.F16)
    slots = torch.tensor([3, 64, 5], dtype=torch.int64)  # 64 = 4 blocks * 16: outside
    st = dev_status()
    pk.pa_kv_cache_write(cache, kin.to(DEV), kin.to(DEV), slots.to(DEV), st)
    torch.cuda.synchronize()
    assert st.item() == 6
    kref, vref = W.as_bits(kc), W.as_bits(vc)
    oracle.cache_write(kref, vref, W.F16, W.as_bits(kin), W.as_bits(kin), W.F16, np.array([3, -1, 5]))
    assert np.array_equal(W.as_bits(cache.k_cache), kref)


@pytest.mark.parametrize("kv_dtype", [W.F16, W.E4M3])
def test_copy_blocks_bit_exact(kv_dtype):
    kc, vc = _setup(6, 12, 8, 16, 128, kv_dtype)
    cache = pk.KVCache(kc.to(DEV), vc.to(DEV))
    pairs = np.array([[1, 7], [3, 0], [11, 2]], np.int32)
    st = dev_status()
    pk.pa_copy_blocks(cache, torch.from_numpy(pairs).to(DEV), st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kref, vref = W.as_bits(kc), W.as_bits(vc)
    oracle.copy_blocks(kref, vref, kv_dtype, pairs)
    assert np.array_equal(W.as_bits(cache.k_cache), kref)
    assert np.array_equal(W.as_bits(cache.v_cache), vref)
    bad = torch.tensor([[0, 99]], dtype=torch.int32, device=DEV)
    pk.pa_copy_blocks(cache, bad, st)
    torch.cuda.synchronize()
    assert st.item() == 6
