"""The C-ABI library loads, exports every function include/pa_kv.h declares,
and rejects bad arguments on the host before launching anything.  No GPU."""
import ctypes as C
import os
import re

import pytest

import paged_kv_cache_75_gb300 as pk
from paged_kv_cache_75_gb300 import build as pkg_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa_kv.h")


@pytest.fixture(scope="module")
def lib():
    pkg_build.build()
    return pk.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("pa_kv_cache_write", "pa_decode", "pa_prefill_varlen", "pa_pool_create", "pa_pool_append",
              "pa_copy_blocks", "pa_decode_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    assert pk.pa_status_str(0) == "ok"
    assert "block" in pk.pa_status_str(6)
    assert pk.pa_version() >= 100


def test_workspace_size_host_rule(lib):
    # one partition needs no workspace; more partitions need lse + partial rows
    assert pk.pa_decode_workspace_size(4, 8, 128, 512, 16, 512) == 0
    n = pk.pa_decode_workspace_size(4, 8, 128, 2048, 16, 512)
    rows = 4 * 8 * 4
    assert n >= rows * (128 + 1) * 4


FAKE = 1 << 20  # a 16-byte aligned, never dereferenced address


def _cache(**kw):
    c = pk._binding._Cache(FAKE, FAKE, 8, 16, 2, 128, pk.PA_F16, 1.0, 1.0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _decode(lib, cache, H=4, q_dtype=pk.PA_F16, bt=FAKE, sl=FAKE, ws=None, ws_bytes=0, P=0, max_len=64):
    return lib.pa_decode(FAKE, FAKE, q_dtype, C.byref(cache), bt, 4, sl, 2, max_len, H, 0.1, P, ws,
                         ws_bytes, None, None)


def test_decode_rejects_bad_arguments_before_launch(lib):
    assert _decode(lib, _cache(), H=3) == 1                      # H % Hkv != 0
    assert _decode(lib, _cache(head_size=96)) == 2               # head size not built
    assert _decode(lib, _cache(block_size=8)) == 2               # block size not built
    assert _decode(lib, _cache(), H=32) == 2                     # group 16 not built
    assert _decode(lib, _cache(), q_dtype=pk.PA_BF16) == 2       # q/cache dtype mismatch
    assert _decode(lib, _cache(k_cache=FAKE + 2)) == 1           # misaligned cache
    assert _decode(lib, _cache(), bt=None) == 1                  # null table
    assert _decode(lib, _cache(), P=24) == 1                     # partition not a block multiple
    assert _decode(lib, _cache(), max_len=4096, P=512) == 1      # split needs a workspace
    assert _decode(lib, _cache(kv_dtype=pk.PA_FP8_E4M3, k_scale=0.0)) == 1  # fp8 needs scales


def test_cache_write_and_prefill_reject_bad_arguments(lib):
    c = _cache()
    assert lib.pa_kv_cache_write(C.byref(c), FAKE, FAKE, pk.PA_BF16, 3, 256, FAKE, None, None) == 2
    assert lib.pa_kv_cache_write(C.byref(c), FAKE, FAKE, pk.PA_F16, 3, 100, FAKE, None, None) == 1
    assert lib.pa_kv_cache_write(C.byref(c), FAKE, FAKE, pk.PA_F16, 0, 256, FAKE, None, None) == 0
    assert lib.pa_copy_blocks(C.byref(c), None, 2, None, None) == 1
    c64 = _cache(head_size=64)
    assert lib.pa_prefill_varlen(FAKE, FAKE, pk.PA_F16, C.byref(c64), FAKE, 4, FAKE, FAKE, 2, 8, 8, 4,
                                 0.1, 1, None, None) == 2
    assert lib.pa_prefill_varlen(FAKE, FAKE, pk.PA_F16, C.byref(c), FAKE, 4, FAKE, FAKE, 2, 8, 8, 3,
                                 0.1, 1, None, None) == 1
