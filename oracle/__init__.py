"""CPU oracle of the paged-KV-cache attention path (fp64, plain loops).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product library
never does.  This module only marshals numpy arrays into the C oracle in
``oracle.c`` (see the citations there); it computes nothing itself.

Arrays of 16-bit formats are passed as their raw bit patterns (``np.uint16``),
E4M3 as ``np.uint8``.
"""
import ctypes as C
import os

import numpy as np

from .build import build_oracle

F16, BF16, E4M3, F32 = 0, 1, 2, 3
OK, ERR_ARG, ERR_BAD_BLOCK = 0, 1, 6

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _configure(C.CDLL(build_oracle()))
    return _lib


def use_library(path):
    """Load the oracle from another build of ``oracle.c`` (the tests use this
    to check that planted mistakes are caught).  Returns the previous one."""
    global _lib
    prev = _lib
    _lib = _configure(C.CDLL(path))
    return prev


def restore_library(prev):
    global _lib
    _lib = prev


def _configure(L):
    if True:
        vp, i32, i64, dbl, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_double, C.c_float
        L.oracle_f16_to_double.argtypes = [C.c_uint16]
        L.oracle_f16_to_double.restype = dbl
        L.oracle_f16_from_double.argtypes = [dbl]
        L.oracle_f16_from_double.restype = C.c_uint16
        L.oracle_bf16_to_double.argtypes = [C.c_uint16]
        L.oracle_bf16_to_double.restype = dbl
        L.oracle_bf16_from_double.argtypes = [dbl]
        L.oracle_bf16_from_double.restype = C.c_uint16
        L.oracle_e4m3_to_double.argtypes = [C.c_uint8]
        L.oracle_e4m3_to_double.restype = dbl
        L.oracle_e4m3_from_float.argtypes = [f32]
        L.oracle_e4m3_from_float.restype = C.c_uint8
        L.oracle_num_threads.argtypes = [C.c_int]
        L.oracle_num_threads.restype = C.c_int
        L.oracle_slot_mapping.argtypes = [vp, i32, i32, vp, vp, i64, vp]
        L.oracle_slot_mapping.restype = None
        L.oracle_cache_write.argtypes = [vp, vp, C.c_int, i64, i32, i32, i32, f32, f32,
                                         vp, vp, C.c_int, i64, i64, vp]
        L.oracle_cache_write.restype = C.c_int
        L.oracle_copy_blocks.argtypes = [vp, vp, C.c_int, i64, i32, i32, i32, vp, i32]
        L.oracle_copy_blocks.restype = C.c_int
        L.oracle_decode.argtypes = [vp, vp, vp, C.c_int, vp, vp, C.c_int, dbl, dbl, i64,
                                    i32, i32, i32, vp, i32, vp, i32, i32, dbl, C.c_int]
        L.oracle_decode.restype = C.c_int
        L.oracle_prefill.argtypes = [vp, vp, vp, C.c_int, vp, vp, C.c_int, dbl, dbl, i64,
                                     i32, i32, i32, vp, i32, vp, vp, i32, i32, dbl, C.c_int,
                                     C.c_int]
        L.oracle_prefill.restype = C.c_int
        L.oracle_attention_dense.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, C.c_int, i64]
        L.oracle_attention_dense.restype = None
    return L


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


_BITS = {F16: np.uint16, BF16: np.uint16, E4M3: np.uint8, F32: np.float32}


def num_threads(n: int = 0) -> int:
    """Set (n > 0) and return the OpenMP thread count the oracle uses."""
    return lib().oracle_num_threads(n)


# --- codecs (vectorised over numpy arrays) ---------------------------------

def f16_to_f64(bits):
    f = lib().oracle_f16_to_double
    return np.array([f(int(b)) for b in np.asarray(bits, np.uint16).ravel()]).reshape(np.shape(bits))


def f16_from_f64(x):
    f = lib().oracle_f16_from_double
    return np.array([f(float(v)) for v in np.asarray(x, np.float64).ravel()], np.uint16).reshape(np.shape(x))


def bf16_to_f64(bits):
    f = lib().oracle_bf16_to_double
    return np.array([f(int(b)) for b in np.asarray(bits, np.uint16).ravel()]).reshape(np.shape(bits))


def bf16_from_f64(x):
    f = lib().oracle_bf16_from_double
    return np.array([f(float(v)) for v in np.asarray(x, np.float64).ravel()], np.uint16).reshape(np.shape(x))


def e4m3_to_f64(codes):
    f = lib().oracle_e4m3_to_double
    return np.array([f(int(c)) for c in np.asarray(codes, np.uint8).ravel()]).reshape(np.shape(codes))


def e4m3_from_f32(x):
    f = lib().oracle_e4m3_from_float
    return np.array([f(float(v)) for v in np.asarray(x, np.float32).ravel()], np.uint8).reshape(np.shape(x))


def decode_bits(bits, dtype):
    """Values (float64) of an array of raw codes of `dtype`."""
    return {F16: f16_to_f64, BF16: bf16_to_f64, E4M3: e4m3_to_f64}[dtype](bits)


# --- path operations --------------------------------------------------------

def slot_mapping(block_table, block_size, seq_idx, pos):
    bt = _c(block_table, np.int32)
    si = _c(seq_idx, np.int32)
    ps = _c(pos, np.int64)
    out = np.empty(ps.shape[0], np.int64)
    lib().oracle_slot_mapping(_ptr(bt), bt.shape[1], block_size, _ptr(si), _ptr(ps), ps.shape[0], _ptr(out))
    return out


def cache_write(k_cache, v_cache, kv_dtype, k, v, in_dtype, slot_mapping, k_scale=1.0, v_scale=1.0,
                token_stride=None):
    """In-place write into numpy caches of raw codes, shape [nb, Hkv, bs, D].
    k, v: raw codes of shape [T, Hkv, D] (or [T, >=Hkv*D] with token_stride)."""
    nb, hkv, bs, d = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    kk = _c(k, _BITS[in_dtype])
    vv = _c(v, _BITS[in_dtype])
    sm = _c(slot_mapping, np.int64)
    T = sm.shape[0]
    stride = token_stride if token_stride is not None else hkv * d
    rc = lib().oracle_cache_write(_ptr(k_cache), _ptr(v_cache), kv_dtype, nb, bs, hkv, d,
                                  k_scale, v_scale, _ptr(kk), _ptr(vv), in_dtype, T, stride, _ptr(sm))
    return rc


def copy_blocks(k_cache, v_cache, kv_dtype, pairs):
    nb, hkv, bs, d = k_cache.shape
    pr = _c(pairs, np.int32).reshape(-1, 2)
    return lib().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), kv_dtype, nb, bs, hkv, d,
                                    _ptr(pr), pr.shape[0])


def decode(q, q_dtype, k_cache, v_cache, kv_dtype, block_table, seq_lens, scale,
           k_scale=1.0, v_scale=1.0, nthreads=0, want_codes=True):
    """Returns (out_codes [B,H,D] in q_dtype or None, out_f64 [B,H,D], status)."""
    qq = _c(q, _BITS[q_dtype])
    B, H, D = qq.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == D
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    out = np.zeros((B, H, D), _BITS[q_dtype]) if want_codes else None
    out64 = np.zeros((B, H, D), np.float64)
    rc = lib().oracle_decode(_ptr(out), _ptr(out64), _ptr(qq), q_dtype, _ptr(kc), _ptr(vc), kv_dtype,
                             k_scale, v_scale, nb, bs, hkv, D, _ptr(bt), bt.shape[1], _ptr(sl), B, H,
                             scale, nthreads)
    return out, out64, rc


def prefill(q, q_dtype, k_cache, v_cache, kv_dtype, block_table, cu_seq_lens_q, cu_seq_lens_k,
            scale, causal=True, k_scale=1.0, v_scale=1.0, nthreads=0, want_codes=True):
    """q: [total_q, H, D] raw codes.  Returns (out_codes, out_f64, status)."""
    qq = _c(q, _BITS[q_dtype])
    TQ, H, D = qq.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == D
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    bt = _c(block_table, np.int32)
    cq = _c(cu_seq_lens_q, np.int32)
    ck = _c(cu_seq_lens_k, np.int32)
    B = cq.shape[0] - 1
    assert cq[-1] == TQ
    out = np.zeros((TQ, H, D), _BITS[q_dtype]) if want_codes else None
    out64 = np.zeros((TQ, H, D), np.float64)
    rc = lib().oracle_prefill(_ptr(out), _ptr(out64), _ptr(qq), q_dtype, _ptr(kc), _ptr(vc), kv_dtype,
                              k_scale, v_scale, nb, bs, hkv, D, _ptr(bt), bt.shape[1], _ptr(cq),
                              _ptr(ck), B, H, scale, 1 if causal else 0, nthreads)
    return out, out64, rc


def attention_dense(q, k, v, scale, causal=False, causal_shift=0):
    """Brute force over dense float64 rows: q [Lq, D], k/v [Lk, D]."""
    qq = _c(q, np.float64)
    kk = _c(k, np.float64)
    vv = _c(v, np.float64)
    lq, D = qq.shape
    lk = kk.shape[0]
    out = np.zeros((lq, D), np.float64)
    lib().oracle_attention_dense(_ptr(out), _ptr(qq), _ptr(kk), _ptr(vv), lq, lk, D, scale,
                                 1 if causal else 0, causal_shift)
    return out
