"""ctypes marshalling for libpa_kv.so (see include/pa_kv.h for semantics)."""
import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional

import torch

PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
_TORCH_CODE = {torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.float8_e4m3fn: PA_FP8_E4M3}

library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa_kv.so")
_lib = None


class PaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, pa_status_str(status), status))


class _Cache(C.Structure):
    _fields_ = [("k_cache", C.c_void_p), ("v_cache", C.c_void_p), ("num_blocks", C.c_int64),
                ("block_size", C.c_int32), ("num_kv_heads", C.c_int32), ("head_size", C.c_int32),
                ("kv_dtype", C.c_int), ("k_scale", C.c_float), ("v_scale", C.c_float)]


def library():
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError("libpa_kv.so is missing: run __graft_entry__.build() "
                               "(or python -m paged_kv_cache_75_gb300.build)")
        L = C.CDLL(library_path)
        vp, i32, i64, sz, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_float
        pc = C.POINTER(_Cache)
        sig = {
            "pa_status_str": ([C.c_int], C.c_char_p),
            "pa_version": ([], i32),
            "pa_kv_cache_write": ([pc, vp, vp, C.c_int, i64, i64, vp, vp, vp], C.c_int),
            "pa_copy_blocks": ([pc, vp, i32, vp, vp], C.c_int),
            "pa_decode_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
            "pa_decode": ([vp, vp, C.c_int, pc, vp, i32, vp, i32, i32, i32, f32, i32, vp, sz, vp, vp],
                          C.c_int),
            "pa_prefill_varlen": ([vp, vp, C.c_int, pc, vp, i32, vp, vp, i32, i32, i32, i32, f32, i32,
                                   vp, vp], C.c_int),
            "pa_pool_create": ([i64, i32, vp, C.POINTER(vp)], C.c_int),
            "pa_pool_destroy": ([vp], None),
            "pa_pool_add_seq": ([vp, i64], C.c_int),
            "pa_pool_append": ([vp, i64, i32, vp, vp, vp], C.c_int),
            "pa_pool_fork": ([vp, i64, i64], C.c_int),
            "pa_pool_free_seq": ([vp, i64], C.c_int),
            "pa_pool_block_table": ([vp, vp, i32, i32, vp, vp], C.c_int),
            "pa_pool_num_free": ([vp], i64),
            "pa_pool_ref_count": ([vp, i64], i32),
            "pa_pool_seq_len": ([vp, i64], i32),
            "pa_slot_mapping": ([vp, i32, i32, i32, vp, vp, i64, vp], C.c_int),
            "pa_swap_blocks": ([pc, vp, vp, i64, vp, i32, i32, vp, vp], C.c_int),
            "pa_varlen_mixed_workspace_size": ([i32, i32, i32, i32, i32], sz),
            "pa_varlen_mixed": ([vp, vp, C.c_int, pc, vp, i32, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp, sz, vp,
                                 vp], C.c_int),
            "pa_decode_append": ([vp, vp, vp, vp, C.c_int, pc, vp, i32, vp, i32, i32, i32, f32, i32, vp, sz, vp,
                                  vp], C.c_int),
            "pa_prefill_varlen_packed": ([vp, vp, vp, vp, C.c_int, vp, vp, i32, i32, i32, i64, i32, i32, i32, f32,
                                          i32, vp, vp], C.c_int),
            "pa_decode_static_ws": ([vp, vp, C.c_int, pc, vp, i32, vp, i32, i32, i32, f32, i32, vp, vp],
                                    C.c_int),
            "pa_decode_test_wait_timeout": ([vp, vp, C.c_int, pc, vp, i32, vp, i32, i32, i32, f32, i32, vp, sz, vp,
                                             vp], C.c_int),
            "pa_decode_cascade_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
            "pa_decode_partition_size": ([i32, i32, i32, i32], i32),
            "pa_decode_cascade": ([vp, vp, C.c_int, pc, vp, i32, vp, i32, i32, i32, f32, vp, vp, i32, i32, i32,
                                   i32, vp, sz, vp, vp], C.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def pa_status_str(status: int) -> str:
    return library().pa_status_str(int(status)).decode()


def pa_version() -> int:
    return library().pa_version()


def _check(status, where):
    if status != 0:
        raise PaError(status, where)


def torch_dtype_code(dt) -> int:
    if dt not in _TORCH_CODE:
        raise TypeError("unsupported dtype %s" % dt)
    return _TORCH_CODE[dt]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return C.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t, name, dtype=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a tensor" % name)
    if cuda and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


@dataclass
class KVCache:
    """One layer's paged cache: k_cache, v_cache [num_blocks, num_kv_heads,
    block_size, head_size] (float16 / bfloat16 / float8_e4m3fn)."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: float = 1.0
    v_scale: float = 1.0

    def __post_init__(self):
        _need(self.k_cache, "k_cache")
        _need(self.v_cache, "v_cache")
        if self.k_cache.shape != self.v_cache.shape or self.k_cache.dtype != self.v_cache.dtype:
            raise ValueError("k_cache and v_cache must match")
        if self.k_cache.dim() != 4:
            raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_size]")

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def num_kv_heads(self):
        return self.k_cache.shape[1]

    @property
    def block_size(self):
        return self.k_cache.shape[2]

    @property
    def head_size(self):
        return self.k_cache.shape[3]

    @property
    def dtype_code(self):
        return torch_dtype_code(self.k_cache.dtype)

    def c_struct(self) -> _Cache:
        nb, hkv, bs, d = self.k_cache.shape
        return _Cache(self.k_cache.data_ptr(), self.v_cache.data_ptr(), nb, bs, hkv, d,
                      self.dtype_code, float(self.k_scale), float(self.v_scale))


def pa_kv_cache_write(cache: KVCache, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                      dev_status: Optional[torch.Tensor] = None):
    """k, v: [T, num_kv_heads, head_size] (or [T, >= num_kv_heads*head_size]
    rows with a common token stride); slot_mapping int64 [T] (< 0 skips)."""
    _need(slot_mapping, "slot_mapping", torch.int64)
    T = slot_mapping.shape[0]
    for name, t in (("k", k), ("v", v)):
        if not t.is_cuda or t.stride(-1) != 1 or t.shape[0] != T:
            raise ValueError("%s must be a CUDA tensor of [T, ...] rows" % name)
    if k.stride(0) != v.stride(0) or k.dtype != v.dtype:
        raise ValueError("k and v must share dtype and token stride")
    cs = cache.c_struct()
    st = library().pa_kv_cache_write(C.byref(cs), _ptr(k), _ptr(v), torch_dtype_code(k.dtype), T,
                                     k.stride(0), _ptr(slot_mapping), _ptr(dev_status), _stream(k))
    _check(st, "pa_kv_cache_write")


def pa_copy_blocks(cache: KVCache, src_dst_pairs: torch.Tensor, dev_status: Optional[torch.Tensor] = None):
    _need(src_dst_pairs, "src_dst_pairs", torch.int32)
    cs = cache.c_struct()
    n = src_dst_pairs.numel() // 2
    st = library().pa_copy_blocks(C.byref(cs), _ptr(src_dst_pairs), n, _ptr(dev_status),
                                  _stream(cache.k_cache))
    _check(st, "pa_copy_blocks")


def pa_prefill_varlen_packed(out: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                             cu_seq_lens_q: torch.Tensor, cu_seq_lens_k: torch.Tensor, max_seqlen_q: int,
                             max_seqlen_k: int, scale: float, causal: bool = True,
                             dev_status: Optional[torch.Tensor] = None):
    """Varlen attention over packed K/V [Σk, Hkv, D] (no cache)."""
    for name, t in (("out", out), ("q", q), ("k", k), ("v", v)):
        _need(t, name)
    _need(cu_seq_lens_q, "cu_seq_lens_q", torch.int32)
    _need(cu_seq_lens_k, "cu_seq_lens_k", torch.int32)
    if k.dim() != 3 or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k, v must be [total_k, num_kv_heads, head_size] of q's dtype")
    st = library().pa_prefill_varlen_packed(_ptr(out), _ptr(q), _ptr(k), _ptr(v), torch_dtype_code(q.dtype),
                                            _ptr(cu_seq_lens_q), _ptr(cu_seq_lens_k), cu_seq_lens_q.numel() - 1,
                                            max_seqlen_q, max_seqlen_k, k.shape[0], q.shape[1], k.shape[1],
                                            q.shape[2], scale, 1 if causal else 0, _ptr(dev_status), _stream(q))
    _check(st, "pa_prefill_varlen_packed")


def pa_varlen_mixed_workspace_size(num_seqs, num_heads, head_size, max_seqlen_k, block_size) -> int:
    return int(library().pa_varlen_mixed_workspace_size(num_seqs, num_heads, head_size, max_seqlen_k, block_size))


def pa_varlen_mixed(out: torch.Tensor, q: torch.Tensor, cache: KVCache, block_table: torch.Tensor,
                    cu_seq_lens_q: torch.Tensor, cu_seq_lens_k: torch.Tensor, host_cu_seq_lens_q, max_seqlen_q: int,
                    max_seqlen_k: int, scale: float, causal: bool = True, workspace: Optional[torch.Tensor] = None,
                    dev_status: Optional[torch.Tensor] = None):
    """pa_prefill_varlen with the trailing one-token sequences sent to the
    decode kernel; host_cu_seq_lens_q: the same offsets on the host."""
    import numpy as np
    _need(q, "q")
    _need(out, "out", q.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(cu_seq_lens_q, "cu_seq_lens_q", torch.int32)
    _need(cu_seq_lens_k, "cu_seq_lens_k", torch.int32)
    hq = np.ascontiguousarray(host_cu_seq_lens_q, np.int32)
    if hq.shape[0] != cu_seq_lens_q.numel():
        raise ValueError("host_cu_seq_lens_q must match cu_seq_lens_q")
    if workspace is not None:
        _need(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    cs = cache.c_struct()
    st = library().pa_varlen_mixed(_ptr(out), _ptr(q), torch_dtype_code(q.dtype), C.byref(cs), _ptr(block_table),
                                   block_table.shape[1], _ptr(cu_seq_lens_q), _ptr(cu_seq_lens_k),
                                   hq.ctypes.data_as(C.c_void_p), hq.shape[0] - 1, int(max_seqlen_q),
                                   int(max_seqlen_k), q.shape[1], float(scale), 1 if causal else 0, _ptr(workspace),
                                   ws_bytes, _ptr(dev_status), _stream(q))
    _check(st, "pa_varlen_mixed")


def pa_swap_blocks(cache: KVCache, host_k: torch.Tensor, host_v: torch.Tensor, pairs: torch.Tensor,
                   to_host: bool, dev_status: Optional[torch.Tensor] = None):
    """Copies whole blocks between the cache and pinned host tensors shaped
    like the cache ([host_blocks, Hkv, bs, D]); pairs: device int32 [n, 2] of
    (device block, host block)."""
    _need(pairs, "pairs", torch.int32)
    for name, t in (("host_k", host_k), ("host_v", host_v)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous host tensor" % name)
        if t.dtype != cache.k_cache.dtype or t.shape[1:] != cache.k_cache.shape[1:]:
            raise ValueError("%s must match the cache's dtype and block shape" % name)
    cs = cache.c_struct()
    st = library().pa_swap_blocks(C.byref(cs), C.c_void_p(host_k.data_ptr()), C.c_void_p(host_v.data_ptr()),
                                  host_k.shape[0], _ptr(pairs), pairs.numel() // 2, 1 if to_host else 0,
                                  _ptr(dev_status), _stream(cache.k_cache))
    _check(st, "pa_swap_blocks")


def pa_decode_workspace_size(num_seqs, num_heads, head_size, max_seq_len, block_size, partition_size=0) -> int:
    return int(library().pa_decode_workspace_size(num_seqs, num_heads, head_size, max_seq_len,
                                                  block_size, partition_size))


def pa_decode(out: torch.Tensor, q: torch.Tensor, cache: KVCache, block_table: torch.Tensor,
              seq_lens: torch.Tensor, max_seq_len: int, scale: float, partition_size: int = 0,
              workspace: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None):
    """out, q: [num_seqs, num_heads, head_size]; block_table int32 [num_seqs,
    max_blocks_per_seq]; seq_lens int32 [num_seqs] (attended lengths)."""
    _need(q, "q")
    _need(out, "out", q.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, H, D = q.shape
    if workspace is not None:
        _need(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    cs = cache.c_struct()
    st = library().pa_decode(_ptr(out), _ptr(q), torch_dtype_code(q.dtype), C.byref(cs), _ptr(block_table),
                             block_table.shape[1], _ptr(seq_lens), B, int(max_seq_len), H, float(scale),
                             int(partition_size), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(q))
    _check(st, "pa_decode")


def pa_decode_test_wait_timeout(out: torch.Tensor, q: torch.Tensor, cache: KVCache, block_table: torch.Tensor,
                                seq_lens: torch.Tensor, max_seq_len: int, scale: float, partition_size: int = 0,
                                workspace: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None):
    """Test hook: pa_decode whose copies are never issued, so every wait of
    the kernel runs out (PA_ERR_TIMEOUT in dev_status after about 2 s)."""
    _need(q, "q")
    _need(out, "out", q.dtype)
    B, H, D = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    cs = cache.c_struct()
    st = library().pa_decode_test_wait_timeout(_ptr(out), _ptr(q), torch_dtype_code(q.dtype), C.byref(cs),
                                               _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
                                               int(max_seq_len), H, float(scale), int(partition_size),
                                               _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(q))
    _check(st, "pa_decode_test_wait_timeout")


def pa_decode_partition_size(num_seqs, num_heads, num_kv_heads, max_seq_len) -> int:
    """The partition size pa_decode chooses for partition_size = 0 on the current device."""
    return int(library().pa_decode_partition_size(num_seqs, num_heads, num_kv_heads, max_seq_len))


def pa_decode_cascade_workspace_size(num_seqs, num_heads, head_size, max_seq_len, block_size,
                                     partition_size=0) -> int:
    return int(library().pa_decode_cascade_workspace_size(num_seqs, num_heads, head_size, max_seq_len,
                                                          block_size, partition_size))


def pa_decode_cascade(out: torch.Tensor, q: torch.Tensor, cache: KVCache, block_table: torch.Tensor,
                      seq_lens: torch.Tensor, max_seq_len: int, scale: float, cu_groups: torch.Tensor,
                      shared_lens: torch.Tensor, max_group_size: int, max_shared_len: int,
                      workspace: torch.Tensor, partition_size: int = 0,
                      dev_status: Optional[torch.Tensor] = None):
    """pa_decode for groups of sequences that share their first blocks:
    cu_groups int32 [num_groups+1] (group g = rows cu_groups[g] ..
    cu_groups[g+1]-1), shared_lens int32 [num_groups] (tokens, whole blocks)."""
    _need(q, "q")
    _need(out, "out", q.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    _need(cu_groups, "cu_groups", torch.int32)
    _need(shared_lens, "shared_lens", torch.int32)
    _need(workspace, "workspace")
    B, H, D = q.shape
    G = shared_lens.shape[0]
    if cu_groups.shape[0] != G + 1:
        raise ValueError("cu_groups must have num_groups + 1 entries")
    cs = cache.c_struct()
    st = library().pa_decode_cascade(_ptr(out), _ptr(q), torch_dtype_code(q.dtype), C.byref(cs), _ptr(block_table),
                                     block_table.shape[1], _ptr(seq_lens), B, int(max_seq_len), H, float(scale),
                                     _ptr(cu_groups), _ptr(shared_lens), G, int(max_group_size),
                                     int(max_shared_len), int(partition_size), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(q))
    _check(st, "pa_decode_cascade")


def pa_decode_append(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                     cache: KVCache, block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                     scale: float, partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                     dev_status: Optional[torch.Tensor] = None):
    """pa_kv_cache_write of each sequence's new token (k_new, v_new:
    [num_seqs, num_kv_heads, head_size], position seq_lens-1) fused with
    pa_decode over seq_lens tokens."""
    _need(q, "q")
    _need(out, "out", q.dtype)
    _need(k_new, "k_new", q.dtype)
    _need(v_new, "v_new", q.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, H, D = q.shape
    if tuple(k_new.shape) != (B, cache.num_kv_heads, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new, v_new must be [num_seqs, num_kv_heads, head_size]")
    if workspace is not None:
        _need(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    cs = cache.c_struct()
    st = library().pa_decode_append(_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), torch_dtype_code(q.dtype),
                                    C.byref(cs), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
                                    int(max_seq_len), H, float(scale), int(partition_size), _ptr(workspace),
                                    ws_bytes, _ptr(dev_status), _stream(q))
    _check(st, "pa_decode_append")


def pa_decode_static_ws(out: torch.Tensor, q: torch.Tensor, cache: KVCache, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, max_seq_len: int, scale: float, partition_size: int = 0,
                        dev_status: Optional[torch.Tensor] = None):
    """pa_decode without a workspace argument: the library's built-in scratch
    (for callers that cannot allocate device memory; see include/pa_kv.h)."""
    _need(q, "q")
    _need(out, "out", q.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, H, D = q.shape
    cs = cache.c_struct()
    st = library().pa_decode_static_ws(_ptr(out), _ptr(q), torch_dtype_code(q.dtype), C.byref(cs),
                                       _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
                                       int(max_seq_len), H, float(scale), int(partition_size),
                                       _ptr(dev_status), _stream(q))
    _check(st, "pa_decode_static_ws")


def pa_prefill_varlen(out: torch.Tensor, q: torch.Tensor, cache: KVCache, block_table: torch.Tensor,
                      cu_seq_lens_q: torch.Tensor, cu_seq_lens_k: torch.Tensor, max_seqlen_q: int,
                      max_seqlen_k: int, scale: float, causal: bool = True,
                      dev_status: Optional[torch.Tensor] = None):
    """q, out: [total_q, num_heads, head_size]; cu_seq_lens_q/k int32 [B+1]."""
    _need(q, "q")
    _need(out, "out", q.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(cu_seq_lens_q, "cu_seq_lens_q", torch.int32)
    _need(cu_seq_lens_k, "cu_seq_lens_k", torch.int32)
    H = q.shape[1]
    B = cu_seq_lens_q.shape[0] - 1
    cs = cache.c_struct()
    st = library().pa_prefill_varlen(_ptr(out), _ptr(q), torch_dtype_code(q.dtype), C.byref(cs),
                                     _ptr(block_table), block_table.shape[1], _ptr(cu_seq_lens_q),
                                     _ptr(cu_seq_lens_k), B, int(max_seqlen_q), int(max_seqlen_k), H,
                                     float(scale), 1 if causal else 0, _ptr(dev_status), _stream(q))
    _check(st, "pa_prefill_varlen")


def pa_slot_mapping(block_table, block_size: int, seq_idx, pos):
    """Host helper: slots of new tokens (numpy int32 table [B, max_blocks],
    seq_idx int32 [n], pos int64 [n]) -> numpy int64 [n]."""
    import numpy as np
    bt = np.ascontiguousarray(block_table, np.int32)
    si = np.ascontiguousarray(seq_idx, np.int32)
    ps = np.ascontiguousarray(pos, np.int64)
    out = np.empty(ps.shape[0], np.int64)
    st = library().pa_slot_mapping(bt.ctypes.data_as(C.c_void_p), bt.shape[0], bt.shape[1], block_size,
                                   si.ctypes.data_as(C.c_void_p), ps.ctypes.data_as(C.c_void_p), ps.shape[0],
                                   out.ctypes.data_as(C.c_void_p))
    _check(st, "pa_slot_mapping")
    return out


class BlockPool:
    """Host block pool (FIFO free list, reference counts, fork, copy-on-write)."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        L = library()
        self._h = C.c_void_p()
        order = None
        if free_order is not None:
            order = (C.c_int32 * num_blocks)(*[int(x) for x in free_order])
        _check(L.pa_pool_create(num_blocks, block_size, order, C.byref(self._h)), "pa_pool_create")
        self.block_size = block_size

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pa_pool_destroy(self._h)
            self._h = None

    def add_seq(self, seq_id: int):
        _check(library().pa_pool_add_seq(self._h, seq_id), "pa_pool_add_seq")

    def append(self, seq_id: int, n: int):
        """Returns (slots list, cow pairs list)."""
        slots = (C.c_int64 * max(n, 1))()
        cow = (C.c_int32 * 2)()
        ncow = C.c_int32(0)
        _check(library().pa_pool_append(self._h, seq_id, n, slots, cow, C.byref(ncow)), "pa_pool_append")
        return list(slots[:n]), [(cow[0], cow[1])] if ncow.value else []

    def fork(self, parent: int, child: int):
        _check(library().pa_pool_fork(self._h, parent, child), "pa_pool_fork")

    def free_seq(self, seq_id: int):
        _check(library().pa_pool_free_seq(self._h, seq_id), "pa_pool_free_seq")

    def block_table(self, seq_ids, max_blocks: int):
        n = len(seq_ids)
        ids = (C.c_int64 * max(n, 1))(*seq_ids)
        table = (C.c_int32 * max(n * max_blocks, 1))()
        lens = (C.c_int32 * max(n, 1))()
        _check(library().pa_pool_block_table(self._h, ids, n, max_blocks, table, lens), "pa_pool_block_table")
        return [list(table[r * max_blocks:(r + 1) * max_blocks]) for r in range(n)], list(lens[:n])

    def num_free(self) -> int:
        return library().pa_pool_num_free(self._h)

    def ref_count(self, block: int) -> int:
        return library().pa_pool_ref_count(self._h, block)

    def seq_len(self, seq_id: int) -> int:
        return library().pa_pool_seq_len(self._h, seq_id)
