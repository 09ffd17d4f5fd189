"""fp8_paged_kv_kvq_gb300 -- an FP8 E4M3 paged KV cache for NVIDIA GB300.

Python binding of ``libkvq.so`` (C ABI: ``include/kvq.h``).  Every function
here only marshals arguments -- PyTorch tensors in, raw device pointers, sizes
and the current CUDA stream out -- and calls the C entry point of the same
name; all computation happens in the library's sm_103a kernels.  There is no
fallback: if the library has not been built, or a call returns an error status,
a ``KvqError`` is raised.

Row format (ROCm/ATOM PR #2655 "fix(qwen4-exp): register the QSA FP8 scale
planes for KV offload", PR description; FlashML-org/FreeToken PR #354
"feat(kvcache): store the KV cache as fp8 e4m3 codes", PR description): every
cached (token, KV head) row of K or V is head_dim e4m3 bytes, in a uint8 buffer
shaped like the 16-bit cache, and one fp32 scale = row amax / 448.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from dataclasses import dataclass

import torch

__all__ = [
    "KvqError", "Cache", "load", "abi_version", "cache_bytes", "quantize_scatter",
    "paged_decode", "paged_decode_partials", "paged_decode_combine",
    "paged_decode_workspace_size", "paged_decode_partition_tokens", "dequant_rows",
    "header_functions", "LIB_PATH", "HEADER_PATH",
    "IndexCache", "INDEX_FP8", "INDEX_MXFP4", "index_cache_bytes", "index_quantize_scatter",
    "index_dequant_rows",
    "ERRF_SLOT_RANGE", "ERRF_BLOCK_RANGE", "ERRF_CONTEXT_RANGE",
    "CODES_E4M3", "CODES_E5M2", "quantize_scatter_unscaled", "paged_decode_codes",
    "paged_decode_codes_workspace_size",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libkvq.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "kvq.h")

INDEX_FP8 = 0
INDEX_MXFP4 = 1

CODES_E4M3 = 0
CODES_E5M2 = 1

ERRF_SLOT_RANGE = 1
ERRF_BLOCK_RANGE = 2
ERRF_CONTEXT_RANGE = 4

_STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARGUMENT", 2: "KVQ_ERR_UNSUPPORTED",
           3: "KVQ_ERR_MISALIGNED", 4: "KVQ_ERR_WORKSPACE_TOO_SMALL", 5: "KVQ_ERR_CUDA"}


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)} "
                         f"({load().kvq_status_string(status).decode()})")


class _CacheStruct(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("num_slots", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32)]


class _IndexCacheStruct(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("exponents", ctypes.c_void_p), ("num_slots", ctypes.c_int64),
                ("format", ctypes.c_int32), ("dim", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libkvq.so (built by ``fp8_paged_kv_kvq_gb300.build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libkvq.so not found at {p}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(or fp8_paged_kv_kvq_gb300/build.py); there is no CPU fallback")
        lib = ctypes.CDLL(p)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        CP = ctypes.POINTER(_CacheStruct)
        sigs = {
            "kvq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "kvq_abi_version": (i32, []),
            "kvq_cache_bytes": (sz, [i64, i32, i32]),
            "kvq_quantize_scatter": (ctypes.c_int, [CP, P, i64, P, i64, i64, P, P, P]),
            "kvq_paged_decode_partition_tokens": (i32, [i32, i32, i32, i32, i32, i32]),
            "kvq_paged_decode_workspace_size": (sz, [i32, i32, i32, i32, i32, i32, i32, i32]),
            "kvq_paged_decode": (ctypes.c_int, [CP, P, i32, i32, i32, P, i32, P, i32,
                                                ctypes.c_float, i32, P, P, sz, P, P]),
            "kvq_paged_decode_partials": (ctypes.c_int, [CP, P, i32, i32, i32, P, i32, P, i32,
                                                         ctypes.c_float, i32, P, P, sz, P, P]),
            "kvq_paged_decode_combine": (ctypes.c_int, [CP, i32, i32, i32, i32, P, i32, i32,
                                                        P, P, sz, P]),
            "kvq_paged_decode_append_partials": (ctypes.c_int, [CP, P, i64, P, i64, P, i32, i32,
                                                                i32, P, i32, P, i32,
                                                                ctypes.c_float, i32, P, P, sz,
                                                                P, P]),
            "kvq_paged_decode_append": (ctypes.c_int, [CP, P, i64, P, i64, P, i32, i32, i32, P,
                                                       i32, P, i32, ctypes.c_float, i32, P, P,
                                                       sz, P, P]),
            "kvq_dequant_rows": (ctypes.c_int, [CP, P, i64, i32, P, P, P, P]),
            "kvq_quantize_scatter_unscaled": (ctypes.c_int, [CP, i32, P, i64, P, i64, i64, P,
                                                             P, P]),
            "kvq_paged_decode_codes_workspace_size": (sz, [i32, i32, i32, i32, i32, i32, i32]),
            "kvq_paged_decode_codes": (ctypes.c_int, [CP, i32, P, i32, i32, i32, P, i32, P, i32,
                                                      ctypes.c_float, P, P, sz, P, P]),
            "kvq_index_cache_bytes": (sz, [i64, i32, i32]),
            "kvq_index_quantize_scatter": (ctypes.c_int, [ctypes.POINTER(_IndexCacheStruct), P,
                                                          i64, i64, P, P, P]),
            "kvq_index_dequant_rows": (ctypes.c_int, [ctypes.POINTER(_IndexCacheStruct), P, i64,
                                                      i32, P, P, P]),
            "kvq_index_scores": (ctypes.c_int, [ctypes.POINTER(_IndexCacheStruct), i32, P, i32,
                                                i32, i32, P, i32, P, i32, P, P, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def header_functions(path: str = HEADER_PATH) -> list[str]:
    """Names of the functions declared in include/kvq.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def _check(status: int, where: str):
    if status != 0:
        raise KvqError(status, where)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


@dataclass
class Cache:
    """Device tensors of one FP8 paged cache; codes and scales travel together.

    k_codes, v_codes: uint8 [num_slots, num_kv_heads, head_dim]
    k_scales, v_scales: float32 [num_slots, num_kv_heads]"""
    k_codes: torch.Tensor
    v_codes: torch.Tensor
    k_scales: torch.Tensor
    v_scales: torch.Tensor
    block_size: int

    @staticmethod
    def empty(num_slots: int, num_kv_heads: int, head_dim: int = 128, block_size: int = 16,
              device="cuda") -> "Cache":
        return Cache(
            torch.zeros(num_slots, num_kv_heads, head_dim, dtype=torch.uint8, device=device),
            torch.zeros(num_slots, num_kv_heads, head_dim, dtype=torch.uint8, device=device),
            torch.zeros(num_slots, num_kv_heads, dtype=torch.float32, device=device),
            torch.zeros(num_slots, num_kv_heads, dtype=torch.float32, device=device),
            block_size)

    @property
    def num_slots(self) -> int:
        return self.k_codes.shape[0]

    @property
    def num_kv_heads(self) -> int:
        return self.k_codes.shape[1]

    @property
    def head_dim(self) -> int:
        return self.k_codes.shape[2]

    def struct(self) -> _CacheStruct:
        for t, dt in ((self.k_codes, torch.uint8), (self.v_codes, torch.uint8),
                      (self.k_scales, torch.float32), (self.v_scales, torch.float32)):
            if t.dtype != dt or not t.is_contiguous():
                raise ValueError("cache tensors must be contiguous uint8 codes / fp32 scales")
        return _CacheStruct(self.k_codes.data_ptr(), self.v_codes.data_ptr(),
                            self.k_scales.data_ptr(), self.v_scales.data_ptr(),
                            self.num_slots, self.num_kv_heads, self.head_dim, self.block_size)


def abi_version() -> int:
    return load().kvq_abi_version()


def cache_bytes(num_slots: int, num_kv_heads: int, head_dim: int = 128) -> int:
    return load().kvq_cache_bytes(num_slots, num_kv_heads, head_dim)


def _rows_view(x: torch.Tensor, H: int, D: int, name: str) -> int:
    """Token stride (elements) of a [T, H, D] (or [T, H*D]) bf16 view whose rows
    are contiguous within a token."""
    if x.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16")
    if x.dim() == 2:
        if x.shape[1] != H * D or x.stride(1) != 1:
            raise ValueError(f"{name}: expected [T, {H * D}] with unit inner stride")
    elif x.dim() == 3:
        if tuple(x.shape[1:]) != (H, D) or x.stride(2) != 1 or x.stride(1) != D:
            raise ValueError(f"{name}: expected [T, {H}, {D}] with contiguous heads")
    else:
        raise ValueError(f"{name}: expected a 2-D or 3-D view")
    return x.stride(0)


def quantize_scatter(cache: Cache, k: torch.Tensor, v: torch.Tensor, slot_ids: torch.Tensor,
                     err_flags: torch.Tensor | None = None, stream=None) -> None:
    """kvq_quantize_scatter: quantise bf16 K/V rows [T, H, D] (views allowed,
    each with its own token stride) into ``cache`` at device int64 ``slot_ids``."""
    H, D = cache.num_kv_heads, cache.head_dim
    ks = _rows_view(k, H, D, "k")
    vs = _rows_view(v, H, D, "v")
    T = k.shape[0]
    if v.shape[0] != T or slot_ids.numel() != T or slot_ids.dtype != torch.int64:
        raise ValueError("k, v and slot_ids (int64) must have the same token count")
    st = cache.struct()
    _check(load().kvq_quantize_scatter(ctypes.byref(st), _ptr(k), ks, _ptr(v), vs, T,
                                       _ptr(slot_ids), _ptr(err_flags), _stream(stream)),
           "kvq_quantize_scatter")


def paged_decode_partition_tokens(num_requests: int, rows_per_request: int, num_q_heads: int,
                                  num_kv_heads: int, block_size: int,
                                  max_context_len: int) -> int:
    return load().kvq_paged_decode_partition_tokens(num_requests, rows_per_request, num_q_heads,
                                                    num_kv_heads, block_size, max_context_len)


def paged_decode_workspace_size(num_requests: int, rows_per_request: int, num_q_heads: int,
                                num_kv_heads: int, head_dim: int, block_size: int,
                                max_context_len: int, partition_tokens: int = 0) -> int:
    return load().kvq_paged_decode_workspace_size(num_requests, rows_per_request, num_q_heads,
                                                  num_kv_heads, head_dim, block_size,
                                                  max_context_len, partition_tokens)


def _decode_args(cache, q, block_tables, context_lens, rows_per_request):
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be a contiguous bf16 [num_requests*R, Hq, D] tensor")
    if block_tables.dtype != torch.int32 or not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous int32 [N, max_blocks]")
    if context_lens.dtype != torch.int32 or not context_lens.is_contiguous():
        raise ValueError("context_lens must be contiguous int32 [N]")
    N = block_tables.shape[0]
    if q.shape[0] != N * rows_per_request or context_lens.numel() != N:
        raise ValueError("q rows must equal num_requests * rows_per_request")
    return N, q.shape[1], block_tables.shape[1]


def paged_decode(cache: Cache, q: torch.Tensor, block_tables: torch.Tensor,
                 context_lens: torch.Tensor, max_context_len: int, sm_scale: float,
                 rows_per_request: int = 1, partition_tokens: int = 0,
                 out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                 err_flags: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvq_paged_decode: paged GQA decode / verify attention; returns ``out``
    (bf16, shape of q).  ``workspace`` (uint8, >= paged_decode_workspace_size;
    no initialisation needed) is allocated here, by PyTorch, when not given."""
    N, Hq, mb = _decode_args(cache, q, block_tables, context_lens, rows_per_request)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = paged_decode_workspace_size(N, rows_per_request, Hq, cache.num_kv_heads,
                                           cache.head_dim, cache.block_size, max_context_len,
                                           partition_tokens)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = cache.struct()
    _check(load().kvq_paged_decode(ctypes.byref(st), _ptr(q), N, rows_per_request, Hq,
                                   _ptr(block_tables), mb, _ptr(context_lens), max_context_len,
                                   float(sm_scale), partition_tokens, _ptr(out), _ptr(workspace),
                                   workspace.numel(), _ptr(err_flags), _stream(stream)),
           "kvq_paged_decode")
    return out


def _append_rows(cache: Cache, k_new, v_new, n_rows: int):
    H, D = cache.num_kv_heads, cache.head_dim
    ks = _rows_view(k_new, H, D, "k_new")
    vs = _rows_view(v_new, H, D, "v_new")
    if k_new.shape[0] != n_rows or v_new.shape[0] != n_rows:
        raise ValueError("k_new and v_new need num_requests * rows_per_request rows")
    return ks, vs


def paged_decode_append(cache: Cache, k_new: torch.Tensor, v_new: torch.Tensor,
                        q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                        max_context_len: int, sm_scale: float, rows_per_request: int = 1,
                        partition_tokens: int = 0, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None,
                        err_flags: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvq_paged_decode_append: one decode step -- the step's new K/V rows
    [N*R, H, D] (views allowed) stored at positions L_r - R + i of each
    request's block table, then the attention over the cache that holds them;
    returns ``out`` (bf16, shape of q)."""
    N, Hq, mb = _decode_args(cache, q, block_tables, context_lens, rows_per_request)
    ks, vs = _append_rows(cache, k_new, v_new, N * rows_per_request)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = paged_decode_workspace_size(N, rows_per_request, Hq, cache.num_kv_heads,
                                           cache.head_dim, cache.block_size, max_context_len,
                                           partition_tokens)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = cache.struct()
    _check(load().kvq_paged_decode_append(
        ctypes.byref(st), _ptr(k_new), ks, _ptr(v_new), vs, _ptr(q), N, rows_per_request, Hq,
        _ptr(block_tables), mb, _ptr(context_lens), max_context_len, float(sm_scale),
        partition_tokens, _ptr(out), _ptr(workspace), workspace.numel(), _ptr(err_flags),
        _stream(stream)), "kvq_paged_decode_append")
    return out


def paged_decode_append_partials(cache: Cache, k_new, v_new, q, block_tables, context_lens,
                                 max_context_len: int, sm_scale: float, rows_per_request: int,
                                 partition_tokens: int, out: torch.Tensor,
                                 workspace: torch.Tensor | None,
                                 err_flags: torch.Tensor | None = None, stream=None) -> None:
    """kvq_paged_decode_append_partials (the step's store and split-K launch;
    kvq_paged_decode_combine follows)."""
    N, Hq, mb = _decode_args(cache, q, block_tables, context_lens, rows_per_request)
    ks, vs = _append_rows(cache, k_new, v_new, N * rows_per_request)
    st = cache.struct()
    _check(load().kvq_paged_decode_append_partials(
        ctypes.byref(st), _ptr(k_new), ks, _ptr(v_new), vs, _ptr(q), N, rows_per_request, Hq,
        _ptr(block_tables), mb, _ptr(context_lens), max_context_len, float(sm_scale),
        partition_tokens, _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(err_flags), _stream(stream)),
        "kvq_paged_decode_append_partials")


def paged_decode_partials(cache: Cache, q, block_tables, context_lens, max_context_len: int,
                          sm_scale: float, rows_per_request: int, partition_tokens: int,
                          out: torch.Tensor, workspace: torch.Tensor | None,
                          err_flags: torch.Tensor | None = None, stream=None) -> None:
    """kvq_paged_decode_partials (the split-K launch of kvq_paged_decode)."""
    N, Hq, mb = _decode_args(cache, q, block_tables, context_lens, rows_per_request)
    st = cache.struct()
    _check(load().kvq_paged_decode_partials(
        ctypes.byref(st), _ptr(q), N, rows_per_request, Hq, _ptr(block_tables), mb,
        _ptr(context_lens), max_context_len, float(sm_scale), partition_tokens, _ptr(out),
        _ptr(workspace), 0 if workspace is None else workspace.numel(), _ptr(err_flags),
        _stream(stream)), "kvq_paged_decode_partials")


def paged_decode_combine(cache: Cache, num_requests: int, rows_per_request: int,
                         num_q_heads: int, max_blocks_per_req: int, context_lens: torch.Tensor,
                         max_context_len: int, partition_tokens: int, out: torch.Tensor,
                         workspace: torch.Tensor | None, stream=None) -> None:
    """kvq_paged_decode_combine (the merge launch of kvq_paged_decode)."""
    st = cache.struct()
    _check(load().kvq_paged_decode_combine(
        ctypes.byref(st), num_requests, rows_per_request, num_q_heads, max_blocks_per_req,
        _ptr(context_lens), max_context_len, partition_tokens, _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream)),
        "kvq_paged_decode_combine")


def quantize_scatter_unscaled(cache: Cache, k: torch.Tensor, v: torch.Tensor,
                              slot_ids: torch.Tensor, code_format: int = CODES_E4M3,
                              err_flags: torch.Tensor | None = None, stream=None) -> None:
    """kvq_quantize_scatter_unscaled: cast bf16 K/V rows to e4m3 or e5m2 codes
    with no scale (scale planes set to 1) -- the codec ablation's caches."""
    H, D = cache.num_kv_heads, cache.head_dim
    ks = _rows_view(k, H, D, "k")
    vs = _rows_view(v, H, D, "v")
    T = k.shape[0]
    if v.shape[0] != T or slot_ids.numel() != T or slot_ids.dtype != torch.int64:
        raise ValueError("k, v and slot_ids (int64) must have the same token count")
    st = cache.struct()
    _check(load().kvq_quantize_scatter_unscaled(ctypes.byref(st), code_format, _ptr(k), ks,
                                                _ptr(v), vs, T, _ptr(slot_ids), _ptr(err_flags),
                                                _stream(stream)),
           "kvq_quantize_scatter_unscaled")


def paged_decode_codes_workspace_size(num_requests: int, rows_per_request: int,
                                      num_q_heads: int, num_kv_heads: int, head_dim: int,
                                      block_size: int, max_context_len: int) -> int:
    return load().kvq_paged_decode_codes_workspace_size(num_requests, rows_per_request,
                                                        num_q_heads, num_kv_heads, head_dim,
                                                        block_size, max_context_len)


def paged_decode_codes(cache: Cache, code_format: int, q: torch.Tensor,
                       block_tables: torch.Tensor, context_lens: torch.Tensor,
                       max_context_len: int, sm_scale: float, rows_per_request: int = 1,
                       out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       err_flags: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvq_paged_decode_codes: paged attention over a cache of e4m3 or e5m2
    codes (the rows-on-M kernel for every shape); returns ``out``."""
    N, Hq, mb = _decode_args(cache, q, block_tables, context_lens, rows_per_request)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = paged_decode_codes_workspace_size(N, rows_per_request, Hq, cache.num_kv_heads,
                                                 cache.head_dim, cache.block_size,
                                                 max_context_len)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = cache.struct()
    _check(load().kvq_paged_decode_codes(ctypes.byref(st), code_format, _ptr(q), N,
                                         rows_per_request, Hq, _ptr(block_tables), mb,
                                         _ptr(context_lens), max_context_len, float(sm_scale),
                                         _ptr(out), _ptr(workspace), workspace.numel(),
                                         _ptr(err_flags), _stream(stream)),
           "kvq_paged_decode_codes")
    return out


def dequant_rows(cache: Cache, slot_ids: torch.Tensor, out_dtype=torch.float32,
                 out_k: torch.Tensor | None = None, out_v: torch.Tensor | None = None,
                 err_flags: torch.Tensor | None = None, stream=None):
    """kvq_dequant_rows: fp32 or bf16 rows [n, H, D] of K and V at ``slot_ids``."""
    if slot_ids.dtype != torch.int64:
        raise ValueError("slot_ids must be int64")
    code = {torch.float32: 0, torch.bfloat16: 1}[out_dtype]
    n = slot_ids.numel()
    shape = (n, cache.num_kv_heads, cache.head_dim)
    if out_k is None:
        out_k = torch.empty(shape, dtype=out_dtype, device=cache.k_codes.device)
    if out_v is None:
        out_v = torch.empty(shape, dtype=out_dtype, device=cache.k_codes.device)
    st = cache.struct()
    _check(load().kvq_dequant_rows(ctypes.byref(st), _ptr(slot_ids), n, code, _ptr(out_k),
                                   _ptr(out_v), _ptr(err_flags), _stream(stream)),
           "kvq_dequant_rows")
    return out_k, out_v


# ---------------------------------------------------------------------------
# compressed index keys

@dataclass
class IndexCache:
    """Device tensors of an index-key cache (one row of ``dim`` values per slot).

    FP8:   codes uint8 [num_slots, dim], scales float32 [num_slots]
    MXFP4: codes uint8 [num_slots, dim/2] (E2M1 pairs), exponents uint8
           [num_slots, dim/32] (E8M0)"""
    format: int
    codes: torch.Tensor
    scales: torch.Tensor | None = None
    exponents: torch.Tensor | None = None

    @staticmethod
    def empty(num_slots: int, format: int, dim: int = 128, device="cuda") -> "IndexCache":
        if format == INDEX_FP8:
            return IndexCache(format,
                              torch.zeros(num_slots, dim, dtype=torch.uint8, device=device),
                              scales=torch.zeros(num_slots, dtype=torch.float32, device=device))
        if format == INDEX_MXFP4:
            return IndexCache(format,
                              torch.zeros(num_slots, dim // 2, dtype=torch.uint8, device=device),
                              exponents=torch.zeros(num_slots, dim // 32, dtype=torch.uint8,
                                                    device=device))
        raise ValueError("format must be INDEX_FP8 or INDEX_MXFP4")

    @property
    def num_slots(self) -> int:
        return self.codes.shape[0]

    @property
    def dim(self) -> int:
        return self.codes.shape[1] * (1 if self.format == INDEX_FP8 else 2)

    def struct(self) -> _IndexCacheStruct:
        for t in (self.codes, self.scales, self.exponents):
            if t is not None and not t.is_contiguous():
                raise ValueError("index cache tensors must be contiguous")
        return _IndexCacheStruct(self.codes.data_ptr(),
                                 0 if self.scales is None else self.scales.data_ptr(),
                                 0 if self.exponents is None else self.exponents.data_ptr(),
                                 self.num_slots, self.format, self.dim)


def index_cache_bytes(num_slots: int, format: int, dim: int = 128) -> int:
    return load().kvq_index_cache_bytes(num_slots, format, dim)


def index_quantize_scatter(cache: IndexCache, x: torch.Tensor, slot_ids: torch.Tensor,
                           err_flags: torch.Tensor | None = None, stream=None) -> None:
    """kvq_index_quantize_scatter: bf16 rows [T, dim] (a view with unit inner
    stride; any token stride) into ``cache`` at device int64 ``slot_ids``."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != cache.dim or x.stride(1) != 1:
        raise ValueError(f"x: expected bf16 [T, {cache.dim}] with unit inner stride")
    if slot_ids.dtype != torch.int64 or slot_ids.numel() != x.shape[0]:
        raise ValueError("slot_ids must be int64 with one id per row")
    st = cache.struct()
    _check(load().kvq_index_quantize_scatter(ctypes.byref(st), _ptr(x), x.stride(0), x.shape[0],
                                             _ptr(slot_ids), _ptr(err_flags), _stream(stream)),
           "kvq_index_quantize_scatter")


def index_dequant_rows(cache: IndexCache, slot_ids: torch.Tensor, out_dtype=torch.float32,
                       err_flags: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvq_index_dequant_rows: fp32 or bf16 rows [n, dim] at ``slot_ids``."""
    if slot_ids.dtype != torch.int64:
        raise ValueError("slot_ids must be int64")
    code = {torch.float32: 0, torch.bfloat16: 1}[out_dtype]
    n = slot_ids.numel()
    out = torch.empty((n, cache.dim), dtype=out_dtype, device=cache.codes.device)
    st = cache.struct()
    _check(load().kvq_index_dequant_rows(ctypes.byref(st), _ptr(slot_ids), n, code, _ptr(out),
                                         _ptr(err_flags), _stream(stream)),
           "kvq_index_dequant_rows")
    return out


def index_scores(cache: IndexCache, block_size: int, q: torch.Tensor, block_tables: torch.Tensor,
                 context_lens: torch.Tensor, max_context_len: int,
                 out: torch.Tensor | None = None, err_flags: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """kvq_index_scores: stacked index scores fp32 [N * R, max_context_len] for
    bf16 queries ``q`` [N, R, H, dim] over the paged index keys; -inf where a
    row does not see a token."""
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 4 \
            or q.shape[3] != cache.dim:
        raise ValueError(f"q must be a contiguous bf16 [N, R, H, {cache.dim}] tensor")
    if block_tables.dtype != torch.int32 or not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous int32 [N, max_blocks]")
    if context_lens.dtype != torch.int32 or not context_lens.is_contiguous():
        raise ValueError("context_lens must be contiguous int32 [N]")
    N, R, H = q.shape[0], q.shape[1], q.shape[2]
    if block_tables.shape[0] != N or context_lens.numel() != N:
        raise ValueError("block_tables / context_lens must have one entry per request")
    if out is None:
        out = torch.empty((N * R, max_context_len), dtype=torch.float32, device=q.device)
    elif out.dtype != torch.float32 or not out.is_contiguous() \
            or tuple(out.shape) != (N * R, max_context_len):
        raise ValueError("out must be contiguous fp32 [N * R, max_context_len]")
    st = cache.struct()
    _check(load().kvq_index_scores(ctypes.byref(st), block_size, _ptr(q), N, R, H,
                                   _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                   max_context_len, _ptr(out), _ptr(err_flags), _stream(stream)),
           "kvq_index_scores")
    return out
