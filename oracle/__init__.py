"""CPU oracle for the FP8 E4M3 paged KV cache -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg import this package.  The product (``fp8_paged_kv_kvq_gb300``, its
CUDA library and C ABI) never imports, links or calls it, and it imports nothing
from the product: the two share no code.  The arithmetic lives in
``kvq_oracle.c`` (plain C11, fp64 attention, IEEE binary32 quantisation) and in
``dense.py`` (a numpy brute-force attention used to cross-check it); this module
only compiles the C file with gcc and marshals numpy arrays through ctypes.

Pages followed (title and section):
  * ROCm/ATOM PR #2655 "fix(qwen4-exp): register the QSA FP8 scale planes for
    KV offload" -- PR description, K/V bullet (per-row FP32 scale = amax / FP8
    max; key scale on the score, value scale on the probability).
  * FlashML-org/FreeToken PR #354 "feat(kvcache): store the KV cache as fp8 e4m3
    codes" -- PR description (uint8 codes + fp32 row-scale sidecar, fused
    quantize+scatter to device slot ids) and the fix commit "give the V tensor
    its own row pitch in the fp8 KV store".
  * sgl-project/sglang-jax #1776 "feat(dsa): implement fp8 KV cache (e4m3) with
    a bf16 indexer cache" -- design points (448 range, 0.0156 normal floor, ~6%
    worst-case relative error of e4m3).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None

ERR_SLOT_RANGE = 1
ERR_BLOCK_RANGE = 2
ERR_CONTEXT_RANGE = 4


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into a shared library (gcc, -O2, no fp contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            lib.kvqo_e4m3_decode.restype = f64
            lib.kvqo_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.kvqo_e4m3_encode.restype = ctypes.c_uint8
            lib.kvqo_e4m3_encode.argtypes = [ctypes.c_float]
            lib.kvqo_float_to_bf16.restype = ctypes.c_uint16
            lib.kvqo_float_to_bf16.argtypes = [ctypes.c_float]
            lib.kvqo_e4m3_encode_array.restype = None
            lib.kvqo_e4m3_encode_array.argtypes = [P, i64, P]
            lib.kvqo_float_to_bf16_array.restype = None
            lib.kvqo_float_to_bf16_array.argtypes = [P, i64, P]
            lib.kvqo_quantize_row.restype = None
            lib.kvqo_quantize_row.argtypes = [P, ctypes.c_int, P, P]
            lib.kvqo_quantize_rows.restype = None
            lib.kvqo_quantize_rows.argtypes = [P, i64, ctypes.c_int, P, P]
            lib.kvqo_quantize_scatter.restype = i32
            lib.kvqo_quantize_scatter.argtypes = [P, i64, P, i64, i64, ctypes.c_int,
                                                  ctypes.c_int, P, i64, P, P, P, P]
            lib.kvqo_dequant_rows.restype = None
            lib.kvqo_e5m2_decode.restype = f64
            lib.kvqo_e5m2_decode.argtypes = [ctypes.c_uint8]
            lib.kvqo_e5m2_encode.restype = ctypes.c_uint8
            lib.kvqo_e5m2_encode.argtypes = [ctypes.c_float]
            lib.kvqo_e5m2_encode_array.restype = None
            lib.kvqo_e5m2_encode_array.argtypes = [P, i64, P]
            lib.kvqo_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.kvqo_e2m1_decode.restype = ctypes.c_double
            lib.kvqo_e2m1_encode.argtypes = [ctypes.c_double]
            lib.kvqo_e2m1_encode.restype = ctypes.c_uint8
            lib.kvqo_mxfp4_group_exponent.argtypes = [ctypes.c_double]
            lib.kvqo_mxfp4_group_exponent.restype = ctypes.c_int
            lib.kvqo_mxfp4_quantize_rows.argtypes = [P, i64, ctypes.c_int, P, P]
            lib.kvqo_mxfp4_quantize_rows.restype = None
            lib.kvqo_mxfp4_dequant_rows.argtypes = [P, P, i64, ctypes.c_int, P]
            lib.kvqo_mxfp4_dequant_rows.restype = None
            lib.kvqo_index_scores.argtypes = [ctypes.c_int, P, P, P, i64, ctypes.c_int,
                                              ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, P, ctypes.c_int, P]
            lib.kvqo_index_scores.restype = ctypes.c_int32
            lib.kvqo_dequant_rows.argtypes = [P, P, i64, ctypes.c_int, ctypes.c_int, P,
                                              i64, ctypes.c_int, P]
            lib.kvqo_paged_attention.restype = i32
            lib.kvqo_paged_attention.argtypes = [P, P, P, P, i64, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, P,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 P, ctypes.c_int, P, f64, P]
            lib.kvqo_paged_attention_units.restype = i32
            lib.kvqo_paged_attention_units.argtypes = [P, P, P, P, i64, ctypes.c_int,
                                                       ctypes.c_int, ctypes.c_int, P,
                                                       ctypes.c_int, ctypes.c_int,
                                                       ctypes.c_int, P, ctypes.c_int, P,
                                                       f64, P, i64, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------
# codec

def e4m3_decode(codes) -> np.ndarray:
    """Exact value of each e4m3 code (float64; NaN for 0x7F / 0xFF)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.kvqo_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e4m3_encode(q) -> np.ndarray:
    """Round-to-nearest-even, saturating e4m3 code of each finite float32."""
    lib = _load()
    shape = np.shape(q)
    qa = _c(np.reshape(q, -1), np.float32)
    out = np.empty(qa.shape, dtype=np.uint8)
    lib.kvqo_e4m3_encode_array(_ptr(qa), qa.size, _ptr(out))
    return out.reshape(shape)


def e5m2_decode(codes) -> np.ndarray:
    """Exact value of each e5m2 code (float64; +-inf for 0x7C / 0xFC, NaN for
    the other exponent-31 codes)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.kvqo_e5m2_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e5m2_encode(q) -> np.ndarray:
    """Round-to-nearest-even, saturating e5m2 code of each finite float32."""
    lib = _load()
    shape = np.shape(q)
    qa = _c(np.reshape(q, -1), np.float32)
    out = np.empty(qa.shape, dtype=np.uint8)
    lib.kvqo_e5m2_encode_array(_ptr(qa), qa.size, _ptr(out))
    return out.reshape(shape)


def float_to_bf16_bits(x) -> np.ndarray:
    lib = _load()
    shape = np.shape(x)
    xa = _c(np.reshape(x, -1), np.float32)
    out = np.empty(xa.shape, dtype=np.uint16)
    lib.kvqo_float_to_bf16_array(_ptr(xa), xa.size, _ptr(out))
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# quantize

def quantize_rows(x_bf16_bits: np.ndarray):
    """Quantise rows [..., D] of bf16 (given as uint16 bit patterns).

    Returns (codes uint8 [..., D], scales float32 [...])."""
    lib = _load()
    x = _c(x_bf16_bits, np.uint16)
    D = x.shape[-1]
    rows = x.reshape(-1, D)
    codes = np.empty(rows.shape, dtype=np.uint8)
    scales = np.empty(rows.shape[0], dtype=np.float32)
    lib.kvqo_quantize_rows(_ptr(rows), rows.shape[0], D, _ptr(codes), _ptr(scales))
    return codes.reshape(x.shape), scales.reshape(x.shape[:-1])


def quantize_scatter(k_bits: np.ndarray, k_token_stride: int,
                     v_bits: np.ndarray, v_token_stride: int,
                     num_tokens: int, H: int, D: int, slot_ids: np.ndarray,
                     cache: dict) -> int:
    """Quantise K/V rows given as flat uint16 buffers with their own token
    pitches (elements) and scatter them into ``cache`` (numpy arrays
    k_codes/v_codes [S, H, D] uint8, k_scales/v_scales [S, H] float32), in
    place.  Returns the error word."""
    lib = _load()
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    sid = _c(slot_ids, np.int64)
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        a = cache[name]
        assert a.flags["C_CONTIGUOUS"], name
    need_k = (num_tokens - 1) * k_token_stride + H * D if num_tokens else 0
    need_v = (num_tokens - 1) * v_token_stride + H * D if num_tokens else 0
    assert k.size >= need_k and v.size >= need_v, "source buffer too small"
    S = cache["k_codes"].shape[0]
    return int(lib.kvqo_quantize_scatter(
        _ptr(k), k_token_stride, _ptr(v), v_token_stride, num_tokens, H, D,
        _ptr(sid), S, _ptr(cache["k_codes"]), _ptr(cache["v_codes"]),
        _ptr(cache["k_scales"]), _ptr(cache["v_scales"])))


def e2m1_decode(codes) -> np.ndarray:
    """E2M1 code (low 4 bits) -> value, float64 (MXFP4 element format)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.kvqo_e2m1_decode(int(x)) for x in c.ravel()]).reshape(c.shape)


def e2m1_encode(q) -> np.ndarray:
    """Nearest E2M1 code to each value (ties to even), sign kept."""
    lib = _load()
    a = np.asarray(q, dtype=np.float64)
    return np.array([lib.kvqo_e2m1_encode(float(x)) for x in a.ravel()],
                    dtype=np.uint8).reshape(a.shape)


def mxfp4_group_exponent(amax: float) -> int:
    """Smallest X with amax <= 6 * 2^X, clamped to [-127, 127]."""
    return int(_load().kvqo_mxfp4_group_exponent(float(amax)))


def mxfp4_quantize_rows(x_bf16_bits: np.ndarray):
    """MXFP4 rows: x [..., D] bf16 bit patterns (D a multiple of 32) ->
    (codes uint8 [..., D/2] packed pairs, exps uint8 [..., D/32] E8M0)."""
    lib = _load()
    x = _c(x_bf16_bits, np.uint16)
    D = x.shape[-1]
    assert D % 32 == 0
    rows = x.reshape(-1, D)
    codes = np.empty((rows.shape[0], D // 2), dtype=np.uint8)
    exps = np.empty((rows.shape[0], D // 32), dtype=np.uint8)
    lib.kvqo_mxfp4_quantize_rows(_ptr(rows), rows.shape[0], D, _ptr(codes), _ptr(exps))
    return codes.reshape(x.shape[:-1] + (D // 2,)), exps.reshape(x.shape[:-1] + (D // 32,))


def mxfp4_dequant_rows(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    """codes [n, D/2], exps [n, D/32] -> float32 [n, D]."""
    lib = _load()
    c = _c(codes, np.uint8)
    e = _c(exps, np.uint8)
    n, half = c.shape
    out = np.empty((n, 2 * half), dtype=np.float32)
    lib.kvqo_mxfp4_dequant_rows(_ptr(c), _ptr(e), n, 2 * half, _ptr(out))
    return out


def empty_cache(num_slots: int, H: int, D: int) -> dict:
    return {
        "k_codes": np.zeros((num_slots, H, D), dtype=np.uint8),
        "v_codes": np.zeros((num_slots, H, D), dtype=np.uint8),
        "k_scales": np.zeros((num_slots, H), dtype=np.float32),
        "v_scales": np.zeros((num_slots, H), dtype=np.float32),
    }


def dequant_rows(codes: np.ndarray, scales: np.ndarray, slot_ids, out_dtype: int = 0):
    """Dequantise the rows at ``slot_ids``: fp32 (out_dtype 0) or bf16 bit
    patterns as uint16 (out_dtype 1); shape [n, H, D]."""
    lib = _load()
    c = _c(codes, np.uint8)
    s = _c(scales, np.float32)
    S, H, D = c.shape
    sid = _c(slot_ids, np.int64)
    n = sid.size
    out = np.empty((n, H, D), dtype=np.float32 if out_dtype == 0 else np.uint16)
    lib.kvqo_dequant_rows(_ptr(c), _ptr(s), S, H, D, _ptr(sid), n, out_dtype, _ptr(out))
    return out


# ---------------------------------------------------------------------------
# attention

def paged_attention(cache: dict, q_bits: np.ndarray, N: int, R: int, Hq: int,
                    block_tables: np.ndarray, context_lens: np.ndarray,
                    block_size: int, sm_scale: float):
    """fp64 paged GQA attention over the dequantised cache.

    q_bits: bf16 bit patterns [N*R, Hq, D].  Returns (out float64
    [N*R, Hq, D], error word)."""
    lib = _load()
    kc, vc = _c(cache["k_codes"], np.uint8), _c(cache["v_codes"], np.uint8)
    ks, vs = _c(cache["k_scales"], np.float32), _c(cache["v_scales"], np.float32)
    S, H, D = kc.shape
    q = _c(q_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.zeros((N * R, Hq, D), dtype=np.float64)
    err = lib.kvqo_paged_attention(_ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), S, H, D,
                                   block_size, _ptr(q), N, R, Hq, _ptr(bt), bt.shape[1],
                                   _ptr(cl), float(sm_scale), _ptr(out))
    if err < 0:
        raise MemoryError("oracle attention: allocation failed")
    return out, int(err)


def paged_attention_units(cache: dict, q_bits: np.ndarray, N: int, R: int, Hq: int,
                          block_tables: np.ndarray, context_lens: np.ndarray,
                          block_size: int, sm_scale: float, units):
    """Same as ``paged_attention`` for a list of (request, row, q head) units.
    Returns (out float64 [len(units), D], error word)."""
    lib = _load()
    kc, vc = _c(cache["k_codes"], np.uint8), _c(cache["v_codes"], np.uint8)
    ks, vs = _c(cache["k_scales"], np.float32), _c(cache["v_scales"], np.float32)
    S, H, D = kc.shape
    q = _c(q_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    u = _c(np.asarray(units).reshape(-1, 3), np.int32)
    out = np.zeros((u.shape[0], D), dtype=np.float64)
    err = lib.kvqo_paged_attention_units(_ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), S, H,
                                         D, block_size, _ptr(q), N, R, Hq, _ptr(bt),
                                         bt.shape[1], _ptr(cl), float(sm_scale),
                                         _ptr(u), u.shape[0], _ptr(out))
    if err < 0:
        raise ValueError("oracle attention: bad unit or allocation failure")
    return out, int(err)


def index_scores(fmt: int, codes: np.ndarray, scales, exps, block_tables: np.ndarray,
                 block_size: int, context_lens: np.ndarray, R: int, H: int,
                 q_bits: np.ndarray, max_len: int):
    """Index scores in float64 [N*R, max_len]: sum over heads of max(0, q . k),
    -inf where a row does not see the token (format 0 FP8 keys with scales,
    1 MXFP4 keys with exponents).  Returns (scores, error word)."""
    lib = _load()
    c = _c(codes, np.uint8)
    S = c.shape[0]
    D = c.shape[1] if fmt == 0 else 2 * c.shape[1]
    sc = _c(scales if scales is not None else np.zeros(1, np.float32), np.float32)
    ex = _c(exps if exps is not None else np.zeros(1, np.uint8), np.uint8)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    qb = _c(q_bits, np.uint16)
    N = cl.size
    out = np.empty((N * R, max_len), dtype=np.float64)
    err = lib.kvqo_index_scores(fmt, _ptr(c), _ptr(sc), _ptr(ex), S, D, block_size, _ptr(bt),
                                bt.shape[1], _ptr(cl), N, R, H, _ptr(qb), max_len, _ptr(out))
    return out, int(err)
