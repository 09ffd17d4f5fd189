"""The C ABI without a GPU: libkvq.so builds for sm_103a, loads, exports every
function include/kvq.h declares, and its host-side validation and size
helpers answer before anything would be launched."""
import ctypes
import subprocess

import pytest

import fp8_paged_kv_kvq_gb300 as kvq
from fp8_paged_kv_kvq_gb300 import build as kbuild

OK, INVALID, UNSUPPORTED, MISALIGNED, WS_SMALL = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvq.load()


def test_header_declares_the_boundary():
    names = kvq.header_functions()
    for n in ("kvq_quantize_scatter", "kvq_paged_decode", "kvq_dequant_rows"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in kvq.header_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_library_targets_sm_103a_only():
    assert kbuild.ARCH == "-gencode=arch=compute_103a,code=sm_103a"
    flags = kbuild._flags()
    assert "-ftz=false" in flags and "-prec-div=true" in flags
    assert not any("fast-math" in f for f in flags)


def _cache(head_dim=128, block_size=16, slots=64, ptr=0x10000):
    return kvq._CacheStruct(ptr, ptr + 0x100000, ptr + 0x200000, ptr + 0x300000, slots, 8,
                            head_dim, block_size)


def test_status_strings_and_version(lib):
    assert lib.kvq_abi_version() == 3
    for s in range(6):
        assert lib.kvq_status_string(s)


def test_cache_bytes_counts_codes_and_scales(lib):
    # FreeToken PR #354: the pool counts codes plus the fp32 sidecar
    assert lib.kvq_cache_bytes(1000, 8, 128) == 2 * 1000 * 8 * (128 + 4)
    assert lib.kvq_cache_bytes(-1, 8, 128) == 0


def test_quantize_validation_happens_before_launch(lib):
    P = ctypes.c_void_p
    c = _cache()
    q = lib.kvq_quantize_scatter
    assert q(ctypes.byref(c), P(0), 0, P(0), 0, 0, P(0), P(0), P(0)) == OK
    assert q(None, P(16), 0, P(16), 0, 1, P(8), P(0), P(0)) == INVALID
    assert q(ctypes.byref(c), P(0), 1024, P(16), 1024, 4, P(8), P(0), P(0)) == INVALID
    assert q(ctypes.byref(c), P(16), 1024, P(16), 1024, -1, P(8), P(0), P(0)) == INVALID
    assert q(ctypes.byref(c), P(18), 1024, P(16), 1024, 4, P(8), P(0), P(0)) == MISALIGNED
    assert q(ctypes.byref(c), P(16), 1028, P(16), 1024, 4, P(8), P(0), P(0)) == MISALIGNED
    assert q(ctypes.byref(c), P(16), 1024, P(16), 1024, 4, P(12), P(0), P(0)) == MISALIGNED
    bad = _cache(head_dim=64)
    assert q(ctypes.byref(bad), P(16), 1024, P(16), 1024, 4, P(8), P(0), P(0)) == UNSUPPORTED
    mis = _cache(ptr=0x10008)
    assert q(ctypes.byref(mis), P(16), 1024, P(16), 1024, 4, P(8), P(0), P(0)) == MISALIGNED


def _decode(lib, c, q=16, N=2, R=1, Hq=32, bt=16, mb=4, cl=16, maxc=64, sm=0.1, part=0, out=16,
            ws=0, wsb=0):
    P = ctypes.c_void_p
    return lib.kvq_paged_decode(ctypes.byref(c) if c is not None else None, P(q), N, R, Hq, P(bt),
                                mb, P(cl), maxc, sm, part, P(out), P(ws), wsb, P(0), P(0))


def test_decode_validation_happens_before_launch(lib):
    c = _cache()
    assert _decode(lib, c, N=0) == OK
    assert _decode(lib, None) == INVALID
    assert _decode(lib, c, Hq=30) == INVALID                   # not a multiple of H
    assert _decode(lib, c, R=0) == INVALID
    assert _decode(lib, c, part=100) == INVALID                # not a multiple of 64
    assert _decode(lib, c, sm=float("nan")) == INVALID
    assert _decode(lib, c, R=5, Hq=256, part=64) == UNSUPPORTED   # 160 rows, fixed partitions
    assert _decode(lib, c, R=300, Hq=256) == UNSUPPORTED       # 9600 rows per KV head
    assert _decode(lib, _cache(head_dim=256)) == UNSUPPORTED
    assert _decode(lib, _cache(block_size=24)) == UNSUPPORTED  # not a power of two
    assert _decode(lib, _cache(block_size=0)) == INVALID
    assert _decode(lib, c, q=24) == MISALIGNED
    assert _decode(lib, c, out=8) == MISALIGNED
    assert _decode(lib, c, bt=2) == MISALIGNED
    assert _decode(lib, c, maxc=128, part=64) == WS_SMALL      # two partitions need a workspace
    need = lib.kvq_paged_decode_workspace_size(2, 1, 32, 8, 128, 16, 128, 64)
    assert _decode(lib, c, maxc=128, part=64, ws=256, wsb=need - 1) == WS_SMALL


def test_workspace_size_of_the_rows_split(lib):
    """More than 8 stacked rows per KV head with partition_tokens 0: one 64-bit
    ticket per (request, KV head, 128-row tile), rounded to 256 bytes, then two
    pieces per SM of rows-per-tile (32, 64 or 128) partial rows of 128 fp32 and
    their (max, denominator) pairs, each part rounded to 256 bytes."""
    sms = lib.kvq_test_sm_count() if hasattr(lib, "kvq_test_sm_count") else 152

    def expect(N, H, rows):
        T = (rows + 127) // 128
        rc = 32 if rows <= 32 else (64 if rows <= 64 else 128)
        r256 = lambda x: (x + 255) // 256 * 256
        return r256(N * H * T * 8) + r256(sms * 2 * rc * 128 * 4) + r256(sms * 2 * rc * 8)
    assert lib.kvq_paged_decode_workspace_size(64, 4, 64, 8, 128, 64, 32768, 0) == expect(64, 8, 32)
    # an explicit partition keeps 9..32 rows on the partitioned tcgen05 kernel
    assert lib.kvq_paged_decode_workspace_size(64, 4, 64, 8, 128, 64, 32768, 4096) != \
        expect(64, 8, 32)
    assert lib.kvq_paged_decode_workspace_size(4, 4, 32, 8, 128, 256, 4096, 0) == expect(4, 8, 16)
    assert lib.kvq_paged_decode_workspace_size(3, 3, 48, 4, 128, 16, 500, 0) == expect(3, 4, 36)
    assert lib.kvq_paged_decode_workspace_size(1, 512, 32, 8, 128, 64, 4096, 0) == expect(1, 8, 2048)


def test_workspace_size_formula(lib):
    n = lib.kvq_paged_decode_workspace_size(32, 1, 32, 8, 128, 16, 8192, 512)
    rows, parts = 32 * 32, 16
    o = rows * parts * 128 * 4
    ml = rows * parts * 2 * 4
    assert n == ((((o + 255) // 256) * 256 + ml + 255) // 256) * 256
    assert lib.kvq_paged_decode_workspace_size(32, 1, 32, 8, 128, 16, 512, 512) == 0
    assert lib.kvq_paged_decode_workspace_size(32, 1, 32, 8, 64, 16, 512, 512) == 0  # invalid


def test_partition_heuristic_is_a_power_of_two_multiple_of_64(lib):
    for N, maxc in ((1, 64), (32, 8192), (64, 32768), (2, 1 << 20)):
        p = lib.kvq_paged_decode_partition_tokens(N, 1, 32, 8, 16, maxc)
        assert p % 64 == 0 and (p & (p - 1)) == 0 and 256 <= p <= 8192
    # 9..32 stacked rows per KV head (tensor-core verify): longer partitions,
    # within the kernel's 512 pages per partition
    for N, bs, maxc in ((64, 64, 32768), (64, 16, 32768), (2, 128, 1 << 20)):
        p = lib.kvq_paged_decode_partition_tokens(N, 4, 64, 8, bs, maxc)
        assert p % 64 == 0 and (p & (p - 1)) == 0 and 256 <= p <= min(32768, 512 * bs)


def test_dequant_validation(lib):
    P = ctypes.c_void_p
    c = _cache()
    d = lib.kvq_dequant_rows
    assert d(ctypes.byref(c), P(8), 0, 0, P(16), P(16), P(0), P(0)) == OK
    assert d(ctypes.byref(c), P(8), 4, 2, P(16), P(16), P(0), P(0)) == INVALID
    assert d(ctypes.byref(c), P(0), 4, 0, P(16), P(16), P(0), P(0)) == INVALID
    assert d(ctypes.byref(c), P(8), 4, 0, P(20), P(16), P(0), P(0)) == MISALIGNED


def _index_cache(fmt=1, slots=64, ptr=0x10000):
    return kvq._IndexCacheStruct(ptr, ptr + 0x100000 if fmt == 0 else 0,
                                 ptr + 0x200000 if fmt == 1 else 0, slots, fmt, 128)


def test_index_cache_bytes_and_validation(lib):
    P = ctypes.c_void_p
    assert lib.kvq_index_cache_bytes(1000, 0, 128) == 1000 * 132
    assert lib.kvq_index_cache_bytes(1000, 1, 128) == 1000 * 68
    assert lib.kvq_index_cache_bytes(1000, 2, 128) == 0
    c = _index_cache()
    q = lib.kvq_index_quantize_scatter
    assert q(ctypes.byref(c), P(16), 128, 0, P(8), P(0), P(0)) == OK
    assert q(ctypes.byref(c), P(16), 129, 4, P(8), P(0), P(0)) == MISALIGNED
    bad = _index_cache()
    bad.format = 5
    assert q(ctypes.byref(bad), P(16), 128, 4, P(8), P(0), P(0)) == INVALID
    nodim = _index_cache()
    nodim.dim = 64
    assert q(ctypes.byref(nodim), P(16), 128, 4, P(8), P(0), P(0)) == UNSUPPORTED


def test_index_scores_validation_happens_before_launch(lib):
    """kvq_index_scores: R * H <= 16 with H in {1, 2, 4, 8}, a power-of-two
    block size, a 16-byte aligned query; empty batches launch nothing."""
    P = ctypes.c_void_p
    s = lib.kvq_index_scores
    c = _index_cache()

    def call(bs=16, q=16, N=2, R=4, H=4, mb=8, maxc=128, out=16):
        return s(ctypes.byref(c), bs, P(q), N, R, H, P(64), mb, P(128), maxc, P(out), P(0),
                 P(0))
    assert call(N=0) == OK and call(maxc=0) == OK
    assert call(H=3) == UNSUPPORTED
    assert call(R=5, H=4) == UNSUPPORTED
    assert call(bs=24) == UNSUPPORTED
    assert call(bs=8) == UNSUPPORTED
    assert call(bs=0) == INVALID
    assert call(R=0) == INVALID
    assert call(N=70000) == UNSUPPORTED
    assert call(q=24) == MISALIGNED
    assert call(out=18) == MISALIGNED
    assert call(q=0) == INVALID


def test_index_scores_binding_rejects_bad_tensors():
    """The Python binding checks dtypes and shapes before it calls the library
    (every call here raises before anything could be launched)."""
    import torch
    cache = kvq.IndexCache.empty(64, kvq.INDEX_MXFP4, device="cpu")
    bt = torch.zeros(2, 4, dtype=torch.int32)
    lens = torch.zeros(2, dtype=torch.int32)
    q = torch.zeros(2, 4, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kvq.index_scores(cache, 16, q.float(), bt, lens, 64)                 # not bf16
    with pytest.raises(ValueError):
        kvq.index_scores(cache, 16, q[..., :64], bt, lens, 64)               # wrong dim
    with pytest.raises(ValueError):
        kvq.index_scores(cache, 16, q, bt.long(), lens, 64)                  # int64 table
    with pytest.raises(ValueError):
        kvq.index_scores(cache, 16, q, bt[:1], lens, 64)                     # one table row
    with pytest.raises(ValueError):
        kvq.index_scores(cache, 16, q, bt, lens, 64,
                         out=torch.empty(8, 32, dtype=torch.float32))        # wrong out shape
