"""kvq_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (it uses a fixed scratch array inside the library
instead of a caller workspace).  Called through the C ABI and checked against
kvq_paged_decode on the same inputs, twice in a row, with shapes that need the
split-K scratch; with the default partition choice (the load-balanced kernel,
which keeps its piece counts and slots in the array) against the oracle, twice
in a row with different lengths; plus the refusal of a shape larger than the
array.

This file is collected last so that a run stopping at its first failure has
already run every other test; it builds its own inputs and passes alone."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import workloads
from fp8_paged_kv_kvq_gb300 import build as kbuild
from kvq_testlib import (REL_L2, assert_attention_close, attention_errors, build_paged,
                         oracle_decode)

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def _noalloc_fn():
    kbuild.build()
    lib = kvq.load()
    fn = lib.kvq_paged_decode_noalloc
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(kvq._CacheStruct), P, i32, i32, i32, P, i32, P, i32,
                   ctypes.c_float, i32, P, P, P]
    return fn


def _call(fn, cache, q, bt, cl, maxc, sm, R, part, out, err):
    st = cache.struct()
    return fn(ctypes.byref(st), ctypes.c_void_p(q.data_ptr()), bt.shape[0], R, q.shape[1],
              ctypes.c_void_p(bt.data_ptr()), bt.shape[1], ctypes.c_void_p(cl.data_ptr()), maxc,
              sm, part, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(err.data_ptr()),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_the_workspace_decode_twice_in_a_row():
    fn = _noalloc_fn()
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=4)
    lens = np.array([700, 2500, 64, 3000], dtype=np.int32)
    built = build_paged(w, lens, oracle_side=False)
    cache = built["cache"]
    bt = torch.from_numpy(built["bt"]).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, (P, seed, ln) in enumerate([(256, 1, lens), (128, 2, lens - np.array([0, 900, 0, 5]))]):
        g = workloads.generator(seed, 55)
        q = torch.randn(4, w.num_q_heads, 128, generator=g).to(torch.bfloat16).cuda()
        cl = torch.from_numpy(ln.astype(np.int32)).cuda()
        need = kvq.paged_decode_workspace_size(4, 1, w.num_q_heads, w.num_kv_heads, 128,
                                               w.block_size, 3000, P)
        assert 0 < need <= SCRATCH_BYTES          # the shape does use the scratch
        out = torch.full_like(q, float("nan"))
        assert _call(fn, cache, q, bt, cl, 3000, w.sm_scale, 1, P, out, err) == 0
        ref = kvq.paged_decode(cache, q, bt, cl, 3000, w.sm_scale, partition_tokens=P)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        mx, rel, _, _ = attention_errors(out, ref.float().cpu().numpy().astype(np.float64))
        assert mx <= 1.0 and rel <= REL_L2, (call, mx, rel)


def test_noalloc_default_partition_against_the_oracle():
    """partition_tokens = 0 on a small decode batch: the library picks its
    load-balanced kernel, which keeps its piece counts and slots in the
    scratch array.  Two calls in a row with different context lengths (and a
    different number of pieces per request) are checked against the oracle, so
    nothing the first call left in the array leaks into the second."""
    fn = _noalloc_fn()
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=5)
    lens = np.array([4096, 300, 1, 2000, 777], dtype=np.int32)
    built = build_paged(w, lens, oracle_side=True)
    cache = built["cache"]
    bt = torch.from_numpy(built["bt"]).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, (seed, ln) in enumerate([(3, lens), (4, np.array([1500, 299, 0, 2000, 20]))]):
        ln = ln.astype(np.int32)
        need = kvq.paged_decode_workspace_size(5, 1, w.num_q_heads, w.num_kv_heads, 128,
                                               w.block_size, 4096, 0)
        assert 0 < need <= SCRATCH_BYTES
        g = workloads.generator(seed, 56)
        q = torch.randn(5, w.num_q_heads, 128, generator=g).to(torch.bfloat16)
        out = torch.full((5, w.num_q_heads, 128), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        assert _call(fn, cache, q.cuda(), bt, torch.from_numpy(ln).cuda(), 4096, w.sm_scale, 1,
                     0, out, err) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref, e = oracle_decode(built, q, 1, w.num_q_heads, w.sm_scale, lens=ln)
        assert e == 0
        assert_attention_close(out, ref, f"noalloc default partition, call {call}")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    fn = _noalloc_fn()
    cache = kvq.Cache.empty(64, 8, 128, 64)
    q = torch.zeros(64, 32, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(64, 1024, dtype=torch.int32, device="cuda")
    cl = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    need = kvq.paged_decode_workspace_size(64, 1, 32, 8, 128, 64, 65536, 256)
    assert need > SCRATCH_BYTES
    assert _call(fn, cache, q, bt, cl, 65536, 0.1, 1, 256, out, err) == 4   # WORKSPACE_TOO_SMALL
