"""kvq_paged_decode on the GPU against the fp64 oracle (the oracle quantises
the same seeded bf16 rows itself): decode and multi-row verify shapes,
single-partition and split-K paths, ragged tails, edge cases, and the large
workloads at full size on every output (verify: every request of one KV
head)."""
import numpy as np
import pytest
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import oracle
import workloads
from kvq_testlib import (assert_attention_close, assert_cache_equal, build_custom, build_paged,
                         gpu_decode, oracle_decode)

pytestmark = pytest.mark.gpu


def _queries(w, N, R, seed):
    g = workloads.generator(seed, 77)
    return torch.randn(N * R, w.num_q_heads, w.head_dim, generator=g).to(torch.bfloat16)


def test_tiny_workload():
    w = workloads.WORKLOADS["tiny"]
    lens = workloads.context_lengths(w)
    built = build_paged(w, lens, spare_blocks=0)
    assert_cache_equal(built["cache"], built["ocache"])
    q = workloads.queries(w)
    out = gpu_decode(built, q, 1, w.sm_scale)
    ref, err = oracle_decode(built, q, 1, w.num_q_heads, w.sm_scale)
    assert err == 0
    assert_attention_close(out, ref, "tiny")


@pytest.mark.parametrize("partition_tokens", [0, 64, 128, 256, 1024])
def test_decode_batch_scaled(partition_tokens):
    """The decode-batch shape (GQA 4, block size 16, log-normal rows) with
    fewer, shorter requests; ragged lengths exercise partial stages."""
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=5)
    lens = np.array([1, 63, 64, 700, 1500], dtype=np.int32)
    built = build_paged(w, lens)
    assert_cache_equal(built["cache"], built["ocache"])
    q = _queries(w, 5, 1, 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(built, q, 1, w.sm_scale, partition_tokens=partition_tokens, err=err)
    ref, _ = oracle_decode(built, q, 1, w.num_q_heads, w.sm_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, f"decode P={partition_tokens}")


@pytest.mark.parametrize("R,Hq,H,bs", [
    (4, 64, 8, 64),    # the verify shape: 4 rows x GQA 8 = 32 stacked rows
    (4, 32, 8, 16),    # 16 rows
    (2, 32, 8, 16),    # 8 rows
    (1, 8, 8, 16),     # MHA
    (4, 128, 8, 64),   # 64 rows: two row groups
    (3, 12, 4, 32),    # 9 rows, odd group
    (1, 32, 8, 4),     # block size 4: cp.async staging
    (2, 16, 4, 8),     # block size 8: smallest TMA page box
    (4, 64, 8, 128),   # block larger than a 64-token stage
    (4, 32, 8, 256),   # 16 rows on 256-token pages: the rows-on-M kernel, 32-row tiles
    (4, 96, 8, 32),    # 48 rows: the rows-on-M kernel, 64-row tiles
])
@pytest.mark.parametrize("partition_tokens", [0, 128])
def test_verify_shapes(R, Hq, H, bs, partition_tokens):
    w = workloads.scaled(workloads.WORKLOADS["verify"], num_requests=3, rows_per_request=R,
                         num_q_heads=Hq, num_kv_heads=H, block_size=bs)
    lens = np.array([R, 333, 520], dtype=np.int32)
    built = build_paged(w, lens)
    q = _queries(w, 3, R, 2)
    out = gpu_decode(built, q, R, w.sm_scale, partition_tokens=partition_tokens)
    ref, _ = oracle_decode(built, q, R, Hq, w.sm_scale)
    assert_attention_close(out, ref, f"R={R} Hq={Hq} H={H} P={partition_tokens}")


def _many_lens(n, hi, seed):
    return [int(x) for x in np.random.default_rng(seed).integers(0, hi + 1, n)]


@pytest.mark.parametrize("R,Hq,H,lens", [
    (1, 32, 8, [0, 1, 15, 16, 17, 300, 1000, 2047, 33, 4096, 5, 0, 777]),
    (2, 16, 4, [3, 129, 640, 64, 2]),      # 8 stacked rows: 2 query rows x GQA 4
    (1, 8, 8, [6000, 20, 40]),             # one dominant request: 15 pieces per head group
    # enough chunks for the weighted split, many short segments per CTA (the
    # next segment's query rows staged while the current one runs)
    (1, 32, 8, _many_lens(300, 700, 11)),
    (2, 16, 4, _many_lens(200, 900, 12)),
    (1, 8, 4, _many_lens(1024, 48, 13)),     # the most requests it takes: a full prefix
])
def test_load_balanced_split(R, Hq, H, lens):
    """The library's own choice for small batches of <= 8 stacked rows on
    pages of >= 16 tokens: the batch's 16-token chunks spread over a
    persistent grid (equal ranges, or ranges weighted by the grid's thirds
    once every range still cuts a (request, head group) into at most 16
    pieces), the pieces merged by the combine; empty contexts give zero
    rows."""
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=len(lens),
                         rows_per_request=R, num_q_heads=Hq, num_kv_heads=H)
    lens = np.array(lens, dtype=np.int32)
    built = build_paged(w, lens)
    q = _queries(w, len(lens), R, 5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(built, q, R, w.sm_scale, err=err)
    ref, _ = oracle_decode(built, q, R, Hq, w.sm_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    empty = np.repeat(lens == 0, R)
    assert not out.float()[torch.from_numpy(empty)].any()
    assert_attention_close(out, ref, f"balanced R={R} Hq={Hq} H={H}")


@pytest.mark.parametrize("R,Hq,H,bs", [
    (1, 32, 8, 32),
    (2, 16, 4, 64),
    (1, 8, 4, 256),
])
def test_load_balanced_block_sizes(R, Hq, H, bs):
    """The load-balanced kernel on pages of 32 to 256 tokens (a 16-token
    chunk always lies within one page): contexts ending on and just past page
    edges, long ones spanning many pages, empty requests."""
    lens = [bs, bs + 1, 1, 0, 2 * bs - 1] + _many_lens(30, 3000, 40 + bs)
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=len(lens),
                         rows_per_request=R, num_q_heads=Hq, num_kv_heads=H, block_size=bs)
    lens = np.array(lens, dtype=np.int32)
    built = build_paged(w, lens)
    q = _queries(w, len(lens), R, 9)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(built, q, R, w.sm_scale, err=err)
    ref, _ = oracle_decode(built, q, R, Hq, w.sm_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, f"balanced bs={bs} R={R} Hq={Hq} H={H}")


@pytest.mark.parametrize("R,Hq,H,bs", [
    (4, 32, 8, 16),    # 16 stacked rows, 32-row tiles
    (4, 64, 4, 32),    # 64 stacked rows, 64-row tiles
])
def test_rows_kernel_most_requests(R, Hq, H, bs):
    """The rows-on-M kernel at the most requests it takes (1024: the request
    prefix fills its shared-memory array), short ragged contexts and empty
    requests among them, so that units are cut across CTAs all over the
    batch."""
    lens = np.array(_many_lens(1024, 300, 31), dtype=np.int32)
    lens[:R] = np.arange(R)                   # contexts shorter than the rows
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=len(lens),
                         rows_per_request=R, num_q_heads=Hq, num_kv_heads=H, block_size=bs)
    built = build_paged(w, lens, gen_device="cuda")
    q = _queries(w, len(lens), R, 8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(built, q, R, w.sm_scale, err=err)
    ref, _ = oracle_decode(built, q, R, Hq, w.sm_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, f"1024 requests R={R} Hq={Hq} H={H}")


@pytest.mark.parametrize("partition_tokens", [0, 1024, 8192])
def test_verify_climbing_scores_move_every_reference(partition_tokens):
    """The verify shape (32 stacked rows per KV head) with keys that grow along
    the context in the query's direction, so every row's score climbs by about
    25 (log2 units) per 128 tokens and every stage moves every row's softmax
    reference: the partitioned tcgen05 kernel switches through all of its
    accumulator buffers and then rescales in place; the rows-on-M kernel
    (partition 0) moves references in the middle of chunks and rescales both
    of its O buffers.  Value magnitudes grow too, sixfold over the longer
    context (the running bound on the value scales moves).  (The stated bound
    is absolute, for values of unit scale: with values grown 14-fold, the f16
    rounding of P'' alone -- the same in both tensor-core kernels -- already
    reaches 0.6 of it, so the growth stays moderate.)"""
    w = workloads.scaled(workloads.WORKLOADS["verify"], num_requests=2)
    R, Hq, H, D = w.rows_per_request, w.num_q_heads, w.num_kv_heads, w.head_dim
    G = Hq // H
    g = workloads.generator(31, 1)
    u = torch.randn(H, D, generator=g)                      # one direction per KV head
    kvs = []
    for L in (5120, 3001):
        t = torch.arange(L, dtype=torch.float32)[:, None, None]
        k = 0.012 * t * u[None] + 0.3 * torch.randn(L, H, D, generator=g)
        v = torch.randn(L, H, D, generator=g) * (1.0 + t / 1000.0)
        kvs.append((k.to(torch.bfloat16), v.to(torch.bfloat16)))
    built = build_custom(w, kvs)
    q = (u.repeat_interleave(G, dim=0)[None].expand(2 * R, Hq, D) +
         0.1 * torch.randn(2 * R, Hq, D, generator=g)).to(torch.bfloat16)
    out = gpu_decode(built, q, R, w.sm_scale, partition_tokens=partition_tokens)
    ref, err = oracle_decode(built, q, R, Hq, w.sm_scale)
    assert err == 0
    assert_attention_close(out, ref, f"climbing scores P={partition_tokens}")


def test_rows_that_see_nothing_and_empty_requests():
    w = workloads.scaled(workloads.WORKLOADS["verify"], num_requests=4, rows_per_request=4,
                         num_q_heads=16, num_kv_heads=4, block_size=16)
    lens = np.array([0, 1, 2, 200], dtype=np.int32)   # L < R: leading rows see nothing
    built = build_paged(w, lens)
    q = _queries(w, 4, 4, 3)
    for P in (0, 64):
        out = gpu_decode(built, q, 4, w.sm_scale, partition_tokens=P, max_context_len=256)
        ref, _ = oracle_decode(built, q, 4, 16, w.sm_scale)
        assert torch.all(out[:4].float() == 0)                  # request 0: L = 0
        assert torch.all(out[4:7].float() == 0)                 # request 1: rows 0..2 see nothing
        assert_attention_close(out, ref, f"edge P={P}")


def test_split_and_single_partition_agree():
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=2)
    lens = np.array([2000, 4096], dtype=np.int32)
    built = build_paged(w, lens, oracle_side=False)
    q = _queries(w, 2, 1, 4)
    one = gpu_decode(built, q, 1, w.sm_scale, partition_tokens=4096).float()
    many = gpu_decode(built, q, 1, w.sm_scale, partition_tokens=64).float()
    rel = (one - many).norm() / one.norm()
    assert rel < 3e-3


def test_bad_block_ids_and_lengths_are_flagged_not_faulted():
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=2)
    lens = np.array([100, 300], dtype=np.int32)
    built = build_paged(w, lens, oracle_side=False)
    q = _queries(w, 2, 1, 5).cuda()
    bt = torch.from_numpy(built["bt"]).cuda()
    bad = bt.clone()
    bad[1, 3] = 1 << 30
    bad[1, 4] = -5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cl = torch.from_numpy(lens).cuda()
    kvq.paged_decode(built["cache"], q, bad, cl, 300, w.sm_scale, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvq.ERRF_BLOCK_RANGE
    err.zero_()
    cl_bad = torch.tensor([100, 10 ** 6], dtype=torch.int32, device="cuda")
    out = kvq.paged_decode(built["cache"], q, bt, cl_bad, 300, w.sm_scale, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvq.ERRF_CONTEXT_RANGE
    assert torch.all(torch.isfinite(out.float()))


def test_graph_capture_of_decode():
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=3)
    lens = np.array([300, 900, 50], dtype=np.int32)
    built = build_paged(w, lens)
    q = _queries(w, 3, 1, 6).cuda()
    bt = torch.from_numpy(built["bt"]).cuda()
    cl = torch.from_numpy(lens).cuda()
    P = 128
    need = kvq.paged_decode_workspace_size(3, 1, w.num_q_heads, w.num_kv_heads, 128,
                                           w.block_size, 1024, P)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kvq.paged_decode(built["cache"], q, bt, cl, 1024, w.sm_scale, partition_tokens=P,
                         out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kvq.paged_decode(built["cache"], q, bt, cl, 1024, w.sm_scale, partition_tokens=P,
                         out=out, workspace=ws)
    out.zero_()
    q.mul_(-1.0)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    ref, _ = oracle_decode(built, q.cpu(), 1, w.num_q_heads, w.sm_scale)
    assert_attention_close(out, ref, "graph replay")


def _full_size(name, one_head=None, append=False):
    """The named workload at full size, in the configuration the benchmark
    times (default partition size, hence the same kernels and split), checked
    against the oracle on every (request, KV head) unit -- or, with `one_head`,
    on every request for that KV head.  The oracle quantises each unit's bf16
    rows itself (codes and both scale planes compared bit for bit) and computes
    its attention in fp64; the units run on all host cores (the oracle's C
    calls release the GIL).  With `append`, the cache holds each request's
    first L - R tokens and the decode step's call stores the last R itself."""
    import concurrent.futures
    import os
    w = workloads.WORKLOADS[name]
    lens = workloads.context_lengths(w)
    bt, nblk = workloads.block_tables(lens, w.block_size, w.seed)
    S = nblk * w.block_size
    H, D, G, R = w.num_kv_heads, w.head_dim, w.group, w.rows_per_request
    cache = kvq.Cache.empty(S, H, D, w.block_size)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ct = workloads.chunk_tokens(w)
    for r in range(w.num_requests):
        L = int(lens[r])
        n_prev = L - R if append else L
        slots_all = workloads.token_slots(bt, r, L, w.block_size)
        for c0 in range(0, n_prev, ct):
            n = min(ct, n_prev - c0)
            k, v = workloads.request_kv(w, r, c0, n, device="cuda")
            kvq.quantize_scatter(cache, k, v, torch.from_numpy(slots_all[c0:c0 + n]).cuda(), err)
    q = workloads.queries(w, device="cuda")
    btd, cld = torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda()
    if append:
        new = [workloads.request_kv(w, r, int(lens[r]) - R, R, device="cuda")
               for r in range(w.num_requests)]
        out = kvq.paged_decode_append(cache, torch.cat([k for k, _ in new]),
                                      torch.cat([v for _, v in new]), q, btd, cld,
                                      int(lens.max()), w.sm_scale, rows_per_request=R,
                                      err_flags=err)
    else:
        out = kvq.paged_decode(cache, q, btd, cld, int(lens.max()), w.sm_scale,
                               rows_per_request=R, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    out_h = out.float().cpu().numpy().astype(np.float64)
    q_h = workloads.bf16_bits(q.cpu())
    heads = list(range(H)) if one_head is None else [one_head]

    def unit(r, h, kb, vb, got_codes, got_scales):
        """Oracle side of one (request, KV head): its own one-head cache."""
        L = int(lens[r])
        slots = workloads.token_slots(bt, r, L, w.block_size)
        oc = oracle.empty_cache(S, 1, D)
        oracle.quantize_scatter(kb, D, vb, D, L, 1, D, slots, oc)
        for nm in ("k_codes", "v_codes"):
            assert np.array_equal(got_codes[nm], oc[nm][slots, 0]), f"{name} r={r} h={h} {nm}"
        for nm in ("k_scales", "v_scales"):
            assert np.array_equal(got_scales[nm].view(np.uint32),
                                  oc[nm][slots, 0].view(np.uint32)), f"{name} r={r} h={h} {nm}"
        qh = np.ascontiguousarray(q_h[r * R:(r + 1) * R, h * G:(h + 1) * G])
        ref, e = oracle.paged_attention(oc, qh, 1, R, G, bt[r:r + 1], lens[r:r + 1],
                                        w.block_size, w.sm_scale)
        assert e == 0
        return r, h, ref

    workers = max(1, len(os.sched_getaffinity(0)))
    gpu_all, ref_all, pending = [], [], []

    def collect(fut):
        r, h, ref = fut.result()
        gpu_all.append(out_h[r * R:(r + 1) * R, h * G:(h + 1) * G].reshape(-1))
        ref_all.append(ref.reshape(-1))

    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for r in range(w.num_requests):
            L = int(lens[r])
            sl = torch.from_numpy(workloads.token_slots(bt, r, L, w.block_size)).cuda()
            for h in heads:
                # the unit's rows, redrawn on the device chunk by chunk (one
                # head at a time keeps the host memory in flight small)
                kparts, vparts = [], []
                for c0 in range(0, L, ct):
                    n = min(ct, L - c0)
                    k, v = workloads.request_kv(w, r, c0, n, device="cuda")
                    kparts.append(workloads.bf16_bits(k[:, h]))
                    vparts.append(workloads.bf16_bits(v[:, h]))
                got_codes = {"k_codes": cache.k_codes[sl, h].cpu().numpy(),
                             "v_codes": cache.v_codes[sl, h].cpu().numpy()}
                got_scales = {"k_scales": cache.k_scales[sl, h].cpu().numpy(),
                              "v_scales": cache.v_scales[sl, h].cpu().numpy()}
                kb = np.concatenate(kparts).reshape(-1)
                vb = np.concatenate(vparts).reshape(-1)
                pending.append(ex.submit(unit, r, h, kb, vb, got_codes, got_scales))
                while len(pending) >= 2 * workers:      # bound the host memory in flight
                    collect(pending.pop(0))
        while pending:
            collect(pending.pop(0))
    n_units = len(ref_all)
    assert n_units == w.num_requests * len(heads)
    assert_attention_close(np.concatenate(gpu_all), np.concatenate(ref_all),
                           f"{name} full size, {n_units} (request, KV head) units, "
                           f"{workers} host threads")


def test_decode_batch_full_size():
    _full_size("decode")


def test_decode_step_with_append_full_size():
    """The benchmark's decode step: the new row of every request stored by the
    attention launch itself (kvq_paged_decode_append)."""
    _full_size("decode", append=True)


def test_verify_full_size():
    _full_size("verify", one_head=5)


def test_verify_step_with_append_full_size():
    """The verify step through kvq_paged_decode_append: 4 new rows per request
    stored at their block-table positions by the store's own launch (more
    than two rows per request), then the rows-on-M kernel."""
    _full_size("verify", one_head=2, append=True)


def test_long_context_full_size():
    _full_size("longctx")


def _constructed_cache(L, bs, k_code_fn, v_code_fn, ks_fn, vs_fn):
    """A cache written directly (codes and scales chosen by the test, not by
    the quantiser): one request, one KV head, tokens in permuted blocks."""
    lens = np.array([L], dtype=np.int32)
    bt, nblk = workloads.block_tables(lens, bs, 123, spare_blocks=2)
    S = nblk * bs
    oc = oracle.empty_cache(S, 1, 128)
    slots = workloads.token_slots(bt, 0, L, bs)
    j = np.arange(L)[:, None]
    d = np.arange(128)[None, :]
    oc["k_codes"][slots, 0] = k_code_fn(j, d).astype(np.uint8)
    oc["v_codes"][slots, 0] = v_code_fn(j, d).astype(np.uint8)
    oc["k_scales"][slots, 0] = ks_fn(np.arange(L)).astype(np.float32)
    oc["v_scales"][slots, 0] = vs_fn(np.arange(L)).astype(np.float32)
    cache = kvq.Cache(*(torch.from_numpy(oc[n]).cuda() for n in
                        ("k_codes", "v_codes", "k_scales", "v_scales")), bs)
    return {"cache": cache, "ocache": oc, "bt": bt, "lens": lens, "S": S}


def _no_nan(c):
    c = np.where((c & 0x7F) == 0x7F, c & 0x80, c)
    return c


@pytest.mark.parametrize("vscale", [1000.0, 2.0 ** 110, 2.0 ** -100])
def test_every_code_value_through_the_attention(vscale):
    """Uniform attention (all K codes zero) over V rows built from chosen codes:
    dims 0..7 hold the subnormal codes 0..7 in every token (so a flushed
    subnormal would show), the rest cycle through every finite code; value
    scales range over many binades around `vscale`."""
    L, bs = 384, 16
    built = _constructed_cache(
        L, bs, lambda j, d: np.zeros((j.size, d.size)),
        lambda j, d: np.where(d < 8, d + 0 * j, _no_nan((j * 7 + d * 3) % 256)),
        lambda j: np.ones_like(j, dtype=np.float64),
        lambda j: vscale * np.exp2((j % 9) - 4.0))
    q = _queries(workloads.scaled(workloads.WORKLOADS["tiny"], num_q_heads=1,
                                  num_kv_heads=1), 1, 1, 9)
    for P in (0, 64):
        out = gpu_decode(built, q, 1, 0.1, partition_tokens=P)
        ref, _ = oracle_decode(built, q, 1, 1, 0.1)
        g = out.float().cpu().numpy().astype(np.float64)
        rel = np.abs(g - ref) / np.abs(ref).max()
        assert rel.max() < 5e-3, (P, rel.max())
        # the subnormal-code dims: mean of d * 2^-9 * v_scale over tokens
        assert np.allclose(g[0, 0, 1:8], ref[0, 0, 1:8], rtol=8e-3, atol=0)


def test_scores_with_extreme_key_scales():
    """Key scales spanning 2^-60..2^60 with chosen codes: the score column
    scaling happens in fp32 after the code dot."""
    L, bs = 200, 16
    built = _constructed_cache(
        L, bs, lambda j, d: _no_nan((j * 5 + d * 11) % 256),
        lambda j, d: _no_nan((j * 3 + d * 7 + 1) % 256),
        lambda j: np.exp2((j % 13) * 10.0 - 60.0) * 1e-3,
        lambda j: np.exp2((j % 5) - 2.0))
    q = _queries(workloads.scaled(workloads.WORKLOADS["tiny"], num_q_heads=1,
                                  num_kv_heads=1), 1, 1, 10)
    out = gpu_decode(built, q, 1, 1.0 / np.sqrt(128))
    ref, _ = oracle_decode(built, q, 1, 1, 1.0 / np.sqrt(128))
    assert_attention_close(out, ref, "extreme key scales")


def _split_case(tiny: bool, R: int, G: int, H: int = 4, L: int = 96, bs: int = 16, seed=0):
    """Query rows whose element 0 is the row maximum 1.0 and whose other 127
    elements are bf16 values of 8 significant bits and random sign, either in
    [2^-16, 2^-10) (below the split's exactness threshold amax * 2^-9) or in
    [2^-9, 2^-1) (above it).  Every cached key holds, in dims 1..127, the code
    of 448 with the sign of the query element in even tokens and the opposite
    sign in odd tokens, so the scores come from those elements alone: s_even =
    +s, s_odd = -s, s near 0.5.  Values are +1 (even tokens) and -1 (odd).  The
    attention output is then a convex mix of +-1 whose derivative with respect
    to any score is at most 2 in magnitude."""
    rng = np.random.default_rng(seed)
    D = 128
    Hq = G * H
    mant = rng.integers(128, 256, size=(R * Hq, D - 1)).astype(np.float64) / 128.0
    ex = rng.integers(-16, -10, size=(R * Hq, D - 1)) if tiny else \
        rng.integers(-9, -1, size=(R * Hq, D - 1))
    sign = np.where(rng.random((R * Hq, D - 1)) < 0.5, -1.0, 1.0)
    qv = np.concatenate([np.ones((R * Hq, 1)), sign * mant * np.exp2(ex)], axis=1)
    q = torch.from_numpy(qv).to(torch.bfloat16).reshape(R, Hq, D)
    assert torch.equal(q.double(), torch.from_numpy(qv).reshape(R, Hq, D))   # exact in bf16
    # one KV head's query rows must agree on the key sign pattern: use the
    # pattern of the head's first row for every row of the head (the other
    # rows' scores are then smaller, never larger)
    lens = np.array([L], dtype=np.int32)
    bt, nblk = workloads.block_tables(lens, bs, 321, spare_blocks=2)
    S = nblk * bs
    oc = oracle.empty_cache(S, H, D)
    slots = workloads.token_slots(bt, 0, L, bs)
    c448 = 0x7E
    for h in range(H):
        sg = np.sign(qv[h * G, 1:])
        for j in range(L):
            pos = (sg > 0) if j % 2 == 0 else (sg < 0)
            oc["k_codes"][slots[j], h, 1:] = np.where(pos, c448, c448 | 0x80)
            oc["k_codes"][slots[j], h, 0] = 0
            oc["v_codes"][slots[j], h, :] = 0x38 if j % 2 == 0 else 0xB8   # +-1.0
    sm = 1.0 / np.sqrt(128.0)
    sum_abs = np.abs(qv[:, 1:]).sum(axis=1).max() * 448.0
    ks = np.float32(0.5 / (sm * sum_abs))
    oc["k_scales"][slots, :] = ks
    oc["v_scales"][slots, :] = np.float32(1.0)
    cache = kvq.Cache(*(torch.from_numpy(oc[n]).cuda() for n in
                        ("k_codes", "v_codes", "k_scales", "v_scales")), bs)
    built = {"cache": cache, "ocache": oc, "bt": bt, "lens": lens, "S": S}
    # the split's bound: an element below amax 2^-9 carries an absolute error
    # of at most 2^-10 2^e = 2^-17 (amax = 1, 2^e = 2^-7), so a score moves by
    # at most sm * ks * 127 * 448 * 2^-17
    ds = sm * float(ks) * 127 * 448 * 2.0 ** -17
    return built, q, sm, ds


@pytest.mark.parametrize("R,G", [(1, 4), (4, 8)])
def test_query_split_error_bound(R, G):
    """The two-piece e4m3 query split q = 2^e (p1 + p2): exact for every element
    of magnitude >= amax * 2^-9, and off by at most 2^-10 * 2^e (amax * 2^-17
    here) for smaller ones.  Scores built only from such elements move the
    output by at most twice the score error (plus f16-P and bf16 rounding);
    scores built from elements above the threshold are exact."""
    H = 4
    for tiny in (False, True):
        built, q, sm, ds = _split_case(tiny, R, G, H)
        out = gpu_decode(built, q, R, sm)
        ref, e = oracle_decode(built, q, R, G * H, sm)
        assert e == 0
        g = out.float().cpu().numpy().astype(np.float64)
        err = np.abs(g - ref)
        rounding = 2.0 ** -9 * np.abs(ref) + 2.0 ** -10
        bound = rounding + (2.0 * ds if tiny else 0.0)
        worst = float((err / bound).max())
        print(f"split R={R} G={G} tiny={tiny}: worst err / bound {worst:.3f}, "
              f"max err {err.max():.3e}, score bound {ds:.3e}")
        assert worst <= 1.0, (tiny, worst)


@pytest.mark.parametrize("R,Hq,H,bs,lens", [
    (1, 32, 8, 16, [5000, 300, 0, 2000]),      # the load-balanced decode kernel and its combine
    (4, 128, 8, 64, [3000, 900]),              # 64 rows: the rows-on-M kernel, cut units
])
def test_workspace_needs_no_initialisation(R, Hq, H, bs, lens):
    """A workspace full of arbitrary bytes (here 0xA5 and random) needs no
    clearing: the load-balanced decode writes its piece counts every call, and the
    rows-on-M kernel counts a cut unit's pieces in words tagged with the call.
    Calls in a row on it, and a captured CUDA graph replayed three times, all
    give the oracle's result."""
    w = workloads.scaled(workloads.WORKLOADS["verify"], num_requests=len(lens), rows_per_request=R,
                         num_q_heads=Hq, num_kv_heads=H, block_size=bs)
    lens = np.array(lens, dtype=np.int32)
    built = build_paged(w, lens)
    q = _queries(w, len(lens), R, 21)
    ref, _ = oracle_decode(built, q, R, Hq, w.sm_scale)
    bt = torch.from_numpy(built["bt"]).cuda()
    cl = torch.from_numpy(lens).cuda()
    maxc = int(lens.max())
    need = kvq.paged_decode_workspace_size(len(lens), R, Hq, H, 128, bs, maxc, 0)
    assert need > 0
    g = torch.Generator(device="cuda").manual_seed(5)
    for fill in ("a5", "random"):
        ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda") if fill == "a5" else \
            torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda", generator=g)
        for call in range(2):
            out = kvq.paged_decode(built["cache"], q.cuda(), bt, cl, maxc, w.sm_scale,
                                   rows_per_request=R, workspace=ws)
            torch.cuda.synchronize()
            assert_attention_close(out, ref, f"workspace {fill}, call {call}")
    qd = q.cuda()
    out = torch.empty_like(qd)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kvq.paged_decode(built["cache"], qd, bt, cl, maxc, w.sm_scale, rows_per_request=R,
                         out=out, workspace=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kvq.paged_decode(built["cache"], qd, bt, cl, maxc, w.sm_scale, rows_per_request=R,
                         out=out, workspace=ws)
    for rep in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_attention_close(out, ref, f"graph replay {rep}")
