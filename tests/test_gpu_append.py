"""kvq_paged_decode_append on the GPU against the oracle: one decode step's
store of the new K/V rows (at positions L - R .. L - 1 of each request's block
table) and the attention that reads them, in one launch where the shape takes
the load-balanced kernel, as two launches elsewhere.  The cache holds each
request's earlier tokens; the oracle stores the same bf16 rows itself, so the
codes and scales of every position are compared bit for bit and the outputs
against fp64 attention."""
import numpy as np
import pytest
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import oracle
import workloads
from kvq_testlib import assert_attention_close

pytestmark = pytest.mark.gpu


def _step(w, lens, R, seed, fused_qkv=False, spare_blocks=3):
    """GPU and oracle caches holding each request's first L - R tokens, the
    step's new rows (N*R of them; rows at negative positions are never
    stored) and the queries."""
    lens = np.asarray(lens, dtype=np.int32)
    N, H, D, Hq = len(lens), w.num_kv_heads, w.head_dim, w.num_q_heads
    bt, nblk = workloads.block_tables(lens, w.block_size, w.seed, spare_blocks=spare_blocks)
    S = nblk * w.block_size
    cache = kvq.Cache.empty(S, H, D, w.block_size)
    ocache = oracle.empty_cache(S, H, D)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(N):
        prev = int(lens[r]) - R
        if prev <= 0:
            continue
        k, v = workloads.request_kv(w, r, 0, prev)
        slots = workloads.token_slots(bt, r, prev, w.block_size)
        kvq.quantize_scatter(cache, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), err)
        oracle.quantize_scatter(workloads.bf16_bits(k).reshape(-1), H * D,
                                workloads.bf16_bits(v).reshape(-1), H * D, prev, H, D, slots,
                                ocache)
    g = workloads.generator(seed, 91)
    k_new, v_new = workloads.kv_rows(w.kv_rows, N * R, H, D, g)
    kb, vb = workloads.bf16_bits(k_new), workloads.bf16_bits(v_new)
    for r in range(N):
        for i in range(R):
            pos = int(lens[r]) - R + i
            if pos < 0:
                continue
            slot = workloads.token_slots(bt, r, pos + 1, w.block_size)[pos:pos + 1]
            t = r * R + i
            oracle.quantize_scatter(kb[t].reshape(-1), H * D, vb[t].reshape(-1), H * D, 1, H, D,
                                    slot, ocache)
    if fused_qkv:
        # the new rows as strided views of one fused projection output [T, (Hq + 2H) D]
        qkv = torch.zeros(N * R, (Hq + 2 * H) * D, dtype=torch.bfloat16)
        qkv[:, Hq * D:(Hq + H) * D] = k_new.reshape(N * R, H * D)
        qkv[:, (Hq + H) * D:] = v_new.reshape(N * R, H * D)
        qkv = qkv.cuda()
        kg, vg = qkv[:, Hq * D:(Hq + H) * D], qkv[:, (Hq + H) * D:]
    else:
        kg, vg = k_new.cuda(), v_new.cuda()
    q = torch.randn(N * R, Hq, D, generator=workloads.generator(seed, 92)).to(torch.bfloat16)
    return {"cache": cache, "ocache": ocache, "bt": bt, "lens": lens, "err": err,
            "k_new": kg, "v_new": vg, "q": q}


def _check_cache(st, R):
    """Codes and scales of every position < L of every request, bit for bit."""
    cache, oc, bt, lens = st["cache"], st["ocache"], st["bt"], st["lens"]
    bs = cache.block_size
    slots = np.concatenate([workloads.token_slots(bt, r, int(L), bs)
                            for r, L in enumerate(lens) if L > 0] or [np.zeros(0, np.int64)])
    sl = torch.from_numpy(slots).cuda()
    for nm in ("k_codes", "v_codes"):
        got = getattr(cache, nm)[sl].cpu().numpy()
        bad = int((got != oc[nm][slots]).sum())
        assert bad == 0, f"{nm}: {bad} codes differ"
    for nm in ("k_scales", "v_scales"):
        got = getattr(cache, nm)[sl].cpu().numpy()
        assert np.array_equal(got.view(np.uint32), oc[nm][slots].view(np.uint32)), nm


def _run(w, lens, R, partition_tokens=0, seed=1, fused_qkv=False):
    st = _step(w, lens, R, seed, fused_qkv=fused_qkv)
    lens = st["lens"]
    out = kvq.paged_decode_append(st["cache"], st["k_new"], st["v_new"], st["q"].cuda(),
                                  torch.from_numpy(st["bt"]).cuda(),
                                  torch.from_numpy(lens).cuda(), int(max(lens.max(), 1)),
                                  w.sm_scale, rows_per_request=R,
                                  partition_tokens=partition_tokens, err_flags=st["err"])
    torch.cuda.synchronize()
    assert int(st["err"].item()) == 0
    _check_cache(st, R)
    ref, e = oracle.paged_attention(st["ocache"], workloads.bf16_bits(st["q"]), len(lens), R,
                                    w.num_q_heads, st["bt"], lens, w.block_size, w.sm_scale)
    assert e == 0
    return out, ref


def _many_lens(n, hi, seed):
    return [int(x) for x in np.random.default_rng(seed).integers(0, hi + 1, n)]


@pytest.mark.parametrize("R,Hq,H,bs,lens,P", [
    # the load-balanced kernel stores the rows itself
    (1, 32, 8, 16, [1, 15, 16, 17, 300, 1000, 33, 0, 4096, 5], 0),
    (2, 16, 4, 16, [17, 2, 1, 640, 64, 33], 0),     # rows across a chunk edge; a negative position
    (1, 32, 8, 16, _many_lens(300, 700, 21), 0),    # weighted split, many segments per CTA
    (2, 16, 4, 32, _many_lens(150, 900, 22), 0),
    (1, 8, 4, 16, _many_lens(1024, 40, 23), 0),    # 1024 requests
    # larger pages: the new rows at the end of a page, across two pages
    (1, 32, 8, 64, [64, 65, 1, 2, 128, 129] + _many_lens(30, 3000, 24), 0),
    (2, 16, 4, 256, [256, 257, 2, 3, 512] + _many_lens(25, 2500, 25), 0),
    # other kernels, or more than two new rows: the store's own launch, then
    # the attention
    (4, 16, 8, 16, [4, 3, 100, 31, 2000], 0),       # 8 stacked rows, 4 new rows each
    (1, 32, 8, 16, [1, 15, 16, 17, 300, 1000, 33, 0, 4096, 5], 128),
    (4, 32, 8, 64, [4, 333, 520], 0),               # 16 stacked rows: the rows-on-M kernel
    (4, 32, 8, 64, [4, 333, 520], 256),             # the partitioned tensor-core kernel
])
def test_append_matches_the_oracle(R, Hq, H, bs, lens, P):
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=len(lens),
                         rows_per_request=R, num_q_heads=Hq, num_kv_heads=H, block_size=bs)
    out, ref = _run(w, lens, R, partition_tokens=P)
    assert_attention_close(out, ref, f"append R={R} Hq={Hq} H={H} bs={bs} P={P}")


def test_append_from_a_fused_qkv_view():
    """The new K and V rows as strided column blocks of one [T, (Hq + 2H) D]
    projection output."""
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=6)
    out, ref = _run(w, [40, 16, 1, 777, 2048, 3], 1, fused_qkv=True)
    assert_attention_close(out, ref, "append from a fused qkv view")


def test_append_partials_then_combine_equals_append():
    """The two-launch form (append partials, then the combine) gives the same
    bytes as the one-call form."""
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=8)
    lens = [100, 3000, 17, 1, 4000, 64, 900, 2]
    a = _step(w, lens, 1, 5)
    b = _step(w, lens, 1, 5)
    bt = torch.from_numpy(a["bt"]).cuda()
    cl = torch.from_numpy(a["lens"]).cuda()
    q = a["q"].cuda()
    maxc = int(a["lens"].max())
    out1 = kvq.paged_decode_append(a["cache"], a["k_new"], a["v_new"], q, bt, cl, maxc,
                                   w.sm_scale)
    need = kvq.paged_decode_workspace_size(len(lens), 1, w.num_q_heads, w.num_kv_heads,
                                           w.head_dim, w.block_size, maxc)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    out2 = torch.empty_like(q)
    kvq.paged_decode_append_partials(b["cache"], b["k_new"], b["v_new"], q, bt, cl, maxc,
                                     w.sm_scale, 1, 0, out2, ws)
    kvq.paged_decode_combine(b["cache"], len(lens), 1, w.num_q_heads, bt.shape[1], cl, maxc, 0,
                             out2, ws)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    for nm in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert torch.equal(getattr(a["cache"], nm), getattr(b["cache"], nm)), nm


def test_graph_capture_of_the_step():
    """The step (store + attention + combine) captured in a CUDA graph and
    replayed with new rows and new queries written into the captured buffers."""
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=5)
    lens = [50, 1200, 16, 3000, 7]
    st = _step(w, lens, 1, 7)
    bt = torch.from_numpy(st["bt"]).cuda()
    cl = torch.from_numpy(st["lens"]).cuda()
    q = st["q"].cuda()
    k_new = torch.zeros_like(st["k_new"])
    v_new = torch.zeros_like(st["v_new"])
    maxc = int(st["lens"].max())
    need = kvq.paged_decode_workspace_size(len(lens), 1, w.num_q_heads, w.num_kv_heads,
                                           w.head_dim, w.block_size, maxc)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        kvq.paged_decode_append(st["cache"], k_new, v_new, q, bt, cl, maxc, w.sm_scale,
                                out=out, workspace=ws, err_flags=st["err"], stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            kvq.paged_decode_append(st["cache"], k_new, v_new, q, bt, cl, maxc, w.sm_scale,
                                    out=out, workspace=ws, err_flags=st["err"], stream=s)
    torch.cuda.synchronize()
    k_new.copy_(st["k_new"])
    v_new.copy_(st["v_new"])
    out.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert int(st["err"].item()) == 0
    _check_cache(st, 1)
    ref, e = oracle.paged_attention(st["ocache"], workloads.bf16_bits(st["q"]), len(lens), 1,
                                    w.num_q_heads, st["bt"], st["lens"], w.block_size,
                                    w.sm_scale)
    assert e == 0
    assert_attention_close(out, ref, "graph replay of the step")


@pytest.mark.parametrize("P", [0, 128])
def test_append_to_a_bad_page_is_flagged_and_skipped(P):
    """A new row whose page id is out of range (too large, negative) is not
    stored -- no write lands anywhere in the cache -- and the call sets
    KVQ_ERRF_BLOCK_RANGE; the other requests' rows and outputs are those of
    the oracle.  P = 0: the load-balanced kernel stores the rows; P = 128: the
    store's own launch."""
    w = workloads.scaled(workloads.WORKLOADS["decode"], num_requests=4)
    lens = [200, 333, 1000, 64]
    st = _step(w, lens, 1, 9)
    bs = w.block_size
    bt_bad = st["bt"].copy()
    bt_bad[1, (333 - 1) // bs] = 1 << 30          # the page of request 1's new row
    bt_bad[3, (64 - 1) // bs] = -7                 # and of request 3's
    before = {nm: getattr(st["cache"], nm).clone() for nm in ("k_codes", "v_codes", "k_scales",
                                                                "v_scales")}
    lens_a = st["lens"]
    out = kvq.paged_decode_append(st["cache"], st["k_new"], st["v_new"], st["q"].cuda(),
                                  torch.from_numpy(bt_bad).cuda(), torch.from_numpy(lens_a).cuda(),
                                  int(lens_a.max()), w.sm_scale, partition_tokens=P,
                                  err_flags=st["err"])
    torch.cuda.synchronize()
    assert int(st["err"].item()) & kvq.ERRF_BLOCK_RANGE
    # only requests 0 and 2 stored their rows: every other slot is unchanged
    bsz = st["cache"].block_size
    new_slots = [int(workloads.token_slots(st["bt"], r, int(lens_a[r]), bsz)[-1]) for r in (0, 2)]
    for nm, b in before.items():
        now = getattr(st["cache"], nm)
        changed = torch.nonzero((now != b).reshape(now.shape[0], -1).any(dim=1)).flatten().tolist()
        assert set(changed) <= set(new_slots), (nm, changed, new_slots)
    # requests 0 and 2 (pages intact) match the oracle
    ref, e = oracle.paged_attention(st["ocache"], workloads.bf16_bits(st["q"]), len(lens), 1,
                                    w.num_q_heads, st["bt"], lens_a, w.block_size, w.sm_scale)
    assert e == 0
    for r in (0, 2):
        assert_attention_close(out[r:r + 1], ref[r:r + 1], f"append, bad pages elsewhere, r={r} P={P}")
