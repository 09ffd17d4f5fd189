"""Chunked-prefill attention over the FP8 paged cache on the GPU against the
fp64 oracle (sgl-project/sglang-jax #1776 "feat(dsa): implement fp8 KV cache
(e4m3) with a bf16 indexer cache", Modifications: a prefill chunk attends over
the cached blocks, causally, and its probabilities are never rounded to fp8).

A chunk of R new tokens of a request whose cache holds L tokens (the chunk's
own included) is kvq_paged_decode with rows_per_request = R: row i sees the
first L - R + 1 + i tokens.  With G query heads per KV head that is R * G
stacked rows per KV head, run by the rows-on-M tensor-core kernel in tiles of
128 rows; chunks of 256 to 2,048 tokens are checked, on pure prefill (L = R)
and on chunks appended to a cached context, with ragged lengths."""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import oracle
import workloads
from kvq_testlib import assert_attention_close, build_custom, build_paged

pytestmark = pytest.mark.gpu


def _oracle_by_head(built, q_bits, R, G, H, sm_scale, lens):
    """fp64 oracle output [N*R, H*G, D], one KV head per host thread (each
    thread gets the oracle cache's planes of its head)."""
    oc = built["ocache"]
    N = len(lens)
    D = 128

    def one(h):
        sub = {k: np.ascontiguousarray(oc[k][:, h:h + 1]) for k in oc}
        qh = np.ascontiguousarray(q_bits[:, h * G:(h + 1) * G])
        ref, err = oracle.paged_attention(sub, qh, N, R, G, built["bt"], lens,
                                          built["cache"].block_size, sm_scale)
        assert err == 0
        return h, ref

    out = np.zeros((N * R, H * G, D))
    workers = max(1, min(H, len(os.sched_getaffinity(0))))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for h, ref in ex.map(one, range(H)):
            out[:, h * G:(h + 1) * G] = ref
    return out


@pytest.mark.parametrize("R,lens,H,G,bs", [
    (256, [256], 8, 4, 64),                 # pure prefill of a 256-token prompt
    (256, [1000, 256, 700], 8, 4, 16),      # chunks after cached contexts, 16-token pages
    (512, [2048, 777], 4, 4, 64),           # 2048 rows per KV head, ragged context
    (1000, [1500], 4, 8, 32),               # a chunk that is not a multiple of the tile
    (2048, [2048, 4096], 4, 4, 64),         # 2,048-token chunks: 8,192 rows per KV head
])
def test_prefill_chunks_match_the_oracle(R, lens, H, G, bs):
    w = workloads.scaled(workloads.WORKLOADS["prefill"], num_requests=len(lens),
                         rows_per_request=R, num_q_heads=H * G, num_kv_heads=H, block_size=bs)
    lens = np.array(lens, dtype=np.int32)
    built = build_paged(w, lens)
    g = workloads.generator(11, R, len(lens))
    q = torch.randn(len(lens) * R, H * G, 128, generator=g).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = torch.from_numpy(built["bt"]).cuda()
    cl = torch.from_numpy(lens).cuda()
    out = kvq.paged_decode(built["cache"], q.cuda(), bt, cl, int(lens.max()), w.sm_scale,
                           rows_per_request=R, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = _oracle_by_head(built, workloads.bf16_bits(q), R, G, H, w.sm_scale, lens)
    assert_attention_close(out, ref, f"prefill R={R} lens={list(lens)} H={H} G={G} bs={bs}")


def test_prefill_twice_in_a_row_with_a_shared_workspace():
    """Two calls sharing one workspace: the per-unit tickets the first call
    leaves at zero serve the second (the workspace is zeroed only once)."""
    w = workloads.scaled(workloads.WORKLOADS["prefill"], num_requests=2, rows_per_request=384,
                         num_q_heads=16, num_kv_heads=4, block_size=64)
    lens = np.array([3000, 384], dtype=np.int32)
    built = build_paged(w, lens)
    bt = torch.from_numpy(built["bt"]).cuda()
    cl = torch.from_numpy(lens).cuda()
    need = kvq.paged_decode_workspace_size(2, 384, 16, 4, 128, 64, 3000, 0)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for seed in (1, 2):
        g = workloads.generator(12, seed)
        q = torch.randn(2 * 384, 16, 128, generator=g).to(torch.bfloat16)
        out = kvq.paged_decode(built["cache"], q.cuda(), bt, cl, 3000, w.sm_scale,
                               rows_per_request=384, workspace=ws)
        torch.cuda.synchronize()
        ref = _oracle_by_head(built, workloads.bf16_bits(q), 384, 4, 4, w.sm_scale, lens)
        assert_attention_close(out, ref, f"prefill shared workspace, call {seed}")


def test_prefill_climbing_scores_move_references_mid_chunk():
    """Tiles of 128 rows store P'' 16 tokens at a time and move a row's
    references before a group's exponentials, rescaling the P'' already in
    tensor memory.  Keys that grow along the context in the query's direction
    make every row's score climb by about 3 (log2 units) per 16 tokens, so
    references move inside most chunks; value magnitudes grow too (the value
    bound moves)."""
    R, H, G, D = 256, 4, 4, 128
    w = workloads.scaled(workloads.WORKLOADS["prefill"], num_requests=2, rows_per_request=R,
                         num_q_heads=H * G, num_kv_heads=H, block_size=64)
    g = workloads.generator(37, 2)
    u = torch.randn(H, D, generator=g)
    kvs = []
    for L in (1536, 700):
        t = torch.arange(L, dtype=torch.float32)[:, None, None]
        k = 0.012 * t * u[None] + 0.3 * torch.randn(L, H, D, generator=g)
        v = torch.randn(L, H, D, generator=g) * (1.0 + t / 300.0)
        kvs.append((k.to(torch.bfloat16), v.to(torch.bfloat16)))
    built = build_custom(w, kvs)
    lens = built["lens"]
    q = (u.repeat_interleave(G, dim=0)[None].expand(2 * R, H * G, D) +
         0.1 * torch.randn(2 * R, H * G, D, generator=g)).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvq.paged_decode(built["cache"], q.cuda(), torch.from_numpy(built["bt"]).cuda(),
                           torch.from_numpy(lens).cuda(), int(lens.max()), w.sm_scale,
                           rows_per_request=R, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = _oracle_by_head(built, workloads.bf16_bits(q), R, G, H, w.sm_scale, lens)
    assert_attention_close(out, ref, "prefill, climbing scores")
