"""kvq_index_scores on the GPU against the oracle (ATOM PR #2655, PR
description: the decode-time scorer multiplies a request's query rows x
index heads against each cached index key in one product, loading each key
once, and clips each head's dot at zero before adding the heads).

Scores must lie within the bound the kernel's arithmetic gives (f16 products
of exactly converted keys and power-of-two-scaled queries, fp32 accumulation;
MXFP4 groups more than 2^23 below the token's largest group are not exact in
f16):
    |gpu - exact| <= 1e-5 * sum_h sum_d |q_hd * k_d| + 2^-22 * max_d |k_d| * sum_h sum_d |q_hd|
and the -inf pattern (tokens a row does not see) must match exactly."""
import numpy as np
import pytest
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _exact_keys(fmt, codes, scales, exps):
    """Dequantised keys in double (every value exact)."""
    if fmt == kvq.INDEX_FP8:
        return oracle.e4m3_decode(codes).astype(np.float64) * scales.astype(np.float64)[:, None]
    lo = oracle.e2m1_decode(codes & 0xF)
    hi = oracle.e2m1_decode(codes >> 4)
    v = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], 128).astype(np.float64)
    X = exps.astype(np.float64) - 127.0
    return v * np.repeat(np.exp2(X), 32, axis=1)


def _upload(fmt, codes, scales, exps):
    S = codes.shape[0]
    cache = kvq.IndexCache.empty(S, fmt)
    cache.codes.copy_(torch.from_numpy(codes))
    if fmt == kvq.INDEX_FP8:
        cache.scales.copy_(torch.from_numpy(scales))
    else:
        cache.exponents.copy_(torch.from_numpy(exps))
    return cache


def _check(fmt, codes, scales, exps, bt, bs, lens, q, max_len, got, requests=None):
    """Compare GPU scores `got` [N*R, max_len] with the oracle on `requests`."""
    N, R, H, _ = q.shape
    requests = range(N) if requests is None else requests
    qf = q.double().numpy()
    qb = _bits(q)
    for r in requests:
        sub_bt = bt[r:r + 1]
        want, err = oracle.index_scores(fmt, codes, scales, exps, sub_bt, bs, lens[r:r + 1], R, H,
                                        qb[r].reshape(R * H, 128), max_len)
        assert err == 0
        L = int(lens[r])
        pos = np.arange(L)
        sl = bt[r, pos // bs].astype(np.int64) * bs + pos % bs
        k = _exact_keys(fmt, codes[sl], None if scales is None else scales[sl],
                        None if exps is None else exps[sl])                # [L, 128]
        absdot = np.einsum("ihd,td->it", np.abs(qf[r]), np.abs(k))       # [R, L]
        bound = 1e-5 * absdot + 2.0 ** -22 * np.abs(k).max(axis=1)[None, :] * \
            np.abs(qf[r]).sum(axis=(1, 2))[:, None]
        for i in range(R):
            g = got[r * R + i]
            vis = max(L - R + 1 + i, 0)
            assert np.all(np.isneginf(g[vis:])), (r, i)
            assert np.all(np.isneginf(want[0 + i][vis:]))
            d = np.abs(g[:vis].astype(np.float64) - want[i][:vis])
            assert np.all(d <= bound[i, :vis] + 1e-30), \
                (r, i, float(d.max()), int(np.argmax(d - bound[i, :vis])))


def _realistic_keys(fmt, S, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(S, 4, 32, generator=g) * torch.exp(2.0 * torch.randn(S, 4, 1, generator=g))
    xb = _bits(x.reshape(S, 128).to(torch.bfloat16))
    if fmt == kvq.INDEX_FP8:
        codes, scales = oracle.quantize_rows(xb)
        return codes, scales, None
    codes, exps = oracle.mxfp4_quantize_rows(xb)
    return codes, None, exps


SHAPES = [(1, 1, 16), (4, 4, 64), (2, 8, 16), (16, 1, 128), (8, 2, 32), (1, 8, 16), (3, 4, 16),
          (5, 2, 64)]


@pytest.mark.parametrize("fmt", [kvq.INDEX_MXFP4, kvq.INDEX_FP8])
@pytest.mark.parametrize("R,H,bs", SHAPES)
def test_scores_match_oracle(fmt, R, H, bs):
    """Ragged contexts spanning several 512-token CTAs and a tail that is not
    a multiple of the 16-token tile; an empty request; a request shorter than
    its row count."""
    lens = np.array([1300, 17, 0, 600, 513, 2], dtype=np.int32)
    max_len = 1400
    bt, nblk = workloads.block_tables(lens, bs, seed=R * 10 + H, spare_blocks=2)
    codes, scales, exps = _realistic_keys(fmt, nblk * bs, R * 100 + H + fmt)
    q = workloads.index_queries(len(lens), R, H, seed=R + 7 * H)
    cache = _upload(fmt, codes, scales, exps)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = kvq.index_scores(cache, bs, q.cuda(), torch.from_numpy(bt).cuda(),
                           torch.from_numpy(lens).cuda(), max_len, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _check(fmt, codes, scales, exps, bt, bs, lens, q, max_len, got.cpu().numpy())


def test_mxfp4_groups_far_below_the_largest():
    """MXFP4 tokens whose groups sit 0 .. 60 binary orders below the token's
    largest group, with the queries weighting the small groups 2^20 times
    more: the f16 renormalisation is exact down to 23 orders (normal and
    subnormal f16 factors) and the rest stays inside the bound."""
    S, bs = 2048, 16
    g = workloads.generator(11, 1)
    codes = torch.randint(0, 256, (S, 64), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    top = torch.randint(120, 135, (S,), generator=g).numpy()
    deltas = np.array([0, -1, -9, -14, -15, -16, -20, -23, -24, -25, -30, -60])
    pick = torch.randint(0, len(deltas), (S, 3), generator=g).numpy()
    exps = np.empty((S, 4), dtype=np.int64)
    exps[:, 0] = top
    exps[:, 1:] = np.maximum(top[:, None] + deltas[pick], 0)
    exps = exps.astype(np.uint8)
    lens = np.array([S], dtype=np.int32)
    bt, _ = workloads.block_tables(lens, bs, seed=12)
    q = workloads.index_queries(1, 4, 4, seed=13).float()
    q[..., 32:] *= 2.0 ** 20
    q = q.to(torch.bfloat16)
    cache = _upload(kvq.INDEX_MXFP4, codes, None, exps)
    got = kvq.index_scores(cache, bs, q.cuda(), torch.from_numpy(bt).cuda(),
                           torch.from_numpy(lens).cuda(), S)
    _check(kvq.INDEX_MXFP4, codes, None, exps, bt, bs, lens, q, S, got.cpu().numpy())


def test_degenerate_shapes():
    """max_context_len 1 and a tail of one token; a request with L = R - 1
    (row 0 sees nothing); queries of zeros (scores 0, not -inf)."""
    bs = 16
    for fmt in (kvq.INDEX_FP8, kvq.INDEX_MXFP4):
        codes, scales, exps = _realistic_keys(fmt, 64, 21 + fmt)
        cache = _upload(fmt, codes, scales, exps)
        bt = np.array([[0, 1, 2, 3]], dtype=np.int32)
        for L, R, max_len in ((1, 1, 1), (3, 4, 17), (49, 2, 64), (64, 16, 64)):
            lens = np.array([L], dtype=np.int32)
            q = workloads.index_queries(1, R, 1, seed=L)
            got = kvq.index_scores(cache, bs, q.cuda(), torch.from_numpy(bt).cuda(),
                                   torch.from_numpy(lens).cuda(), max_len).cpu().numpy()
            _check(fmt, codes, scales, exps, bt, bs, lens, q, max_len, got)
        z = torch.zeros(1, 2, 4, 128, dtype=torch.bfloat16)
        got = kvq.index_scores(cache, bs, z.cuda(), torch.from_numpy(bt).cuda(),
                               torch.tensor([40], dtype=torch.int32).cuda(), 64).cpu().numpy()
        assert np.all(got[0, :39] == 0.0) and np.all(np.isneginf(got[0, 39:]))
        assert np.all(got[1, :40] == 0.0) and np.all(np.isneginf(got[1, 40:]))


def test_bad_block_ids_and_lengths_are_flagged_not_faulted():
    bs = 16
    codes, scales, exps = _realistic_keys(kvq.INDEX_MXFP4, 64, 31)
    cache = _upload(kvq.INDEX_MXFP4, codes, scales, exps)
    q = workloads.index_queries(3, 2, 4, seed=32).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = torch.tensor([[0, 1, 4, 2], [3, -1, 0, 0], [0, 1, 2, 3]], dtype=torch.int32)
    lens = torch.tensor([40, 20, 10], dtype=torch.int32)
    out = kvq.index_scores(cache, bs, q, bt.cuda(), lens.cuda(), 64, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvq.ERRF_BLOCK_RANGE
    # the request with a valid table is still scored correctly
    _check(kvq.INDEX_MXFP4, codes, None, exps, bt.numpy(), bs, lens.numpy(), q.cpu(), 64,
           out.cpu().numpy(), requests=[2])
    err.zero_()
    kvq.index_scores(cache, bs, q, bt.cuda(), torch.tensor([10, 10, 65], dtype=torch.int32).cuda(),
                     64, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvq.ERRF_CONTEXT_RANGE


@pytest.mark.parametrize("fmt", [kvq.INDEX_MXFP4, kvq.INDEX_FP8])
def test_full_size_sampled(fmt):
    """The index-scoring workload at full size (64 requests x 4 rows x 4
    heads, context 32,768, block size 64), as the benchmark launches it; the
    oracle checks two sampled requests, and every other row the -inf tail
    and the absence of NaN."""
    w = workloads.INDEX_SCORES
    lens = np.full(w.num_requests, w.context, dtype=np.int32)
    bt, nblk = workloads.block_tables(lens, w.block_size, w.seed)
    codes, scales, exps = workloads.index_key_codes(fmt, nblk * w.block_size, w.seed)
    q = workloads.index_queries(w.num_requests, w.rows, w.heads, w.seed)
    cache = _upload(fmt, codes, scales, exps)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = kvq.index_scores(cache, w.block_size, q.cuda(), torch.from_numpy(bt).cuda(),
                           torch.from_numpy(lens).cuda(), w.context, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g = got.cpu().numpy()
    assert not np.isnan(g).any()
    R = w.rows
    for i in range(R):
        vis = w.context - R + 1 + i
        assert np.all(np.isneginf(g[i::R, vis:]))
        assert np.all(g[i::R, :vis] >= 0.0)
    _check(fmt, codes, scales, exps, bt, w.block_size, lens, q, w.context, g, requests=[0, 37])
