"""Pins of the oracle's fp64 paged attention: agreement with a dense brute
force built from library routines (torch float8 decode, matmul, softmax) on
tiny inputs, closed-form special cases, invariance to where pages live, and
the causal rule for multi-row verify."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import dense


def _make(N, R, Hq, H, D, bs, lens, seed, spare=3, lognormal=True):
    lens = np.asarray(lens, dtype=np.int32)
    bt, nblk = workloads.block_tables(lens, bs, seed, spare_blocks=spare)
    S = nblk * bs
    cache = oracle.empty_cache(S, H, D)
    g = torch.Generator().manual_seed(seed)
    for r in range(N):
        L = int(lens[r])
        if L == 0:
            continue
        k = torch.randn(L, H, D, generator=g)
        v = torch.randn(L, H, D, generator=g)
        if lognormal:
            k = k * torch.exp(torch.randn(L, H, 1, generator=g))
            v = v * torch.exp(torch.randn(L, H, 1, generator=g))
        k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
        slots = workloads.token_slots(bt, r, L, bs)
        oracle.quantize_scatter(workloads.bf16_bits(k).reshape(-1), H * D,
                                workloads.bf16_bits(v).reshape(-1), H * D, L, H, D, slots, cache)
    q = torch.randn(N * R, Hq, D, generator=g).to(torch.bfloat16)
    return cache, workloads.bf16_bits(q), bt, lens


@pytest.mark.parametrize("N,R,Hq,H,bs,lens", [
    (1, 1, 32, 8, 16, [64]),            # the tiny workload's shape
    (3, 1, 8, 2, 16, [1, 17, 50]),
    (2, 4, 16, 4, 8, [4, 37]),          # verify rows, causal
    (2, 2, 6, 3, 4, [1, 9]),            # row 0 of request 0 sees nothing
])
def test_paged_oracle_equals_dense_brute_force(N, R, Hq, H, bs, lens):
    D = 128
    cache, q, bt, L = _make(N, R, Hq, H, D, bs, lens, seed=sum(lens))
    sm = 1 / np.sqrt(D)
    ours, err = oracle.paged_attention(cache, q, N, R, Hq, bt, L, bs, sm)
    ref = dense.dense_attention(cache, q, N, R, Hq, bt, L, bs, sm)
    assert err == 0
    assert np.max(np.abs(ours - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_units_form_matches_full_form():
    cache, q, bt, L = _make(3, 2, 8, 2, 128, 16, [20, 33, 7], seed=9)
    full, _ = oracle.paged_attention(cache, q, 3, 2, 8, bt, L, 16, 0.1)
    units = [(2, 1, 7), (0, 0, 0), (1, 1, 3)]
    part, _ = oracle.paged_attention_units(cache, q, 3, 2, 8, bt, L, 16, 0.1, units)
    for u, (r, i, h) in enumerate(units):
        assert np.array_equal(part[u], full[r * 2 + i, h])


def test_single_token_returns_its_value_row():
    cache, q, bt, L = _make(1, 1, 4, 1, 128, 16, [1], seed=3)
    out, _ = oracle.paged_attention(cache, q, 1, 1, 4, bt, L, 16, 0.3)
    slot = int(bt[0, 0]) * 16
    vhat = oracle.e4m3_decode(cache["v_codes"][slot, 0]) * float(cache["v_scales"][slot, 0])
    for h in range(4):
        assert np.array_equal(out[0, h], vhat)


def test_identical_keys_give_the_mean_of_values():
    cache, q, bt, L = _make(1, 1, 2, 1, 128, 16, [40], seed=4)
    slots = workloads.token_slots(bt, 0, 40, 16)
    cache["k_codes"][slots] = cache["k_codes"][slots[0]]
    cache["k_scales"][slots] = cache["k_scales"][slots[0]]
    out, _ = oracle.paged_attention(cache, q, 1, 1, 2, bt, L, 16, 0.2)
    vhat = oracle.e4m3_decode(cache["v_codes"][slots, 0]) * \
        cache["v_scales"][slots, 0].astype(np.float64)[:, None]
    assert np.allclose(out[0, 0], vhat.mean(axis=0), rtol=0, atol=1e-12)


def test_dominant_score_selects_its_value_row():
    D = 128
    cache, q, bt, L = _make(1, 1, 1, 1, D, 16, [30], seed=5)
    slots = workloads.token_slots(bt, 0, 30, 16)
    qv = torch.zeros(1, 1, D)
    qv[0, 0, 0] = 1.0
    q = workloads.bf16_bits(qv.to(torch.bfloat16))
    cache["k_codes"][slots] = 0
    cache["k_scales"][slots] = 1.0
    cache["k_codes"][slots[17], 0, 0] = 0x7E  # 448 on dim 0 of token 17
    out, _ = oracle.paged_attention(cache, q, 1, 1, 1, bt, L, 16, 1.0)
    vhat = oracle.e4m3_decode(cache["v_codes"][slots[17], 0]) * float(cache["v_scales"][slots[17], 0])
    assert np.allclose(out[0, 0], vhat, rtol=0, atol=1e-150)


def test_moving_pages_does_not_change_the_result():
    bs, H, D = 8, 2, 128
    cache, q, bt, L = _make(2, 1, 4, H, D, bs, [30, 19], seed=6, spare=10)
    out, _ = oracle.paged_attention(cache, q, 2, 1, 4, bt, L, bs, 0.1)
    # move every used block to a fresh permutation of the pool
    nblk = cache["k_codes"].shape[0] // bs
    perm = np.random.default_rng(1).permutation(nblk).astype(np.int32)
    moved = {k: np.zeros_like(v) for k, v in cache.items()}
    for b in range(nblk):
        for name in moved:
            moved[name][perm[b] * bs:(perm[b] + 1) * bs] = cache[name][b * bs:(b + 1) * bs]
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, _ = oracle.paged_attention(moved, q, 2, 1, 4, bt2, L, bs, 0.1)
    assert np.array_equal(out, out2)


def test_verify_row_equals_decode_over_its_visible_prefix():
    R, Hq, H, D, bs = 4, 8, 2, 128, 16
    cache, q, bt, L = _make(1, R, Hq, H, D, bs, [45], seed=7)
    out, _ = oracle.paged_attention(cache, q, 1, R, Hq, bt, L, bs, 0.09)
    for i in range(R):
        qi = q.reshape(R, Hq, D)[i:i + 1]
        d, _ = oracle.paged_attention(cache, qi, 1, 1, Hq, bt, np.array([45 - R + 1 + i], np.int32),
                                      bs, 0.09)
        assert np.array_equal(out[i], d[0])


def test_gqa_heads_read_their_own_kv_head():
    Hq, H, D, bs = 8, 4, 128, 16
    cache, q, bt, L = _make(1, 1, Hq, H, D, bs, [25], seed=8)
    out, _ = oracle.paged_attention(cache, q, 1, 1, Hq, bt, L, bs, 0.1)
    changed = {k: v.copy() for k, v in cache.items()}
    changed["v_codes"][:, 2] = 0x38  # perturb KV head 2 only (every code -> 1.0)
    out2, _ = oracle.paged_attention(changed, q, 1, 1, Hq, bt, L, bs, 0.1)
    diff = np.abs(out2 - out).max(axis=-1)[0]
    assert np.all(diff[[4, 5]] > 0) and np.all(diff[[0, 1, 2, 3, 6, 7]] == 0)


def test_empty_context_and_bad_ids_are_reported():
    cache, q, bt, L = _make(2, 1, 2, 1, 128, 16, [0, 5], seed=10)
    out, err = oracle.paged_attention(cache, q, 2, 1, 2, bt, L, 16, 0.1)
    assert err == 0 and np.all(out[0] == 0) and np.any(out[1] != 0)
    bad = bt.copy()
    bad[1, 0] = 10 ** 6
    out, err = oracle.paged_attention(cache, q, 2, 1, 2, bad, L, 16, 0.1)
    assert err == oracle.ERR_BLOCK_RANGE and np.all(out[1] == 0)
    out, err = oracle.paged_attention(cache, q, 2, 1, 2, bt, np.array([0, 10 ** 6], np.int32), 16, 0.1)
    assert err & oracle.ERR_CONTEXT_RANGE
