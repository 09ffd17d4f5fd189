"""Pins for the oracle's unscaled-cache ablation (sgl-project/sglang-jax #1776,
design points and accuracy tests: e4m3 or e5m2 cast with no scale; about 6 %
against 12.5 % worst-case relative error; attention error about twice as large
for e5m2), checked against PyTorch's own float8 dtypes, brute force over the
code grid, the formats' closed-form error bounds, the power-of-two argument the
page makes, and the C oracle's paged attention."""
import numpy as np
import pytest
import torch

import oracle
import oracle.ablation as A
import workloads


def test_e5m2_decode_matches_torch_float8_e5m2():
    """All 256 codes against torch's float8_e5m2 (an independent library
    decode), plus values worked by hand from the format."""
    got = oracle.e5m2_decode(np.arange(256))
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e5m2) \
        .to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # 1.0 = exponent 15, mantissa 0; 57344 = 1.75 * 2^15; 2^-16 the smallest
    # subnormal, 2^-14 the smallest normal; 0x7C infinity
    assert got[0x3C] == 1.0 and got[0x7B] == 57344.0 and got[0x01] == 2.0 ** -16
    assert got[0x04] == 2.0 ** -14 and np.isposinf(got[0x7C]) and got[0xBC] == -1.0


def test_e5m2_encode_brute_force_and_torch():
    """Nearest finite e5m2 value with ties to the even mantissa, by search over
    the whole grid; and torch's float -> float8_e5m2 cast inside the range."""
    grid = oracle.e5m2_decode(np.arange(0x7C))
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(3000) * np.exp(rng.uniform(-12, 10, 3000)),
                        (grid[:-1] + grid[1:]) / 2,            # every midpoint
                        -(grid[:-1] + grid[1:]) / 2, grid, [0.0, -0.0, 60000.0, -1e30]])
    x = x.astype(np.float32)
    got = oracle.e5m2_encode(x)
    for v, c in zip(x.astype(np.float64), got):
        a = min(abs(v), 57344.0)
        d = np.abs(grid - a)
        cand = np.flatnonzero(d == d.min())
        want = cand[0] if len(cand) == 1 else [k for k in cand if k % 2 == 0][0]
        assert c == (want | (0x80 if np.signbit(v) else 0)), (v, c)
    inr = np.abs(x) < 57344.0
    tref = torch.from_numpy(x[inr]).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(got[inr], tref)


@pytest.mark.parametrize("fmt,m,lo,hi", [("e4m3", 3, 2.0 ** -6, 448.0),
                                          ("e5m2", 2, 2.0 ** -14, 57344.0)])
def test_worst_case_relative_error_is_half_an_ulp(fmt, m, lo, hi):
    """Over the normal range the rounding error is at most 2^-(m+1) of the
    value (6.25 % for e4m3, 12.5 % for e5m2 -- the page's ~6 % and ~12.5 %),
    and just above a power of two it comes within 1/(1 + 2^-(m+1)) of it."""
    x = np.exp(np.linspace(np.log(lo), np.log(hi) - 1e-9, 400001)).astype(np.float32)
    enc, dec = (oracle.e4m3_encode, oracle.e4m3_decode) if fmt == "e4m3" else \
        (oracle.e5m2_encode, oracle.e5m2_decode)
    xd = x.astype(np.float64)
    rel = np.abs(dec(enc(x)) - xd) / xd
    u = 2.0 ** -(m + 1)
    assert rel.max() <= u
    assert rel.max() >= 0.999 * u / (1 + u)
    # the tight maximum, u / (1 + u), sits at 1 + u of a binade: 1/17 and 1/9
    assert rel.max() <= u / (1 + u) + 1e-7


def test_e5m2_bound_is_the_pages_number(golden_dir):
    """The page's worst-case figure for e5m2 (golden fixture, about 12.5 %) is
    the half-ulp bound 2^-3 of a 2-bit mantissa."""
    import json
    import os
    facts = json.load(open(os.path.join(golden_dir, "pages_facts.json")))
    w = facts["worst_case_rel_error"]
    assert abs(w["e5m2"] - 2.0 ** -3) <= w["approx_rel"] * w["e5m2"]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_power_of_two_rescale_changes_nothing(fmt):
    """fp8 precision is relative: inside the normal range the cast of x * 2^k
    is exactly 2^k times the cast of x."""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(20000) * 2.0).astype(np.float32)
    x = x[np.abs(x) >= 2.0 ** -2]        # x * 2^-3 stays clear of e4m3's subnormals (2^-6)
    base = A.cache_values(fmt, oracle.float_to_bf16_bits(x))
    for k in (-3, -1, 1, 4):
        xs = (x.astype(np.float64) * 2.0 ** k).astype(np.float32)
        got = A.cache_values(fmt, oracle.float_to_bf16_bits(xs))
        assert np.array_equal(got, base * 2.0 ** k)


def test_fp64_attention_matches_the_paged_oracle():
    """The ablation's attention on the per-row-scaled cache's values equals the
    C oracle's paged attention on the same cache (two independent forms)."""
    g = workloads.generator(31, 0)
    H, Hq, D, L, R, bs = 2, 8, 128, 70, 3, 16
    k = workloads.unit_rms_rows(L, H, D, g)
    v = workloads.unit_rms_rows(L, H, D, g)
    q = torch.randn(R, Hq, D, generator=g).to(torch.bfloat16)
    kb, vb, qb = (workloads.bf16_bits(t) for t in (k, v, q))
    K, V = A.cache_values("e4m3_row", kb), A.cache_values("e4m3_row", vb)
    got = A.attention_fp64(A.bf16_values(qb), K, V, D ** -0.5)
    oc = oracle.empty_cache(L + 10, H, D)
    bt = np.arange((L + bs - 1) // bs, dtype=np.int32)[None, :]
    slots = np.arange(L, dtype=np.int64)
    oracle.quantize_scatter(kb.reshape(-1), H * D, vb.reshape(-1), H * D, L, H, D, slots, oc)
    ref, err = oracle.paged_attention(oc, qb, 1, R, Hq, bt, np.array([L], np.int32), bs,
                                      D ** -0.5)
    assert err == 0
    assert np.allclose(got, ref.reshape(R, Hq, D), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("R,L", [(1, 2048), (64, 512)])
def test_e5m2_error_is_about_twice_e4m3(R, L):
    """On unit-RMS rows the attention error against the bf16 cache grows by
    about the extra mantissa bit, e5m2 against e4m3 (the page measured 1.87 to
    2.10), for a decode row and a prefill chunk."""
    g = workloads.generator(32, R)
    H, Hq, D = 2, 8, 128
    k = workloads.bf16_bits(workloads.unit_rms_rows(L, H, D, g))
    v = workloads.bf16_bits(workloads.unit_rms_rows(L, H, D, g))
    q = A.bf16_values(workloads.bf16_bits(torch.randn(R, Hq, D, generator=g)
                                          .to(torch.bfloat16)))
    ref = A.attention_fp64(q, A.cache_values("bf16", k), A.cache_values("bf16", v), D ** -0.5)
    err = {f: A.rel_l2(A.attention_fp64(q, A.cache_values(f, k), A.cache_values(f, v),
                                        D ** -0.5), ref)
           for f in ("e4m3", "e5m2", "e4m3_row")}
    # the page measured 1.87-2.10 on its model; seeds of this recipe give 1.95-2.11
    assert 1.8 <= err["e5m2"] / err["e4m3"] <= 2.25, err
    assert err["e4m3"] < 0.1 and err["e4m3_row"] < 0.1


def test_fp64_attention_matches_torch_sdpa_on_a_prefill_chunk():
    """A prefill chunk (64 new rows over a 200-token context, GQA 4) against
    torch's scaled_dot_product_attention with the causal-with-offset mask
    written out (a library routine; float64 on the CPU)."""
    g = workloads.generator(33, 0)
    H, Hq, D, L, R = 2, 8, 128, 200, 64
    K = torch.randn(L, H, D, generator=g, dtype=torch.float64)
    V = torch.randn(L, H, D, generator=g, dtype=torch.float64)
    q = torch.randn(R, Hq, D, generator=g, dtype=torch.float64)
    got = A.attention_fp64(q.numpy(), K.numpy(), V.numpy(), 0.1)
    mask = torch.arange(L)[None, :] <= (L - R + torch.arange(R))[:, None]      # [R, L]
    Kx = K.repeat_interleave(Hq // H, dim=1).permute(1, 0, 2)                  # [Hq, L, D]
    Vx = V.repeat_interleave(Hq // H, dim=1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2), Kx, Vx, attn_mask=mask, scale=0.1).permute(1, 0, 2)
    assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-13)
