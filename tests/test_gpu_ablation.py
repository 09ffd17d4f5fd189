"""The codec ablation on the GPU (sgl-project/sglang-jax #1776 "feat(dsa):
implement fp8 KV cache (e4m3) with a bf16 indexer cache", design points and
accuracy tests): caches of O(1) values cast to e4m3 or e5m2 with no scale,
against this library's per-row-scaled e4m3 cache and the bf16 rows.

  * the unscaled store is bit-exact against the oracle's codecs (and writes
    scales of 1);
  * attention over each cache (the same rows-on-M kernel for both formats)
    matches fp64 attention over the same dequantised codes;
  * the errors against the bf16 cache keep the page's order: e5m2 about twice
    e4m3 (the oracle's pinned band 1.8-2.25), the per-row scale no worse than
    the unscaled e4m3 cast."""
import numpy as np
import pytest
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import oracle
import workloads
from oracle import ablation
from kvq_testlib import assert_attention_close

pytestmark = pytest.mark.gpu

D = 128


def _special_rows():
    """Values at the formats' edges: beyond both saturations, at and around the
    e4m3 / e5m2 maxima, subnormals of both, signed zeros, tiny negatives."""
    vals = [0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, -2.0 ** -10, 2.0 ** -9, 2.0 ** -17, -2.0 ** -16,
            440.0, 448.0, 460.0, -500.0, 57344.0, -60000.0, 1e6, -3e38, 0.3, -1.7, 17.0, 2.5e-3,
            -6.1e-5, 6.103515625e-05, 1.52587890625e-05]
    x = torch.tensor(vals * 8, dtype=torch.float32)[:D * (len(vals) * 8 // D)]
    return x.reshape(-1, 1, D).expand(-1, 4, D).to(torch.bfloat16).contiguous()


@pytest.mark.parametrize("fmt", [kvq.CODES_E4M3, kvq.CODES_E5M2])
def test_unscaled_store_is_bit_exact(fmt):
    g = workloads.generator(41, fmt)
    H = 4
    rows = torch.cat([workloads.unit_rms_rows(300, H, D, g) * 37.0, _special_rows()])
    T = rows.shape[0]
    k = rows
    v = (-rows).contiguous()
    cache = kvq.Cache.empty(T + 5, H, D, 16)
    slots = torch.randperm(T + 5, generator=g)[:T].to(torch.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.quantize_scatter_unscaled(cache, k.cuda(), v.cuda(), slots.cuda(), fmt, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    enc = oracle.e4m3_encode if fmt == kvq.CODES_E4M3 else oracle.e5m2_encode
    sl = slots.numpy()
    for name, x in (("k", k), ("v", v)):
        want = enc(ablation.bf16_values(workloads.bf16_bits(x)).astype(np.float32))
        got = getattr(cache, f"{name}_codes").cpu().numpy()[sl]
        bad = int((got != want).sum())
        assert bad == 0, f"{name}: {bad} codes differ"
        sc = getattr(cache, f"{name}_scales").cpu().numpy()[sl]
        assert np.all(sc == 1.0)


def _caches(H, Hq, L, bs, seed):
    g = workloads.generator(seed, 1)
    k = workloads.unit_rms_rows(L, H, D, g)
    v = workloads.unit_rms_rows(L, H, D, g)
    lens = np.array([L], dtype=np.int32)
    bt, nblk = workloads.block_tables(lens, bs, seed, spare_blocks=2)
    slots = torch.from_numpy(workloads.token_slots(bt, 0, L, bs)).cuda()
    out = {}
    for name in ("e4m3_row", "e4m3", "e5m2"):
        c = kvq.Cache.empty(nblk * bs, H, D, bs)
        if name == "e4m3_row":
            kvq.quantize_scatter(c, k.cuda(), v.cuda(), slots)
        else:
            kvq.quantize_scatter_unscaled(c, k.cuda(), v.cuda(), slots,
                                          kvq.CODES_E4M3 if name == "e4m3" else kvq.CODES_E5M2)
        out[name] = c
    torch.cuda.synchronize()
    return k, v, lens, torch.from_numpy(bt).cuda(), out


@pytest.mark.parametrize("R,L", [(1, 2048), (64, 512)])
def test_unscaled_attention_parity_and_error_order(R, L):
    H, Hq, bs = 4, 16, 64
    k, v, lens, bt, caches = _caches(H, Hq, L, bs, seed=43 + R)
    g = workloads.generator(44, R)
    q = workloads.unit_rms_rows(R, Hq, D, g)
    sm = 1.0 / np.sqrt(D)
    cl = torch.from_numpy(lens).cuda()
    kb, vb, qb = workloads.bf16_bits(k), workloads.bf16_bits(v), workloads.bf16_bits(q)
    qv = ablation.bf16_values(qb)
    exact = ablation.attention_fp64(qv, ablation.cache_values("bf16", kb),
                                    ablation.cache_values("bf16", vb), sm)
    errs = {}
    for name, cache in caches.items():
        if name == "e4m3_row":
            out = kvq.paged_decode(cache, q.cuda(), bt, cl, L, sm, rows_per_request=R)
        else:
            fmt = kvq.CODES_E4M3 if name == "e4m3" else kvq.CODES_E5M2
            out = kvq.paged_decode_codes(cache, fmt, q.cuda(), bt, cl, L, sm, rows_per_request=R)
        torch.cuda.synchronize()
        # parity: the same arithmetic in fp64 over the same dequantised codes
        ref = ablation.attention_fp64(qv, ablation.cache_values(name, kb),
                                      ablation.cache_values(name, vb), sm)
        assert_attention_close(out, ref, f"{name} R={R} L={L}")
        errs[name] = ablation.rel_l2(out.float().cpu().numpy().astype(np.float64), exact)
    print(f"R={R} L={L}: rel-L2 against the bf16 cache {errs}, "
          f"e5m2 / e4m3 = {errs['e5m2'] / errs['e4m3']:.3f}")
    assert 1.8 <= errs["e5m2"] / errs["e4m3"] <= 2.25, errs
    assert errs["e4m3_row"] <= 1.1 * errs["e4m3"], errs
