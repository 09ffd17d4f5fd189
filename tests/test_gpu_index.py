"""kvq_index_quantize_scatter / kvq_index_dequant_rows on the GPU against the
oracle (ROCm/ATOM PR #2655, PR description, index-key bullet: index keys as
FP8 plus an FP32 scale for each row, or MXFP4 -- two E2M1 codes per byte and
an E8M0 exponent for every 32 dims, large enough that no element overflows): codes, scales and
exponents bit-exact, dequantised rows exact, on random rows and on rows built
to sit on every rounding decision."""
import numpy as np
import pytest
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import oracle

pytestmark = pytest.mark.gpu

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _rows(n, seed):
    """bf16 rows [n, 128]: N(0,1) times a log-normal magnitude per 32-dim group,
    plus rows built for the rounding decisions."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, 4, 32, generator=g) * torch.exp(torch.randn(n, 4, 1, generator=g) * 4)
    x = x.reshape(n, 128)
    special = []
    for X in (-30, -4, 0, 3, 60):
        s = 2.0 ** X
        # every E2M1 midpoint, both signs, next to a group max of exactly 6 * 2^X
        mids = [(E2M1[i] + E2M1[i + 1]) / 2 for i in range(7)]
        grp = [6.0] + mids + [-m for m in mids] + E2M1[1:] + [-0.0] * 2
        grp = (grp + [0.25] * 32)[:32]
        special.append(torch.tensor(grp * 4) * s)
    # group amax with mantissa exactly 1.5, and the next bf16 above it
    for a in (1.5, 1.5078125, 1.0, 1.9921875):
        row = torch.full((128,), 0.3)
        row[::32] = a * 2.0 ** 7
        special.append(row)
    special.append(torch.zeros(128))
    special.append(-torch.zeros(128))
    tiny = torch.full((128,), 2.0 ** -130)                 # bf16 subnormals
    tiny[1::2] *= -3
    special.append(tiny)
    big = torch.full((128,), 3.0e38)                       # near the bf16 maximum
    big[1::3] = -1.0e38
    special.append(big)
    x = torch.cat([x, torch.stack(special)])
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("fmt", [kvq.INDEX_MXFP4, kvq.INDEX_FP8])
def test_codes_bit_exact_through_scatter(fmt):
    x = _rows(700, 1)
    T = x.shape[0]
    S = T + 64
    g = torch.Generator().manual_seed(2)
    slots = torch.randperm(S, generator=g)[:T].to(torch.int64)
    slots[5] = -1                                           # padding: skipped
    slots[9] = S + 3                                        # out of range: flagged, skipped
    # a strided view: rows live in a wider buffer
    wide = torch.zeros(T, 192, dtype=torch.bfloat16)
    wide[:, 32:160] = x
    xv = wide.cuda()[:, 32:160]
    cache = kvq.IndexCache.empty(S, fmt)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.index_quantize_scatter(cache, xv, slots.cuda(), err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvq.ERRF_SLOT_RANGE
    xb = _bits(x)
    ok = [t for t in range(T) if 0 <= slots[t] < S]
    sl = slots[ok].numpy()
    if fmt == kvq.INDEX_MXFP4:
        want_c, want_e = oracle.mxfp4_quantize_rows(xb[ok])
        got_c = cache.codes.cpu().numpy()[sl]
        got_e = cache.exponents.cpu().numpy()[sl]
        assert np.array_equal(got_e, want_e)
        assert np.array_equal(got_c, want_c)
    else:
        want_c, want_s = oracle.quantize_rows(xb[ok])
        got_c = cache.codes.cpu().numpy()[sl]
        got_s = cache.scales.cpu().numpy()[sl]
        assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32))
        assert np.array_equal(got_c, want_c)
    # slots nobody wrote stay zero
    untouched = np.setdiff1d(np.arange(S), sl)
    assert not cache.codes.cpu().numpy()[untouched].any()


@pytest.mark.parametrize("fmt", [kvq.INDEX_MXFP4, kvq.INDEX_FP8])
def test_dequant_rows_exact(fmt):
    x = _rows(300, 3)
    T = x.shape[0]
    cache = kvq.IndexCache.empty(T, fmt)
    ids = torch.arange(T, dtype=torch.int64)
    kvq.index_quantize_scatter(cache, x.cuda(), ids.cuda())
    probe = torch.cat([ids, torch.tensor([-4, T + 9], dtype=torch.int64)])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out32 = kvq.index_dequant_rows(cache, probe.cuda(), torch.float32, err).cpu().numpy()
    out16 = kvq.index_dequant_rows(cache, probe.cuda(), torch.bfloat16).cpu()
    torch.cuda.synchronize()
    assert int(err.item()) == kvq.ERRF_SLOT_RANGE
    if fmt == kvq.INDEX_MXFP4:
        want = oracle.mxfp4_dequant_rows(cache.codes.cpu().numpy(), cache.exponents.cpu().numpy())
    else:
        c = cache.codes.cpu().numpy()[:, None, :]
        s = cache.scales.cpu().numpy()[:, None]
        want = oracle.dequant_rows(c, s, np.arange(T))[:, 0, :]
    assert np.array_equal(out32[:T].view(np.uint32), want.view(np.uint32))
    assert not out32[T:].any()
    want16 = torch.from_numpy(want).to(torch.bfloat16)
    assert torch.equal(out16[:T].view(torch.int16), want16.view(torch.int16))


def test_mxfp4_never_clips_on_device():
    """Every group's largest element decodes to within half a grid step of its
    value: the exponent leaves it inside E2M1's range."""
    x = _rows(200, 5)[:200]
    cache = kvq.IndexCache.empty(200, kvq.INDEX_MXFP4)
    ids = torch.arange(200, dtype=torch.int64, device="cuda")
    kvq.index_quantize_scatter(cache, x.cuda(), ids)
    deq = kvq.index_dequant_rows(cache, ids).cpu().double().reshape(200, 4, 32)
    xf = x.double().reshape(200, 4, 32)
    X = cache.exponents.cpu().double() - 127
    amax = xf.abs().amax(dim=2)
    assert bool((amax <= 6.0 * 2.0 ** X).all())
    i = xf.abs().argmax(dim=2, keepdim=True)
    err = (deq.gather(2, i) - xf.gather(2, i)).abs().squeeze(2)
    assert bool((err <= 2.0 ** X).all())           # half the largest spacing (2 * 2^X)
