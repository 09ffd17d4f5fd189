"""kvq_quantize_scatter and kvq_dequant_rows on the GPU against the oracle:
codes and scales bit-exact (FreeToken PR #354 review: only a codes-level check
catches store bugs), strided K/V pitches, the fused-qkv store workload at full
size, CUDA-graph capture, padding and out-of-range slot ids, guard bands."""
import numpy as np
import pytest
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import oracle
import workloads
from kvq_testlib import assert_cache_equal

pytestmark = pytest.mark.gpu

B = workloads.bf16_bits


def _flat(x: torch.Tensor) -> np.ndarray:
    """The elements of a strided [T, ...] view as a flat uint16 buffer laid out
    with the view's own token pitch (its first element at index 0)."""
    T = x.shape[0]
    rowlen = x.shape[1] * x.shape[2] if x.dim() == 3 else x.shape[1]
    span = (T - 1) * x.stride(0) + rowlen
    base = torch.as_strided(x, (span,), (1,), x.storage_offset())
    return B(base.contiguous())


def _quantize_both(k, v, slots, S, H, D=128):
    cache = kvq.Cache.empty(S, H, D)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.quantize_scatter(cache, k, v, slots.cuda(), err)
    torch.cuda.synchronize()
    oc = oracle.empty_cache(S, H, D)
    oerr = oracle.quantize_scatter(_flat(k), k.stride(0), _flat(v), v.stride(0), k.shape[0], H, D,
                                   slots.cpu().numpy(), oc)
    return cache, oc, int(err.item()), oerr


def test_tiny_workload_bit_exact():
    w = workloads.WORKLOADS["tiny"]
    k, v = workloads.request_kv(w, 0, 0, 64)
    slots = torch.randperm(64, generator=workloads.generator(0, 9)).to(torch.int64)
    cache, oc, e, oe = _quantize_both(k.cuda(), v.cuda(), slots, 64, 8)
    assert e == 0 and oe == 0
    assert_cache_equal(cache, oc)


@pytest.mark.parametrize("kind", ["normal", "lognormal_rows"])
def test_random_rows_bit_exact(kind):
    T, H = 3000, 8
    k, v = workloads.kv_rows(kind, T, H, 128, workloads.generator(5, 1))
    slots = torch.randperm(T, generator=workloads.generator(5, 2)).to(torch.int64)
    cache, oc, e, oe = _quantize_both(k.cuda(), v.cuda(), slots, T, H)
    assert_cache_equal(cache, oc)


def test_every_bf16_value_encodes_like_the_oracle():
    # rows whose amax is exactly 448 have scale 1, so every bf16 value with
    # |x| <= 448 is encoded as itself
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(x) & (np.abs(x) <= 448)
    vals = torch.from_numpy(bits[keep].view(np.int16)).view(torch.bfloat16)
    n = vals.numel()
    rows = (n + 126) // 127
    buf = torch.zeros(rows * 127, dtype=torch.bfloat16)
    buf[:n] = vals
    body = buf.view(rows, 127)
    k = torch.cat([torch.full((rows, 1), 448.0, dtype=torch.bfloat16), body], dim=1)
    k = k.view(rows, 1, 128)
    v = (-k).contiguous()
    slots = torch.arange(rows, dtype=torch.int64)
    cache, oc, _, _ = _quantize_both(k.cuda(), v.cuda(), slots, rows, 1)
    assert torch.all(cache.k_scales == 1.0)
    assert_cache_equal(cache, oc)


def test_tiny_and_zero_rows():
    T, H = 64, 4
    g = workloads.generator(7, 1)
    k = torch.randn(T, H, 128, generator=g)
    k[0:8] *= 1e-38            # fp32 subnormal scales
    k[8:16] *= 1e-30
    k[16] = 0.0                # all-zero rows
    k[17] = -0.0               # negative zeros
    k[18, :, ::2] = -0.0
    k[19] *= 3e37              # near the top of the range
    k = k.to(torch.bfloat16)
    v = k.flip(0).contiguous()
    slots = torch.arange(T, dtype=torch.int64)
    cache, oc, _, _ = _quantize_both(k.cuda(), v.cuda(), slots, T, H)
    assert_cache_equal(cache, oc)
    assert torch.all(cache.k_scales[16:18] == 0) and torch.all(cache.k_codes[16:18] == 0)


def _rows_near_midpoints(rows: int, seed: int) -> torch.Tensor:
    """bf16 rows [rows, 128] whose amax spans every bf16 binade (subnormal
    amax included, so scales from fp32 subnormals up to 2^119) and whose other
    elements are the bf16 values nearest to (e4m3 midpoint) * scale, +-2 bf16
    ulps: their quotients x / scale fall within an ulp of an e4m3 rounding
    boundary far more often than random data, exercising the division and the
    nearest-even rounding at the cases where either could go wrong."""
    rng = np.random.default_rng(seed)
    expo = rng.integers(0, 255, rows, dtype=np.uint32)
    mant = rng.integers(0, 128, rows, dtype=np.uint32)
    mant[expo == 0] |= 1                                   # no zero amax here
    amax_bits = ((expo << 7) | mant).astype(np.uint16)
    amax = (amax_bits.astype(np.uint32) << 16).view(np.float32)
    s = (amax / np.float32(448.0)).astype(np.float32)      # IEEE binary32
    grid = oracle.e4m3_decode(np.arange(0x7F))
    mids = np.concatenate([(grid[:-1] + grid[1:]) / 2, grid])
    pick = mids[rng.integers(0, mids.size, (rows, 127))]
    target = torch.from_numpy(pick * s.astype(np.float64)[:, None])
    xb = B(target.to(torch.bfloat16)).astype(np.int32)
    xb = np.clip(xb + rng.integers(-2, 3, xb.shape), 0, None)
    xb = np.minimum(xb, amax_bits.astype(np.int32)[:, None])  # |x| <= amax
    sign = rng.integers(0, 2, xb.shape).astype(np.int32) << 15
    body = (xb | sign).astype(np.uint16)
    full = np.concatenate([amax_bits[:, None], body], axis=1)
    perm = rng.permuted(np.tile(np.arange(128), (rows, 1)), axis=1)
    full = np.take_along_axis(full, perm, axis=1)
    return torch.from_numpy(full.view(np.int16)).view(torch.bfloat16)


def test_rounding_boundaries_every_scale_bit_exact():
    T, H = 8192, 2
    k = _rows_near_midpoints(T * H, 21).view(T, H, 128)
    v = _rows_near_midpoints(T * H, 22).view(T, H, 128)
    slots = torch.arange(T, dtype=torch.int64)
    cache, oc, _, _ = _quantize_both(k.cuda(), v.cuda(), slots, T, H)
    assert_cache_equal(cache, oc)


@pytest.mark.parametrize("swap", [False, True])
def test_strided_pitch_regression(swap):
    """FreeToken PR #354 review: K a view of the qkv slice (pitch 1152), V dense
    (pitch 384), 8 tokens x 3 heads x 128; 0 of 3072 codes may differ."""
    T, H, D = 8, 3, 128
    g = workloads.generator(11, 1)
    qkv = torch.randn(T, 3 * H * D, generator=g).to(torch.bfloat16).cuda()
    k_view = qkv[:, H * D:2 * H * D].view(T, H, D)
    v_dense = (torch.randn(T, H * D, generator=g).to(torch.bfloat16).clamp(-448, 448)
               .cuda().view(T, H, D))
    assert k_view.stride(0) == 1152 and v_dense.stride(0) == 384
    a, b = (v_dense, k_view) if swap else (k_view, v_dense)
    slots = torch.arange(T, dtype=torch.int64)
    cache, oc, _, _ = _quantize_both(a, b, slots, T, H)
    ek, _ = oracle.quantize_rows(B(a.contiguous()))
    ev, _ = oracle.quantize_rows(B(b.contiguous()))
    assert int((cache.k_codes.cpu().numpy() != ek).sum()) == 0
    assert int((cache.v_codes.cpu().numpy() != ev).sum()) == 0
    assert_cache_equal(cache, oc)


def test_store_workload_full_size_bit_exact_and_graph_replay():
    """The prefill-sized store: 16,384 tokens as strided views of a fused qkv
    [16384, 6144] with outliers and zero rows, permuted int64 slot ids on the
    device, captured once in a CUDA graph and replayed."""
    w = workloads.WORKLOADS["store"]
    qkv, k, v, slots, S = workloads.store_qkv(w, device="cpu")
    qkv = qkv.cuda()
    Hq, H, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    k = qkv[:, Hq * D:(Hq + H) * D].view(-1, H, D)
    v = qkv[:, (Hq + H) * D:].view(-1, H, D)
    slots_d = slots.cuda()
    cache = kvq.Cache.empty(S, H, D, w.block_size)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        kvq.quantize_scatter(cache, k, v, slots_d, err)  # warm up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        kvq.quantize_scatter(cache, k, v, slots_d, err)
    # new values in the same buffers, then replay
    qkv.mul_(-0.5)
    cache.k_codes.zero_()
    cache.v_scales.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oc = oracle.empty_cache(S, H, D)
    qh = B(qkv.cpu()).reshape(-1)
    oracle.quantize_scatter(qh[Hq * D:], qkv.stride(0), qh[(Hq + H) * D:], qkv.stride(0),
                            qkv.shape[0], H, D, slots.numpy(), oc)
    assert_cache_equal(cache, oc)
    assert int((cache.k_scales == 0).sum()) + int((cache.v_scales == 0).sum()) >= 2


def test_padding_out_of_range_and_guard_bands():
    T, H, D, S = 16, 2, 128, 12
    k, v = workloads.kv_rows("normal", T, H, D, workloads.generator(13, 1))
    slots = torch.arange(T, dtype=torch.int64)
    slots[3] = -1          # padding: skipped silently
    slots[5] = S           # out of range: skipped and flagged
    slots[6] = S + 1000
    # the rest unique and in range (ids must be unique: two tokens writing one
    # slot race); slot 3 is never written
    slots[7:] = torch.tensor([7, 8, 9, 10, 11, 5, 6, -1, -1], dtype=torch.int64)
    guard = 4096
    sentinel = 0xA5
    big = torch.full((2 * guard + S * H * D,), sentinel, dtype=torch.uint8, device="cuda")
    big_v = torch.full_like(big, sentinel)
    kc = big[guard:guard + S * H * D].view(S, H, D)
    vc = big_v[guard:guard + S * H * D].view(S, H, D)
    fs = torch.full((2 * 64 + S * H,), -7.0, device="cuda")
    ks = fs[64:64 + S * H].view(S, H)
    fv = torch.full_like(fs, -7.0)
    vs = fv[64:64 + S * H].view(S, H)
    cache = kvq.Cache(kc, vc, ks, vs, 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.quantize_scatter(cache, k.cuda(), v.cuda(), slots.cuda(), err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvq.ERRF_SLOT_RANGE
    for b in (big, big_v):
        assert torch.all(b[:guard] == sentinel) and torch.all(b[-guard:] == sentinel)
    for f in (fs, fv):
        assert torch.all(f[:64] == -7.0) and torch.all(f[-64:] == -7.0)
    # slot 3 was never written (token 3 is padding, no other token maps there)
    assert torch.all(kc[3] == sentinel) and torch.all(ks[3] == -7.0)
    oc = oracle.empty_cache(S, H, D)
    oc["k_codes"][:] = sentinel
    oc["v_codes"][:] = sentinel
    oc["k_scales"][:] = -7.0
    oc["v_scales"][:] = -7.0
    oe = oracle.quantize_scatter(B(k).reshape(-1), H * D, B(v).reshape(-1), H * D, T, H, D,
                                 slots.numpy(), oc)
    assert oe == oracle.ERR_SLOT_RANGE
    assert_cache_equal(cache, oc)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_dequant_rows_bit_exact(out_dtype):
    T, H, D = 500, 8, 128
    k, v = workloads.kv_rows("lognormal_rows", T, H, D, workloads.generator(17, 1))
    k[3] *= 1e-38
    slots = torch.randperm(T, generator=workloads.generator(17, 2)).to(torch.int64)
    cache, oc, _, _ = _quantize_both(k.cuda(), v.cuda(), slots, T, H)
    sel = torch.tensor([0, 5, 499, -1, 250, 1000, 7], dtype=torch.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ok, ov = kvq.dequant_rows(cache, sel.cuda(), out_dtype, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvq.ERRF_SLOT_RANGE
    code = 0 if out_dtype == torch.float32 else 1
    ek = oracle.dequant_rows(oc["k_codes"], oc["k_scales"], sel.numpy(), code)
    ev = oracle.dequant_rows(oc["v_codes"], oc["v_scales"], sel.numpy(), code)
    iv = torch.int32 if code == 0 else torch.int16
    nv = np.uint32 if code == 0 else np.uint16
    gk = ok.cpu().contiguous().view(iv).numpy().view(nv)
    gv = ov.cpu().contiguous().view(iv).numpy().view(nv)
    assert np.array_equal(gk, ek.view(nv))
    assert np.array_equal(gv, ev.view(nv))
