"""Shared helpers for the GPU parity tests: build the same cache through the
CUDA path and through the oracle from the same seeded bf16 rows, and compare.

The oracle never sees anything the CUDA path produced: it quantises the
generator's bf16 rows itself."""
from __future__ import annotations

import numpy as np
import torch

import fp8_paged_kv_kvq_gb300 as kvq
import oracle
import workloads

# Attention tolerance.  The stated bound is max |err| <= 1e-2 and rel-L2 <= 5e-3
# for bf16 output against fp64 attention over the same dequantised codes.  A
# bf16 output cannot be closer to the exact value than half a bf16 ulp, which
# exceeds 1e-2 once |out| >= 4, so the elementwise bound is applied as
# max(1e-2, one bf16 ulp at |ref|), the ulp being 2^(floor(log2 |ref|) - 7)
# (between 2^-8 |ref| and 2^-7 |ref|): a correctly rounded output plus the
# fp32 / f16 arithmetic error of the kernels stays inside it.  rel-L2 is
# applied as stated.
MAX_ABS = 1e-2
REL_L2 = 5e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """One bf16 ulp at |x| (2^(floor(log2|x|) - 7); 0 for x = 0)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(a)                  # a = m 2^e, m in [0.5, 1)
    return np.where(a > 0, np.ldexp(1.0, e - 8), 0.0)


def attention_errors(gpu, ref: np.ndarray):
    """(worst |err| / max(1e-2, bf16 ulp of |ref|), rel-L2, worst raw |err|, |ref| there)."""
    if isinstance(gpu, torch.Tensor):
        g = gpu.float().cpu().numpy().astype(np.float64)
    else:
        g = np.asarray(gpu, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g))
    err = np.abs(g - ref)
    scaled = err / np.maximum(MAX_ABS, bf16_ulp(ref))
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(g - ref) / denom if denom > 0 else np.linalg.norm(g - ref)
    if not scaled.size:
        return 0.0, float(rel), 0.0, 0.0
    i = int(np.argmax(scaled))
    return float(scaled.flat[i]), float(rel), float(err.flat[i]), float(np.abs(ref).flat[i])


def assert_attention_close(gpu, ref, what=""):
    mx, rel, raw, at = attention_errors(gpu, ref)
    msg = (f"{what}: worst |err| / max(1e-2, bf16 ulp) = {mx:.3f} (|err| {raw:.3e} at "
           f"|ref| {at:.3e}), rel-L2 {rel:.3e}")
    print(msg)
    assert mx <= 1.0, msg
    assert rel <= REL_L2, msg
    return mx, rel


def build_paged(w: workloads.Workload, lens, device="cuda", spare_blocks=3, oracle_side=True,
                gen_device="cpu"):
    """Quantise every request's context into a GPU cache (through
    kvq_quantize_scatter) and, if asked, into an oracle cache from the same
    bf16 rows.  Returns a dict with the GPU cache, oracle cache, block tables."""
    lens = np.asarray(lens, dtype=np.int32)
    bt, nblk = workloads.block_tables(lens, w.block_size, w.seed, spare_blocks=spare_blocks)
    S = nblk * w.block_size
    H, D = w.num_kv_heads, w.head_dim
    cache = kvq.Cache.empty(S, H, D, w.block_size, device=device)
    ocache = oracle.empty_cache(S, H, D) if oracle_side else None
    err = torch.zeros(1, dtype=torch.int32, device=device)
    for r in range(len(lens)):
        L = int(lens[r])
        if L == 0:
            continue
        k, v = workloads.request_kv(w, r, 0, L, device=gen_device)
        slots = workloads.token_slots(bt, r, L, w.block_size)
        kvq.quantize_scatter(cache, k.to(device), v.to(device),
                             torch.from_numpy(slots).to(device), err)
        if oracle_side:
            oracle.quantize_scatter(workloads.bf16_bits(k).reshape(-1), H * D,
                                    workloads.bf16_bits(v).reshape(-1), H * D, L, H, D, slots,
                                    ocache)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return {"cache": cache, "ocache": ocache, "bt": bt, "lens": lens, "S": S}


def build_custom(w, kv_per_request, spare_blocks=3):
    """GPU and oracle caches from given bf16 K/V rows [L, H, D] per request."""
    lens = np.array([k.shape[0] for k, _ in kv_per_request], dtype=np.int32)
    bt, nblk = workloads.block_tables(lens, w.block_size, w.seed, spare_blocks=spare_blocks)
    S = nblk * w.block_size
    H, D = w.num_kv_heads, w.head_dim
    cache = kvq.Cache.empty(S, H, D, w.block_size)
    ocache = oracle.empty_cache(S, H, D)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r, (k, v) in enumerate(kv_per_request):
        L = k.shape[0]
        slots = workloads.token_slots(bt, r, L, w.block_size)
        kvq.quantize_scatter(cache, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), err)
        oracle.quantize_scatter(workloads.bf16_bits(k).reshape(-1), H * D,
                                workloads.bf16_bits(v).reshape(-1), H * D, L, H, D, slots, ocache)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return {"cache": cache, "ocache": ocache, "bt": bt, "lens": lens, "S": S}


def assert_cache_equal(cache: kvq.Cache, ocache: dict):
    for name in ("k_codes", "v_codes"):
        got = getattr(cache, name).cpu().numpy()
        exp = ocache[name]
        bad = int((got != exp).sum())
        assert bad == 0, f"{name}: {bad} of {got.size} codes differ"
    for name in ("k_scales", "v_scales"):
        got = getattr(cache, name).cpu().numpy()
        exp = ocache[name]
        assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), f"{name} differ"


def gpu_decode(built, q_bf16, R, sm_scale, partition_tokens=0, max_context_len=None,
               err=None, lens=None):
    cache = built["cache"]
    bt = torch.from_numpy(built["bt"]).cuda()
    ln = built["lens"] if lens is None else np.asarray(lens, dtype=np.int32)
    cl = torch.from_numpy(ln).cuda()
    maxc = int(ln.max()) if max_context_len is None else max_context_len
    return kvq.paged_decode(cache, q_bf16.cuda(), bt, cl, maxc, sm_scale, rows_per_request=R,
                            partition_tokens=partition_tokens, err_flags=err)


def oracle_decode(built, q_bf16, R, Hq, sm_scale, lens=None):
    ln = built["lens"] if lens is None else np.asarray(lens, dtype=np.int32)
    return oracle.paged_attention(built["ocache"], workloads.bf16_bits(q_bf16), len(ln), R, Hq,
                                  built["bt"], ln, built["cache"].block_size, sm_scale)
