"""Seeded synthetic workloads for the FP8 paged KV cache.

This module holds only input generation: shapes, seeds and random draws.  It
holds none of the method's arithmetic (no scale, no encode, no attention), so
both the CPU oracle and the CUDA path can take its outputs as their inputs.

The five workloads follow the shapes the pages' deployments imply (GQA decode
with head_dim 128, paged caches with block size 16 or 64, a fused qkv
projection output, MTP-style verify with 3 draft tokens, a 1M-token context):

  tiny       64 tokens x 8 KV heads x 128, bf16 N(0,1), block size 16, blocks
             randomly permuted; decode for 1 request, 32 q heads (GQA 4),
             context 64, q N(0,1), sm_scale 1/sqrt(128).            (seed 0)
  decode     32 requests, context lengths uniform in [1024, 8192], 32 q heads /
             8 KV heads, block size 16, non-contiguous random block tables; K, V
             rows N(0,1) times a per-row log-normal(0,1) magnitude; 1 query row
             per request.                                           (seed 1)
  store      16,384 tokens as strided K and V views of a fused bf16 qkv tensor
             [16384, (32+8+8)*128], N(0,1) with 1% of elements x50 (outliers)
             and all-zero (token, head) rows with probability 1/128; slot ids a
             random permutation (device int64); block size 64.      (seed 2)
  verify     64 requests x 4 query rows, 64 q heads / 8 KV heads, context
             32,768, block size 64; K, V as in ``decode``.          (seed 3)
  longctx    2 requests x 1,048,576 tokens, 32 q heads / 8 KV heads, block size
             64; K, V as in ``decode``; 1 query row per request.    (seed 4)
  prefill    4 requests, each a chunk of 2,048 new tokens at the end of an
             8,192-token context (chunked prefill: the chunk's rows attend
             causally to everything cached before them and to each other), 32 q
             heads / 8 KV heads, block size 64; K, V as in ``decode``.  (seed 7)

One more workload feeds the stacked index scorer:

  index_scores  64 requests x 4 query rows x 4 index heads, context 32,768,
             block size 64, one 128-dim index key per token; the key codes are
             drawn directly (every drawn byte a finite code of its format), the
             queries N(0,1).                                          (seed 6)

Large caches are generated chunk by chunk on the device with a generator seeded
from (workload seed, request, chunk), so that any chunk can be drawn again on
its own (the parity tests sample requests of the large workloads that way).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    num_requests: int
    rows_per_request: int          # R: 1 decode, 4 verify (3 draft tokens + 1)
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    context_min: int               # context lengths uniform in [min, max]
    context_max: int
    kv_rows: str                   # "normal" or "lognormal_rows"
    store_tokens: int = 0          # prefill-sized store workload only

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


WORKLOADS = {
    "tiny": Workload("tiny", 0, 1, 1, 32, 8, HEAD_DIM, 16, 64, 64, "normal"),
    "decode": Workload("decode", 1, 32, 1, 32, 8, HEAD_DIM, 16, 1024, 8192, "lognormal_rows"),
    "store": Workload("store", 2, 0, 1, 32, 8, HEAD_DIM, 64, 0, 0, "normal", store_tokens=16384),
    "verify": Workload("verify", 3, 64, 4, 64, 8, HEAD_DIM, 64, 32768, 32768, "lognormal_rows"),
    "longctx": Workload("longctx", 4, 2, 1, 32, 8, HEAD_DIM, 64, 1 << 20, 1 << 20, "lognormal_rows"),
    "prefill": Workload("prefill", 7, 4, 2048, 32, 8, HEAD_DIM, 64, 8192, 8192, "lognormal_rows"),
}


def generator(seed: int, *parts: int, device="cpu") -> torch.Generator:
    """A torch generator seeded from a workload seed and sub-stream ids."""
    s = int(seed) & 0xFFFFFFFF
    for p in parts:
        s = (s * 1_000_003 + int(p) + 0x9E3779B9) & 0x7FFFFFFFFFFFFFFF
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def context_lengths(w: Workload) -> np.ndarray:
    g = generator(w.seed, 1)
    if w.context_min == w.context_max:
        return np.full(w.num_requests, w.context_min, dtype=np.int32)
    lens = torch.randint(w.context_min, w.context_max + 1, (w.num_requests,), generator=g)
    return lens.numpy().astype(np.int32)


def block_tables(lens: np.ndarray, block_size: int, seed: int, spare_blocks: int = 0):
    """Random non-contiguous paging: every request gets ceil(L / bs) blocks, the
    physical block ids are a seeded random permutation of the whole pool.
    Returns (block_tables int32 [N, max_blocks], num_blocks)."""
    need = [(int(L) + block_size - 1) // block_size for L in lens]
    max_blocks = max(max(need), 1) if len(need) else 1
    total = sum(need) + spare_blocks
    g = generator(seed, 2)
    perm = torch.randperm(max(total, 1), generator=g).numpy().astype(np.int32)
    bt = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(need):
        bt[r, :n] = perm[off:off + n]
        off += n
    return bt, max(total, 1)


def token_slots(bt: np.ndarray, r: int, L: int, block_size: int) -> np.ndarray:
    pos = np.arange(L, dtype=np.int64)
    return bt[r, pos // block_size].astype(np.int64) * block_size + pos % block_size


def kv_rows(w_kind: str, num_tokens: int, H: int, D: int, g: torch.Generator,
            device="cpu"):
    """K and V rows [T, H, D] bf16 for one chunk of tokens.

    ``normal``: N(0,1).  ``lognormal_rows``: N(0,1) times one exp(N(0,1))
    magnitude per (token, head) row, drawn independently for K and V."""
    k = torch.randn(num_tokens, H, D, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(num_tokens, H, D, generator=g, device=device, dtype=torch.float32)
    if w_kind == "lognormal_rows":
        k = k * torch.exp(torch.randn(num_tokens, H, 1, generator=g, device=device))
        v = v * torch.exp(torch.randn(num_tokens, H, 1, generator=g, device=device))
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def request_kv(w: Workload, r: int, start: int, count: int, device="cpu"):
    """K, V rows of tokens [start, start+count) of request r, drawn in chunks of
    ``chunk_tokens(w)`` so the same token always gets the same values."""
    ct = chunk_tokens(w)
    ks, vs = [], []
    c0, c1 = start // ct, (start + count - 1) // ct
    for c in range(c0, c1 + 1):
        g = generator(w.seed, 10, r, c, device=device)
        k, v = kv_rows(w.kv_rows, ct, w.num_kv_heads, w.head_dim, g, device)
        lo = max(start, c * ct) - c * ct
        hi = min(start + count, (c + 1) * ct) - c * ct
        ks.append(k[lo:hi])
        vs.append(v[lo:hi])
    return torch.cat(ks), torch.cat(vs)


def chunk_tokens(w: Workload) -> int:
    return 1024 if w.context_max <= 8192 else 16384


def queries(w: Workload, device="cpu") -> torch.Tensor:
    """bf16 q [N*R, Hq, D], N(0,1)."""
    g = generator(w.seed, 3, device=device)
    q = torch.randn(w.num_requests * w.rows_per_request, w.num_q_heads, w.head_dim,
                    generator=g, device=device)
    return q.to(torch.bfloat16)


def store_qkv(w: Workload, device="cpu"):
    """The prefill-sized store workload: a fused qkv tensor [T, (Hq+2H)*D] bf16,
    N(0,1), 1% of elements x50, and all-zero K or V (token, head) rows with
    probability 1/128 (at least one of each).  Returns (qkv, k_view, v_view,
    slot_ids int64 [T], num_slots)."""
    T, Hq, H, D = w.store_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    g = generator(w.seed, 4, device=device)
    x = torch.randn(T, (Hq + 2 * H) * D, generator=g, device=device)
    outlier = torch.rand(x.shape, generator=g, device=device) < 0.01
    x = torch.where(outlier, x * 50.0, x)
    x = x.to(torch.bfloat16)
    zero_rows = torch.rand(T, 2, H, generator=g, device=device) < (1.0 / 128.0)
    zero_rows[0, 0, 0] = True
    zero_rows[T - 1, 1, H - 1] = True
    kv = x[:, Hq * D:].view(T, 2, H, D)
    kv.masked_fill_(zero_rows[..., None], 0.0)
    k_view = x[:, Hq * D:(Hq + H) * D].view(T, H, D)
    v_view = x[:, (Hq + H) * D:].view(T, H, D)
    slot_ids = torch.randperm(T, generator=g, device=device).to(torch.int64)
    return x, k_view, v_view, slot_ids, T


def scaled(w: Workload, **changes) -> Workload:
    """A smaller copy of a workload with the same structure (for parity tests
    the oracle finishes in seconds)."""
    return dataclasses.replace(w, **changes)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (same shape)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclasses.dataclass(frozen=True)
class IndexScoreWorkload:
    num_requests: int = 64
    rows: int = 4
    heads: int = 4
    context: int = 32768
    block_size: int = 64
    seed: int = 6


INDEX_SCORES = IndexScoreWorkload()


def index_key_codes(fmt: int, num_slots: int, seed: int, exp_spread: int = 8):
    """Random index-key codes for ``num_slots`` tokens of 128 dims, as numpy.

    fmt 0 (FP8): codes uint8 [S, 128] uniform over the 254 finite e4m3 codes
    (0x7F and 0xFF left out), scales fp32 [S] = exp(N(0,1)) / 448.
    fmt 1 (MXFP4): codes uint8 [S, 64] uniform over all bytes (every nibble is
    an E2M1 code), exponent bytes uint8 [S, 4] uniform in 127 +- exp_spread.
    Returns (codes, scales or None, exponents or None)."""
    g = generator(seed, 7, fmt)
    if fmt == 0:
        c = torch.randint(0, 254, (num_slots, HEAD_DIM), generator=g, dtype=torch.int32)
        c = c + (c >= 0x7F).to(torch.int32)                 # skip 0x7F; 0xFF never drawn
        sc = torch.exp(torch.randn(num_slots, generator=g)) / 448.0
        return c.to(torch.uint8).numpy(), sc.to(torch.float32).numpy(), None
    c = torch.randint(0, 256, (num_slots, HEAD_DIM // 2), generator=g, dtype=torch.int32)
    e = torch.randint(127 - exp_spread, 128 + exp_spread, (num_slots, HEAD_DIM // 32),
                      generator=g, dtype=torch.int32)
    return c.to(torch.uint8).numpy(), None, e.to(torch.uint8).numpy()


def index_queries(num_requests: int, rows: int, heads: int, seed: int) -> torch.Tensor:
    """bf16 query vectors [N, R, H, 128], N(0,1)."""
    g = generator(seed, 8)
    return torch.randn(num_requests, rows, heads, HEAD_DIM, generator=g).to(torch.bfloat16)


def unit_rms_rows(num_tokens: int, H: int, D: int, g: torch.Generator) -> torch.Tensor:
    """bf16 rows [T, H, D] with unit RMS each (N(0,1) divided by the row's
    RMS): the O(1) post-LayerNorm values an unscaled fp8 cache is meant for."""
    x = torch.randn(num_tokens, H, D, generator=g, dtype=torch.float64)
    x = x / torch.sqrt((x * x).mean(dim=-1, keepdim=True))
    return x.to(torch.bfloat16)
