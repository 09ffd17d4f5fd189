"""Dense brute-force attention over a gathered cache -- TEST INFRASTRUCTURE ONLY.

A second, deliberately different formulation of the attention the C oracle
computes, used only to cross-check it on tiny inputs: it takes no block-table
walk inside the loop and no running softmax.  The K/V rows of each request are
first gathered into contiguous [L, H, D] tensors (plain indexing), the e4m3
codes are decoded by PyTorch's own ``float8_e4m3fn`` dtype (an independent
library routine), and the attention is one fp64 matrix product, a library
softmax and a second matrix product per (request, row, head).

Pages: ROCm/ATOM PR #2655 (PR description, K/V bullet) for the per-row scales
and GQA sharing; FlashML-org/FreeToken PR #354 (PR description) for the
[slot, head, dim] cache geometry.
"""
from __future__ import annotations

import numpy as np
import torch


def decode_codes_torch(codes: np.ndarray) -> torch.Tensor:
    """e4m3 codes -> float64 values, through torch's float8_e4m3fn dtype."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64)


def bf16_bits_to_torch(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64)


def gather_request(cache: dict, block_table: np.ndarray, length: int, block_size: int):
    """Dequantised K, V of one request, contiguous: two float64 [L, H, D]."""
    pos = np.arange(length)
    slots = block_table[pos // block_size].astype(np.int64) * block_size + pos % block_size
    kc = decode_codes_torch(cache["k_codes"][slots])
    vc = decode_codes_torch(cache["v_codes"][slots])
    ks = torch.from_numpy(cache["k_scales"][slots].astype(np.float64))
    vs = torch.from_numpy(cache["v_scales"][slots].astype(np.float64))
    return kc * ks[..., None], vc * vs[..., None]


def dense_attention(cache: dict, q_bits: np.ndarray, N: int, R: int, Hq: int,
                    block_tables: np.ndarray, context_lens: np.ndarray,
                    block_size: int, sm_scale: float) -> np.ndarray:
    """fp64 attention, [N*R, Hq, D], with the same row/visibility rules as the
    C oracle (row i of a request with R rows sees its first L - R + 1 + i tokens;
    GQA head hq reads KV head hq // (Hq // H); nothing visible gives zeros)."""
    H = cache["k_codes"].shape[1]
    D = cache["k_codes"].shape[2]
    G = Hq // H
    q = bf16_bits_to_torch(q_bits).reshape(N * R, Hq, D)
    out = torch.zeros(N * R, Hq, D, dtype=torch.float64)
    for r in range(N):
        L = int(context_lens[r])
        K, V = gather_request(cache, block_tables[r], L, block_size)
        for i in range(R):
            vis = L - R + 1 + i
            if vis <= 0:
                continue
            for hq in range(Hq):
                kh = hq // G
                s = sm_scale * (K[:vis, kh, :] @ q[r * R + i, hq])
                p = torch.softmax(s, dim=0)
                out[r * R + i, hq] = p @ V[:vis, kh, :]
    return out.numpy()
