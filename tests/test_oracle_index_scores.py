"""Pins for the oracle's index scorer (ROCm/ATOM PR #2655, PR description:
the decode-time scorer multiplies R query rows x H index heads against each
cached index key in one product; each head's dot is clipped at zero before
the heads are added), checked
against scores worked by hand, a dense numpy evaluation on the dequantised
keys, and the block-table indirection."""
import numpy as np
import torch

import oracle


def _bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_scores_worked_by_hand():
    """One MXFP4 key: dim 5 holds code 7 (6.0) in group 0 with exponent 1 ->
    12.0, all else 0.  The query's four heads are 0.5, -1, 2 and 0 times e_5:
    dots 6, -12, 24, 0 -> ReLU and sum = 30.  Token 1 is all zero -> 0."""
    codes = np.zeros((4, 64), dtype=np.uint8)
    exps = np.full((4, 4), 127, dtype=np.uint8)
    codes[0, 2] = 0x70                          # dim 5 = high nibble of byte 2
    exps[0, 0] = 128                            # X = 1
    q = np.zeros((1, 4, 128), dtype=np.float32)
    q[0, :, 5] = [0.5, -1.0, 2.0, 0.0]
    bt = np.array([[0, 1]], dtype=np.int32)
    out, err = oracle.index_scores(1, codes, None, exps, bt, 2, np.array([2], np.int32), 1, 4,
                                   _bits(q), 5)
    assert err == 0
    assert out[0, 0] == 30.0 and out[0, 1] == 0.0
    assert np.all(np.isneginf(out[0, 2:]))


def test_verify_rows_are_causal():
    """R = 2 rows, L = 3: row 0 sees tokens 0, 1; row 1 sees 0, 1, 2."""
    codes = np.full((8, 128), 0x38, dtype=np.uint8)      # e4m3 1.0 everywhere
    scales = np.ones(8, dtype=np.float32)
    q = np.full((2, 1, 128), 1.0 / 128, dtype=np.float32)
    bt = np.array([[0, 1]], dtype=np.int32)
    out, err = oracle.index_scores(0, codes, scales, None, bt, 4, np.array([3], np.int32), 2, 1,
                                   _bits(q), 6)
    assert err == 0
    assert np.allclose(out[0, :2], 1.0) and np.all(np.isneginf(out[0, 2:]))
    assert np.allclose(out[1, :3], 1.0) and np.all(np.isneginf(out[1, 3:]))


def _random_case(fmt, seed):
    rng = np.random.default_rng(seed)
    N, R, H, bs = 3, 2, 4, 8
    lens = np.array([17, 40, 5], dtype=np.int32)
    nblk = 16
    S = nblk * bs
    x = (rng.standard_normal((S, 128)) * np.exp(rng.standard_normal((S, 1)))).astype(np.float32)
    if fmt == 0:
        codes, scales = oracle.quantize_rows(_bits(x))
        exps = None
        # exact key values: code value times scale, in double
        keys = oracle.e4m3_decode(codes).astype(np.float64) * scales[:, None].astype(np.float64)
    else:
        codes, exps = oracle.mxfp4_quantize_rows(_bits(x))
        scales = None
        keys = oracle.mxfp4_dequant_rows(codes, exps)
    bt = rng.permutation(nblk)[:15].reshape(3, 5).astype(np.int32)
    q = rng.standard_normal((N * R, H, 128)).astype(np.float32)
    qf = torch.from_numpy(_bits(q).view(np.int16)).view(torch.bfloat16).double().numpy()
    return fmt, codes, scales, exps, bt, bs, lens, R, H, q, qf, keys.astype(np.float64)


def test_matches_dense_numpy_on_dequantised_keys():
    for fmt in (0, 1):
        fmt, codes, scales, exps, bt, bs, lens, R, H, q, qf, keys = _random_case(fmt, fmt + 4)
        max_len = 44
        out, err = oracle.index_scores(fmt, codes, scales, exps, bt, bs, lens, R, H, _bits(q),
                                       max_len)
        assert err == 0
        for r in range(len(lens)):
            # gather the request's keys contiguously, then one matrix product
            pos = np.arange(lens[r])
            slots = bt[r, pos // bs] * bs + pos % bs
            k = keys[slots]                                        # [L, 128]
            dots = np.einsum("ihd,td->iht", qf[r * R:(r + 1) * R], k)
            want = np.maximum(dots, 0.0).sum(axis=1)               # [R, L]
            for i in range(R):
                vis = lens[r] - R + 1 + i
                got = out[r * R + i]
                assert np.allclose(got[:vis], want[i, :vis], rtol=1e-12, atol=1e-12)
                assert np.all(np.isneginf(got[vis:]))
