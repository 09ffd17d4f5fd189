"""Pins for the oracle's MXFP4 index-key codec (ROCm/ATOM PR #2655, PR
description, index-key bullet: two E2M1 codes per byte, an E8M0 exponent for
every 32 dims, large enough that no element overflows), checked against values worked by
hand from the format, brute force over all 16 codes, and properties that must
hold for every input."""
import numpy as np
import torch

import oracle

# The E2M1 element format (1 sign, 2 exponent bits with bias 1, 1 mantissa
# bit), its eight magnitudes listed from the format's definition: subnormal
# 0 and 0.5, then 1, 1.5 (exponent 1), 2, 3 (exponent 2), 4, 6 (exponent 3).
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_e2m1_decode_table():
    for c in range(16):
        mag = E2M1_MAGNITUDES[c & 7]
        v = oracle.e2m1_decode(np.array([c]))[0]
        assert v == (-mag if c & 8 else mag) and np.signbit(v) == bool(c & 8)


def test_e2m1_ties_and_saturation_worked_by_hand():
    # midpoints go to the even code (mantissa bit 0): 0.25 -> 0, 0.75 -> 1.0,
    # 1.25 -> 1.0, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4; 6.5 and up saturate
    q = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 0.2, 0.3, 5.1, -2.6, -0.0, -0.1]
    want = [0, 2, 2, 4, 4, 6, 6, 7, 0, 1, 7, 0xD, 0x8, 0x8]
    assert oracle.e2m1_encode(np.array(q)).tolist() == want


def test_e2m1_encode_brute_force():
    """Against a search over all 16 codes: the nearest value, and at equal
    distance the code with the even mantissa bit; the sign of the input."""
    rng = np.random.default_rng(7)
    q = np.concatenate([rng.uniform(-7, 7, 4000),
                        np.array([m + s * d for m in E2M1_MAGNITUDES for s in (-1, 1)
                                  for d in (0.0, 0.125, 0.25, 0.5, 1.0)])])
    got = oracle.e2m1_encode(q)
    for x, c in zip(q, got):
        a = min(abs(x), 6.0)
        dist = [abs(a - m) for m in E2M1_MAGNITUDES]
        best = min(dist)
        cands = [i for i, d in enumerate(dist) if d == best]
        mag = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        assert c == (mag | (8 if np.signbit(x) else 0)), (x, c)


def test_group_exponent_is_the_smallest_that_does_not_clip():
    """Every positive finite bf16 amax: 6 * 2^X >= amax and 6 * 2^(X-1) < amax
    (unless X sits at the E8M0 clamp)."""
    bits = np.arange(1, 0x7F80, dtype=np.uint16)
    amax = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    for a in amax.astype(np.float64):
        X = oracle.mxfp4_group_exponent(a)
        assert -127 <= X <= 127
        if X > -127:
            assert 6.0 * 2.0 ** X >= a and 6.0 * 2.0 ** (X - 1) < a, a
        else:
            assert 6.0 * 2.0 ** X >= a
    assert oracle.mxfp4_group_exponent(0.0) == -127
    assert oracle.mxfp4_group_exponent(6.0) == 0
    assert oracle.mxfp4_group_exponent(1.5) == -2
    assert oracle.mxfp4_group_exponent(7.0) == 1


def test_row_layout_worked_by_hand():
    """Group 0 has amax 6 (X = 0, E8M0 127): 1.0 -> 2, 6.0 -> 7 share byte 0 as
    0x72 (even element in the low nibble); -0.5 -> 9, 3.0 -> 5 make 0x59.
    Group 1 is 0.75 and 0.1 elsewhere (X = -3: 0.75 = 6 / 8): 0.75 * 8 = 6 ->
    7, 0.1 * 8 = 0.8 -> 1.0 -> 2.  Groups 2 and 3 are zero: X = -127, code 0."""
    row = np.zeros(128, dtype=np.float32)
    row[0:4] = [1.0, 6.0, -0.5, 3.0]
    row[32:64] = 0.1
    row[32] = 0.75
    codes, exps = oracle.mxfp4_quantize_rows(_bf16_bits(row)[None, :])
    assert exps.tolist() == [[127, 124, 0, 0]]
    assert codes[0, 0] == 0x72 and codes[0, 1] == 0x59 and not codes[0, 2:16].any()
    # 0.1 in bf16 is 0.10009765625: times 8 = 0.80078 -> 1.0 (code 2)
    assert codes[0, 16] == 0x27 and (codes[0, 17:32] == 0x22).all()
    assert not codes[0, 32:].any()


def test_never_clips_and_nearest_in_every_group():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 128)) * np.exp(rng.standard_normal((64, 1)) * 3)).astype(
        np.float32)
    xb = _bf16_bits(x)
    xf = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).double().numpy()
    codes, exps = oracle.mxfp4_quantize_rows(xb)
    deq = oracle.mxfp4_dequant_rows(codes, exps).astype(np.float64)
    for r in range(64):
        for g in range(4):
            grp = xf[r, 32 * g:32 * g + 32]
            X = int(exps[r, g]) - 127
            assert np.abs(grp).max() <= 6.0 * 2.0 ** X
            # every element's value is the nearest grid point of its group
            grid = np.array(E2M1_MAGNITUDES) * 2.0 ** X
            for d in range(32):
                err = abs(deq[r, 32 * g + d] - grp[d])
                assert err <= np.abs(grid - abs(grp[d])).min() + 0.0


def test_round_trip_of_representable_values():
    """Values that are decode(c) * 2^X quantise back to the same codes and
    exponent when the group's largest magnitude is 6 * 2^X (the exponent the
    rule picks)."""
    rng = np.random.default_rng(3)
    for X in (-20, -3, 0, 5, 40):
        mags = rng.integers(0, 16, size=(8, 32))
        mags[:, 0] = 7                                  # one element at 6 * 2^X
        vals = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])[mags] * 2.0 ** X
        row = np.tile(vals.reshape(8, 32), (1, 4)).astype(np.float32)
        codes, exps = oracle.mxfp4_quantize_rows(_bf16_bits(row))
        assert (exps == X + 127).all()
        deq = oracle.mxfp4_dequant_rows(codes, exps)
        assert np.array_equal(deq, row)
