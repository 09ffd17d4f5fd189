"""Pins of the oracle's row quantiser and scatter: invariants the method fixes
(the amax element maps to +-448, the e4m3 error bound, zero rows), the
hand-derived row in tests/golden/e4m3_worked_examples.json, the multiset check
and the strided-V regression shape printed in the FreeToken PR #354 review."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads


def _bits(x: torch.Tensor) -> np.ndarray:
    return workloads.bf16_bits(x)


def _rows(n, D=128, seed=0, lognormal=True, tiny=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, D, generator=g)
    if lognormal:
        x = x * torch.exp(2.0 * torch.randn(n, 1, generator=g))
    if tiny:
        x = x * 1e-39  # bf16 subnormal territory: fp32 subnormal scales
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("tiny", [False, True])
def test_amax_element_encodes_to_448(tiny):
    x = _rows(4000, seed=1, tiny=tiny)
    codes, scales = oracle.quantize_rows(_bits(x))
    xf = x.float().numpy()
    nz = np.abs(xf).max(axis=1) > 0
    assert nz.sum() > 3000
    idx = np.abs(xf).argmax(axis=1)
    c = codes[np.arange(len(idx)), idx]
    sgn = np.signbit(xf[np.arange(len(idx)), idx])
    assert np.all(c[nz] == np.where(sgn[nz], 0xFE, 0x7E))
    assert not np.any((codes & 0x7F) == 0x7F)


def test_scale_is_amax_over_448_in_fp32():
    x = _rows(3000, seed=2)
    codes, scales = oracle.quantize_rows(_bits(x))
    amax = np.abs(x.float().numpy()).max(axis=1).astype(np.float32)
    assert np.array_equal(scales, (amax / np.float32(448.0)).astype(np.float32))


def test_reconstruction_error_bounds():
    x = _rows(3000, seed=3)
    codes, scales = oracle.quantize_rows(_bits(x))
    xf = x.double().numpy()
    rec = oracle.e4m3_decode(codes) * scales.astype(np.float64)[:, None]
    err = np.abs(rec - xf)
    q = np.abs(xf) / scales.astype(np.float64)[:, None]
    normal = q >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xf[normal]))
    sub = ~normal
    assert sub.sum() > 0
    bound = (2.0 ** -10 + 2.0 ** -20) * np.broadcast_to(scales[:, None], err.shape)[sub]
    assert np.all(err[sub] <= bound)


def test_zero_rows_and_signed_zeros():
    x = torch.zeros(3, 128, dtype=torch.bfloat16)
    x[1] = -0.0
    x[2, 5] = -0.0
    x[2, 7] = 2.0
    x[2, 9] = -1e-30
    codes, scales = oracle.quantize_rows(_bits(x))
    assert scales[0] == 0 and scales[1] == 0
    assert np.all(codes[0] == 0) and np.all(codes[1] == 0)
    assert scales[2] == np.float32(2.0) / np.float32(448.0)
    assert codes[2, 5] == 0x80 and codes[2, 9] == 0x80 and codes[2, 0] == 0x00
    assert codes[2, 7] == 0x7E


def test_hand_derived_row(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "e4m3_worked_examples.json")))["quantize_row"]
    x = torch.zeros(ex["head_dim"], dtype=torch.bfloat16)
    x[: len(ex["row_head"])] = torch.tensor(ex["row_head"])
    codes, scale = oracle.quantize_rows(_bits(x[None]))
    assert scale[0] == np.float32(3.0) / np.float32(448.0)
    assert [int(c) for c in codes[0, :4]] == [int(c, 16) for c in ex["codes_head"]]
    assert np.all(codes[0, 4:] == 0)


def test_scatter_is_a_permutation_of_rows():
    T, H, D = 96, 4, 128
    k = _rows(T * H, seed=4).view(T, H, D)
    v = _rows(T * H, seed=5).view(T, H, D)
    perm = np.random.default_rng(0).permutation(T).astype(np.int64)
    cache = oracle.empty_cache(T, H, D)
    err = oracle.quantize_scatter(_bits(k).reshape(-1), H * D, _bits(v).reshape(-1), H * D,
                                  T, H, D, perm, cache)
    assert err == 0
    kc, ks = oracle.quantize_rows(_bits(k))
    assert np.array_equal(cache["k_codes"][perm], kc)
    assert np.array_equal(cache["k_scales"][perm], ks)
    # the multiset check from the FreeToken review: sorted codes agree
    assert np.array_equal(np.sort(cache["v_codes"].reshape(-1)),
                          np.sort(oracle.quantize_rows(_bits(v))[0].reshape(-1)))


def test_scatter_skips_padding_and_flags_out_of_range():
    T, H, D = 4, 2, 128
    k = _rows(T * H, seed=6).view(T, H, D)
    cache = oracle.empty_cache(3, H, D)
    err = oracle.quantize_scatter(_bits(k).reshape(-1), H * D, _bits(k).reshape(-1), H * D,
                                  T, H, D, np.array([2, -1, 3, 0], dtype=np.int64), cache)
    assert err == oracle.ERR_SLOT_RANGE
    kc, _ = oracle.quantize_rows(_bits(k))
    assert np.array_equal(cache["k_codes"][2], kc[0]) and np.array_equal(cache["k_codes"][0], kc[3])
    assert np.all(cache["k_codes"][1] == 0)


def _strided_case(golden_dir):
    f = json.load(open(os.path.join(golden_dir, "pages_facts.json")))["strided_v_regression"]
    T, H, D = f["tokens"], f["num_heads"], f["head_dim"]
    g = torch.Generator().manual_seed(0)
    qkv = torch.randn(T, f["k_token_pitch"], generator=g).to(torch.bfloat16)
    k_rows = qkv[:, H * D:2 * H * D]        # view: token pitch 1152
    v_rows = torch.randn(T, H * D, generator=g).to(torch.bfloat16).clamp(-448, 448)
    assert k_rows.stride(0) == f["k_token_pitch"] and v_rows.stride(0) == f["v_token_pitch"]
    return f, qkv, k_rows, v_rows


def test_strided_k_and_v_pitches(golden_dir):
    f, qkv, k_rows, v_rows = _strided_case(golden_dir)
    T, H, D = f["tokens"], f["num_heads"], f["head_dim"]
    slots = np.arange(T, dtype=np.int64)
    flat_k = _bits(qkv).reshape(-1)[H * D:]  # K's rows start H*D elements in
    flat_v = _bits(v_rows).reshape(-1)
    for swap in (False, True):
        cache = oracle.empty_cache(T, H, D)
        if not swap:
            oracle.quantize_scatter(flat_k, f["k_token_pitch"], flat_v, f["v_token_pitch"],
                                    T, H, D, slots, cache)
            kk, vv = k_rows, v_rows
            ck, cv = cache["k_codes"], cache["v_codes"]
        else:
            oracle.quantize_scatter(flat_v, f["v_token_pitch"], flat_k, f["k_token_pitch"],
                                    T, H, D, slots, cache)
            kk, vv = v_rows, k_rows
            ck, cv = cache["k_codes"], cache["v_codes"]
        ek, _ = oracle.quantize_rows(_bits(kk.contiguous().view(T, H, D)))
        ev, _ = oracle.quantize_rows(_bits(vv.contiguous().view(T, H, D)))
        assert ck.size == f["codes_per_tensor"]
        assert int((ck != ek).sum()) == f["fixed_mismatches"]["k"]
        assert int((cv != ev).sum()) == f["fixed_mismatches"]["v"]


def test_planted_shared_pitch_bug_is_caught_by_codes(golden_dir):
    """Plant the reviewed bug in the oracle's input handling (V read at K's pitch,
    on the CPU) and check its fingerprint: token 0 right, tokens 1-2 wrong.
    The reads past the data are replaced by zeros here."""
    f, qkv, k_rows, v_rows = _strided_case(golden_dir)
    T, H, D = f["tokens"], f["num_heads"], f["head_dim"]
    flat_v = _bits(v_rows).reshape(-1)
    padded_v = np.zeros((T - 1) * f["k_token_pitch"] + H * D, dtype=np.uint16)
    padded_v[: flat_v.size] = flat_v
    cache = oracle.empty_cache(T, H, D)
    oracle.quantize_scatter(_bits(qkv).reshape(-1)[H * D:], f["k_token_pitch"], padded_v,
                            f["k_token_pitch"], T, H, D, np.arange(T, dtype=np.int64), cache)
    ev, _ = oracle.quantize_rows(_bits(v_rows.contiguous().view(T, H, D)))
    wrong_tok = [(cache["v_codes"][t] != ev[t]).any() for t in range(T)]
    for t in f["buggy_correct_tokens"]:
        assert not wrong_tok[t]
    for t in f["buggy_wrong_in_range_tokens"]:
        assert wrong_tok[t]
    assert sum(wrong_tok) == T - len(f["buggy_correct_tokens"])


def test_dequant_rows_bf16_matches_torch_rounding():
    x = _rows(64, seed=8).view(16, 4, 128)
    codes, scales = oracle.quantize_rows(_bits(x))
    sl = np.array([3, 0, 15, -1], dtype=np.int64)
    f32 = oracle.dequant_rows(codes, scales, sl, 0)
    b16 = oracle.dequant_rows(codes, scales, sl, 1)
    exact = oracle.e4m3_decode(codes) * scales[..., None].astype(np.float64)
    assert np.array_equal(f32[:3].astype(np.float64), exact[sl[:3]].astype(np.float32))
    assert np.all(f32[3] == 0)
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b16, ref)


def test_sidecar_overhead_fact(golden_dir):
    f = json.load(open(os.path.join(golden_dir, "pages_facts.json")))
    D = 128
    fp8_row = D * 1 + 4
    bf16_row = D * 2
    assert abs(4 / D - f["scale_sidecar_overhead_at_head_dim_128"]["value"]) <= \
        f["scale_sidecar_overhead_at_head_dim_128"]["approx_abs"]
    assert D * 1 / bf16_row == f["fp8_halves_bytes_per_token"]["value"]
    assert fp8_row / bf16_row == pytest.approx(0.5 + 4 / (2 * D))
