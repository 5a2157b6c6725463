"""Pins of the oracle's FP8 K/V storage (pogovet.com article, detail 5: compressed KV entries in
FP8, only the RoPE dims in BF16), CPU only: a hand-worked example, the power-of-two scale rule at
its boundaries, torch's own float8 / bfloat16 casts as an independent rounding, exact survival of
representable values, the error bound, and the K/V split of the RoPE dims."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "kv_fp8_worked.txt")


def _worked():
    vals = {"k": np.zeros((2, 128)), "v": np.zeros((1, 128))}
    expect, scales = [], []
    for ln in open(GOLD):
        ln = ln.split("#")[0].split()
        if not ln:
            continue
        if ln[0] == "scale":
            scales.append((ln[1], int(ln[2]), int(ln[3]), int(ln[4])))
            continue
        kind, r, c, x, code, deq = ln[0], int(ln[1]), int(ln[2]), float(ln[3]), int(ln[4], 16), float(ln[5])
        vals[kind][r, c] = x
        expect.append((kind, r, c, code, deq))
    return vals, expect, scales


def test_worked_example():
    vals, expect, scales = _worked()
    out = {"k": oracle.quant_kv_fp8(vals["k"], 64), "v": oracle.quant_kv_fp8(vals["v"], 0)}
    deq = {"k": oracle.dequant_kv_fp8(*out["k"], 128), "v": oracle.dequant_kv_fp8(*out["v"], 128)}
    for kind, r, c, code, d in expect:
        codes, _, keep = out[kind]
        got = codes[r, c] if c < codes.shape[1] else keep[r, c - codes.shape[1]]
        assert got == code, (kind, r, c, hex(got), hex(code))
        assert deq[kind][r, c] == d, (kind, r, c, deq[kind][r, c], d)
    for kind, r, b, byte in scales:
        assert out[kind][1][r, b] == byte, (kind, r, b)
    # the unlisted values are zero and stay zero
    listed = {(k, r, c) for k, r, c, _, _ in expect}
    for kind in ("k", "v"):
        for r in range(vals[kind].shape[0]):
            for c in range(128):
                if (kind, r, c) not in listed:
                    assert deq[kind][r, c] == 0.0


@pytest.mark.parametrize("e", [-20, -7, 0, 5])
def test_scale_is_the_smallest_power_of_two_that_fits(e):
    x = np.zeros((3, 64))
    x[0, 9] = 448.0 * 2.0 ** e                        # exactly at the bound: e itself, max code 7E
    x[1, 9] = np.float32(448.0 * 2.0 ** e) * (1 + 2 ** -20)   # just above (in float32): e + 1
    x[2, 9] = 449.0 * 2.0 ** (e - 1)                  # above 448 * 2^(e-1): e
    codes, sc, _ = oracle.quant_kv_fp8(x, 0)
    assert list(sc[:, 0]) == [e + 127, e + 128, e + 127]
    assert codes[0, 9] == 0x7E
    assert not codes[:, :9].any() and not codes[:, 10:].any()


def test_codes_match_torch_float8_cast_of_the_scaled_values():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 192)) * np.exp(rng.uniform(-12, 12, size=(64, 1)))
    x[5] = 0.0
    x[7, :64] = 0.0                                    # one zero block beside a non-zero one
    codes, sc, keep = oracle.quant_kv_fp8(x, 64)
    x32 = x.astype(np.float32).astype(np.float64)
    for b in range(2):
        e = sc[:, b].astype(np.int64) - 127
        y = torch.from_numpy(x32[:, 64 * b: 64 * b + 64] * np.ldexp(1.0, -e)[:, None])
        ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(codes[:, 64 * b: 64 * b + 64], ref)
    assert sc[5, 0] == 127 and sc[7, 0] == 127 and not codes[7, :64].any()
    ref_bf16 = torch.from_numpy(x[:, 128:].astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    np.testing.assert_array_equal(keep.view(np.int16), ref_bf16)


def test_representable_values_survive_and_the_error_is_half_a_step():
    rng = np.random.default_rng(4)
    # values code * 2^e come back exactly
    e = rng.integers(-30, 10, size=(16, 1))
    codes = rng.integers(0, 0x7F, size=(16, 64)).astype(np.uint8)      # no NaN code
    codes[:, 0] = 0x7E                                 # amax 448 * 2^e: the scale is 2^e
    x = np.array([[oracle.e4m3_decode(int(c)) for c in row] for row in codes]) * np.ldexp(1.0, e)
    c2, s2, _ = oracle.quant_kv_fp8(x, 0)
    np.testing.assert_array_equal(s2[:, 0], (e[:, 0] + 127).astype(np.uint8))
    np.testing.assert_array_equal(oracle.dequant_kv_fp8(c2, s2, None, 64), x)
    # anything else: within half an E4M3 step of its scaled value
    y = rng.standard_normal((32, 64)) * 10.0
    c3, s3, _ = oracle.quant_kv_fp8(y, 0)
    deq = oracle.dequant_kv_fp8(c3, s3, None, 64)
    ee = s3[:, :1].astype(np.int64) - 127
    z = np.abs(y.astype(np.float32).astype(np.float64)) * np.ldexp(1.0, -ee)
    step = np.where(z < 2.0 ** -6, 2.0 ** -9, np.ldexp(1.0, np.floor(np.log2(np.maximum(z, 2.0 ** -6))).astype(int) - 3))
    assert (np.abs(deq - y.astype(np.float32)) <= 0.5 * step * np.ldexp(1.0, ee) + 0.0).all()


def test_only_the_last_64_dims_of_k_stay_bf16():
    x = np.zeros((1, 128))
    x[0, :64] = 1000.0                                 # a large block: its small values flush
    x[0, 1] = 1e-3
    x[0, 64:] = 1e-3                                   # RoPE dims: BF16 keeps them
    codes, sc, keep = oracle.quant_kv_fp8(x, 64)
    deq = oracle.dequant_kv_fp8(codes, sc, keep, 128)
    assert deq[0, 1] == 0.0 and deq[0, 0] == 1024.0    # 1000 -> 1024 at scale 2^2 (grid 64)
    bf = float(torch.tensor(1e-3, dtype=torch.float32).to(torch.bfloat16).float())
    assert (deq[0, 64:] == bf).all()
    cv, sv, _ = oracle.quant_kv_fp8(x, 0)              # a V row: all 128 dims in FP8
    assert cv.shape == (1, 128) and sv.shape == (1, 2)
    # block 1: amax 1e-3 <= 448 * 2^-18 (> 448 * 2^-19): e = -18; 1e-3 * 2^18 = 262.1 -> 256 (grid 32)
    assert sv[0, 1] == 127 - 18
    assert (oracle.dequant_kv_fp8(cv, sv, None, 128)[0, 64:] == 2.0 ** -10).all()
