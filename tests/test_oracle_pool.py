"""Pins for the oracle's softmax-gated pooling (compression of m tokens into one entry).

Method: pogovet.com DeepSeek-V4 article, detail 4 (m=4 softmax-gated pooling with a learned
position bias; HCA m=128); honbul.tistory.com/221 sections "CSA" and "HCA".
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.golden import load


def test_worked_example_two_blocks():
    g = load("pool_m4_worked.txt")
    m, d = int(g["m"][0]), int(g["d"][0])
    x = np.array(g["x"], dtype=np.float32).reshape(-1, d)
    out, alpha = oracle.pool(x, np.array(g["gate"], np.float32), np.array(g["bias"], np.float32), m)
    np.testing.assert_allclose(alpha.ravel(), g["alpha"], rtol=1e-6)
    np.testing.assert_allclose(out.ravel(), g["expected"], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("m", [1, 4, 128])
def test_constant_block_pools_to_constant(m):
    rng = np.random.default_rng(1)
    d, nb = 16, 5
    const = rng.standard_normal((nb, d)).astype(np.float32)
    x = np.repeat(const, m, axis=0)
    gate = rng.standard_normal(nb * m).astype(np.float32) * 3
    bias = rng.standard_normal(m).astype(np.float32)
    out, alpha = oracle.pool(x, gate, bias, m)
    np.testing.assert_allclose(out, const, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(alpha.sum(1), 1.0, rtol=0, atol=1e-14)
    assert (alpha > 0).all()


def test_m1_is_identity():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((37, 8)).astype(np.float32)
    out, alpha = oracle.pool(x, np.zeros(37, np.float32), np.zeros(1, np.float32), 1)
    np.testing.assert_array_equal(out, x.astype(np.float64))
    np.testing.assert_array_equal(alpha, 1.0)


def test_bias_is_per_slot_not_per_block():
    # A dominant bias on slot 0 selects the first token of EVERY block.
    rng = np.random.default_rng(3)
    m, nb, d = 4, 6, 8
    x = rng.standard_normal((m * nb, d)).astype(np.float32)
    gate = rng.standard_normal(m * nb).astype(np.float32)
    bias = np.array([200.0, 0.0, 0.0, 0.0], np.float32)
    out, _ = oracle.pool(x, gate, bias, m)
    np.testing.assert_allclose(out, x[0::m].astype(np.float64), rtol=0, atol=1e-12)
    bias2 = np.array([0.0, 0.0, 200.0, 0.0], np.float32)
    out2, _ = oracle.pool(x, gate, bias2, m)
    np.testing.assert_allclose(out2, x[2::m].astype(np.float64), rtol=0, atol=1e-12)


@pytest.mark.parametrize("m", [4, 128])
def test_matches_library_softmax_per_block(m):
    # Reduces to torch.softmax (library) followed by a weighted sum, block by block.
    rng = np.random.default_rng(4)
    nb, d = 3, 24
    x = rng.standard_normal((m * nb, d)).astype(np.float32)
    gate = rng.standard_normal(m * nb).astype(np.float32)
    bias = (0.5 * rng.standard_normal(m)).astype(np.float32)
    out, _ = oracle.pool(x, gate, bias, m)
    z = torch.from_numpy(gate.astype(np.float64)).view(nb, m) + torch.from_numpy(bias.astype(np.float64))
    a = torch.softmax(z, dim=-1)
    ref = torch.einsum("ji,jid->jd", a, torch.from_numpy(x.astype(np.float64)).view(nb, m, d))
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_bf16_input_and_rounding():
    rng = np.random.default_rng(5)
    x32 = rng.standard_normal((8, 4)).astype(np.float32)
    xb = torch.from_numpy(x32).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_to_f64(bits), xb.to(torch.float64).numpy())
    out, _ = oracle.pool(bits, np.zeros(8, np.float32), np.zeros(4, np.float32), 4)
    np.testing.assert_allclose(out, xb.to(torch.float64).view(2, 4, 4).mean(1).numpy(), rtol=1e-15)
    # round-to-nearest-even to bf16 agrees with torch's (library) conversion
    vals = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                           [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1e-40, -3e-39]])
    mine = oracle.round_bf16(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, ref)


@pytest.mark.parametrize("L,m", [(4099, 4), (4096, 128), (1 << 20, 128), (127, 128)])
def test_compressed_bytes_closed_form(L, m):
    # Compressed K and V cache bytes = 2 * floor(L/m) * d * sizeof(storage dtype).
    d = 8
    n = L // m
    x = np.zeros((L, d), np.uint16)
    gate = np.zeros(L, np.float32)
    ck, cv = oracle.compress(x, x, gate, np.zeros(m, np.float32), m, oracle.BF16)
    assert ck.nbytes + cv.nbytes == 2 * math.floor(L / m) * d * 2 == 2 * n * d * 2
