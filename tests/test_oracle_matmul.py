"""Pins for the oracle's fused decode + product reference (CPU only).

y[m, n] = sum_k X[m, k] * W[n, k] with W = DequantizePacked(w, [N, K], T),
T FLOAT or BFLOAT16, and bfloat16 activations X, summed in binary64.

* One-hot activation rows pick single decoded weights (the index wiring:
  W is [N, K], the product contracts K).
* Integer weights and activations reduce the product to numpy's exact
  int64 matrix product (q8_0 and q4_0 with unit scales).
* Rows of X are independent, yabs bounds |y|, and empty extents give
  empty or zero results.
"""
import numpy as np
import pytest
import torch

import synth

BF16_ONE = 0x3F80


def bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("fmt", ["gguf:q4_k", "gguf:q6_k", "gguf:iq2_xs", "nvfp4", "fp8_e4m3fn_row_fp16"])
@pytest.mark.parametrize("weights", ["bfloat16", "float32"])
def test_one_hot_rows_pick_decoded_weights(orc, fmt, weights):
    B = synth.GEOMETRY[fmt][0]
    N, K = 5, 2 * max(B, 32)
    w = synth.payload(fmt, (N, K), seed=3)
    dec = orc.decode(fmt, (N, K), w, weights)
    W = (bf16_values(dec) if weights == "bfloat16" else dec).astype(np.float64)
    ks = [0, 1, K // 2 + 3, K - 1]
    x = np.zeros((len(ks), K), np.uint16)
    for m, k in enumerate(ks):
        x[m, k] = BF16_ONE
    y, yabs = orc.matmul_packed(fmt, N, K, w, x, weights)
    for m, k in enumerate(ks):
        assert np.array_equal(y[m], W[:, k]), (fmt, k)
        assert np.array_equal(yabs[m], np.abs(W[:, k]))


@pytest.mark.parametrize("fmt,lo,hi", [("gguf:q8_0", -127, 128), ("gguf:q4_0", 0, 16)])
def test_integer_case_is_numpy_int_matmul(orc, fmt, lo, hi):
    rng = np.random.default_rng(5)
    N, K, M = 7, 96, 3
    B, S = synth.GEOMETRY[fmt]
    blk = synth.payload(fmt, (N, K), seed=1).reshape(-1, S).copy()
    blk[:, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)  # d = 1
    if fmt == "gguf:q8_0":
        codes = blk[:, 2:].view(np.int8).astype(np.int64).reshape(N, K)
    else:  # P(q,4,16): 16 low nibbles, then 16 high nibbles, minus 8
        q = blk[:, 2:].astype(np.int64)
        codes = np.concatenate([q & 15, q >> 4], axis=1).reshape(N, K) - 8
    xi = rng.integers(-8, 9, size=(M, K))
    for weights in ("bfloat16", "float32"):
        y, _ = orc.matmul_packed(fmt, N, K, blk.reshape(-1), bf16_bits(xi), weights)
        assert np.array_equal(y, (xi @ codes.T).astype(np.float64))


def test_rows_of_x_are_independent(orc):
    fmt, N, K = "gguf:q5_k", 6, 512
    w = synth.payload(fmt, (N, K), seed=8)
    x = bf16_bits(np.random.default_rng(9).standard_normal((4, K)))
    y, yabs = orc.matmul_packed(fmt, N, K, w, x)
    for m in range(4):
        ym, ya = orc.matmul_packed(fmt, N, K, w, x[m:m + 1])
        assert np.array_equal(ym[0], y[m]) and np.array_equal(ya[0], yabs[m])
    assert (yabs >= np.abs(y)).all()


def test_empty_extents(orc):
    y, _ = orc.matmul_packed("gguf:q4_0", 0, 32, np.zeros(0, np.uint8), np.zeros((2, 32), np.uint16))
    assert y.shape == (2, 0)
    y, _ = orc.matmul_packed("gguf:q4_0", 3, 0, np.zeros(0, np.uint8), np.zeros((2, 0), np.uint16))
    assert y.shape == (2, 3) and not y.any()
