"""Pins of the oracle's layers: torch CPU float64 library routines, closed
forms (identity / shifted-delta / zero kernels), linearity, pool/upsample
invariants."""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import layers


def _torch_conv(x, w, b, relu):
    t = torch.from_numpy(np.ascontiguousarray(x.transpose(2, 0, 1)))[None]
    y = F.conv2d(t, torch.from_numpy(w), torch.from_numpy(b), padding=1)
    if relu:
        y = torch.relu(y)
    return y[0].numpy().transpose(1, 2, 0)


@pytest.mark.parametrize("seed", range(12))
def test_conv_matches_torch_conv2d(seed):
    rng = np.random.default_rng(seed)
    h, w = rng.integers(1, 8, size=2)
    cin, cout = rng.integers(1, 10, size=2)
    x = rng.standard_normal((h, w, cin))
    wt = rng.standard_normal((cout, cin, 3, 3))
    b = rng.standard_normal(cout)
    for relu in (False, True):
        got = layers.conv3x3(x, wt, b, relu)
        ref = _torch_conv(x, wt, b, relu)
        assert got.shape == (h, w, cout)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_conv_identity_kernel_is_relu():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 5, 4))
    wt = np.zeros((4, 4, 3, 3))
    for c in range(4):
        wt[c, c, 1, 1] = 1.0
    out = layers.conv3x3(x, wt, np.zeros(4), relu=True)
    assert np.array_equal(out, np.maximum(x, 0.0))


@pytest.mark.parametrize("ky,kx", [(ky, kx) for ky in range(3) for kx in range(3)])
def test_conv_shifted_delta_is_shift_with_zero_fill(ky, kx):
    rng = np.random.default_rng(2)
    h, w, c = 5, 7, 3
    x = rng.standard_normal((h, w, c))
    wt = np.zeros((c, c, 3, 3))
    for i in range(c):
        wt[i, i, ky, kx] = 1.0
    out = layers.conv3x3(x, wt, np.zeros(c), relu=False)
    expected = np.zeros_like(x)
    for y in range(h):
        for xx in range(w):
            sy, sx = y + ky - 1, xx + kx - 1
            if 0 <= sy < h and 0 <= sx < w:
                expected[y, xx] = x[sy, sx]
    assert np.array_equal(out, expected)


def test_conv_linearity_without_relu():
    rng = np.random.default_rng(3)
    x1 = rng.standard_normal((7, 6, 5))
    x2 = rng.standard_normal((7, 6, 5))
    wt = rng.standard_normal((4, 5, 3, 3))
    b = rng.standard_normal(4)
    a1, a2 = 0.7, -1.3
    lhs = layers.conv3x3(a1 * x1 + a2 * x2, wt, b, False) - b
    rhs = a1 * (layers.conv3x3(x1, wt, b, False) - b) + a2 * (layers.conv3x3(x2, wt, b, False) - b)
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-12)


def test_conv_zero_weights_gives_relu_bias():
    b = np.array([-1.0, 0.5, 2.0])
    out = layers.conv3x3(np.ones((3, 4, 2)), np.zeros((3, 2, 3, 3)), b, relu=True)
    assert np.array_equal(out, np.broadcast_to(np.maximum(b, 0), (3, 4, 3)))


@pytest.mark.parametrize("h,w", [(1, 1), (2, 2), (3, 5), (4, 7), (8, 8), (9, 6)])
def test_pool_matches_torch_ceil_mode(h, w):
    rng = np.random.default_rng(h * 31 + w)
    x = rng.standard_normal((h, w, 3))
    got = layers.maxpool2x2(x)
    t = torch.from_numpy(np.ascontiguousarray(x.transpose(2, 0, 1)))[None]
    ref = F.max_pool2d(t, 2, 2, ceil_mode=True)[0].numpy().transpose(1, 2, 0)
    assert got.shape == ((h + 1) // 2, (w + 1) // 2, 3)
    assert np.array_equal(got, ref)


def test_upsample_and_pool_invariants():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 6, 2))
    up = layers.upsample2x(x, 10, 12)
    for y in range(5):
        for xx in range(6):
            for py in range(2):
                for px in range(2):
                    assert np.array_equal(up[2 * y + py, 2 * xx + px], x[y, xx])
    assert np.array_equal(layers.maxpool2x2(up), x)
    t = torch.from_numpy(np.ascontiguousarray(x.transpose(2, 0, 1)))[None]
    ref = F.interpolate(t, scale_factor=2, mode="nearest")[0].numpy().transpose(1, 2, 0)
    assert np.array_equal(up, ref)
    # cropped (odd target) keeps the top-left part
    assert np.array_equal(layers.upsample2x(x, 9, 11), up[:9, :11])


def test_decoder_input_channel_order():
    low = np.full((2, 2, 3), 7.0)
    skip = np.full((4, 3, 2), -1.0)
    cat = layers.decoder_input(low, skip)
    assert cat.shape == (4, 3, 5)
    assert (cat[..., :3] == 7.0).all() and (cat[..., 3:] == -1.0).all()
