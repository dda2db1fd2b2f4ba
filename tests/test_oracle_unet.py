"""Pins of the oracle network and denoise: closed forms through each path
(bottom path, level-0 skip), translation equivariance on the 16-grid,
torch CPU float64 composition, tiled == untiled bit for bit."""

import numpy as np
import torch
import torch.nn.functional as F

import synth
from oracle import unet, tiles, passes


def _zero_weights(in_channels=9):
    shapes = synth.unet_shapes(in_channels)
    return {n: (np.zeros((co, ci, 3, 3), np.float32), np.zeros(co, np.float32))
            for n, (co, ci) in shapes.items()}


def test_final_bias_only_gives_constant_output():
    wts = _zero_weights()
    wts["dec_conv0"][1][:] = [0.25, -3.0, 7.5]
    x = np.random.default_rng(0).uniform(size=(32, 48, 9)).astype(np.float16)
    out = unet.forward(x, wts, "fp16")
    assert np.array_equal(out, np.broadcast_to(np.float32([0.25, -3.0, 7.5]), (32, 48, 3)))


def test_skip_path_at_full_resolution():
    # Only the level-0 skip of dec_conv1a carries input channel 4 through.
    wts = _zero_weights()
    w1a = wts["dec_conv1a"][0]
    w1a[0, 64 + 4, 1, 1] = 1.0          # skip channels follow the 64 upsampled ones
    wts["dec_conv1b"][0][0, 0, 1, 1] = 1.0
    for c in range(3):
        wts["dec_conv0"][0][c, 0, 1, 1] = 1.0
    x = np.random.default_rng(1).uniform(size=(16, 32, 9)).astype(np.float16)
    out = unet.forward(x, wts, "fp16")
    for c in range(3):
        assert np.array_equal(out[..., c], x[..., 4].astype(np.float32))


def test_bottom_path_carries_a_constant():
    # Centre deltas along channel 0 through every encoder conv, the bottom and
    # the upsampled part of every decoder conv: a constant input survives.
    wts = _zero_weights()
    for name in synth.UNET_LAYERS:
        wts[name][0][0, 0, 1, 1] = 1.0
    x = np.zeros((32, 32, 9), np.float16)
    x[..., 0] = 0.375
    out = unet.forward(x, wts, "fp16")
    # dec_conv0 centre delta only into channel 0
    assert np.array_equal(out[..., 0], np.full((32, 32), 0.375, np.float32))
    assert not out[..., 1:].any()


def _torch_unet(x, weights):
    """Composition of torch CPU float64 library ops (fp32 mode)."""
    t = torch.from_numpy(x.transpose(2, 0, 1).astype(np.float64))[None]
    W = {n: (torch.from_numpy(w.astype(np.float64)), torch.from_numpy(b.astype(np.float64)))
         for n, (w, b) in weights.items()}

    def c(n, v, relu=True):
        y = F.conv2d(v, W[n][0], W[n][1], padding=1)
        y = torch.relu(y) if relu else y
        return y.to(torch.float32).to(torch.float64)

    def p(v):
        return F.max_pool2d(v, 2, 2, ceil_mode=True)

    def up(v, skip):
        u = F.interpolate(v, scale_factor=2, mode="nearest")
        return torch.cat([u[..., :skip.shape[2], :skip.shape[3]], skip], dim=1)

    e = c("enc_conv1", c("enc_conv0", t))
    p1 = p(e)
    p2 = p(c("enc_conv2", p1))
    p3 = p(c("enc_conv3", p2))
    p4 = p(c("enc_conv4", p3))
    b = c("enc_conv5b", c("enc_conv5a", p4))
    d = c("dec_conv4b", c("dec_conv4a", up(b, p3)))
    d = c("dec_conv3b", c("dec_conv3a", up(d, p2)))
    d = c("dec_conv2b", c("dec_conv2a", up(d, p1)))
    d = c("dec_conv1b", c("dec_conv1a", up(d, t)))
    o = c("dec_conv0", d, relu=False)
    return o[0].numpy().transpose(1, 2, 0).astype(np.float32)


def test_network_matches_torch_composition_fp32():
    weights = synth.unet_weights(9, bias_scale=0.05)
    for h, w in ((32, 48), (20, 36)):   # second case has odd extents below level 2
        x = np.random.default_rng(h).uniform(size=(h, w, 9)).astype(np.float32)
        got = unet.forward(x, weights, "fp32")
        ref = _torch_unet(x, weights)
        assert got.shape == (h, w, 3)
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


def test_translation_equivariance_on_the_16_grid():
    weights = synth.unet_weights(9, bias_scale=0.05)
    x = np.random.default_rng(7).uniform(size=(48, 96, 9)).astype(np.float16)
    shifted = np.zeros_like(x)
    shifted[:, 16:] = x[:, :-16]
    a = unet.forward(x, weights, "fp16")
    b = unet.forward(shifted, weights, "fp16")
    # far from every border the output shifts with the input
    np.testing.assert_allclose(b[:, 16 + 40:-40], a[:, 40:-40 - 16], rtol=0, atol=1e-6)


def test_tiled_denoise_equals_single_tile_bitwise():
    weights = synth.unet_weights(9, bias_scale=0.05)
    w, h = 300, 70
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    whole = unet.denoise(imgs, weights, hdr=True, max_tile_size=0, precision="fp16")
    grid = tiles.plan_tile_grid(w, h, 256, 96)
    assert len(grid) >= 2
    tiled = unet.denoise(imgs, weights, hdr=True, max_tile_size=256, precision="fp16")
    assert np.array_equal(whole.view(np.uint32), tiled.view(np.uint32))


def test_conv_flops_of_the_1080p_tile():
    flops = unet.conv_flops(synth.unet_shapes(9), 1920, 1088)
    assert abs(flops / 1920 / 1088 - 250812) < 1  # per-pixel total, levels exact at /16
