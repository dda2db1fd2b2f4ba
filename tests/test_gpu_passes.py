"""Input pass (pack) bit for bit and output pass (unpack) on the GPU against
the oracle, including NaN/Inf colour, clamp-to-edge padding and 1/2/3
sources."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from oracle import passes, tiles
from tests._gpu import Denoiser, ulp_diff_f32

import conv2d_implicit_gemm_gb300 as ox


def _images(w, h, sources, hdr, nan_fraction):
    imgs = synth.denoise_inputs(w, h, sources, hdr=hdr, nan_fraction=nan_fraction)
    if sources >= 3:
        imgs[2][0, 0, :3] = [np.nan, np.inf, -np.inf]   # normals get specials too
    if sources >= 2:
        imgs[1][0, 1, :3] = [np.nan, 2.0, -0.0]
    return imgs


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
@pytest.mark.parametrize("sources", [1, 2, 3])
@pytest.mark.parametrize("hdr", [True, False])
def test_pack_and_unpack_match_oracle(precision, sources, hdr):
    w, h = 150, 37                         # padded to 160 x 48: clamp-to-edge
    imgs = _images(w, h, sources, hdr, 0.05)
    scale = 0.75 if hdr else 1.0
    weights = synth.unet_weights(3 * sources, bias_scale=0.05)
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    d = Denoiser(weights, prec, imgs, hdr, input_scale=scale, keep=True)
    try:
        out = d.run()
        grid = tiles.plan_tile_grid(w, h, 0, 96)
        assert len(grid) == 1
        ix, iy, iw, ih = grid[0]["input"]
        packed = d.activation(0, ih, iw, 3 * sources)
        ref = passes.pack_tile(imgs, (ix, iy, iw, ih), hdr, scale, precision)
        assert np.array_equal(packed.view(np.uint32), ref.astype(np.float32).view(np.uint32))
        net = d.activation(16, ih, iw, 3)
    finally:
        d.close()
    ref_out = passes.unpack_rect(net[:h, :w], imgs[0], hdr, scale)
    assert np.array_equal(out[..., 3].view(np.uint32), imgs[0][..., 3].view(np.uint32))
    if hdr:
        fin = np.isfinite(ref_out[..., :3])
        assert np.array_equal(np.isfinite(out[..., :3]), fin)
        assert ulp_diff_f32(out[..., :3][fin], ref_out[..., :3][fin]).max() <= 8
    else:
        assert np.array_equal(out.view(np.uint32), ref_out.view(np.uint32))


def test_pack_hdr_transfer_is_correctly_rounded_everywhere():
    # dense sweep of colour values through the fp16 input pass: every code
    # must equal the correctly rounded fp16 of log2(1 + x)
    w, h = 512, 64
    vals = np.logspace(-9, 6, w * h * 3).astype(np.float32)
    color = np.ones((h, w, 4), np.float32)
    color[..., :3] = vals.reshape(h, w, 3)
    imgs = [color, synth.albedo(w, h), synth.normal(w, h)]
    d = Denoiser(synth.unet_weights(9), ox.PRECISION_FP16, imgs, True, keep=True)
    try:
        d.run()
        packed = d.activation(0, h, w, 9)
    finally:
        d.close()
    ref = passes.pack_tile(imgs, (0, 0, w, h), True, 1.0, "fp16")
    assert np.array_equal(packed[..., :3].view(np.uint32),
                          ref[..., :3].astype(np.float32).view(np.uint32))
