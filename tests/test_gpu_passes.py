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



def _near_fp32_midpoints(n, rel, seed):
    """Colour values whose log2(1 + x) lies within rel (relative) of a
    rounding boundary between two fp32 codes: the hardest inputs for any
    evaluation that is not exact."""
    rng = np.random.default_rng(seed)
    x = np.concatenate([(10.0 ** rng.uniform(-18, 38, n)),
                        rng.uniform(0.0, 2.0 ** -9, n),
                        rng.uniform(0.0, 8.0, n)]).astype(np.float32)
    x = x[x > 0]
    f = np.log1p(x.astype(np.float64)) / np.log(2.0)
    y = f.astype(np.float32)
    other = np.nextafter(y, np.where(f > y, np.float32(np.inf), np.float32(0)))
    mid = (y.astype(np.float64) + other.astype(np.float64)) / 2
    return x[np.abs(f - mid) < rel * f]


def test_pack_hdr_transfer_fp32_is_correctly_rounded_everywhere():
    # fp32 input pass: every stored value must equal the correctly rounded
    # fp32 of log2(1 + x), over a dense sweep from subnormal colour to
    # FLT_MAX, the small-value range, the edges of the evaluation's ranges
    # and values whose F lies within 2^-36 of a rounding boundary
    f32max = np.finfo(np.float32).max
    edges = np.array([0.0, 2.0 ** -149, 2.0 ** -61, 2.0 ** -60, 2.0 ** -24, 2.0 ** -23,
                      2.0 ** -9, 2.0 ** -8, 0.5, 1.0, 2.0, 2.0 ** 24, 2.0 ** 24 + 2,
                      2.0 ** 25 + 4, 2.0 ** 126, 2.0 ** 127, f32max], np.float32)
    edges = np.concatenate([edges, np.nextafter(edges, np.float32(0)),
                            np.nextafter(edges, np.float32(np.inf))])
    edges = edges[np.isfinite(edges)]
    hard = _near_fp32_midpoints(1 << 20, 2.0 ** -36, 7)
    assert hard.size > 100
    vals = np.concatenate([np.logspace(-44, 38.5, 90000).astype(np.float32),
                           np.random.default_rng(3).uniform(0, 2.0 ** -8, 20000).astype(np.float32),
                           edges, hard])
    w = 512
    h = -(-vals.size // (3 * w * 16)) * 16   # a whole number of 16-row blocks: one tile
    flat = np.ones(w * h * 3, np.float32)
    flat[:vals.size] = vals
    color = np.ones((h, w, 4), np.float32)
    color[..., :3] = flat.reshape(h, w, 3)
    imgs = [color, synth.albedo(w, h), synth.normal(w, h)]
    d = Denoiser(synth.unet_weights(9), ox.PRECISION_FP32, imgs, True, keep=True)
    try:
        d.run()
        packed = d.activation(0, h, w, 9)
    finally:
        d.close()
    ref = passes.pack_tile(imgs, (0, 0, w, h), True, 1.0, "fp32")
    got = packed[..., :3].astype(np.float32)
    bad = np.flatnonzero(got.view(np.uint32) != ref[..., :3].astype(np.float32).view(np.uint32))
    assert bad.size == 0, (bad.size, flat[bad[:5]], got.reshape(-1)[bad[:5]],
                           ref[..., :3].reshape(-1)[bad[:5]])

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
