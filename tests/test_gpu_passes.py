"""Input pass (pack) bit for bit and output pass (unpack) on the GPU against
the oracle, including NaN/Inf colour, clamp-to-edge padding and 1/2/3
sources."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from oracle import passes, tiles
from oracle.numerics import hdr_inverse_exact
from tests._gpu import Denoiser, empty_dev, stream, to_dev, to_host

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
    # HDR: (2^d - 1) / inputScale correctly rounded, as the oracle's single
    # rounding of its float64 value; LDR and alpha: copies and clamps
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


def _near_inverse_midpoints(n, scale, lo_rel, hi_rel, seed):
    """Network outputs d whose (2^d - 1) / scale lies between lo_rel and
    hi_rel (relative) from a rounding boundary between two fp32 values: the
    inputs a pair evaluation must hand to its exact fallback.  lo_rel keeps
    them far enough from the boundary that the oracle's float64 value
    (within 2^-50) decides them."""
    rng = np.random.default_rng(seed)
    d = np.concatenate([2.0 ** rng.uniform(-60, 6.97, n), rng.uniform(0, 8, n)]).astype(np.float32)
    with np.errstate(over="ignore"):
        f = hdr_inverse_exact(d) / np.float64(scale)
        y = f.astype(np.float32)
    ok = np.isfinite(y) & (y > 0)
    d, f, y = d[ok], f[ok], y[ok]
    other = np.nextafter(y, np.where(f > y, np.float32(np.inf), np.float32(0)))
    dist = np.abs(f - (y.astype(np.float64) + other.astype(np.float64)) / 2) / f
    return d[(dist < hi_rel) & (dist > lo_rel)]


@pytest.mark.parametrize("scale", [1.0, 0.75, 3.0, 2.0 ** -20, 1e-30, 1e30, 0.0])
def test_output_pass_hdr_is_correctly_rounded(scale):
    """Output pass alone on a dense sweep of network outputs: every HDR value
    must be the correctly rounded fp32 of (2^d - 1) / inputScale (the oracle's
    float64 value rounded once), alpha copied bit for bit; specials (NaN,
    +-Inf, negatives, -0, subnormals, FLT_MAX) sanitized first."""
    f32max = np.finfo(np.float32).max
    specials = np.array([np.nan, np.inf, -np.inf, -1.0, -0.0, 0.0, 2.0 ** -149, 2.0 ** -126,
                         2.0 ** -61, 2.0 ** -60, 2.0 ** -9, 1.0 / 512, 0.5, 1.0, 2.0, 125.99,
                         126.0, 127.0, 127.9999, 128.0, 150.0, 1023.0, 1025.0, f32max], np.float32)
    eff = 1.0 if scale == 0.0 else scale
    hard = _near_inverse_midpoints(1 << 20, np.float32(eff), 2.0 ** -46, 2.0 ** -36, 11)
    assert hard.size > 50
    rng = np.random.default_rng(5)
    vals = np.concatenate([specials,
                           np.logspace(-45, 2.2, 60000).astype(np.float32),
                           rng.uniform(0, 1, 30000).astype(np.float32),
                           rng.uniform(0, 20, 30000).astype(np.float32), hard])
    w = 256
    h = -(-vals.size // w)
    net = np.zeros((h, w, 4), np.float32)
    net.reshape(-1, 4)[:, 0] = np.resize(vals, h * w)
    net.reshape(-1, 4)[:, 1] = np.resize(vals[::-1], h * w)
    net.reshape(-1, 4)[:, 2] = np.resize(np.roll(vals, 7), h * w)
    color = synth.hdr_color(w, h)
    f = ox.oidnx_filter_create(ox.write_weight_blob(synth.unet_weights(9)), ox.PRECISION_FP16)
    try:
        d_net, d_col, d_out = to_dev(net), to_dev(color), empty_dev(w * h * 16)
        for hdr in (1, 0):
            d_out.fill_(0xFF)
            ox.oidnx_output_pass(f, d_net.data_ptr(), w, h, d_col.data_ptr(), d_out.data_ptr(),
                                 hdr, scale, stream())
            ox.oidnx_filter_sync_status(f)
            got = to_host(d_out, np.float32, (h, w, 4))
            ref = passes.unpack_rect(net, color, bool(hdr), scale)
            bad = np.flatnonzero(got.view(np.uint32) != ref.view(np.uint32))
            assert bad.size == 0, (hdr, bad.size, net.reshape(-1)[bad[:4]], got.reshape(-1)[bad[:4]],
                                   ref.reshape(-1)[bad[:4]])
    finally:
        ox.oidnx_filter_release(f)


def test_output_pass_rejects_bad_arguments():
    f = ox.oidnx_filter_create(ox.write_weight_blob(synth.unet_weights(9)), ox.PRECISION_FP16)
    try:
        buf = empty_dev(4096)
        p = buf.data_ptr()
        for args in [(0, 4, 0, 1, 1.0), (4, 4, 0, 2, 1.0), (4, 4, 0, 1, -1.0), (4, 4, 0, 1, float("nan")),
                     (4, 4, 32, 1, 1.0), (4, 70000, 0, 1, 1.0)]:
            w, h, stride, hdr, scale = args
            with pytest.raises(ox.OidnxError) as e:
                ox.oidnx_output_pass(f, p, w, h, p, p, hdr, scale, stream(), color_stride=stride)
            assert e.value.status == ox.ERR_INVALID_ARGUMENT
    finally:
        ox.oidnx_filter_release(f)
