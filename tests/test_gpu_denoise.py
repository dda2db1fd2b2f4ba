"""Whole denoise on the GPU against the oracle for the four image workloads:
128x128 fp32 (full image), 1920x1080 fp16 (single tile), 3840x2160 fp16
tiled (maxTileSize 1024, overlap 96), 3840x2160 fp32 LDR colour-only with 5%
NaN/Inf.  Full-size runs are checked on 16-aligned crops that the oracle can
afford: with a margin of the default overlap (96 >= the network's dependency
radius 94) the oracle's output on a crop equals the full-frame output in the
crop's interior, so the interior is compared pixel by pixel."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from oracle import passes, unet
from oracle.numerics import FLT_MAX, sanitize
from tests._gpu import Denoiser, rel_l2

import conv2d_implicit_gemm_gb300 as ox

MARGIN = 96


def _crop_check(net_gpu, imgs, weights, precision, hdr, scale, crop, tile_w, tile_h, tol):
    cx, cy, cw, ch = crop
    packed = passes.pack_tile(imgs, crop, hdr, scale, precision)
    ref = unet.forward(packed, weights, precision)
    ml = 0 if cx == 0 else MARGIN
    mt = 0 if cy == 0 else MARGIN
    mr = 0 if cx + cw == tile_w else MARGIN
    mb = 0 if cy + ch == tile_h else MARGIN
    r = ref[mt:ch - mb, ml:cw - mr]
    g = net_gpu[cy + mt:cy + ch - mb, cx + ml:cx + cw - mr]
    assert r.size > 0
    if precision == "fp16":
        top = FLT_MAX if hdr else 1.0
        diff = np.abs(sanitize(g, 0, top).astype(np.float64) - sanitize(r, 0, top))
        assert diff.max() <= tol, diff.max()
    else:
        assert rel_l2(g, r) <= tol


def test_config_128x128_fp32_full_image():
    w = h = 128
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9)
    d = Denoiser(weights, ox.PRECISION_FP32, imgs, True, keep=True)
    try:
        out = d.run()
        net = d.activation(16, h, w, 3)
    finally:
        d.close()
    ref = unet.denoise(imgs, weights, hdr=True, precision="fp32")
    ref_net = unet.forward(passes.pack_tile(imgs, (0, 0, w, h), True, 1.0, "fp32"),
                           weights, "fp32")
    # the stated fp32 bound applies to the network (per layer, and here to its
    # output); the output pass F^-1(y) = 2^y - 1 scales relative errors by its
    # condition number y ln2 / (1 - 2^-y), so the image gets that factor
    assert rel_l2(net, ref_net) <= 1e-4
    y = np.clip(ref_net.astype(np.float64), 1e-6, None)
    kappa = float((y * np.log(2.0) / (1.0 - 2.0 ** -y)).max())
    assert rel_l2(out[..., :3], ref[..., :3]) <= 1e-4 * kappa
    assert np.array_equal(out[..., 3].view(np.uint32), imgs[0][..., 3].view(np.uint32))


def test_config_1080p_fp16_single_tile():
    w, h = 1920, 1080
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9)
    # keep=True: the network output is read back (with the output pass in
    # the final conv's epilogue it is not stored otherwise)
    d = Denoiser(weights, ox.PRECISION_FP16, imgs, True, keep=True)
    try:
        out = d.run()
        assert ox.oidnx_filter_get_int(d.f, "tiles") == 1
        net = d.activation(16, 1088, 1920, 3)
    finally:
        d.close()
    assert np.isfinite(out[..., :3]).all()
    for crop in [(0, 0, 256, 256), (832, 416, 256, 256), (1664, 832, 256, 256)]:
        _crop_check(net, imgs, weights, "fp16", True, 1.0, crop, 1920, 1088, 2e-2)
    # final HDR image on one interior window
    ref = unet.denoise([im[400:656, 800:1056] for im in imgs], weights, hdr=True)
    got = out[400 + MARGIN:656 - MARGIN, 800 + MARGIN:1056 - MARGIN, :3]
    assert rel_l2(got, ref[MARGIN:-MARGIN, MARGIN:-MARGIN, :3]) <= 2e-2


def test_config_4k_fp16_tiled_equals_single_tile():
    w, h = 3840, 2160
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9)
    d = Denoiser(weights, ox.PRECISION_FP16, imgs, True, max_tile_size=1024)
    try:
        tiled = d.run()
        assert ox.oidnx_filter_get_int(d.f, "tiles") == 15
    finally:
        d.close()
    d = Denoiser(weights, ox.PRECISION_FP16, imgs, True, max_tile_size=0, keep=True)
    try:
        whole = d.run()
        net = d.activation(16, 2160, 3840, 3)   # 2160 is already 16-aligned
    finally:
        d.close()
    assert np.array_equal(tiled.view(np.uint32), whole.view(np.uint32))
    _crop_check(net, imgs, weights, "fp16", True, 1.0, (2144, 1008, 256, 256), 3840, 2160, 2e-2)


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
@pytest.mark.parametrize("w,h", [(1, 1), (1, 37), (37, 1), (17, 5)])
def test_degenerate_image_shapes_match_oracle(w, h, precision):
    """One-pixel, one-row and one-column images through the whole filter
    path: the tile is padded to 16 x 16 with clamp-to-edge reads, and the
    output pass writes only the image's pixels."""
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9, bias_scale=0.05)
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    d = Denoiser(weights, prec, imgs, True)
    try:
        out = d.run()
    finally:
        d.close()
    ref = unet.denoise(imgs, weights, hdr=True, precision=precision)
    assert np.array_equal(out[..., 3].view(np.uint32), imgs[0][..., 3].view(np.uint32))
    if precision == "fp16":
        assert rel_l2(out[..., :3], ref[..., :3]) <= 2e-2
    else:
        assert rel_l2(out[..., :3], ref[..., :3]) <= 3e-4   # 1e-4 on the network output x kappa


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
def test_tiled_denoise_matches_oracle_tiled_denoise(precision):
    """A ragged tile grid (500 x 300, maxTileSize 256, overlap 96) against the
    oracle's own tiled denoise: the same tile rectangles, per-tile input and
    output passes and stitching, with inputScale != 1."""
    w, h = 500, 300
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9, bias_scale=0.05)
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    d = Denoiser(weights, prec, imgs, True, input_scale=0.8, max_tile_size=256, overlap=96)
    try:
        out = d.run()
        tiles = ox.oidnx_filter_get_int(d.f, "tiles")
    finally:
        d.close()
    ref = unet.denoise(imgs, weights, hdr=True, input_scale=0.8, max_tile_size=256, overlap=96,
                       precision=precision)
    assert tiles > 4
    assert np.array_equal(out[..., 3].view(np.uint32), imgs[0][..., 3].view(np.uint32))
    if precision == "fp16":
        assert rel_l2(out[..., :3], ref[..., :3]) <= 2e-2
    else:
        assert rel_l2(out[..., :3], ref[..., :3]) <= 3e-4   # 1e-4 on the network output x kappa


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
def test_stacked_tile_groups_equal_tile_by_tile(precision):
    """A 10-tile frame (ragged edges) denoised tile by tile (stackTiles 1), in
    stacks of at most 4 and 3 tiles (a partial last group each: 4 + 4 + 2 and
    3 + 3 + 3 + 1) and as one stack (0: the memory budget allows all ten):
    the same bits, since every conv sees the same zero padding at a tile's
    edges whether it comes from the image border or the gap rows."""
    w, h = 300, 120
    imgs = synth.denoise_inputs(w, h, 3, hdr=True, nan_fraction=0.02)
    weights = synth.unet_weights(9, bias_scale=0.05)
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    outs = []
    for stack, expect in ((1, 1), (4, 4), (3, 3), (0, 10)):
        d = Denoiser(weights, prec, imgs, True, input_scale=0.9, max_tile_size=224, overlap=96)
        try:
            ox.oidnx_filter_set_int(d.f, "stackTiles", stack)
            ox.oidnx_filter_commit(d.f)
            assert ox.oidnx_filter_get_int(d.f, "tiles") == 10
            assert ox.oidnx_filter_get_int(d.f, "stackedTiles") == expect
            outs.append(d.run())
            outs.append(d.run())   # graph replay
        finally:
            d.close()
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def test_8k_single_tile_with_activations_over_4gib():
    """8192 x 8192 as one tile: dec_conv1a's fp16 output alone is 8 GiB, so
    the 64-bit offsets of every kernel are exercised.  The output image is
    checked on an interior window and on the bottom-right corner window
    (whose image-edge sides need no margin) against the oracle."""
    w = h = 8192
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9)
    d = Denoiser(weights, ox.PRECISION_FP16, imgs, True, max_tile_size=0)
    try:
        out = d.run()
        assert ox.oidnx_filter_get_int(d.f, "tiles") == 1
    finally:
        d.close()
    assert np.isfinite(out[..., :3]).all()
    for y0, x0, edge in [(4000, 4000, False), (h - 256, w - 256, True)]:
        ref = unet.denoise([im[y0:y0 + 256, x0:x0 + 256] for im in imgs], weights, hdr=True)
        end = 256 if edge else 256 - MARGIN
        got = out[y0 + MARGIN:y0 + end, x0 + MARGIN:x0 + end, :3]
        assert rel_l2(got, ref[MARGIN:end, MARGIN:end, :3]) <= 2e-2


def test_config_4k_fp32_ldr_color_only_nan_inf():
    w, h = 3840, 2160
    imgs = synth.denoise_inputs(w, h, 1, hdr=False, nan_fraction=0.05)
    weights = synth.unet_weights(3)
    d = Denoiser(weights, ox.PRECISION_FP32, imgs, False, keep=True)
    try:
        out = d.run()
        net = d.activation(16, 2160, 3840, 3)
    finally:
        d.close()
    assert np.isfinite(out).sum() == out[..., :3].size + np.isfinite(imgs[0][..., 3]).sum()
    assert (out[..., :3] >= 0).all() and (out[..., :3] <= 1).all()
    _crop_check(net, imgs, weights, "fp32", False, 1.0, (3584, 1904, 256, 256), 3840, 2160, 1e-4)
    ref = passes.unpack_rect(net[:h, :w], imgs[0], False, 1.0)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
def test_subpixel_decoder_denoise_matches_oracle(precision):
    """Sub-pixel decoder mode (the default) against the expansion mode and the
    oracle through the whole filter path (the input pass and the pool
    epilogues also write the parity-split skip copies)."""
    w, h = 400, 272
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9, bias_scale=0.05)
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    ref = unet.forward(passes.pack_tile(imgs, (0, 0, w, h), True, 1.0, precision), weights, precision)
    outs = []
    for mode in (0, 1):
        d = Denoiser(weights, prec, imgs, True, keep=True)
        try:
            ox.oidnx_filter_set_int(d.f, "subpixelDecoder", mode)
            ox.oidnx_filter_commit(d.f)
            outs.append(d.run())
            net = d.activation(16, 272, 400, 3)
        finally:
            d.close()
        if precision == "fp16":
            diff = np.abs(sanitize(net, 0, FLT_MAX).astype(np.float64) - sanitize(ref, 0, FLT_MAX))
            assert diff.max() <= 2e-2
        else:
            assert rel_l2(net, ref) <= 1e-4
    if precision == "fp16":
        assert rel_l2(outs[1][..., :3], outs[0][..., :3]) <= 2e-2
    else:
        # both within 1e-4 of the oracle's network output; the output pass
        # scales relative errors by at most kappa = max y ln2 / (1 - 2^-y)
        y = np.clip(ref.astype(np.float64), 1e-6, None)
        kappa = float((y * np.log(2.0) / (1.0 - 2.0 ** -y)).max())
        ref_out = passes.unpack_rect(ref, imgs[0], True, 1.0)
        for out in outs:
            assert rel_l2(out[..., :3], ref_out[..., :3]) <= 1e-4 * kappa


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
@pytest.mark.parametrize("hdr", [True, False])
def test_output_pass_in_final_conv_equals_separate_pass(hdr, precision):
    """The output pass run in the final conv's epilogue gives the bits of the
    separate output pass kernel, over a tile grid with ragged edges (so the
    output rectangles are offset inside their tiles)."""
    w, h = 700, 430
    imgs = synth.denoise_inputs(w, h, 3, hdr=hdr, nan_fraction=0.02)
    weights = synth.unet_weights(9, bias_scale=0.05)
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    outs = []
    for fuse in (1, 0):
        d = Denoiser(weights, prec, imgs, hdr, input_scale=0.7 if hdr else 1.0,
                     max_tile_size=256, overlap=96)
        try:
            ox.oidnx_filter_set_int(d.f, "fuseOutput", fuse)
            ox.oidnx_filter_commit(d.f)
            assert ox.oidnx_filter_get_int(d.f, "tiles") > 4
            outs.append(d.run())
        finally:
            d.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0][..., 3].view(np.uint32), imgs[0][..., 3].view(np.uint32))
