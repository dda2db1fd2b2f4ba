"""The input pass fused into enc_conv0 on the GPU: the packed input of each
conv tile's halo is computed from the source images in shared memory, and
only its column-parity copy (dec_conv1a's skip source) is stored.  The
kernel uses the input pass's per-pixel code and sums enc_conv0's products
in the plain conv kernel's order, so every denoise must give the bits of
the separate input pass and enc_conv0 (themselves checked against the
oracle: bit-exact pack, per-layer conv checks), over 1-, 2- and 3-source
models, HDR and LDR, NaN/Inf inputs, input scales, extents that cut the
8-row x 128-pixel tiles raggedly, and tile grids run tile by tile."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from oracle import unet
from tests._gpu import Denoiser, rel_l2

import conv2d_implicit_gemm_gb300 as ox


def _denoise(weights, imgs, hdr, head, scale=1.0, max_tile=0, stack=0, keep=False, profile=False):
    d = Denoiser(weights, ox.PRECISION_FP16, imgs, hdr, input_scale=scale, max_tile_size=max_tile,
                 overlap=96, keep=keep)
    try:
        ox.oidnx_filter_set_int(d.f, "fuseInput", head)
        ox.oidnx_filter_set_int(d.f, "stackTiles", stack)
        ox.oidnx_filter_commit(d.f)
        assert ox.oidnx_filter_get_int(d.f, "fuseInput") == head
        if profile:
            ox.oidnx_profile_next(d.f)
        out = d.run()
        ids = [l["id"] for l in ox.oidnx_get_profile(d.f)["layers"]] if profile else None
    finally:
        d.close()
    return out, ids


@pytest.mark.parametrize("sources", [3, 2, 1])
@pytest.mark.parametrize("hdr", [True, False])
@pytest.mark.parametrize("w,h", [(64, 48), (700, 430), (130, 22), (2, 2)])
def test_head_denoise_equals_separate(sources, hdr, w, h):
    imgs = synth.denoise_inputs(w, h, sources, hdr=hdr, nan_fraction=0.02)
    weights = synth.unet_weights(3 * sources, bias_scale=0.05)
    scale = 0.7 if hdr else 1.0
    fused, ids = _denoise(weights, imgs, hdr, 1, scale, profile=True)
    plain, ids0 = _denoise(weights, imgs, hdr, 0, scale, profile=True)
    assert np.array_equal(fused.view(np.uint32), plain.view(np.uint32))
    assert "input-pack+enc_conv0" in ids and "input-pack" not in ids and "enc_conv0" not in ids
    assert "input-pack" in ids0 and "enc_conv0" in ids0
    if w * h <= 64 * 48 and sources == 3:
        ref = unet.denoise(imgs, weights, hdr=hdr, input_scale=scale)
        assert rel_l2(fused[..., :3], ref[..., :3]) <= 2e-2


def test_head_1080p_frame_equals_separate():
    w, h = 1920, 1080
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9)
    fused, _ = _denoise(weights, imgs, True, 1)
    plain, _ = _denoise(weights, imgs, True, 0)
    assert np.array_equal(fused.view(np.uint32), plain.view(np.uint32))


def test_head_tile_by_tile_equals_separate():
    """A tile grid run one tile at a time (stackTiles 1): the head reads each
    tile's rectangle of the images, clamp-to-edge at the frame border."""
    w, h = 700, 430
    imgs = synth.denoise_inputs(w, h, 3, hdr=True, nan_fraction=0.02)
    weights = synth.unet_weights(9, bias_scale=0.05)
    fused, ids = _denoise(weights, imgs, True, 1, 0.7, max_tile=256, stack=1, profile=True)
    plain, _ = _denoise(weights, imgs, True, 0, 0.7, max_tile=256, stack=1)
    assert np.array_equal(fused.view(np.uint32), plain.view(np.uint32))
    assert "input-pack+enc_conv0" in ids


def test_head_off_with_kept_activations_or_expansion_decoders():
    # kept activations read the packed input back; expansion decoders
    # (subpixelDecoder 0) read the plain packed input as their skip source:
    # both run the separate input pass
    w, h = 64, 48
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9, bias_scale=0.05)
    fused, ids = _denoise(weights, imgs, True, 1, keep=True, profile=True)
    plain, _ = _denoise(weights, imgs, True, 0, keep=True)
    assert np.array_equal(fused.view(np.uint32), plain.view(np.uint32))
    assert "input-pack" in ids and "input-pack+enc_conv0" not in ids
    outs = []
    for head in (1, 0):
        d = Denoiser(weights, ox.PRECISION_FP16, imgs, True)
        try:
            ox.oidnx_filter_set_int(d.f, "subpixelDecoder", 0)
            ox.oidnx_filter_set_int(d.f, "fuseInput", head)
            ox.oidnx_filter_commit(d.f)
            ox.oidnx_profile_next(d.f)
            outs.append(d.run())
            ids = [l["id"] for l in ox.oidnx_get_profile(d.f)["layers"]]
            assert "input-pack" in ids and "input-pack+enc_conv0" not in ids
        finally:
            d.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
