"""The fused tail on the GPU: dec_conv1b and dec_conv0 (and, in a denoise,
the output pass) as one kernel, dec_conv1b's map handed to dec_conv0 inside
tensor memory.  The kernel sums every product in the order of the unfused
kernels (dec_conv1b's plain conv, dec_conv0's folded final conv) and rounds
the intermediate map to fp16 as they store it, so its results must equal
theirs bit for bit; the unfused kernels are themselves checked against the
oracle layer by layer, and each case here is also held to the oracle end to
end.  Extents cut the 126-pixel x 6-row output tiles raggedly, fall below
one tile, and reach the 1920 x 1080 frame; the larger ones make the CTAs
walk groups of tiles that pass conv-1 rows on in tensor memory."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from oracle import unet
from oracle.numerics import round_storage
from tests import _layout
from tests._gpu import Denoiser, empty_dev, rel_l2, stream, to_dev, to_host

import conv2d_implicit_gemm_gb300 as ox


def _network(f, x):
    h, w, _ = x.shape
    src = to_dev(_layout.to_internal(x, "fp16"))
    out = empty_dev(w * h * 16)
    ox.oidnx_network_execute(f, src.data_ptr(), w, h, out.data_ptr(), stream())
    ox.oidnx_filter_sync_status(f)
    return to_host(out, np.float32, (h, w, 4)).copy()


def _filter(weights, tail):
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), ox.PRECISION_FP16)
    ox.oidnx_filter_set_int(f, "fuseTail", tail)
    return f


# from (512, 300) on, the CTAs walk groups of 2 to 13 row tiles and carry
# conv-1 rows from tile to tile
@pytest.mark.parametrize("w,h", [(1, 1), (3, 2), (17, 5), (126, 6), (127, 7), (130, 21),
                                 (252, 12), (300, 37), (512, 64), (379, 131), (512, 300),
                                 (1000, 601), (1283, 997)])
def test_tail_network_equals_unfused(w, h):
    weights = synth.unet_weights(9, bias_scale=0.05)
    x = round_storage(synth.uniform_activations(h, w, 9, seed=7 * w + h, low=0.0, high=1.0), "fp16")
    outs = []
    for tail in (1, 0):
        f = _filter(weights, tail)
        try:
            assert ox.oidnx_filter_get_int(f, "fuseTail") == tail
            outs.append(_network(f, x))
        finally:
            ox.oidnx_filter_release(f)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert not outs[0][..., 3].any()
    if w * h <= 300 * 37:
        ref = unet.forward(x, weights, "fp16")
        assert np.abs(outs[0][..., :3] - ref).max() <= 2e-2


def test_tail_repeated_runs_equal_unfused():
    """The kernel's warps hand tensor-memory columns to one another through
    barriers; a missing handoff shows as a few wrong pixels in some runs
    only, so one frame with long tile groups runs several times."""
    w, h = 1000, 601
    weights = synth.unet_weights(9, bias_scale=0.05)
    x = round_storage(synth.uniform_activations(h, w, 9, seed=11, low=0.0, high=1.0), "fp16")
    f, g = _filter(weights, 1), _filter(weights, 0)
    try:
        ref = _network(g, x).view(np.uint32)
        for _ in range(6):
            assert np.array_equal(_network(f, x).view(np.uint32), ref)
    finally:
        ox.oidnx_filter_release(f)
        ox.oidnx_filter_release(g)


def test_tail_runs_as_one_launch_and_keeps_no_map():
    weights = synth.unet_weights(9)
    x = round_storage(synth.uniform_activations(24, 40, 9, seed=2, low=0.0, high=1.0), "fp16")
    f = _filter(weights, 1)
    try:
        ox.oidnx_profile_next(f)
        _network(f, x)
        ids = [l["id"] for l in ox.oidnx_get_profile(f)["layers"]]
        assert "dec_conv1b+dec_conv0" in ids
        assert "dec_conv1b" not in ids and "dec_conv0" not in ids
        with pytest.raises(ox.OidnxError) as e:
            ox.oidnx_debug_read_activation(f, 15)
        assert "not stored" in str(e.value)
        # kept activations turn the fusion off: every map can be read back
        ox.oidnx_filter_set_int(f, "keepActivations", 1)
        ox.oidnx_profile_next(f)
        _network(f, x)
        ids = [l["id"] for l in ox.oidnx_get_profile(f)["layers"]]
        assert "dec_conv1b" in ids and "dec_conv0" in ids
        assert ox.oidnx_debug_read_activation(f, 15).size == 24 * 40 * 32
    finally:
        ox.oidnx_filter_release(f)


def test_tail_noalloc_equals_planned_unfused():
    weights = synth.unet_weights(9, bias_scale=0.05)
    f = _filter(weights, 1)
    g = _filter(weights, 0)
    try:
        for (w, h, seed) in [(200, 136, 1), (96, 72, 2), (33, 9, 3)]:
            x = round_storage(synth.uniform_activations(h, w, 9, seed=seed, low=0.0, high=1.0), "fp16")
            src = to_dev(_layout.to_internal(x, "fp16"))
            got = empty_dev(w * h * 16)
            got.fill_(0xFF)
            ox.oidnx_network_execute_noalloc(f, src.data_ptr(), w, h, got.data_ptr(), stream())
            ox.oidnx_filter_sync_status(f)
            ref = _network(g, x)
            assert np.array_equal(to_host(got, np.uint32, (h, w, 4)), ref.view(np.uint32))
    finally:
        ox.oidnx_filter_release(f)
        ox.oidnx_filter_release(g)


@pytest.mark.parametrize("hdr", [True, False])
@pytest.mark.parametrize("w,h", [(700, 430), (37, 11), (1, 1)])
def test_tail_output_pass_equals_unfused(hdr, w, h):
    """One tile: the output pass runs in the tail's epilogue (fuseOutput on)
    or after it (off); both give the bits of the unfused kernels."""
    imgs = synth.denoise_inputs(w, h, 3, hdr=hdr, nan_fraction=0.02)
    weights = synth.unet_weights(9, bias_scale=0.05)
    outs = []
    for tail, fuse_out in ((1, 1), (1, 0), (0, 1)):
        d = Denoiser(weights, ox.PRECISION_FP16, imgs, hdr, input_scale=0.7 if hdr else 1.0)
        try:
            ox.oidnx_filter_set_int(d.f, "fuseTail", tail)
            ox.oidnx_filter_set_int(d.f, "fuseOutput", fuse_out)
            ox.oidnx_filter_commit(d.f)
            assert ox.oidnx_filter_get_int(d.f, "tiles") == 1
            outs.append(d.run())
        finally:
            d.close()
    for o in outs[1:]:
        assert np.array_equal(outs[0].view(np.uint32), o.view(np.uint32))
    assert np.array_equal(outs[0][..., 3].view(np.uint32), imgs[0][..., 3].view(np.uint32))
    if w * h <= 37 * 11:
        ref = unet.denoise(imgs, weights, hdr=hdr, input_scale=0.7 if hdr else 1.0)
        assert rel_l2(outs[0][..., :3], ref[..., :3]) <= 2e-2


def test_tail_1080p_frame_equals_unfused():
    """The frame the benchmark times (1920 x 1080, colour + albedo + normal,
    HDR, one tile): fused and unfused give the same bits; one interior window
    is held to the oracle's denoise (a 16-aligned crop, so that the oracle's
    pooling grid matches the frame's)."""
    w, h = 1920, 1080
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    weights = synth.unet_weights(9)
    outs = []
    for tail in (1, 0):
        d = Denoiser(weights, ox.PRECISION_FP16, imgs, True)
        try:
            ox.oidnx_filter_set_int(d.f, "fuseTail", tail)
            ox.oidnx_filter_commit(d.f)
            outs.append(d.run())
        finally:
            d.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    m = 96
    ref = unet.denoise([im[592:848, 1504:1760] for im in imgs], weights, hdr=True)
    got = outs[0][592 + m:848 - m, 1504 + m:1760 - m, :3]
    assert rel_l2(got, ref[m:-m, m:-m, :3]) <= 2e-2


@pytest.mark.parametrize("stack", [0, 3])
def test_tail_stacked_tiles_equal_unfused(stack):
    """A frame of several tiles, stacked (one group, or groups of 3 with a
    short last one): each tile's fused tail reads that tile's rows of
    dec_conv1a's output, its halo beyond them read as zeros like the gap rows
    the separate dec_conv1b sees, so the bits equal the separate kernels'."""
    w, h = 700, 430
    imgs = synth.denoise_inputs(w, h, 3, hdr=True, nan_fraction=0.02)
    weights = synth.unet_weights(9, bias_scale=0.05)
    outs = []
    for tail in (1, 0):
        d = Denoiser(weights, ox.PRECISION_FP16, imgs, True, input_scale=0.7, max_tile_size=256, overlap=96)
        try:
            ox.oidnx_filter_set_int(d.f, "fuseTail", tail)
            ox.oidnx_filter_set_int(d.f, "stackTiles", stack)
            ox.oidnx_filter_commit(d.f)
            assert ox.oidnx_filter_get_int(d.f, "tiles") > 4
            assert ox.oidnx_filter_get_int(d.f, "stackedTiles") > 1
            if tail:
                ox.oidnx_profile_next(d.f)
            outs.append(d.run())
            if tail:
                ids = [l["id"] for l in ox.oidnx_get_profile(d.f)["layers"]]
                assert ids[-1] == "dec_conv1b+dec_conv0+output" and "dec_conv1b" not in ids
        finally:
            d.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
