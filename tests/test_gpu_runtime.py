"""Runtime behaviour on the GPU: graph replay is bit-identical to the eager
(profiled) run, the host-buffer path equals the device path, the LRU shape
cache evicts safely, the profile and resource reports are well formed."""

import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import synth
from oracle.numerics import round_storage
from tests import _layout
from tests._gpu import Denoiser, empty_dev, stream, to_dev, to_host

import conv2d_implicit_gemm_gb300 as ox


@pytest.fixture(scope="module")
def weights():
    return synth.unet_weights(9, bias_scale=0.05)


def test_graph_replay_equals_eager_and_host_path(weights):
    w, h = 300, 120        # 10 tiles of 224 x 128 (maxTileSize 224, overlap 96)
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    d = Denoiser(weights, ox.PRECISION_FP16, imgs, True, max_tile_size=224, overlap=96)
    try:
        ox.oidnx_profile_next(d.f)
        eager = d.run()
        prof = ox.oidnx_get_profile(d.f)
        graph1 = d.run()
        graph2 = d.run()
        host_out = np.zeros((h, w, 4), np.float32)
        ox.oidnx_filter_execute_host(d.f, imgs[0], imgs[1], imgs[2], host_out, stream())
        info = ox.oidnx_get_resource_info(d.f)
    finally:
        d.close()
    assert np.array_equal(eager.view(np.uint32), graph1.view(np.uint32))
    assert np.array_equal(graph1.view(np.uint32), graph2.view(np.uint32))
    assert np.array_equal(graph1.view(np.uint32), host_out.view(np.uint32))
    ids = [l["id"] for l in prof["layers"]]
    # input pass, 14 convs, then dec_conv1b + dec_conv0 with the output pass
    # in one kernel (the fused tail)
    last = "dec_conv1b+dec_conv0+output"
    assert ids[0] == "input-pack" and ids[-1] == last and len(ids) == 16
    # the 10 tiles are stacked: one input pass and one tail per tile, each
    # other conv once over the stack
    for l in prof["layers"]:
        assert l["launches"] == (10 if l["id"] in ("input-pack", last) else 1), l
    assert all(l["ms"] > 0 for l in prof["layers"])
    assert prof["totalMs"] >= sum(l["ms"] for l in prof["layers"]) * 0.99
    # one graph for the bound device images, one for the host path's staging set
    assert info["graphs"] == 2 and info["plans"] >= 1 and info["weightBytes"] > 0


def test_profile_every_execution_through_the_graph(weights):
    w, h = 96, 64
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    d = Denoiser(weights, ox.PRECISION_FP16, imgs, True)
    try:
        plain = d.run()
        ox.oidnx_filter_set_int(d.f, "profile", 1)
        profiled = d.run()
        prof = ox.oidnx_get_profile(d.f)
    finally:
        d.close()
    assert np.array_equal(plain.view(np.uint32), profiled.view(np.uint32))
    # input pass, 14 convs, then dec_conv1b + dec_conv0 + the output pass as
    # one kernel (the fused tail, on by default for a one-tile frame)
    ids = [l["id"] for l in prof["layers"]]
    assert len(ids) == 16 and ids[-1] == "dec_conv1b+dec_conv0+output", ids


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
def test_profile_counts_executed_tensor_flops(weights, precision):
    """mmaFlop against per-pixel counts at a 256 x 128 tile, which the conv
    tiles cover exactly (no padded rows or columns): enc_conv1 (32 -> 32,
    plain) executes its logical FLOPs; dec_conv1a (sub-pixel, 64 upsampled +
    9 skip channels -> 64) executes 4 taps on the upsampled channels and 9 on
    the skip lanes padded to one K block (16 fp16 lanes, 16 fp32 lanes as two
    8-lane blocks), x3 for the three tf32 products of fp32 storage."""
    w, h = 256, 128
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    d = Denoiser(weights, prec, imgs, True)
    try:
        ox.oidnx_profile_next(d.f)
        d.run()
        prof = {l["id"]: l for l in ox.oidnx_get_profile(d.f)["layers"]}
    finally:
        d.close()
    px = w * h
    passes = 1 if precision == "fp16" else 3
    assert prof["enc_conv1"]["flop"] == 2 * 9 * 32 * 32 * px
    assert prof["enc_conv1"]["mmaFlop"] == passes * prof["enc_conv1"]["flop"]
    assert prof["dec_conv1a"]["flop"] == 2 * 9 * 73 * 64 * px
    assert prof["dec_conv1a"]["mmaFlop"] == passes * 2 * (4 * 64 + 9 * 16) * 64 * px
    assert prof["input-pack"]["mmaFlop"] == 0
    if precision == "fp16":
        # the fused tail: 3 x 22 tiles of 126 x 6 outputs, each its own group
        # at this size (all 8 conv-1 rows computed); per tile conv 1 issues
        # 8 rows x 3 ky x 3 kx x 4 K blocks at N 32, conv 2 6 rows x 3 ky x
        # 2 K blocks at N 16, each M 128 x K 16
        tail = prof["dec_conv1b+dec_conv0+output"]
        assert tail["flop"] == 2 * 9 * (64 * 32 + 32 * 3) * px
        assert tail["mmaFlop"] == 66 * 2 * 128 * 16 * (8 * 3 * 3 * 4 * 32 + 6 * 3 * 2 * 16)


def test_shape_cache_eviction_with_work_in_flight(weights):
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), ox.PRECISION_FP16)
    try:
        ox.oidnx_filter_set_int(f, "shapeCacheSize", 1)
        shapes = [(64, 48), (96, 32), (64, 48), (40, 40)]
        bufs, outs = [], []
        for (w, h) in shapes:
            x = round_storage(synth.uniform_activations(h, w, 9, seed=w * h, low=0, high=1), "fp16")
            src = to_dev(_layout.to_internal(x, "fp16"))
            out = empty_dev(w * h * 16)
            ox.oidnx_network_execute(f, src.data_ptr(), w, h, out.data_ptr(), stream())
            bufs.append(src)
            outs.append((out, w, h))
        ox.oidnx_filter_sync_status(f)
        results = [to_host(o, np.float32, (h, w, 4)).copy() for (o, w, h) in outs]
        info = ox.oidnx_get_resource_info(f)
        assert info["plans"] == 1
        # same shape, same input -> same bits, even across an eviction
        assert np.array_equal(results[0].view(np.uint32), results[2].view(np.uint32))
    finally:
        ox.oidnx_filter_release(f)


def test_execute_requires_commit_and_release_is_final(weights):
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), ox.PRECISION_FP16)
    with pytest.raises(ox.OidnxError) as e:
        ox.oidnx_filter_execute(f, stream())
    assert e.value.status == ox.ERR_NOT_COMMITTED
    with pytest.raises(ox.OidnxError) as e:
        ox.oidnx_filter_commit(f)                 # no images bound
    assert e.value.status == ox.ERR_INVALID_ARGUMENT
    ox.oidnx_filter_set_int(f, "hdr", 1)
    ox.oidnx_filter_set_int(f, "transfer", ox.TRANSFER_PU)
    ox.oidnx_filter_set_int(f, "width", 8)
    ox.oidnx_filter_set_int(f, "height", 8)
    img = empty_dev(8 * 8 * 16)
    for i in range(4):
        ox.oidnx_filter_set_image(f, i, img.data_ptr(), 0)
    with pytest.raises(ox.OidnxError) as e:
        ox.oidnx_filter_commit(f)
    assert e.value.status == ox.ERR_UNSUPPORTED
    ox.oidnx_filter_release(f)
    torch.cuda.synchronize()


def test_degenerate_dimensions_and_input_scale(weights):
    """Non-positive image dimensions, other out-of-range integer parameters
    and a negative or non-finite inputScale are rejected when set, leaving
    the committed filter as it was; an
    inputScale of 0 stands for 1 (the pages' default): an HDR denoise with
    inputScale 0 gives the bits of one with inputScale 1."""
    w, h = 80, 48
    imgs = synth.denoise_inputs(w, h, 3, hdr=True)
    outs = []
    for scale in (1.0, 0.0):
        d = Denoiser(weights, ox.PRECISION_FP16, imgs, True, input_scale=scale)
        try:
            outs.append(d.run())
            for bad in (-1.0, float("nan"), float("inf")):
                with pytest.raises(ox.OidnxError) as e:
                    ox.oidnx_filter_set_float(d.f, "inputScale", bad)
                assert e.value.status == ox.ERR_INVALID_ARGUMENT
            for name, value in (("width", 0), ("height", -3), ("stackTiles", -1),
                                ("maxTileSize", -16), ("overlap", 40), ("shapeCacheSize", 0)):
                with pytest.raises(ox.OidnxError) as e:
                    ox.oidnx_filter_set_int(d.f, name, value)
                assert e.value.status == ox.ERR_INVALID_ARGUMENT
            again = d.run()
            assert np.array_equal(again.view(np.uint32), outs[-1].view(np.uint32))
        finally:
            d.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_oversized_single_tile_reports_out_of_memory_and_filter_stays_usable(weights):
    """A 65536 x 65536 single tile needs an activation arena of over a
    terabyte: commit (which plans and allocates, and launches nothing)
    reports OUT_OF_MEMORY, and the same filter then commits and runs a small
    image.  No buffer limit below device memory applies: sizes are 64-bit."""
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), ox.PRECISION_FP16)
    try:
        img = empty_dev(64 * 64 * 16)
        for i in range(4):
            ox.oidnx_filter_set_image(f, i, img.data_ptr(), 0)
        ox.oidnx_filter_set_int(f, "width", 65536)
        ox.oidnx_filter_set_int(f, "height", 65536)
        ox.oidnx_filter_set_int(f, "maxTileSize", 0)
        with pytest.raises(ox.OidnxError) as e:
            ox.oidnx_filter_commit(f)
        assert e.value.status == ox.ERR_OUT_OF_MEMORY
        assert "arena" in str(e.value)
        imgs = synth.denoise_inputs(64, 64, 3, hdr=False)
        dev = [to_dev(im) for im in imgs]
        out = empty_dev(64 * 64 * 16)
        for i, t in enumerate(dev):
            ox.oidnx_filter_set_image(f, i, t.data_ptr(), 0)
        ox.oidnx_filter_set_image(f, ox.IMAGE_OUTPUT, out.data_ptr(), 0)
        ox.oidnx_filter_set_int(f, "width", 64)
        ox.oidnx_filter_set_int(f, "height", 64)
        ox.oidnx_filter_commit(f)
        ox.oidnx_filter_execute(f, stream())
        ox.oidnx_filter_sync_status(f)
        got = to_host(out, np.float32, (64, 64, 4))
        assert np.isfinite(got).all() and (got[..., :3] >= 0).all() and (got[..., :3] <= 1).all()
    finally:
        ox.oidnx_filter_release(f)
    torch.cuda.synchronize()


def test_bounded_device_wait_reports_timeout_and_context_survives(weights):
    """A device wait that nothing completes gives up after its limit, sets the
    filter's error word (reported once as ERR_TIMEOUT) and leaves the context
    usable: a network execution afterwards still matches the one before."""
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), ox.PRECISION_FP16)
    try:
        w, h = 40, 24
        x = round_storage(synth.uniform_activations(h, w, 9, seed=5, low=0, high=1), "fp16")
        src = to_dev(_layout.to_internal(x, "fp16"))
        out0, out1 = empty_dev(w * h * 16), empty_dev(w * h * 16)
        ox.oidnx_network_execute(f, src.data_ptr(), w, h, out0.data_ptr(), stream())
        ox.oidnx_filter_sync_status(f)
        with pytest.raises(ox.OidnxError) as e:
            ox.oidnx_debug_wait_probe(f, 0)
        assert e.value.status == ox.ERR_INVALID_ARGUMENT
        t0 = time.perf_counter()
        ox.oidnx_debug_wait_probe(f, 20000, stream())      # 20 ms limit
        with pytest.raises(ox.OidnxError) as e:
            ox.oidnx_filter_sync_status(f)
        elapsed = time.perf_counter() - t0
        assert e.value.status == ox.ERR_TIMEOUT
        assert "0x10" in str(e.value)
        assert 0.015 <= elapsed < 5.0
        ox.oidnx_filter_sync_status(f)                      # the word was cleared
        ox.oidnx_network_execute(f, src.data_ptr(), w, h, out1.data_ptr(), stream())
        ox.oidnx_filter_sync_status(f)
        assert torch.equal(out0, out1)
    finally:
        ox.oidnx_filter_release(f)


def test_host_async_frame_stream_equals_sync_calls(weights):
    # five frames in flight through the two staging sets: every output equals
    # the synchronous host call's, bit for bit, whatever the overlap
    w, h = 200, 120
    frames = []
    for k in range(5):
        imgs = synth.denoise_inputs(w, h, 3, hdr=True)
        frames.append([np.ascontiguousarray(im * np.float32(1.0 + 0.25 * k)) for im in imgs])
        frames[-1][0][..., 3] = np.float32(k)   # distinct alpha per frame
    d = Denoiser(weights, ox.PRECISION_FP16, frames[0], True)
    try:
        sync = []
        for fr in frames:
            out = np.zeros((h, w, 4), np.float32)
            ox.oidnx_filter_execute_host(d.f, fr[0], fr[1], fr[2], out, stream())
            sync.append(out)
        outs = [np.full((h, w, 4), np.nan, np.float32) for _ in frames]
        for fr, out in zip(frames, outs):
            ox.oidnx_filter_execute_host_async(d.f, fr[0], fr[1], fr[2], out, stream())
        ox.oidnx_filter_wait_host(d.f)
        info = ox.oidnx_get_resource_info(d.f)
    finally:
        d.close()
    for k in range(len(frames)):
        assert np.array_equal(outs[k].view(np.uint32), sync[k].view(np.uint32)), k
        assert (outs[k][..., 3] == k).all()
    assert not np.array_equal(sync[0], sync[1])
    assert info["graphs"] == 2 and info["hostImageBytes"] == 2 * 4 * w * h * 16
