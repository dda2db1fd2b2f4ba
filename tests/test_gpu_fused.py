"""The fused layer pairs on the GPU against the oracle: enc_conv0 +
enc_conv1 + 2x2 max-pool and dec_conv1b + dec_conv0, each run as one kernel
that keeps the 32-channel map between its convs on chip.  Each pair's output
is checked in isolation (the oracle's two layers applied to the GPU's own
stored input of the pair), the chained output end to end, over widths that
cut the column strips raggedly, odd heights (a half pool window at the
bottom) and inputs smaller than one strip."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from oracle import unet
from oracle.numerics import round_storage
from tests._gpu import rel_l2
from tests.test_gpu_network import (VALUE_NAMES, _isolated, _run_network,
                                    assert_layer_elementwise)

import conv2d_implicit_gemm_gb300 as ox


def _shapes(ref):
    return {k: (ref[name].shape if k < 16 else ref["dec_conv0"].shape)
            for k, name in enumerate(VALUE_NAMES)}


@pytest.mark.parametrize("w,h", [(64, 48), (80, 34), (130, 21), (250, 37), (512, 64), (300, 9),
                                 (17, 5), (3, 2), (1, 1)])
@pytest.mark.parametrize("in_channels", [9, 3])
def test_fused_pairs_match_oracle(w, h, in_channels):
    weights = synth.unet_weights(in_channels, bias_scale=0.05)
    x = round_storage(synth.uniform_activations(h, w, in_channels, seed=3 * w + h, low=0.0, high=1.0),
                      "fp16")
    flat, final = _run_network(weights, x, "fp16", subpixel=1, fuse=1)
    ref = unet.forward(x, weights, "fp16", keep=True)
    shp = _shapes(ref)
    acts = {k: flat[k].reshape(shp[k]) for k in range(17) if flat[k] is not None}
    assert 1 not in acts and 15 not in acts
    # encoder pair from the GPU's packed input
    mid = {0: acts[0], 1: _isolated(1, acts, weights, "fp16")}
    iso = _isolated(2, mid, weights, "fp16")
    assert rel_l2(acts[2], iso) <= 1e-2, "enc pair"
    assert_pair_elementwise(acts[2], iso, mid, 2, weights)
    # decoder pair from the GPU's dec_conv1a output
    mid = {14: acts[14], 15: _isolated(15, acts, weights, "fp16")}
    iso = _isolated(16, mid, weights, "fp16")
    assert rel_l2(acts[16], iso) <= 1e-2, "dec pair"
    assert_pair_elementwise(acts[16], iso, mid, 16, weights)
    # the layers between the pairs still match in isolation, value by value
    for k in range(3, 15):
        iso = _isolated(k, acts, weights, "fp16")
        assert rel_l2(acts[k], iso) <= 1e-2, VALUE_NAMES[k]
        assert_layer_elementwise(k, acts[k], iso, acts, weights, "fp16", 1)
    assert np.array_equal(final[..., :3], acts[16].astype(np.float32))
    assert not final[..., 3].any()
    assert np.abs(final[..., :3] - ref["dec_conv0"]).max() <= 2e-2


def assert_pair_elementwise(got, iso, mid, k, weights):
    """Second conv of a fused pair, value by value: the oracle's input (its
    own fp16 rounding of the first conv) may differ from the kernel's
    on-chip one by one fp16 step per value (2^-11 relative), which moves an
    output by at most 2^-11 (|W| * |mid|); plus the bound of an unfused
    layer (one fp16 step / 1e-4; the final conv: 2^-14 (|W| * |x| + |b|))."""
    from tests.test_gpu_network import _magnitude
    got = np.asarray(got, np.float64)
    iso = np.asarray(iso, np.float64)
    diff = np.abs(got - iso)
    mag = _magnitude(k, mid, weights)
    if k == 16:
        close = diff <= 2.0 ** -11 * mag + 2.0 ** -14 * mag
    else:
        code = np.abs(got.astype(np.float16).view(np.int16).astype(np.int32) -
                      iso.astype(np.float16).view(np.int16).astype(np.int32))
        close = (code <= 1) | (diff <= 1e-4 + 2.0 ** -11 * mag)
    assert close.all(), (k, int((~close).sum()), float(diff[~close].max()))


def test_fused_and_unfused_networks_agree():
    # the fused kernels round the intermediate map to fp16 like the unfused
    # layers; only fp32 summation order differs
    weights = synth.unet_weights(9, bias_scale=0.05)
    w, h = 384, 200
    x = round_storage(synth.uniform_activations(h, w, 9, seed=5, low=0.0, high=1.0), "fp16")
    _, fused = _run_network(weights, x, "fp16", subpixel=1, fuse=1)
    _, plain = _run_network(weights, x, "fp16", subpixel=1, fuse=0)
    ref = unet.forward(x, weights, "fp16")
    assert np.abs(fused[..., :3] - ref).max() <= 2e-2
    assert np.abs(plain[..., :3] - ref).max() <= 2e-2
    assert rel_l2(fused[..., :3], plain[..., :3]) <= 1e-2


def test_fused_intermediate_is_not_stored():
    weights = synth.unet_weights(9)
    x = round_storage(synth.uniform_activations(16, 32, 9, seed=1, low=0.0, high=1.0), "fp16")
    prec = ox.PRECISION_FP16
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), prec)
    try:
        assert ox.oidnx_filter_get_int(f, "fuseLayers") == 0
    finally:
        ox.oidnx_filter_release(f)
    flat, _ = _run_network(weights, x, "fp16", fuse=1)
    assert flat[1] is None and flat[15] is None
    with pytest.raises(ox.OidnxError) as e:
        _read_fused_intermediate(weights, x)
    assert e.value.status == ox.ERR_INVALID_ARGUMENT
    assert "not stored" in str(e.value)


def _read_fused_intermediate(weights, x):
    from tests import _layout
    from tests._gpu import empty_dev, stream, to_dev
    h, w, _ = x.shape
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), ox.PRECISION_FP16)
    try:
        ox.oidnx_filter_set_int(f, "keepActivations", 1)
        ox.oidnx_filter_set_int(f, "fuseLayers", 1)
        src = to_dev(_layout.to_internal(x, "fp16"))
        out = empty_dev(w * h * 16)
        ox.oidnx_network_execute(f, src.data_ptr(), w, h, out.data_ptr(), stream())
        ox.oidnx_filter_sync_status(f)
        ox.oidnx_debug_read_activation(f, 15)
    finally:
        ox.oidnx_filter_release(f)


def test_fused_noalloc_matches_planned_run():
    # the fixed-array entry point builds the same fused launches
    from tests import _layout
    from tests._gpu import empty_dev, stream, to_dev, to_host
    weights = synth.unet_weights(9, bias_scale=0.05)
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), ox.PRECISION_FP16)
    try:
        ox.oidnx_filter_set_int(f, "fuseLayers", 1)
        for (w, h, seed) in [(200, 136, 1), (96, 72, 2)]:
            x = round_storage(synth.uniform_activations(h, w, 9, seed=seed, low=0.0, high=1.0), "fp16")
            src = to_dev(_layout.to_internal(x, "fp16"))
            ref = empty_dev(w * h * 16)
            got = empty_dev(w * h * 16)
            got.fill_(0xFF)
            ox.oidnx_network_execute(f, src.data_ptr(), w, h, ref.data_ptr(), stream())
            ox.oidnx_network_execute_noalloc(f, src.data_ptr(), w, h, got.data_ptr(), stream())
            ox.oidnx_filter_sync_status(f)
            r = to_host(ref, np.float32, (h, w, 4))
            g = to_host(got, np.float32, (h, w, 4))
            assert np.array_equal(g.view(np.uint32), r.view(np.uint32))
            assert np.abs(g[..., :3] - unet.forward(x, weights, "fp16")).max() <= 2e-2
    finally:
        ox.oidnx_filter_release(f)
