"""The 16-layer network on the GPU against the oracle: every stored
activation checked in isolation (the oracle's layer applied to the GPU's own
input activations) and the chained output checked end to end."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from oracle import layers, unet
from oracle.numerics import round_storage
from tests import _layout
from tests._gpu import empty_dev, rel_l2, stream, to_dev, to_host

import conv2d_implicit_gemm_gb300 as ox

# activation index (0 = input, k = output of layer k-1) -> its sources and op
LAYER_OPS = {
    1: (0, None, "plain"), 2: (1, None, "pool"), 3: (2, None, "pool"),
    4: (3, None, "pool"), 5: (4, None, "pool"), 6: (5, None, "plain"),
    7: (6, None, "plain"), 8: (7, 4, "dec"), 9: (8, None, "plain"),
    10: (9, 3, "dec"), 11: (10, None, "plain"), 12: (11, 2, "dec"),
    13: (12, None, "plain"), 14: (13, 0, "dec"), 15: (14, None, "plain"),
    16: (15, None, "final"),
}
VALUE_NAMES = ["input", "enc_conv0", "pool1", "pool2", "pool3", "pool4",
               "enc_conv5a", "enc_conv5b", "dec_conv4a", "dec_conv4b",
               "dec_conv3a", "dec_conv3b", "dec_conv2a", "dec_conv2b",
               "dec_conv1a", "dec_conv1b", "dec_conv0"]


def _isolated(k, acts, weights, precision):
    s0, s1, op = LAYER_OPS[k]
    name = ox.LAYER_NAMES[k - 1]
    w, b = weights[name]
    wq = round_storage(w, precision).astype(np.float64)
    x = acts[s0].astype(np.float64)
    if op == "dec":
        x = layers.decoder_input(x, acts[s1].astype(np.float64))
    y = layers.conv3x3(x, wq, b.astype(np.float64), relu=op != "final")
    y = round_storage(y, "fp32" if op == "final" else precision).astype(np.float64)
    if op == "pool":
        y = layers.maxpool2x2(y)
    return y


def _fp16_code_diff(a, b):
    ai = np.asarray(a).astype(np.float16).view(np.int16).astype(np.int32)
    bi = np.asarray(b).astype(np.float16).view(np.int16).astype(np.int32)
    return np.abs(ai - bi)


def _magnitude(k, acts, weights, channels=None):
    """|W| * |x| + |b| of layer k on the GPU's own inputs (the sum of the
    absolute values of every term of each output), optionally over the
    first `channels` input channels only (bias then left out); pooled like
    the layer's output."""
    s0, s1, op = LAYER_OPS[k]
    w, b = weights[ox.LAYER_NAMES[k - 1]]
    x = np.abs(acts[s0].astype(np.float64))
    if op == "dec":
        x = layers.decoder_input(x, np.abs(acts[s1].astype(np.float64)))
    aw = np.abs(np.asarray(w, np.float64))
    bias = np.abs(np.asarray(b, np.float64))
    if channels is not None:
        x, aw, bias = x[..., :channels], aw[:, :channels], np.zeros_like(bias)
    m = layers.conv3x3(x, aw, bias, relu=False)
    return layers.maxpool2x2(m) if op == "pool" else m


def _subpixel_layer(k, acts, subpixel):
    """Whether the GPU ran decoder layer k in sub-pixel form (even conv
    extent, exactly twice the upsampled source's)."""
    s0, _, op = LAYER_OPS[k]
    if op != "dec" or not subpixel:
        return False
    h, w = acts[k].shape[:2]
    h0, w0 = acts[s0].shape[:2]
    return h % 2 == 0 and w % 2 == 0 and 2 * h0 == h and 2 * w0 == w


def assert_layer_elementwise(k, got, ref, acts, weights, precision, subpixel):
    """Every value of layer k against the oracle's layer on the GPU's inputs:
      fp16 layers: within one fp16 step, or within 1e-4 absolute where the
        sum cancels below the fp32 accumulation's rounding; a sub-pixel
        decoder may add 2^-11 (|W_up| * |up(x)|) and one more fp16 step: it
        sums the fp16 weights of the taps that read one low-resolution pixel
        and rounds the sum to fp16 once more (relative error <= 2^-11 per
        summed weight), before both sides round the result to fp16;
      the fp16 network's final layer (fp32 output): within 2^-14 (|W| * |x| +
        |b|), the fp32 accumulation of at most ~100 partial sums;
      fp32 layers (3xTF32 products): within 2^-13 (|W| * |x| + |b|): each
        product within 3 * 2^-22 (the dropped lo * lo term and the tf32
        rounding of both lo parts), plus at most ~540 fp32 accumulation steps
        of 2^-24 each."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = np.abs(got - ref)
    final = LAYER_OPS[k][2] == "final"
    if precision == "fp16" and not final:
        tol = 1e-4
        if _subpixel_layer(k, acts, subpixel):
            # the re-rounding bound, plus both sides' fp16 storage rounding
            # (half an fp16 step each at the larger magnitude)
            c0 = acts[LAYER_OPS[k][0]].shape[-1]
            step = np.spacing(np.maximum(np.abs(got), np.abs(ref)).astype(np.float16)).astype(np.float64)
            tol = tol + 2.0 ** -11 * _magnitude(k, acts, weights, channels=c0) + step
        close = (_fp16_code_diff(got, ref) <= 1) | (diff <= tol)
    else:
        bound = 2.0 ** (-14 if precision == "fp16" else -13) * _magnitude(k, acts, weights)
        close = diff <= bound + np.abs(ref) * 2.0 ** -23
    assert close.all(), (VALUE_NAMES[k], int((~close).sum()), float(diff[~close].max()),
                         np.argwhere(~close)[:3].tolist())


def _run_network(weights, packed_logical, precision, subpixel=0, fuse=0):
    # fuse=1: the fused pairs' intermediate maps (activations 1 and 15) are
    # never stored and come back as None
    h, w, c = packed_logical.shape
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights), prec)
    try:
        ox.oidnx_filter_set_int(f, "keepActivations", 1)
        ox.oidnx_filter_set_int(f, "subpixelDecoder", subpixel)
        ox.oidnx_filter_set_int(f, "fuseLayers", fuse)
        src = to_dev(_layout.to_internal(packed_logical, precision))
        out = empty_dev(w * h * 16)
        ox.oidnx_network_execute(f, src.data_ptr(), w, h, out.data_ptr(), stream())
        ox.oidnx_filter_sync_status(f)
        skip = (1, 15) if fuse and precision == "fp16" else ()
        acts = [None if k in skip else ox.oidnx_debug_read_activation(f, k) for k in range(17)]
        final = to_host(out, np.float32, (h, w, 4)).copy()
    finally:
        ox.oidnx_filter_release(f)
    return acts, final


@pytest.mark.parametrize("precision,subpixel", [("fp16", 0), ("fp16", 1), ("fp32", 0), ("fp32", 1)])
@pytest.mark.parametrize("w,h", [(64, 48), (80, 34), (130, 20), (512, 64), (1, 1), (33, 17)])
def test_network_layers_match_oracle(precision, subpixel, w, h):
    weights = synth.unet_weights(9, bias_scale=0.05)
    x = synth.uniform_activations(h, w, 9, seed=w + h, low=0.0, high=1.0)
    x = round_storage(x, precision)
    acts_flat, final = _run_network(weights, x, precision, subpixel)
    ref = unet.forward(x, weights, precision, keep=True)
    acts = []
    for k, name in enumerate(VALUE_NAMES):
        shape = ref[name].shape if k < 16 else ref["dec_conv0"].shape
        acts.append(acts_flat[k].reshape(shape))
    assert np.array_equal(acts[0], np.asarray(x, np.float32))
    tol = 1e-2 if precision == "fp16" else 1e-4
    for k in range(1, 17):
        iso = _isolated(k, acts, weights, precision)
        err = rel_l2(acts[k], iso)
        assert err <= tol, (VALUE_NAMES[k], err)
        assert_layer_elementwise(k, acts[k], iso, acts, weights, precision, subpixel)
    # chained end to end
    out = ref["dec_conv0"]
    assert np.array_equal(final[..., :3], acts[16].astype(np.float32))
    assert not final[..., 3].any()
    if precision == "fp16":
        assert np.abs(final[..., :3] - out).max() <= 2e-2
    else:
        assert rel_l2(final[..., :3], out) <= 1e-4


def test_network_one_pixel_and_tiny_inputs():
    weights = synth.unet_weights(9, bias_scale=0.05)
    for (w, h) in [(1, 1), (3, 2), (17, 5)]:
        x = round_storage(synth.uniform_activations(h, w, 9, seed=w, low=0, high=1), "fp16")
        _, final = _run_network(weights, x, "fp16")
        ref = unet.forward(x, weights, "fp16")
        assert np.abs(final[..., :3] - ref).max() <= 2e-2


@pytest.mark.parametrize("precision,subpixel", [("fp16", 1), ("fp32", 0), ("fp32", 1)])
@pytest.mark.parametrize("in_channels", [3, 6])
def test_colour_only_and_colour_albedo_models_match_oracle(precision, subpixel, in_channels):
    """The 3- and 6-channel model variants (colour; colour + albedo): the
    input block and dec_conv1a's skip have fewer lanes.  Every stored
    activation is checked in isolation, the output end to end."""
    weights = synth.unet_weights(in_channels, bias_scale=0.05)
    w, h = 130, 36
    x = round_storage(synth.uniform_activations(h, w, in_channels, seed=in_channels, low=0, high=1),
                      precision)
    acts_flat, final = _run_network(weights, x, precision, subpixel)
    ref = unet.forward(x, weights, precision, keep=True)
    acts = []
    for k, name in enumerate(VALUE_NAMES):
        shape = ref[name].shape if k < 16 else ref["dec_conv0"].shape
        acts.append(acts_flat[k].reshape(shape))
    tol = 1e-2 if precision == "fp16" else 1e-4
    for k in range(1, 17):
        iso = _isolated(k, acts, weights, precision)
        err = rel_l2(acts[k], iso)
        assert err <= tol, (VALUE_NAMES[k], err)
        assert_layer_elementwise(k, acts[k], iso, acts, weights, precision, subpixel)
    out = ref["dec_conv0"]
    if precision == "fp16":
        assert np.abs(final[..., :3] - out).max() <= 2e-2
    else:
        assert rel_l2(final[..., :3], out) <= 1e-4
