"""Single conv layer on the GPU (tcgen05 fp16 path and the 3xTF32 fp32 path)
against the oracle, element by element, through the C ABI."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from oracle import layers
from oracle.numerics import round_storage
from tests import _layout
from tests._gpu import empty_dev, rel_l2, stream, to_dev, to_host

ox = pytest.importorskip("conv2d_implicit_gemm_gb300")


def _run_conv(x, w, b, precision):
    h, wd, cin = x.shape
    cout = w.shape[0]
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    c = ox.oidnx_conv_create(w, b, prec)
    try:
        src = to_dev(_layout.to_internal(x, precision))
        out = empty_dev(_layout.internal_nbytes(h, wd, cout, precision))
        ox.oidnx_conv_execute(c, src.data_ptr(), out.data_ptr(), wd, h, 1, stream())
        import torch
        torch.cuda.synchronize()
        dt = np.float16 if precision == "fp16" else np.float32
        raw = to_host(out, dt)
        return _layout.from_internal(raw, h, wd, cout, precision).astype(np.float64), raw
    finally:
        ox.oidnx_conv_release(c)


def _oracle_conv(x, w, b, precision):
    wq = round_storage(w, precision).astype(np.float64)
    y = layers.conv3x3(x.astype(np.float64), wq, b.astype(np.float64), relu=True)
    return round_storage(y, precision).astype(np.float64)


def _fp16_code_diff(a, b):
    ai = a.astype(np.float16).view(np.int16).astype(np.int32)
    bi = b.astype(np.float16).view(np.int16).astype(np.int32)
    return np.abs(ai - bi)


def _assert_near_fp16(got, ref):
    """fp32 accumulation vs the exact sum: every stored fp16 value is within
    one fp16 step of the oracle's, or within 1e-4 absolute where the sum
    cancels to a value whose fp16 spacing is finer than the fp32 rounding."""
    close = (_fp16_code_diff(got, ref) <= 1) | (np.abs(got - ref) <= 1e-4)
    assert close.all(), (np.abs(got - ref)[~close].max(), (~close).sum())


CASES = [  # (width, height, cin, cout)
    (128, 4, 16, 16), (130, 5, 32, 32), (1, 1, 16, 16), (37, 9, 9, 32),
    (257, 3, 64, 48), (64, 20, 80, 96), (200, 7, 112, 112), (50, 6, 160, 96),
    (300, 2, 73, 64), (17, 33, 32, 3),
    # 184 tiles on a 152-CTA grid: the last wave's 32 tiles run as sub-tiles
    # of 2 rows (R = 8) and of 1 row (R = 4)
    (1024, 184, 32, 32), (1024, 92, 64, 64),
]


@pytest.mark.parametrize("w,h,cin,cout", CASES)
@pytest.mark.parametrize("precision", ["fp16", "fp32"])
def test_conv_layer_matches_oracle(w, h, cin, cout, precision):
    x = synth.uniform_activations(h, w, cin, seed=w * 7 + h)
    if precision == "fp16":
        x = x.astype(np.float16)
    wt, b = synth.he_uniform_conv(cout, cin, seed=cin * 13 + cout, bias_scale=0.1)
    got, _ = _run_conv(x, wt, b, precision)
    ref = _oracle_conv(x, wt, b, precision)
    assert got.shape == ref.shape
    err = rel_l2(got, ref)
    if precision == "fp16":
        assert err <= 1e-2, err
        _assert_near_fp16(got, ref)
    else:
        assert err <= 1e-4, err


def test_conv_padded_lanes_stay_zero():
    x = synth.uniform_activations(9, 140, 24, seed=3).astype(np.float16)
    wt, b = synth.he_uniform_conv(40, 24, seed=4, bias_scale=0.5)
    _, raw = _run_conv(x, wt, b, "fp16")
    full = raw.reshape(9, -1, 140, 8).transpose(0, 2, 1, 3).reshape(9, 140, -1)
    assert full.shape[-1] == 48
    assert not full[..., 40:].any()


def test_single_conv_512x512_64_to_64_full_size():
    """The single-layer workload: 512x512, Cin = Cout = 64, fp16, fp32 acc."""
    x = synth.uniform_activations(512, 512, 64, seed=11).astype(np.float16)
    wt, b = synth.he_uniform_conv(64, 64, seed=1001, bias_scale=0.1)
    got, _ = _run_conv(x, wt, b, "fp16")
    ref = _oracle_conv(x, wt, b, "fp16")
    assert rel_l2(got, ref) <= 1e-2
    _assert_near_fp16(got, ref)
