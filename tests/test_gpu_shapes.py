"""Conv layers of the common tile shapes run kernels compiled for that shape
(rows per tile, rows stacked per MMA, epilogue mode); option "shapeKernels"
0 makes every conv select its issue sequence at run time instead.  Both
forms issue the same MMAs in the same order, so a denoise gives the same bits
either way.  The profile names the shape each conv launch ran, so each case
also checks that the compiled shapes were used (and not with the option 0).
The cases cover one-tile frames whose levels take tiles of 8, 4, 2 and 1 rows
(with split last waves), a stacked frame of tiles, and fp32 storage."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import synth
from tests._gpu import Denoiser

import conv2d_implicit_gemm_gb300 as ox


def _run(weights, precision, imgs, shape_kernels, **kw):
    d = Denoiser(weights, precision, imgs, True, input_scale=0.7, **kw)
    try:
        ox.oidnx_filter_set_int(d.f, "shapeKernels", shape_kernels)
        ox.oidnx_filter_commit(d.f)
        assert ox.oidnx_filter_get_int(d.f, "shapeKernels") == shape_kernels
        ox.oidnx_profile_next(d.f)
        out = d.run()
        shapes = [l["shape"] for l in ox.oidnx_get_profile(d.f)["layers"]]
        return out, shapes
    finally:
        d.close()


@pytest.mark.parametrize("precision,w,h,tile", [
    (ox.PRECISION_FP16, 960, 544, 0),
    (ox.PRECISION_FP16, 700, 430, 0),
    (ox.PRECISION_FP16, 1283, 611, 0),
    (ox.PRECISION_FP16, 700, 430, 256),
    (ox.PRECISION_FP32, 384, 256, 0),
])
def test_shape_kernels_equal_run_time_form(precision, w, h, tile):
    imgs = synth.denoise_inputs(w, h, 3, hdr=True, nan_fraction=0.01)
    weights = synth.unet_weights(9, bias_scale=0.05)
    kw = {"max_tile_size": tile, "overlap": 96} if tile else {}
    a, shapes_a = _run(weights, precision, imgs, 1, **kw)
    b, shapes_b = _run(weights, precision, imgs, 0, **kw)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert any(s != 0 for s in shapes_a)
    assert all(s == 0 for s in shapes_b)
