"""oidnx_network_execute_noalloc: the network forward for callers that may
not allocate device memory after set-up (fixed-budget renderers, plug-ins
whose host owns all device memory).  Its intermediate activations live in
the library's fixed device array instead of a filter-allocated arena.

Checked against oidnx_network_execute on two calls in a row with different
shapes and data, so that contents left in the shared array by the first call
cannot leak into the second, and checked to leave the device's free memory
unchanged once set up.  This file is collected last on purpose."""

import gc

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import synth
from oracle.numerics import round_storage
from tests import _layout
from tests._gpu import empty_dev, stream, to_dev, to_host

import conv2d_implicit_gemm_gb300 as ox


def _packed(w, h, seed, precision):
    x = synth.uniform_activations(h, w, 9, seed=seed, low=0.0, high=1.0)
    return to_dev(_layout.to_internal(round_storage(x, precision), precision))


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
def test_noalloc_matches_network_execute_two_calls_in_a_row(precision):
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    f = ox.oidnx_filter_create(ox.write_weight_blob(synth.unet_weights(9, bias_scale=0.05)), prec)
    try:
        for (w, h, seed) in [(200, 136, 1), (96, 72, 2)]:
            src = _packed(w, h, seed, precision)
            ref = empty_dev(w * h * 16)
            got = empty_dev(w * h * 16)
            got.fill_(0xFF)   # NaN pattern: every output value must be written
            ox.oidnx_network_execute(f, src.data_ptr(), w, h, ref.data_ptr(), stream())
            ox.oidnx_network_execute_noalloc(f, src.data_ptr(), w, h, got.data_ptr(), stream())
            ox.oidnx_filter_sync_status(f)
            r = to_host(ref, np.float32, (h, w, 4))
            g = to_host(got, np.float32, (h, w, 4))
            assert np.isfinite(g).all()
            if precision == "fp16":
                np.testing.assert_allclose(g, r, rtol=0, atol=2e-2)
            else:
                num = np.linalg.norm((g - r).ravel())
                assert num <= 1e-4 * np.linalg.norm(r.ravel())
            # same kernels with the same launch parameters: the bits agree too
            assert np.array_equal(g.view(np.uint32), r.view(np.uint32))
    finally:
        ox.oidnx_filter_release(f)


def test_noalloc_rejects_inputs_beyond_the_array():
    f = ox.oidnx_filter_create(ox.write_weight_blob(synth.unet_weights(9)), ox.PRECISION_FP16)
    try:
        src = empty_dev(16)
        with pytest.raises(ox.OidnxError) as e:
            ox.oidnx_network_execute_noalloc(f, src.data_ptr(), 512, 512, src.data_ptr(), stream())
        assert e.value.status == ox.ERR_INVALID_ARGUMENT
        assert "bytes of activation scratch" in str(e.value)
    finally:
        ox.oidnx_filter_release(f)
    torch.cuda.synchronize()


@pytest.mark.parametrize("precision,side", [("fp16", 384), ("fp32", 256)])
def test_noalloc_accepts_the_documented_maximum(precision, side):
    """The largest square input the header promises (the fp16 one with the
    sub-pixel decoders' parity-split copies) runs and writes every output."""
    prec = ox.PRECISION_FP16 if precision == "fp16" else ox.PRECISION_FP32
    f = ox.oidnx_filter_create(ox.write_weight_blob(synth.unet_weights(9, bias_scale=0.05)), prec)
    try:
        src = _packed(side, side, 3, precision)
        got = empty_dev(side * side * 16)
        got.fill_(0xFF)
        ox.oidnx_network_execute_noalloc(f, src.data_ptr(), side, side, got.data_ptr(), stream())
        ox.oidnx_filter_sync_status(f)
        assert np.isfinite(to_host(got, np.float32, (side, side, 4))).all()
    finally:
        ox.oidnx_filter_release(f)


def test_noalloc_allocates_nothing_after_set_up():
    """After one warm-up call (which also loads the kernels it launches),
    further calls must not change the device's free memory, the filter's own
    arena bytes or torch's allocator counters: the call's only memory is
    the library's fixed array, placed when the filter was created."""
    f = ox.oidnx_filter_create(ox.write_weight_blob(synth.unet_weights(9, bias_scale=0.05)),
                               ox.PRECISION_FP16)
    try:
        w, h = 256, 160
        src = _packed(w, h, 4, "fp16")
        out = empty_dev(w * h * 16)
        ox.oidnx_network_execute_noalloc(f, src.data_ptr(), w, h, out.data_ptr(), stream())
        ox.oidnx_filter_sync_status(f)
        # tensors left by earlier tests are collected now, not during the
        # loop (torch's counters may still only go down, never up)
        gc.collect()
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        arena0 = ox.oidnx_get_resource_info(f)
        alloc0 = torch.cuda.memory_allocated()
        reserved0 = torch.cuda.memory_reserved()
        for _ in range(5):
            ox.oidnx_network_execute_noalloc(f, src.data_ptr(), w, h, out.data_ptr(), stream())
        ox.oidnx_filter_sync_status(f)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0
        assert ox.oidnx_get_resource_info(f) == arena0
        assert torch.cuda.memory_allocated() <= alloc0
        assert torch.cuda.memory_reserved() <= reserved0
    finally:
        ox.oidnx_filter_release(f)
