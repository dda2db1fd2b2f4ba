"""Helpers shared by the GPU tests: device buffers via torch (plumbing only),
filter set-up through the C ABI, and the oracle-side comparisons."""

import numpy as np
import torch

import conv2d_implicit_gemm_gb300 as ox


def to_dev(arr):
    """Copy a numpy array to a CUDA tensor with the same bytes."""
    a = np.ascontiguousarray(arr)
    t = torch.from_numpy(a.view(np.uint8).reshape(-1).copy())
    return t.cuda()


def empty_dev(nbytes):
    return torch.zeros(nbytes, dtype=torch.uint8, device="cuda")


def to_host(t, dtype, shape=None):
    a = t.cpu().numpy().view(dtype)
    return a.reshape(shape) if shape is not None else a


def stream():
    return torch.cuda.current_stream().cuda_stream


class Denoiser:
    """One filter over device images (colour, albedo, normal, output)."""

    def __init__(self, weights, precision, images, hdr, input_scale=1.0,
                 max_tile_size=0, overlap=-1, keep=False, blob_dtype="f32"):
        self.f = ox.oidnx_filter_create(ox.write_weight_blob(weights, blob_dtype), precision)
        h, w = images[0].shape[:2]
        self.w, self.h = w, h
        self.inputs = [to_dev(img.astype(np.float32)) for img in images]
        self.output = empty_dev(w * h * 16)
        for i, t in enumerate(self.inputs):
            ox.oidnx_filter_set_image(self.f, i, t.data_ptr(), 0)
        ox.oidnx_filter_set_image(self.f, ox.IMAGE_OUTPUT, self.output.data_ptr(), 0)
        ox.oidnx_filter_set_int(self.f, "width", w)
        ox.oidnx_filter_set_int(self.f, "height", h)
        ox.oidnx_filter_set_int(self.f, "hdr", int(hdr))
        ox.oidnx_filter_set_int(self.f, "transfer", ox.TRANSFER_LOG)
        ox.oidnx_filter_set_int(self.f, "maxTileSize", max_tile_size)
        ox.oidnx_filter_set_int(self.f, "overlap", overlap)
        ox.oidnx_filter_set_int(self.f, "keepActivations", int(keep))
        ox.oidnx_filter_set_float(self.f, "inputScale", input_scale)
        ox.oidnx_filter_commit(self.f)

    def run(self):
        ox.oidnx_filter_execute(self.f, stream())
        ox.oidnx_filter_sync_status(self.f)
        return to_host(self.output, np.float32, (self.h, self.w, 4)).copy()

    def activation(self, layer, h, w, c):
        return ox.oidnx_debug_read_activation(self.f, layer).reshape(h, w, c)

    def close(self):
        ox.oidnx_filter_release(self.f)


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref.ravel())
    return np.linalg.norm((got - ref).ravel()) / max(den, 1e-30)


def ulp_diff_f32(a, b):
    """|a - b| in float32 ulps (same-sign finite values)."""
    ai = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(ai - bi)
