"""Per-tile input pass (pack) and output pass (unpack).

Source: "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts",
inputShader and outputShader; channel order as in "oidn-web 0.3.4 -> 0.4.0,
nativeUNet.ts", createInputPackShader (channel c of the network input is
channel c % 3 of source image c / 3; lanes past 3*S are zero).
"""

import numpy as np

from .numerics import (FLT_MAX, hdr_forward_exact, hdr_inverse_exact,
                       round_storage, sanitize)


def effective_scale(input_scale):
    """inputScale 0 means 1 (the config word convention of program.ts)."""
    return np.float32(1.0) if input_scale == 0 else np.float32(input_scale)


def pack_tile(images, rect, hdr, input_scale, precision):
    """Network input of one tile, logical channels [h, w, 3*S].

    images: list of S float32 [H, W, 4] arrays in order colour, albedo,
    normal.  rect = (x, y, w, h): the tile's input rectangle; pixels are read
    at clamp(position, 0, size - 1) (clamp-to-edge).
    Colour: HDR -> F(sanitize(rgb * inputScale, 0, FLT_MAX)); LDR ->
    sanitize(rgb, 0, 1).  Albedo: sanitize(rgb, 0, 1).  Normal:
    sanitize(rgb, -1, 1) * 0.5 + 0.5.  All steps but F are float32 as in the
    shader; F is evaluated exactly (float64) and every channel is rounded
    once to the storage precision.
    Returns float16 or float32 array [h, w, 3*S].
    """
    x0, y0, w, h = rect
    height, width = images[0].shape[:2]
    ys = np.clip(np.arange(y0, y0 + h), 0, height - 1)
    xs = np.clip(np.arange(x0, x0 + w), 0, width - 1)
    chans = []
    for index, img in enumerate(images):
        rgb = np.asarray(img, np.float32)[ys][:, xs, :3]
        if index == 0:
            if hdr:
                scaled = sanitize(rgb * effective_scale(input_scale), 0.0, FLT_MAX)
                chans.append(round_storage(hdr_forward_exact(scaled), precision))
            else:
                chans.append(round_storage(sanitize(rgb, 0.0, 1.0), precision))
        elif index == 1:
            chans.append(round_storage(sanitize(rgb, 0.0, 1.0), precision))
        else:
            n = sanitize(rgb, -1.0, 1.0) * np.float32(0.5) + np.float32(0.5)
            chans.append(round_storage(n.astype(np.float32), precision))
    return np.concatenate(chans, axis=-1)


def unpack_rect(net, color, hdr, input_scale):
    """Output pass for one rectangle.

    net: float32 [h, w, >=3] network output at the rectangle's pixels;
    color: float32 [h, w, 4] input colour at the same pixels.
    rgb = sanitize(net.rgb, 0, hdr ? FLT_MAX : 1); HDR: F^-1(rgb) / inputScale
    evaluated exactly and rounded once to float32; alpha = colour alpha,
    copied bit for bit.  Returns float32 [h, w, 4].
    """
    d = sanitize(np.asarray(net, np.float32)[..., :3], 0.0,
                 FLT_MAX if hdr else 1.0)
    out = np.empty(d.shape[:2] + (4,), np.float32)
    if hdr:
        scale = np.float64(effective_scale(input_scale))
        with np.errstate(over="ignore"):
            out[..., :3] = (hdr_inverse_exact(d) / scale).astype(np.float32)
    else:
        out[..., :3] = d
    bits = np.ascontiguousarray(color[..., 3]).view(np.uint32)
    out.view(np.uint32)[..., 3] = bits
    return out
