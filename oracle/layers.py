"""Layers of the U-Net as their plain definitions, float64, [H, W, C] arrays.

Activations here are logical-channel arrays (no lane padding); the vec4
blocking of the pages is a storage layout and does not change any value
("nativeUNet.ts", packConvTensors: padded lanes are zero and stay zero).
"""

import numpy as np


def conv3x3(x, weight, bias, relu):
    """Same-padded 3x3 convolution + bias, then ReLU if `relu`.

    out[y, x, o] = bias[o] + sum_{ky,kx in 0..2} sum_i W[o, i, ky, kx] *
                   in[y + ky - 1, x + kx - 1, i],
    taps outside the image contributing zero ("nativeUNet.ts",
    createConvShader: out-of-bounds taps are skipped; bias initialises the
    accumulator; activationExpression applies max(acc, 0)).

    The sum over input channels of one tap is a matrix product (a library
    primitive); the nine taps are added in (ky, kx) order.
    x: [H, W, Cin] float64; weight: [Cout, Cin, 3, 3]; bias: [Cout].
    Returns the unrounded float64 result [H, W, Cout].
    """
    x = np.asarray(x, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    bias = np.asarray(bias, dtype=np.float64)
    h, w, cin = x.shape
    cout = weight.shape[0]
    assert weight.shape == (cout, cin, 3, 3)
    padded = np.zeros((h + 2, w + 2, cin), np.float64)
    padded[1:h + 1, 1:w + 1] = x
    out = np.broadcast_to(bias, (h, w, cout)).copy()
    for ky in range(3):
        for kx in range(3):
            window = padded[ky:ky + h, kx:kx + w].reshape(h * w, cin)
            out += (window @ weight[:, :, ky, kx].T).reshape(h, w, cout)
    if relu:
        out = np.maximum(out, 0.0)
    return out


def pooled_size(n):
    """Pool output extent: ceil(n / 2) (reading for odd extents)."""
    return (n + 1) // 2


def maxpool2x2(x):
    """2x2 / stride 2 max-pool over the valid pixels of each window
    ("nativeUNet.ts", createMaxPoolShader: out-of-range inputs skipped).
    """
    x = np.asarray(x)
    h, w, c = x.shape
    ho, wo = pooled_size(h), pooled_size(w)
    out = np.full((ho, wo, c), -np.inf, dtype=np.float64)
    for py in range(2):
        for px in range(2):
            part = x[py::2, px::2].astype(np.float64)
            out[:part.shape[0], :part.shape[1]] = np.maximum(
                out[:part.shape[0], :part.shape[1]], part)
    return out


def upsample2x(x, height, width):
    """Nearest 2x upsample cropped to [height, width]: out[y, x] =
    in[y >> 1, x >> 1] ("nativeUNet.ts", createTiledDecoderShader: the
    upsampled source is read at (x/2, y/2))."""
    x = np.asarray(x)
    rows = np.arange(height) >> 1
    cols = np.arange(width) >> 1
    return x[rows][:, cols]


def concat(a, b):
    """Channel concatenation [a, b] (reading: the upsampled source first)."""
    return np.concatenate([np.asarray(a), np.asarray(b)], axis=-1)


def decoder_input(low, skip):
    """Decoder conv input: concat(upsample2x(low) cropped to skip, skip)."""
    h, w = skip.shape[:2]
    return concat(upsample2x(low, h, w), skip)
