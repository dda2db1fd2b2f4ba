"""Test helpers: conversions between logical [H, W, C] arrays and the
library's activation layout (16-byte channel blocks, block index above x):
fp16 [H][L/8][W][8] with L = C rounded up to 16, fp32 [H][L/4][W][4] with
L = C rounded up to 4; padded lanes zero."""

import numpy as np


def lanes(c, precision):
    return -(-c // 16) * 16 if precision == "fp16" else -(-c // 4) * 4


def to_internal(x, precision):
    h, w, c = x.shape
    per = 8 if precision == "fp16" else 4
    dt = np.float16 if precision == "fp16" else np.float32
    full = np.zeros((h, w, lanes(c, precision)), dt)
    full[..., :c] = x.astype(dt)
    return np.ascontiguousarray(full.reshape(h, w, -1, per).transpose(0, 2, 1, 3))


def from_internal(buf, h, w, c, precision):
    per = 8 if precision == "fp16" else 4
    arr = np.asarray(buf).reshape(h, -1, w, per).transpose(0, 2, 1, 3).reshape(h, w, -1)
    return arr[..., :c]


def internal_nbytes(h, w, c, precision):
    return h * w * lanes(c, precision) * (2 if precision == "fp16" else 4)
