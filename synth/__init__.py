"""Seeded synthetic inputs for the U-Net denoiser forward pass.

This module only draws random numbers; it holds none of the denoiser's
arithmetic.  Both the CPU oracle and the CUDA path (tests, bench) take their
inputs from here, so the two sides see the same bytes.

Workload recipe (the pages publish no dataset; these stand in for images):

* colour (seed 1): rgb i.i.d. lognormal(mu=-1, sigma=1.5) for HDR runs, or
  U[0,1] for LDR runs; alpha U[0,1] so that the alpha copy is exercised.
* albedo (seed 2): rgb U[0,1], alpha 1.
* normal (seed 3): rgb = a random unit vector (normalised standard normal
  draw), components in [-1,1], alpha 1.
* NaN/Inf mask (seed 4): a fraction of pixels whose rgb is replaced by one of
  {NaN, +Inf, -Inf}, chosen uniformly per pixel.
* conv weights (seed 1000 + layer index): He-uniform
  W ~ U[-sqrt(6/(9*Cin)), +sqrt(6/(9*Cin))], OIHW float32; bias zero unless
  a bias scale is asked for (tests use a non-zero bias to exercise the add).
* single-layer activations: U[-1,1].

All images are float32 arrays of shape [H, W, 4] (RGBA, row-major), the
layout the denoise call takes.
"""

import numpy as np

# Layer names and logical channel counts of the OIDN-shaped U-Net used by
# the workloads (encoder 9->32->32,pool,->48,pool,->64,pool,->80,pool,->96->96;
# decoder up+cat 160->112->112, up+cat 160->96->96, up+cat 128->64->64,
# up+cat 73->64->32->3).  Only the shapes live here: the dataflow between the
# layers is part of the method and is written separately by each side.
UNET_LAYERS = (
    "enc_conv0", "enc_conv1", "enc_conv2", "enc_conv3", "enc_conv4",
    "enc_conv5a", "enc_conv5b",
    "dec_conv4a", "dec_conv4b", "dec_conv3a", "dec_conv3b",
    "dec_conv2a", "dec_conv2b", "dec_conv1a", "dec_conv1b", "dec_conv0",
)


def unet_shapes(in_channels=9):
    """(Cout, Cin) per layer for the OIDN-shaped U-Net with `in_channels`."""
    ec1, ec2, ec3, ec4, ec5 = 32, 48, 64, 80, 96
    dc4, dc3, dc2, dc1 = 112, 96, 64, 32
    return {
        "enc_conv0": (ec1, in_channels),
        "enc_conv1": (ec1, ec1),
        "enc_conv2": (ec2, ec1),
        "enc_conv3": (ec3, ec2),
        "enc_conv4": (ec4, ec3),
        "enc_conv5a": (ec5, ec4),
        "enc_conv5b": (ec5, ec5),
        "dec_conv4a": (dc4, ec5 + ec3),
        "dec_conv4b": (dc4, dc4),
        "dec_conv3a": (dc3, dc4 + ec2),
        "dec_conv3b": (dc3, dc3),
        "dec_conv2a": (dc2, dc3 + ec1),
        "dec_conv2b": (dc2, dc2),
        "dec_conv1a": (64, dc2 + in_channels),
        "dec_conv1b": (dc1, 64),
        "dec_conv0": (3, dc1),
    }


def he_uniform_conv(cout, cin, seed, bias_scale=0.0):
    """One 3x3 conv: He-uniform OIHW float32 weight and float32 bias."""
    rng = np.random.Generator(np.random.PCG64(seed))
    bound = np.sqrt(6.0 / (9.0 * cin))
    w = rng.uniform(-bound, bound, size=(cout, cin, 3, 3)).astype(np.float32)
    if bias_scale:
        b = rng.uniform(-bias_scale, bias_scale, size=(cout,)).astype(np.float32)
    else:
        b = np.zeros((cout,), np.float32)
    return w, b


def unet_weights(in_channels=9, seed_base=1000, bias_scale=0.0):
    """dict layer name -> (weight OIHW f32, bias f32) for the whole U-Net."""
    shapes = unet_shapes(in_channels)
    out = {}
    for index, name in enumerate(UNET_LAYERS):
        cout, cin = shapes[name]
        out[name] = he_uniform_conv(cout, cin, seed_base + index, bias_scale)
    return out


def hdr_color(width, height, seed=1):
    rng = np.random.Generator(np.random.PCG64(seed))
    img = np.empty((height, width, 4), np.float32)
    img[..., :3] = rng.lognormal(mean=-1.0, sigma=1.5, size=(height, width, 3))
    img[..., 3] = rng.uniform(0.0, 1.0, size=(height, width))
    return img


def ldr_color(width, height, seed=1):
    rng = np.random.Generator(np.random.PCG64(seed))
    img = np.empty((height, width, 4), np.float32)
    img[..., :3] = rng.uniform(0.0, 1.0, size=(height, width, 3))
    img[..., 3] = rng.uniform(0.0, 1.0, size=(height, width))
    return img


def albedo(width, height, seed=2):
    rng = np.random.Generator(np.random.PCG64(seed))
    img = np.ones((height, width, 4), np.float32)
    img[..., :3] = rng.uniform(0.0, 1.0, size=(height, width, 3))
    return img


def normal(width, height, seed=3):
    rng = np.random.Generator(np.random.PCG64(seed))
    v = rng.standard_normal(size=(height, width, 3))
    n = v / np.maximum(np.linalg.norm(v, axis=-1, keepdims=True), 1e-30)
    img = np.ones((height, width, 4), np.float32)
    img[..., :3] = np.clip(n, -1.0, 1.0)
    return img


def inject_nan_inf(img, fraction=0.05, seed=4):
    """Copy of `img` with `fraction` of its pixels' rgb set to NaN/+Inf/-Inf."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = img.copy()
    h, w = img.shape[:2]
    mask = rng.uniform(0.0, 1.0, size=(h, w)) < fraction
    kind = rng.integers(0, 3, size=(h, w))
    specials = np.array([np.nan, np.inf, -np.inf], np.float32)
    vals = specials[kind]
    for c in range(3):
        out[..., c] = np.where(mask, vals, out[..., c])
    return out


def uniform_activations(height, width, channels, seed=5, low=-1.0, high=1.0):
    """[H, W, C] float32 activations drawn U[low, high]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.uniform(low, high, size=(height, width, channels)).astype(np.float32)


def denoise_inputs(width, height, sources=3, hdr=True, nan_fraction=0.0):
    """The colour/albedo/normal images of one workload, in input order."""
    color = hdr_color(width, height) if hdr else ldr_color(width, height)
    if nan_fraction:
        color = inject_nan_inf(color, nan_fraction)
    imgs = [color, albedo(width, height), normal(width, height)]
    return imgs[:sources]
