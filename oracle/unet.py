"""The 16-layer OIDN-style U-Net and the whole tiled denoise, float64.

Dataflow ("oidn-web 0.3.4 -> 0.4.0, nativeUNet.ts", the graph the executor
runs: conv2d, fused conv+ReLU+max-pool, fused upsample+concat+conv):

  enc_conv0 -> enc_conv1 -> pool1 -> enc_conv2 -> pool2 -> enc_conv3 -> pool3
  -> enc_conv4 -> pool4 -> enc_conv5a -> enc_conv5b
  -> dec_conv4a(up(enc_conv5b) ++ pool3) -> dec_conv4b
  -> dec_conv3a(up(dec_conv4b) ++ pool2) -> dec_conv3b
  -> dec_conv2a(up(dec_conv3b) ++ pool1) -> dec_conv2b
  -> dec_conv1a(up(dec_conv2b) ++ input) -> dec_conv1b -> dec_conv0

Every conv has ReLU except dec_conv0.  Precision modes:

* "fp32": weights and activations stored as float32;
* "fp16": weights rounded to fp16, bias kept float32 ("packConvTensors":
  bias stays f32), every stored activation rounded to fp16, the final layer
  stored as float32 (the executor allocates the output at 4 bytes/scalar).

Accumulation is exact up to float64 rounding in both modes (reading: the
pages' fp16 kernels sum fp16 partials; this build accumulates in fp32 and
compares against the float64 sum within a tolerance).
"""

import numpy as np

from . import layers
from .numerics import round_storage
from .passes import pack_tile, unpack_rect
from .tiles import default_overlap, plan_tile_grid

ENCODER = ("enc_conv0", "enc_conv1", "enc_conv2", "enc_conv3", "enc_conv4")


def _weights_in_precision(weights, precision):
    out = {}
    for name, (w, b) in weights.items():
        wq = round_storage(np.asarray(w, np.float32), precision).astype(np.float64)
        out[name] = (wq, np.asarray(b, np.float32).astype(np.float64))
    return out


def forward(packed_input, weights, precision, keep=False):
    """Run the network on one packed input.

    packed_input: [h, w, Cin] array already in storage precision (the pack
    pass output).  weights: dict name -> (OIHW float32, bias float32).
    Returns the float32 network output [h, w, 3]; with keep=True a dict of
    every stored value (layer name, plus 'pool1'..'pool4') as float64.
    """
    wts = _weights_in_precision(weights, precision)
    x = np.asarray(packed_input).astype(np.float64)
    values = {"input": x}

    def conv(name, inp, relu=True, final=False):
        w, b = wts[name]
        y = layers.conv3x3(inp, w, b, relu)
        y = round_storage(y, "fp32" if final else precision).astype(np.float64)
        values[name] = y
        return y

    def pool(name, inp):
        y = layers.maxpool2x2(inp)
        values[name] = y
        return y

    e = conv("enc_conv0", x)
    e = conv("enc_conv1", e)
    p1 = pool("pool1", e)
    p2 = pool("pool2", conv("enc_conv2", p1))
    p3 = pool("pool3", conv("enc_conv3", p2))
    p4 = pool("pool4", conv("enc_conv4", p3))
    b = conv("enc_conv5b", conv("enc_conv5a", p4))
    d = conv("dec_conv4b", conv("dec_conv4a", layers.decoder_input(b, p3)))
    d = conv("dec_conv3b", conv("dec_conv3a", layers.decoder_input(d, p2)))
    d = conv("dec_conv2b", conv("dec_conv2a", layers.decoder_input(d, p1)))
    d = conv("dec_conv1b", conv("dec_conv1a", layers.decoder_input(d, x)))
    out = conv("dec_conv0", d, relu=False, final=True)
    if keep:
        return values
    return out.astype(np.float32)


def denoise(images, weights, hdr, input_scale=1.0, max_tile_size=0,
            overlap=None, precision="fp16"):
    """Whole denoise of a W x H image ("denoise.ts", recordDenoiseExecution):
    per tile of the grid, the input pass, the network, and the output pass
    into the tile's output rectangle.  Returns float32 [H, W, 4]."""
    height, width = images[0].shape[:2]
    if overlap is None:
        overlap = default_overlap()
    out = np.zeros((height, width, 4), np.float32)
    for tile in plan_tile_grid(width, height, max_tile_size, overlap):
        ix, iy, iw, ih = tile["input"]
        ox, oy, ow, oh = tile["output"]
        packed = pack_tile(images, (ix, iy, iw, ih), hdr, input_scale, precision)
        net = forward(packed, weights, precision)
        region = net[oy - iy:oy - iy + oh, ox - ix:ox - ix + ow]
        color = images[0][oy:oy + oh, ox:ox + ow]
        out[oy:oy + oh, ox:ox + ow] = unpack_rect(region, color, hdr, input_scale)
    return out


def conv_flops(shapes, width, height):
    """Logical conv FLOPs of one network pass on a width x height tile:
    sum over layers of 2 * 9 * Cin * Cout * (pixels at the layer's level)."""
    level_of = {
        "enc_conv0": 0, "enc_conv1": 0, "enc_conv2": 1, "enc_conv3": 2,
        "enc_conv4": 3, "enc_conv5a": 4, "enc_conv5b": 4,
        "dec_conv4a": 3, "dec_conv4b": 3, "dec_conv3a": 2, "dec_conv3b": 2,
        "dec_conv2a": 1, "dec_conv2b": 1, "dec_conv1a": 0, "dec_conv1b": 0,
        "dec_conv0": 0,
    }
    total = 0
    for name, (cout, cin) in shapes.items():
        w, h = width, height
        for _ in range(level_of[name]):
            w, h = (w + 1) // 2, (h + 1) // 2
        total += 2 * 9 * cin * cout * w * h
    return total
