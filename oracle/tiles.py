"""Overlapping tile grid and the network's dependency radius.

The tile planner and OIDN_TILE_ALIGNMENT are imported by "oidn-webgpu
0.0.0-stage -> 0.6.0, src/native/denoise.ts" (recordDenoiseExecution) but not
shown.  That function fixes: overlap = alignUp(receptiveField / 2, ALIGN);
tile limit = maxTileSize, or alignUp(max(W, H), ALIGN) when maxTileSize is 0;
tiles carry an input rectangle and an output rectangle.  The rest is the
reading below (per axis, on the padded extent Ea = alignUp(E, 16)):

* T' = floor16(limit).  If Ea <= T': one tile, input [0, Ea), output [0, E).
* Else the smallest n >= 2 with c + 2*O <= T', c = alignUp(ceil(Ea / n), 16);
  none -> error.  Every tile's input size is S = c + 2*O.
* Output cuts o_i = i*c (i < n), o_n = Ea; input start
  s_i = clamp(o_i - O, 0, Ea - S); output [o_i, min(o_{i+1}, E)).
"""

ALIGN = 16


def align_up(v, a=ALIGN):
    return -(-v // a) * a


def plan_axis(extent, limit, overlap):
    """List of (input_start, input_size, output_start, output_size)."""
    if extent <= 0 or overlap < 0 or overlap % ALIGN:
        raise ValueError("bad axis")
    ea = align_up(extent)
    tmax = (limit // ALIGN) * ALIGN
    if ea <= tmax:
        return [(0, ea, 0, extent)]
    n = 2
    while True:
        c = align_up(-(-ea // n))
        if c + 2 * overlap <= tmax:
            break
        if c <= ALIGN:
            raise ValueError("maxTileSize too small for the overlap")
        n += 1
    size = c + 2 * overlap
    tiles = []
    for i in range(n):
        o = i * c
        o_next = (i + 1) * c if i + 1 < n else ea
        s = min(max(o - overlap, 0), ea - size)
        tiles.append((s, size, o, min(o_next, extent) - o))
    return [t for t in tiles if t[3] > 0]


def plan_tile_grid(width, height, max_tile_size, overlap):
    """Tiles as dicts {input: (x, y, w, h), output: (x, y, w, h)}, row-major."""
    limit = max_tile_size if max_tile_size > 0 else align_up(max(width, height))
    xs = plan_axis(width, limit, overlap)
    ys = plan_axis(height, limit, overlap)
    tiles = []
    for (sy, sh, oy, ohh) in ys:
        for (sx, sw, ox, oww) in xs:
            tiles.append({"input": (sx, sy, sw, sh), "output": (ox, oy, oww, ohh)})
    return tiles


def dependency_interval(p, levels=4):
    """Input positions (1-D) that network output position p depends on.

    Walks the U-Net backwards with interval arithmetic: a same-padded 3x3
    conv widens [a, b] to [a-1, b+1]; a 2x2 pool's input for output [a, b]
    is [2a, 2b+1]; a nearest upsample's source for [a, b] is [a>>1, b>>1];
    a concat is the union of its two sources.  Network: enc_conv0, enc_conv1,
    pool (skip 1); per further level one conv and a pool (skips 2..levels-1,
    then the bottom pool); two convs at the bottom; per decoder level
    up + concat(skip) and two convs; the finest skip is the network input;
    a final conv.
    """
    def conv(iv):
        return (iv[0] - 1, iv[1] + 1)

    def pool_src(iv):
        return (2 * iv[0], 2 * iv[1] + 1)

    def up_src(iv):
        return (iv[0] >> 1, iv[1] >> 1)

    def union(a, b):
        return (min(a[0], b[0]), max(a[1], b[1]))

    def pooled(iv, level):
        """Input interval for interval `iv` of the pooled value at `level`
        (level 0 is the network input itself)."""
        if level == 0:
            return iv
        src = conv(pool_src(iv))          # conv that feeds this pool
        if level == 1:
            return conv(src)              # enc_conv0 feeds enc_conv1
        return pooled(src, level - 1)

    def decoded(iv, level):
        """Input interval for `iv` of the decoder output at `level`
        (level == levels means the bottom: two convs on the last pool)."""
        if level == levels:
            return pooled(conv(conv(iv)), levels)
        cat = conv(conv(iv))              # the level's two convs
        return union(decoded(up_src(cat), level + 1), pooled(cat, level))

    return decoded(conv((p, p)), 0)


def dependency_radius(levels=4, align=ALIGN):
    """Largest one-sided distance from an output position to an input
    position it depends on, over positions at every residue mod `align`."""
    base = 10 * align * (1 << levels)
    r = 0
    for res in range(align):
        p = base + res
        lo, hi = dependency_interval(p, levels)
        r = max(r, p - lo, hi - p)
    return r


def default_overlap(levels=4):
    """alignUp(receptiveField / 2, ALIGN) with the receptive field taken as
    the full dependency span 2 * radius (+1 for the centre)."""
    radius = dependency_radius(levels)
    return align_up((2 * radius + 1) // 2)
