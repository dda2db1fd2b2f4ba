"""Pins of the oracle's input/output passes (golden closed-form fixture,
clamp-to-edge, lane order) and of its tile planner (brute-force invariants,
dependency radius measured by perturbing the oracle network)."""

import os

import numpy as np
import pytest

from oracle import passes, tiles, unet
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pass_cases.txt")


def _golden(kind):
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == kind:
                rows.append(parts[1:])
    assert rows
    return rows


@pytest.mark.parametrize("precision", ["fp16", "fp32"])
def test_pack_golden_cases(precision):
    sources = {"color": 0, "albedo": 1, "normal": 2}
    for source, hdr, scale, value, expected in _golden("pack"):
        imgs = [np.full((1, 1, 4), 0.25, np.float32) for _ in range(3)]
        imgs[sources[source]][0, 0, :3] = np.float32(float(value))
        out = passes.pack_tile(imgs, (0, 0, 1, 1), bool(int(hdr)), float(scale), precision)
        ch = out[0, 0, 3 * sources[source]:3 * sources[source] + 3].astype(np.float64)
        assert np.array_equal(ch, np.full(3, float(expected))), (source, hdr, scale, value, ch)


def test_unpack_golden_cases():
    for hdr, scale, value, expected in _golden("unpack"):
        net = np.full((1, 1, 4), np.float32(float(value)))
        color = np.zeros((1, 1, 4), np.float32)
        out = passes.unpack_rect(net, color, bool(int(hdr)), float(scale))
        assert np.array_equal(out[0, 0, :3], np.full(3, np.float32(float(expected)))), (hdr, scale, value)


def test_unpack_copies_alpha_bits():
    color = np.zeros((1, 4, 4), np.float32)
    alpha_bits = np.array([0x7FC01234, 0x3F800000, 0x80000000, 0x00000001], np.uint32)
    color[..., 3] = alpha_bits.view(np.float32)
    out = passes.unpack_rect(np.ones((1, 4, 4), np.float32), color, True, 1.0)
    assert np.array_equal(out[..., 3].view(np.uint32)[0], alpha_bits)


def test_pack_lane_order_and_clamp_to_edge():
    w, h = 3, 2
    imgs = []
    for s in range(3):
        img = np.zeros((h, w, 4), np.float32)
        for y in range(h):
            for x in range(w):
                img[y, x, :3] = [(s * 100 + y * 10 + x + c * 0.5) / 1000 for c in range(3)]
        imgs.append(img)
    out = passes.pack_tile(imgs, (-2, -1, 6, 4), False, 1.0, "fp32")
    assert out.shape == (4, 6, 9)
    for ty in range(4):
        for tx in range(6):
            sy = min(max(ty - 1, 0), h - 1)
            sx = min(max(tx - 2, 0), w - 1)
            for s in range(3):
                for c in range(3):
                    v = imgs[s][sy, sx, c]
                    if s == 2:
                        v = np.float32(v) * np.float32(0.5) + np.float32(0.5)
                    assert out[ty, tx, 3 * s + c] == np.float32(v)
    # fewer sources: only the first 3*S channels
    assert passes.pack_tile(imgs[:1], (0, 0, 3, 2), False, 1.0, "fp16").shape == (2, 3, 3)
    assert passes.pack_tile(imgs[:2], (0, 0, 3, 2), False, 1.0, "fp16").shape == (2, 3, 6)


def _check_axis(extent, limit, overlap):
    plan = tiles.plan_axis(extent, limit, overlap)
    ea = tiles.align_up(extent)
    covered = np.zeros(extent, np.int32)
    sizes = {t[1] for t in plan}
    assert len(sizes) == 1
    for s, size, o, n in plan:
        assert s % 16 == 0 and size % 16 == 0
        assert 0 <= s and s + size <= ea
        assert s <= o and o + n <= s + size
        covered[o:o + n] += 1
        if len(plan) > 1:
            assert size <= (limit // 16) * 16
            assert o - s >= overlap or s == 0
            assert s + size - (o + n) >= overlap or s + size == ea
    assert (covered == 1).all()
    return plan


def test_tile_planner_invariants_brute_force():
    count = 0
    for extent in list(range(1, 200, 7)) + [1080, 1920, 2160, 3840, 4097]:
        for limit in (128, 224, 256, 300, 512, 1024, 5000):
            for overlap in (0, 16, 32, 48, 96):
                if limit // 16 * 16 < 2 * overlap + 16 and tiles.align_up(extent) > limit // 16 * 16:
                    with pytest.raises(ValueError):
                        tiles.plan_axis(extent, limit, overlap)
                    continue
                _check_axis(extent, limit, overlap)
                count += 1
    assert count > 500


def test_tile_planner_4k_plan():
    # 3840x2160, maxTileSize 1024, overlap 96 (hand-worked from the reading)
    grid = tiles.plan_tile_grid(3840, 2160, 1024, 96)
    assert len(grid) == 15
    xs = sorted({t["input"][0] for t in grid})
    ys = sorted({t["input"][1] for t in grid})
    assert xs == [0, 672, 1440, 2208, 2880]
    assert ys == [0, 624, 1248]
    assert {t["input"][2:] for t in grid} == {(960, 912)}
    single = tiles.plan_tile_grid(1920, 1080, 0, 96)
    assert single == [{"input": (0, 0, 1920, 1088), "output": (0, 0, 1920, 1080)}]


def test_dependency_radius_is_covered_by_default_overlap():
    assert tiles.dependency_radius() == 94
    assert tiles.default_overlap() == 96


def test_dependency_radius_by_perturbing_the_network():
    """Brute force: change one input pixel, see which outputs move."""
    weights = synth.unet_weights(in_channels=3, bias_scale=0.1)
    w = 384
    rng = np.random.default_rng(0)
    x = rng.uniform(0.0, 1.0, size=(16, w, 3))
    base = unet.forward(x, weights, "fp32")
    worst = 0
    for p in (160, 167, 175):
        xp = x.copy()
        xp[5:11, p, :] += 1.0
        moved = np.abs(unet.forward(xp, weights, "fp32") - base).max(axis=(0, 2)) > 0
        idx = np.nonzero(moved)[0]
        worst = max(worst, p - idx.min(), idx.max() - p)
    assert 0 < worst <= tiles.dependency_radius()
