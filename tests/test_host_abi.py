"""CPU tests of the C-ABI library: it loads, exports every declared symbol,
and its host-only logic (tile planner, overlap, blob validation, argument
checks) agrees with the oracle's reading.  No kernel runs here."""

import os
import re
import subprocess

import numpy as np
import pytest

import synth
from oracle import tiles

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ox():
    import conv2d_implicit_gemm_gb300 as m
    return m


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "oidnx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oidnx_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol(ox):
    declared = _declared_symbols()
    assert len(declared) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", ox.LIBRARY_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    for s in declared:
        assert hasattr(ox._lib, s)


def test_default_overlap_matches_oracle(ox):
    assert ox.oidnx_default_overlap() == tiles.default_overlap() == 96


def test_tile_planner_matches_oracle(ox):
    cases = [(1920, 1080, 0, 96), (3840, 2160, 1024, 96), (300, 70, 256, 96),
             (1, 1, 0, 96), (17, 33, 0, 16), (4097, 100, 512, 32), (640, 480, 224, 96)]
    for w in range(1, 700, 37):
        for limit in (256, 300, 1024):
            cases.append((w, 200, limit, 96))
    for w, h, limit, overlap in cases:
        ref = tiles.plan_tile_grid(w, h, limit, overlap)
        got = ox.oidnx_plan_tiles(w, h, limit, overlap)
        assert got == [(t["input"], t["output"]) for t in ref], (w, h, limit, overlap)


def test_tile_planner_rejects_small_tiles(ox):
    with pytest.raises(ox.OidnxError) as e:
        ox.oidnx_plan_tiles(1000, 1000, 128, 96)
    assert e.value.status == ox.ERR_INVALID_ARGUMENT
    with pytest.raises(ox.OidnxError):
        ox.oidnx_plan_tiles(0, 10, 0, 96)


def _blob(ox, in_channels=9, **changes):
    w = synth.unet_weights(in_channels)
    w.update(changes)
    return ox.write_weight_blob(w)


@pytest.mark.parametrize("mutate,expected", [
    (lambda b: b"XXXX" + b[4:], "magic"),
    (lambda b: b[:4] + b"\x02\x00\x00\x00" + b[8:], "version"),
    (lambda b: b[:len(b) // 2], "truncated"),
    (lambda b: b[:16], "truncated"),
])
def test_corrupt_blob_is_invalid_model(ox, mutate, expected):
    blob = mutate(_blob(ox))
    with pytest.raises(ox.OidnxError) as e:
        ox.oidnx_filter_create(blob, ox.PRECISION_FP16)
    assert e.value.status == ox.ERR_INVALID_MODEL
    assert expected in str(e.value) or "missing" in str(e.value)


def test_wrong_topology_is_invalid_model(ox):
    w = synth.unet_weights(9)
    w["dec_conv4a"] = synth.he_uniform_conv(112, 150, 7)   # should be 160 inputs
    with pytest.raises(ox.OidnxError) as e:
        ox.oidnx_filter_create(ox.write_weight_blob(w))
    assert e.value.status == ox.ERR_INVALID_MODEL and "dec_conv4a" in str(e.value)
    w = synth.unet_weights(9)
    del w["enc_conv2"]
    with pytest.raises(ox.OidnxError) as e:
        ox.oidnx_filter_create(ox.write_weight_blob(w))
    assert "enc_conv2" in str(e.value)


def test_input_channel_count_is_validated(ox):
    # 4 input channels: not 3, 6 or 9
    w = synth.unet_weights(4)
    with pytest.raises(ox.OidnxError) as e:
        ox.oidnx_filter_create(ox.write_weight_blob(w))
    assert e.value.status == ox.ERR_INVALID_MODEL
    assert "3, 6, or 9" in str(e.value)


def test_null_arguments_are_rejected(ox):
    assert ox._lib.oidnx_filter_create(None, 0, 0, None) == ox.ERR_INVALID_ARGUMENT
    assert "NULL" in ox.oidnx_last_error()
    assert ox._lib.oidnx_filter_commit(None) == ox.ERR_INVALID_ARGUMENT
    assert ox._lib.oidnx_filter_execute(None, None) == ox.ERR_INVALID_ARGUMENT
    ox.oidnx_filter_release(None)   # ignored
    assert ox._lib.oidnx_conv_execute(None, None, None, 1, 1, 1, None) == ox.ERR_INVALID_ARGUMENT
    with pytest.raises(ox.OidnxError):
        ox.oidnx_filter_create(_blob(ox), precision=7)


def test_blob_writer_round_trips_half_weights(ox):
    # f16 blobs parse too (the parser widens them exactly); validation passes
    # and only the device step can fail on a machine without a GPU.
    blob = ox.write_weight_blob(synth.unet_weights(9), dtype="f16")
    try:
        f = ox.oidnx_filter_create(blob, ox.PRECISION_FP16)
    except ox.OidnxError as e:
        assert e.status in (ox.ERR_CUDA, ox.ERR_OUT_OF_MEMORY)
    else:
        ox.oidnx_filter_release(f)
