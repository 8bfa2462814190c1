"""Pins for the oracle's scheduling units and chunk plan (CPU only).

Against the numbers the teardown prints for the shipped configuration
(tests/golden/unit_rhythm.txt), against a brute-force walk of the codec's
latents (glue the one-frame latent of each group of five to its neighbour,
then count), and against the structural facts the plan must satisfy: units
partition the latents, chunks follow one another without gaps, and the recent
history of a chunk ends where the chunk begins.
"""
import os

import pytest

from oracle import chunk_plan, latent_rgb_frames, unit_latents, units_latents

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


G = _golden("unit_rhythm.txt")


def _units_brute(n_units, merge=True):
    """Walk latents in codec groups of five; with merging, the group's first
    latent (one RGB frame) joins the next latent in one unit."""
    units, lat = [], 0
    while len(units) < n_units:
        if merge and lat % 5 == 0:
            units.append([lat, lat + 1])
            lat += 2
        else:
            units.append([lat])
            lat += 1
    return units


def test_codec_group_of_five_latents_is_seventeen_frames():
    assert sum(latent_rgb_frames(l) for l in range(G["latents_per_group"])) == G["rgb_frames_per_group"]
    assert sum(latent_rgb_frames(l) for l in range(5, 10)) == G["rgb_frames_per_group"]


def test_units_match_the_brute_force_walk():
    units = _units_brute(40)
    assert [len(u) for u in units] == [unit_latents(u) for u in range(40)]
    assert [len(u) for u in units[:8]] == [2, 1, 1, 1, 2, 1, 1, 1]
    flat = [l for u in units for l in u]
    assert flat == list(range(len(flat)))           # units partition the latents
    assert all(unit_latents(u, False) == 1 for u in range(10))


def test_shipped_config_numbers_from_the_page():
    kw = dict(bootstrap_units=G["bootstrap_units"], chunk_units=G["chunk_units"],
              window_units=G["window_units"], sink_units=G["sink_units"])
    p0 = chunk_plan(0, **kw)
    assert p0["n_frames"] == G["bootstrap_latents"] and p0["hist_frames"] == 0
    assert sum(latent_rgb_frames(l) for l in range(p0["n_frames"])) == G["bootstrap_rgb_frames"]
    lat = []
    rgb = []
    for c in range(1, 9):
        p = chunk_plan(c, **kw)
        lat.append(p["n_frames"])
        rgb.append(sum(latent_rgb_frames(l) for l in range(p["first_latent"], p["first_latent"] + p["n_frames"])))
    assert lat == [G["chunk_latents_a"], G["chunk_latents_b"]] * 4
    assert rgb == [G["chunk_rgb_frames_a"], G["chunk_rgb_frames_b"]] * 4
    assert rgb[0] + rgb[1] == G["rgb_frames_per_two_chunks"]
    assert round(1000 * rgb[0] / G["fps"]) == G["chunk_ms_a"]
    assert int(1000 * rgb[1] / G["fps"]) == G["chunk_ms_b"]
    assert int(1000 * (rgb[0] + rgb[1]) / 2 / G["fps"]) == G["mean_chunk_ms"]
    side = G["vae_downsample"] * G["patch"]
    assert (G["video_height"] // side) * (G["video_width"] // side) == G["tokens_per_latent"]


@pytest.mark.parametrize("boot,cu,wu,su,merge", [(7, 2, 2, 2, True), (7, 2, 5, 4, True), (3, 1, 2, 1, True),
                                                 (7, 2, 2, 2, False), (9, 3, 4, 2, True)])
def test_plan_against_brute_force_units(boot, cu, wu, su, merge):
    units = _units_brute(boot + 30 * cu + 4, merge)
    nxt = 0
    for c in range(30):
        p = chunk_plan(c, boot, cu, wu, su, merge)
        u0 = 0 if c == 0 else boot + (c - 1) * cu
        mine = units[u0:u0 + (boot if c == 0 else cu)]
        lats = [l for u in mine for l in u]
        assert p["first_latent"] == lats[0] == nxt       # chunks follow one another without gaps
        assert p["n_frames"] == len(lats)
        nxt = lats[-1] + 1
        if c == 0:
            assert p["hist_frames"] == 0
        else:
            hist = [l for u in units[max(0, u0 - wu):u0] for l in u]
            assert p["hist_frames"] == len(hist)
            assert not hist or hist[-1] + 1 == p["first_latent"]   # history ends where the chunk begins
        assert p["sink_frames"] == len([l for u in units[:su] for l in u])
        assert units_latents(0, u0, merge) == p["first_latent"]


def test_negative_chunk_index_is_rejected():
    with pytest.raises(ValueError):
        chunk_plan(-1)
