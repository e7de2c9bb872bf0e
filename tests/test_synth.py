"""The seeded input generator: voxelisation against brute force, determinism, targets."""
import numpy as np
import pytest
import torch

from synth import CONFIGS, ellipsoid_shell, make_coords, make_values, round_to_bf16, torus_shell
from synth.shells import uniform_rotation


def brute_grid(res):
    z, y, x = np.meshgrid(np.arange(res), np.arange(res), np.arange(res), indexing="ij")
    return np.stack([z.ravel(), y.ravel(), x.ravel()], axis=1).astype(np.float64)


def as_set(pts):
    return set(map(tuple, np.asarray(pts, np.int64).tolist()))


@pytest.mark.parametrize("seed", range(6))
def test_ellipsoid_shell_equals_full_grid_scan(seed):
    rng = np.random.default_rng(seed)
    res = 40
    axes = 4 + 14 * rng.random(3)
    rot = uniform_rotation(rng)
    c = 6 + 28 * rng.random(3)          # may cross the grid edge: clipping is part of the test
    P = brute_grid(res)
    u = (P - c) @ rot
    q = np.sqrt(((u / axes) ** 2).sum(1))
    want = P[np.abs(q - 1) * axes.mean() <= 0.5]
    assert as_set(ellipsoid_shell(res, c, axes, rot)) == as_set(want)


@pytest.mark.parametrize("seed", range(6))
def test_torus_shell_equals_full_grid_scan(seed):
    rng = np.random.default_rng(100 + seed)
    res = 48
    R, r = 6 + 12 * rng.random(), 1.5 + 5 * rng.random()
    rot = uniform_rotation(rng) if seed else np.eye(3)     # seed 0: axis along x exactly
    c = 10 + 28 * rng.random(3)
    P = brute_grid(res)
    u = (P - c) @ rot
    d = np.hypot(np.hypot(u[:, 0], u[:, 1]) - R, u[:, 2])
    want = P[np.abs(d - r) <= 0.5]
    assert as_set(torus_shell(res, c, R, r, rot)) == as_set(want)


def test_rotation_is_orthonormal():
    rng = np.random.default_rng(0)
    for _ in range(20):
        R = uniform_rotation(rng)
        np.testing.assert_allclose(R @ R.T, np.eye(3), atol=1e-12)
        assert np.linalg.det(R) > 0


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(100_000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3.0e38, -1e-40],
                                 np.float32)])
    v, bits = round_to_bf16(x)
    t = torch.from_numpy(x).to(torch.bfloat16)
    np.testing.assert_array_equal(bits, t.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(v, t.to(torch.float32).numpy())


@pytest.mark.parametrize("cfg_id", [1, 2, 3, 4])
def test_workload_counts_and_determinism(cfg_id):
    cfg = CONFIGS[cfg_id]
    c, info = make_coords(cfg_id)
    c2, _ = make_coords(cfg_id)
    np.testing.assert_array_equal(c, c2)
    assert c.dtype == np.int32 and c.shape[1] == 4
    keys = ((c[:, 0].astype(np.int64) * cfg["res"] + c[:, 1]) * cfg["res"] + c[:, 2]) * cfg["res"] + c[:, 3]
    assert (np.diff(keys) > 0).all()                       # raster order, no duplicates
    assert c[:, 1:].min() >= 0 and c[:, 1:].max() < cfg["res"]
    assert set(np.unique(c[:, 0])) == set(range(cfg["batch"]))
    if cfg["target"]:
        for b in range(cfg["batch"]):
            n = int((c[:, 0] == b).sum())
            assert abs(n - cfg["target"]) <= 0.2 * cfg["target"]
    else:
        assert 250 <= c.shape[0] <= 450                     # sphere shell r = 5 in 16^3
    s, _ = make_coords(cfg_id, "shuffled")
    assert as_set(s) == as_set(c) and not np.array_equal(s, c)


def test_values_distribution():
    v = make_values(20_000, 64, 48, "bf16", 3)
    assert v["feats"].shape == (20_000, 64) and v["weight"].shape == (48, 3, 3, 3, 64)
    assert abs(v["feats"].std() - 1) < 0.01
    assert abs(v["weight"].std() - 1 / np.sqrt(27 * 64)) < 0.01 / np.sqrt(27 * 64) * 5
    assert abs(v["bias"].std() - 0.1) < 0.05
    back, _ = round_to_bf16(v["feats"])
    np.testing.assert_array_equal(back, v["feats"])
