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


def test_make_residual_is_seeded_bf16_exact_and_standard_normal():
    from synth import make_residual, make_values
    r1, bits1 = make_residual(5000, 64, "bf16", 5)
    r2, bits2 = make_residual(5000, 64, "bf16", 5)
    np.testing.assert_array_equal(bits1, bits2)
    np.testing.assert_array_equal(r1, r2)
    # bf16-exact: the low 16 bits of every float32 are zero, and the bits are the high half
    u = r1.view(np.uint32)
    assert not (u & 0xFFFF).any()
    np.testing.assert_array_equal((u >> 16).astype(np.uint16), bits1)
    assert abs(r1.mean()) < 0.02 and abs(r1.std() - 1) < 0.02
    # its own stream: not a copy of the features drawn from the same seed
    f = make_values(5000, 64, 64, "bf16", 5)["feats"]
    assert not np.array_equal(f, r1)
    r3, none = make_residual(10, 3, "f32", 1)
    assert none is None and r3.dtype == np.float32 and r3.shape == (10, 3)


def test_bench_roofline_bytes_with_and_without_residual():
    import bench
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 1000.0}
    N, P, I, O = 1000, 11000, 64, 64
    a = bench.roofline(N, P, I, O, 1e-3, peaks, "measured", "none", e=2)
    b = bench.roofline(N, P, I, O, 1e-3, peaks, "measured", "none", e=2, residual=True)
    assert a["algorithmic_bytes"] == P * I * 2 + N * O * 2 + 108 * N + 27 * I * O * 2
    assert b["algorithmic_bytes"] - a["algorithmic_bytes"] == N * O * 2
    assert b["compulsory_bytes"] - a["compulsory_bytes"] == N * O * 2
    assert abs(a["frac"] - a["algorithmic_bytes"] / 1e-3 / 1e9 / 1000.0) < 1e-12
    c = bench.roofline(N, P, I, O, 1e-3, peaks, "measured", "none", e=4)
    assert c["kernel"] == "fwd_simt" and c["algorithmic_bytes"] == 2 * a["algorithmic_bytes"] - 108 * N
