"""Pins for the CPU oracle: each test checks it against something other than itself.

* brute-force pairwise neighbour search and a dense index-grid lookup (kernel map);
* a dense zero-padded Conv3d (torch CPU, float64, padding 1) on small grids, masked
  to the active sites -- equal to the submanifold convolution because inactive
  sites hold zeros;
* a hand-worked example (tests/golden/hand_worked.json);
* invariants: isolated voxel, single asymmetric tap, translation and permutation
  equivariance, linearity, batch independence, grid-boundary voxels, errors;
* the C++ oracle against all of the above and against the Python oracle.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import cpu, ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def random_set(rng, res, batch, n):
    """n distinct random lattice points per batch item (b, z, y, x) int32."""
    rows = []
    for b in range(batch):
        flat = rng.choice(res ** 3, size=n, replace=False)
        z, rem = np.divmod(flat, res * res)
        y, x = np.divmod(rem, res)
        rows.append(np.stack([np.full(n, b), z, y, x], axis=1))
    c = np.concatenate(rows).astype(np.int32)
    return c[rng.permutation(c.shape[0])]


def dense_masked_conv3d(coords, feats, weight, bias, res):
    """Dense zero-padded Conv3d (padding 1) on the densified grid, read at the active sites."""
    coords = np.asarray(coords)
    B = int(coords[:, 0].max()) + 1
    I = feats.shape[1]
    grid = torch.zeros(B, I, res, res, res, dtype=torch.float64)
    b, z, y, x = (torch.from_numpy(coords[:, k].astype(np.int64)) for k in range(4))
    grid[b, :, z, y, x] = torch.from_numpy(np.asarray(feats, np.float64))
    w = torch.from_numpy(np.asarray(weight, np.float64)).permute(0, 4, 1, 2, 3).contiguous()
    bt = None if bias is None else torch.from_numpy(np.asarray(bias, np.float64))
    out = F.conv3d(grid, w, bt, stride=1, padding=1)
    return out[b, :, z, y, x].numpy()


def brute_force_nbr(coords):
    """O(N^2): nbr[i, k] = j whenever coords[j] - coords[i] is offset k in the same batch item."""
    c = np.asarray(coords, np.int64)
    N = c.shape[0]
    nbr = np.full((N, 27), -1, np.int32)
    for i in range(N):
        d = c[:, 1:] - c[i, 1:]
        same = (c[:, 0] == c[i, 0]) & (np.abs(d).max(axis=1) <= 1)
        for j in np.nonzero(same)[0]:
            dz, dy, dx = d[j]
            nbr[i, 9 * (dz + 1) + 3 * (dy + 1) + (dx + 1)] = j
    return nbr


def dense_lookup_nbr(coords, res):
    """Index grid filled with -1, padded by one cell, read at the 27 shifted positions."""
    c = np.asarray(coords, np.int64)
    B = int(c[:, 0].max()) + 1
    grid = np.full((B, res + 2, res + 2, res + 2), -1, np.int64)
    grid[c[:, 0], c[:, 1] + 1, c[:, 2] + 1, c[:, 3] + 1] = np.arange(c.shape[0])
    cols = []
    for dz in (-1, 0, 1):
        for dy in (-1, 0, 1):
            for dx in (-1, 0, 1):
                cols.append(grid[c[:, 0], c[:, 1] + 1 + dz, c[:, 2] + 1 + dy, c[:, 3] + 1 + dx])
    return np.stack(cols, axis=1).astype(np.int32)


def rand_values(rng, N, I, O, with_bias=True):
    f = rng.standard_normal((N, I))
    w = rng.standard_normal((O, 3, 3, 3, I))
    b = rng.standard_normal(O) if with_bias else None
    return f, w, b


# ----------------------------------------------------------------------------- kernel map

@pytest.mark.parametrize("seed,res,batch,n", [(0, 4, 1, 20), (1, 5, 2, 40), (2, 6, 1, 120),
                                               (3, 3, 2, 27), (4, 7, 3, 60)])
def test_kernel_map_brute_force_and_dense_lookup(seed, res, batch, n):
    rng = np.random.default_rng(seed)
    c = random_set(rng, res, batch, n)
    want = brute_force_nbr(c)
    np.testing.assert_array_equal(ref.kernel_map(c, res), want)
    np.testing.assert_array_equal(dense_lookup_nbr(c, res), want)
    np.testing.assert_array_equal(cpu.kernel_map(c, res), want)


def test_kernel_map_full_block_and_symmetry():
    # a full 3x3x3 block: the centre sees all 27 neighbours, tap k holding the voxel at offset k
    c = np.array([[0, z, y, x] for z in range(3) for y in range(3) for x in range(3)], np.int32)
    nbr = ref.kernel_map(c, 3)
    np.testing.assert_array_equal(nbr[13], np.arange(27))
    # neighbour relation is symmetric: nbr[i, k] = j  <=>  nbr[j, 26 - k] = i
    rng = np.random.default_rng(7)
    c = random_set(rng, 6, 2, 90)
    nbr = ref.kernel_map(c, 6)
    for i, k in zip(*np.nonzero(nbr >= 0)):
        assert nbr[nbr[i, k], 26 - k] == i
    assert (nbr[:, 13] == np.arange(c.shape[0])).all()


def test_kernel_map_grid_boundary_and_batches():
    res = 5
    c = np.array([[0, 0, 0, 0], [0, 4, 4, 4], [1, 0, 0, 0], [1, 4, 4, 4], [0, 1, 1, 1]], np.int32)
    nbr = ref.kernel_map(c, res)
    # the corner voxels see nothing outside the grid, only their in-grid neighbours
    assert nbr[0, 26] == 4 and (np.delete(nbr[0], [13, 26]) == -1).all()
    assert (np.delete(nbr[1], 13) == -1).all()
    # identical (z, y, x) in another batch item is not a neighbour
    assert (np.delete(nbr[2], 13) == -1).all()
    np.testing.assert_array_equal(cpu.kernel_map(c, res), nbr)


@pytest.mark.parametrize("mod", [ref, cpu])
def test_errors(mod):
    with pytest.raises(ref.OracleError):
        mod.kernel_map(np.array([[0, 0, 0, 4]], np.int32), 4)
    with pytest.raises(ref.OracleError):
        mod.kernel_map(np.array([[0, -1, 0, 0]], np.int32), 4)
    with pytest.raises(ref.OracleError):
        mod.kernel_map(np.array([[-1, 0, 0, 0]], np.int32), 4)
    with pytest.raises(ref.OracleError):
        mod.kernel_map(np.array([[0, 1, 2, 3], [0, 0, 0, 0], [0, 1, 2, 3]], np.int32), 4)


# ----------------------------------------------------------------------------- forward

@pytest.mark.parametrize("seed,res,batch,n,I,O", [(0, 4, 1, 30, 3, 5), (1, 6, 2, 70, 4, 2),
                                                   (2, 8, 1, 200, 2, 3), (3, 5, 3, 50, 5, 4),
                                                   (4, 3, 1, 27, 2, 2)])
def test_forward_matches_dense_conv3d(seed, res, batch, n, I, O):
    rng = np.random.default_rng(seed)
    c = random_set(rng, res, batch, n)
    f, w, b = rand_values(rng, c.shape[0], I, O, with_bias=seed % 2 == 0)
    want = dense_masked_conv3d(c, f, w, b, res)
    got = ref.subm_conv3d(c, f, w, b, res)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * max(1.0, np.abs(want).max()))
    got_cpp = cpu.forward_rows(c, f.astype(np.float32), w.astype(np.float32),
                               None if b is None else b.astype(np.float32), res)
    want32 = dense_masked_conv3d(c, f.astype(np.float32), w.astype(np.float32),
                                 None if b is None else b.astype(np.float32), res)
    np.testing.assert_allclose(got_cpp, want32, rtol=0, atol=1e-12 * max(1.0, np.abs(want32).max()))


def test_forward_on_shell_matches_dense_conv3d():
    from synth import ellipsoid_shell, union_coords, uniform_rotation
    rng = np.random.default_rng(11)
    pts = ellipsoid_shell(20, (9.6, 10.2, 9.1), (6.5, 4.2, 7.7), uniform_rotation(rng))
    c = union_coords([(0, pts), (1, pts[::2])], 20)
    f, w, b = rand_values(rng, c.shape[0], 6, 7)
    want = dense_masked_conv3d(c, f, w, b, 20)
    np.testing.assert_allclose(ref.subm_conv3d(c, f, w, b, 20), want, rtol=0, atol=1e-11)
    np.testing.assert_allclose(
        cpu.forward_rows(c, f.astype(np.float32), w.astype(np.float32), b.astype(np.float32), 20),
        dense_masked_conv3d(c, f.astype(np.float32), w.astype(np.float32), b.astype(np.float32), 20),
        rtol=0, atol=1e-11)


def test_hand_worked_golden():
    spec = json.load(open(GOLDEN))
    for cs in spec["cases"]:
        c = np.array(cs["coords"], np.int32)
        N = c.shape[0]
        w = np.zeros((1, 3, 3, 3, 1))
        for kz in range(3):
            for ky in range(3):
                for kx in range(3):
                    w[0, kz, ky, kx, 0] = 1 + 9 * kz + 3 * ky + kx
        f = np.array(cs["feats"], np.float64).reshape(N, 1)
        b = np.array([cs["bias"]])
        want_nbr = np.full((N, 27), -1)
        for i, pairs in enumerate(cs["nbr_nonabsent"]):
            for k, j in pairs:
                want_nbr[i, k] = j
        for mod in (ref, cpu):
            np.testing.assert_array_equal(mod.kernel_map(c, cs["res"]), want_nbr, err_msg=cs["name"])
        np.testing.assert_array_equal(ref.subm_conv3d(c, f, w, b, cs["res"])[:, 0], cs["out"])
        np.testing.assert_array_equal(
            cpu.forward_rows(c, f.astype(np.float32), w.astype(np.float32),
                             b.astype(np.float32), cs["res"])[:, 0], cs["out"])


def test_isolated_voxel_sees_only_centre_tap():
    rng = np.random.default_rng(3)
    c = np.array([[0, 2, 2, 2], [0, 6, 6, 6], [1, 2, 2, 2]], np.int32)
    f, w, b = rand_values(rng, 3, 4, 5)
    out = ref.subm_conv3d(c, f, w, b, 9)
    for i in range(3):
        np.testing.assert_allclose(out[i], w[:, 1, 1, 1, :] @ f[i] + b, rtol=1e-14)


@pytest.mark.parametrize("tap", [(2, 1, 0), (0, 2, 1), (1, 0, 2), (0, 0, 0), (2, 2, 2)])
def test_single_asymmetric_tap_orientation(tap):
    """Only tap (kz, ky, kx) is non-zero: out at p reads the input at p + (tap - 1)."""
    rng = np.random.default_rng(5)
    c = random_set(rng, 5, 1, 60)
    f, _, _ = rand_values(rng, c.shape[0], 3, 2)
    w = np.zeros((2, 3, 3, 3, 3))
    w[:, tap[0], tap[1], tap[2], :] = rng.standard_normal((2, 3))
    out = ref.subm_conv3d(c, f, w, None, 5)
    index = {tuple(r): i for i, r in enumerate(c.tolist())}
    d = np.array(tap) - 1
    for i, (b, z, y, x) in enumerate(c.tolist()):
        j = index.get((b, z + d[0], y + d[1], x + d[2]))
        want = np.zeros(2) if j is None else w[:, tap[0], tap[1], tap[2], :] @ f[j]
        np.testing.assert_allclose(out[i], want, rtol=1e-14, atol=0)
    np.testing.assert_allclose(cpu.forward_rows(c, f.astype(np.float32), w.astype(np.float32),
                                                None, 5),
                               ref.subm_conv3d(c, f.astype(np.float32), w.astype(np.float32),
                                               None, 5), rtol=1e-13, atol=1e-13)


def test_translation_and_permutation_equivariance():
    rng = np.random.default_rng(9)
    c = random_set(rng, 6, 2, 80)
    f, w, b = rand_values(rng, c.shape[0], 3, 4)
    out = ref.subm_conv3d(c, f, w, b, 12)
    t = np.array([0, 3, 5, 2], np.int32)
    np.testing.assert_allclose(ref.subm_conv3d(c + t, f, w, b, 12), out, rtol=0, atol=1e-12)
    p = rng.permutation(c.shape[0])
    np.testing.assert_allclose(ref.subm_conv3d(c[p], f[p], w, b, 12), out[p], rtol=0, atol=1e-12)
    f32, w32, b32 = f.astype(np.float32), w.astype(np.float32), b.astype(np.float32)
    np.testing.assert_allclose(cpu.forward_rows(c[p], f32[p], w32, b32, 12),
                               cpu.forward_rows(c, f32, w32, b32, 12)[p], rtol=0, atol=1e-12)


def test_linearity_in_feats_and_weight():
    rng = np.random.default_rng(13)
    c = random_set(rng, 5, 1, 50)
    f1, w1, _ = rand_values(rng, c.shape[0], 3, 4)
    f2, w2, _ = rand_values(rng, c.shape[0], 3, 4)
    a, s = 0.7, -1.9
    conv = lambda f, w: ref.subm_conv3d(c, f, w, None, 5)
    np.testing.assert_allclose(conv(a * f1 + s * f2, w1), a * conv(f1, w1) + s * conv(f2, w1),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(conv(f1, a * w1 + s * w2), a * conv(f1, w1) + s * conv(f1, w2),
                               rtol=0, atol=1e-12)


def test_batch_items_are_independent():
    rng = np.random.default_rng(17)
    c0 = random_set(rng, 5, 1, 40)
    c1 = c0.copy()
    c1[:, 0] = 1
    f, w, b = rand_values(rng, 40, 3, 4)
    both = ref.subm_conv3d(np.concatenate([c0, c1]), np.concatenate([f, f]), w, b, 5)
    np.testing.assert_array_equal(both[:40], both[40:])
    np.testing.assert_array_equal(both[:40], ref.subm_conv3d(c0, f, w, b, 5))


def test_rows_subset_matches_full():
    rng = np.random.default_rng(19)
    c = random_set(rng, 7, 2, 100)
    f, w, b = (v.astype(np.float32) for v in rand_values(rng, c.shape[0], 4, 3))
    full = ref.subm_conv3d(c, f, w, b, 7)
    rows = [0, 5, 199, 17, 17]
    np.testing.assert_array_equal(ref.subm_conv3d_rows(c, f, w, b, 7, rows), full[rows])
    np.testing.assert_allclose(cpu.forward_rows(c, f, w, b, 7, rows=rows), full[rows],
                               rtol=0, atol=1e-12)


def _golden_inputs(cs):
    c = np.array(cs["coords"], np.int32)
    w = np.zeros((1, 3, 3, 3, 1))
    w.reshape(-1)[:] = np.arange(1, 28)
    f = np.array(cs["feats"]).reshape(-1, 1)
    return c, f, w, np.array([cs["bias"]])


def test_planted_convolution_flip_is_caught(monkeypatch):
    """Planting a flipped tap (true convolution instead of correlation) in the oracle
    must break the hand-worked example."""
    monkeypatch.setattr(ref, "tap", lambda dz, dy, dx: (1 - dz, 1 - dy, 1 - dx))
    for cs in json.load(open(GOLDEN))["cases"][:2]:
        c, f, w, b = _golden_inputs(cs)
        got = ref.subm_conv3d(c, f, w, b, cs["res"])[:, 0]
        assert not np.array_equal(got, cs["out"]), cs["name"]


def test_planted_axis_swap_is_caught(monkeypatch):
    """Planting a z/x swap of the tap axes in the oracle must break the example."""
    monkeypatch.setattr(ref, "tap", lambda dz, dy, dx: (dx + 1, dy + 1, dz + 1))
    for cs in json.load(open(GOLDEN))["cases"][:2]:
        c, f, w, b = _golden_inputs(cs)
        got = ref.subm_conv3d(c, f, w, b, cs["res"])[:, 0]
        assert not np.array_equal(got, cs["out"]), cs["name"]


def test_planted_offset_enumeration_mistake_is_caught(monkeypatch):
    """Planting a reversed offset enumeration in the oracle must break the kernel map pin."""
    monkeypatch.setattr(ref, "OFFSETS", ref.OFFSETS[::-1])
    rng = np.random.default_rng(0)
    c = random_set(rng, 4, 1, 20)
    assert not np.array_equal(ref.kernel_map(c, 4), brute_force_nbr(c))


# ----------------------------------------------------------------- fused block epilogue

_TORCH_ACT = {"none": lambda t: t, "relu": F.relu, "silu": F.silu}


def dense_block(coords, feats, weight, bias, residual, act, res):
    """act(dense masked Conv3d + residual) with torch's own activation routines."""
    y = torch.from_numpy(dense_masked_conv3d(coords, feats, weight, bias, res))
    if residual is not None:
        y = y + torch.from_numpy(np.asarray(residual, np.float64))
    return _TORCH_ACT[act](y).numpy()


@pytest.mark.parametrize("act", ref.ACTIVATIONS)
@pytest.mark.parametrize("with_residual", [False, True])
def test_block_epilogue_matches_dense_block(act, with_residual):
    rng = np.random.default_rng(20 + len(act) + with_residual)
    c = random_set(rng, 6, 2, 60)
    f, w, b = rand_values(rng, c.shape[0], 4, 5)
    r = rng.standard_normal((c.shape[0], 5)) if with_residual else None
    want = dense_block(c, f, w, b, r, act, 6)
    got = ref.block_epilogue(ref.subm_conv3d(c, f, w, b, 6), r, act)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * max(1.0, np.abs(want).max()))
    # the negative side of every activation is exercised
    assert (ref.subm_conv3d(c, f, w, b, 6) < -0.5).any()


def test_activation_closed_forms_and_odd_part():
    ln3 = np.log(3.0)
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    np.testing.assert_allclose(ref.activation([ln3, -ln3, 0.0], "silu"),
                               [0.75 * ln3, -0.25 * ln3, 0.0], rtol=1e-15, atol=0)
    np.testing.assert_array_equal(ref.activation([-2.0, 0.0, 3.5], "relu"), [0.0, 0.0, 3.5])
    np.testing.assert_array_equal(ref.activation([-2.0, 3.5], "none"), [-2.0, 3.5])
    y = np.random.default_rng(5).standard_normal(1000) * 6
    # f(y) - f(-y) = y for relu and silu (y sigmoid(y) + y sigmoid(-y) = y)
    for act in ("relu", "silu"):
        np.testing.assert_allclose(ref.activation(y, act) - ref.activation(-y, act), y,
                                   rtol=0, atol=1e-12)
    # silu tends to the identity above and to 0 below, without overflow to nan
    assert abs(ref.activation([40.0], "silu")[0] - 40.0) < 1e-14
    big = ref.activation([-800.0, 800.0], "silu")
    assert np.isfinite(big).all() and big[0] == 0.0 and big[1] == 800.0
    with pytest.raises(ref.OracleError):
        ref.activation([1.0], "gelu")


def test_block_epilogue_residual_only_and_shape_check():
    """Zero weight and bias leave act(residual): the epilogue sees only the skip path."""
    rng = np.random.default_rng(8)
    c = random_set(rng, 5, 1, 30)
    f = rng.standard_normal((30, 3))
    r = rng.standard_normal((30, 4))
    conv = ref.subm_conv3d(c, f, np.zeros((4, 3, 3, 3, 3)), np.zeros(4), 5)
    for act in ref.ACTIVATIONS:
        np.testing.assert_allclose(ref.block_epilogue(conv, r, act),
                                   _TORCH_ACT[act](torch.from_numpy(r)).numpy(), rtol=1e-15,
                                   atol=1e-16)
    with pytest.raises(ref.OracleError):
        ref.block_epilogue(conv, r[:, :3], "relu")


def test_planted_silu_sign_mistake_is_caught(monkeypatch):
    """Planting y * sigmoid(-y) for silu in the oracle must break the dense-block pin."""
    real = ref.activation

    def wrong(y, act):
        return -real(-np.asarray(y, np.float64), act) if act == "silu" else real(y, act)

    monkeypatch.setattr(ref, "activation", wrong)
    rng = np.random.default_rng(21)
    c = random_set(rng, 6, 1, 40)
    f, w, b = rand_values(rng, 40, 3, 3)
    got = ref.block_epilogue(ref.subm_conv3d(c, f, w, b, 6), None, "silu")
    assert not np.allclose(got, dense_block(c, f, w, b, None, "silu", 6), atol=1e-6)


# ------------------------------------------------- SparseDownsample(2) / SparseUpsample(2)

def _morton_less(p, q):
    """Z-order comparison without building a code: the axis whose coordinates differ in
    the highest bit decides; on equal highest bits z outranks y outranks x."""
    j, best = 0, 0
    for k in range(3):
        d = p[k] ^ q[k]
        if best < d and best < (best ^ d):    # msb(best) < msb(d)
            j, best = k, d
    return p[j] < q[j]


def dense_pool(coords, feats, res, mode):
    """Parents, pooled features and child counts from torch's dense 2x2x2 pooling on the
    densified grid (ceil mode for odd sides)."""
    coords = np.asarray(coords)
    B = int(coords[:, 0].max()) + 1
    C = feats.shape[1]
    b, z, y, x = (torch.from_numpy(coords[:, k].astype(np.int64)) for k in range(4))
    occ = torch.zeros(B, 1, res, res, res, dtype=torch.float64)
    occ[b, 0, z, y, x] = 1.0
    cnt = F.avg_pool3d(occ, 2, 2, ceil_mode=True, divisor_override=1)
    if mode == "mean":
        g = torch.zeros(B, C, res, res, res, dtype=torch.float64)
        g[b, :, z, y, x] = torch.from_numpy(np.asarray(feats, np.float64))
        pooled = F.avg_pool3d(g, 2, 2, ceil_mode=True, divisor_override=1) / cnt.clamp(min=1)
    else:
        g = torch.full((B, C, res, res, res), -np.inf, dtype=torch.float64)
        g[b, :, z, y, x] = torch.from_numpy(np.asarray(feats, np.float64))
        pooled = F.max_pool3d(g, 2, 2, ceil_mode=True)
    return cnt[:, 0], pooled


@pytest.mark.parametrize("mode", ref.POOL_MODES)
@pytest.mark.parametrize("seed,res,batch,n", [(0, 4, 1, 30), (1, 7, 2, 120), (2, 9, 3, 200),
                                               (3, 2, 1, 8), (4, 5, 2, 1)])
def test_downsample_matches_dense_pooling(mode, seed, res, batch, n):
    rng = np.random.default_rng(seed)
    c = random_set(rng, res, batch, n)
    f = rng.standard_normal((c.shape[0], 3))
    coarse, pooled, parent, mask = ref.downsample(c, f, res, mode)
    cnt, dense = dense_pool(c, f, res, mode)
    # the coarse set is exactly the occupied 2x2x2 cells
    occ = torch.nonzero(cnt > 0).numpy()
    assert sorted(map(tuple, coarse.tolist())) == sorted(map(tuple, occ.tolist()))
    # pooled rows and child counts equal the dense pooling at those cells
    cb, cz, cy, cx = (coarse[:, k] for k in range(4))
    np.testing.assert_allclose(pooled, dense.numpy()[cb, :, cz, cy, cx], rtol=0, atol=1e-12)
    np.testing.assert_array_equal([bin(int(m)).count("1") for m in mask], cnt.numpy()[cb, cz, cy, cx])
    # every fine row points at the cell that holds it, with its own bit set in the mask
    for i, (b, z, y, x) in enumerate(c.tolist()):
        assert tuple(coarse[parent[i]]) == (b, z // 2, y // 2, x // 2)
        assert mask[parent[i]] >> ((z & 1) << 2 | (y & 1) << 1 | (x & 1)) & 1


def test_downsample_order_is_batch_then_z_order():
    rng = np.random.default_rng(12)
    c = random_set(rng, 32, 3, 400)
    coarse = ref.downsample(c, None, 32)[0].tolist()
    for p, q in zip(coarse, coarse[1:]):
        assert p[0] < q[0] or (p[0] == q[0] and _morton_less(p[1:], q[1:])), (p, q)


def test_upsample_inverts_structure_and_max_of_single_children():
    rng = np.random.default_rng(13)
    c = random_set(rng, 8, 2, 100)
    f = rng.standard_normal((c.shape[0], 4))
    coarse, pooled, parent, mask = ref.downsample(c, f, 8, "mean")
    up = ref.upsample(pooled, parent)
    # each fine row gets its cell's mean; summing a cell's children gives count x mean
    for p in range(len(coarse)):
        kids = np.nonzero(parent == p)[0]
        np.testing.assert_allclose(up[kids].sum(axis=0), f[kids].sum(axis=0), rtol=0, atol=1e-12)
    # voxels alone in their cell come back unchanged (both modes)
    iso = np.array([[0, 0, 0, 0], [0, 2, 4, 6], [1, 5, 5, 5]], np.int32)
    g = rng.standard_normal((3, 2))
    for mode in ref.POOL_MODES:
        _, pl, par, mk = ref.downsample(iso, g, 8, mode)
        np.testing.assert_array_equal(ref.upsample(pl, par), g)
        assert all(bin(int(m)).count("1") == 1 for m in mk)
    with pytest.raises(ref.OracleError):
        ref.upsample(pooled, np.array([len(coarse)]))
    with pytest.raises(ref.OracleError):
        ref.downsample(c, f, 8, "sum")
    with pytest.raises(ref.OracleError):
        ref.downsample(np.array([[0, 1, 1, 1], [0, 1, 1, 1]], np.int32), None, 4)


def test_planted_morton_axis_swap_is_caught(monkeypatch):
    """Planting x as the most significant axis of the Z-order code in the oracle must
    break the order pin."""
    monkeypatch.setattr(ref, "morton_code", lambda z, y, x: sum(
        (((z >> t) & 1) << (3 * t) | ((y >> t) & 1) << (3 * t + 1) | ((x >> t) & 1) << (3 * t + 2))
        for t in range(16)))
    c = random_set(np.random.default_rng(12), 32, 1, 300)
    coarse = ref.downsample(c, None, 32)[0].tolist()
    assert not all(_morton_less(p[1:], q[1:]) for p, q in zip(coarse, coarse[1:]))


# ------------------------------------------- SparseSpatial2Channel(2) / channel2spatial

def dense_unshuffle(coords, feats, res, coarse):
    """3-D pixel-unshuffle of the densified grid by reshape and permute: channel block k
    of a cell holds the child at (dz, dy, dx) with k = 4 dz + 2 dy + dx; read at the
    coarse cells."""
    coords = np.asarray(coords)
    B = int(coords[:, 0].max()) + 1
    C = feats.shape[1]
    R = res + (res & 1)
    g = torch.zeros(B, C, R, R, R, dtype=torch.float64)
    b, z, y, x = (torch.from_numpy(coords[:, k].astype(np.int64)) for k in range(4))
    g[b, :, z, y, x] = torch.from_numpy(np.asarray(feats, np.float64))
    h = R // 2
    g = g.view(B, C, h, 2, h, 2, h, 2).permute(0, 3, 5, 7, 1, 2, 4, 6).reshape(B, 8 * C, h, h, h)
    cb, cz, cy, cx = (torch.from_numpy(coarse[:, k].astype(np.int64)) for k in range(4))
    return g[cb, :, cz, cy, cx].numpy()


@pytest.mark.parametrize("seed,res,batch,n,C", [(0, 6, 2, 100, 3), (1, 9, 1, 400, 2),
                                                 (2, 2, 1, 8, 4), (3, 5, 3, 1, 1)])
def test_spatial2channel_matches_dense_unshuffle(seed, res, batch, n, C):
    rng = np.random.default_rng(seed)
    c = random_set(rng, res, batch, n)
    f = rng.standard_normal((c.shape[0], C))
    coarse, out, parent, mask = ref.spatial2channel(c, f, res)
    np.testing.assert_array_equal(out, dense_unshuffle(c, f, res, coarse))
    ds = ref.downsample(c, None, res)
    np.testing.assert_array_equal(coarse, ds[0])
    np.testing.assert_array_equal(parent, ds[2])
    # absent children are zero blocks, present ones are not (random features)
    for p, m in enumerate(mask):
        for k in range(8):
            blk = out[p, k * C:(k + 1) * C]
            assert (np.abs(blk).sum() > 0) == bool(m >> k & 1)
    # channel2spatial undoes it exactly
    np.testing.assert_array_equal(ref.channel2spatial(out, c, parent), f)


def test_channel2spatial_errors_and_planted_bit_order(monkeypatch):
    c = np.array([[0, 0, 0, 1], [0, 1, 0, 0]], np.int32)
    f = np.array([[1.0], [2.0]])
    coarse, out, parent, _ = ref.spatial2channel(c, f, 4)
    np.testing.assert_array_equal(out, [[0, 1, 0, 0, 2, 0, 0, 0]])   # x -> block 1, z -> block 4
    with pytest.raises(ref.OracleError):
        ref.channel2spatial(out[:, :7], c, parent)
    with pytest.raises(ref.OracleError):
        ref.channel2spatial(out, c, np.array([0, 1]))
    # planting x as the high bit of the child index must break the dense pin
    monkeypatch.setattr(ref, "child_bit", lambda z, y, x: ((x & 1) << 2) | ((y & 1) << 1) | (z & 1))
    rng = np.random.default_rng(3)
    cs = random_set(rng, 6, 1, 80)
    fs = rng.standard_normal((80, 2))
    co, o2, _, _ = ref.spatial2channel(cs, fs, 6)
    assert not np.array_equal(o2, dense_unshuffle(cs, fs, 6, co))


# ------------------------------------------------- tile plan of the grouped forward

def test_morton_codes_give_z_order_and_match_the_scalar_code():
    rng = np.random.default_rng(31)
    c = np.concatenate([random_set(rng, 64, 2, 300),
                        np.array([[0, 65534, 3, 40000], [1, 0, 65534, 1]], np.int32)])
    m = ref.morton_codes(c)
    for i in range(0, c.shape[0], 7):
        assert int(m[i]) == ref.morton_code(int(c[i, 1]), int(c[i, 2]), int(c[i, 3]))
    order = np.lexsort((m, c[:, 0]))
    pts = [tuple(int(v) for v in c[i]) for i in order]
    for p, q in zip(pts, pts[1:]):
        assert p[0] < q[0] or (p[0] == q[0] and _morton_less(p[1:], q[1:])), (p, q)


def test_neighbour_masks_by_hand():
    # k = 9 (dz + 1) + 3 (dy + 1) + (dx + 1). From (5,5,5): (5,5,6) is (0,0,+1), k = 14, and
    # (4,5,5) is (-1,0,0), k = 4. From (5,5,6): (5,5,5) is (0,0,-1), k = 12, and (4,5,5) is
    # (-1,0,-1), k = 3. From (4,5,5): (5,5,5) is (+1,0,0), k = 22, and (5,5,6) is (+1,0,+1),
    # k = 23. (9,9,9) is alone: the centre, k = 13, only.
    c = np.array([[0, 5, 5, 5], [0, 5, 5, 6], [0, 4, 5, 5], [0, 9, 9, 9]], np.int32)
    m = ref.neighbour_masks(ref.kernel_map(c, 16))
    assert m.tolist() == [(1 << 13) | (1 << 14) | (1 << 4), (1 << 13) | (1 << 12) | (1 << 3),
                          (1 << 13) | (1 << 22) | (1 << 23), 1 << 13]


def _check_plan(c, nbr, window, perm, pnbr, tmask, tile=128):
    N = c.shape[0]
    assert sorted(perm.tolist()) == list(range(N))                        # a permutation
    assert np.array_equal(pnbr, nbr[perm])
    masks = ref.neighbour_masks(nbr)[perm]
    # windows: consecutive stretches of the (batch, Z-order) sequence, each a stretch of
    # `window` voxels -- checked with the comparator, without a Morton code
    key = lambda i: (int(c[i, 0]),) + tuple(int(v) for v in c[i, 1:])
    for w0 in range(0, N, window):
        seg = perm[w0:w0 + window]
        if w0 + window < N:   # everything in this window precedes everything after it
            last = max(seg, key=lambda i: _zkey_rank(c, i))
            nxt = perm[w0 + window:]
            first_next = min(nxt, key=lambda i: _zkey_rank(c, i))
            assert _zless(c, last, first_next), (key(last), key(first_next))
        ms = masks[w0:w0 + window]
        assert np.all(ms[1:] >= ms[:-1])                                    # masks ascend
        for a, b in zip(range(len(seg) - 1), range(1, len(seg))):
            if ms[a] == ms[b]:
                assert _zless(c, seg[a], seg[b])                            # Z-order among ties
    nt = (N + tile - 1) // tile
    for t in range(nt):
        want = 0
        for r in range(t * tile, min(N, (t + 1) * tile)):
            want |= int(masks[r])
        assert int(tmask[t]) == want


def _zless(c, i, j):
    p, q = c[i], c[j]
    if p[0] != q[0]:
        return p[0] < q[0]
    return _morton_less(tuple(int(v) for v in p[1:]), tuple(int(v) for v in q[1:]))


_zrank_cache = {}


def _zkey_rank(c, i):
    # rank of row i in the comparator's (batch, Z) order, computed once per array
    key = id(c)
    if key not in _zrank_cache:
        import functools
        idx = list(range(c.shape[0]))
        idx.sort(key=functools.cmp_to_key(lambda a, b: -1 if _zless(c, a, b) else (1 if _zless(c, b, a) else 0)))
        _zrank_cache[key] = {v: r for r, v in enumerate(idx)}
    return _zrank_cache[key][i]


@pytest.mark.parametrize("window", [1, 128, 256, 1 << 20])
def test_tile_plan_properties(window):
    rng = np.random.default_rng(7 + window % 97)
    from synth import ellipsoid_shell, union_coords, uniform_rotation
    parts = [(b, ellipsoid_shell(24, (11.7, 12.2, 12.4), (8.0, 6.5, 9.5), uniform_rotation(rng)))
             for b in range(2)]
    c = union_coords(parts, 24)
    c = c[rng.permutation(c.shape[0])]
    nbr = ref.kernel_map(c, 24)
    perm, pnbr, tmask = ref.tile_plan(c, nbr, window)
    _check_plan(c, nbr, window, perm, pnbr, tmask)
    _zrank_cache.clear()


def test_tile_plan_window_one_is_z_order_and_huge_window_sorts_by_mask():
    rng = np.random.default_rng(3)
    c = random_set(rng, 12, 2, 150)
    nbr = ref.kernel_map(c, 12)
    perm1 = ref.tile_plan(c, nbr, 1)[0]
    for a, b in zip(perm1, perm1[1:]):
        assert _zless(c, a, b)
    permh = ref.tile_plan(c, nbr, 1 << 30)[0]
    assert np.all(np.diff(ref.neighbour_masks(nbr)[permh].astype(np.int64)) >= 0)


def test_planted_unstable_grouping_is_caught(monkeypatch):
    rng = np.random.default_rng(5)
    from synth import ellipsoid_shell, union_coords, uniform_rotation
    c = union_coords([(0, ellipsoid_shell(20, (9.6, 10.1, 9.8), (7.0, 8.0, 6.0),
                                          uniform_rotation(rng)))], 20)
    nbr = ref.kernel_map(c, 20)
    real = np.lexsort

    def unstable(keys):   # drops the Morton tie-break of the grouping sort
        keys = tuple(keys)
        if len(keys) == 3 and keys[0].dtype.kind == "i" and np.array_equal(keys[0], np.arange(len(keys[0]))):
            return real((keys[0][::-1], keys[1], keys[2]))
        return real(keys)
    monkeypatch.setattr(np, "lexsort", unstable)
    perm, pnbr, tmask = ref.tile_plan(c, nbr, 128)
    monkeypatch.setattr(np, "lexsort", real)
    with pytest.raises(AssertionError):
        _check_plan(c, nbr, 128, perm, pnbr, tmask)
    _zrank_cache.clear()
