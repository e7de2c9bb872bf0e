"""Kernel map on the GPU, bit-exact against the CPU oracle."""
import numpy as np
import pytest
import torch

from oracle import cpu, ref
from submanifold_sparse_convolution_04_b300 import (Subm3dError, subm3d_build_kmap,
                                                    subm3d_build_kmap_ex,
                                                    subm3d_kmap_workspace_bytes)
from submanifold_sparse_convolution_04_b300 import _binding as B
from tests.conftest import cached_case
from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def gpu_nbr(coords_np, res, dev, **kw):
    c = torch.from_numpy(np.ascontiguousarray(coords_np, np.int32)).to(dev)
    return subm3d_build_kmap(c, res, **kw).cpu().numpy()


@pytest.mark.parametrize("cfg_id", [1, 2, 3, 4, 5])
def test_kmap_bit_exact_on_workloads(dev, cfg_id):
    case = cached_case(cfg_id)
    got = gpu_nbr(case["coords"], case["res"], dev)
    np.testing.assert_array_equal(got, cpu.kernel_map(case["coords"], case["res"]))


@pytest.mark.parametrize("cfg_id", [2, 4])
def test_kmap_bit_exact_shuffled_order(dev, cfg_id):
    case = cached_case(cfg_id, "shuffled")
    got = gpu_nbr(case["coords"], case["res"], dev)
    np.testing.assert_array_equal(got, cpu.kernel_map(case["coords"], case["res"]))


def random_set(rng, res, batch, n):
    rows = []
    for b in range(batch):
        flat = rng.choice(res ** 3, size=n, replace=False)
        z, rem = np.divmod(flat, res * res)
        y, x = np.divmod(rem, res)
        rows.append(np.stack([np.full(n, b), z, y, x], axis=1))
    c = np.concatenate(rows).astype(np.int32)
    return c[rng.permutation(c.shape[0])]


@pytest.mark.parametrize("seed,res,batch,n", [(0, 4, 1, 1), (1, 3, 1, 27), (2, 5, 3, 70),
                                               (3, 8, 2, 500), (4, 2, 4, 8), (5, 31, 1, 4000),
                                               (6, 1, 5, 1), (7, 17, 7, 333)])
def test_kmap_random_sets(dev, seed, res, batch, n):
    rng = np.random.default_rng(seed)
    c = random_set(rng, res, batch, n)
    np.testing.assert_array_equal(gpu_nbr(c, res, dev), ref.kernel_map(c, res))


def test_kmap_extreme_coordinates(dev):
    res = 65535
    c = np.array([[0, 0, 0, 0], [0, 65534, 65534, 65534], [0, 65533, 65534, 65534],
                  [65534, 65534, 0, 1], [65534, 65534, 1, 1], [3, 1, 1, 1], [3, 0, 0, 0]],
                 np.int32)
    np.testing.assert_array_equal(gpu_nbr(c, res, dev), ref.kernel_map(c, res))


def test_kmap_empty(dev):
    c = torch.zeros((0, 4), dtype=torch.int32, device=dev)
    assert subm3d_build_kmap(c, 16).shape == (0, 27)


def test_kmap_morton_order(dev):
    case = cached_case(3)
    c = torch.from_numpy(case["coords"]).to(dev)
    nbr, order = subm3d_build_kmap_ex(c, case["res"], order=True)
    o = order.cpu().numpy()
    assert np.array_equal(np.sort(o), np.arange(len(o)))
    # Morton key written out independently: interleave bits of z, y, x (z highest of each triple)
    co = case["coords"].astype(np.int64)
    m = np.zeros(len(co), np.int64)
    for t in range(8):
        m |= ((co[:, 3] >> t) & 1) << (3 * t)
        m |= ((co[:, 2] >> t) & 1) << (3 * t + 1)
        m |= ((co[:, 1] >> t) & 1) << (3 * t + 2)
    key = (co[:, 0] << 24) | m
    want = np.lexsort((np.arange(len(co)), key))       # stable ascending order
    np.testing.assert_array_equal(o, want)
    np.testing.assert_array_equal(nbr.cpu().numpy(), cpu.kernel_map(case["coords"], case["res"]))


@pytest.mark.parametrize("res", [1, 2, 3, 4, 5])
def test_kmap_morton_order_small_grids_with_batches(dev, res):
    # grids below 4 per side: the sort key still keeps the batch above a whole 4x4x4
    # block's Morton bits; the order is (b, Morton(z, y, x)) ascending, stable
    rng = np.random.default_rng(res)
    cells = np.array([(b, z, y, x) for b in range(3) for z in range(res) for y in range(res)
                      for x in range(res)], np.int32)
    c = cells[rng.permutation(len(cells))[: max(1, (2 * len(cells)) // 3)]]
    ct = torch.from_numpy(c).to(dev)
    nbr, order = subm3d_build_kmap_ex(ct, res, order=True)
    co = c.astype(np.int64)
    m = np.zeros(len(co), np.int64)
    for t in range(4):
        m |= ((co[:, 3] >> t) & 1) << (3 * t)
        m |= ((co[:, 2] >> t) & 1) << (3 * t + 1)
        m |= ((co[:, 1] >> t) & 1) << (3 * t + 2)
    want = np.lexsort((np.arange(len(co)), m, co[:, 0]))   # by batch, then Morton, stable
    np.testing.assert_array_equal(order.cpu().numpy(), want)
    np.testing.assert_array_equal(nbr.cpu().numpy(), ref.kernel_map(c, res))


def test_kmap_errors_and_recovery(dev):
    good = np.array([[0, 1, 1, 1], [0, 1, 1, 2]], np.int32)
    for bad, code in [
        (np.array([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], np.int32), B.ERR_DUPLICATE),
        (np.array([[0, 1, 1, 1], [0, 8, 0, 0]], np.int32), B.ERR_COORD_RANGE),
        (np.array([[0, 1, 1, 1], [0, 0, -1, 0]], np.int32), B.ERR_COORD_RANGE),
        (np.array([[-1, 1, 1, 1]], np.int32), B.ERR_COORD_RANGE),
        (np.array([[65535, 1, 1, 1]], np.int32), B.ERR_COORD_RANGE),
    ]:
        with pytest.raises(Subm3dError) as e:
            gpu_nbr(bad, 8, dev)
        assert e.value.code == code
        np.testing.assert_array_equal(gpu_nbr(good, 8, dev), ref.kernel_map(good, 8))


def test_kmap_hash_full_is_reported(dev):
    # 100 voxels, each in an aligned 4x4x4 block of its own: 100 occupied blocks
    rng = np.random.default_rng(3)
    cells = rng.choice(16 ** 3, size=100, replace=False)
    c = np.zeros((100, 4), np.int32)
    c[:, 1], c[:, 2], c[:, 3] = 4 * (cells // 256), 4 * ((cells // 16) % 16), 4 * (cells % 16)
    c[:, 1:] += rng.integers(0, 4, size=(100, 3)).astype(np.int32)
    ct = torch.from_numpy(c).to(dev)
    with pytest.raises(Subm3dError) as e:
        subm3d_build_kmap_ex(ct, 64, hash_capacity=64)
    assert e.value.code == B.ERR_HASH_FULL
    # the smallest capacity that holds the blocks works, with long probe chains
    nbr, _ = subm3d_build_kmap_ex(ct, 64, hash_capacity=128)
    np.testing.assert_array_equal(nbr.cpu().numpy(), ref.kernel_map(c, 64))


def test_kmap_reuses_dirty_workspace(dev):
    case = cached_case(2)
    c = torch.from_numpy(case["coords"]).to(dev)
    ws = torch.full((subm3d_kmap_workspace_bytes(c.shape[0]),), 0xA5, dtype=torch.uint8, device=dev)
    a = subm3d_build_kmap(c, case["res"], workspace=ws).cpu().numpy()
    b = subm3d_build_kmap(c, case["res"], workspace=ws).cpu().numpy()
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, cpu.kernel_map(case["coords"], case["res"]))
    with pytest.raises(Subm3dError) as e:
        subm3d_build_kmap(c, case["res"], workspace=ws[:1024])
    assert e.value.code == B.ERR_WORKSPACE


def sparse_pairs(rng, res, batch, n):
    """Isolated voxels, about half with a +x neighbour (often across a 4x4x4 block's
    face): roughly one voxel per occupied block."""
    rows = []
    for b in range(batch):
        flat = rng.choice((res // 8) ** 3, size=n, replace=False)
        z, rem = np.divmod(flat, (res // 8) ** 2)
        y, x = np.divmod(rem, res // 8)
        p = np.stack([np.full(n, b), 8 * z + 3, 8 * y + rng.integers(0, 8, n), 8 * x + 3], 1)
        q = p[rng.random(n) < 0.5].copy()
        q[:, 3] += 1
        rows += [p, q]
    c = np.concatenate(rows).astype(np.int32)
    return c[rng.permutation(c.shape[0])]


def test_kmap_hashed_table_grows(dev):
    # the nbr-only build first sizes its block table for N/4 blocks; here there are about
    # N of them, so it rebuilds the table at full size, with the same answer
    rng = np.random.default_rng(11)
    c = sparse_pairs(rng, 1024, 2, 20000)
    got = gpu_nbr(c, 1024, dev)
    np.testing.assert_array_equal(got, ref.kernel_map(c, 1024))
    assert (got[:, 12] >= 0).sum() + (got[:, 14] >= 0).sum() > 0   # some pairs


@pytest.mark.parametrize("cfg_id", [3, 5])
def test_kmap_front_ends_agree(dev, cfg_id):
    # nbr alone (hashed blocks, no sort) and with the Morton order (radix-sort front end)
    case = cached_case(cfg_id)
    c = torch.from_numpy(case["coords"]).to(dev)
    hashed = subm3d_build_kmap(c, case["res"]).cpu().numpy()
    sorted_nbr, _ = subm3d_build_kmap_ex(c, case["res"], order=True)
    np.testing.assert_array_equal(hashed, sorted_nbr.cpu().numpy())
    np.testing.assert_array_equal(hashed, cpu.kernel_map(case["coords"], case["res"]))


def one_voxel_per_block(rng, res, n):
    """n voxels in n distinct 4x4x4 blocks of a res^3 grid, each at a random place."""
    nb = res // 4
    blocks = rng.choice(nb ** 3, size=n, replace=False)
    bz, rem = np.divmod(blocks, nb * nb)
    by, bx = np.divmod(rem, nb)
    off = rng.integers(0, 4, size=(n, 3))
    c = np.stack([np.zeros(n, np.int64), 4 * bz + off[:, 0], 4 * by + off[:, 1],
                  4 * bx + off[:, 2]], axis=1)
    return c.astype(np.int32)


def test_kmap_growth_duplicates_and_full_table_one_voxel_per_block(dev):
    # 6000 voxels, one per 4x4x4 block of a 128^3 grid, plus 600 +x neighbours: the
    # blocks overfill the first (N/4) table, so it grows first. Then a duplicate and a
    # fixed table that is too small, at this size.
    rng = np.random.default_rng(21)
    c = one_voxel_per_block(rng, 128, 6000)
    c = np.concatenate([c, c[:600] + np.array([0, 0, 0, 1], np.int32)])
    c = np.unique(c[(c[:, 3] < 128)], axis=0)
    c = c[rng.permutation(len(c))]
    want = ref.kernel_map(c, 128)
    np.testing.assert_array_equal(gpu_nbr(c, 128, dev), want)
    assert (want[:, 14] >= 0).sum() > 0
    # a repeated row: ERR_DUPLICATE, and the next build is clean again
    with pytest.raises(Subm3dError) as e:
        gpu_nbr(np.concatenate([c, c[17:18]]), 128, dev)
    assert e.value.code == B.ERR_DUPLICATE
    np.testing.assert_array_equal(gpu_nbr(c, 128, dev), want)
    # a fixed table smaller than the blocks: ERR_HASH_FULL; one that holds them works
    nblk = len(np.unique(c[:, 1:] // 4, axis=0))
    small = 1 << (nblk.bit_length() - 1)      # < nblk
    ct = torch.from_numpy(c).to(dev)
    with pytest.raises(Subm3dError) as e:
        subm3d_build_kmap_ex(ct, 128, hash_capacity=small)
    assert e.value.code == B.ERR_HASH_FULL
    nbr, _ = subm3d_build_kmap_ex(ct, 128, hash_capacity=4 * small)
    np.testing.assert_array_equal(nbr.cpu().numpy(), want)


@pytest.mark.parametrize("batch,res,n", [(3, 64, 3000), (2, 128, 5000), (1, 1024, 3000)])
def test_kmap_key_range_edges(dev, batch, res, n):
    # blocks at both ends of the block-key range (the grid's first and last cell, in the
    # first and last batch), one voxel per block elsewhere, in batches
    rng = np.random.default_rng(batch * 7 + res)
    rows = []
    for b in range(batch):
        c = one_voxel_per_block(rng, min(res, 128), n)
        c[:, 0] = b
        rows.append(c)
    c = np.concatenate(rows)
    corners = np.array([[0, 0, 0, 0], [batch - 1, res - 1, res - 1, res - 1],
                        [batch - 1, res - 1, res - 1, res - 2]], np.int32)
    c = np.unique(np.concatenate([c, corners]), axis=0)
    c = c[rng.permutation(len(c))]
    np.testing.assert_array_equal(gpu_nbr(c, res, dev), ref.kernel_map(c, res))
