"""subm3d_build_kmap_noalloc: the kernel map for callers that cannot allocate device
memory (a host application that owns all device memory through its own pool, or a
latency-critical loop where an allocation is not acceptable). Called through the C
ABI with caller-owned coords and nbr only, its result must equal that of
subm3d_build_kmap (bit-exact: the neighbour table is integer data), on two calls in a
row with different voxel sets, since the built-in scratch keeps the previous call's
contents. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from submanifold_sparse_convolution_04_b300 import _binding as B
from submanifold_sparse_convolution_04_b300 import subm3d_build_kmap
from synth import ellipsoid_shell, union_coords, uniform_rotation
from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu

MAX_VOXELS = 131072


def shells(seed, res, batch):
    rng = np.random.default_rng(seed)
    parts = []
    for b in range(batch):
        a = res * (0.2 + 0.2 * rng.random(3))
        parts.append((b, ellipsoid_shell(res, res / 2 + rng.random(3), a, uniform_rotation(rng))))
    return union_coords(parts, res)


def noalloc_nbr(L, coords, res):
    nbr = torch.full((coords.shape[0], 27), -7, dtype=torch.int32, device=coords.device)
    rc = L.subm3d_build_kmap_noalloc(ctypes.c_void_p(coords.data_ptr()), coords.shape[0], res,
                                     ctypes.c_void_p(nbr.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == B.OK, B.subm3d_last_error()
    torch.cuda.synchronize()
    return nbr


def test_noalloc_matches_workspace_entry_point_twice():
    dev = require_gpu()
    L = B.lib()
    first = torch.from_numpy(shells(1, 96, 2)).to(dev)     # ~30 k voxels
    second = torch.from_numpy(shells(2, 48, 3)).to(dev)    # a smaller, different set
    assert first.shape[0] > second.shape[0] > 1000
    for coords, res in ((first, 96), (second, 48)):
        got = noalloc_nbr(L, coords, res)
        want = subm3d_build_kmap(coords, res)
        assert torch.equal(got, want)


def test_noalloc_at_the_size_limit_and_beyond():
    dev = require_gpu()
    L = B.lib()
    rng = np.random.default_rng(3)
    flat = rng.choice(64 ** 3, size=MAX_VOXELS, replace=False)
    z, rem = np.divmod(flat, 64 * 64)
    y, x = np.divmod(rem, 64)
    coords = torch.from_numpy(np.stack([np.zeros_like(z), z, y, x], 1).astype(np.int32)).to(dev)
    assert torch.equal(noalloc_nbr(L, coords, 64), subm3d_build_kmap(coords, 64))
    rc = L.subm3d_build_kmap_noalloc(ctypes.c_void_p(16), MAX_VOXELS + 1, 64, ctypes.c_void_p(16),
                                     None)
    assert rc == B.ERR_ARG and "131072" in B.subm3d_last_error()
