"""CPU oracle for submanifold sparse 3D convolution (SubMConv3d, kernel 3, stride 1,
no padding) -- the plain definition, written out.

TEST INFRASTRUCTURE ONLY. This module is imported by the tests, by the smoke check
and by the benchmark's CPU-baseline leg, and by nothing else. The CUDA library
never calls it and shares no code with it.

Sources (page titles and sections):
* "pixal3d_mrp_mlx README", section "Scope, measured against the shared core":
  every SparseConv3d in the model is (c, out, 3), i.e. stride 1 and no padding,
  which is the submanifold variant. "pixal3d_mrp_mlx CLAUDE.md", section
  "Measured facts": stride 1 with padding None dispatches to SubMConv3d.
* The same README's commit header: tensors are carried channels-last and the
  weight is stored as [O, kz, ky, kx, I]; its "Status" section: the converter
  remaps the kernel to [K^3, in, out] as a pure permutation.
* Submanifold means the output sites are exactly the active input sites; a
  neighbour that is inactive or outside the grid contributes nothing.

Readings taken where the pages are silent (each is pinned by a test):
* Orientation is cross-correlation, the convention of a dense Conv3d: the input
  at p + d meets weight tap (kz, ky, kx) = (dz + 1, dy + 1, dx + 1).
* Coordinate columns (b, z, y, x) pair with the weight axes (kz, ky, kx) in order.
* Offsets are enumerated k = 9 (dz + 1) + 3 (dy + 1) + (dx + 1); k = 13 is the centre.
* Coordinates outside 0 <= z, y, x < res, a batch index outside [0, 65534], and
  duplicate coordinates are errors, not clamps or merges.
* Arithmetic: every product and sum in float64 from the exact stored input values.

Pure-Python loops: meant for small inputs (a few thousand voxels). The C++ file
in this directory computes the same definition for the large workloads.
"""
from __future__ import annotations

import numpy as np

__all__ = ["OFFSETS", "CENTER", "ACTIVATIONS", "POOL_MODES", "OracleError", "tap",
           "coordinate_dict", "kernel_map", "subm_conv3d", "subm_conv3d_rows", "activation",
           "block_epilogue", "morton_code", "child_bit", "downsample", "upsample",
           "spatial2channel", "channel2spatial", "morton_codes", "neighbour_masks", "tile_plan"]

# k -> (dz, dy, dx), k = 9 (dz + 1) + 3 (dy + 1) + (dx + 1)
OFFSETS = [(dz, dy, dx) for dz in (-1, 0, 1) for dy in (-1, 0, 1) for dx in (-1, 0, 1)]
CENTER = 13
ACTIVATIONS = ("none", "relu", "silu")
POOL_MODES = ("mean", "max")
MAX_BATCH = 65534
MAX_RES = 65535


def tap(dz, dy, dx):
    """Weight tap (kz, ky, kx) that meets the neighbour at offset (dz, dy, dx):
    cross-correlation, as a dense Conv3d."""
    return dz + 1, dy + 1, dx + 1


class OracleError(ValueError):
    """Invalid input: out-of-range or duplicate coordinates, or bad shapes."""


def coordinate_dict(coords, res):
    """S = {(b, z, y, x): input row index}, after validating every coordinate."""
    coords = np.asarray(coords)
    if coords.ndim != 2 or coords.shape[1] != 4:
        raise OracleError("coords must be [N, 4] (b, z, y, x)")
    if not (1 <= int(res) <= MAX_RES):
        raise OracleError(f"res={res} outside [1, {MAX_RES}]")
    S = {}
    for i, row in enumerate(coords.tolist()):
        b, z, y, x = row
        if not (0 <= b <= MAX_BATCH) or not (0 <= z < res and 0 <= y < res and 0 <= x < res):
            raise OracleError(f"coordinate {i} = {row} outside the grid (res={res})")
        key = (b, z, y, x)
        if key in S:
            raise OracleError(f"duplicate coordinate {row} at rows {S[key]} and {i}")
        S[key] = i
    return S


def kernel_map(coords, res):
    """nbr[i, k] = index of the active voxel at coords[i] + OFFSETS[k], or -1.

    A neighbour position outside [0, res)^3 is absent. Returns int32 [N, 27].
    """
    S = coordinate_dict(coords, res)
    coords = np.asarray(coords).tolist()
    nbr = np.full((len(coords), 27), -1, dtype=np.int32)
    for i, (b, z, y, x) in enumerate(coords):
        for k, (dz, dy, dx) in enumerate(OFFSETS):
            q = (b, z + dz, y + dy, x + dx)
            if 0 <= q[1] < res and 0 <= q[2] < res and 0 <= q[3] < res:
                nbr[i, k] = S.get(q, -1)
    return nbr


def _check_values(N, feats, weight, bias):
    feats = np.asarray(feats, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    if feats.ndim != 2 or feats.shape[0] != N:
        raise OracleError("feats must be [N, I]")
    I = feats.shape[1]
    if weight.ndim != 5 or weight.shape[1:] != (3, 3, 3, I):
        raise OracleError("weight must be [O, 3, 3, 3, I]")
    O = weight.shape[0]
    if bias is None:
        bias = np.zeros(O, dtype=np.float64)
    bias = np.asarray(bias, dtype=np.float64)
    if bias.shape != (O,):
        raise OracleError("bias must be [O]")
    return feats, weight, bias


def subm_conv3d_rows(coords, feats, weight, bias, res, rows):
    """Output rows `rows` of the convolution, float64 [len(rows), O]:

    out[i, o] = bias[o] + sum_{k : nbr[i,k] >= 0} sum_c weight[o, kz, ky, kx, c] * feats[nbr[i,k], c]
    with (kz, ky, kx) = OFFSETS[k] + 1.
    """
    coords = np.asarray(coords)
    N = coords.shape[0]
    feats, weight, bias = _check_values(N, feats, weight, bias)
    S = coordinate_dict(coords, res)
    clist = coords.tolist()
    out = np.empty((len(rows), weight.shape[0]), dtype=np.float64)
    for r, i in enumerate(rows):
        b, z, y, x = clist[i]
        acc = bias.copy()
        for dz, dy, dx in OFFSETS:
            zz, yy, xx = z + dz, y + dy, x + dx
            if not (0 <= zz < res and 0 <= yy < res and 0 <= xx < res):
                continue
            j = S.get((b, zz, yy, xx), -1)
            if j < 0:
                continue
            kz, ky, kx = tap(dz, dy, dx)
            acc += weight[:, kz, ky, kx, :] @ feats[j]
        out[r] = acc
    return out


def subm_conv3d(coords, feats, weight, bias, res):
    """All output rows, float64 [N, O] (see subm_conv3d_rows)."""
    N = np.asarray(coords).shape[0]
    return subm_conv3d_rows(coords, feats, weight, bias, res, range(N))


def activation(y, act):
    """Elementwise activation in float64: "none" is the identity, "relu" is max(y, 0),
    "silu" is y * sigmoid(y) = y / (1 + exp(-y))."""
    y = np.asarray(y, dtype=np.float64)
    if act == "none":
        return y.copy()
    if act == "relu":
        return np.where(y > 0.0, y, 0.0)
    if act == "silu":
        with np.errstate(over="ignore"):      # exp(-y) = inf for y << 0 gives -0.0
            return y / (1.0 + np.exp(-y))
    raise OracleError(f"activation {act!r} is not one of {ACTIVATIONS}")


def block_epilogue(conv, residual=None, act="none"):
    """Tail of a residual block on top of the convolution, float64:

    out = act(conv + residual), conv being the convolution output with its bias.

    The "pixal3d_mrp_mlx README" scope table ("Scope, measured against the shared
    core" and its correction) lists ResBlock-style and ConvNeXt-style sparse blocks and
    activations beside SubMConv3d, but not their internals; a residual add and an
    activation are the steps such a block applies to a convolution's output.
    """
    y = np.asarray(conv, dtype=np.float64)
    if residual is not None:
        residual = np.asarray(residual, dtype=np.float64)
        if residual.shape != y.shape:
            raise OracleError(f"residual shape {residual.shape} != output shape {y.shape}")
        y = y + residual
    return activation(y, act)


def morton_code(z, y, x):
    """Z-order code of a lattice point: bit t of x goes to bit 3t, of y to 3t + 1, of z to
    3t + 2 (z the most significant axis of each bit triple)."""
    m, t = 0, 0
    while (z >> t) or (y >> t) or (x >> t):
        m |= ((x >> t) & 1) << (3 * t)
        m |= ((y >> t) & 1) << (3 * t + 1)
        m |= ((z >> t) & 1) << (3 * t + 2)
        t += 1
    return m


def child_bit(z, y, x):
    """Place of a fine voxel inside its parent's 2x2x2 cell: (z&1)<<2 | (y&1)<<1 | (x&1)."""
    return ((z & 1) << 2) | ((y & 1) << 1) | (x & 1)


def downsample(coords, feats, res, mode="mean"):
    """SparseDownsample(2) and the subdivision it stores for its paired upsample.

    The "pixal3d_mrp_mlx README" scope table lists SparseDownsample(2) (its status notes
    say the shared core's downsample takes a pooling mode) and SparseUpsample(2) as the
    cache-paired inverse that needs the subdivision stored by the matching downsample.
    Readings: the coarse voxel of a fine voxel (b, z, y, x) is (b, z//2, y//2, x//2);
    the coarse set is the set of those parents, ordered by batch, then Morton code;
    a coarse feature pools its children's features ("mean" or "max"); the subdivision
    is each fine row's parent row plus each parent's 8-bit child mask (child_bit).

    Returns (coarse_coords int32 [M, 4], coarse_feats float64 [M, C] or None,
    parent int32 [N], child_mask uint8 [M]).
    """
    if mode not in POOL_MODES:
        raise OracleError(f"pooling mode {mode!r} is not one of {POOL_MODES}")
    coordinate_dict(coords, res)    # validates range and duplicates
    clist = np.asarray(coords).tolist()
    groups = {}
    for i, (b, z, y, x) in enumerate(clist):
        groups.setdefault((b, z // 2, y // 2, x // 2), []).append(i)
    order = sorted(groups, key=lambda q: (q[0], morton_code(q[1], q[2], q[3])))
    M = len(order)
    coarse = np.array(order, dtype=np.int32).reshape(M, 4)
    parent = np.empty(len(clist), dtype=np.int32)
    mask = np.zeros(M, dtype=np.uint8)
    for p, q in enumerate(order):
        for i in groups[q]:
            parent[i] = p
            b, z, y, x = clist[i]
            mask[p] |= 1 << child_bit(z, y, x)
    pooled = None
    if feats is not None:
        f = np.asarray(feats, dtype=np.float64)
        if f.ndim != 2 or f.shape[0] != len(clist):
            raise OracleError("feats must be [N, C]")
        pooled = np.empty((M, f.shape[1]), dtype=np.float64)
        for p, q in enumerate(order):
            rows = f[groups[q]]
            pooled[p] = rows.sum(axis=0) / len(rows) if mode == "mean" else rows.max(axis=0)
    return coarse, pooled, parent, mask


def upsample(coarse_feats, parent):
    """SparseUpsample(2) with a stored subdivision: each fine row takes its parent's
    coarse row (the fine set is exactly the one the paired downsample saw), float64."""
    c = np.asarray(coarse_feats, dtype=np.float64)
    parent = np.asarray(parent)
    if parent.size and (parent.min() < 0 or parent.max() >= c.shape[0]):
        raise OracleError("parent index outside the coarse rows")
    return c[parent]


def spatial2channel(coords, feats, res):
    """SparseSpatial2Channel(2), the sparse pixel-unshuffle the "pixal3d_mrp_mlx README"
    scope table lists beside the down/upsample (cache-backed, paired with the same
    subdivision). Reading: each parent cell's row holds its eight children's feature
    rows side by side in child_bit order, zeros where a child is absent:

        out[p, k*C:(k+1)*C] = feats[i] if fine row i is child k of parent p, else 0.

    Returns (coarse_coords [M, 4], out float64 [M, 8C], parent [N], child_mask [M]) with
    the coarse set, order and subdivision of downsample()."""
    coarse, _, parent, mask = downsample(coords, None, res)
    f = np.asarray(feats, dtype=np.float64)
    C = f.shape[1]
    out = np.zeros((coarse.shape[0], 8 * C), dtype=np.float64)
    for i, (b, z, y, x) in enumerate(np.asarray(coords).tolist()):
        k = child_bit(z, y, x)
        out[parent[i], k * C:(k + 1) * C] = f[i]
    return coarse, out, parent, mask


def channel2spatial(coarse_feats, coords, parent):
    """The inverse of spatial2channel on the stored subdivision: fine row i takes the
    C-wide slice of its parent's row at its child_bit, float64 [N, C]."""
    c = np.asarray(coarse_feats, dtype=np.float64)
    if c.shape[1] % 8:
        raise OracleError("coarse rows must hold 8 x C channels")
    C = c.shape[1] // 8
    parent = np.asarray(parent)
    if parent.size and (parent.min() < 0 or parent.max() >= c.shape[0]):
        raise OracleError("parent index outside the coarse rows")
    out = np.empty((parent.shape[0], C), dtype=np.float64)
    for i, (b, z, y, x) in enumerate(np.asarray(coords).tolist()):
        k = child_bit(z, y, x)
        out[i] = c[parent[i], k * C:(k + 1) * C]
    return out


# ---------------------------------------------------------------------------------
# Occupancy-grouped tiles (the tile plan of the grouped forward). This is not part of
# the convolution's definition -- the grouped forward computes the same sums -- but the
# plan the GPU builds is a deterministic function of the voxel set and the window, so
# it is written out here as plainly as the rest and compared bit-exactly.

def morton_codes(coords):
    """morton_code(z, y, x) of every row of coords [N, 4] (b, z, y, x), as uint64 (the
    same bit interleave, one bit plane at a time over the whole array)."""
    c = np.asarray(coords, dtype=np.int64)
    m = np.zeros(c.shape[0], dtype=np.uint64)
    for t in range(16):
        for axis, col in ((0, 3), (1, 2), (2, 1)):       # x -> 3t, y -> 3t + 1, z -> 3t + 2
            bitv = ((c[:, col] >> t) & 1).astype(np.uint64)
            m |= bitv << np.uint64(3 * t + axis)
    return m


def neighbour_masks(nbr):
    """27-bit mask per row of a kernel map: bit k set when nbr[i, k] >= 0."""
    present = np.asarray(nbr) >= 0
    return (present.astype(np.uint64) << np.arange(27, dtype=np.uint64)).sum(axis=1).astype(np.uint32)


def tile_plan(coords, nbr, window, tile=128):
    """(perm [N], plan_nbr [N, 27], tile_mask [ceil(N / tile)]) of the grouped forward.

    The voxels in (batch, Morton code) order, ties by input row, are cut into windows of
    `window` consecutive voxels; inside each window they are sorted by neighbour mask
    (as an integer), keeping Morton order among equal masks. perm[r] is the input row
    at plan row r, plan_nbr the kernel map's rows in that order, and tile_mask[t] the OR
    of the masks of plan rows [tile t, tile t + tile)."""
    c = np.asarray(coords, dtype=np.int64)
    N = c.shape[0]
    rows = np.arange(N)
    morton_order = np.lexsort((rows, morton_codes(c), c[:, 0]))
    masks = neighbour_masks(nbr)
    window_of = rows // int(window)                       # window of each sorted position
    grouped = np.lexsort((rows, masks[morton_order], window_of))
    perm = morton_order[grouped].astype(np.int32)
    ntiles = (N + tile - 1) // tile
    padded = np.zeros(ntiles * tile, dtype=np.uint32)
    padded[:N] = masks[perm]
    tile_mask = np.bitwise_or.reduce(padded.reshape(ntiles, tile), axis=1).astype(np.uint32)
    return perm, np.asarray(nbr)[perm], tile_mask
