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

__all__ = ["OFFSETS", "CENTER", "ACTIVATIONS", "OracleError", "tap", "coordinate_dict",
           "kernel_map", "subm_conv3d", "subm_conv3d_rows", "activation", "block_epilogue"]

# k -> (dz, dy, dx), k = 9 (dz + 1) + 3 (dy + 1) + (dx + 1)
OFFSETS = [(dz, dy, dx) for dz in (-1, 0, 1) for dy in (-1, 0, 1) for dx in (-1, 0, 1)]
CENTER = 13
ACTIVATIONS = ("none", "relu", "silu")
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
