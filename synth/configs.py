"""The five synthetic workloads and their seeded value draws.

Each workload is a set of surface shells on a cubic grid plus channels-last
features, a weight [O, 3, 3, 3, I] and a bias [O]:

  1  tiny fp32:  batch 1, 16^3, sphere shell centre 8 radius 5 (+-0.5), I = O = 32
  2  batch 1, 64^3, one ellipsoid shell, semi-axes U[16, 28], ~3.6 k voxels, I = O = 128, bf16
  3  batch 2, 256^3, per item an ellipsoid shell plus 3 torus shells, ~150 k voxels
     per item, I = O = 256, bf16
  4  batch 1, 512^3, union of 8 ellipsoid shells, ~700 k voxels, I = O = 128, bf16
  5  batch 1, 1024^3, union of 16 ellipsoid / torus shells, ~3 M voxels, I = O = 64, bf16

Values: feats ~ N(0, 1); weight ~ N(0, sigma = 1/sqrt(27 I)); bias ~ N(0, 0.1),
drawn in fp32 and rounded to bf16 (round to nearest even) for the bf16 workloads.

Shape parameters are drawn from numpy PCG64(seed = workload number); a draw whose
voxel count misses the target by more than 20 % is redrawn from the same stream,
so the accepted set is a deterministic function of the seed. Values come from an
independent stream PCG64([seed, 1]) so they do not depend on how many redraws the
geometry needed.
"""
from __future__ import annotations

import numpy as np

from .shells import ellipsoid_shell, torus_shell, union_coords, uniform_rotation

__all__ = ["CONFIGS", "make_coords", "make_values", "make_case", "round_to_bf16"]

CONFIGS = {
    1: dict(name="sphere16_tiny_fp32", res=16, batch=1, I=32, O=32, dtype="f32", target=None),
    2: dict(name="ellipsoid64", res=64, batch=1, I=128, O=128, dtype="bf16", target=3600),
    3: dict(name="ellipsoid_tori256_b2", res=256, batch=2, I=256, O=256, dtype="bf16",
            target=150_000),
    4: dict(name="ellipsoids8_512", res=512, batch=1, I=128, O=128, dtype="bf16",
            target=700_000),
    5: dict(name="shells16_1024", res=1024, batch=1, I=64, O=64, dtype="bf16",
            target=3_000_000),
}


def _center(rng, res, extent):
    lo = extent
    hi = res - 1 - extent
    if hi <= lo:
        return np.full(3, (res - 1) / 2.0)
    return lo + (hi - lo) * rng.random(3)


def _ellipsoid(rng, res, amin, amax):
    axes = amin + (amax - amin) * rng.random(3)
    rot = uniform_rotation(rng)
    c = _center(rng, res, axes.max() + 1.0)
    return ellipsoid_shell(res, c, axes, rot)


def _torus(rng, res, rmaj, rmin):
    R = rmaj[0] + (rmaj[1] - rmaj[0]) * rng.random()
    r = rmin[0] + (rmin[1] - rmin[0]) * rng.random()
    rot = uniform_rotation(rng)
    c = _center(rng, res, R + r + 1.0)
    return torus_shell(res, c, R, r, rot)


def _draw_item(cfg_id, rng, res):
    """One batch item's shapes for workload cfg_id: a list of [M, 3] point arrays."""
    if cfg_id == 2:
        return [_ellipsoid(rng, res, 16.0, 28.0)]
    if cfg_id == 3:
        return [_ellipsoid(rng, res, 60.0, 100.0)] + [
            _torus(rng, res, (30.0, 60.0), (8.0, 16.0)) for _ in range(3)]
    if cfg_id == 4:
        return [_ellipsoid(rng, res, 60.0, 110.0) for _ in range(8)]
    if cfg_id == 5:
        out = []
        for _ in range(16):
            if rng.random() < 0.5:
                out.append(_ellipsoid(rng, res, 90.0, 160.0))
            else:
                out.append(_torus(rng, res, (120.0, 250.0), (15.0, 35.0)))
        return out
    raise ValueError(cfg_id)


def make_coords(cfg_id: int, order: str = "raster", max_redraws: int = 64):
    """Coordinates int32 [N, 4] (b, z, y, x) of workload cfg_id and a record of the draw.

    order="raster" gives (b, z, y, x) lexicographic order; order="shuffled" applies a
    seeded random permutation to the rows (a robustness case for the kernels).
    """
    cfg = CONFIGS[cfg_id]
    res, batch = cfg["res"], cfg["batch"]
    rng = np.random.Generator(np.random.PCG64(cfg_id))
    if cfg_id == 1:
        pts = ellipsoid_shell(res, (8.0, 8.0, 8.0), (5.0, 5.0, 5.0), np.eye(3))
        coords = union_coords([(0, pts)], res)
        info = dict(redraws=0)
    else:
        target = cfg["target"]
        parts = []
        redraws = 0
        for b in range(batch):
            for attempt in range(max_redraws):
                shapes = _draw_item(cfg_id, rng, res)
                item = union_coords([(0, np.concatenate(shapes, axis=0))], res)
                if abs(item.shape[0] - target) <= 0.2 * target:
                    break
                redraws += 1
            else:
                raise RuntimeError(f"workload {cfg_id}: no draw within 20% of {target}")
            parts.append((b, item[:, 1:].astype(np.int64)))
        coords = union_coords(parts, res)
        info = dict(redraws=redraws)
    if order == "shuffled":
        prng = np.random.Generator(np.random.PCG64([cfg_id, 2]))
        coords = coords[prng.permutation(coords.shape[0])]
    elif order != "raster":
        raise ValueError(order)
    info.update(N=int(coords.shape[0]), res=res, batch=batch, order=order)
    return np.ascontiguousarray(coords), info


def round_to_bf16(x: np.ndarray):
    """Round finite float32 values to bfloat16, nearest-even.

    Returns (values as float32, exactly representable in bf16; raw bf16 bits uint16).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32), (r >> np.uint32(16)).astype(np.uint16)


def make_values(N: int, I: int, O: int, dtype: str, seed: int):
    """feats [N, I], weight [O, 3, 3, 3, I], bias [O] as float32 arrays.

    For dtype "bf16" every value is exactly representable in bf16 and the raw bf16
    bits are returned too (keys feats_bits, weight_bits, bias_bits).
    """
    rng = np.random.Generator(np.random.PCG64([seed, 1]))
    feats = rng.standard_normal((N, I), dtype=np.float32)
    weight = rng.standard_normal((O, 3, 3, 3, I), dtype=np.float32) * np.float32(
        1.0 / np.sqrt(27.0 * I))
    bias = rng.standard_normal(O, dtype=np.float32) * np.float32(0.1)
    out = dict(feats=feats, weight=weight.astype(np.float32), bias=bias.astype(np.float32))
    if dtype == "bf16":
        for k in ("feats", "weight", "bias"):
            v, bits = round_to_bf16(out[k])
            out[k] = v
            out[k + "_bits"] = bits
    elif dtype != "f32":
        raise ValueError(dtype)
    return out


def make_residual(N: int, O: int, dtype: str, seed: int):
    """Skip-path input [N, O] of the fused block epilogue: N(0, 1) float32 values (its
    own stream of the seed), rounded to bf16 for dtype "bf16". Returns (values, bf16
    bits or None)."""
    rng = np.random.Generator(np.random.PCG64([seed, 2]))
    r = rng.standard_normal((N, O), dtype=np.float32)
    if dtype == "bf16":
        return round_to_bf16(r)
    if dtype != "f32":
        raise ValueError(dtype)
    return r, None


def make_case(cfg_id: int, order: str = "raster"):
    """Coordinates and values of workload cfg_id (see the module docstring)."""
    cfg = CONFIGS[cfg_id]
    coords, info = make_coords(cfg_id, order)
    vals = make_values(coords.shape[0], cfg["I"], cfg["O"], cfg["dtype"], cfg_id)
    case = dict(cfg_id=cfg_id, name=cfg["name"], res=cfg["res"], I=cfg["I"], O=cfg["O"],
                dtype=cfg["dtype"], coords=coords, info=info)
    case.update(vals)
    return case
