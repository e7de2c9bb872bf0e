"""Submanifold sparse 3D convolution (SubMConv3d: kernel 3, stride 1, no padding)
for NVIDIA B300 (sm_103a).

The convolution runs in libsubm3d.so (CUDA kernels behind the C ABI of
include/subm3d.h); this package is its Python binding, with the same names:

    nbr = subm3d_build_kmap(coords, res)                 # int32 [N, 27]
    out = subm3d_forward(feats, nbr, weight, bias)       # [N, O]
    y = subm3d_forward_ex(feats, nbr, weight, bias, residual=x, act="relu")

coords int32 [N, 4] (b, z, y, x); feats [N, I] bf16 or fp32 (channels-last);
weight [O, 3, 3, 3, I] ([O, kz, ky, kx, I]); bias [O] or None. subm3d_forward_ex fuses a
residual add and an activation (none, relu, silu) into the same kernel; one nbr serves
every convolution at its resolution. subm3d_downsample / subm3d_upsample are
SparseDownsample(2) (mean or max pooling) and its cache-paired SparseUpsample(2);
subm3d_spatial2channel / subm3d_channel2spatial the sparse pixel-unshuffle and its
inverse on the same subdivision.

Occupancy-grouped tiles: plan = subm3d_build_kmap_grouped(coords, res) orders the voxels
so that each 128-row tile's rows share their neighbour offsets, and
subm3d_forward_grouped(feats, plan, weight, bias) runs only the offsets each tile has;
out stays in input order.
"""
from ._binding import (ACTIVATIONS, BF16, F32, GROUP_MORTON, GROUP_WINDOW, LIB_PATH, POOL_MODES, Subm3dError,
                       lib, plan_views, subm3d_build_kmap, subm3d_build_kmap_async,
                       subm3d_build_kmap_ex, subm3d_build_kmap_grouped, subm3d_build_kmap_noalloc,
                       subm3d_forward_grouped, subm3d_kmap_grouped_workspace_bytes,
                       subm3d_plan_bytes, subm3d_kmap_stage_timing, subm3d_kmap_stage_times,
                       subm3d_downsample, subm3d_forward, subm3d_forward_ex, subm3d_forward_status,
                       subm3d_kernel_launches, subm3d_kmap_workspace_bytes, subm3d_last_error,
                       subm3d_upsample, subm3d_spatial2channel, subm3d_channel2spatial)

__all__ = ["ACTIVATIONS", "BF16", "F32", "GROUP_MORTON", "GROUP_WINDOW", "LIB_PATH", "POOL_MODES", "Subm3dError",
           "lib", "plan_views", "subm3d_build_kmap", "subm3d_build_kmap_async",
           "subm3d_build_kmap_ex", "subm3d_build_kmap_grouped", "subm3d_build_kmap_noalloc",
           "subm3d_forward_grouped", "subm3d_kmap_grouped_workspace_bytes", "subm3d_plan_bytes",
           "subm3d_kmap_stage_timing", "subm3d_kmap_stage_times",
           "subm3d_downsample", "subm3d_forward", "subm3d_forward_ex", "subm3d_forward_status",
           "subm3d_kernel_launches", "subm3d_kmap_workspace_bytes", "subm3d_last_error",
           "subm3d_upsample", "subm3d_spatial2channel", "subm3d_channel2spatial"]
