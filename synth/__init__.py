"""Seeded synthetic surface-shell voxel sets and feature/weight values.

This module is shared by the tests, the benchmark and the smoke check. It holds
no part of the convolution itself: it only draws integer lattice coordinates
(shells of ellipsoids, spheres and tori) and random feature, weight and bias
values. Both the CUDA path and the CPU oracle consume what it produces.
"""
from .shells import ellipsoid_shell, torus_shell, union_coords, uniform_rotation
from .configs import (CONFIGS, make_case, make_coords, make_residual, make_values,
                      round_to_bf16)

__all__ = ["ellipsoid_shell", "torus_shell", "union_coords", "uniform_rotation", "CONFIGS",
           "make_case", "make_coords", "make_residual", "make_values", "round_to_bf16"]
