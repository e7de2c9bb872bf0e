"""CPU oracle for submanifold sparse 3D convolution (kernel 3, stride 1, no padding).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this package; the CUDA library and its Python binding never
do, and the two share no code. `ref` is the dict-of-coordinates triple loop in
float64 (small inputs); `cpu` loads the same definition written in plain C++ with
OpenMP over voxels (large inputs).

Pins (tests/test_oracle_pins.py): brute-force pairwise neighbour search, a dense
zero-padded Conv3d (torch CPU, float64) on small grids masked to the active sites,
a hand-worked example under tests/golden/, and invariants (isolated voxel sees only
the centre tap, translation and permutation equivariance, linearity, batch
independence, orientation of a single asymmetric tap).
"""
