"""The C ABI without a GPU: the library loads, exports every entry point that
include/subm3d.h declares, and host-side argument checks return before any CUDA call."""
import ctypes
import os
import re

import pytest

from submanifold_sparse_convolution_04_b300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "subm3d.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SUBM3D_API\s+[\w\s\*]+?\b(subm3d_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from submanifold_sparse_convolution_04_b300.build import build
    build()
    return B.lib()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("subm3d_build_kmap", "subm3d_forward", "subm3d_kmap_workspace_bytes",
                 "subm3d_last_error"):
        assert name in syms


def test_every_declared_symbol_is_exported(L):
    for name in declared_symbols():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read().split()
    exported = sorted(s for s in out if s.startswith("subm3d_"))
    assert exported == declared_symbols()


def test_workspace_bytes_host_only(L):
    assert L.subm3d_kmap_workspace_bytes(-1) == 0
    w0 = L.subm3d_kmap_workspace_bytes(0)
    w1 = L.subm3d_kmap_workspace_bytes(1000)
    w2 = L.subm3d_kmap_workspace_bytes(3_000_000)
    assert 0 < w0 < w1 < w2
    # two sort-key and three index buffers (28 B per voxel), the sort passes' status
    # words (8 B x 256 digits per 512-key tile: 4 B per voxel) and the block table
    # reserved for its worst case (8 M slots of 32 B) dominate at 3 M voxels
    lower = 3_000_000 * 32 + 32 * (1 << 23)
    assert lower <= w2 < 1.05 * lower + (1 << 22)
    assert L.subm3d_kmap_workspace_bytes_ex(1000, 64) < w1
    assert L.subm3d_kmap_workspace_bytes_ex(1000, 0) == w1


def test_empty_inputs_are_noops(L):
    assert L.subm3d_build_kmap(None, 0, 16, None, None, 0, None) == B.OK
    assert L.subm3d_forward(None, None, None, None, None, 0, 32, 32, B.BF16, None) == B.OK


@pytest.mark.parametrize("args,code", [
    ((None, -1, 16, None, None, 0, None), B.ERR_ARG),               # N < 0
    ((None, 10, 0, None, None, 0, None), B.ERR_ARG),                # res < 1
    ((None, 10, 65536, None, None, 0, None), B.ERR_ARG),            # res too large
    ((None, 10, 16, None, None, 0, None), B.ERR_ARG),               # NULL pointers
    ((16, 10, 16, 24, 256, 1 << 20, None), B.ERR_ARG),              # nbr not 16-byte aligned
    ((16, 10, 16, 32, 128, 1 << 20, None), B.ERR_WORKSPACE),        # workspace not 256-aligned
    ((16, 10, 16, 32, 256, 100, None), B.ERR_WORKSPACE),            # workspace too small
])
def test_build_kmap_argument_errors(L, args, code):
    vp = [ctypes.c_void_p(a) if isinstance(a, int) and i in (0, 3, 4) else a
          for i, a in enumerate(args)]
    assert L.subm3d_build_kmap(*vp) == code
    assert B.subm3d_last_error()


def test_build_kmap_ex_capacity_checks(L):
    p = ctypes.c_void_p
    for cap in (-8, 3, 12, 1 << 41):
        assert L.subm3d_build_kmap_ex(p(16), 10, 16, p(32), None, cap, p(256), 1 << 20, None) == B.ERR_ARG


@pytest.mark.parametrize("N,I,O,dtype,code", [
    (-1, 32, 32, B.BF16, B.ERR_ARG), (10, 0, 32, B.BF16, B.ERR_ARG), (10, 32, 5000, B.F32, B.ERR_ARG),
    (10, 32, 32, 7, B.ERR_ARG), (10, 12, 32, B.BF16, B.ERR_UNSUPPORTED),
    (10, 32, 20, B.BF16, B.ERR_UNSUPPORTED)])
def test_forward_argument_errors(L, N, I, O, dtype, code):
    p = ctypes.c_void_p
    assert L.subm3d_forward(p(256), p(512), p(768), None, p(1024), N, I, O, dtype, None) == code


def test_forward_null_and_alignment(L):
    p = ctypes.c_void_p
    assert L.subm3d_forward(None, p(512), p(768), None, p(1024), 10, 32, 32, B.BF16, None) == B.ERR_ARG
    assert L.subm3d_forward(p(256), p(512), p(768), p(8), p(1024), 10, 32, 32, B.BF16, None) == B.ERR_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    from submanifold_sparse_convolution_04_b300 import subm3d_build_kmap, subm3d_forward
    with pytest.raises(ValueError):
        subm3d_build_kmap(torch.zeros((4, 4), dtype=torch.int32), 8)
    with pytest.raises(ValueError):
        subm3d_forward(torch.zeros((4, 8)), torch.zeros((4, 27), dtype=torch.int32),
                       torch.zeros((8, 3, 3, 3, 8)))


def test_forward_ex_argument_errors(L):
    p = ctypes.c_void_p
    args = lambda res, act, out: (p(256), p(512), p(768), None, res, act, out, 10, 32, 32, B.BF16, None)
    assert L.subm3d_forward_ex(*args(None, 7, p(1024))) == B.ERR_ARG          # unknown activation
    assert b"activation" in L.subm3d_last_error()
    assert L.subm3d_forward_ex(*args(p(1032), 1, p(4096))) == B.ERR_ARG       # residual misaligned
    assert L.subm3d_forward_ex(*args(p(4096 + 64), 2, p(4096))) == B.ERR_ARG  # partial overlap
    assert b"overlaps" in L.subm3d_last_error()
    assert L.subm3d_forward_ex(p(256), p(512), p(768), None, None, 1, None, 0, 32, 32, B.BF16,
                               None) == B.OK                                    # N = 0


def test_downsample_host_checks(L):
    p = ctypes.c_void_p
    M = ctypes.c_int64(-5)
    ws = L.subm3d_downsample_workspace_bytes
    assert ws(-1) == 0 and 0 < ws(0) < ws(1000) < ws(3_000_000)
    # no block table: below the kernel map's workspace at the same N
    assert ws(3_000_000) < L.subm3d_kmap_workspace_bytes(3_000_000)

    def call(coords=16, N=10, res=16, feats=None, C=0, dtype=B.BF16, mode=0, cc=32, cf=None,
             parent=48, mask=64, m=M, w=256, nbytes=1 << 30):
        return L.subm3d_downsample(p(coords) if coords else None, N, res,
                                   p(feats) if feats else None, C, dtype, mode,
                                   p(cc) if cc else None, p(cf) if cf else None,
                                   p(parent) if parent else None, p(mask) if mask else None,
                                   ctypes.byref(m) if m is not None else None,
                                   p(w) if w else None, nbytes, None)
    assert call(m=None) == B.ERR_ARG
    assert call(N=-1) == B.ERR_ARG and M.value == 0
    assert call(res=0) == B.ERR_ARG
    assert call(mode=5) == B.ERR_ARG
    assert call(feats=80, C=0, cf=96) == B.ERR_ARG
    assert call(feats=80, C=8, dtype=9, cf=96) == B.ERR_ARG
    assert call(N=0) == B.OK and M.value == 0
    assert call(coords=None) == B.ERR_ARG
    assert call(feats=80, C=8, cf=None) == B.ERR_ARG          # feats without coarse_feats
    assert call(parent=52) == B.ERR_ARG                       # misaligned
    assert call(w=128) == B.ERR_WORKSPACE                     # workspace not 256-aligned
    assert call(nbytes=100) == B.ERR_WORKSPACE
    assert b"workspace" in L.subm3d_last_error()


def test_downsample_async_host_checks(L):
    p = ctypes.c_void_p

    def call(M=1024, N=10, res=16, order=None, w=256, nbytes=1 << 30, mode=0):
        return L.subm3d_downsample_async(p(16), N, res, p(order) if order else None, None, 0,
                                         B.BF16, mode, p(32), None, p(48), p(64),
                                         p(M) if M else None, p(w), nbytes, None)
    assert call(M=None) == B.ERR_ARG                  # the device word for M is required
    assert call(M=1028) == B.ERR_ARG                  # and 8-byte aligned
    assert call(N=-1) == B.ERR_ARG and call(res=0) == B.ERR_ARG and call(mode=7) == B.ERR_ARG
    assert call(order=20) == B.ERR_ARG                # order not 16-byte aligned
    assert call(nbytes=100) == B.ERR_WORKSPACE
    assert b"subm3d_downsample" in L.subm3d_last_error()


def test_upsample_and_pixel_shuffle_host_checks(L):
    p = ctypes.c_void_p
    assert L.subm3d_upsample(p(16), 4, 8, p(32), -1, B.BF16, p(64), None) == B.ERR_ARG
    assert L.subm3d_upsample(p(16), 4, 0, p(32), 10, B.BF16, p(64), None) == B.ERR_ARG
    assert L.subm3d_upsample(p(16), 4, 8, p(32), 10, 7, p(64), None) == B.ERR_ARG
    assert L.subm3d_upsample(p(16), 4, 8, p(32), 0, B.BF16, p(64), None) == B.OK
    assert L.subm3d_upsample(p(16), 4, 8, None, 10, B.BF16, p(64), None) == B.ERR_ARG
    assert L.subm3d_upsample(p(16), 4, 8, p(36), 10, B.BF16, p(64), None) == B.ERR_ARG
    s2c = L.subm3d_spatial2channel
    assert s2c(p(16), p(32), p(48), p(60), 10, 4, 0, B.F32, p(64), None) == B.ERR_ARG
    assert s2c(p(16), p(32), p(48), p(60), 10, -4, 8, B.F32, p(64), None) == B.ERR_ARG
    assert s2c(None, None, None, None, 0, 0, 8, B.F32, None, None) == B.OK
    assert s2c(p(16), p(32), p(48), None, 10, 4, 8, B.F32, p(64), None) == B.ERR_ARG
    assert s2c(p(16), p(32), p(48), p(61), 10, 4, 8, B.F32, p(72), None) == B.ERR_ARG
    c2s = L.subm3d_channel2spatial
    assert c2s(p(16), p(32), p(48), 0, 4, 8, B.BF16, p(64), None) == B.OK
    assert c2s(p(16), p(32), p(48), 10, 4, 4097, B.BF16, p(64), None) == B.ERR_ARG
    assert c2s(p(16), None, p(48), 10, 4, 8, B.BF16, p(64), None) == B.ERR_ARG
    assert c2s(p(24), p(32), p(48), 10, 4, 8, B.BF16, p(64), None) == B.ERR_ARG


def test_binding_refuses_bad_arguments_without_a_gpu():
    import torch
    from submanifold_sparse_convolution_04_b300 import (subm3d_channel2spatial, subm3d_downsample,
                                                        subm3d_forward_ex, subm3d_spatial2channel,
                                                        subm3d_upsample)
    f = torch.zeros((4, 8))
    nbr = torch.zeros((4, 27), dtype=torch.int32)
    w = torch.zeros((8, 3, 3, 3, 8))
    with pytest.raises(ValueError):
        subm3d_forward_ex(f, nbr, w, act="gelu")
    with pytest.raises(ValueError):
        subm3d_forward_ex(f, nbr, w, act="relu")                  # CPU tensors
    with pytest.raises(ValueError):
        subm3d_downsample(torch.zeros((4, 4), dtype=torch.int32), 8, mode="sum")
    with pytest.raises(ValueError):
        subm3d_downsample(torch.zeros((4, 4), dtype=torch.int32), 8)
    with pytest.raises(ValueError):
        subm3d_upsample(f, torch.zeros(4, dtype=torch.int32))
    with pytest.raises(ValueError):
        subm3d_channel2spatial(torch.zeros((2, 12)), torch.zeros((4, 4), dtype=torch.int32),
                               torch.zeros(4, dtype=torch.int32))   # 12 channels: not 8 x C
    with pytest.raises(ValueError):
        subm3d_spatial2channel(f, torch.zeros((4, 4), dtype=torch.int32),
                               torch.zeros(4, dtype=torch.int32), torch.zeros(2, dtype=torch.uint8))


def test_launchers_refuse_without_a_device_error_word(L):
    # Every forward, upsample and pixel-shuffle launcher fetches its device's error word
    # first and returns ERR_CUDA, launching nothing, when it cannot be had (here: no
    # CUDA device). The pointers are never dereferenced on that path.
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a host without a CUDA device")
    p = ctypes.c_void_p
    for I, O, dt in ((64, 64, B.BF16), (128, 128, B.BF16), (64, 520, B.BF16), (32, 32, B.F32)):
        assert L.subm3d_forward(p(256), p(512), p(768), None, p(1024), 10, I, O, dt, None) == B.ERR_CUDA
        assert b"error word" in L.subm3d_last_error() or b"cudaGetDevice" in L.subm3d_last_error()
    assert L.subm3d_upsample(p(16), 4, 8, p(32), 10, B.BF16, p(64), None) == B.ERR_CUDA
    assert L.subm3d_spatial2channel(p(16), p(32), p(48), p(64), 10, 4, 8, B.F32, p(80),
                                    None) == B.ERR_CUDA
    assert L.subm3d_channel2spatial(p(16), p(32), p(48), 10, 4, 8, B.BF16, p(64), None) == B.ERR_CUDA
    assert L.subm3d_forward_status(None) == B.ERR_CUDA


def test_tile_plan_host_checks(L):
    p = ctypes.c_void_p
    # a plan holds perm (4 B) and the nbr rows (108 B) per voxel and one offset mask per
    # 128-row tile, each part 256-byte aligned
    for N in (1, 1000, 3_000_000):
        pb = L.subm3d_plan_bytes(N)
        least = N * 112 + ((N + 127) // 128) * 4
        assert least <= pb < least + 4096
        assert L.subm3d_kmap_grouped_workspace_bytes(N) > L.subm3d_kmap_workspace_bytes(N)
    assert L.subm3d_plan_bytes(-1) == 0
    assert L.subm3d_build_kmap_grouped(None, 0, 16, 1, None, 0, None, 0, 0, None) == B.OK
    good = dict(coords=p(16), N=10, res=16, window=1, plan=p(256), pb=L.subm3d_plan_bytes(10),
                ws=p(512), wb=1 << 24, flags=0)

    def call(**kw):
        d = dict(good, **kw)
        return L.subm3d_build_kmap_grouped(d["coords"], d["N"], d["res"], d["window"], d["plan"],
                                           d["pb"], d["ws"], d["wb"], d["flags"], None)

    for w in (3, -4, 1 << 31, 6):         # not a power of two in [1, 2^30] (0 is the default)
        assert call(window=w) == B.ERR_ARG
    assert call(pb=good["pb"] - 1) == B.ERR_ARG      # plan too small
    assert call(plan=p(128)) == B.ERR_ARG            # plan not 256-byte aligned
    assert call(plan=None) == B.ERR_ARG
    assert call(coords=p(8)) == B.ERR_ARG            # coords not 16-byte aligned
    assert call(wb=100) == B.ERR_WORKSPACE
    assert call(ws=p(384)) == B.ERR_WORKSPACE        # workspace not 256-byte aligned
    assert call(flags=4) == B.ERR_ARG                # unknown flag
    assert call(res=0) == B.ERR_ARG and call(N=-1) == B.ERR_ARG
    assert B.subm3d_last_error()
    # the forward on a plan: no plan, a misaligned one, N out of range, bad shapes
    f = L.subm3d_forward_grouped
    assert f(p(256), None, p(768), None, None, 0, p(1024), 10, 32, 32, B.BF16, None) == B.ERR_ARG
    assert f(p(256), p(128), p(768), None, None, 0, p(1024), 10, 32, 32, B.BF16, None) == B.ERR_ARG
    assert f(p(256), p(256), p(768), None, None, 0, p(1024), -1, 32, 32, B.BF16, None) == B.ERR_ARG
    assert f(p(256), p(256), p(768), None, None, 0, p(1024), 10, 12, 32, B.BF16, None) == \
        B.ERR_UNSUPPORTED
    assert f(None, None, None, None, None, 0, None, 0, 32, 32, B.BF16, None) == B.OK
