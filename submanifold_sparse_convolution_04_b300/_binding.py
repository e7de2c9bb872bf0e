"""ctypes binding of libsubm3d.so (include/subm3d.h). Argument marshalling only:
every step of the convolution runs in the library's CUDA kernels; PyTorch supplies
device memory and the current stream. There is no other code path: if the library
is missing or the tensors are not on a CUDA device, the calls raise."""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsubm3d.so")

OK, ERR_ARG, ERR_COORD_RANGE, ERR_DUPLICATE, ERR_HASH_FULL, ERR_CUDA, ERR_UNSUPPORTED, \
    ERR_WORKSPACE, ERR_DEVICE = 0, -1, -2, -3, -4, -5, -6, -7, -8
F32, BF16 = 0, 1
_DTYPES = {torch.float32: F32, torch.bfloat16: BF16}
ACTIVATIONS = {"none": 0, "relu": 1, "silu": 2}   # subm3d_act
POOL_MODES = {"mean": 0, "max": 1}                 # subm3d_pool
_NAMES = {0: "OK", -1: "ERR_ARG", -2: "ERR_COORD_RANGE", -3: "ERR_DUPLICATE", -4: "ERR_HASH_FULL",
          -5: "ERR_CUDA", -6: "ERR_UNSUPPORTED", -7: "ERR_WORKSPACE", -8: "ERR_DEVICE"}

_lib = None


class Subm3dError(RuntimeError):
    """A libsubm3d call returned a non-zero status."""

    def __init__(self, code: int, message: str):
        super().__init__(f"{_NAMES.get(code, code)}: {message}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m submanifold_sparse_convolution_04_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        L.subm3d_kmap_workspace_bytes.argtypes = [i64]
        L.subm3d_kmap_workspace_bytes.restype = sz
        L.subm3d_kmap_workspace_bytes_ex.argtypes = [i64, i64]
        L.subm3d_kmap_workspace_bytes_ex.restype = sz
        L.subm3d_build_kmap.argtypes = [vp, i64, i32, vp, vp, sz, vp]
        L.subm3d_build_kmap.restype = ctypes.c_int
        L.subm3d_build_kmap_ex.argtypes = [vp, i64, i32, vp, vp, i64, vp, sz, vp]
        L.subm3d_build_kmap_ex.restype = ctypes.c_int
        L.subm3d_build_kmap_noalloc.argtypes = [vp, i64, i32, vp, vp]
        L.subm3d_build_kmap_noalloc.restype = ctypes.c_int
        L.subm3d_build_kmap_async.argtypes = [vp, i64, i32, vp, vp, sz, vp]
        L.subm3d_build_kmap_async.restype = ctypes.c_int
        L.subm3d_plan_bytes.argtypes = [i64]
        L.subm3d_plan_bytes.restype = sz
        L.subm3d_kmap_grouped_workspace_bytes.argtypes = [i64]
        L.subm3d_kmap_grouped_workspace_bytes.restype = sz
        L.subm3d_build_kmap_grouped.argtypes = [vp, i64, i32, i64, vp, sz, vp, sz, ctypes.c_uint,
                                                vp]
        L.subm3d_build_kmap_grouped.restype = ctypes.c_int
        L.subm3d_forward_grouped.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, vp, i64, i32, i32,
                                             ctypes.c_int, vp]
        L.subm3d_forward_grouped.restype = ctypes.c_int
        L.subm3d_forward.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, ctypes.c_int, vp]
        L.subm3d_forward.restype = ctypes.c_int
        L.subm3d_forward_ex.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, vp, i64, i32, i32,
                                        ctypes.c_int, vp]
        L.subm3d_forward_ex.restype = ctypes.c_int
        L.subm3d_downsample_workspace_bytes.argtypes = [i64]
        L.subm3d_downsample_workspace_bytes.restype = sz
        L.subm3d_downsample.argtypes = [vp, i64, i32, vp, i32, ctypes.c_int, ctypes.c_int, vp, vp,
                                        vp, vp, ctypes.POINTER(ctypes.c_int64), vp, sz, vp]
        L.subm3d_downsample.restype = ctypes.c_int
        L.subm3d_downsample_sorted.argtypes = [vp, i64, i32, vp, vp, i32, ctypes.c_int,
                                               ctypes.c_int, vp, vp, vp, vp,
                                               ctypes.POINTER(ctypes.c_int64), vp, sz, vp]
        L.subm3d_downsample_sorted.restype = ctypes.c_int
        L.subm3d_downsample_async.argtypes = [vp, i64, i32, vp, vp, i32, ctypes.c_int,
                                              ctypes.c_int, vp, vp, vp, vp, vp, vp, sz, vp]
        L.subm3d_downsample_async.restype = ctypes.c_int
        L.subm3d_upsample.argtypes = [vp, i64, i32, vp, i64, ctypes.c_int, vp, vp]
        L.subm3d_upsample.restype = ctypes.c_int
        L.subm3d_spatial2channel.argtypes = [vp, vp, vp, vp, i64, i64, i32, ctypes.c_int, vp, vp]
        L.subm3d_spatial2channel.restype = ctypes.c_int
        L.subm3d_channel2spatial.argtypes = [vp, vp, vp, i64, i64, i32, ctypes.c_int, vp, vp]
        L.subm3d_channel2spatial.restype = ctypes.c_int
        L.subm3d_forward_status.argtypes = [vp]
        L.subm3d_forward_status.restype = ctypes.c_int
        L.subm3d_kmap_stage_timing.argtypes = [ctypes.c_int]
        L.subm3d_kmap_stage_timing.restype = None
        L.subm3d_kmap_stage_times.argtypes = [ctypes.POINTER(ctypes.c_float),
                                              ctypes.POINTER(ctypes.c_char_p), ctypes.c_int]
        L.subm3d_kmap_stage_times.restype = ctypes.c_int
        L.subm3d_last_error.argtypes = []
        L.subm3d_last_error.restype = ctypes.c_char_p
        L.subm3d_kernel_launches.argtypes = []
        L.subm3d_kernel_launches.restype = ctypes.c_int64
        _lib = L
    return _lib


def _check(rc: int):
    if rc != OK:
        raise Subm3dError(rc, subm3d_last_error())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def subm3d_last_error() -> str:
    return lib().subm3d_last_error().decode()


def subm3d_kernel_launches() -> int:
    return int(lib().subm3d_kernel_launches())


def subm3d_kmap_workspace_bytes(N: int, hash_capacity: int = 0) -> int:
    if hash_capacity:
        return int(lib().subm3d_kmap_workspace_bytes_ex(N, hash_capacity))
    return int(lib().subm3d_kmap_workspace_bytes(N))


def _workspace(N, hash_capacity, workspace, device):
    need = subm3d_kmap_workspace_bytes(N, hash_capacity)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace, _dev(workspace, "workspace", torch.uint8), workspace.numel()


def subm3d_build_kmap(coords: torch.Tensor, res: int, nbr: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """nbr int32 [N, 27] of the voxel set coords int32 [N, 4] (b, z, y, x)."""
    N = coords.shape[0]
    pc = _dev(coords, "coords", torch.int32, (N, 4))
    if nbr is None:
        nbr = torch.empty((N, 27), dtype=torch.int32, device=coords.device)
    pn = _dev(nbr, "nbr", torch.int32, (N, 27))
    workspace, pw, nbytes = _workspace(N, 0, workspace, coords.device)
    _check(lib().subm3d_build_kmap(pc, N, int(res), pn, pw, nbytes, _stream(stream)))
    return nbr


def subm3d_build_kmap_ex(coords: torch.Tensor, res: int, nbr: torch.Tensor | None = None,
                         order: torch.Tensor | bool | None = None, hash_capacity: int = 0,
                         workspace: torch.Tensor | None = None, stream=None):
    """(nbr, order): order int32 [N] is the Morton order if requested (order=True or a
    tensor), else None."""
    N = coords.shape[0]
    pc = _dev(coords, "coords", torch.int32, (N, 4))
    if nbr is None:
        nbr = torch.empty((N, 27), dtype=torch.int32, device=coords.device)
    pn = _dev(nbr, "nbr", torch.int32, (N, 27))
    if order is True:
        order = torch.empty(N, dtype=torch.int32, device=coords.device)
    elif order is False:
        order = None
    po = None if order is None else _dev(order, "order", torch.int32, (N,))
    workspace, pw, nbytes = _workspace(N, hash_capacity, workspace, coords.device)
    _check(lib().subm3d_build_kmap_ex(pc, N, int(res), pn, po, int(hash_capacity), pw, nbytes,
                                      _stream(stream)))
    return nbr, order


def subm3d_build_kmap_noalloc(coords: torch.Tensor, res: int, nbr: torch.Tensor,
                              stream=None) -> torch.Tensor:
    """nbr int32 [N, 27] of coords int32 [N, 4], written into the caller's nbr, with the
    library's built-in scratch instead of a workspace (N <= 131072). Allocates nothing."""
    N = coords.shape[0]
    pc = _dev(coords, "coords", torch.int32, (N, 4))
    pn = _dev(nbr, "nbr", torch.int32, (N, 27))
    _check(lib().subm3d_build_kmap_noalloc(pc, N, int(res), pn, _stream(stream)))
    return nbr


def subm3d_build_kmap_async(coords: torch.Tensor, res: int, nbr: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """subm3d_build_kmap without waiting for the stream; device-side errors surface at the
    next subm3d_forward_status()."""
    N = coords.shape[0]
    pc = _dev(coords, "coords", torch.int32, (N, 4))
    if nbr is None:
        nbr = torch.empty((N, 27), dtype=torch.int32, device=coords.device)
    pn = _dev(nbr, "nbr", torch.int32, (N, 27))
    workspace, pw, nbytes = _workspace(N, 0, workspace, coords.device)
    _check(lib().subm3d_build_kmap_async(pc, N, int(res), pn, pw, nbytes, _stream(stream)))
    return nbr


KMAP_ASYNC = 1
GROUP_WINDOW = 262144
GROUP_MORTON = 1   # window 1: tiles of the Morton order (no grouping sort)


def subm3d_plan_bytes(N: int) -> int:
    return int(lib().subm3d_plan_bytes(N))


def subm3d_kmap_grouped_workspace_bytes(N: int) -> int:
    return int(lib().subm3d_kmap_grouped_workspace_bytes(N))


def plan_views(plan: torch.Tensor, N: int):
    """(perm int32 [N], nbr int32 [N, 27], tile_mask int32 [ceil(N/128)]) views of a tile
    plan buffer, at the offsets include/subm3d.h documents (each part 256-byte aligned;
    tile_mask holds uint32 bit patterns)."""
    a256 = lambda x: (x + 255) // 256 * 256
    o_nbr = a256(4 * N)
    o_mask = a256(o_nbr + 4 * 27 * N)
    nt = (N + 127) // 128
    b = plan.view(torch.uint8)
    perm = b[0:4 * N].view(torch.int32)
    nbr = b[o_nbr:o_nbr + 4 * 27 * N].view(torch.int32).view(N, 27)
    mask = b[o_mask:o_mask + 4 * nt].view(torch.int32)
    return perm, nbr, mask


def subm3d_build_kmap_grouped(coords: torch.Tensor, res: int, window: int = 0,
                              plan: torch.Tensor | None = None,
                              workspace: torch.Tensor | None = None, async_: bool = False,
                              stream=None) -> torch.Tensor:
    """The kernel map as a tile plan (uint8 device buffer; see plan_views). window 0 is
    the default grouping window; GROUP_MORTON (1) gives tiles of the Morton order."""
    N = coords.shape[0]
    dev = coords.device
    pc = _dev(coords, "coords", torch.int32, (N, 4))
    if plan is None:
        plan = torch.empty(max(subm3d_plan_bytes(N), 256), dtype=torch.uint8, device=dev)
    pp = _dev(plan, "plan", torch.uint8)
    need = subm3d_kmap_grouped_workspace_bytes(N)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    pw = _dev(workspace, "workspace", torch.uint8)
    _check(lib().subm3d_build_kmap_grouped(pc, N, int(res), int(window), pp, plan.numel(), pw,
                                           workspace.numel(), KMAP_ASYNC if async_ else 0,
                                           _stream(stream)))
    return plan


def subm3d_forward_grouped(feats: torch.Tensor, plan: torch.Tensor, weight: torch.Tensor,
                           bias: torch.Tensor | None = None, residual: torch.Tensor | None = None,
                           act: str = "none", out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """subm3d_forward_ex on a tile plan from subm3d_build_kmap_grouped (same voxels)."""
    if feats.dtype not in _DTYPES:
        raise ValueError(f"feats dtype {feats.dtype} is not float32 or bfloat16")
    if act not in ACTIVATIONS:
        raise ValueError(f"act {act!r} is not one of {sorted(ACTIVATIONS)}")
    N, I = feats.shape
    O = weight.shape[0]
    pf = _dev(feats, "feats")
    pp = _dev(plan, "plan", torch.uint8)
    if plan.numel() < subm3d_plan_bytes(N):
        raise ValueError(f"plan has {plan.numel()} bytes, a plan for N={N} needs "
                         f"{subm3d_plan_bytes(N)}")
    pw = _dev(weight, "weight", feats.dtype, (O, 3, 3, 3, I))
    pb = None if bias is None else _dev(bias, "bias", feats.dtype, (O,))
    pr = None if residual is None else _dev(residual, "residual", feats.dtype, (N, O))
    if out is None:
        out = torch.empty((N, O), dtype=feats.dtype, device=feats.device)
    po = _dev(out, "out", feats.dtype, (N, O))
    _check(lib().subm3d_forward_grouped(pf, pp, pw, pb, pr, ACTIVATIONS[act], po, N, I, O,
                                        _DTYPES[feats.dtype], _stream(stream)))
    return out


def subm3d_forward(feats: torch.Tensor, nbr: torch.Tensor, weight: torch.Tensor,
                   bias: torch.Tensor | None = None, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """out [N, O] = submanifold convolution of feats [N, I] with weight [O, 3, 3, 3, I]."""
    if feats.dtype not in _DTYPES:
        raise ValueError(f"feats dtype {feats.dtype} is not float32 or bfloat16")
    N, I = feats.shape
    O = weight.shape[0]
    pf = _dev(feats, "feats")
    pn = _dev(nbr, "nbr", torch.int32, (N, 27))
    pw = _dev(weight, "weight", feats.dtype, (O, 3, 3, 3, I))
    pb = None if bias is None else _dev(bias, "bias", feats.dtype, (O,))
    if out is None:
        out = torch.empty((N, O), dtype=feats.dtype, device=feats.device)
    po = _dev(out, "out", feats.dtype, (N, O))
    _check(lib().subm3d_forward(pf, pn, pw, pb, po, N, I, O, _DTYPES[feats.dtype],
                                _stream(stream)))
    return out


def subm3d_forward_ex(feats: torch.Tensor, nbr: torch.Tensor, weight: torch.Tensor,
                      bias: torch.Tensor | None = None, residual: torch.Tensor | None = None,
                      act: str = "none", out: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """out [N, O] = act(convolution + bias + residual), the fused block epilogue.

    residual [N, O] of feats' dtype or None; it may be `out` itself (in place).
    act is "none", "relu" or "silu"."""
    if feats.dtype not in _DTYPES:
        raise ValueError(f"feats dtype {feats.dtype} is not float32 or bfloat16")
    if act not in ACTIVATIONS:
        raise ValueError(f"act {act!r} is not one of {sorted(ACTIVATIONS)}")
    N, I = feats.shape
    O = weight.shape[0]
    pf = _dev(feats, "feats")
    pn = _dev(nbr, "nbr", torch.int32, (N, 27))
    pw = _dev(weight, "weight", feats.dtype, (O, 3, 3, 3, I))
    pb = None if bias is None else _dev(bias, "bias", feats.dtype, (O,))
    pr = None if residual is None else _dev(residual, "residual", feats.dtype, (N, O))
    if out is None:
        out = torch.empty((N, O), dtype=feats.dtype, device=feats.device)
    po = _dev(out, "out", feats.dtype, (N, O))
    _check(lib().subm3d_forward_ex(pf, pn, pw, pb, pr, ACTIVATIONS[act], po, N, I, O,
                                   _DTYPES[feats.dtype], _stream(stream)))
    return out


def subm3d_downsample(coords: torch.Tensor, res: int, feats: torch.Tensor | None = None,
                      mode: str = "mean", workspace: torch.Tensor | None = None, stream=None,
                      order: torch.Tensor | None = None, async_: bool = False, out=None):
    """SparseDownsample(2): (coarse_coords int32 [M, 4], coarse_feats [M, C] or None,
    parent int32 [N], child_mask uint8 [M]) for coords int32 [N, 4] (b, z, y, x) on a
    grid of side res. Coarse voxels come in (batch, Morton) order; parent and
    child_mask are the subdivision subm3d_upsample takes. Synchronises the stream once.
    order: the Morton order subm3d_build_kmap_ex gave for the same coords (int32 [N]);
    when given, the radix sort is skipped (subm3d_downsample_sorted).
    async_: subm3d_downsample_async -- no wait; returns (coarse_coords [N, 4],
    coarse_feats [N, C] or None, parent [N], child_mask [N], M) with M an int64 device
    tensor of one element and only the first M rows of the coarse outputs written.
    out: that tuple from an earlier call of the same N and C, to write into again."""
    if mode not in POOL_MODES:
        raise ValueError(f"mode {mode!r} is not one of {sorted(POOL_MODES)}")
    N = coords.shape[0]
    dev = coords.device
    pc = _dev(coords, "coords", torch.int32, (N, 4))
    C, dt, pf, cf, pcf = 0, F32, None, None, None
    if feats is not None:
        if feats.dtype not in _DTYPES:
            raise ValueError(f"feats dtype {feats.dtype} is not float32 or bfloat16")
        C = feats.shape[1]
        dt = _DTYPES[feats.dtype]
        pf = _dev(feats, "feats", feats.dtype, (N, C))
    if out is not None:
        cc, cf, parent, mask, m_dev = out
    else:
        cf = None if feats is None else torch.empty((N, C), dtype=feats.dtype, device=dev)
        cc = torch.empty((N, 4), dtype=torch.int32, device=dev)
        parent = torch.empty(N, dtype=torch.int32, device=dev)
        mask = torch.empty(N, dtype=torch.uint8, device=dev)
        m_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    if cf is not None:
        pcf = _dev(cf, "coarse_feats", feats.dtype, (N, C))
    need = lib().subm3d_downsample_workspace_bytes(N)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    pw = _dev(workspace, "workspace", torch.uint8)
    if async_:
        po = None if order is None else _dev(order, "order", torch.int32, (N,))
        _check(lib().subm3d_downsample_async(pc, N, int(res), po, pf, C, dt, POOL_MODES[mode],
                                             _dev(cc, "cc", torch.int32, (N, 4)), pcf,
                                             _dev(parent, "parent", torch.int32, (N,)),
                                             _dev(mask, "mask", torch.uint8, (N,)),
                                             _dev(m_dev, "M", torch.int64, (1,)), pw,
                                             workspace.numel(), _stream(stream)))
        return cc, cf, parent, mask, m_dev
    M = ctypes.c_int64(0)
    if order is None:
        _check(lib().subm3d_downsample(pc, N, int(res), pf, C, dt, POOL_MODES[mode],
                                       _dev(cc, "cc"), pcf, _dev(parent, "parent"),
                                       _dev(mask, "mask"), ctypes.byref(M), pw, workspace.numel(),
                                       _stream(stream)))
    else:
        po = _dev(order, "order", torch.int32, (N,))
        _check(lib().subm3d_downsample_sorted(pc, N, int(res), po, pf, C, dt, POOL_MODES[mode],
                                              _dev(cc, "cc"), pcf, _dev(parent, "parent"),
                                              _dev(mask, "mask"), ctypes.byref(M), pw,
                                              workspace.numel(), _stream(stream)))
    m = M.value
    return cc[:m], (None if cf is None else cf[:m]), parent, mask[:m]


def subm3d_upsample(coarse_feats: torch.Tensor, parent: torch.Tensor,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """SparseUpsample(2) with a stored subdivision: out [N, C] with out[i] =
    coarse_feats[parent[i]] (parent from subm3d_downsample)."""
    if coarse_feats.dtype not in _DTYPES:
        raise ValueError(f"coarse_feats dtype {coarse_feats.dtype} is not float32 or bfloat16")
    M, C = coarse_feats.shape
    N = parent.shape[0]
    pcf = _dev(coarse_feats, "coarse_feats")
    pp = _dev(parent, "parent", torch.int32, (N,))
    if out is None:
        out = torch.empty((N, C), dtype=coarse_feats.dtype, device=coarse_feats.device)
    po = _dev(out, "out", coarse_feats.dtype, (N, C))
    _check(lib().subm3d_upsample(pcf, M, C, pp, N, _DTYPES[coarse_feats.dtype], po,
                                 _stream(stream)))
    return out


def subm3d_spatial2channel(feats: torch.Tensor, coords: torch.Tensor, parent: torch.Tensor,
                           child_mask: torch.Tensor, out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """SparseSpatial2Channel(2): out [M, 8C], the eight children's rows of each parent side
    by side in child-bit order (zeros for absent children); parent and child_mask from
    subm3d_downsample on the same coords."""
    if feats.dtype not in _DTYPES:
        raise ValueError(f"feats dtype {feats.dtype} is not float32 or bfloat16")
    N, C = feats.shape
    M = child_mask.shape[0]
    pf = _dev(feats, "feats")
    pc = _dev(coords, "coords", torch.int32, (N, 4))
    pp = _dev(parent, "parent", torch.int32, (N,))
    pm = _dev(child_mask, "child_mask", torch.uint8, (M,))
    if out is None:
        out = torch.empty((M, 8 * C), dtype=feats.dtype, device=feats.device)
    po = _dev(out, "out", feats.dtype, (M, 8 * C))
    _check(lib().subm3d_spatial2channel(pf, pc, pp, pm, N, M, C, _DTYPES[feats.dtype], po,
                                        _stream(stream)))
    return out


def subm3d_channel2spatial(coarse_feats: torch.Tensor, coords: torch.Tensor, parent: torch.Tensor,
                           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The inverse: out [N, C] with out[i] = the C-wide block of coarse_feats[parent[i]] at
    fine voxel i's child bit."""
    if coarse_feats.dtype not in _DTYPES:
        raise ValueError(f"coarse_feats dtype {coarse_feats.dtype} is not float32 or bfloat16")
    M, C8 = coarse_feats.shape
    if C8 % 8:
        raise ValueError(f"coarse_feats has {C8} channels, not a multiple of 8")
    C = C8 // 8
    N = parent.shape[0]
    pcf = _dev(coarse_feats, "coarse_feats")
    pc = _dev(coords, "coords", torch.int32, (N, 4))
    pp = _dev(parent, "parent", torch.int32, (N,))
    if out is None:
        out = torch.empty((N, C), dtype=coarse_feats.dtype, device=coarse_feats.device)
    po = _dev(out, "out", coarse_feats.dtype, (N, C))
    _check(lib().subm3d_channel2spatial(pcf, pc, pp, N, M, C, _DTYPES[coarse_feats.dtype], po,
                                        _stream(stream)))
    return out


def subm3d_kmap_stage_timing(enable: bool) -> None:
    """Turns the per-stage event recording of kernel-map builds on or off (this thread)."""
    lib().subm3d_kmap_stage_timing(1 if enable else 0)


def subm3d_kmap_stage_times() -> list:
    """[(stage name, GPU ms)] of this thread's last kernel-map build made with stage
    timing on (waits for its events)."""
    ms = (ctypes.c_float * 40)()
    names = (ctypes.c_char_p * 40)()
    n = lib().subm3d_kmap_stage_times(ms, names, 40)
    if n < 0:
        _check(n)
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


def subm3d_forward_status(stream=None) -> None:
    """Waits for the stream and raises Subm3dError if a forward kernel recorded an error."""
    _check(lib().subm3d_forward_status(_stream(stream)))
