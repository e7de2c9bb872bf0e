"""Occupancy-grouped tiles on the GPU: the tile plan bit-exact against the oracle's
(ref.tile_plan: windows of the Morton order sorted by neighbour mask), and the grouped
forward against the oracle on every output row -- and equal in value to the plain
forward, which accumulates the same present offsets in the same order. Also the
asynchronous kernel-map builds and their errors, reported by subm3d_forward_status."""
import numpy as np
import pytest
import torch

from oracle import cpu, ref
from submanifold_sparse_convolution_04_b300 import (GROUP_WINDOW, Subm3dError, plan_views,
                                                    subm3d_build_kmap, subm3d_build_kmap_async,
                                                    subm3d_build_kmap_grouped, subm3d_forward,
                                                    subm3d_forward_ex, subm3d_forward_grouped,
                                                    subm3d_forward_status, subm3d_plan_bytes)
from submanifold_sparse_convolution_04_b300 import _binding as B
from synth import make_residual, make_values
from tests.conftest import cached_case
from tests.gpu_util import assert_close, bf16_tensor, require_gpu, to_device
from tests.test_forward_gpu import multi_tile_case, shell_case
from tests.test_kmap_gpu import random_set

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def gpu_plan(coords, res, dev, window=0, **kw):
    c = torch.from_numpy(np.ascontiguousarray(coords, np.int32)).to(dev)
    plan = subm3d_build_kmap_grouped(c, res, window=window, **kw)
    return plan


def check_plan(plan, coords, res, window, nbr=None):
    N = coords.shape[0]
    perm, pnbr, tmask = (t.cpu().numpy() for t in plan_views(plan, N))
    if nbr is None:
        nbr = cpu.kernel_map(coords, res)
    want_perm, want_nbr, want_mask = ref.tile_plan(coords, nbr, window or GROUP_WINDOW)
    np.testing.assert_array_equal(perm, want_perm)
    np.testing.assert_array_equal(pnbr, want_nbr)
    np.testing.assert_array_equal(tmask.view(np.uint32), want_mask | (1 << 13))


@pytest.mark.parametrize("cfg_id", [1, 2, 3, 4, 5])
def test_plan_bit_exact_on_workloads(dev, cfg_id):
    case = cached_case(cfg_id)
    plan = gpu_plan(case["coords"], case["res"], dev)
    check_plan(plan, case["coords"], case["res"], 0)


@pytest.mark.parametrize("cfg_id,window", [(3, 128), (3, 4096), (4, 1 << 30), (5, 1 << 16),
                                           (2, 256), (5, 1), (3, 1), (4, 2), (1, 1)])
def test_plan_bit_exact_other_windows(dev, cfg_id, window):
    case = cached_case(cfg_id)
    plan = gpu_plan(case["coords"], case["res"], dev, window=window)
    check_plan(plan, case["coords"], case["res"], window)


def test_plan_bit_exact_shuffled_and_random_sets(dev):
    case = cached_case(4, "shuffled")
    check_plan(gpu_plan(case["coords"], case["res"], dev), case["coords"], case["res"], 0)
    for seed, res, batch, n in [(0, 4, 1, 1), (2, 5, 3, 70), (3, 8, 2, 500), (6, 1, 5, 1),
                                (7, 17, 7, 333), (5, 31, 1, 4000)]:
        c = random_set(np.random.default_rng(seed), res, batch, n)
        for window in (128, 1):
            check_plan(gpu_plan(c, res, dev, window=window), c, res, window, ref.kernel_map(c, res))


def run_both(coords, res, v, dtype, dev, residual=None, act="none", window=0):
    mk = (lambda a: bf16_tensor(a, dev)) if dtype == "bf16" else (lambda a: torch.from_numpy(a).to(dev))
    c = torch.from_numpy(coords).to(dev)
    f, w, b = mk(v["feats"]), mk(v["weight"]), mk(v["bias"])
    r = None if residual is None else mk(residual)
    plan = subm3d_build_kmap_grouped(c, res, window=window)
    out_g = subm3d_forward_grouped(f, plan, w, b, residual=r, act=act)
    nbr = subm3d_build_kmap(c, res)
    out_p = subm3d_forward_ex(f, nbr, w, b, residual=r, act=act)
    subm3d_forward_status()
    return out_g, out_p


@pytest.mark.parametrize("cfg_id,window", [(1, 0), (2, 0), (3, 0), (4, 0), (5, 0), (2, 1),
                                           (3, 1), (5, 1)])
def test_grouped_forward_every_row(dev, cfg_id, window):
    # window 0: mask-grouped tiles (staged row copies in the narrow kernel); window 1: the
    # Morton order (per-thread row loads)
    case = cached_case(cfg_id)
    out_g, out_p = run_both(case["coords"], case["res"], case, case["dtype"], dev, window=window)
    # the same present offsets, in the same order: equal values (signed zeros aside)
    assert bool((out_g == out_p).all())
    want = cpu.forward_rows(case["coords"], case["feats"], case["weight"], case["bias"],
                            case["res"])
    assert_close(out_g.float().cpu().numpy(), want, case["dtype"], case["name"])


@pytest.mark.parametrize("I,O,dtype", [(64, 64, "bf16"), (16, 16, "bf16"), (48, 32, "bf16"),
                                       (128, 128, "bf16"), (96, 256, "bf16"), (64, 264, "bf16"),
                                       (32, 32, "f32")])
def test_grouped_forward_several_tiles_per_cta(dev, I, O, dtype):
    coords, v = multi_tile_case(I * 3 + O + 1, I, O, dtype)
    want = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 256)
    for window in (0, 1):
        out_g, out_p = run_both(coords, 256, v, dtype, dev, window=window)
        assert bool((out_g == out_p).all())
        assert_close(out_g.float().cpu().numpy(), want, dtype, f"window {window} I={I} O={O}")


@pytest.mark.parametrize("I,O,act", [(64, 64, "relu"), (128, 128, "silu"), (32, 32, "none")])
def test_grouped_forward_epilogue(dev, I, O, act):
    coords, v = shell_case(I + 2 * O, 48, I, O, "bf16", batch=2)
    N = coords.shape[0]
    r_np, _ = make_residual(N, O, "bf16", 9)
    out_g, out_p = run_both(coords, 48, v, "bf16", dev, residual=r_np, act=act)
    assert bool((out_g == out_p).all())
    conv = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 48)
    assert_close(out_g.float().cpu().numpy(), ref.block_epilogue(conv, r_np, act), "bf16", act)


def test_grouped_forward_in_place_residual(dev):
    coords, v = shell_case(21, 40, 64, 64, "bf16", batch=2)
    N = coords.shape[0]
    r_np, _ = make_residual(N, 64, "bf16", 4)
    c = torch.from_numpy(coords).to(dev)
    plan = subm3d_build_kmap_grouped(c, 40)
    buf = bf16_tensor(r_np, dev)
    subm3d_forward_grouped(bf16_tensor(v["feats"], dev), plan, bf16_tensor(v["weight"], dev),
                           bf16_tensor(v["bias"], dev), residual=buf, act="relu", out=buf)
    subm3d_forward_status()
    conv = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 40)
    assert_close(buf.float().cpu().numpy(), ref.block_epilogue(conv, r_np, "relu"), "bf16", "in place")


def test_grouped_empty_and_tiny(dev):
    c = torch.zeros((0, 4), dtype=torch.int32, device=dev)
    plan = subm3d_build_kmap_grouped(c, 8)
    f = torch.zeros((0, 64), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((64, 3, 3, 3, 64), dtype=torch.bfloat16, device=dev)
    assert subm3d_forward_grouped(f, plan, w).shape == (0, 64)
    coords = np.array([[0, 1, 1, 1], [0, 5, 5, 5], [1, 1, 1, 1]], np.int32)
    v = make_values(3, 64, 64, "bf16", 5)
    out_g, _ = run_both(coords, 8, v, "bf16", dev)
    want = v["feats"].astype(np.float64) @ v["weight"][:, 1, 1, 1, :].astype(np.float64).T + v["bias"]
    assert_close(out_g.float().cpu().numpy(), want, "bf16", "isolated")


def test_async_kmap_matches_and_reports_errors(dev):
    case = cached_case(4)
    c = torch.from_numpy(case["coords"]).to(dev)
    nbr = subm3d_build_kmap_async(c, case["res"])
    subm3d_forward_status()
    np.testing.assert_array_equal(nbr.cpu().numpy(), cpu.kernel_map(case["coords"], case["res"]))
    plan = subm3d_build_kmap_grouped(c, case["res"], async_=True)
    subm3d_forward_status()
    check_plan(plan, case["coords"], case["res"], 0)
    # a duplicate: the build returns OK, the status call reports it, then the word is clear
    dup = np.concatenate([case["coords"][:5000], case["coords"][17:18]])
    d = torch.from_numpy(dup).to(dev)
    for build in (lambda: subm3d_build_kmap_async(d, case["res"]),
                  lambda: subm3d_build_kmap_grouped(d, case["res"], async_=True)):
        build()
        with pytest.raises(Subm3dError) as e:
            subm3d_forward_status()
        assert e.value.code == B.ERR_DUPLICATE
        subm3d_forward_status()
    bad = case["coords"][:1000].copy()
    bad[10, 2] = case["res"]
    subm3d_build_kmap_async(torch.from_numpy(bad).to(dev), case["res"])
    with pytest.raises(Subm3dError) as e:
        subm3d_forward_status()
    assert e.value.code == B.ERR_COORD_RANGE
    subm3d_forward_status()


def test_grouped_sync_errors(dev):
    case = cached_case(2)
    dup = np.concatenate([case["coords"], case["coords"][3:4]])
    with pytest.raises(Subm3dError) as e:
        subm3d_build_kmap_grouped(torch.from_numpy(dup).to(dev), case["res"])
    assert e.value.code == B.ERR_DUPLICATE
    c = torch.from_numpy(case["coords"]).to(dev)
    with pytest.raises(Subm3dError):
        subm3d_build_kmap_grouped(c, case["res"], window=100)          # not a power of two
    with pytest.raises(Subm3dError):
        subm3d_build_kmap_grouped(c, case["res"], window=-4)
    small = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(Subm3dError):
        subm3d_build_kmap_grouped(c, case["res"], plan=small)
    # recovery: a good build right after
    check_plan(subm3d_build_kmap_grouped(c, case["res"]), case["coords"], case["res"], 0)


def test_grouped_forward_reports_a_bad_plan_row(dev):
    coords, v = shell_case(13, 24, 32, 32, "bf16")
    N = coords.shape[0]
    c = torch.from_numpy(coords).to(dev)
    plan = subm3d_build_kmap_grouped(c, 24)
    perm, _, _ = plan_views(plan, N)
    good_row = int(perm[5].item())
    perm[5] = N + 7
    out = torch.zeros((N, 32), dtype=torch.bfloat16, device=dev)
    subm3d_forward_grouped(bf16_tensor(v["feats"], dev), plan, bf16_tensor(v["weight"], dev),
                           bf16_tensor(v["bias"], dev), out=out)
    with pytest.raises(Subm3dError) as e:
        subm3d_forward_status()
    assert e.value.code == B.ERR_DEVICE
    subm3d_forward_status()
    assert bool((out[good_row] == 0).all())          # the skipped row was not written
    want = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 24)
    keep = np.ones(N, bool)
    keep[good_row] = False
    assert_close(out.float().cpu().numpy()[keep], want[keep], "bf16", "other rows")
