"""Forward pass on the GPU against the CPU oracle (float64), within max|err| <=
1e-4 max|ref| (fp32) and 2e-2 max|ref| (bf16; the tests also hold bf16 to a tighter
4e-3). Every workload, the full-size ones included, is compared on every output row,
in the same launch configuration the benchmark times; sets large enough that every
persistent CTA runs at least four tiles check the reuse of accumulators, stage slots
and neighbour-block buffers element by element on every kernel."""
import numpy as np
import pytest
import torch

from oracle import cpu, ref
from submanifold_sparse_convolution_04_b300 import (Subm3dError, subm3d_build_kmap,
                                                    subm3d_forward, subm3d_forward_status,
                                                    subm3d_kernel_launches)
from submanifold_sparse_convolution_04_b300 import _binding as B
from synth import ellipsoid_shell, make_values, union_coords, uniform_rotation
from tests.conftest import cached_case
from tests.gpu_util import assert_close, bf16_tensor, require_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def run(case, dev, rows=None):
    c, f, w, b = to_device(case, dev)
    nbr = subm3d_build_kmap(c, case["res"])
    out = subm3d_forward(f, nbr, w, b)
    subm3d_forward_status()
    out = out.float().cpu().numpy()
    return out if rows is None else out[rows]


def sample_rows(N, seed, n_random=1500):
    rng = np.random.default_rng(seed)
    edges = [r for t in range(0, N, 128) for r in (t, t + 127) if r < N][:400]
    tail = list(range(max(0, N - 300), N))
    rows = np.unique(np.concatenate([rng.integers(0, N, n_random), edges, tail]))
    return rows.astype(np.int64)


@pytest.mark.parametrize("cfg_id", [1, 2])
def test_forward_small_workloads_every_element(dev, cfg_id):
    case = cached_case(cfg_id)
    got = run(case, dev)
    want = ref.subm_conv3d(case["coords"], case["feats"], case["weight"], case["bias"], case["res"])
    assert_close(got, want, case["dtype"], case["name"])


@pytest.mark.parametrize("cfg_id", [3, 4, 5])
def test_forward_full_workloads_every_row(dev, cfg_id):
    case = cached_case(cfg_id)
    got = run(case, dev)
    want = cpu.forward_rows(case["coords"], case["feats"], case["weight"], case["bias"],
                            case["res"])
    assert_close(got, want, case["dtype"], case["name"])


def test_forward_shuffled_order(dev):
    case = cached_case(4, "shuffled")
    got = run(case, dev)
    want = cpu.forward_rows(case["coords"], case["feats"], case["weight"], case["bias"],
                            case["res"])
    assert_close(got, want, "bf16", "shuffled")


def multi_tile_case(seed, I, O, dtype, min_tiles_per_sm=4):
    """Shells on a 256^3 grid (two batch items) with at least 148 x 128 x min_tiles_per_sm
    voxels and a ragged last tile: every persistent CTA runs several tiles."""
    rng = np.random.default_rng(seed)
    res = 256
    need = 148 * 128 * min_tiles_per_sm
    parts = []
    coords = np.zeros((0, 4), np.int32)
    while coords.shape[0] < need or coords.shape[0] % 128 == 0:
        b = len(parts) % 2
        a = res * (0.18 + 0.12 * rng.random(3))
        parts.append((b, ellipsoid_shell(res, res / 2 + rng.random(3), a, uniform_rotation(rng))))
        coords = union_coords(parts, res)
    return coords, make_values(coords.shape[0], I, O, dtype, seed)


@pytest.mark.parametrize("I,O,dtype", [(64, 64, "bf16"), (32, 48, "bf16"), (16, 16, "bf16"),
                                       (128, 128, "bf16"), (96, 256, "bf16"), (64, 264, "bf16"),
                                       (32, 32, "f32")])
def test_forward_several_tiles_per_cta_every_row(dev, I, O, dtype):
    coords, v = multi_tile_case(I * 5 + O, I, O, dtype)
    N = coords.shape[0]
    assert N >= 148 * 128 * 4 and N % 128 != 0
    mk = (lambda a: bf16_tensor(a, dev)) if dtype == "bf16" else (lambda a: torch.from_numpy(a).to(dev))
    nbr = subm3d_build_kmap(torch.from_numpy(coords).to(dev), 256)
    out = subm3d_forward(mk(v["feats"]), nbr, mk(v["weight"]), mk(v["bias"]))
    subm3d_forward_status()
    want = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 256)
    assert_close(out.float().cpu().numpy(), want, dtype, f"N={N} I={I} O={O}")


def shell_case(seed, res, I, O, dtype, batch=1):
    rng = np.random.default_rng(seed)
    parts = []
    for b in range(batch):
        a = res * (0.2 + 0.15 * rng.random(3))
        parts.append((b, ellipsoid_shell(res, res / 2 + rng.random(3), a, uniform_rotation(rng))))
    coords = union_coords(parts, res)
    v = make_values(coords.shape[0], I, O, dtype, seed)
    return coords, v


@pytest.mark.parametrize("I,O", [(16, 16), (32, 64), (64, 32), (96, 96), (128, 256), (256, 128),
                                 (8, 8), (24, 40), (72, 136), (264, 48), (64, 256), (256, 256),
                                 (40, 264), (8, 520),
                                 # rows by TMA gathers (I a multiple of 64); above
                                 # O = 128 with the weight taps in a ring of their own
                                 (64, 128), (192, 80), (128, 16), (64, 72), (192, 144),
                                 (64, 208)])
def test_forward_bf16_shapes(dev, I, O):
    coords, v = shell_case(I * 7 + O, 40, I, O, "bf16", batch=2)
    N = coords.shape[0]
    assert N % 128 != 0
    c = torch.from_numpy(coords).to(dev)
    nbr = subm3d_build_kmap(c, 40)
    use_bias = (I + O) % 3 != 0
    out = subm3d_forward(bf16_tensor(v["feats"], dev), nbr, bf16_tensor(v["weight"], dev),
                         bf16_tensor(v["bias"], dev) if use_bias else None)
    subm3d_forward_status()
    rows = np.arange(N) if N * I * O < 3e8 else sample_rows(N, 1, 600)
    want = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"] if use_bias else None, 40,
                            rows=rows)
    assert_close(out.float().cpu().numpy()[rows], want, "bf16", f"I={I} O={O}")


@pytest.mark.parametrize("I,O", [(16, 48), (48, 16), (48, 48), (64, 64), (64, 16), (32, 32)])
def test_forward_narrow_kernel_shapes(dev, I, O):
    # I, O in {16, 32, 48, 64}: the kernel that keeps the gathered rows in tensor memory
    coords, v = shell_case(I * 11 + O * 3, 40, I, O, "bf16", batch=2)
    N = coords.shape[0]
    assert N % 128 != 0
    nbr = subm3d_build_kmap(torch.from_numpy(coords).to(dev), 40)
    out = subm3d_forward(bf16_tensor(v["feats"], dev), nbr, bf16_tensor(v["weight"], dev),
                         bf16_tensor(v["bias"], dev))
    subm3d_forward_status()
    want = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 40)
    assert_close(out.float().cpu().numpy(), want, "bf16", f"I={I} O={O}")


def test_forward_narrow_shape_with_16_byte_aligned_feats(dev):
    # a feats pointer that is 16-byte but not 32-byte aligned gives the same result
    coords, v = shell_case(77, 40, 64, 64, "bf16", batch=2)
    N = coords.shape[0]
    nbr = subm3d_build_kmap(torch.from_numpy(coords).to(dev), 40)
    f32b = bf16_tensor(v["feats"], dev)
    flat = torch.empty(N * 64 + 8, dtype=torch.bfloat16, device=dev)
    f16b = flat[8:].view(N, 64)
    f16b.copy_(f32b)
    assert f32b.data_ptr() % 32 == 0 and f16b.data_ptr() % 32 == 16
    w, b = bf16_tensor(v["weight"], dev), bf16_tensor(v["bias"], dev)
    o1 = subm3d_forward(f32b, nbr, w, b)
    o2 = subm3d_forward(f16b, nbr, w, b)
    subm3d_forward_status()
    want = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 40)
    assert_close(o1.float().cpu().numpy(), want, "bf16", "32-byte aligned")
    assert_close(o2.float().cpu().numpy(), want, "bf16", "16-byte aligned")


@pytest.mark.parametrize("I,O", [(32, 32), (16, 8), (3, 5), (64, 96), (1, 1), (130, 70)])
def test_forward_fp32_shapes(dev, I, O):
    coords, v = shell_case(I + 1000 * O, 24, I, O, "f32")
    c = torch.from_numpy(coords).to(dev)
    nbr = subm3d_build_kmap(c, 24)
    out = subm3d_forward(torch.from_numpy(v["feats"]).to(dev), nbr,
                         torch.from_numpy(v["weight"]).to(dev), torch.from_numpy(v["bias"]).to(dev))
    subm3d_forward_status()
    want = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 24)
    assert_close(out.cpu().numpy(), want, "f32", f"I={I} O={O}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_forward_tiny_and_isolated(dev, dtype):
    # N = 1, then a handful of isolated voxels: only the centre tap contributes
    for coords in (np.array([[0, 3, 3, 3]], np.int32),
                   np.array([[0, 1, 1, 1], [0, 5, 5, 5], [1, 1, 1, 1], [2, 9, 0, 9]], np.int32)):
        v = make_values(coords.shape[0], 64, 64, dtype, 5)
        mk = (lambda a: bf16_tensor(a, dev)) if dtype == "bf16" else (lambda a: torch.from_numpy(a).to(dev))
        nbr = subm3d_build_kmap(torch.from_numpy(coords).to(dev), 10)
        out = subm3d_forward(mk(v["feats"]), nbr, mk(v["weight"]), mk(v["bias"]))
        subm3d_forward_status()
        want = v["feats"].astype(np.float64) @ v["weight"][:, 1, 1, 1, :].astype(np.float64).T + v["bias"]
        assert_close(out.float().cpu().numpy(), want, dtype, "isolated")


def test_forward_empty(dev):
    f = torch.zeros((0, 64), dtype=torch.bfloat16, device=dev)
    nbr = torch.zeros((0, 27), dtype=torch.int32, device=dev)
    w = torch.zeros((64, 3, 3, 3, 64), dtype=torch.bfloat16, device=dev)
    assert subm3d_forward(f, nbr, w).shape == (0, 64)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_forward_invalid_nbr_is_reported_not_dereferenced(dev, dtype):
    coords, v = shell_case(9, 20, 32, 32, dtype)
    N = coords.shape[0]
    c = torch.from_numpy(coords).to(dev)
    nbr = subm3d_build_kmap(c, 20)
    bad = nbr.clone()
    bad[5, 0] = N + 1000
    bad[7, 26] = -7
    mk = (lambda a: bf16_tensor(a, dev)) if dtype == "bf16" else (lambda a: torch.from_numpy(a).to(dev))
    out = subm3d_forward(mk(v["feats"]), bad, mk(v["weight"]), mk(v["bias"]))
    with pytest.raises(Subm3dError) as e:
        subm3d_forward_status()
    assert e.value.code == B.ERR_DEVICE
    subm3d_forward_status()   # the word was cleared
    # the bad entries were treated as absent
    fixed = nbr.clone().cpu().numpy()
    fixed[5, 0] = -1
    fixed[7, 26] = -1
    o2 = subm3d_forward(mk(v["feats"]), torch.from_numpy(fixed).to(dev), mk(v["weight"]), mk(v["bias"]))
    subm3d_forward_status()
    assert torch.equal(out, o2)


def test_forward_is_deterministic_and_counts_launches(dev):
    case = cached_case(2)
    c, f, w, b = to_device(case, dev)
    nbr = subm3d_build_kmap(c, case["res"])
    n0 = subm3d_kernel_launches()
    o1 = subm3d_forward(f, nbr, w, b)
    o2 = subm3d_forward(f, nbr, w, b)
    subm3d_forward_status()
    assert subm3d_kernel_launches() - n0 == 2
    assert torch.equal(o1, o2)


def test_forward_on_side_stream(dev):
    case = cached_case(2)
    c, f, w, b = to_device(case, dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        nbr = subm3d_build_kmap(c, case["res"])
        out = subm3d_forward(f, nbr, w, b)
    subm3d_forward_status(s)
    torch.cuda.synchronize()
    want = ref.subm_conv3d(case["coords"], case["feats"], case["weight"], case["bias"], case["res"])
    assert_close(out.float().cpu().numpy(), want, "bf16", "side stream")
