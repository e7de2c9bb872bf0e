"""SparseDownsample(2) / SparseUpsample(2) and SparseSpatial2Channel(2) /
channel2spatial on the GPU against the CPU oracle (oracle.ref): coarse coordinates,
parent rows and child masks bit-exact; pooled features within the forward's tolerances
(fp32 1e-4, bf16 2e-2 of max|ref|, bf16 also the tighter 4e-3); the pixel-(un)shuffle
pair moves values without arithmetic, so it is compared bit-exactly."""
import numpy as np
import pytest
import torch

from oracle import ref
from submanifold_sparse_convolution_04_b300 import (Subm3dError, subm3d_channel2spatial,
                                                    subm3d_downsample, subm3d_forward_status,
                                                    subm3d_spatial2channel, subm3d_upsample)
from submanifold_sparse_convolution_04_b300 import _binding as B
from synth import round_to_bf16
from tests.conftest import cached_case
from tests.gpu_util import assert_close, require_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def random_set(rng, res, batch, n):
    rows = []
    for b in range(batch):
        flat = rng.choice(res ** 3, size=min(n, res ** 3), replace=False)
        z, rem = np.divmod(flat, res * res)
        y, x = np.divmod(rem, res)
        rows.append(np.stack([np.full(len(flat), b), z, y, x], axis=1))
    c = np.concatenate(rows).astype(np.int32)
    return c[rng.permutation(c.shape[0])]


def values(rng, N, C, dtype):
    f = rng.standard_normal((N, C)).astype(np.float32)
    if dtype == "bf16":
        f, _ = round_to_bf16(f)
    return f


def as_tensor(a, dtype, dev):
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return (t.to(torch.bfloat16) if dtype == "bf16" else t).to(dev)


def check_structure(got, want):
    cc, _, parent, mask = got
    wc, _, wp, wm = want
    np.testing.assert_array_equal(cc.cpu().numpy(), wc)
    np.testing.assert_array_equal(parent.cpu().numpy(), wp)
    np.testing.assert_array_equal(mask.cpu().numpy(), wm)


@pytest.mark.parametrize("mode", ["mean", "max"])
@pytest.mark.parametrize("dtype,C", [("f32", 3), ("f32", 8), ("bf16", 64), ("bf16", 12)])
@pytest.mark.parametrize("seed,res,batch,n", [(0, 9, 2, 300), (1, 40, 3, 5000), (2, 1, 2, 1),
                                               (3, 2, 1, 8), (4, 129, 1, 7000)])
def test_downsample_matches_oracle(dev, mode, dtype, C, seed, res, batch, n):
    rng = np.random.default_rng(seed * 7 + C)
    c = random_set(rng, res, batch, n)
    f = values(rng, c.shape[0], C, dtype)
    got = subm3d_downsample(torch.from_numpy(c).to(dev), res, as_tensor(f, dtype, dev), mode)
    want = ref.downsample(c, f, res, mode)
    check_structure(got, want)
    assert_close(got[1].float().cpu().numpy(), want[1], dtype, f"{mode} {dtype} C={C}")


def test_downsample_structure_only_and_empty(dev):
    rng = np.random.default_rng(5)
    c = random_set(rng, 17, 2, 900)
    got = subm3d_downsample(torch.from_numpy(c).to(dev), 17)
    assert got[1] is None
    check_structure(got, ref.downsample(c, None, 17))
    e = subm3d_downsample(torch.zeros((0, 4), dtype=torch.int32, device=dev), 8,
                          torch.zeros((0, 16), dtype=torch.bfloat16, device=dev))
    assert e[0].shape == (0, 4) and e[1].shape == (0, 16) and e[2].shape == (0,)


@pytest.mark.parametrize("dtype,C", [("f32", 5), ("bf16", 64), ("bf16", 24)])
def test_upsample_matches_oracle(dev, dtype, C):
    rng = np.random.default_rng(C)
    c = random_set(rng, 24, 2, 3000)
    f = values(rng, c.shape[0], C, dtype)
    cc, cf, parent, mask = subm3d_downsample(torch.from_numpy(c).to(dev), 24,
                                             as_tensor(f, dtype, dev), "mean")
    up = subm3d_upsample(cf, parent)
    subm3d_forward_status()
    # the oracle upsamples the GPU's coarse rows (exact values) with the GPU's subdivision
    # (checked bit-exact above); the copy itself must be exact
    want = ref.upsample(cf.float().cpu().numpy(), parent.cpu().numpy())
    np.testing.assert_array_equal(up.float().cpu().numpy(), want)
    # and the whole round trip matches the oracle's
    _, wf, wp, _ = ref.downsample(c, f, 24, "mean")
    assert_close(up.float().cpu().numpy(), ref.upsample(wf, wp), dtype, "round trip")


def test_upsample_bad_parent_is_reported(dev):
    cf = torch.ones((4, 8), dtype=torch.bfloat16, device=dev)
    parent = torch.tensor([0, 3, 4, -1, 2], dtype=torch.int32, device=dev)
    up = subm3d_upsample(cf, parent)
    with pytest.raises(Subm3dError) as e:
        subm3d_forward_status()
    assert e.value.code == B.ERR_DEVICE and "parent" in str(e.value)
    subm3d_forward_status()   # cleared
    np.testing.assert_array_equal(up.float().cpu().numpy()[:, 0], [1, 1, 0, 0, 1])


def test_downsample_errors(dev):
    dup = torch.tensor([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=torch.int32, device=dev)
    with pytest.raises(Subm3dError) as e:
        subm3d_downsample(dup, 4)
    assert e.value.code == B.ERR_DUPLICATE
    out = torch.tensor([[0, 1, 1, 1], [0, 4, 0, 0]], dtype=torch.int32, device=dev)
    with pytest.raises(Subm3dError) as e:
        subm3d_downsample(out, 4)
    assert e.value.code == B.ERR_COORD_RANGE
    with pytest.raises(ValueError):
        subm3d_downsample(out, 4, mode="sum")
    ok = torch.tensor([[0, 1, 1, 1], [0, 2, 2, 2]], dtype=torch.int32, device=dev)
    with pytest.raises(Subm3dError) as e:
        subm3d_downsample(ok, 4, workspace=torch.empty(256, dtype=torch.uint8, device=dev))
    assert e.value.code == B.ERR_WORKSPACE
    # the library recovers: a valid call after the failures
    got = subm3d_downsample(ok, 4)
    check_structure(got, ref.downsample(ok.cpu().numpy(), None, 4))


def _morton(co):
    m = np.zeros(len(co), np.int64)
    for t in range(16):
        m |= ((co[:, 3] >> t) & 1) << (3 * t)
        m |= ((co[:, 2] >> t) & 1) << (3 * t + 1)
        m |= ((co[:, 1] >> t) & 1) << (3 * t + 2)
    return m


@pytest.mark.parametrize("mode", ["mean", "max"])
def test_downsample_full_workload(dev, mode):
    """The 1024^3 workload (2.9 M voxels, C = 64, bf16), as the benchmark runs it: the
    structure checked on every row through properties that fix it (parent cells, masks,
    distinct parents in (batch, Morton) order), the pooled rows of sampled parents
    against the oracle on their children."""
    case = cached_case(5)
    co = case["coords"]
    N = co.shape[0]
    c, f, _, _ = to_device(case, dev)
    cc, cf, parent, mask = subm3d_downsample(c, case["res"], f, mode)
    cc, parent, mask = cc.cpu().numpy(), parent.cpu().numpy(), mask.cpu().numpy()
    M = cc.shape[0]
    assert 0 < M <= N
    np.testing.assert_array_equal(cc[parent, 0], co[:, 0])
    np.testing.assert_array_equal(cc[parent, 1:], co[:, 1:] >> 1)
    bit = ((co[:, 1] & 1) << 2) | ((co[:, 2] & 1) << 1) | (co[:, 3] & 1)
    want_mask = np.zeros(M, np.uint8)
    np.bitwise_or.at(want_mask, parent, (1 << bit).astype(np.uint8))
    np.testing.assert_array_equal(mask, want_mask)
    assert np.bincount(parent, minlength=M).min() >= 1          # no empty parent
    key = (cc[:, 0].astype(np.int64) << 48) | _morton(cc.astype(np.int64))
    assert (np.diff(key) > 0).all()                              # distinct, ascending
    rng = np.random.default_rng(7)
    sample = np.unique(np.concatenate([rng.integers(0, M, 400), [0, M - 1]]))
    rows = np.nonzero(np.isin(parent, sample))[0]
    sub = ref.downsample(co[rows], case["feats"][rows], case["res"], mode)
    # the oracle's parents of the sampled children are exactly the sampled parents, in order
    np.testing.assert_array_equal(sub[0], cc[sample])
    assert_close(cf[torch.from_numpy(sample).to(dev)].float().cpu().numpy(), sub[1], "bf16",
                 f"1024^3 {mode}")
    up = subm3d_upsample(cf, torch.from_numpy(parent).to(dev))
    subm3d_forward_status()
    np.testing.assert_array_equal(up[torch.from_numpy(rows).to(dev)].float().cpu().numpy(),
                                  cf.float().cpu().numpy()[parent[rows]])


@pytest.mark.parametrize("dtype,C", [("f32", 3), ("f32", 8), ("bf16", 64), ("bf16", 12)])
@pytest.mark.parametrize("seed,res,batch,n", [(0, 9, 2, 300), (1, 40, 3, 4000), (2, 1, 2, 1),
                                               (3, 2, 1, 8)])
def test_spatial2channel_matches_oracle(dev, dtype, C, seed, res, batch, n):
    rng = np.random.default_rng(seed * 11 + C)
    c = random_set(rng, res, batch, n)
    f = values(rng, c.shape[0], C, dtype)
    ct = torch.from_numpy(c).to(dev)
    ft = as_tensor(f, dtype, dev)
    _, _, parent, mask = subm3d_downsample(ct, res)
    out = subm3d_spatial2channel(ft, ct, parent, mask)
    back = subm3d_channel2spatial(out, ct, parent)
    subm3d_forward_status()
    want = ref.spatial2channel(c, f, res)
    np.testing.assert_array_equal(out.float().cpu().numpy(), want[1])
    np.testing.assert_array_equal(back.float().cpu().numpy(), f)


def test_spatial2channel_full_workload_and_bad_parent(dev):
    """The 1024^3 workload (2.9 M voxels, C = 64): the round trip is exact on every row,
    sampled parents' rows equal the oracle's on their children, and a bad parent entry is
    reported."""
    case = cached_case(5)
    co = case["coords"]
    c, f, _, _ = to_device(case, dev)
    cc, _, parent, mask = subm3d_downsample(c, case["res"])
    out = subm3d_spatial2channel(f, c, parent, mask)
    back = subm3d_channel2spatial(out, c, parent)
    subm3d_forward_status()
    assert torch.equal(back, f)
    M = cc.shape[0]
    p_np = parent.cpu().numpy()
    rng = np.random.default_rng(9)
    sample = np.unique(np.concatenate([rng.integers(0, M, 300), [0, M - 1]]))
    rows = np.nonzero(np.isin(p_np, sample))[0]
    sub = ref.spatial2channel(co[rows], case["feats"][rows], case["res"])
    np.testing.assert_array_equal(sub[0], cc.cpu().numpy()[sample])
    np.testing.assert_array_equal(out[torch.from_numpy(sample).to(dev)].float().cpu().numpy(),
                                  sub[1])
    bad = parent.clone()
    bad[3] = M
    fine = subm3d_channel2spatial(out, c, bad)
    with pytest.raises(Subm3dError) as e:
        subm3d_forward_status()
    assert e.value.code == B.ERR_DEVICE and "parent" in str(e.value)
    assert float(fine[3].float().abs().sum()) == 0.0
    assert torch.equal(fine[4:], f[4:])


@pytest.mark.parametrize("seed,res,batch,n,C", [(0, 9, 2, 300, 8), (1, 40, 3, 5000, 64),
                                                 (2, 1, 2, 1, 16), (4, 129, 1, 7000, 12)])
def test_downsample_on_the_kernel_maps_order(dev, seed, res, batch, n, C):
    # the Morton order the kernel map wrote for the same coords: the same result as the
    # downsample that sorts by itself, bit for bit (structure and pooled rows)
    from submanifold_sparse_convolution_04_b300 import subm3d_build_kmap_ex
    rng = np.random.default_rng(seed + 100)
    c = random_set(rng, res, batch, n)
    f = values(rng, c.shape[0], C, "bf16")
    ct, ft = torch.from_numpy(c).to(dev), as_tensor(f, "bf16", dev)
    _, order = subm3d_build_kmap_ex(ct, res, order=True)
    for mode in ("mean", "max"):
        got = subm3d_downsample(ct, res, ft, mode, order=order)
        plain = subm3d_downsample(ct, res, ft, mode)
        want = ref.downsample(c, f, res, mode)
        check_structure(got, want)
        assert torch.equal(got[1], plain[1])
        assert_close(got[1].float().cpu().numpy(), want[1], "bf16", f"sorted {mode}")


def test_downsample_on_order_full_workload_and_a_wrong_order(dev):
    from submanifold_sparse_convolution_04_b300 import subm3d_build_kmap_ex
    case = cached_case(5)
    c, f, _, _ = to_device(case, dev)
    _, order = subm3d_build_kmap_ex(c, case["res"], order=True)
    got = subm3d_downsample(c, case["res"], f, "mean", order=order)
    plain = subm3d_downsample(c, case["res"], f, "mean")
    for a, b in zip(got, plain):
        assert torch.equal(a, b)
    bad = order.clone()
    bad[[10, 11]] = bad[[11, 10]]           # two positions swapped: keys no longer ascend
    with pytest.raises(Subm3dError) as e:
        subm3d_downsample(c, case["res"], f, "mean", order=bad)
    assert e.value.code == B.ERR_ARG
    bad[10] = c.shape[0] + 5                 # a row outside [0, N)
    with pytest.raises(Subm3dError):
        subm3d_downsample(c, case["res"], f, "mean", order=bad)
    # recovery
    got2 = subm3d_downsample(c, case["res"], f, "mean", order=order)
    assert torch.equal(got2[1], plain[1])


def test_downsample_async_matches_and_reports_errors(dev):
    # the asynchronous downsample (M on the device, no wait): the same first M rows as the
    # synchronous call, with and without the kernel map's order; twice into one set of
    # outputs; device-side errors at the next status call, with M set to 0
    from submanifold_sparse_convolution_04_b300 import subm3d_build_kmap_ex
    case = cached_case(4)
    c, f, _, _ = to_device(case, dev)
    res = case["res"]
    want = subm3d_downsample(c, res, f, "mean")
    M = want[0].shape[0]
    _, order = subm3d_build_kmap_ex(c, res, order=True)
    out = None
    for o in (None, order, order):
        out = subm3d_downsample(c, res, f, "mean", order=o, async_=True, out=out)
        subm3d_forward_status()
        assert int(out[4].item()) == M
        for a, b in zip((out[0][:M], out[1][:M], out[2], out[3][:M]), want):
            assert torch.equal(a, b)
    dup = torch.cat([c[:3000], c[7:8]])
    d = subm3d_downsample(dup, res, async_=True)
    with pytest.raises(Subm3dError) as e:
        subm3d_forward_status()
    assert e.value.code == B.ERR_DUPLICATE
    assert int(d[4].item()) == 0
    bad = order.clone()
    bad[[10, 11]] = bad[[11, 10]]
    subm3d_downsample(c, res, f, "mean", order=bad, async_=True)
    with pytest.raises(Subm3dError) as e:
        subm3d_forward_status()
    assert e.value.code == B.ERR_ARG
    subm3d_forward_status()
