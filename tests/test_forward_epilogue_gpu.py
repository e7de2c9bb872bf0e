"""Fused block epilogue (subm3d_forward_ex: out = act(conv + bias + residual)) on the GPU
against the CPU oracle (convolution rows in float64, then the oracle's block_epilogue),
for every forward kernel: the narrow tensor-memory kernel (I, O in {16..64}), the
shared-memory tcgen05 kernel (other O <= 256), the CUDA-core kernel (bf16 O > 256 and
fp32). Same tolerances as the plain forward."""
import numpy as np
import pytest
import torch

from oracle import cpu, ref
from submanifold_sparse_convolution_04_b300 import (Subm3dError, subm3d_build_kmap,
                                                    subm3d_forward, subm3d_forward_ex,
                                                    subm3d_forward_status)
from submanifold_sparse_convolution_04_b300 import _binding as B
from synth import make_residual
from tests.conftest import cached_case
from tests.gpu_util import assert_close, bf16_tensor, require_gpu, to_device
from tests.test_forward_gpu import sample_rows, shell_case

pytestmark = pytest.mark.gpu

# (I, O, dtype): which kernel runs is fixed by the shape (see subm3d.h)
SHAPES = [(64, 64, "bf16"), (32, 48, "bf16"),      # narrow tensor-memory kernel
          (128, 96, "bf16"), (72, 136, "bf16"),    # shared-memory tcgen05 kernel
          (16, 264, "bf16"),                       # CUDA-core kernel, bf16
          (32, 32, "f32"), (3, 5, "f32")]          # CUDA-core kernel, fp32
MODES = [("none", "separate"), ("relu", None), ("relu", "inplace"), ("silu", "separate"),
         ("silu", "inplace")]


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _tensor(a, dtype, dev):
    return bf16_tensor(a, dev) if dtype == "bf16" else torch.from_numpy(np.ascontiguousarray(a)).to(dev)


@pytest.mark.parametrize("act,rmode", MODES)
@pytest.mark.parametrize("I,O,dtype", SHAPES)
def test_epilogue_every_kernel(dev, I, O, dtype, act, rmode):
    coords, v = shell_case(I * 5 + O, 36, I, O, dtype, batch=2)
    N = coords.shape[0]
    assert N % 128 != 0 and N % 32 != 0
    nbr = subm3d_build_kmap(torch.from_numpy(coords).to(dev), 36)
    f, w, b = (_tensor(v[k], dtype, dev) for k in ("feats", "weight", "bias"))
    r_np = None
    r = out = None
    if rmode is not None:
        r_np, _ = make_residual(N, O, dtype, I + O)
        r = _tensor(r_np, dtype, dev)
        if rmode == "inplace":
            out = r          # the residual buffer is overwritten with the result
    got = subm3d_forward_ex(f, nbr, w, b, residual=r, act=act, out=out)
    subm3d_forward_status()
    if rmode == "inplace":
        assert got.data_ptr() == r.data_ptr()
    conv = cpu.forward_rows(coords, v["feats"], v["weight"], v["bias"], 36)
    want = ref.block_epilogue(conv, r_np, act)
    assert_close(got.float().cpu().numpy(), want, dtype, f"I={I} O={O} {act} {rmode}")


@pytest.mark.parametrize("I,O,dtype", [(64, 64, "bf16"), (128, 128, "bf16"), (32, 32, "f32")])
def test_epilogue_none_equals_plain_forward_bitwise(dev, I, O, dtype):
    """act none and no residual is the plain forward, bit for bit (same kernel, same sums)."""
    coords, v = shell_case(3 * I + O, 30, I, O, dtype)
    nbr = subm3d_build_kmap(torch.from_numpy(coords).to(dev), 30)
    f, w, b = (_tensor(v[k], dtype, dev) for k in ("feats", "weight", "bias"))
    o1 = subm3d_forward(f, nbr, w, b)
    o2 = subm3d_forward_ex(f, nbr, w, b, residual=None, act="none")
    subm3d_forward_status()
    assert torch.equal(o1, o2)


def test_epilogue_shares_one_kernel_map_across_convolutions(dev):
    """Two convolutions of a residual block at one resolution on one nbr:
    h = relu(conv1(x)), y = conv2(h) + x (the plain reading of a ResBlock tail)."""
    coords, v1 = shell_case(101, 32, 64, 64, "bf16", batch=2)
    N = coords.shape[0]
    _, v2 = shell_case(101, 32, 64, 64, "bf16", batch=2)
    w2 = np.asarray(v2["weight"])[::-1].copy()   # a different weight, still bf16-exact
    nbr = subm3d_build_kmap(torch.from_numpy(coords).to(dev), 32)
    x = bf16_tensor(v1["feats"], dev)
    h = subm3d_forward_ex(x, nbr, bf16_tensor(v1["weight"], dev), bf16_tensor(v1["bias"], dev),
                          act="relu")
    y = subm3d_forward_ex(h, nbr, bf16_tensor(w2, dev), None, residual=x)
    subm3d_forward_status()
    h_got = h.float().cpu().numpy()
    h_want = ref.block_epilogue(cpu.forward_rows(coords, v1["feats"], v1["weight"], v1["bias"], 32),
                                None, "relu")
    assert_close(h_got, h_want, "bf16", "conv1 + relu")
    # the second convolution consumes the GPU's bf16 h (exact values), as a user's would
    y_want = ref.block_epilogue(cpu.forward_rows(coords, h_got, w2, None, 32), v1["feats"], "none")
    assert_close(y.float().cpu().numpy(), y_want, "bf16", "conv2 + skip")
    assert N == h.shape[0]


def test_epilogue_full_workload_every_row(dev):
    """The 1024^3 workload in the launch configuration the benchmark times with
    --residual --act relu, on every row."""
    case = cached_case(5)
    N = case["coords"].shape[0]
    c, f, w, b = to_device(case, dev)
    r_np, _ = make_residual(N, case["O"], case["dtype"], 5)
    r = bf16_tensor(r_np, dev)
    nbr = subm3d_build_kmap(c, case["res"])
    out = subm3d_forward_ex(f, nbr, w, b, residual=r, act="relu")
    subm3d_forward_status()
    conv = cpu.forward_rows(case["coords"], case["feats"], case["weight"], case["bias"],
                            case["res"])
    want = ref.block_epilogue(conv, r_np, "relu")
    assert_close(out.float().cpu().numpy(), want, "bf16", "1024^3 residual + relu")


def test_epilogue_argument_errors(dev):
    coords, v = shell_case(3, 20, 16, 16, "bf16")
    N = coords.shape[0]
    nbr = subm3d_build_kmap(torch.from_numpy(coords).to(dev), 20)
    f, w = bf16_tensor(v["feats"], dev), bf16_tensor(v["weight"], dev)
    with pytest.raises(ValueError):
        subm3d_forward_ex(f, nbr, w, act="gelu")
    with pytest.raises(ValueError):     # residual shape is checked by the binding
        subm3d_forward_ex(f, nbr, w, residual=torch.zeros((N, 8), dtype=torch.bfloat16, device=dev))
    # the C ABI rejects an unknown activation code and a partial overlap with out
    buf = torch.zeros(N * 16 + 8, dtype=torch.bfloat16, device=dev)
    out = buf[:N * 16]
    res = buf[8:]
    rc = B.lib().subm3d_forward_ex(f.data_ptr(), nbr.data_ptr(), w.data_ptr(), None,
                                   res.data_ptr(), 0, out.data_ptr(), N, 16, 16, B.BF16, None)
    assert rc == B.ERR_ARG and b"overlaps" in B.lib().subm3d_last_error()
    rc = B.lib().subm3d_forward_ex(f.data_ptr(), nbr.data_ptr(), w.data_ptr(), None, None, 7,
                                   out.data_ptr(), N, 16, 16, B.BF16, None)
    assert rc == B.ERR_ARG and b"activation" in B.lib().subm3d_last_error()
    torch.cuda.synchronize()
    with pytest.raises(Subm3dError):
        B._check(-1)
