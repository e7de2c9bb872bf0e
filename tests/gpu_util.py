"""Helpers shared by the GPU parity tests."""
import numpy as np
import pytest
import torch

# Tolerances of the parity bar: max |err| <= TOL * max |ref|.
TOL = {"f32": 1e-4, "bf16": 2e-2}
# Tighter bound this implementation is held to for bf16 (output rounding is 2^-9
# relative; fp32 accumulation adds far less): catches small systematic errors.
TIGHT_BF16 = 4e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from submanifold_sparse_convolution_04_b300.build import build
    build()
    return torch.device("cuda:0")


def to_device(case, dev):
    """coords, feats, weight, bias as device tensors of the workload's dtype."""
    c = torch.from_numpy(case["coords"]).to(dev)
    if case["dtype"] == "bf16":
        f = torch.from_numpy(case["feats_bits"].view(np.int16)).view(torch.bfloat16).to(dev)
        w = torch.from_numpy(case["weight_bits"].view(np.int16)).view(torch.bfloat16).to(dev)
        b = torch.from_numpy(case["bias_bits"].view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        f = torch.from_numpy(case["feats"]).to(dev)
        w = torch.from_numpy(case["weight"]).to(dev)
        b = torch.from_numpy(case["bias"]).to(dev)
    return c, f, w, b


def bf16_tensor(x: np.ndarray, dev):
    """A float32 array (bf16-exact values) as a bf16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).to(dev)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    err = float(np.abs(got.astype(np.float64) - ref).max()) if ref.size else 0.0
    assert np.isfinite(got).all(), what
    assert err <= TOL[dtype] * max(scale, 1e-30), f"{what}: max err {err:.3e} vs max |ref| {scale:.3e}"
    if dtype == "bf16":
        assert err <= TIGHT_BF16 * max(scale, 1e-30), f"{what}: max err {err:.3e} (tight bound)"
    return err / max(scale, 1e-30)
