"""Kernel-level checks of the tensor-core projection GEMM against an exact float64 product
of the same bf16 inputs (the oracle's definition of a projection)."""
import numpy as np
import pytest
import torch

from block_diffusion_drafter_forward_gb300 import dflash_gemm_bf16
from synth.inputs import draw
from synth.torch_io import to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("N,K,M", [(128, 64, 16), (256, 512, 16), (5120, 2048, 16), (384, 128, 48),
                                   (1000, 256, 100), (2048, 6144, 512), (640, 4096, 272)])
def test_gemm_bf16_matches_exact_product(N, K, M):
    w = draw(7, f"w{N}_{K}", (N, K), 0.0, 0.02, "bf16")
    x = draw(8, f"x{M}_{K}", (M, K), 0.0, 1.0, "bf16")
    W, X = to_torch(w, "bf16"), to_torch(x, "bf16")
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    dflash_gemm_bf16(W.data_ptr(), N, K, X.data_ptr(), M, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = bf16_to_f64(x) @ bf16_to_f64(w).T
    got = out.double().cpu().numpy()
    # fp32 accumulation of K products: error well below 1e-5 of the output scale
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert np.isfinite(got).all() and err < 2e-5, err
