"""The allocation-free split-K GEMM entry point, for callers that cannot allocate device
memory while running.  Checked through the C ABI against the regular GEMM entry point
(same kernel without split-K) and against the exact float64 product of the same bf16
inputs, on two calls in a row so the shared fixed scratch is reused; and at the edge of
its fixed capacity.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from block_diffusion_drafter_forward_gb300 import _lib
from synth.inputs import draw
from synth.torch_io import to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _regular(W, X, N, K, M, st):
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    rc = _lib.load().dflash_gemm_bf16(ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_void_p(X.data_ptr()), M,
                                      ctypes.c_void_p(out.data_ptr()), 1, ctypes.c_void_p(st))
    assert rc == 0
    return out


def _noalloc(W, X, N, K, M, nsplit, st):
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    rc = _lib.load().dflash_gemm_bf16_noalloc(ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_void_p(X.data_ptr()),
                                              M, ctypes.c_void_p(out.data_ptr()), nsplit, ctypes.c_void_p(st))
    assert rc == 0
    return out


def _exact(W, X):
    """The float64 product of the same bf16 inputs (fp32 accumulation differs only by rounding)."""
    return X.double() @ W.double().t()


# (N, K, M, nsplit): one token tile, several token tiles of 128 (M > 128: more than one tile
# along the grid's token axis), no split at all, and a ragged weight-row tail
CASES = [(5120, 2048, 16, 4), (2048, 6144, 48, 8), (1000, 512, 100, 3), (1024, 2048, 300, 4),
         (1536, 1024, 64, 1)]


@pytest.mark.parametrize("N,K,M,nsplit", CASES)
def test_noalloc_split_k_matches_regular_gemm_twice(N, K, M, nsplit):
    """Two calls in a row (the fixed scratch is reused and its counters re-zeroed): each equal
    to the regular entry point and to the exact product of the same inputs."""
    st = torch.cuda.current_stream().cuda_stream
    W = to_torch(draw(31, f"na_w{N}_{K}", (N, K), 0.0, 0.02, "bf16"), "bf16")
    for call in range(2):
        X = to_torch(draw(32 + call, f"na_x{M}_{K}", (M, K), 0.0, 1.0, "bf16"), "bf16")
        ref = _regular(W, X, N, K, M, st)
        got = _noalloc(W, X, N, K, M, nsplit, st)
        torch.cuda.synchronize()
        ex = _exact(W, X)
        err = ((got - ref).abs().max() / ref.abs().max()).item()
        err_exact = ((got.double() - ex).abs().max() / ex.abs().max()).item()
        assert torch.isfinite(got).all() and err < 1e-5 and err_exact < 1e-5, (call, err, err_exact)


def test_noalloc_at_the_capacity_limit():
    """tiles * nsplit * 128 * TN == 2^21 floats is accepted and exact; one more weight row
    (one more tile) is rejected with ECAPACITY before anything runs."""
    st = torch.cuda.current_stream().cuda_stream
    N, K, M, ns = 256 * 128, 256, 16, 4          # 256 tiles x 4 splits x 128 x 16 = 2^21
    W = to_torch(draw(35, "na_cap_w", (N + 1, K), 0.0, 0.02, "bf16"), "bf16")
    X = to_torch(draw(36, "na_cap_x", (M, K), 0.0, 1.0, "bf16"), "bf16")
    got = _noalloc(W, X, N, K, M, ns, st)
    torch.cuda.synchronize()
    ex = _exact(W[:N], X)
    assert ((got.double() - ex).abs().max() / ex.abs().max()).item() < 1e-5
    out = torch.full((M, N + 1), 7.0, dtype=torch.float32, device="cuda")
    rc = _lib.load().dflash_gemm_bf16_noalloc(ctypes.c_void_p(W.data_ptr()), N + 1, K, ctypes.c_void_p(X.data_ptr()),
                                              M, ctypes.c_void_p(out.data_ptr()), ns, ctypes.c_void_p(st))
    torch.cuda.synchronize()
    assert rc == _lib.DFLASH_ECAPACITY
    assert bool((out == 7.0).all())


def test_noalloc_rejects_shapes_beyond_the_fixed_scratch():
    st = torch.cuda.current_stream().cuda_stream
    W = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    X = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((16, 128), dtype=torch.float32, device="cuda")
    lib = _lib.load()
    # 600 000 weight rows x 256 tokens x 2 splits needs far more than 8 MiB of partials
    big = lib.dflash_gemm_bf16_noalloc(ctypes.c_void_p(W.data_ptr()), 600000, 128, ctypes.c_void_p(X.data_ptr()),
                                       256, ctypes.c_void_p(out.data_ptr()), 2, ctypes.c_void_p(st))
    assert big == _lib.DFLASH_ECAPACITY
    assert lib.dflash_gemm_bf16_noalloc(ctypes.c_void_p(W.data_ptr()), 128, 64, ctypes.c_void_p(X.data_ptr()), 16,
                                        ctypes.c_void_p(out.data_ptr()), 2, ctypes.c_void_p(st)) == _lib.DFLASH_EINVAL
