"""Kernel-level checks of the tensor-core projection GEMM against an exact float64 product
of the same bf16 inputs (the oracle's definition of a projection)."""
import numpy as np
import pytest
import torch

from block_diffusion_drafter_forward_gb300 import dflash_attention_check, dflash_gemm_bf16
from synth import CONFIGS, make_workload
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


@pytest.mark.parametrize("cfgname,ctx", [("qwen3_8l_bf16", [4096]), ("qwen3_8l_bf16", [0, 17, 300, 129]),
                                         ("wide_5l_yarn_bf16", [3000]),
                                         # long ranges: the super-chunk kernel (>= 4 chunks per CTA)
                                         ("qwen3_8l_bf16", [8000, 7000, 6100, 5000, 3000, 8100, 100, 7777]),
                                         ("wide_5l_yarn_bf16", [6000, 5000, 9000, 4000])])
def test_tensor_core_attention_matches_cuda_core(cfgname, ctx):
    """Same queries, same paged pool: the tcgen05 attention (split-KV, chunked online
    softmax, bf16 probabilities) against the CUDA-core one (fp32 online softmax)."""
    from helpers import Rig
    cfg = CONFIGS[cfgname]
    wl = make_workload(cfg, 61, ctx)
    rig = Rig(wl)
    rig.propose()
    M = wl.nb * 16
    layers = [cfg.n_layers - 1] + ([0] if cfg.sliding(0) else [])
    for layer in layers:
        a = torch.zeros((M, cfg.q_dim), dtype=torch.bfloat16, device="cuda")
        b = torch.zeros_like(a)
        dflash_attention_check(rig.drafter.handle, layer, rig.ctx_lens.data_ptr(), rig.page_tables.data_ptr(),
                               wl.nb, wl.max_ctx_len, a.data_ptr(), b.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert rig.drafter.device_status() == 0
        err = ((a.float() - b.float()).abs().max() / a.float().abs().max()).item()
        assert err < 1e-2, (layer, err)


@pytest.mark.parametrize("ctx", [[5, 17, 3, 40], [0, 2, 900, 1]])
def test_stream_k_attention_under_a_loose_max_context(ctx):
    """max_ctx_len far above every context (20000): the host picks the stream-K kernel from it,
    while the batch holds fewer key chunks than the kernel has CTAs (most CTAs get no chunk, a
    unit's chunks sit in one CTA or span a few).  Same comparison as above."""
    from helpers import Rig
    cfg = CONFIGS["qwen3_8l_bf16"]
    wl = make_workload(cfg, 63, ctx, extra_pages_per_seq=1260)
    rig = Rig(wl)
    rig.propose()
    M = wl.nb * 16
    layer = cfg.n_layers - 1
    a = torch.zeros((M, cfg.q_dim), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros_like(a)
    dflash_attention_check(rig.drafter.handle, layer, rig.ctx_lens.data_ptr(), rig.page_tables.data_ptr(),
                           wl.nb, 20000, a.data_ptr(), b.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rig.drafter.device_status() == 0
    err = ((a.float() - b.float()).abs().max() / a.float().abs().max()).item()
    assert err < 1e-2, err
