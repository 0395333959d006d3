"""The FP8 drafter lane (every layer's q/k/v/o/gate/up/down and the lm_head in e4m3 with per-row
fp32 scales; the context-K/V writer on the bf16 weights) through the C ABI: the create-time codes
and scales byte for byte against the oracle's quantiser, and the forward against the oracle's
FP8 forward at the bf16 tolerances."""
import numpy as np
import pytest
import torch

from block_diffusion_drafter_forward_gb300 import dflash_fp8_layer
from oracle.dflash_oracle import fp8_quantize_rows, to_f64
from synth import CONFIGS, WORKLOADS, make_workload

from helpers import DevView, Rig

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_drafter_forward_gb300._lib as L
    L.load()


def _packed(W, l, proj, cfg):
    """The packed weight the library quantises (q|k|v rows; gate/up in 64-row blocks)."""
    g = lambda t: to_f64(W.get(f"L{l}.{t}"), "bf16").astype(np.float32)  # noqa: E731
    if proj == 0:
        return np.concatenate([g("wq"), g("wk"), g("wv")])
    if proj == 1:
        return g("wo")
    if proj == 3:
        return g("w_down")
    gate, up = g("w_gate"), g("w_up")
    blocks = []
    for b in range(cfg.n_ff // 64):
        blocks += [gate[64 * b:64 * b + 64], up[64 * b:64 * b + 64]]
    return np.concatenate(blocks)


def test_fp8_layer_codes_and_scales_bit_exact():
    wl = make_workload(CONFIGS["qwen3_8l_fp8w"], 101, [16])
    rig = Rig(wl, write=False)
    assert not rig.drafter.persistent
    for l, proj in ((0, 0), (0, 1), (7, 2), (7, 3)):
        w = _packed(rig.W, l, proj, wl.cfg)
        rows, cols = w.shape
        cp, sp = dflash_fp8_layer(rig.drafter.handle, l, proj)
        codes = torch.as_tensor(DevView(cp, rows * cols, "|u1"), device="cuda").view(rows, cols).cpu().numpy()
        scale = torch.as_tensor(DevView(sp, rows, "<f4"), device="cuda").cpu().numpy()
        rc, rs = fp8_quantize_rows(w)
        assert np.array_equal(codes, rc), (l, proj)
        assert np.array_equal(scale, rs), (l, proj)


def test_fp8_layers_forward_small():
    from test_gpu_parity import run_and_check
    run_and_check(make_workload(CONFIGS["qwen3_8l_fp8w"], 102, [600]))
    run_and_check(make_workload(CONFIGS["qwen3_8l_fp8w"], 103, [0, 77, 1500]))


def test_fp8_layers_full_size_nb1_and_nb32_sampled():
    from test_gpu_parity import run_and_check
    run_and_check(WORKLOADS["fp8w_nb1_ctx4096"](), check_kv=False)
    run_and_check(WORKLOADS["fp8w_nb32_ragged"](), bands=[0, 17, 31], check_kv=False)
