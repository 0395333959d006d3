"""dflash_propose_ex: per-sequence RoPE start (q_rope_pos) and active block width, both read on
the device, against the oracle's b-row block at that RoPE start; on the single-launch forward
(nb = 1), the per-projection kernels (a ragged batch) and the CUDA-core fp32 path; graph replays
that change the values in place; and the out-of-range width flag."""
import numpy as np
import pytest
import torch

from block_diffusion_drafter_forward_gb300._lib import DFLASH_DEV_BAD_WIDTH
from oracle.dflash_oracle import Oracle
from synth import CONFIGS, make_workload
from synth.torch_io import to_torch

from helpers import TOL, Rig, as_f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_drafter_forward_gb300._lib as L
    L.load()


def run_ex(rig, rope, widths):
    nb, g, cfg = rig.wl.nb, rig.cfg.gamma, rig.cfg
    dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    z = torch.empty((nb * g, cfg.vocab), dtype=dt, device="cuda")
    h = torch.empty((nb * g, cfg.hidden), dtype=dt, device="cuda")
    d = rig.drafter.propose(rig.bonus, rig.ctx_lens, rig.page_tables, rig.wl.max_ctx_len, logits=z, hidden=h,
                            q_rope_pos=rope, widths=widths)
    torch.cuda.synchronize()
    return d, z, h


def check_ex(rig, rope_np, widths_np, o=None):
    wl, cfg = rig.wl, rig.cfg
    tol = TOL[cfg.dtype]
    rope = to_torch(np.asarray(rope_np, dtype=np.int32), "i32") if rope_np is not None else None
    widths = to_torch(np.asarray(widths_np, dtype=np.int32), "i32") if widths_np is not None else None
    d, z, h = run_ex(rig, rope, widths)
    assert rig.drafter.device_status() == 0
    o = o or Oracle(cfg, rig.W, cache=True)
    for s in range(wl.nb):
        c = int(wl.ctx_lens[s])
        b = int(widths_np[s]) if widths_np is not None else 16
        rp = int(rope_np[s]) if rope_np is not None else None
        from synth import workload_taps
        ref = o.run_sequence(workload_taps(wl, s, 0, c), wl.ctx_positions(s, 0, c), int(wl.bonus[s]),
                             block_pos0=rp, width=b)
        assert rel_err(as_f64(h[16 * s:16 * s + b]), ref["h"]) <= tol["hidden"], s
        assert rel_err(as_f64(z[16 * s:16 * s + b]), ref["logits"]) <= tol["logits"], s
        got = d[s].cpu().numpy().astype(np.int64)
        sure = ref["margin"] > tol["margin"]
        assert np.array_equal(got[:b - 1][sure], ref["tokens"][sure]), (s, got, ref["tokens"])
        assert np.all(got[b - 1:] == -1), (s, got)
    return d


def test_propose_ex_single_launch_nb1():
    rig = Rig(make_workload(CONFIGS["qwen3_8l_bf16"], 81, [300]))
    assert rig.drafter.persistent
    check_ex(rig, [300 + 777], [9])
    check_ex(rig, None, [2])
    check_ex(rig, [5], None)


def test_propose_ex_per_projection_ragged():
    rig = Rig(make_workload(CONFIGS["qwen3_8l_bf16"], 82, [40, 0, 1000]))
    check_ex(rig, [40 + 3, 9000, 1000], [16, 5, 2])


def test_propose_ex_stream_k_attention():
    """Long contexts: the per-projection path's stream-K attention with per-sequence widths and
    RoPE starts."""
    rig = Rig(make_workload(CONFIGS["qwen3_8l_bf16"], 87, [3000, 2500, 4000, 3500]))
    check_ex(rig, [3000 + 5, 2500, 100, 3500], [16, 7, 2, 12])


def test_propose_ex_fp32_path():
    rig = Rig(make_workload(CONFIGS["tiny_fp32"], 83, [64, 17]))
    check_ex(rig, [64 + 200, 17], [4, 13])


def test_propose_ex_markov_head_stops_at_the_width():
    rig = Rig(make_workload(CONFIGS["tiny_fp32_markov"], 84, [50, 20]))
    rope = to_torch(np.array([50, 20], dtype=np.int32), "i32")
    widths = to_torch(np.array([6, 16], dtype=np.int32), "i32")
    d, z, h = run_ex(rig, rope, widths)
    assert rig.drafter.device_status() == 0
    o = Oracle(rig.cfg, rig.W, cache=True)
    from synth import workload_taps
    for s, b in ((0, 6), (1, 16)):
        c = int(rig.wl.ctx_lens[s])
        ref = o.run_sequence(workload_taps(rig.wl, s, 0, c), rig.wl.ctx_positions(s, 0, c), int(rig.wl.bonus[s]),
                             width=b)
        _, adj, tok, margin = o.drafts_markov(ref["h"], int(rig.wl.bonus[s]))
        unsure = np.nonzero(margin <= TOL["f32"]["margin"])[0]
        stop = int(unsure[0]) if unsure.size else b - 1
        got = d[s].cpu().numpy()
        assert np.array_equal(got[:stop], tok[:stop]) and np.all(got[b - 1:] == -1), (s, got, tok)


def test_propose_ex_graph_replay_follows_new_values():
    """Same buffers, new values: the captured graph reads widths and RoPE starts at run time."""
    wl = make_workload(CONFIGS["qwen3_8l_bf16"], 85, [200])
    rig = Rig(wl)
    rope = to_torch(np.array([200], dtype=np.int32), "i32")
    widths = to_torch(np.array([16], dtype=np.int32), "i32")
    d1, _, _ = run_ex(rig, rope, widths)
    rope.fill_(4000)
    widths.fill_(3)
    d2, z2, h2 = run_ex(rig, rope, widths)
    from synth import workload_taps
    ref = Oracle(wl.cfg, rig.W, cache=True).run_sequence(workload_taps(wl, 0, 0, 200), wl.ctx_positions(0, 0, 200),
                                                         int(wl.bonus[0]), block_pos0=4000, width=3)
    assert rel_err(as_f64(h2[:3]), ref["h"]) <= TOL["bf16"]["hidden"]
    assert np.all(d2[0].cpu().numpy()[2:] == -1)


def test_width_out_of_range_is_flagged_and_clamped():
    rig = Rig(make_workload(CONFIGS["tiny_fp32"], 86, [30]))
    for bad in (1, 40):
        widths = to_torch(np.array([bad], dtype=np.int32), "i32")
        d, z, h = run_ex(rig, None, widths)
        assert rig.drafter.device_status() & DFLASH_DEV_BAD_WIDTH
        clamped = 2 if bad < 2 else 16
        assert np.all(d[0].cpu().numpy()[clamped - 1:] == -1) and torch.isfinite(h[:clamped]).all()
    assert rig.drafter.device_status() == 0
