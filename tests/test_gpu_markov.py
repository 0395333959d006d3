"""Parity of the DSpark Markov head (through the C ABI) with the CPU oracle's chain.

Each band's chain is compared with the oracle's position by position up to the first row whose
adjusted top-1/top-2 margin is within the config's near-tie margin (after such a row the two
chains may legitimately part, and every later bias with them); the adjusted logits of the rows
up to and including that one are compared at the logits tolerance, and row 0 (no bias) too."""
import numpy as np
import pytest
import torch

from oracle.dflash_oracle import Oracle
from synth import CONFIGS, make_workload

from helpers import TOL, Rig, as_f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_drafter_forward_gb300._lib as L
    L.load()


def check_markov(wl):
    rig = Rig(wl)
    assert not rig.drafter.persistent
    drafts, z, h = rig.propose()
    assert rig.drafter.device_status() == 0
    tol = TOL[wl.cfg.dtype]
    o = Oracle(wl.cfg, rig.W, cache=True)
    plain_differs = 0
    for s in range(wl.nb):
        ref = rig.oracle_band(s, o)
        z0, adj, tok, margin = o.drafts_markov(ref["h"], int(wl.bonus[s]))
        assert rel_err(as_f64(h[16 * s:16 * s + 16]), ref["h"]) <= tol["hidden"]
        zs = as_f64(z[16 * s:16 * s + 16])
        unsure = np.nonzero(margin <= tol["margin"])[0]
        stop = int(unsure[0]) if unsure.size else 15           # first row where chains may part
        got = drafts[s].cpu().numpy().astype(np.int64)
        assert np.array_equal(got[:stop], tok[:stop]), (s, stop, got, tok, margin)
        rows = min(stop + 1, 15)
        assert rel_err(zs[0], z0) <= tol["logits"]
        assert rel_err(zs[1:1 + rows], adj[:rows]) <= tol["logits"], s
        plain_differs += int(not np.array_equal(tok, ref["tokens"]))
    assert int(drafts.min()) >= 0 and int(drafts.max()) < wl.cfg.vocab
    # the head changed the drafts of at least one band (it is not a no-op)
    assert plain_differs > 0
    return rig


def test_markov_tiny_fp32():
    check_markov(make_workload(CONFIGS["tiny_fp32_markov"], 61, [64]))
    check_markov(make_workload(CONFIGS["tiny_fp32_markov"], 62, [0, 30, 77]))


def test_markov_8l_bf16_nb1_and_ragged_batch():
    check_markov(make_workload(CONFIGS["qwen3_8l_markov"], 63, [500]))
    check_markov(make_workload(CONFIGS["qwen3_8l_markov"], 64, [16, 1200, 3, 700]))


def test_markov_graph_replay_follows_new_bonus_tokens():
    """The captured graph re-reads the bonus tokens (the chain's start) on every replay."""
    wl = make_workload(CONFIGS["tiny_fp32_markov"], 65, [40, 40])
    rig = Rig(wl)
    d1, _, _ = rig.propose()
    rig.bonus.copy_(torch.tensor([int(wl.bonus[1]), int(wl.bonus[0])], dtype=torch.int32, device="cuda"))
    d2, _, _ = rig.propose()
    wl.bonus[:] = wl.bonus[::-1].copy()
    o = Oracle(wl.cfg, rig.W, cache=True)
    for s in range(2):
        ref = rig.oracle_band(s, o)
        _, _, tok, margin = o.drafts_markov(ref["h"], int(wl.bonus[s]))
        unsure = np.nonzero(margin <= TOL["f32"]["margin"])[0]
        stop = int(unsure[0]) if unsure.size else 15
        assert np.array_equal(d2[s].cpu().numpy()[:stop], tok[:stop])
