"""The single-launch persistent forward (batch 1, bf16 lm_head) against the oracle, against
the per-projection kernels, and on its edge cases (empty context, a full page table, a bad
page id, repeated launches)."""
import numpy as np
import pytest
import torch

from oracle.dflash_oracle import Oracle
from synth import CONFIGS, make_workload

from helpers import TOL, Rig, as_f64, check_band, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_drafter_forward_gb300._lib as L
    L.load()


def _check_vs_oracle(rig, drafts, z, h):
    tol = TOL[rig.cfg.dtype]
    ref = rig.oracle_band(0, Oracle(rig.cfg, rig.W))
    return check_band(rig, 0, ref, drafts, z, h, tol)


def test_persistent_is_default_for_one_sequence():
    rig = Rig(make_workload(CONFIGS["qwen3_8l_bf16"], 61, [200]))
    assert rig.drafter.persistent
    d, z, h = rig.propose()
    assert rig.drafter.device_status() == 0
    _check_vs_oracle(rig, d, z, h)


def test_persistent_and_per_projection_agree():
    rig = Rig(make_workload(CONFIGS["qwen3_8l_bf16"], 62, [1500]))
    d1, z1, h1 = rig.propose()
    assert rig.drafter.device_status() == 0
    e1 = _check_vs_oracle(rig, d1, z1, h1)
    rig.drafter.set_persistent(False)
    assert not rig.drafter.persistent
    d2, z2, h2 = rig.propose()
    assert rig.drafter.device_status() == 0
    e2 = _check_vs_oracle(rig, d2, z2, h2)
    # same arithmetic, different split-K summation order; each bf16 intermediate (xb, q,
    # attention output, MLP activation) then rounds differently, so the two paths sit as far
    # from each other as each sits from the oracle: the oracle's bar applies between them
    tol = TOL["bf16"]
    assert rel_err(as_f64(h1), as_f64(h2)) <= tol["hidden"], (e1, e2)
    assert rel_err(as_f64(z1), as_f64(z2)) <= tol["logits"], (e1, e2)
    rig.drafter.set_persistent(True)
    d3, z3, h3 = rig.propose()
    assert torch.equal(z3, z1) and torch.equal(d3, d1)


def test_persistent_repeated_launches_bit_identical():
    rig = Rig(make_workload(CONFIGS["qwen3_8l_bf16"], 63, [700]))
    outs = [rig.propose() for _ in range(3)]
    for d, z, h in outs[1:]:
        assert torch.equal(d, outs[0][0]) and torch.equal(z, outs[0][1]) and torch.equal(h, outs[0][2])
    assert rig.drafter.device_status() == 0


def test_persistent_empty_context():
    rig = Rig(make_workload(CONFIGS["qwen3_8l_bf16"], 64, [0]))
    d, z, h = rig.propose()
    assert rig.drafter.device_status() == 0
    _check_vs_oracle(rig, d, z, h)


def test_persistent_page_table_full():
    # context + block fill every page of the table exactly
    wl = make_workload(CONFIGS["qwen3_8l_bf16"], 65, [4096 - 16])
    rig = Rig(wl)
    assert (int(wl.ctx_lens[0]) + 16) % 16 == 0
    d, z, h = rig.propose()
    assert rig.drafter.device_status() == 0
    _check_vs_oracle(rig, d, z, h)


def test_persistent_bad_page_sets_flag_without_fault():
    from block_diffusion_drafter_forward_gb300._lib import DFLASH_DEV_BAD_PAGE

    wl = make_workload(CONFIGS["qwen3_8l_bf16"], 66, [100])
    rig = Rig(wl)
    pt = rig.page_tables.clone()
    pt[0, 2] = wl.num_pages + 5  # a context page out of range
    rig.page_tables = pt
    rig.propose()
    assert rig.drafter.device_status() & DFLASH_DEV_BAD_PAGE
    # the handle stays usable
    rig.page_tables = torch.as_tensor(wl.page_tables, dtype=torch.int32, device="cuda")
    d, z, h = rig.propose()
    assert rig.drafter.device_status() == 0
    _check_vs_oracle(rig, d, z, h)


def test_persistent_wide_window_config():
    rig = Rig(make_workload(CONFIGS["wide_5l_yarn_bf16"], 67, [2500]))
    assert rig.drafter.persistent
    d, z, h = rig.propose()
    assert rig.drafter.device_status() == 0
    _check_vs_oracle(rig, d, z, h)


def test_fp8_head_uses_per_projection_kernels():
    rig = Rig(make_workload(CONFIGS["qwen3_8l_fp8head"], 68, [300]), write=False)
    assert not rig.drafter.persistent
    from block_diffusion_drafter_forward_gb300 import DflashError

    with pytest.raises(DflashError):
        rig.drafter.set_persistent(True)


def test_persistent_hidden_only_outputs():
    # logits and hidden outputs are optional: drafts alone must match
    rig = Rig(make_workload(CONFIGS["qwen3_8l_bf16"], 69, [333]))
    d_full, _, _ = rig.propose()
    d_only, _, _ = rig.propose(logits=False, hidden=False)
    assert torch.equal(d_full, d_only)
    assert np.all(d_only.cpu().numpy() >= 0)


def test_graph_replay_reads_new_inputs():
    # dflash_propose replays a captured graph for the same buffers: new values written into the
    # same bonus-token buffer must be used (on both launch shapes)
    wl = make_workload(CONFIGS["qwen3_8l_bf16"], 70, [500])
    rig = Rig(wl)
    g, V = rig.cfg.gamma, rig.cfg.vocab
    drafts = torch.empty((1, g - 1), dtype=torch.int32, device="cuda")
    z = torch.empty((g, V), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((g, rig.cfg.hidden), dtype=torch.bfloat16, device="cuda")
    first = int(wl.bonus[0])
    for persistent in (True, False):
        rig.drafter.set_persistent(persistent)
        for bonus in (first, (first + 12345) % V, first):
            wl.bonus[0] = bonus
            rig.bonus.fill_(bonus)
            rig.drafter.propose(rig.bonus, rig.ctx_lens, rig.page_tables, wl.max_ctx_len, drafts=drafts, logits=z,
                                hidden=h)
            torch.cuda.synchronize()
            assert rig.drafter.device_status() == 0
            _check_vs_oracle(rig, drafts, z, h)
