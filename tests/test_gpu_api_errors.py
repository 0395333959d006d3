"""The C ABI's checks on a GPU.

Host side: every argument that include/dflash.h rejects before a launch returns its status code
and a message, launches nothing (the draft buffer and the K/V pool keep their bytes), and leaves
the handle usable.

Device side: a context length outside [0, max_ctx_len] or past the page table, or a bonus token
outside [0, vocab), sets its status flag without a fault. The other sequences of the batch are
computed exactly as before, and the next valid call reproduces the earlier outputs bit for bit.

The three drafters exercise the three launch shapes: the CUDA-core kernels (tiny fp32), the
single-launch forward (8-layer bf16, one sequence) and the per-projection tensor-core kernels
(8-layer bf16, two sequences)."""
import ctypes

import pytest
import torch

import block_diffusion_drafter_forward_gb300._lib as L
from block_diffusion_drafter_forward_gb300 import DflashError
from synth import CONFIGS, make_workload

from helpers import Rig, pool_view

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_fp32_nb2": ("tiny_fp32", 81, [40, 7]),
    "bf16_nb1_persistent": ("qwen3_8l_bf16", 82, [300]),
    "bf16_nb2_per_projection": ("qwen3_8l_bf16", 83, [100, 20]),
}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.load()


@pytest.fixture(scope="module", params=list(CASES))
def rig(request):
    cfg, seed, ctxs = CASES[request.param]
    # one spare page per sequence: room for a context length above max_ctx_len that still fits
    r = Rig(make_workload(CONFIGS[cfg], seed, ctxs, extra_pages_per_seq=1))
    r.base = r.propose()
    assert r.drafter.device_status() == 0
    # the handle's flag: set for every bf16-head drafter; a batch of one takes the single launch
    assert r.drafter.persistent == (cfg == "qwen3_8l_bf16")
    yield r
    r.drafter.close()


def _raw_bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int32) if t.element_size() == 4 else t.view(torch.int16)


def _expect(code, call):
    with pytest.raises(DflashError) as e:
        call()
    assert e.value.code == code, str(e.value)
    assert str(e.value).split(": ", 1)[1], "no message"


def _assert_same_as_base(rig, bands=None):
    d, z, h = rig.propose()
    assert rig.drafter.device_status() == 0
    g = rig.cfg.gamma
    d0, z0, h0 = rig.base
    for s in bands if bands is not None else range(rig.wl.nb):
        assert torch.equal(d[s], d0[s]), s
        assert torch.equal(_raw_bits(z[s * g:(s + 1) * g]), _raw_bits(z0[s * g:(s + 1) * g])), s
        assert torch.equal(_raw_bits(h[s * g:(s + 1) * g]), _raw_bits(h0[s * g:(s + 1) * g])), s


def test_propose_rejects_bad_arguments(rig):
    wl, c = rig.wl, rig.drafter.ccfg
    drafts = torch.full((wl.nb, rig.cfg.gamma - 1), -7, dtype=torch.int32, device="cuda")
    ok = dict(bonus=rig.bonus.data_ptr(), ctx=rig.ctx_lens.data_ptr(), pt=rig.page_tables.data_ptr(),
              nb=wl.nb, max_ctx=wl.max_ctx_len, drafts=drafts.data_ptr())

    def call(**kw):
        a = {**ok, **kw}
        return lambda: L.dflash_propose(rig.drafter.handle, a["bonus"], a["ctx"], a["pt"], a["nb"], a["max_ctx"],
                                        a["drafts"])

    _expect(L.DFLASH_EINVAL, call(nb=0))
    _expect(L.DFLASH_EINVAL, call(nb=-1))
    _expect(L.DFLASH_ECAPACITY, call(nb=c.max_batch + 1))
    _expect(L.DFLASH_EINVAL, call(max_ctx=-1))
    # max_ctx_len + gamma must fit the page-table row
    _expect(L.DFLASH_ECAPACITY, call(max_ctx=16 * c.max_pages_per_seq - rig.cfg.gamma + 1))
    for k in ("bonus", "ctx", "pt", "drafts"):
        _expect(L.DFLASH_EINVAL, call(**{k: 0}))
    torch.cuda.synchronize()
    assert bool((drafts == -7).all()), "a rejected call launched work"
    # the largest max_ctx_len the page table admits is accepted; the attention's key split is
    # sized from it, so the summation order (not the inputs) may differ from the first call
    L.dflash_propose(rig.drafter.handle, ok["bonus"], ok["ctx"], ok["pt"], wl.nb,
                     16 * c.max_pages_per_seq - rig.cfg.gamma, ok["drafts"])
    torch.cuda.synchronize()
    assert rig.drafter.device_status() == 0
    assert int(drafts.min()) >= 0 and int(drafts.max()) < rig.cfg.vocab
    _assert_same_as_base(rig)


def test_write_rejects_bad_arguments(rig):
    c = rig.drafter.ccfg
    cap = 16 * c.max_pages_per_seq
    before = _raw_bits(pool_view(rig.drafter)).clone()
    taps = rig.taps_dev(0, 0, 2)
    pos = torch.arange(2, dtype=torch.int32, device="cuda")
    pt = rig.page_tables[0]
    h = rig.drafter.handle

    def call(tp=taps.data_ptr(), ps=pos.data_ptr(), pg=pt.data_ptr(), first=0, n=2):
        return lambda: L.dflash_write_ctx_kv(h, tp, ps, pg, first, n)

    _expect(L.DFLASH_EINVAL, call(first=-1))
    _expect(L.DFLASH_EINVAL, call(n=-1))
    _expect(L.DFLASH_ECAPACITY, call(first=cap - 1, n=2))
    _expect(L.DFLASH_EINVAL, call(tp=0))
    _expect(L.DFLASH_EINVAL, call(ps=0))
    _expect(L.DFLASH_EINVAL, call(pg=0))
    # n = 0 is a no-op, whatever the pointers
    L.dflash_write_ctx_kv(h, 0, 0, 0, cap, 0)
    torch.cuda.synchronize()
    assert torch.equal(_raw_bits(pool_view(rig.drafter)), before), "a rejected write touched the pool"
    assert rig.drafter.device_status() == 0
    _assert_same_as_base(rig)


@pytest.mark.parametrize("kind", ["negative", "above_max_ctx_len", "past_page_table"])
def test_bad_context_length_sets_flag(rig, kind):
    wl = rig.wl
    m = wl.max_ctx_len
    bad = {"negative": -3, "above_max_ctx_len": m + 1,
           "past_page_table": 16 * rig.drafter.ccfg.max_pages_per_seq - rig.cfg.gamma + 1}[kind]
    # the spare page keeps m + 1 inside the page table: only the max_ctx_len bound is broken
    assert kind != "above_max_ctx_len" or bad + rig.cfg.gamma <= 16 * rig.drafter.ccfg.max_pages_per_seq
    good = rig.ctx_lens.clone()
    rig.ctx_lens[0] = bad
    try:
        d, z, h = rig.propose()
        assert rig.drafter.device_status() & L.DFLASH_DEV_BAD_CTX
        # the other sequences are untouched by the bad one
        g, (d0, z0, h0) = rig.cfg.gamma, rig.base
        for s in range(1, wl.nb):
            assert torch.equal(d[s], d0[s]) and torch.equal(_raw_bits(z[s * g:]), _raw_bits(z0[s * g:])), s
    finally:
        rig.ctx_lens.copy_(good)
    _assert_same_as_base(rig)


@pytest.mark.parametrize("token", ["vocab", "negative"])
def test_bad_bonus_token_sets_flag(rig, token):
    wl = rig.wl
    good = rig.bonus.clone()
    rig.bonus[0] = rig.cfg.vocab if token == "vocab" else -1
    try:
        d, z, h = rig.propose()
        assert rig.drafter.device_status() & L.DFLASH_DEV_BAD_TOKEN
        # the anchor row is embedded as zeros: the forward stays finite
        assert bool(torch.isfinite(h.float()).all()) and bool(torch.isfinite(z.float()).all())
        assert int(d.min()) >= 0 and int(d.max()) < rig.cfg.vocab
        g, (d0, z0, h0) = rig.cfg.gamma, rig.base
        for s in range(1, wl.nb):
            assert torch.equal(d[s], d0[s]) and torch.equal(_raw_bits(h[s * g:]), _raw_bits(h0[s * g:])), s
    finally:
        rig.bonus.copy_(good)
    _assert_same_as_base(rig)


def test_last_error_names_the_failed_check(rig):
    wl = rig.wl
    drafts = torch.empty((wl.nb, rig.cfg.gamma - 1), dtype=torch.int32, device="cuda")
    with pytest.raises(DflashError) as e:
        L.dflash_propose(rig.drafter.handle, rig.bonus.data_ptr(), rig.ctx_lens.data_ptr(),
                         rig.page_tables.data_ptr(), rig.drafter.ccfg.max_batch + 1, wl.max_ctx_len,
                         drafts.data_ptr())
    assert "max_batch" in str(e.value)
    # a successful call clears it
    rig.propose()
    msg = L.load().dflash_last_error(ctypes.c_void_p(rig.drafter.handle))
    assert not msg
