"""Parity of the CUDA path (through the C ABI) with the CPU oracle on seeded inputs.

Bars: bit-exact placement of every K/V row in the paged pool and of the draft tokens
wherever the oracle's top-1/top-2 logit margin exceeds the config's margin (0.1 for
bf16, 1e-3 for fp32); relative max error <= 2e-2 (bf16) / 1e-4 (fp32) on final hidden
states and <= 3e-2 / 1e-4 on logits."""
import numpy as np
import pytest
import torch

from block_diffusion_drafter_forward_gb300 import dflash_fp8_lm_head
from block_diffusion_drafter_forward_gb300._lib import DFLASH_DEV_BAD_PAGE
from oracle.dflash_oracle import Oracle, fp8_quantize_rows, page_slots, to_f64
from synth import CONFIGS, WORKLOADS, make_workload
from synth.torch_io import to_torch

from helpers import TOL, DevView, Rig, as_f64, check_band, pool_rows, pool_view, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_drafter_forward_gb300._lib as L
    L.load()


def run_and_check(wl, bands=None, max_write_rows=4096, check_kv=True, rig=None):
    rig = rig or Rig(wl, max_write_rows=max_write_rows)
    drafts, z, h = rig.propose()
    assert rig.drafter.device_status() == 0
    tol = TOL[wl.cfg.dtype]
    o = Oracle(wl.cfg, rig.W)
    bands = range(wl.nb) if bands is None else bands
    errs = []
    for s in bands:
        ref = rig.oracle_band(s, o)
        errs.append(check_band(rig, s, ref, drafts, z, h, tol))
        if check_kv and int(wl.ctx_lens[s]) > 0:
            c = int(wl.ctx_lens[s])
            sl = page_slots(wl.page_tables[s], 0, c)
            for l in (0, wl.cfg.n_layers - 1):
                for g in range(wl.cfg.n_kv_heads):
                    k = pool_rows(rig.drafter, l, 0, g, sl // 16, sl % 16)
                    v = pool_rows(rig.drafter, l, 1, g, sl // 16, sl % 16)
                    assert rel_err(k, ref["k"][l][:, g]) <= tol["hidden"]
                    assert rel_err(v, ref["v"][l][:, g]) <= tol["hidden"]
    assert int(drafts.min()) >= 0 and int(drafts.max()) < wl.cfg.vocab
    return rig, errs


# ----------------------------------------------------------------------------- tiny fp32


def test_tiny_fp32_full_size():
    run_and_check(WORKLOADS["tiny_fp32_nb1_ctx64"]())


def test_tiny_fp32_ragged_batch_with_empty_context():
    wl = make_workload(CONFIGS["tiny_fp32"], 11, [0, 5, 77, 16])
    run_and_check(wl)


@pytest.mark.parametrize("cfg_name,ctxs,sentinel", [
    ("tiny_fp32", [37, 50], -12345.0),
    ("qwen3_8l_bf16", [37, 50], -12288.0),   # per-projection kernels, 4 kv heads
    ("qwen3_8l_bf16", [93], -12288.0),       # single-launch forward
])
def test_slot_writeback_exact(cfg_name, ctxs, sentinel):
    """A sentinel-filled pool: the writer changes exactly the slots of rows 0..c-1 and
    propose exactly the slots c..c+15, layer by layer (integer placement, bit-exact).
    The sentinel is exact in the pool's dtype."""
    wl = make_workload(CONFIGS[cfg_name], 12, ctxs)
    rig = Rig(wl, write=False)
    pool = pool_view(rig.drafter)
    pool.fill_(sentinel)
    rig.write_all(chunk=20)
    _, _, st = rig.drafter.kv_layout()
    hd, L, P, nkv = wl.cfg.head_dim, wl.cfg.n_layers, wl.num_pages, wl.cfg.n_kv_heads
    # every tile's base through the published strides (any tile order), then the documented
    # in-tile layouts: K tile element (j, d) -> row j; V tile (j, d) -> row j
    idx = torch.arange
    base = (idx(L)[:, None, None, None] * st[0] + idx(P)[None, :, None, None] * st[1]
            + idx(2)[None, None, :, None] * st[2] + idx(nkv)[None, None, None, :] * st[3]).cuda()
    j = torch.arange(16)[:, None]
    d = torch.arange(hd)[None, :]
    kinner = (((j // 8) * (hd // 8) + d // 8) * 64 + (j % 8) * 8 + d % 8).cuda()
    vinner = (((d // 8) * 2 + j // 8) * 64 + (d % 8) * 8 + j % 8).cuda()

    def changed_rows():
        # [L, P, nkv, 16, hd] booleans for the K tiles and the V tiles
        ch = (pool != sentinel)
        return (ch[base[:, :, 0, :, None, None] + kinner[None, None, None]],
                ch[base[:, :, 1, :, None, None] + vinner[None, None, None]])

    expect = torch.zeros((P, 16), dtype=torch.bool)
    for s in range(wl.nb):
        sl = page_slots(wl.page_tables[s], 0, int(wl.ctx_lens[s]))
        expect[sl // 16, sl % 16] = True
    kk, vv = changed_rows()
    e = expect.cuda()[None, :, None, :, None].expand_as(kk)
    assert torch.equal(kk, e) and torch.equal(vv, e)
    # propose adds the transient block rows c..c+15
    rig.propose()
    for s in range(wl.nb):
        c = int(wl.ctx_lens[s])
        sl = page_slots(wl.page_tables[s], c, 16)
        expect[sl // 16, sl % 16] = True
    kk, vv = changed_rows()
    e = expect.cuda()[None, :, None, :, None].expand_as(kk)
    assert torch.equal(kk, e) and torch.equal(vv, e)


def test_tiny_fp32_writer_chunking_is_bit_exact():
    wl = make_workload(CONFIGS["tiny_fp32"], 13, [100])
    a = Rig(wl, max_write_rows=4096)
    b = Rig(wl, max_write_rows=16, write=False)
    b.write_all(chunk=33)
    torch.cuda.synchronize()
    assert torch.equal(pool_view(a.drafter), pool_view(b.drafter))


def test_tiny_fp32_bands_are_independent():
    """Band s of a batched propose equals a single-sequence propose of sequence s."""
    wl = make_workload(CONFIGS["tiny_fp32"], 14, [30, 64, 9])
    rig = Rig(wl)
    d3, z3, h3 = rig.propose()
    for s in range(3):
        one = make_workload(CONFIGS["tiny_fp32"], 14, [int(wl.ctx_lens[s])], bonus=[int(wl.bonus[s])],
                            taps_rows=wl.taps_rows)
        one.tap_offsets[0] = wl.tap_offsets[s]
        r1 = Rig(one, write=False)
        r1._table = rig._table
        r1.write_all()
        d1, z1, h1 = r1.propose()
        assert torch.equal(d1[0], d3[s])
        assert rel_err(as_f64(h1), as_f64(h3[16 * s:16 * s + 16])) <= 1e-6


def test_bad_page_id_sets_flag_without_fault():
    wl = make_workload(CONFIGS["tiny_fp32"], 15, [20])
    rig = Rig(wl)
    bad = rig.page_tables.clone()
    bad[0, 1] = wl.num_pages + 7          # the page holding rows 16..31 (ctx and block rows)
    rig.drafter.propose(rig.bonus, rig.ctx_lens, bad, wl.max_ctx_len)
    assert rig.drafter.device_status() & DFLASH_DEV_BAD_PAGE
    assert rig.drafter.device_status() == 0   # cleared by the read
    rig.propose()                              # the handle stays usable


# ----------------------------------------------------------------------------- 8-layer bf16


def test_qwen3_8l_short_context():
    run_and_check(make_workload(CONFIGS["qwen3_8l_bf16"], 21, [200]))


def test_qwen3_8l_full_size_nb1_ctx4096():
    run_and_check(WORKLOADS["qwen3_8l_nb1_ctx4096"]())


def test_qwen3_8l_nb32_ragged_full_size_every_band():
    """The 32-sequence ragged batch at full size: every band against the oracle, and the
    context K/V pool rows of layers 0 and 7 of every sequence."""
    wl = WORKLOADS["qwen3_8l_nb32_ragged"]()
    run_and_check(wl)


def test_qwen3_8l_small_batch_all_bands():
    wl = make_workload(CONFIGS["qwen3_8l_bf16"], 22, [16, 300, 1, 47])
    run_and_check(wl)


# ----------------------------------------------------------------------------- wide YaRN + window


def test_wide_yarn_window_ctx3000():
    wl = make_workload(CONFIGS["wide_5l_yarn_bf16"], 41, [3000])
    run_and_check(wl)


@pytest.mark.slow
def test_wide_yarn_full_size_ctx16384():
    run_and_check(WORKLOADS["wide_5l_yarn_nb1_ctx16384"](), check_kv=False)


# ----------------------------------------------------------------------------- FP8 lm_head


def test_fp8_head_small():
    wl = make_workload(CONFIGS["qwen3_8l_fp8head"], 51, [1000, 37])
    run_and_check(wl)


def test_fp8_head_codes_and_scales_bit_exact():
    """The create-time e4m3 quantisation of the lm_head, byte for byte."""
    wl = make_workload(CONFIGS["qwen3_8l_fp8head"], 52, [16])
    rig = Rig(wl, write=False)
    codes_ptr, scale_ptr = dflash_fp8_lm_head(rig.drafter.handle)
    V, H = wl.cfg.vocab, wl.cfg.hidden
    codes = torch.as_tensor(DevView(codes_ptr, V * H, "|u1"), device="cuda").view(V, H)
    scale = torch.as_tensor(DevView(scale_ptr, V, "<f4"), device="cuda")
    lm = rig.W.get("lm_head", keep=False)
    for s0 in range(0, V, 37987):            # several row blocks spread over the vocabulary
        sl = slice(s0, min(V, s0 + 4096))
        rc, rs = fp8_quantize_rows(to_f64(lm[sl], "bf16").astype(np.float32))
        assert np.array_equal(codes[sl].cpu().numpy(), rc)
        assert np.array_equal(scale[sl].cpu().numpy(), rs)


@pytest.mark.parametrize("name,bands", [
    ("fp8head_nb1_ctx32768", [0]),
    ("fp8head_nb4_ctx32768", [2]),
    ("fp8head_nb16_ctx32768", [0, 9, 15]),
    ("fp8head_nb64_ctx32768", [0, 37, 63]),
])
def test_fp8_head_sweep_full_size_sampled(name, bands):
    """The FP8-lm_head throughput sweep at full size (32 768 context rows per sequence): the
    oracle recomputes the sampled bands one by one."""
    run_and_check(WORKLOADS[name](), bands=bands, check_kv=False)


# ----------------------------------------------------------------------------- other accepted shapes


def test_tiny_fp32_with_fp8_head():
    """The e4m3 lm_head on the fp32 drafter (CUDA-core FP8 GEMV over fp32 activations)."""
    rig, _ = run_and_check(make_workload(CONFIGS["tiny_fp32_fp8head"], 53, [64, 9]))
    codes_ptr, scale_ptr = dflash_fp8_lm_head(rig.drafter.handle)
    V, H = rig.cfg.vocab, rig.cfg.hidden
    codes = torch.as_tensor(DevView(codes_ptr, V * H, "|u1"), device="cuda").view(V, H)
    rc, rs = fp8_quantize_rows(rig.W.get("lm_head").astype(np.float32))
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("cfg_name", ["small_gqa4_bf16", "small_gqa8_bf16"])
def test_small_bf16_drafters_on_the_per_projection_kernels(cfg_name):
    """bf16 drafters the single launch does not take: 4 query heads per kv head (CUDA-core
    attention between the tensor-core projections), and 8 per kv head with an o_proj of
    fewer (tile, k-block) units than SMs.  Both at nb = 1 and on a ragged batch."""
    for seed, ctxs in ((54, [300]), (55, [0, 77, 1000])):
        rig, _ = run_and_check(make_workload(CONFIGS[cfg_name], seed, ctxs))
        assert not rig.drafter.persistent
