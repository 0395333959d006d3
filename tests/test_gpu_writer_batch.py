"""The batched context-K/V writer (one call over several sequences' new rows, rows in any order)
through the C ABI: K/V against the oracle, slot placement byte-exact on a sentinel-filled pool,
the fp32 path bit-identical to the per-sequence writer (its GEMM sums every output element in the
same order whatever the batch), the bf16 path within one bf16 rounding of it, and the device-side
row checks."""
import numpy as np
import pytest
import torch

from block_diffusion_drafter_forward_gb300._lib import DFLASH_DEV_BAD_CTX
from oracle.dflash_oracle import Oracle, page_slots
from synth import CONFIGS, make_workload, workload_taps
from synth.torch_io import to_torch

from helpers import TOL, Rig, pool_rows, pool_view, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_drafter_forward_gb300._lib as L
    L.load()


def batch_rows(rig, spans, seed):
    """Rows (sequence s, logical rows first..first+n-1) of every span, shuffled: taps, positions,
    row_seq, row_index as device tensors."""
    taps, pos, rs, ri = [], [], [], []
    for s, first, n in spans:
        taps.append(rig.taps_dev(s, first, n))
        pos.append(rig.wl.ctx_positions(s, first, n))
        rs.append(np.full(n, s, np.int32))
        ri.append(np.arange(first, first + n, dtype=np.int32))
    perm = np.random.default_rng(seed).permutation(sum(n for _, _, n in spans))
    permt = torch.as_tensor(perm, device="cuda")
    return (torch.cat(taps)[permt].contiguous(), to_torch(np.concatenate(pos)[perm], "i32"),
            to_torch(np.concatenate(rs)[perm], "i32"), to_torch(np.concatenate(ri)[perm], "i32"))


def write_batched(rig, spans, seed=0):
    taps, pos, rs, ri = batch_rows(rig, spans, seed)
    rig.drafter.write_ctx_kv_batch(taps, pos, rs, ri, rig.page_tables)
    torch.cuda.synchronize()


def write_each(rig, spans):
    for s, first, n in spans:
        rig.drafter.write_ctx_kv(rig.taps_dev(s, first, n), to_torch(rig.wl.ctx_positions(s, first, n), "i32"),
                                 rig.page_tables[s], first)
    torch.cuda.synchronize()


SPANS = [(0, 0, 300), (1, 0, 41), (2, 0, 100), (2, 100, 517), (3, 16, 33)]


@pytest.mark.parametrize("cfg_name", ["tiny_fp32", "qwen3_8l_bf16"])
def test_batched_writer_against_oracle_and_per_sequence(cfg_name):
    wl = make_workload(CONFIGS[cfg_name], 91, [300, 41, 617, 49])
    a = Rig(wl, write=False, max_write_rows=256)   # several chunks in one batched call
    b = Rig(wl, write=False, max_write_rows=256)
    write_batched(a, SPANS, seed=1)
    write_each(b, SPANS)
    assert a.drafter.device_status() == 0 and b.drafter.device_status() == 0
    pa, pb = pool_view(a.drafter), pool_view(b.drafter)
    if wl.cfg.dtype == "f32":
        assert torch.equal(pa, pb)
    else:
        # same arithmetic; only the split-K summation order of the two GEMMs follows the row count,
        # so the fp32 values before the bf16 rounding differ in their last bits: one bf16 step of
        # the value, or (for elements far below their head's scale, after k_norm) a few fp32 steps
        # of the head's scale
        da, db = pa.float(), pb.float()
        diff = (da - db).abs()
        bound = torch.maximum(da.abs(), db.abs()) * 2.0 ** -7 + 2.0 ** -18 * max(float(da.abs().max()), 1.0)
        worst = float((diff - bound).max())
        assert worst <= 0, (worst, float(diff.max()), int((diff > 0).sum()), diff.numel())
    tol = TOL[wl.cfg.dtype]
    o = Oracle(wl.cfg, a.W, cache=True)
    for s, first, n in SPANS:
        f = o.ctx_features(workload_taps(wl, s, first, n))
        sl = page_slots(wl.page_tables[s], first, n)
        for l in (0, wl.cfg.n_layers - 1):
            k, v = o.ctx_kv_layer(l, f, wl.ctx_positions(s, first, n))
            for g in range(wl.cfg.n_kv_heads):
                assert rel_err(pool_rows(a.drafter, l, 0, g, sl // 16, sl % 16), k[:, g]) <= tol["hidden"]
                assert rel_err(pool_rows(a.drafter, l, 1, g, sl // 16, sl % 16), v[:, g]) <= tol["hidden"]


def test_batched_writer_slot_placement_is_exact():
    wl = make_workload(CONFIGS["qwen3_8l_bf16"], 92, [70, 20, 130])
    rig = Rig(wl, write=False)
    pool = pool_view(rig.drafter)
    pool.fill_(-12288.0)
    spans = [(0, 0, 70), (1, 3, 17), (2, 40, 90)]
    write_batched(rig, spans, seed=2)
    _, _, st = rig.drafter.kv_layout()
    L, P, nkv = wl.cfg.n_layers, wl.num_pages, wl.cfg.n_kv_heads
    changed = (pool != -12288.0).view(L, P, nkv, 2, 16, 128)   # [layer][page][head][K|V][16 x 128 tile]
    assert st[1] == nkv * 2 * 16 * 128 and st[3] == 2 * 16 * 128
    rows_touched = changed.any(dim=-1)                             # every element of a row is written
    expect = torch.zeros((P, 16), dtype=torch.bool)
    for s, first, n in spans:
        sl = page_slots(wl.page_tables[s], first, n)
        expect[sl // 16, sl % 16] = True
    # K tiles (8x8 blocks: row j's dims are spread) and V tiles: compare per page the set of rows
    kinner = torch.tensor([[((j // 8) * 16 + d // 8) * 64 + (j % 8) * 8 + d % 8 for d in range(128)]
                           for j in range(16)], device="cuda")
    vinner = torch.tensor([[((d // 8) * 2 + j // 8) * 64 + (d % 8) * 8 + j % 8 for d in range(128)]
                           for j in range(16)], device="cuda")
    tiles = changed.reshape(L, P, nkv, 2, 2048)
    krows = tiles[:, :, :, 0][..., kinner].all(-1)
    vrows = tiles[:, :, :, 1][..., vinner].all(-1)
    kany = tiles[:, :, :, 0][..., kinner].any(-1)
    e = expect.cuda()[None, :, None, :].expand_as(krows)
    assert torch.equal(krows, e) and torch.equal(kany, e) and torch.equal(vrows, e)
    del rows_touched


def test_batched_writer_flags_rows_out_of_range():
    wl = make_workload(CONFIGS["tiny_fp32"], 93, [40, 40])
    rig = Rig(wl, write=False)
    taps, pos, rs, ri = batch_rows(rig, [(0, 0, 20), (1, 0, 20)], seed=3)
    rs[3] = 7                                  # no such sequence
    ri[5] = 16 * wl.max_pages_per_seq          # past the page table
    rig.drafter.write_ctx_kv_batch(taps, pos, rs, ri, rig.page_tables)
    assert rig.drafter.device_status() & DFLASH_DEV_BAD_CTX
    assert rig.drafter.device_status() == 0
