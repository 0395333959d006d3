"""The Python binding's argument checks (CPU): the C ABI takes raw pointers, so the binding
rejects a tensor of the wrong device, dtype, shape or layout before passing its address."""
import pytest
import torch

from block_diffusion_drafter_forward_gb300 import Drafter, make_cfg
from block_diffusion_drafter_forward_gb300.drafter import check_tensor
from synth import CONFIGS


def test_check_tensor_accepts_the_documented_layout():
    t = torch.zeros(3, 4, dtype=torch.int32)
    check_tensor(t, "t", torch.int32, (3, 4), device_type="cpu")
    check_tensor(t, "t", torch.int32, (2, 4), min_rows=True, device_type="cpu")
    check_tensor(torch.zeros(0, 4, dtype=torch.int32), "t", torch.int32, (0, 4), device_type="cpu")


@pytest.mark.parametrize("t,dtype,shape,kw,msg", [
    (torch.zeros(3, 4, dtype=torch.int32), torch.int64, (3, 4), {}, "expected torch.int64"),
    (torch.zeros(3, 4, dtype=torch.int32), torch.int32, (4, 4), {}, "expected shape"),
    (torch.zeros(3, 4, dtype=torch.int32), torch.int32, (4, 4), {"min_rows": True}, "expected shape"),
    (torch.zeros(3, 4, dtype=torch.int32), torch.int32, (3, 5), {}, "expected shape"),
    (torch.zeros(3, 4, dtype=torch.int32), torch.int32, (12,), {}, "expected shape"),
    (torch.zeros(4, 3, dtype=torch.int32).t(), torch.int32, (3, 4), {}, "contiguous"),
    (torch.zeros(16, 8, dtype=torch.float32), torch.bfloat16, (16, 8), {}, "expected torch.bfloat16"),
])
def test_check_tensor_rejects(t, dtype, shape, kw, msg):
    with pytest.raises(ValueError, match=msg):
        check_tensor(t, "t", dtype, shape, device_type="cpu", **kw)


def test_check_tensor_rejects_host_tensors_for_the_device():
    with pytest.raises(ValueError, match="expected a cuda tensor"):
        check_tensor(torch.zeros(2, dtype=torch.int32), "bonus", torch.int32, (2,))
    with pytest.raises(TypeError):
        check_tensor([1, 2], "bonus", torch.int32, (2,))


def _unbound_drafter():
    # a Drafter whose checks can run without a GPU: no handle was created, so reaching the C ABI
    # would raise DflashError (null handle) instead of the binding's ValueError
    cfg = CONFIGS["tiny_fp32"]
    d = Drafter.__new__(Drafter)
    d.cfg, d.handle = cfg, None
    d.ccfg = make_cfg(cfg, num_pages=8, max_batch=2, max_pages_per_seq=8)
    return d


def test_propose_and_write_check_before_calling_the_library():
    d = _unbound_drafter()
    i32 = dict(dtype=torch.int32)
    with pytest.raises(ValueError, match="bonus"):
        d.propose(torch.zeros(2, **i32), torch.zeros(2, **i32), torch.zeros(2, 8, **i32), 10)
    with pytest.raises(ValueError, match="taps"):
        d.write_ctx_kv(torch.zeros(4, 768), torch.zeros(4, **i32), torch.zeros(8, **i32), 0)
    assert d.act_dtype == torch.float32


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_8l_bf16", "wide_5l_yarn_bf16"])
def test_weight_shapes_match_the_generator(name):
    # the binding's expected shapes against the seeded generator's own table (HF layout)
    from block_diffusion_drafter_forward_gb300.drafter import weight_shapes
    from synth import make_weights
    cfg = CONFIGS[name]
    W = make_weights(cfg, 1)
    shapes = weight_shapes(cfg)
    assert set(shapes) == set(W.names())
    for n, sh in shapes.items():
        assert tuple(W.spec(n)[0]) == sh, n


def test_create_checks_every_weight_first():
    cfg = CONFIGS["tiny_fp32"]
    from block_diffusion_drafter_forward_gb300.drafter import weight_shapes
    tensors = {n: torch.zeros(sh) for n, sh in weight_shapes(cfg).items()}
    with pytest.raises(ValueError, match="expected a cuda tensor"):
        Drafter(cfg, tensors, num_pages=8, max_batch=1, max_pages_per_seq=8)
    del tensors["L0.wq"]
    with pytest.raises(ValueError, match="missing weight L0.wq"):
        Drafter(cfg, tensors, num_pages=8, max_batch=1, max_pages_per_seq=8)
