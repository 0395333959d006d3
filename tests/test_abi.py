"""The C ABI without a GPU: the library loads, exports every function include/*.h
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_diffusion_drafter_forward_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(dflash_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dflash_create", "dflash_destroy", "dflash_write_ctx_kv", "dflash_propose", "dflash_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
    from block_diffusion_drafter_forward_gb300 import _lib
    assert set(_lib.EXPORTS) <= set(names)


def _cfg():
    from block_diffusion_drafter_forward_gb300 import make_cfg
    from synth import CONFIGS
    return make_cfg(CONFIGS["tiny_fp32"], num_pages=8, max_batch=2, max_pages_per_seq=8)


def _create_rc(lib, cfg):
    from block_diffusion_drafter_forward_gb300 import _lib
    w = _lib.dflash_weights()
    out = ctypes.c_void_p()
    return lib.dflash_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(out)), out


@pytest.mark.parametrize("field,value,code", [
    ("gamma", 8, -5), ("page_size", 32, -5), ("head_dim", 96, -5), ("n_kv_heads", 3, -1),
    ("n_layers", 0, -1), ("n_layers", 65, -1), ("dtype", 7, -1), ("lm_head_dtype", 9, -1),
    ("mask_token_id", 5000, -1), ("num_pages", 0, -1), ("max_write_rows", 8, -1), ("hidden", 0, -1),
])
def test_create_rejects_bad_config(lib, field, value, code):
    cfg = _cfg()
    setattr(cfg, field, value)
    rc, out = _create_rc(lib, cfg)
    assert rc == code and not out.value
    assert lib.dflash_last_error(None)


def test_create_rejects_null_weights(lib):
    rc, out = _create_rc(lib, _cfg())
    assert rc == -1 and b"weight" in lib.dflash_last_error(None)


def test_sliding_layer_needs_window(lib):
    cfg = _cfg()
    cfg.layer_sliding[0] = 1
    cfg.sliding_window = 0
    rc, _ = _create_rc(lib, cfg)
    assert rc == -1


def test_calls_on_null_handle(lib):
    assert lib.dflash_propose(None, None, None, None, 1, 0, None, None, None, None) == -1
    assert lib.dflash_write_ctx_kv(None, None, None, None, 0, 0, None) == -1
    assert lib.dflash_destroy(None) == 0
    assert lib.dflash_kv_layout(None, None, None, None) == -1
    assert lib.dflash_set_persistent(None, 1) == -1
    assert lib.dflash_set_persistent(None, 0) == -1
    assert lib.dflash_persistent(None) == 0
