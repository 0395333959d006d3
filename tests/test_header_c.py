"""include/dflash.h as a C user sees it (CPU): the header compiles as strict C99, a C program
links every declared function from libdflash.so, and the struct layouts the C compiler gives
match the ctypes structures of the Python binding field by field."""
import ctypes
import os
import shutil
import subprocess

import pytest

from test_abi import ROOT, declared_functions

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")

STRUCTS = {
    "dflash_cfg": ("hidden", "n_q_heads", "n_kv_heads", "head_dim", "n_ff", "n_layers", "vocab", "gamma",
                   "mask_token_id", "n_taps", "target_hidden", "rms_eps", "rope_theta", "rope_yarn", "yarn_factor",
                   "yarn_orig_max_pos", "yarn_beta_fast", "yarn_beta_slow", "sliding_window", "layer_sliding", "dtype",
                   "lm_head_dtype", "page_size", "num_pages", "max_batch", "max_pages_per_seq", "max_write_rows",
                   "markov_rank", "layer_weight_dtype"),
    "dflash_layer_weights": ("ln_in", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ln_post", "w_gate", "w_up",
                             "w_down"),
    "dflash_weights": ("fc", "hidden_norm", "norm", "embed", "lm_head", "layers", "markov_w1", "markov_w2"),
}


def _program() -> str:
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "dflash.h"', "int main(void) {"]
    # take the address of every declared function: the link fails if one is missing
    fns = declared_functions()
    lines.append("  void (*fns[])(void) = {" + ", ".join(f"(void (*)(void)){f}" for f in fns) + "};")
    lines.append('  printf("fns %d\\n", (int)(sizeof fns / sizeof fns[0]));')
    for s, fields in STRUCTS.items():
        lines.append(f'  printf("{s} size %zu\\n", sizeof({s}));')
        for f in fields:
            lines.append(f'  printf("{s} {f} %zu\\n", offsetof({s}, {f}));')
    lines += ["  return 0;", "}"]
    return "\n".join(lines) + "\n"


@pytest.fixture(scope="module")
def layout(tmp_path_factory):
    from block_diffusion_drafter_forward_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    d = tmp_path_factory.mktemp("c_abi")
    src = d / "abi.c"
    src.write_text(_program())
    exe = d / "abi"
    libdir = os.path.dirname(_lib.LIB_PATH)
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                         str(src), "-o", str(exe), "-L", libdir, "-l:libdflash.so", f"-Wl,-rpath,{libdir}",
                         "-Wl,--no-as-needed"], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    out = {}
    for ln in run.stdout.splitlines():
        parts = ln.split()
        out[tuple(parts[:-1])] = int(parts[-1])
    return out


def test_header_is_c99_and_every_function_links(layout):
    assert layout[("fns",)] == len(declared_functions())


@pytest.mark.parametrize("name", list(STRUCTS))
def test_ctypes_layout_matches_the_c_compiler(layout, name):
    from block_diffusion_drafter_forward_gb300 import _lib
    ct = getattr(_lib, name)
    assert [f for f, _ in ct._fields_] == list(STRUCTS[name])
    assert ctypes.sizeof(ct) == layout[(name, "size")]
    for f in STRUCTS[name]:
        assert getattr(ct, f).offset == layout[(name, f)], (name, f)
