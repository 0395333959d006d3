"""ctypes binding of libdflash.so: the C ABI of include/dflash.h, same names, argument
marshalling only.  Every step of the forward runs in the library's CUDA kernels; there is
no Python or CPU fallback: if the library is missing this module raises on load."""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdflash.so")

DFLASH_OK = 0
DFLASH_EINVAL = -1
DFLASH_ENOMEM = -2
DFLASH_ECUDA = -3
DFLASH_ECAPACITY = -4
DFLASH_EUNSUPPORTED = -5
DFLASH_EDEVICE = -6

DFLASH_F32 = 0
DFLASH_BF16 = 1
DFLASH_FP8E4M3_ROWSCALE = 2

DFLASH_DEV_BAD_PAGE = 0x1
DFLASH_DEV_BAD_CTX = 0x2
DFLASH_DEV_BAD_TOKEN = 0x4
DFLASH_DEV_TIMEOUT = 0x8
DFLASH_DEV_BAD_WIDTH = 0x10

STATUS_NAMES = {0: "OK", -1: "EINVAL", -2: "ENOMEM", -3: "ECUDA", -4: "ECAPACITY", -5: "EUNSUPPORTED",
                -6: "EDEVICE"}


class DflashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dflash {STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class dflash_cfg(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("n_ff", ctypes.c_int32), ("n_layers", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("gamma", ctypes.c_int32), ("mask_token_id", ctypes.c_int32),
        ("n_taps", ctypes.c_int32), ("target_hidden", ctypes.c_int32),
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("rope_yarn", ctypes.c_int32), ("yarn_factor", ctypes.c_float), ("yarn_orig_max_pos", ctypes.c_float),
        ("yarn_beta_fast", ctypes.c_float), ("yarn_beta_slow", ctypes.c_float),
        ("sliding_window", ctypes.c_int32), ("layer_sliding", ctypes.c_uint8 * 64),
        ("dtype", ctypes.c_int32), ("lm_head_dtype", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("max_batch", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32), ("max_write_rows", ctypes.c_int32),
        ("markov_rank", ctypes.c_int32), ("layer_weight_dtype", ctypes.c_int32),
    ]


class dflash_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("ln_in", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ln_post", "w_gate", "w_up", "w_down")]


class dflash_weights(ctypes.Structure):
    _fields_ = [("fc", ctypes.c_void_p), ("hidden_norm", ctypes.c_void_p), ("norm", ctypes.c_void_p),
                ("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("layers", ctypes.POINTER(dflash_layer_weights)),
                ("markov_w1", ctypes.c_void_p), ("markov_w2", ctypes.c_void_p)]


EXPORTS = ("dflash_create", "dflash_destroy", "dflash_write_ctx_kv", "dflash_propose", "dflash_kv_layout",
           "dflash_device_status", "dflash_last_error", "dflash_fp8_lm_head", "dflash_profile",
           "dflash_profile_kinds", "dflash_profile_read", "dflash_gemm_bf16",
           "dflash_attention_check", "dflash_gemm_bf16_noalloc", "dflash_set_persistent", "dflash_persistent",
           "dflash_propose_ex", "dflash_write_ctx_kv_batch", "dflash_fp8_layer")

_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (raises OSError when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} not found: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, c = ctypes.c_void_p, ctypes.c_int32, ctypes
    lib.dflash_create.argtypes = [c.POINTER(dflash_cfg), c.POINTER(dflash_weights), vp, c.POINTER(vp)]
    lib.dflash_create.restype = c.c_int
    lib.dflash_destroy.argtypes = [vp]
    lib.dflash_destroy.restype = c.c_int
    lib.dflash_write_ctx_kv.argtypes = [vp, vp, vp, vp, i32, i32, vp]
    lib.dflash_write_ctx_kv.restype = c.c_int
    lib.dflash_write_ctx_kv_batch.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, vp]
    lib.dflash_write_ctx_kv_batch.restype = c.c_int
    lib.dflash_propose.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp]
    lib.dflash_propose.restype = c.c_int
    lib.dflash_propose_ex.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.dflash_propose_ex.restype = c.c_int
    lib.dflash_kv_layout.argtypes = [vp, c.POINTER(vp), c.POINTER(c.c_size_t), c.POINTER(c.c_int64)]
    lib.dflash_kv_layout.restype = c.c_int
    lib.dflash_device_status.argtypes = [vp, vp, c.POINTER(c.c_uint32)]
    lib.dflash_device_status.restype = c.c_int
    lib.dflash_fp8_lm_head.argtypes = [vp, c.POINTER(vp), c.POINTER(vp)]
    lib.dflash_fp8_lm_head.restype = c.c_int
    lib.dflash_fp8_layer.argtypes = [vp, i32, i32, c.POINTER(vp), c.POINTER(vp)]
    lib.dflash_fp8_layer.restype = c.c_int
    lib.dflash_profile.argtypes = [vp, c.c_int]
    lib.dflash_profile.restype = c.c_int
    lib.dflash_profile_kinds.argtypes = []
    lib.dflash_profile_kinds.restype = c.c_int
    lib.dflash_profile_read.argtypes = [vp, c.c_int, c.POINTER(c.c_char_p), c.POINTER(c.c_double),
                                        c.POINTER(c.c_int64)]
    lib.dflash_profile_read.restype = c.c_int
    lib.dflash_gemm_bf16.argtypes = [vp, i32, i32, vp, i32, vp, i32, vp]
    lib.dflash_gemm_bf16.restype = c.c_int
    lib.dflash_attention_check.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp, vp]
    lib.dflash_attention_check.restype = c.c_int
    lib.dflash_gemm_bf16_noalloc.argtypes = [vp, i32, i32, vp, i32, vp, i32, vp]
    lib.dflash_gemm_bf16_noalloc.restype = c.c_int
    lib.dflash_set_persistent.argtypes = [vp, c.c_int]
    lib.dflash_set_persistent.restype = c.c_int
    lib.dflash_persistent.argtypes = [vp]
    lib.dflash_persistent.restype = c.c_int
    lib.dflash_last_error.argtypes = [vp]
    lib.dflash_last_error.restype = c.c_char_p
    _lib = lib
    return lib


def _check(rc: int, handle) -> None:
    if rc != DFLASH_OK:
        msg = load().dflash_last_error(handle)
        raise DflashError(rc, msg.decode() if msg else "")


def dflash_create(cfg: dflash_cfg, weights: dflash_weights, stream: int = 0) -> int:
    out = ctypes.c_void_p()
    rc = load().dflash_create(ctypes.byref(cfg), ctypes.byref(weights), ctypes.c_void_p(stream), ctypes.byref(out))
    _check(rc, None)
    return out.value


def dflash_destroy(handle: int) -> None:
    _check(load().dflash_destroy(ctypes.c_void_p(handle)), None)


def dflash_write_ctx_kv(handle: int, taps: int, positions: int, page_table: int, first: int, n: int,
                        stream: int = 0) -> None:
    rc = load().dflash_write_ctx_kv(ctypes.c_void_p(handle), ctypes.c_void_p(taps), ctypes.c_void_p(positions),
                                    ctypes.c_void_p(page_table), first, n, ctypes.c_void_p(stream))
    _check(rc, ctypes.c_void_p(handle))


def dflash_write_ctx_kv_batch(handle: int, taps: int, positions: int, row_seq: int, row_index: int,
                              page_tables: int, nseq: int, n: int, stream: int = 0) -> None:
    rc = load().dflash_write_ctx_kv_batch(ctypes.c_void_p(handle), ctypes.c_void_p(taps), ctypes.c_void_p(positions),
                                          ctypes.c_void_p(row_seq), ctypes.c_void_p(row_index),
                                          ctypes.c_void_p(page_tables), nseq, n, ctypes.c_void_p(stream))
    _check(rc, ctypes.c_void_p(handle))


def dflash_propose(handle: int, bonus_tokens: int, ctx_lens: int, page_tables: int, nb: int, max_ctx_len: int,
                   draft_tokens: int, logits: int = 0, final_hidden: int = 0, stream: int = 0) -> None:
    rc = load().dflash_propose(ctypes.c_void_p(handle), ctypes.c_void_p(bonus_tokens), ctypes.c_void_p(ctx_lens),
                               ctypes.c_void_p(page_tables), nb, max_ctx_len, ctypes.c_void_p(draft_tokens),
                               ctypes.c_void_p(logits or None), ctypes.c_void_p(final_hidden or None),
                               ctypes.c_void_p(stream))
    _check(rc, ctypes.c_void_p(handle))


def dflash_propose_ex(handle: int, bonus_tokens: int, ctx_lens: int, page_tables: int, nb: int, max_ctx_len: int,
                      q_rope_pos: int, widths: int, draft_tokens: int, logits: int = 0, final_hidden: int = 0,
                      stream: int = 0) -> None:
    rc = load().dflash_propose_ex(ctypes.c_void_p(handle), ctypes.c_void_p(bonus_tokens), ctypes.c_void_p(ctx_lens),
                                  ctypes.c_void_p(page_tables), nb, max_ctx_len, ctypes.c_void_p(q_rope_pos or None),
                                  ctypes.c_void_p(widths or None), ctypes.c_void_p(draft_tokens),
                                  ctypes.c_void_p(logits or None), ctypes.c_void_p(final_hidden or None),
                                  ctypes.c_void_p(stream))
    _check(rc, ctypes.c_void_p(handle))


def dflash_kv_layout(handle: int) -> Tuple[int, int, Tuple[int, ...]]:
    pool = ctypes.c_void_p()
    nbytes = ctypes.c_size_t()
    strides = (ctypes.c_int64 * 6)()
    _check(load().dflash_kv_layout(ctypes.c_void_p(handle), ctypes.byref(pool), ctypes.byref(nbytes), strides),
           ctypes.c_void_p(handle))
    return pool.value, nbytes.value, tuple(strides)


def dflash_device_status(handle: int, stream: int = 0) -> int:
    """Synchronise, return the device status bits (and clear them)."""
    flags = ctypes.c_uint32()
    rc = load().dflash_device_status(ctypes.c_void_p(handle), ctypes.c_void_p(stream), ctypes.byref(flags))
    if rc not in (DFLASH_OK, DFLASH_EDEVICE):
        _check(rc, ctypes.c_void_p(handle))
    return flags.value


def dflash_last_error(handle: Optional[int]) -> str:
    msg = load().dflash_last_error(ctypes.c_void_p(handle) if handle else None)
    return msg.decode() if msg else ""


def dflash_fp8_lm_head(handle: int) -> Tuple[int, int]:
    """Device pointers of the e4m3 lm_head codes [V, H] and per-row scales [V]."""
    codes, scales = ctypes.c_void_p(), ctypes.c_void_p()
    _check(load().dflash_fp8_lm_head(ctypes.c_void_p(handle), ctypes.byref(codes), ctypes.byref(scales)),
           ctypes.c_void_p(handle))
    return codes.value, scales.value


def dflash_fp8_layer(handle: int, layer: int, proj: int) -> Tuple[int, int]:
    """Device pointers of one FP8 layer projection's e4m3 codes and per-row scales
    (proj 0 qkv, 1 o_proj, 2 gate/up packed, 3 down)."""
    codes, scales = ctypes.c_void_p(), ctypes.c_void_p()
    _check(load().dflash_fp8_layer(ctypes.c_void_p(handle), layer, proj, ctypes.byref(codes), ctypes.byref(scales)),
           ctypes.c_void_p(handle))
    return codes.value, scales.value


def dflash_set_persistent(handle: int, enable: bool) -> None:
    _check(load().dflash_set_persistent(ctypes.c_void_p(handle), 1 if enable else 0), ctypes.c_void_p(handle))


def dflash_persistent(handle: int) -> bool:
    return bool(load().dflash_persistent(ctypes.c_void_p(handle)))


def dflash_profile(handle: int, enable: bool) -> None:
    _check(load().dflash_profile(ctypes.c_void_p(handle), 1 if enable else 0), ctypes.c_void_p(handle))


def dflash_profile_read(handle: int) -> dict:
    """{kernel kind name: (total ms, launches)} since the last dflash_profile call."""
    lib = load()
    out = {}
    for k in range(lib.dflash_profile_kinds()):
        name, ms, n = ctypes.c_char_p(), ctypes.c_double(), ctypes.c_int64()
        _check(lib.dflash_profile_read(ctypes.c_void_p(handle), k, ctypes.byref(name), ctypes.byref(ms),
                                       ctypes.byref(n)), ctypes.c_void_p(handle))
        out[name.value.decode()] = (ms.value, n.value)
    return out


def dflash_gemm_bf16(W: int, N: int, K: int, X: int, M: int, out: int, stream: int = 0) -> None:
    """out[M, N] fp32 = X[M, K] . W[N, K]^T on the tensor-core GEMM (device pointers)."""
    _check(load().dflash_gemm_bf16(ctypes.c_void_p(W), N, K, ctypes.c_void_p(X), M, ctypes.c_void_p(out), 1,
                                   ctypes.c_void_p(stream)), None)


def dflash_attention_check(handle: int, layer: int, ctx_lens: int, page_tables: int, nb: int, max_ctx_len: int,
                           out_cuda_core: int, out_tensor_core: int, stream: int = 0) -> None:
    _check(load().dflash_attention_check(ctypes.c_void_p(handle), layer, ctypes.c_void_p(ctx_lens),
                                         ctypes.c_void_p(page_tables), nb, max_ctx_len,
                                         ctypes.c_void_p(out_cuda_core), ctypes.c_void_p(out_tensor_core),
                                         ctypes.c_void_p(stream)), ctypes.c_void_p(handle))


def dflash_gemm_bf16_noalloc(W: int, N: int, K: int, X: int, M: int, out: int, nsplit: int,
                             stream: int = 0) -> None:
    """Split-K out[M, N] fp32 = X . W^T using the library's fixed device scratch (no
    allocation; calls must not overlap on the GPU)."""
    rc = load().dflash_gemm_bf16_noalloc(ctypes.c_void_p(W), N, K, ctypes.c_void_p(X), M, ctypes.c_void_p(out),
                                         nsplit, ctypes.c_void_p(stream))
    if rc != DFLASH_OK:
        raise DflashError(rc, "dflash_gemm_bf16_noalloc failed")
