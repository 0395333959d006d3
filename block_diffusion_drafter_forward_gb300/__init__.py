"""GB300 (sm_103a) DFlash drafter gamma-block forward behind a C ABI (libdflash.so)."""
from . import _lib  # noqa: F401
from ._lib import (DflashError, dflash_attention_check, dflash_create, dflash_destroy, dflash_device_status,  # noqa: F401
                   dflash_fp8_layer, dflash_fp8_lm_head, dflash_gemm_bf16, dflash_gemm_bf16_noalloc, dflash_kv_layout, dflash_last_error, dflash_profile,
                   dflash_persistent, dflash_profile_read, dflash_propose, dflash_set_persistent, dflash_write_ctx_kv)
from .drafter import Drafter, make_cfg  # noqa: F401
