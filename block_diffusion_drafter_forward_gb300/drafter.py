"""Python handle over the C ABI: keeps the device weights alive (the embedding and the
lm_head are borrowed by the library) and passes torch device buffers as raw pointers.
PyTorch only provides device memory and streams here."""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import torch

from . import _lib as L

_DT = {"f32": L.DFLASH_F32, "bf16": L.DFLASH_BF16, "fp8": L.DFLASH_FP8E4M3_ROWSCALE}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}
LAYER_TENSORS = ("ln_in", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ln_post", "w_gate", "w_up", "w_down")


def make_cfg(cfg, num_pages: int, max_batch: int, max_pages_per_seq: int, max_write_rows: int = 4096) -> L.dflash_cfg:
    """dflash_cfg from a config object carrying the drafter's shape attributes."""
    c = L.dflash_cfg()
    for f in ("hidden", "n_q_heads", "n_kv_heads", "head_dim", "n_ff", "n_layers", "vocab", "gamma",
              "mask_token_id", "n_taps", "target_hidden"):
        setattr(c, f, int(getattr(cfg, f)))
    c.rms_eps = float(cfg.rms_eps)
    c.rope_theta = float(cfg.rope_theta)
    if cfg.yarn is not None:
        c.rope_yarn = 1
        c.yarn_factor, c.yarn_orig_max_pos, c.yarn_beta_fast, c.yarn_beta_slow = (float(v) for v in cfg.yarn)
    c.sliding_window = int(cfg.sliding_window)
    for i, s in enumerate(cfg.layer_sliding or ()):
        c.layer_sliding[i] = 1 if s else 0
    c.dtype = _DT[cfg.dtype]
    c.lm_head_dtype = _DT[cfg.lm_head_dtype]
    c.page_size = int(cfg.page_size)
    c.num_pages = int(num_pages)
    c.max_batch = int(max_batch)
    c.max_pages_per_seq = int(max_pages_per_seq)
    c.max_write_rows = int(max_write_rows)
    c.markov_rank = int(getattr(cfg, "markov_rank", 0))
    c.layer_weight_dtype = _DT[getattr(cfg, "layer_weight_dtype", cfg.dtype)] \
        if getattr(cfg, "layer_weight_dtype", cfg.dtype) == "fp8" else _DT[cfg.dtype]
    return c


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    return (stream or torch.cuda.current_stream()).cuda_stream


def check_tensor(t: torch.Tensor, name: str, dtype: torch.dtype, shape: Tuple[int, ...], min_rows: bool = False,
                 device_type: str = "cuda") -> None:
    """The C ABI takes raw pointers and cannot see sizes or types, so every tensor is checked here
    before its address is passed: a contiguous `dtype` tensor of exactly `shape` (or, with
    `min_rows`, at least shape[0] rows) on a `device_type` device; ValueError otherwise."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.device.type != device_type:
        raise ValueError(f"{name}: expected a {device_type} tensor, got one on {t.device}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    got, want = tuple(t.shape), tuple(shape)
    if len(got) == len(want) and want:
        rows_ok = got[0] >= want[0] if min_rows else got[0] == want[0]
        ok = rows_ok and got[1:] == want[1:]
    else:
        ok = got == want
    if not ok:
        rows = f">={want[0]}" if min_rows and want else ""
        raise ValueError(f"{name}: expected shape {want if not rows else (rows,) + want[1:]}, got {got}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def weight_shapes(cfg) -> Dict[str, Tuple[int, ...]]:
    """Shape of every weight dflash_create reads, HF layout (Linear weights [out, in])."""
    H, F, V, hd = cfg.hidden, cfg.n_ff, cfg.vocab, cfg.head_dim
    qd, kvd = cfg.n_q_heads * hd, cfg.n_kv_heads * hd
    out = {"fc": (H, cfg.n_taps * cfg.target_hidden), "hidden_norm": (H,), "norm": (H,), "embed": (V, H),
           "lm_head": (V, H)}
    layer = {"ln_in": (H,), "wq": (qd, H), "wk": (kvd, H), "wv": (kvd, H), "q_norm": (hd,), "k_norm": (hd,),
             "wo": (H, qd), "ln_post": (H,), "w_gate": (F, H), "w_up": (F, H), "w_down": (H, F)}
    for l in range(cfg.n_layers):
        out.update({f"L{l}.{t}": sh for t, sh in layer.items()})
    R = int(getattr(cfg, "markov_rank", 0))
    if R > 0:
        out.update({"markov_w1": (V, R), "markov_w2": (V, R)})
    return out


class Drafter:
    """One drafter handle.  `tensors` maps fc, hidden_norm, norm, embed, lm_head and
    L{l}.{ln_in, wq, ...} to contiguous device tensors of the config's dtype."""

    def __init__(self, cfg, tensors: Dict[str, torch.Tensor], num_pages: int, max_batch: int,
                 max_pages_per_seq: int, max_write_rows: int = 4096, stream=None):
        self.cfg = cfg
        self.tensors = tensors
        shapes = weight_shapes(cfg)
        missing = [n for n in shapes if n not in tensors]
        if missing:
            raise ValueError(f"missing weight {missing[0]}" + (f" (+{len(missing) - 1} more)" if len(missing) > 1 else ""))
        for name, shape in shapes.items():
            check_tensor(tensors[name], name, self.act_dtype, shape)
        self.ccfg = make_cfg(cfg, num_pages, max_batch, max_pages_per_seq, max_write_rows)
        layers = (L.dflash_layer_weights * cfg.n_layers)()
        for l in range(cfg.n_layers):
            for t in LAYER_TENSORS:
                setattr(layers[l], t, tensors[f"L{l}.{t}"].data_ptr())
        self._layers = layers
        w = L.dflash_weights()
        for t in ("fc", "hidden_norm", "norm", "embed", "lm_head"):
            setattr(w, t, tensors[t].data_ptr())
        if int(getattr(cfg, "markov_rank", 0)) > 0:
            w.markov_w1 = tensors["markov_w1"].data_ptr()
            w.markov_w2 = tensors["markov_w2"].data_ptr()
        w.layers = layers
        self._w = w
        self.handle = L.dflash_create(self.ccfg, w, _stream(stream))

    def close(self) -> None:
        if getattr(self, "handle", None):
            L.dflash_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def act_dtype(self) -> torch.dtype:
        """dtype of the taps, logits and hidden outputs (fp32 drafter: float32, else bfloat16)."""
        return torch.float32 if self.cfg.dtype == "f32" else torch.bfloat16

    def write_ctx_kv(self, taps: torch.Tensor, positions: torch.Tensor, page_table: torch.Tensor, first: int,
                     stream=None) -> None:
        n = int(taps.shape[0]) if taps.dim() >= 1 else -1
        check_tensor(taps, "taps", self.act_dtype, (n, self.cfg.n_taps * self.cfg.target_hidden))
        check_tensor(positions, "positions", torch.int32, (n,))
        check_tensor(page_table, "page_table", torch.int32, (self.ccfg.max_pages_per_seq,))
        L.dflash_write_ctx_kv(self.handle, taps.data_ptr(), positions.data_ptr(), page_table.data_ptr(), first, n,
                              _stream(stream))

    def write_ctx_kv_batch(self, taps: torch.Tensor, positions: torch.Tensor, row_seq: torch.Tensor,
                           row_index: torch.Tensor, page_tables: torch.Tensor, stream=None) -> None:
        """Context rows of several sequences in one call: row i goes to row row_index[i] of
        sequence row_seq[i] (a row of page_tables [nseq, max_pages_per_seq])."""
        n = int(taps.shape[0]) if taps.dim() >= 1 else -1
        check_tensor(taps, "taps", self.act_dtype, (n, self.cfg.n_taps * self.cfg.target_hidden))
        for t, name in ((positions, "positions"), (row_seq, "row_seq"), (row_index, "row_index")):
            check_tensor(t, name, torch.int32, (n,))
        nseq = int(page_tables.shape[0]) if page_tables.dim() == 2 else -1
        check_tensor(page_tables, "page_tables", torch.int32, (nseq, self.ccfg.max_pages_per_seq))
        L.dflash_write_ctx_kv_batch(self.handle, taps.data_ptr(), positions.data_ptr(), row_seq.data_ptr(),
                                    row_index.data_ptr(), page_tables.data_ptr(), nseq, n, _stream(stream))

    def propose(self, bonus: torch.Tensor, ctx_lens: torch.Tensor, page_tables: torch.Tensor, max_ctx_len: int,
                drafts: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                hidden: Optional[torch.Tensor] = None, stream=None, q_rope_pos: Optional[torch.Tensor] = None,
                widths: Optional[torch.Tensor] = None) -> torch.Tensor:
        """One block forward over nb sequences (dflash_propose; dflash_propose_ex when a per-sequence
        RoPE start `q_rope_pos` [nb] or block width `widths` [nb] int32 device tensor is given)."""
        nb = int(bonus.shape[0]) if bonus.dim() == 1 else -1
        g = self.cfg.gamma
        check_tensor(bonus, "bonus", torch.int32, (nb,))
        check_tensor(ctx_lens, "ctx_lens", torch.int32, (nb,))
        check_tensor(page_tables, "page_tables", torch.int32, (nb, self.ccfg.max_pages_per_seq), min_rows=True)
        if drafts is None:
            drafts = torch.empty((nb, g - 1), dtype=torch.int32, device=bonus.device)
        check_tensor(drafts, "drafts", torch.int32, (nb, g - 1))
        if logits is not None:
            check_tensor(logits, "logits", self.act_dtype, (nb * g, self.cfg.vocab))
        if hidden is not None:
            check_tensor(hidden, "hidden", self.act_dtype, (nb * g, self.cfg.hidden))
        if q_rope_pos is None and widths is None:
            L.dflash_propose(self.handle, bonus.data_ptr(), ctx_lens.data_ptr(), page_tables.data_ptr(), nb,
                             int(max_ctx_len), drafts.data_ptr(), logits.data_ptr() if logits is not None else 0,
                             hidden.data_ptr() if hidden is not None else 0, _stream(stream))
            return drafts
        if q_rope_pos is not None:
            check_tensor(q_rope_pos, "q_rope_pos", torch.int32, (nb,))
        if widths is not None:
            check_tensor(widths, "widths", torch.int32, (nb,))
        L.dflash_propose_ex(self.handle, bonus.data_ptr(), ctx_lens.data_ptr(), page_tables.data_ptr(), nb,
                            int(max_ctx_len), q_rope_pos.data_ptr() if q_rope_pos is not None else 0,
                            widths.data_ptr() if widths is not None else 0, drafts.data_ptr(),
                            logits.data_ptr() if logits is not None else 0,
                            hidden.data_ptr() if hidden is not None else 0, _stream(stream))
        return drafts

    def set_persistent(self, enable: bool) -> None:
        L.dflash_set_persistent(self.handle, enable)

    @property
    def persistent(self) -> bool:
        return L.dflash_persistent(self.handle)

    def kv_layout(self) -> Tuple[int, int, Tuple[int, ...]]:
        return L.dflash_kv_layout(self.handle)

    def device_status(self, stream=None) -> int:
        return L.dflash_device_status(self.handle, _stream(stream))
