"""Move seeded numpy inputs onto a torch device (bit-exact transport, no arithmetic)."""
import numpy as np
import torch


def to_torch(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (uint16) -> torch.bfloat16, float32 -> torch.float32, ints as is."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    elif dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def from_torch(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> numpy (bf16 as uint16 bit patterns)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def upload_weights(weights, device="cuda", keep_host: bool = False):
    """All drafter tensors of a synth Weights object as device tensors (drawn one at a
    time so the host never holds all of them unless keep_host)."""
    out = {}
    for name in weights.names():
        out[name] = to_torch(weights.get(name, keep=keep_host), weights.cfg.dtype, device)
    return out
