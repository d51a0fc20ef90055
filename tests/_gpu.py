"""Helpers for the GPU parity tests: host bf16 bits <-> device tensors."""
import numpy as np
import torch


def dev(bits, device="cuda"):
    """numpy uint16 bf16 patterns (or float32) -> CUDA tensor with the same bits."""
    a = np.ascontiguousarray(bits)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def host(t):
    """CUDA bf16 tensor -> numpy uint16 bit patterns (logical element order)."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def stat_report(got, want, rtol=1e-5):
    """Fraction bit-identical and the worst relative difference of fp32 stats."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    both_nan = np.isnan(got) & np.isnan(want)
    same = (got == want) | both_nan
    with np.errstate(invalid="ignore", divide="ignore"):
        rel = np.where(same, 0.0, np.abs(got - want) / np.maximum(np.abs(want), 1e-30))
    return float(same.mean()) if same.size else 1.0, float(rel.max()) if rel.size else 0.0
