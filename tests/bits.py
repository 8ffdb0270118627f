"""bf16 <-> raw-bit helpers shared by the tests (no method arithmetic)."""
import numpy as np
import torch


def to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor (any device) -> numpy uint16 raw bits."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 raw bits -> bf16 torch tensor (CPU)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def bits_to_f32(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, dtype=np.uint32) << 16).view(np.float32)


def bits_to_f64(a: np.ndarray) -> np.ndarray:
    return bits_to_f32(a).astype(np.float64)


def popcount32(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, dtype=np.uint32)
    return np.unpackbits(a.view(np.uint8).reshape(a.shape + (4,)), axis=-1).sum(axis=-1)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits): 2^(floor(log2|v|) - 7)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 7).astype(np.int64))
