"""Seeded synthetic inputs for the bitmask N:M decode SpMV.

This module only draws random numbers and lays them out. It contains none of
the method's arithmetic: no N:M selection, no packing and no products. Both the
CUDA path (through the tests and the benchmark) and the CPU oracle take their
inputs from here, so neither has to import the other.

Distributions follow the synthetic stand-in for the pages' models
(SparseDecoding, "Decoding-Aware Pruning for Accurate and Efficient LLM
Inference"; the workloads are Llama-3.1-8B / Llama-3.3-70B / Qwen3-14B/32B
shaped linears, whose trained weights are not available):

* ``W``  : bf16_rn(N(0, 0.02^2)), row-major ``[rows][K]``.
* ``a``  : fp32 |N(1, 0.3^2)|, one per input column: a stand-in for the
  per-column activation norm sqrt(sum_t X_jt^2) of the Wanda score
  (daiwk.github.io notes on SparseDecoding, section "核心公式").
* ``x``  : bf16_rn(N(0, 1)), ``[batch][K]``.

Random numbers come from torch's own generators, seeded per tensor. A CPU
generator gives the same stream on every host; a CUDA generator gives a
different (but seeded, repeatable) stream and is used for sizes too large to
draw on the host. Tests that compare against the oracle either draw on the CPU
or copy the device draws back.
"""
from __future__ import annotations

import torch

# Matrix ids inside one decoder layer and tensor ids inside one matrix.
MATRICES = ("qkv", "o", "gate_up", "down")
TENSORS = ("W", "a", "x")


def stream_id(config: int, layer: int, matrix: int, tensor: int) -> int:
    """Stable stream id for (config, layer, matrix, tensor).

    The N:M pattern is deliberately not part of the key, so every pattern
    prunes the same dense W.
    """
    return ((config * 4096 + layer) * 8 + matrix) * 4 + tensor


def _generator(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 0x9E3779B1 + int(stream)) % (2**63))
    return g


def weights(rows: int, K: int, seed: int = 0, stream: int = 0, device="cpu") -> torch.Tensor:
    """Dense bf16 weights ~ N(0, 0.02^2), rounded to nearest even."""
    g = _generator(seed, stream, device)
    z = torch.randn(rows, K, generator=g, device=device, dtype=torch.float32)
    return z.mul_(0.02).to(torch.bfloat16)


def col_norms(K: int, seed: int = 0, stream: int = 1, device="cpu") -> torch.Tensor:
    """Per-input-column activation-norm stand-in, fp32 |N(1, 0.3^2)|."""
    g = _generator(seed, stream, device)
    z = torch.randn(K, generator=g, device=device, dtype=torch.float32)
    return z.mul_(0.3).add_(1.0).abs_()


def activations(batch: int, K: int, seed: int = 0, stream: int = 2, device="cpu") -> torch.Tensor:
    """Decode-step inputs x ~ N(0, 1) in bf16, ``[batch][K]``."""
    g = _generator(seed, stream, device)
    z = torch.randn(batch, K, generator=g, device=device, dtype=torch.float32)
    return z.to(torch.bfloat16)


def random_nm_keep(rows: int, K: int, N: int, M: int, seed: int = 0, stream: int = 3,
                   device="cpu") -> torch.Tensor:
    """Boolean ``[rows][K]`` with exactly N True entries in every aligned M-column
    subgroup, positions drawn uniformly at random (a structure generator, not the
    selection rule)."""
    g = _generator(seed, stream, device)
    keys = torch.rand(rows, K // M, M, generator=g, device=device)
    order = keys.argsort(dim=-1)
    keep = torch.zeros(rows, K // M, M, dtype=torch.bool, device=device)
    keep.scatter_(-1, order[..., :N], True)
    return keep.reshape(rows, K)


def dyadic_values(rows: int, K: int, seed: int = 0, stream: int = 4, device="cpu") -> torch.Tensor:
    """bf16 values drawn from {+-1, +-0.5, +-0.25}: products with small integers
    are exact in fp32 and every partial sum is representable."""
    g = _generator(seed, stream, device)
    mag = torch.randint(0, 3, (rows, K), generator=g, device=device)
    sign = torch.randint(0, 2, (rows, K), generator=g, device=device) * 2 - 1
    return (sign.float() * torch.pow(2.0, -mag.float())).to(torch.bfloat16)


def small_int_activations(batch: int, K: int, seed: int = 0, stream: int = 5,
                          device="cpu") -> torch.Tensor:
    """x in {-2, -1, 0, 1, 2} as bf16."""
    g = _generator(seed, stream, device)
    return (torch.randint(-2, 3, (batch, K), generator=g, device=device)).to(torch.bfloat16)


def nm_structured(rows: int, K: int, N: int, M: int, seed: int = 0, dyadic: bool = False,
                  device="cpu") -> torch.Tensor:
    """A dense bf16 matrix that already satisfies N:M: random kept positions,
    kept values nonzero (normal or dyadic), zeros elsewhere."""
    keep = random_nm_keep(rows, K, N, M, seed=seed, device=device)
    if dyadic:
        vals = dyadic_values(rows, K, seed=seed, device=device)
    else:
        vals = weights(rows, K, seed=seed, stream=6, device=device)
        # a kept weight that rounds to zero would make the pattern ambiguous
        vals = torch.where(vals == 0, torch.full_like(vals, 0.015625), vals)
    return torch.where(keep, vals, torch.zeros_like(vals))


# --- workload shapes (rows x K per linear) -------------------------------------

# Llama-3.1-8B decoder layer: qkv, o, gate_up, down.
LLAMA31_8B = {"qkv": (6144, 4096), "o": (4096, 4096), "gate_up": (28672, 4096),
              "down": (4096, 14336), "layers": 32}
QWEN3_14B = {"qkv": (7168, 5120), "o": (5120, 5120), "gate_up": (34816, 5120),
             "down": (5120, 17408), "layers": 40}
QWEN3_32B = {"qkv": (10240, 5120), "o": (5120, 8192), "gate_up": (51200, 5120),
             "down": (5120, 25600), "layers": 64}
LLAMA33_70B = {"qkv": (10240, 8192), "o": (8192, 8192), "gate_up": (57344, 8192),
               "down": (8192, 28672), "layers": 80}
SINGLE_4096 = {"o": (4096, 4096), "layers": 1}

MODELS = {"llama3.1-8b": LLAMA31_8B, "qwen3-14b": QWEN3_14B, "qwen3-32b": QWEN3_32B,
          "llama3.3-70b": LLAMA33_70B}

PATTERNS = ((2, 4), (4, 8), (8, 16), (16, 32))

# Rows of the q and of the k projection inside each model's fused qkv matrix
# (q rows first, then k, then v with as many rows as k).
QKV_SPLIT = {"llama3.1-8b": (4096, 1024), "qwen3-14b": (5120, 1024), "qwen3-32b": (8192, 1024),
             "llama3.3-70b": (8192, 1024)}


def calibration(T: int, K: int, seed: int = 0, stream: int = 5, dead=(), device="cpu") -> torch.Tensor:
    """Calibration inputs X for one linear layer, bf16 ``[T][K]`` (token-major).

    x_tj = s_j * z_tj with z ~ N(0, 1) and per-channel scales s_j ~ |N(1, 0.3^2)|,
    every 64th channel scaled up 8x (a stand-in for the few large-magnitude
    input channels of LLM activations). Channels listed in ``dead`` are zero in
    every token (the case of an input that never fires)."""
    g = _generator(seed, stream, device)
    s = torch.randn(K, generator=g, device=device, dtype=torch.float32).mul_(0.3).add_(1.0).abs_()
    s[::64] *= 8.0
    if len(dead):
        s[torch.as_tensor(list(dead), device=device)] = 0.0
    z = torch.randn(T, K, generator=g, device=device, dtype=torch.float32)
    return (z * s).to(torch.bfloat16)
