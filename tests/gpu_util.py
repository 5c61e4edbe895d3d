"""Helpers shared by the GPU tests: moving fp16 bit patterns between numpy
(where the generator and the oracle live) and CUDA tensors (where the
library runs), plus the workload shapes."""
from __future__ import annotations

import numpy as np

PATTERNS = [(2, 4), (4, 8), (8, 16), (16, 32)]

# The decode-layer workloads (rows x cols = out x in), with their patterns.
WORKLOADS = {
    "single_4096": {"mats": {"W": (4096, 4096)}, "patterns": [(2, 4)]},
    "llama31_8b_layer": {"mats": {"qkv": (6144, 4096), "o": (4096, 4096),
                                  "gate_up": (28672, 4096), "down": (4096, 14336)},
                         "patterns": [(2, 4)]},
    "pattern_sweep": {"mats": {"up": (14336, 4096), "down": (4096, 14336)},
                      "patterns": PATTERNS},
    "qwen3_32b_layer": {"mats": {"qkv": (10240, 5120), "o": (5120, 8192),
                                 "gate_up": (51200, 5120), "down": (5120, 25600)},
                        "patterns": [(2, 4), (16, 32)]},
    "llama33_70b_layer": {"mats": {"qkv": (10240, 8192), "o": (8192, 8192),
                                   "gate_up": (57344, 8192), "down": (8192, 28672)},
                          "patterns": PATTERNS},
}


def to_dev(a: np.ndarray, device="cuda"):
    """uint16 fp16 bit patterns -> CUDA fp16 tensor (same bits)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(torch.float16)


def from_dev(t) -> np.ndarray:
    """CUDA fp16 / int32 tensor -> numpy uint16 / uint32 with the same bits."""
    import torch
    c = t.detach().cpu()
    if c.dtype == torch.float16:
        return c.view(torch.int16).numpy().view(np.uint16)
    if c.dtype == torch.int32:
        return c.numpy().view(np.uint32)
    raise TypeError(c.dtype)


def f16_to_f64(a: np.ndarray) -> np.ndarray:
    return a.view(np.float16).astype(np.float64)
