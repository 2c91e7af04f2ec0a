"""Shared set-up of the GPU parity tests: the same seeded inputs feed the CUDA
path (through the Python binding of the C ABI) and the CPU oracle."""
import math

import numpy as np
import torch

import workloads as wl


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def widen(a: np.ndarray, cfg) -> np.ndarray:
    """fp32 view of an activation array (bf16 bits widened exactly)."""
    return a if cfg.fp32 else wl.bf16_bits_to_f32(a)


def act_dev(a: np.ndarray, cfg) -> torch.Tensor:
    return dev(a) if cfg.fp32 else dev_bf16(a)


def softmax_scale(cfg) -> float:
    return 1.0 / math.sqrt(cfg.D)


def max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(got.astype(np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))


# tolerances stated by the target: max |err| <= 1e-2 max |ref| for bf16 outputs
# with fp32 accumulation, 1e-5 on the fp32 configuration
def tol(cfg) -> float:
    return 1e-5 if cfg.fp32 else 1e-2
