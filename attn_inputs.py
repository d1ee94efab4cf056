"""Seeded synthetic inputs for the attention forward workloads.

This module is the only code shared by the CPU oracle and the CUDA path. It
draws random numbers and converts them to the dtype the kernel reads; it holds
none of the attention arithmetic.

Recipe (the same for every workload):
  * ``numpy.random.default_rng(seed)`` (seed 0 unless stated), drawing Q, then
    K, then V as float32 arrays of shape [B, H, N, d] with ``standard_normal``
    multiplied by the stated standard deviation. This follows the exactness test
    on "Lecture 2 - Online Softmax and Numerical Correctness", section "Build
    it", which draws Q, K, V from ``default_rng(0).standard_normal``.
  * bf16 workloads round the float32 draws to bfloat16 (round to nearest even,
    done by ``torch.Tensor.to``). The oracle then reads those bf16 values widened
    to float64, so both sides see identical inputs.
  * The MXFP8 workload keeps the float32 draws; each side quantises them itself.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    qk_std: float = 1.0
    v_std: float = 1.0
    dtype: str = "bf16"  # "bf16" or "mxfp8"
    seed: int = 0
    direction: str = "fwd"  # "fwd", or "bwd" for the backward pass

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4*B*H*N^2*d, halved for causal (the counting convention of the task);
        the backward's five products count 2.5 times that."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        if self.direction == "bwd":
            f *= 2.5
        return f / 2.0 if self.causal else f

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "B": self.B,
            "H": self.H,
            "N": self.N,
            "d": self.d,
            "causal": self.causal,
            "qk_std": self.qk_std,
            "v_std": self.v_std,
            "dtype": self.dtype,
            "seed": self.seed,
            "pass": self.direction,
        }


# The five workloads: a tiny one the oracle finishes at once, three bf16
# long-sequence ones and the block-scaled FP8 one.
TINY = Workload("tiny_b1h2n256d64", 1, 2, 256, 64, False)
NONCAUSAL_D128 = Workload("bf16_b4h16n4096d128", 4, 16, 4096, 128, False)
CAUSAL_D128_WIDE = Workload("bf16_causal_b2h16n8192d128_qk2", 2, 16, 8192, 128, True, qk_std=2.0)
CAUSAL_D64 = Workload("bf16_causal_b8h16n4096d64", 8, 16, 4096, 64, True)
MXFP8_CAUSAL = Workload("mxfp8_causal_b2h16n16384d128", 2, 16, 16384, 128, True, dtype="mxfp8")

# The backward pass on the two d = 128 shapes (dO from draw_grad; O and LSE
# from the forward).
BWD_D128 = Workload("bwd_bf16_b4h16n4096d128", 4, 16, 4096, 128, False, direction="bwd")
BWD_CAUSAL_D128 = Workload("bwd_bf16_causal_b2h16n8192d128_qk2", 2, 16, 8192, 128, True, qk_std=2.0,
                           direction="bwd")

# The MXFP8 backward (fp32 Q, K, V, dO quantised inside the step) on the bf16
# backward's non-causal shape and on the MXFP8 forward's causal one.
BWD_MXFP8 = Workload("bwd_mxfp8_b4h16n4096d128", 4, 16, 4096, 128, False, dtype="mxfp8", direction="bwd")
BWD_MXFP8_CAUSAL = Workload("bwd_mxfp8_causal_b2h16n16384d128", 2, 16, 16384, 128, True, dtype="mxfp8",
                            direction="bwd")

WORKLOADS = {w.name: w for w in (TINY, NONCAUSAL_D128, CAUSAL_D128_WIDE, CAUSAL_D64, MXFP8_CAUSAL, BWD_D128,
                                 BWD_CAUSAL_D128, BWD_MXFP8, BWD_MXFP8_CAUSAL)}


def draw_fp32(B: int, H: int, N: int, d: int, qk_std: float = 1.0, v_std: float = 1.0,
              seed: int = 0) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Q, K, V as float32 [B,H,N,d], drawn in that order from one generator."""
    rng = np.random.default_rng(seed)
    shape = (B, H, N, d)
    q = rng.standard_normal(shape, dtype=np.float32)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    if qk_std != 1.0:
        q *= np.float32(qk_std)
        k *= np.float32(qk_std)
    if v_std != 1.0:
        v *= np.float32(v_std)
    return q, k, v


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """float32 numpy -> bfloat16 CPU tensor, round to nearest even."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def bf16_qkv(w: Workload) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """The bf16 CPU tensors the kernel reads for a bf16 workload."""
    q, k, v = draw_fp32(w.B, w.H, w.N, w.d, w.qk_std, w.v_std, w.seed)
    return to_bf16(q), to_bf16(k), to_bf16(v)


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Widen a CPU tensor (bf16, fp32, ...) to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def uniform_fp32(n: int, lo: float, hi: float, seed: int = 0) -> np.ndarray:
    """n float32 values uniform on [lo, hi), used for the exp2 accuracy sweeps."""
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=n).astype(np.float32)


def rescale_scores(kind: str, rows: int = 256, keys: int = 8192, seed: int = 0) -> np.ndarray:
    """Synthetic score rows in log2 units for the rescale-rate table of
    "FlashAttention-4's Softmax Tricks", section "Conditional rescaling":
    ``iid1.5`` and ``iid6`` are N(0, 1.5^2) and N(0, 6^2); ``rise24`` and
    ``rise96`` are N(0, 1.5^2) noise plus a linear ramp from 0 to 24 (or 96)
    across the key order. The page does not state the noise of the ramp rows;
    N(0, 1.5^2) is the reading taken here."""
    rng = np.random.default_rng(seed)
    noise = rng.standard_normal((rows, keys))
    if kind == "iid1.5":
        return 1.5 * noise
    if kind == "iid6":
        return 6.0 * noise
    if kind in ("rise24", "rise96"):
        top = 24.0 if kind == "rise24" else 96.0
        return 1.5 * noise + np.linspace(0.0, top, keys)[None, :]
    raise ValueError(kind)


def fp8_sim_values(keys: int = 8192, d: int = 64, seed: int = 1) -> np.ndarray:
    """V [keys, d] for the P-in-FP8 error table of "FlashAttention-4's Softmax
    Tricks", section "Where 'exact' breaks: P in FP8": the page does not state
    V or d; iid N(0, 1) values and d = 64 are the reading taken here."""
    return np.random.default_rng(seed).standard_normal((keys, d))


def draw_grad(B: int, H: int, N: int, d: int, seed: int = 1) -> np.ndarray:
    """An upstream gradient dO for the backward pass: float32 [B,H,N,d]
    standard normals from its own generator (the pages state no recipe for it)."""
    return np.random.default_rng(seed).standard_normal((B, H, N, d), dtype=np.float32)

