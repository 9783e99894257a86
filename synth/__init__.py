"""Seeded synthetic inputs for the MoE expert layer (shared by the oracle and
the CUDA path; holds none of the layer's arithmetic).

The workloads stand in, by shape only, for the MoE layers the pages train:
Qwen3-MoE-shaped (128 experts, top-8) and DeepSeek-V3-shaped (256 experts,
top-8, one shared expert).  No dataset or trained weight is used: every tensor
is drawn here from a counter-based SplitMix64 stream keyed by (seed, tensor id).

Recipe (per configuration):
  x        [T, H]      ~ N(0, 1)            -> bf16
  W_r      [H, E]      ~ N(0, 1/H)          -> fp32   (router)
  gate_up  [E*H, 2I]   ~ N(0, 1/H)          -> bf16   (fan_in = H)
  down     [E*I, H]    ~ N(0, 1/I)          -> bf16   (fan_in = I)
  dY       [T, H]      ~ N(0, 1)            -> bf16   (training configs)
  shared gate_up [H, 2Is] ~ N(0, 1/H), shared down [Is, H] ~ N(0, 1/Is)
  skewed routing: bias_e = -s * c * ln(r_e), s = 1.2, r a random permutation
  of 1..E (Zipf-shaped per-expert bias added to the router logits).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None

# Tensor ids of the streams.
TID_X, TID_WR, TID_GATE_UP, TID_DOWN, TID_DY = 1, 2, 3, 4, 5
TID_SH_GATE_UP, TID_SH_DOWN, TID_ZIPF_PERM, TID_IDS = 6, 7, 8, 9


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so (in place) when missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64, dbl, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal_bf16.argtypes = [u64, u64, i64, dbl, p]
        lib.synth_normal_f32.argtypes = [u64, u64, i64, dbl, p]
        lib.synth_permutation.argtypes = [u64, u64, i64, p]
        lib.synth_distinct_ids.argtypes = [u64, u64, i64, ctypes.c_int, ctypes.c_int, p]
        lib.synth_uniform_ints.argtypes = [u64, u64, i64, i64, p]
        for f in (lib.synth_normal_bf16, lib.synth_normal_f32, lib.synth_permutation,
                  lib.synth_distinct_ids, lib.synth_uniform_ints):
            f.restype = None
        _lib = lib
    return _lib


def _out(shape, dtype, out):
    if out is None:
        return np.empty(shape, dtype=dtype)
    assert out.dtype == dtype and out.flags["C_CONTIGUOUS"] and out.size == int(np.prod(shape))
    return out


def normal_bf16(seed, tid, shape, std, out=None) -> np.ndarray:
    """bf16 bits (uint16) of N(0, std^2) draws."""
    a = _out(shape, np.uint16, out)
    _load().synth_normal_bf16(seed, tid, a.size, float(std), a.ctypes.data)
    return a.reshape(shape)


def normal_f32(seed, tid, shape, std, out=None) -> np.ndarray:
    a = _out(shape, np.float32, out)
    _load().synth_normal_f32(seed, tid, a.size, float(std), a.ctypes.data)
    return a.reshape(shape)


def permutation(seed, tid, n) -> np.ndarray:
    a = np.empty(n, dtype=np.int32)
    _load().synth_permutation(seed, tid, n, a.ctypes.data)
    return a


def distinct_ids(seed, tid, T, k, E) -> np.ndarray:
    """[T, k] int32: k distinct experts per row, uniformly drawn."""
    assert 1 <= k <= E <= 4096
    a = np.empty((T, k), dtype=np.int32)
    _load().synth_distinct_ids(seed, tid, T, k, E, a.ctypes.data)
    return a


def uniform_ints(seed, tid, n, m) -> np.ndarray:
    a = np.empty(n, dtype=np.int32)
    _load().synth_uniform_ints(seed, tid, n, m, a.ctypes.data)
    return a


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to fp32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def zipf_bias(seed: int, E: int, c: float, s: float = 1.2) -> np.ndarray:
    """Per-expert router bias -s*c*ln(r_e), r a seeded permutation of 1..E (fp32)."""
    r = permutation(seed, TID_ZIPF_PERM, E).astype(np.float64) + 1.0
    return (-s * c * np.log(r)).astype(np.float32)


@dataclass(frozen=True)
class MoEConfig:
    """One synthetic MoE-layer workload."""
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    seed: int
    I_shared: int = 0          # 0: no shared expert
    skew: bool = False         # Zipf router bias
    train: bool = False        # forward + backward
    description: str = ""

    @property
    def R(self) -> int:
        return self.T * self.k

    def flops_fwd(self) -> float:
        f = 2.0 * self.R * self.H * 2 * self.I + 2.0 * self.R * self.I * self.H
        if self.I_shared:
            f += 2.0 * self.T * self.H * 2 * self.I_shared + 2.0 * self.T * self.I_shared * self.H
        return f


CONFIGS = {
    "tiny": MoEConfig("tiny", T=64, H=128, E=8, k=2, I=64, seed=0,
                      description="tiny MoE layer fwd, T=64 H=128 E=8 k=2 I=64"),
    "qwen3_moe": MoEConfig("qwen3_moe", T=4096, H=2048, E=128, k=8, I=768, seed=1,
                           description="Qwen3-MoE-shaped layer fwd, T=4096 (4x1024) H=2048 E=128 k=8 I=768"),
    "qwen3_moe_skewed": MoEConfig("qwen3_moe_skewed", T=4096, H=2048, E=128, k=8, I=768, seed=2,
                                  skew=True,
                                  description="Qwen3-MoE shape with Zipf(s=1.2) router bias (hotspot + empty experts)"),
    "qwen3_moe_train": MoEConfig("qwen3_moe_train", T=8192, H=2048, E=128, k=8, I=768, seed=3,
                                 train=True,
                                 description="training step fwd+bwd, T=8192 H=2048 E=128 k=8 I=768"),
    "deepseek_v3": MoEConfig("deepseek_v3", T=16384, H=7168, E=256, k=8, I=2048, seed=4,
                             I_shared=2048,
                             description="DeepSeek-V3-shaped layer fwd, T=16384 H=7168 E=256 k=8 I=2048 + shared I=2048"),
}


@dataclass
class MoEInputs:
    cfg: MoEConfig
    x: np.ndarray            # [T, H] bf16 bits
    w_router: np.ndarray     # [H, E] fp32
    bias: np.ndarray | None  # [E] fp32
    gate_up: np.ndarray      # [E*H, 2I] bf16 bits
    down: np.ndarray         # [E*I, H] bf16 bits
    dy: np.ndarray | None = None
    sh_gate_up: np.ndarray | None = None
    sh_down: np.ndarray | None = None
    extra: dict = field(default_factory=dict)


def skew_scale(cfg: MoEConfig) -> float:
    """The calibrated Zipf bias scale c for a skewed configuration, written by
    tests/golden/make_golden.py (which runs only the oracle)."""
    import json
    path = os.path.join(os.path.dirname(_HERE), "tests", "golden", "skew_bias_scale.json")
    with open(path) as f:
        return float(json.load(f)[cfg.name]["c"])


def make_inputs(cfg: MoEConfig, with_dy: bool | None = None, bias_scale: float | None = None,
                weights: bool = True) -> MoEInputs:
    s = cfg.seed
    T, H, E, I = cfg.T, cfg.H, cfg.E, cfg.I
    x = normal_bf16(s, TID_X, (T, H), 1.0)
    wr = normal_f32(s, TID_WR, (H, E), 1.0 / math.sqrt(H))
    bias = None
    if cfg.skew:
        c = skew_scale(cfg) if bias_scale is None else bias_scale
        bias = zipf_bias(s, E, c)
    gu = dn = None
    if weights:
        gu = normal_bf16(s, TID_GATE_UP, (E * H, 2 * I), 1.0 / math.sqrt(H))
        dn = normal_bf16(s, TID_DOWN, (E * I, H), 1.0 / math.sqrt(I))
    dy = None
    if with_dy if with_dy is not None else cfg.train:
        dy = normal_bf16(s, TID_DY, (T, H), 1.0)
    sgu = sdn = None
    if cfg.I_shared and weights:
        sgu = normal_bf16(s, TID_SH_GATE_UP, (H, 2 * cfg.I_shared), 1.0 / math.sqrt(H))
        sdn = normal_bf16(s, TID_SH_DOWN, (cfg.I_shared, H), 1.0 / math.sqrt(cfg.I_shared))
    return MoEInputs(cfg, x, wr, bias, gu, dn, dy, sgu, sdn)
