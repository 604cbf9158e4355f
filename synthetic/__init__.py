"""Seeded synthetic inputs for the attention forward pass.

This module only draws numbers; it holds none of the attention arithmetic.
It serves both the fp64 oracle (``oracle/``) and the CUDA path, which
consume the same host-generated bf16 bit patterns.

The generator (``synth.c``) is a counter-based splitmix64 stream turned into
standard normals by the Box-Muller transform in double precision and rounded
float64 -> float32 -> bfloat16, each step round-to-nearest-even.  Tensors are
returned as ``numpy.uint16`` arrays of bf16 bit patterns.

Workload recipes (shapes, seeds and value distributions) follow the pages'
benchmark grid: sequence lengths 1k-32k at 32k total tokens, 16 heads of 128
(hidden 2048), head dims 64, 128 and (192, 128), MHA / GQA / MQA
(FlashAttention-4 wiki summary, "Benchmark setting" under Experiments and
results).  No dataset is involved.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libsynth.so")
_lib = None

# stream ids per tensor
STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the generator with gcc into ``synthetic/_build/libsynth.so``."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_double, ctypes.c_int]
        lib.synth_normal_bf16.restype = ctypes.c_int
        lib.synth_normal_offset_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                                 ctypes.c_uint64, ctypes.c_double, ctypes.c_double,
                                                 ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
        lib.synth_normal_offset_bf16.restype = ctypes.c_int
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(shape, seed: int, stream: int, mul: float = 1.0) -> np.ndarray:
    """bf16 bits of ``mul * N(0, 1)`` i.i.d. draws, C-contiguous ``shape``."""
    out = np.empty(tuple(int(s) for s in shape), dtype=np.uint16)
    if out.size:
        rc = _load().synth_normal_bf16(out.ctypes.data, out.size, seed, stream, float(mul), _threads())
        assert rc == 0
    return out


def normal_offset_bf16(shape, seed: int, stream: int, mul: float, off_max: float) -> np.ndarray:
    """bf16 bits of ``mul * N(0,1) + off_max * j / (S - 1)`` for a ``[B, S, H, D]``
    tensor, j the sequence index (axis 1); the offset is added before rounding."""
    b, s, h, d = (int(x) for x in shape)
    out = np.empty((b, s, h, d), dtype=np.uint16)
    if out.size:
        rc = _load().synth_normal_offset_bf16(out.ctypes.data, out.size, seed, stream, float(mul),
                                              float(off_max), h * d, s, _threads())
        assert rc == 0
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bit patterns (nearest even); for building
    hand-made test inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if np.any(nan):
        r[nan] = 0x7FC0
    return r


@dataclass
class Workload:
    """One attention problem: shapes, mask, scale and the input recipe."""
    name: str
    batch: int
    heads_q: int
    heads_kv: int
    seqlen_q: int
    seqlen_k: int
    d_qk: int
    d_v: int
    causal: bool
    seed: int
    q_mul: float = 1.0
    k_offset: float = 0.0      # per-key offset rising linearly 0 -> k_offset along the sequence
    scale: float | None = None  # None: 1 / sqrt(d_qk)
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / float(np.sqrt(self.d_qk))

    @property
    def shapes(self):
        return dict(q=(self.batch, self.seqlen_q, self.heads_q, self.d_qk),
                    k=(self.batch, self.seqlen_k, self.heads_kv, self.d_qk),
                    v=(self.batch, self.seqlen_k, self.heads_kv, self.d_v),
                    o=(self.batch, self.seqlen_q, self.heads_q, self.d_v),
                    lse=(self.batch, self.heads_q, self.seqlen_q))

    def flops(self) -> float:
        """2*B*Hq*Sq*Sk*(d_qk + d_v), halved for causal (nominal convention)."""
        f = 2.0 * self.batch * self.heads_q * self.seqlen_q * self.seqlen_k * (self.d_qk + self.d_v)
        return f / 2 if self.causal else f

    def algorithmic_bytes(self) -> int:
        """Q, K, V read once; O (bf16) and LSE (fp32) written once."""
        s = self.shapes
        n = lambda t: int(np.prod(t))
        return 2 * (n(s["q"]) + n(s["k"]) + n(s["v"]) + n(s["o"])) + 4 * n(s["lse"])

    def generate(self):
        """(q, k, v) bf16 bit arrays in BSHD layout."""
        s = self.shapes
        q = normal_bf16(s["q"], self.seed, STREAM_Q, self.q_mul)
        if self.k_offset:
            k = normal_offset_bf16(s["k"], self.seed, STREAM_K, 1.0, self.k_offset)
        else:
            k = normal_bf16(s["k"], self.seed, STREAM_K, 1.0)
        v = normal_bf16(s["v"], self.seed, STREAM_V, 1.0)
        return q, k, v


CAUSAL_SWEEP = (1024, 2048, 4096, 8192, 16384, 32768)


def workloads() -> dict:
    """The five benchmark configurations (the causal sweep expands to six)."""
    w = {}
    w["tiny"] = Workload("tiny", 1, 1, 1, 128, 128, 64, 64, False, seed=0,
                         notes="B1 H1 S128 d64 non-causal")
    w["mha8k"] = Workload("mha8k", 4, 16, 16, 8192, 8192, 128, 128, False, seed=1,
                          notes="B4 H16 S8192 d128 non-causal (32k tokens)")
    for s in CAUSAL_SWEEP:
        w[f"causal{s // 1024}k"] = Workload(f"causal{s // 1024}k", 32768 // s, 16, 16, s, s, 128, 128,
                                            True, seed=3000 + s // 1024,
                                            notes=f"B{32768 // s} H16 S{s} d128 causal")
    w["gqa"] = Workload("gqa", 4, 32, 8, 8192, 8192, 128, 128, True, seed=3,
                        notes="B4 S8192 Hq32 Hkv8 d128 causal")
    w["mqa"] = Workload("mqa", 4, 32, 1, 8192, 8192, 128, 128, True, seed=30,
                        notes="B4 S8192 Hq32 Hkv1 d128 causal")
    # smaller case of the MHA kernel for detailed profiling (inputs still > L2)
    w["prof_mha"] = Workload("prof_mha", 2, 16, 16, 8192, 8192, 128, 128, False, seed=101,
                             notes="B2 H16 S8192 d128 non-causal (profiling case)")
    w["asym"] = Workload("asym", 2, 16, 16, 16384, 16384, 192, 128, True, seed=4, q_mul=4.0,
                         k_offset=12.0,
                         notes="B2 H16 S16384 d_qk192 d_v128 causal, Q=4N(0,1), K=N(0,1)+0..12")
    return w


# ---------------------------------------------------------------------------
# variable-length batches (sequences packed back to back)
# ---------------------------------------------------------------------------

@dataclass
class VarlenWorkload:
    """A variable-length batch: per-sequence query and key counts, the shared
    heads / head dims / mask, and the input recipe (N(0,1) bf16 from seed)."""
    name: str
    seqlens_q: tuple
    seqlens_k: tuple
    heads_q: int
    heads_kv: int
    d_qk: int
    d_v: int
    causal: bool
    seed: int
    scale: float | None = None
    notes: str = ""

    @property
    def batch(self) -> int:
        return len(self.seqlens_q)

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens_q)]).astype(np.int32)

    @property
    def cu_seqlens_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens_k)]).astype(np.int32)

    @property
    def total_q(self) -> int:
        return int(sum(self.seqlens_q))

    @property
    def total_k(self) -> int:
        return int(sum(self.seqlens_k))

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / float(np.sqrt(self.d_qk))

    @property
    def shapes(self):
        return dict(q=(self.total_q, self.heads_q, self.d_qk), k=(self.total_k, self.heads_kv, self.d_qk),
                    v=(self.total_k, self.heads_kv, self.d_v), o=(self.total_q, self.heads_q, self.d_v),
                    lse=(self.heads_q, self.total_q))

    def flops(self) -> float:
        """Sum over sequences of 2*Hq*sq*sk*(d_qk + d_v), halved for causal."""
        f = sum(2.0 * self.heads_q * sq * sk * (self.d_qk + self.d_v) for sq, sk in zip(self.seqlens_q,
                                                                                        self.seqlens_k))
        return f / 2 if self.causal else f

    def algorithmic_bytes(self) -> int:
        s = self.shapes
        n = lambda t: int(np.prod(t))
        return 2 * (n(s["q"]) + n(s["k"]) + n(s["v"]) + n(s["o"])) + 4 * n(s["lse"])

    def generate(self):
        """(q, k, v) bf16 bit arrays, packed [total, heads, d]."""
        s = self.shapes
        return (normal_bf16(s["q"], self.seed, STREAM_Q, 1.0), normal_bf16(s["k"], self.seed, STREAM_K, 1.0),
                normal_bf16(s["v"], self.seed, STREAM_V, 1.0))


def loguniform_lengths(total: int, lo: int, hi: int, seed: int) -> tuple:
    """Sequence lengths drawn log-uniformly in [lo, hi] (numpy PCG64, seeded)
    until they hold `total` tokens; the last one is cut to fit exactly."""
    rng = np.random.default_rng(seed)
    out, left = [], total
    while left > 0:
        n = int(round(float(np.exp(rng.uniform(np.log(lo), np.log(hi))))))
        n = min(max(n, lo), hi, left)
        out.append(n)
        left -= n
    return tuple(out)


def varlen_workloads() -> dict:
    """Variable-length batches at the benchmark grid's 32k total tokens, 16
    heads of 128 (lengths 128..8192, log-uniform), causal and non-causal."""
    lens = loguniform_lengths(32768, 128, 8192, seed=41)
    w = {}
    w["varlen32k"] = VarlenWorkload("varlen32k", lens, lens, 16, 16, 128, 128, True, seed=41,
                                    notes=f"{len(lens)} sequences, 32768 tokens, lengths 128..8192 log-uniform, "
                                          "H16 d128 causal")
    w["varlen32k_nc"] = VarlenWorkload("varlen32k_nc", lens, lens, 16, 16, 128, 128, False, seed=42,
                                       notes=f"{len(lens)} sequences, 32768 tokens, lengths 128..8192 "
                                             "log-uniform, H16 d128 non-causal")
    return w


def decode_workloads() -> dict:
    """Decode-shaped problems (few queries against a long K/V cache), the
    split-KV path's workloads.  K/V is read once, so they are HBM-bound."""
    w = {}
    w["decode32k"] = Workload("decode32k", 8, 32, 8, 1, 32768, 128, 128, False, seed=51,
                              notes="B8 Hq32 Hkv8 Sq1 Sk32768 d128 (one query per sequence, 32k-key cache)")
    w["decode_mqa"] = Workload("decode_mqa", 32, 32, 1, 1, 16384, 128, 128, False, seed=52,
                               notes="B32 Hq32 Hkv1 Sq1 Sk16384 d128 (MQA decode)")
    w["specdec"] = Workload("specdec", 8, 32, 8, 4, 16384, 128, 128, True, seed=53,
                            notes="B8 Hq32 Hkv8 Sq4 Sk16384 d128 causal (4 draft tokens)")
    # smaller case of the split-KV kernel for detailed profiling (K/V still > L2)
    w["prof_decode"] = Workload("prof_decode", 4, 32, 8, 1, 16384, 128, 128, False, seed=54,
                                notes="B4 Hq32 Hkv8 Sq1 Sk16384 d128 (decode profiling case)")
    return w
