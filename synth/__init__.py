"""Seeded synthetic inputs for the frame step: model shapes, weights and token streams.

This module holds no frame-step arithmetic.  It says what to draw (tensor names,
shapes, distributions, the five workload recipes) and draws it with the
counter-based Philox4x32-10 generator in ``synth.c``.  The CUDA library and the
CPU oracle both consume the host arrays it returns, so both sides see the same
bits.

Workload shapes come from the Moshi/PersonaPlex pages: the temporal transformer
is 4096-d / 32 layers / 32 heads with a 3000-frame ring window (vLLM-Omni
PersonaPlex recipe, "Architecture"), the depformer is 1024-d / 6 layers /
16 heads with 16 per-substep weight sets (mobius PR #368, "P2 - Moshi LM"), and
the per-codebook delays are [0, 0, 1 x 7, 0, 1 x 7] (mobius PR #368, "P3 -
ONNX Runtime example").
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Dict, List, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None

# Per-codebook delays: text row, agent semantic, 7 agent acoustic, user semantic, 7 user acoustic.
DELAYS: Tuple[int, ...] = (0, 0, 1, 1, 1, 1, 1, 1, 1, 0, 1, 1, 1, 1, 1, 1, 1)
N_STREAMS = 17


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, u32, i64 = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64
        vp = ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u32, u64, i64, ctypes.c_float, ctypes.c_float, vp]
        lib.synth_normal_bf16.argtypes = [u64, u32, u64, i64, ctypes.c_float, ctypes.c_float, vp]
        lib.synth_uniform_int.argtypes = [u64, u32, u64, i64, ctypes.c_int32, ctypes.c_int32, vp]
        lib.synth_philox4x32_10.argtypes = [vp, vp, vp]
        lib.synth_bf16_to_f32.argtypes = [vp, i64, vp]
        _lib = lib
    return _lib


def philox4x32_10(ctr, key) -> Tuple[int, int, int, int]:
    c = (ctypes.c_uint32 * 4)(*ctr)
    k = (ctypes.c_uint32 * 2)(*key)
    o = (ctypes.c_uint32 * 4)()
    _load().synth_philox4x32_10(c, k, o)
    return tuple(int(v) for v in o)


def normal_f32(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0,
               offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    out = np.empty(n, np.float32) if out is None else out
    assert out.dtype == np.float32 and out.size == n and out.flags.c_contiguous
    _load().synth_normal_f32(seed, stream, offset, n, mean, std, out.ctypes.data)
    return out


def normal_bf16(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0,
                offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(mean, std) draws rounded to nearest even."""
    out = np.empty(n, np.uint16) if out is None else out
    assert out.dtype == np.uint16 and out.size == n and out.flags.c_contiguous
    _load().synth_normal_bf16(seed, stream, offset, n, mean, std, out.ctypes.data)
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_uniform_int(seed, stream, offset, n, lo, hi, out.ctypes.data)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float32)
    _load().synth_bf16_to_f32(bits.ctypes.data, bits.size, out.ctypes.data)
    return out


# ----------------------------------------------------------------------------- shapes


@dataclasses.dataclass(frozen=True)
class Shape:
    """Model shape and run limits of one workload."""
    d: int
    n_layers: int
    n_heads: int
    head_dim: int
    ffn: int
    text_vocab: int
    card: int
    window: int
    max_pos: int
    dep_d: int
    dep_layers: int
    dep_heads: int
    dep_head_dim: int
    dep_ffn: int
    n_q: int = 16
    dep_steps: int = 16
    delays: Tuple[int, ...] = DELAYS
    rope_theta: float = 10000.0
    eps: float = 1e-8
    weight_dtype: str = "bf16"   # "f32" | "bf16"
    kv_dtype: str = "bf16"       # "f32" | "bf16"
    max_slots: int = 1

    def replace(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


# Tiny Moshi-shaped LM (correctness workload).  Its depformer FFN width is not
# given; 352 = 2.75 x 128 follows the FFN/d ratio of every other block.
TINY = Shape(d=256, n_layers=2, n_heads=4, head_dim=64, ffn=704, text_vocab=1000, card=2048,
             window=64, max_pos=8192, dep_d=128, dep_layers=1, dep_heads=2, dep_head_dim=64,
             dep_ffn=352, weight_dtype="f32", kv_dtype="f32", max_slots=4)

# Full PersonaPlex shape.
FULL = Shape(d=4096, n_layers=32, n_heads=32, head_dim=128, ffn=11264, text_vocab=32000,
             card=2048, window=3000, max_pos=8192, dep_d=1024, dep_layers=6, dep_heads=16,
             dep_head_dim=64, dep_ffn=2816, weight_dtype="bf16", kv_dtype="bf16", max_slots=1)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    batch: int
    prefill: str          # how rings are filled before decoding
    frames: int           # decode frames
    weight_seed: int
    input_seed: int


WORKLOADS: Dict[str, Workload] = {
    "tiny_b1": Workload("tiny_b1", TINY.replace(max_slots=1), 1, "none", 32, 0, 0),
    "full_b1": Workload("full_b1", FULL.replace(max_slots=1), 1, "250", 125, 0, 1),
    "full_b8": Workload("full_b8", FULL.replace(max_slots=8), 8, "uniform_0_3000", 125, 0, 1),
    "full_b32": Workload("full_b32", FULL.replace(max_slots=32), 32, "full_3000_churn", 250, 0, 1),
    "full_b16": Workload("full_b16", FULL.replace(max_slots=16), 16, "prompt_250", 500, 0, 1),
}

# ----------------------------------------------------------------------------- weights


def weight_specs(s: Shape) -> List[Tuple[str, Tuple[int, ...], str]]:
    """(name, shape, init) for every tensor the frame step reads, in a fixed order.

    init is "normal" (N(0, 0.02), in the workload's weight dtype) or "gain"
    (RMSNorm gains, fp32).  The list index is the Philox stream id of the tensor.
    """
    d, F, V, C, S = s.d, s.ffn, s.text_vocab, s.card, s.dep_steps
    dd, dF = s.dep_d, s.dep_ffn
    specs: List[Tuple[str, Tuple[int, ...], str]] = [
        ("emb.text", (V + 1, d), "normal"),
        ("emb.audio", (s.n_q, C + 1, d), "normal"),
    ]
    for l in range(s.n_layers):
        specs += [
            (f"layers.{l}.attn_norm", (d,), "gain"),
            (f"layers.{l}.wqkv", (3 * d, d), "normal"),
            (f"layers.{l}.wo", (d, d), "normal"),
            (f"layers.{l}.ffn_norm", (d,), "gain"),
            (f"layers.{l}.wgu", (2 * F, d), "normal"),
            (f"layers.{l}.wdown", (d, F), "normal"),
        ]
    specs += [
        ("out_norm", (d,), "gain"),
        ("text_head", (V, d), "normal"),
        ("dep.in", (S, dd, d), "normal"),
        ("dep.emb.text", (V, dd), "normal"),
        ("dep.emb.audio", (S - 1, C, dd), "normal"),
    ]
    for l in range(s.dep_layers):
        specs += [
            (f"dep.layers.{l}.attn_norm", (dd,), "gain"),
            (f"dep.layers.{l}.wqkv", (S, 3 * dd, dd), "normal"),
            (f"dep.layers.{l}.wo", (S, dd, dd), "normal"),
            (f"dep.layers.{l}.ffn_norm", (dd,), "gain"),
            (f"dep.layers.{l}.wgu", (S, 2 * dF, dd), "normal"),
            (f"dep.layers.{l}.wdown", (S, dd, dF), "normal"),
        ]
    specs += [
        ("dep.out_norm", (dd,), "gain"),
        ("dep.head", (S, C, dd), "normal"),
    ]
    return specs


def weight_nbytes(s: Shape) -> int:
    wb = 2 if s.weight_dtype == "bf16" else 4
    tot = 0
    for _, shp, init in weight_specs(s):
        tot += int(np.prod(shp)) * (4 if init == "gain" else wb)
    return tot


def make_weights(s: Shape, seed: int, std: float = 0.02, gain_std: float = 0.0) -> Dict[str, np.ndarray]:
    """Draw every tensor of ``weight_specs``.

    Linear and embedding weights are N(0, std) (bf16 bits as uint16, or fp32).
    RMSNorm gains are 1.0 + N(0, gain_std) in fp32 (gain_std = 0 gives all ones,
    the workloads' setting; tests use gain_std > 0 so that a gain that is
    ignored or misplaced shows up).
    """
    out: Dict[str, np.ndarray] = {}
    for sid, (name, shp, init) in enumerate(weight_specs(s)):
        n = int(np.prod(shp))
        if init == "gain":
            if gain_std > 0:
                a = normal_f32(seed, sid, n, 1.0, gain_std)
            else:
                a = np.ones(n, np.float32)
        elif s.weight_dtype == "bf16":
            a = normal_bf16(seed, sid, n, 0.0, std)
        else:
            a = normal_f32(seed, sid, n, 0.0, std)
        out[name] = a.reshape(shp)
    return out


# ----------------------------------------------------------------------------- token streams

STREAM_PROMPT = 1 << 20      # forced prompt / prefill frames
STREAM_USER = 2 << 20        # user audio rows during decode
STREAM_LENGTHS = 3 << 20     # per-slot prefill lengths
STREAM_CHURN = 4 << 20       # which slots leave and rejoin
STREAM_FORCED = 5 << 20      # fully forced decode frames (teacher forcing)


def forced_frames(s: Shape, seed: int, stream: int, T: int, B: int) -> np.ndarray:
    """[T, B, 17] tokens with every row forced: text uniform in [0, V), codes in [0, C)."""
    n = T * B
    text = uniform_int(seed, stream, n, 0, s.text_vocab).reshape(T, B, 1)
    codes = uniform_int(seed, stream + 1, n * 16, 0, s.card).reshape(T, B, 16)
    return np.concatenate([text, codes], axis=2).astype(np.int32)


def user_frames(s: Shape, seed: int, T: int, B: int, stream: int = STREAM_USER) -> np.ndarray:
    """[T, B, 17] decode inputs: rows 0..8 = -1 (generate), user rows 9..16 uniform in [0, C)."""
    out = np.full((T, B, 17), -1, np.int32)
    out[:, :, 9:] = uniform_int(seed, stream, T * B * 8, 0, s.card).reshape(T, B, 8)
    return out


STREAM_STATE = 6 << 20       # synthetic slot states (history and key/value rings)


def slot_state(s: Shape, seed: int, tag: int, pos: int, kv_std: float = 1.0) -> np.ndarray:
    """A synthetic slot state in the slot-state buffer layout (256-byte header:
    int32 version 1, position, window, kv dtype 1 (bf16), history [17][3];
    then keys and values [n_layers][W][d] as bf16).  History holds uniform
    tokens for frames pos-3 .. pos-1 that exist (-1 elsewhere); every ring row
    holds N(0, kv_std) draws.  ``tag`` selects independent draws."""
    assert s.kv_dtype == "bf16"
    ring = s.n_layers * s.window * s.d
    buf = np.zeros(256 + 4 * ring, np.uint8)
    head = np.zeros(4 + 17 * 3, np.int32)
    head[:4] = [1, pos, s.window, 1]
    hist = np.full((17, 3), -1, np.int32)
    toks = uniform_int(seed, STREAM_STATE + 8 * tag, 17 * 3, 0, 1 << 30).reshape(17, 3)
    for f in range(max(0, pos - 3), pos):
        lim = np.array([s.text_vocab] + [s.card] * 16)
        hist[:, f % 3] = toks[:, f % 3] % lim
    head[4:] = hist.reshape(-1)
    buf[:head.nbytes] = np.frombuffer(head.tobytes(), np.uint8)
    kv = buf[256:].view(np.uint16)
    normal_bf16(seed, STREAM_STATE + 8 * tag + 1, ring, 0.0, kv_std, out=kv[:ring])
    normal_bf16(seed, STREAM_STATE + 8 * tag + 2, ring, 0.0, kv_std, out=kv[ring:])
    return buf


def prefill_lengths(seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    """Per-slot prompt lengths uniform in [lo, hi] (inclusive)."""
    return uniform_int(seed, STREAM_LENGTHS, B, lo, hi + 1)


def churn_slots(seed: int, event: int, B: int, k: int) -> np.ndarray:
    """k distinct slots of B chosen for leave/rejoin event number ``event``."""
    keys = uniform_int(seed, STREAM_CHURN + event, B, 0, 1 << 30)
    return np.sort(np.argsort(keys, kind="stable")[:k]).astype(np.int32)
