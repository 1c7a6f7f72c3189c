"""Shared helpers for the GPU tests: contexts from synth shapes, and the
acceptance rules of the frame step against the oracle.

Acceptance (floating point): each logit vector within 2e-2 x its RMS of the
oracle's, elementwise; greedy tokens equal unless the oracle's top-2 margin is
below 0.1 (a legal flip).  Integer work is compared bit for bit.
"""
from __future__ import annotations

import numpy as np

import synth

LOGIT_RTOL = 2e-2       # x rms(oracle logits), elementwise
FLIP_MARGIN = 0.1       # argmax may differ only below this top-2 margin


def config_of(shape):
    from full_duplex_speech_frame_gb300 import mfs
    return mfs.config_from_shape(shape)


def gpu_context(shape, weights):
    from full_duplex_speech_frame_gb300 import mfs
    return mfs.context_with_weights(shape, weights)


def check_logits(gpu: np.ndarray, ref: np.ndarray, what: str) -> float:
    """Elementwise |gpu - ref| <= 2e-2 * rms(ref) per vector (last axis).  Returns the worst ratio."""
    ref = np.asarray(ref, np.float64)
    gpu = np.asarray(gpu, np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    ratio = np.abs(gpu - ref) / rms
    worst = float(ratio.max())
    assert worst <= LOGIT_RTOL, f"{what}: |gpu-ref|/rms = {worst:.3e} > {LOGIT_RTOL}"
    return worst


def top2_margin(logits: np.ndarray) -> np.ndarray:
    part = np.sort(logits, axis=-1)
    return part[..., -1] - part[..., -2]


def argmax_agrees(gpu_am: np.ndarray, ref_logits: np.ndarray) -> np.ndarray:
    """Boolean mask: equal argmax, or the oracle's top-2 margin < 0.1."""
    ref_am = np.argmax(ref_logits, axis=-1)
    return (gpu_am == ref_am) | (top2_margin(ref_logits) < FLIP_MARGIN)


def check_argmax(gpu_am, ref_logits, what: str) -> int:
    ok = argmax_agrees(np.asarray(gpu_am), np.asarray(ref_logits))
    assert ok.all(), f"{what}: greedy token differs with top-2 margin >= {FLIP_MARGIN} at {np.argwhere(~ok)[:5]}"
    return int((np.asarray(gpu_am) != np.argmax(ref_logits, axis=-1)).sum())


def follow_tokens(text, codes, code_argmax) -> np.ndarray:
    """Follow-mode input for the oracle from one GPU step: the GPU's chosen token per
    stream, and for a frame before 0 (output -1) the raw argmax its substep chain used."""
    text = np.asarray(text, np.int32)
    codes = np.asarray(codes, np.int32)
    f = np.empty((text.shape[0], 17), np.int32)
    f[:, 0] = text
    f[:, 1:] = np.where(codes >= 0, codes, np.asarray(code_argmax, np.int32))
    return f


class Tally:
    """Frames compared, the worst |gpu - ref| / rms(ref) and the legal flips of a run."""

    def __init__(self, what: str):
        self.what, self.frames, self.worst, self.flips = what, 0, 0.0, 0

    def step(self, dbg, rows, ref, label: str) -> None:
        """Check GPU rows `rows` of one step against the oracle's results `ref`."""
        self.worst = max(self.worst, check_logits(dbg["text_logits"][rows], ref["text_logits"], f"{label} text logits"))
        self.worst = max(self.worst, check_logits(dbg["dep_logits"][rows], ref["dep_logits"], f"{label} depformer logits"))
        self.flips += check_argmax(dbg["text_argmax"][rows], ref["text_logits"], f"{label} text argmax")
        self.flips += check_argmax(dbg["code_argmax"][rows], ref["dep_logits"], f"{label} code argmax")
        self.frames += len(rows)

    def report(self) -> str:
        return (f"{self.what}: {self.frames} slot-frames compared, worst |gpu-ref|/rms = {self.worst:.3e} "
                f"(limit {LOGIT_RTOL}), {self.flips} legal flips")


def nan_stale_rows(state: np.ndarray, shape, pos: int, all_rows: bool = False) -> np.ndarray:
    """Set to NaN (bf16 0x7FC0) every key/value ring row of a slot state (slot-state
    layout: 256-byte header, then keys and values [n_layers][W][d] bf16) that the next
    step at position `pos` must not read: rows of positions never written (pos < W:
    rows pos .. W-1) or outside the window (pos >= W: the row of position pos - W,
    which the step overwrites before reading).  all_rows: every row."""
    s = shape
    kv = state[256:].view(np.uint16).reshape(2, s.n_layers, s.window, s.d)
    if all_rows:
        kv[...] = 0x7FC0
    elif pos < s.window:
        kv[:, :, pos:, :] = 0x7FC0
    else:
        kv[:, :, pos % s.window, :] = 0x7FC0
    return state
