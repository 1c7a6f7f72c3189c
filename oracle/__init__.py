"""CPU oracle of the lockstep frame step (fp64, one slot at a time).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(``full_duplex_speech_frame_gb300``) never does.  The C source shares no code,
header, table or constant with the CUDA library.

Parity status per function (what pins each one is in tests/test_oracle_pins.py):
  orc_rmsnorm    pinned (closed forms: constant vector, scale invariance; torch rms_norm)
  orc_rope       pinned (complex-exponential closed form, norm and relative-angle invariants)
  orc_attention  pinned (single key, equal keys, torch scaled_dot_product_attention)
  embed / delays pinned (brute-force schedule on tiny inputs, bit-exact)
  temporal layer pinned (torch library composition, float64, tiny shape)
  ring window    pinned (ring storage == full history masked to the last W, bit-exact)
  depformer      pinned (torch library composition; causality invariants)
  end-to-end model values against the real PersonaPlex: parity unpinned (no
  trained weights or goldens exist here).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mfs_oracle.c")
_LIB = os.path.join(_HERE, "libmfs_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp"
        subprocess.check_call(["gcc", "-O3", "-fPIC", "-shared", "-fopenmp", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "d", "n_layers", "n_heads", "head_dim", "ffn", "text_vocab", "card", "n_q", "window",
        "max_pos", "dep_d", "dep_layers", "dep_heads", "dep_head_dim", "dep_ffn", "dep_steps")] + [
        ("delays", ctypes.c_int * 17), ("rope_theta", ctypes.c_double), ("eps", ctypes.c_double),
        ("weight_dtype", ctypes.c_int), ("max_slots", ctypes.c_int), ("brute_force", ctypes.c_int),
        ("kv_dtype", ctypes.c_int), ("mask_oldest", ctypes.c_int)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, ci = ctypes.c_void_p, ctypes.c_int
        lib.orc_create.restype = vp
        lib.orc_create.argtypes = [ctypes.POINTER(_Cfg)]
        lib.orc_destroy.argtypes = [vp]
        lib.orc_last_error.restype = ctypes.c_char_p
        lib.orc_last_error.argtypes = [vp]
        lib.orc_set_weight.argtypes = [vp, ctypes.c_char_p, vp, ctypes.c_longlong]
        lib.orc_reset_slot.argtypes = [vp, ci]
        lib.orc_position.argtypes = [vp, ci]
        lib.orc_step.argtypes = [vp, ci, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_set_sampling.argtypes = [vp, ci, ctypes.c_double, ci, ctypes.c_double, ci]
        lib.orc_rvq_encode.argtypes = [vp, vp, ci, ci, vp, ci, vp, vp]
        lib.orc_sample_topk.restype = ci
        lib.orc_sample_topk.argtypes = [vp, ci, ctypes.c_double, ci, ctypes.c_double]
        lib.orc_prefill.argtypes = [vp, ci, ci, vp]
        lib.orc_import_slot.argtypes = [vp, ci, vp, ctypes.c_longlong]
        lib.orc_export_slot.argtypes = [vp, ci, vp, ctypes.c_longlong]
        lib.orc_rmsnorm.argtypes = [vp, vp, ci, ctypes.c_double, vp]
        lib.orc_rope.argtypes = [vp, ci, ci, ctypes.c_double]
        lib.orc_attention.argtypes = [vp, vp, vp, ci, ci, ctypes.c_long, vp]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    g = np.ascontiguousarray(g, np.float32)
    out = np.empty_like(x)
    _load().orc_rmsnorm(x.ctypes.data, g.ctypes.data, x.size, eps, out.ctypes.data)
    return out


def rope(v: np.ndarray, p: int, theta: float = 10000.0) -> np.ndarray:
    v = np.array(v, np.float64, copy=True)
    _load().orc_rope(v.ctypes.data, v.size, p, theta)
    return v


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """q [hd], K/V [npos, hd] -> [hd]."""
    q = np.ascontiguousarray(q, np.float64)
    K = np.ascontiguousarray(K, np.float64)
    V = np.ascontiguousarray(V, np.float64)
    out = np.empty(q.size, np.float64)
    _load().orc_attention(q.ctypes.data, K.ctypes.data, V.ctypes.data, K.shape[0], q.size,
                          K.shape[1], out.ctypes.data)
    return out


class Oracle:
    """One oracle instance: slots, token histories and fp64 key/value rings."""

    def __init__(self, shape, weights: Dict[str, np.ndarray], brute_force: bool = False, mask_oldest: bool = False):
        s = shape
        c = _Cfg()
        for f in ("d", "n_layers", "n_heads", "head_dim", "ffn", "text_vocab", "card", "n_q",
                  "window", "max_pos", "dep_d", "dep_layers", "dep_heads", "dep_head_dim",
                  "dep_ffn", "dep_steps", "max_slots"):
            setattr(c, f, int(getattr(s, f)))
        c.delays[:] = list(s.delays)
        c.rope_theta = float(s.rope_theta)
        c.eps = float(s.eps)
        c.weight_dtype = 1 if s.weight_dtype == "bf16" else 0
        c.brute_force = 1 if brute_force else 0
        c.kv_dtype = 1 if s.kv_dtype == "bf16" else 0
        c.mask_oldest = 1 if mask_oldest else 0
        self.shape = s
        self._lib = _load()
        self._h = self._lib.orc_create(ctypes.byref(c))
        if not self._h:
            raise MemoryError("orc_create failed")
        self._keep = {}
        for name, arr in weights.items():
            arr = np.ascontiguousarray(arr)
            self._keep[name] = arr
            rc = self._lib.orc_set_weight(self._h, name.encode(), arr.ctypes.data, arr.nbytes)
            if rc != 0:
                raise ValueError(self._lib.orc_last_error(self._h).decode())

    def __del__(self):
        if getattr(self, "_h", None):
            self._lib.orc_destroy(self._h)
            self._h = None

    def position(self, slot: int) -> int:
        return self._lib.orc_position(self._h, slot)

    def import_slot(self, slot: int, buf: np.ndarray) -> None:
        """Replace a slot's state with a buffer in the slot-state layout (position,
        history, key/value ring rows in the cache dtype)."""
        buf = np.ascontiguousarray(buf, dtype=np.uint8)
        if self._lib.orc_import_slot(self._h, slot, buf.ctypes.data, buf.nbytes) != 0:
            raise ValueError("slot state rejected")

    def state_bytes(self) -> int:
        s = self.shape
        return 256 + 2 * s.n_layers * s.window * s.d * (2 if s.kv_dtype == "bf16" else 4)

    def export_slot(self, slot: int) -> np.ndarray:
        buf = np.empty(self.state_bytes(), np.uint8)
        if self._lib.orc_export_slot(self._h, slot, buf.ctypes.data, buf.nbytes) != 0:
            raise ValueError("export failed")
        return buf

    def reset_slot(self, slot: int) -> None:
        if self._lib.orc_reset_slot(self._h, slot) != 0:
            raise ValueError("bad slot")

    def set_sampling(self, slot: int, text_temp: float, text_k: int, audio_temp: float, audio_k: int) -> None:
        if self._lib.orc_set_sampling(self._h, slot, text_temp, text_k, audio_temp, audio_k) != 0:
            raise ValueError("bad slot")

    def step(self, slots, codes, want_logits: bool = False, want_tokens: bool = False, uniforms=None,
             follow=None):
        """codes [n,17] int (-1 = generate); uniforms [n,17] in [0, 1) switches on the
        slots' sampling (stream k of row i draws with uniforms[i][k]).  follow [n,17]
        (follow mode): the token adopted for stream k wherever the oracle would
        generate it (-1: its own choice); supplied tokens still win.  Returns numpy arrays."""
        unif = None if uniforms is None else np.ascontiguousarray(uniforms, np.float64).reshape(len(slots), 17)
        fol = None if follow is None else np.ascontiguousarray(follow, np.int32).reshape(len(slots), 17)
        slots = np.ascontiguousarray(slots, np.int32)
        codes = np.ascontiguousarray(codes, np.int32).reshape(len(slots), 17)
        n, s = len(slots), self.shape
        out = {"text": np.empty(n, np.int32), "codes": np.empty((n, 16), np.int32),
               "text_argmax": np.empty(n, np.int32), "code_argmax": np.empty((n, 16), np.int32)}
        if want_logits:
            out["text_logits"] = np.empty((n, s.text_vocab), np.float64)
            out["dep_logits"] = np.empty((n, 16, s.card), np.float64)
        if want_tokens:
            out["x_tokens"] = np.empty((n, 17), np.int32)
        rc = self._lib.orc_step(self._h, n, slots.ctypes.data, codes.ctypes.data,
                                out["text"].ctypes.data, out["codes"].ctypes.data,
                                _ptr(out.get("text_logits")), _ptr(out.get("dep_logits")),
                                out["text_argmax"].ctypes.data, out["code_argmax"].ctypes.data,
                                _ptr(out.get("x_tokens")), _ptr(unif), _ptr(fol))
        if rc != 0:
            raise ValueError(f"orc_step: {self._lib.orc_last_error(self._h).decode()} ({rc})")
        return out

    def prefill(self, slot: int, codes) -> None:
        codes = np.ascontiguousarray(codes, np.int32).reshape(-1, 17)
        rc = self._lib.orc_prefill(self._h, slot, codes.shape[0], codes.ctypes.data)
        if rc != 0:
            raise ValueError(f"orc_prefill: {self._lib.orc_last_error(self._h).decode()} ({rc})")


def sample_topk(logits, temp: float, k: int, u: float) -> int:
    """The oracle's temperature + top-k draw for one logit vector (fp64)."""
    lg = np.ascontiguousarray(logits, np.float64).reshape(-1)
    return int(_load().orc_sample_topk(lg.ctypes.data, lg.size, float(temp), int(k), float(u)))


def rvq_encode(z_sem, z_ac, codebooks):
    """The oracle's split RVQ encode: z_sem, z_ac [T, D], codebooks [8, Cb, D] (fp32 inputs).
    Returns (codes [T, 8] int32, gap [T, 8] second-best minus best distance)."""
    z_sem = np.ascontiguousarray(z_sem, np.float32)
    z_ac = np.ascontiguousarray(z_ac, np.float32)
    cb = np.ascontiguousarray(codebooks, np.float32)
    T, D = z_sem.shape
    codes = np.empty((T, 8), np.int32)
    gap = np.empty((T, 8), np.float64)
    _load().orc_rvq_encode(z_sem.ctypes.data, z_ac.ctypes.data, T, D, cb.ctypes.data, cb.shape[1],
                           codes.ctypes.data, gap.ctypes.data)
    return codes, gap
