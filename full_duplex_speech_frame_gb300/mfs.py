"""Python binding of the C ABI in include/mfs.h (ctypes; argument marshalling only).

Every step of the frame step runs in the CUDA library ``libmfs.so``; this module
only converts arguments.  There is no fallback: if the library is missing the
import fails with the command that builds it.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# MFS_LIBRARY selects another build of the same library (same ABI).
LIB_PATH = os.environ.get("MFS_LIBRARY") or os.path.join(_HERE, "libmfs.so")

MFS_OK = 0
STATUS = {-1: "MFS_E_ARG", -2: "MFS_E_SLOT", -3: "MFS_E_TOKEN", -4: "MFS_E_RANGE", -5: "MFS_E_STATE",
          -6: "MFS_E_CUDA", -7: "MFS_E_DEVICE", -8: "MFS_E_NOMEM"}
MFS_DTYPE_F32, MFS_DTYPE_BF16 = 0, 1
MFS_MAX_SLOTS = 64


class MfsError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS.get(code, code)}: {message}")
        self.code = code
        self.status = STATUS.get(code, str(code))


class mfs_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "d", "n_layers", "n_heads", "head_dim", "ffn", "text_vocab", "card", "n_q", "window", "max_pos",
        "dep_d", "dep_layers", "dep_heads", "dep_head_dim", "dep_ffn", "dep_steps")] + [
        ("delays", ctypes.c_int * 17), ("rope_theta", ctypes.c_double), ("eps", ctypes.c_double),
        ("weight_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int), ("max_slots", ctypes.c_int)]


def _load_library():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` "
                          "(or python full_duplex_speech_frame_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ci, i32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    sig = {
        "mfs_create": (ci, [ctypes.POINTER(mfs_config), vp, ctypes.POINTER(vp)]),
        "mfs_destroy": (None, [vp]),
        "mfs_last_error": (ctypes.c_char_p, [vp]),
        "mfs_load_weights": (ci, [vp, ctypes.c_char_p, vp, ctypes.c_size_t, ci]),
        "mfs_step": (ci, [vp, ci, i32p, i32p, i32p, i32p]),
        "mfs_step_device": (ci, [vp, ci, i32p, vp, vp, vp]),
        "mfs_sync": (ci, [vp]),
        "mfs_prefill": (ci, [vp, ci, i32p, ci, i32p]),
        "mfs_reset_slot": (ci, [vp, ci]),
        "mfs_position": (ci, [vp, ci]),
        "mfs_read_debug": (ci, [vp, vp, vp, vp, vp]),
        "mfs_set_ring_mask_oldest": (ci, [vp, ci]),
        "mfs_debug_set_seq": (ci, [vp, ctypes.c_uint32]),
        "mfs_set_mode": (ci, [vp, ci]),
        "mfs_launches_per_step": (ci, [vp]),
        "mfs_set_skip_settled": (ci, [vp, ci]),
        "mfs_set_wait_limit": (ci, [vp, ci]),
        "mfs_debug_stall": (ci, [vp, ci]),
        "mfs_set_sampling": (ci, [vp, ci, ctypes.c_float, ci, ctypes.c_float, ci]),
        "mfs_step_sampled": (ci, [vp, ci, i32p, i32p, vp, i32p, i32p]),
        "mfs_set_timing": (ci, [vp, ci]),
        "mfs_kernel_time": (ci, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
        "mfs_phase_times": (ci, [vp, vp, ci]),
        "mfs_argmax_rows_noalloc": (ci, [vp, ci, ci, ctypes.c_longlong, vp, vp]),
        "mfs_rvq_encode": (ci, [vp, vp, ci, ci, vp, ci, vp, vp]),
        "mfs_slot_state_bytes": (ctypes.c_size_t, [vp]),
        "mfs_export_slot": (ci, [vp, ci, vp, ctypes.c_size_t]),
        "mfs_import_slot": (ci, [vp, ci, vp, ctypes.c_size_t]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load_library()


def exported_symbols() -> Sequence[str]:
    return [n for n in dir(_lib) if n.startswith("mfs_")]


class Ctx:
    """Owner of an ``mfs_ctx*``; destroyed with ``mfs_destroy``."""

    def __init__(self, handle: int, cfg: mfs_config):
        self.handle = ctypes.c_void_p(handle)
        self.cfg = cfg
        self.last_n = 0

    def __del__(self):
        if getattr(self, "handle", None) and self.handle.value:
            _lib.mfs_destroy(self.handle)
            self.handle = ctypes.c_void_p(None)


def _check(ctx: Optional[Ctx], rc: int) -> None:
    if rc != MFS_OK:
        h = ctx.handle if ctx is not None else None
        raise MfsError(rc, (_lib.mfs_last_error(h) or b"").decode())


def make_config(d, n_layers, n_heads, head_dim, ffn, text_vocab, card, window, max_pos, dep_d, dep_layers,
                dep_heads, dep_head_dim, dep_ffn, delays, rope_theta=10000.0, eps=1e-8,
                weight_dtype="bf16", kv_dtype="bf16", max_slots=1, n_q=16, dep_steps=16) -> mfs_config:
    c = mfs_config()
    for k, v in dict(d=d, n_layers=n_layers, n_heads=n_heads, head_dim=head_dim, ffn=ffn, text_vocab=text_vocab,
                     card=card, n_q=n_q, window=window, max_pos=max_pos, dep_d=dep_d, dep_layers=dep_layers,
                     dep_heads=dep_heads, dep_head_dim=dep_head_dim, dep_ffn=dep_ffn, dep_steps=dep_steps,
                     max_slots=max_slots).items():
        setattr(c, k, int(v))
    c.delays[:] = [int(x) for x in delays]
    c.rope_theta = float(rope_theta)
    c.eps = float(eps)
    c.weight_dtype = MFS_DTYPE_BF16 if weight_dtype == "bf16" else MFS_DTYPE_F32
    c.kv_dtype = MFS_DTYPE_BF16 if kv_dtype == "bf16" else MFS_DTYPE_F32
    return c


def config_from_shape(shape) -> mfs_config:
    """An mfs_config from any object with the config's field names as attributes
    (dtypes as the strings "bf16" / "f32")."""
    s = shape
    return make_config(d=s.d, n_layers=s.n_layers, n_heads=s.n_heads, head_dim=s.head_dim, ffn=s.ffn,
                       text_vocab=s.text_vocab, card=s.card, window=s.window, max_pos=s.max_pos,
                       dep_d=s.dep_d, dep_layers=s.dep_layers, dep_heads=s.dep_heads,
                       dep_head_dim=s.dep_head_dim, dep_ffn=s.dep_ffn, delays=s.delays,
                       rope_theta=s.rope_theta, eps=s.eps, weight_dtype=s.weight_dtype,
                       kv_dtype=s.kv_dtype, max_slots=s.max_slots, n_q=s.n_q, dep_steps=s.dep_steps)


def context_with_weights(shape, weights) -> "Ctx":
    """A context for `shape` with every named tensor of `weights` loaded."""
    ctx = mfs_create(config_from_shape(shape))
    for name, arr in weights.items():
        mfs_load_weights(ctx, name, arr)
    return ctx


def _current_stream():
    try:
        import torch
        if torch.cuda.is_available():
            return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    except ImportError:
        pass
    return None


def mfs_create(cfg: mfs_config, stream=None) -> Ctx:
    out = ctypes.c_void_p()
    st = _current_stream() if stream is None else ctypes.c_void_p(stream)
    rc = _lib.mfs_create(ctypes.byref(cfg), st, ctypes.byref(out))
    _check(None, rc)
    return Ctx(out.value, cfg)


def mfs_destroy(ctx: Ctx) -> None:
    if ctx.handle.value:
        _lib.mfs_destroy(ctx.handle)
        ctx.handle = ctypes.c_void_p(None)


def mfs_last_error(ctx: Optional[Ctx]) -> str:
    return (_lib.mfs_last_error(ctx.handle if ctx else None) or b"").decode()


def mfs_load_weights(ctx: Ctx, name: str, src) -> None:
    """src: a C-contiguous numpy array (host) or a contiguous CUDA torch tensor."""
    if isinstance(src, np.ndarray):
        src = np.ascontiguousarray(src)
        rc = _lib.mfs_load_weights(ctx.handle, name.encode(), src.ctypes.data, src.nbytes, 0)
    else:
        assert src.is_cuda and src.is_contiguous()
        rc = _lib.mfs_load_weights(ctx.handle, name.encode(), src.data_ptr(),
                                   src.numel() * src.element_size(), 1)
    _check(ctx, rc)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def mfs_step(ctx: Ctx, slots, in_codes):
    """Returns (text_tok [n], codes [n, 16]) as int32 numpy arrays."""
    slots = _i32(slots).reshape(-1)
    n = slots.size
    codes_in = _i32(in_codes).reshape(n, 17)
    text = np.empty(n, np.int32)
    codes = np.empty((n, 16), np.int32)
    rc = _lib.mfs_step(ctx.handle, n, slots.ctypes.data, codes_in.ctypes.data, text.ctypes.data, codes.ctypes.data)
    _check(ctx, rc)
    ctx.last_n = n
    return text, codes


def mfs_set_sampling(ctx: Ctx, slot: int, text_temp: float, text_topk: int, audio_temp: float, audio_topk: int) -> None:
    _check(ctx, _lib.mfs_set_sampling(ctx.handle, int(slot), float(text_temp), int(text_topk), float(audio_temp),
                                      int(audio_topk)))


def mfs_step_sampled(ctx: Ctx, slots, in_codes, uniforms):
    """mfs_step with uniforms [n, 17] in [0, 1) for the slots' sampling heads."""
    slots = _i32(slots).reshape(-1)
    n = slots.size
    codes_in = _i32(in_codes).reshape(n, 17)
    unif = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(n, 17)
    text = np.empty(n, np.int32)
    codes = np.empty((n, 16), np.int32)
    rc = _lib.mfs_step_sampled(ctx.handle, n, slots.ctypes.data, codes_in.ctypes.data, unif.ctypes.data,
                               text.ctypes.data, codes.ctypes.data)
    _check(ctx, rc)
    ctx.last_n = n
    return text, codes


def mfs_step_device(ctx: Ctx, slots, d_in_codes, d_text=None, d_codes=None) -> None:
    """d_* are contiguous int32 CUDA tensors; returns without waiting."""
    slots = _i32(slots).reshape(-1)
    n = slots.size
    rc = _lib.mfs_step_device(ctx.handle, n, slots.ctypes.data, d_in_codes.data_ptr(),
                              d_text.data_ptr() if d_text is not None else None,
                              d_codes.data_ptr() if d_codes is not None else None)
    _check(ctx, rc)
    ctx.last_n = n


def mfs_sync(ctx: Ctx) -> None:
    _check(ctx, _lib.mfs_sync(ctx.handle))


def mfs_prefill(ctx: Ctx, slots, codes) -> None:
    """codes [n, T, 17] int, every entry >= 0."""
    slots = _i32(slots).reshape(-1)
    n = slots.size
    codes = _i32(codes)
    T = codes.shape[1] if codes.ndim == 3 else codes.size // (17 * n)
    codes = codes.reshape(n, T, 17)
    _check(ctx, _lib.mfs_prefill(ctx.handle, n, slots.ctypes.data, T, codes.ctypes.data))


def mfs_reset_slot(ctx: Ctx, slot: int) -> None:
    _check(ctx, _lib.mfs_reset_slot(ctx.handle, int(slot)))


def mfs_position(ctx: Ctx, slot: int) -> int:
    rc = _lib.mfs_position(ctx.handle, int(slot))
    if rc < 0:
        _check(ctx, rc)
    return rc


def mfs_export_slot(ctx: Ctx, slot: int) -> np.ndarray:
    """The slot's state as a uint8 buffer (layout in include/mfs.h)."""
    buf = np.empty(_lib.mfs_slot_state_bytes(ctx.handle), np.uint8)
    _check(ctx, _lib.mfs_export_slot(ctx.handle, int(slot), buf.ctypes.data, buf.nbytes))
    return buf


def mfs_import_slot(ctx: Ctx, slot: int, buf: np.ndarray) -> None:
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    _check(ctx, _lib.mfs_import_slot(ctx.handle, int(slot), buf.ctypes.data, buf.nbytes))


def mfs_read_debug(ctx: Ctx, n: Optional[int] = None) -> dict:
    n = ctx.last_n if n is None else n
    c = ctx.cfg
    out = {"text_logits": np.empty((n, c.text_vocab), np.float32),
           "dep_logits": np.empty((n, 16, c.card), np.float32),
           "text_argmax": np.empty(n, np.int32), "code_argmax": np.empty((n, 16), np.int32)}
    rc = _lib.mfs_read_debug(ctx.handle, out["text_logits"].ctypes.data, out["dep_logits"].ctypes.data,
                             out["text_argmax"].ctypes.data, out["code_argmax"].ctypes.data)
    _check(ctx, rc)
    return out


def mfs_set_ring_mask_oldest(ctx: Ctx, on: bool) -> None:
    """Attend to W - 1 keys once the ring is full (the masked-oldest-slot window variant)."""
    _check(ctx, _lib.mfs_set_ring_mask_oldest(ctx.handle, 1 if on else 0))


def mfs_debug_set_seq(ctx: Ctx, seq: int) -> None:
    """Testing: the next step takes sequence number seq + 1 (see include/mfs.h)."""
    _check(ctx, _lib.mfs_debug_set_seq(ctx.handle, int(seq) & 0xFFFFFFFF))


def mfs_set_mode(ctx: Ctx, mode: int) -> None:
    _check(ctx, _lib.mfs_set_mode(ctx.handle, int(mode)))


def mfs_set_skip_settled(ctx: Ctx, on: bool) -> None:
    """Skip trailing depformer substeps whose outputs are all supplied (include/mfs.h)."""
    _check(ctx, _lib.mfs_set_skip_settled(ctx.handle, int(bool(on))))


def mfs_set_wait_limit(ctx: Ctx, ms: int) -> None:
    _check(ctx, _lib.mfs_set_wait_limit(ctx.handle, int(ms)))


def mfs_debug_stall(ctx: Ctx, slot: int) -> None:
    """Raises MfsError(MFS_E_DEVICE) when the device's bounded waits work (include/mfs.h)."""
    _check(ctx, _lib.mfs_debug_stall(ctx.handle, int(slot)))


def mfs_launches_per_step(ctx: Ctx) -> int:
    return _lib.mfs_launches_per_step(ctx.handle)


def mfs_set_timing(ctx: Ctx, flags) -> None:
    """flags: bit 0 = event timing of each step's kernel, bit 1 = per-phase timer stamps."""
    _check(ctx, _lib.mfs_set_timing(ctx.handle, int(flags)))


def mfs_phase_times(ctx: Ctx) -> np.ndarray:
    """Diagnostic timer values of the last step(s), [phases + 1, 8] (see include/mfs.h)."""
    buf = np.zeros(16384, np.uint64)
    rc = _lib.mfs_phase_times(ctx.handle, buf.ctypes.data, buf.size)
    if rc < 0:
        _check(ctx, rc)
    return buf[:rc].reshape(-1, 8).copy()


def mfs_kernel_time(ctx: Ctx):
    """(summed kernel milliseconds, steps timed) since the previous call."""
    ms, n = ctypes.c_double(), ctypes.c_int()
    _check(ctx, _lib.mfs_kernel_time(ctx.handle, ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def mfs_argmax_rows_noalloc(logits, out, stream=None) -> None:
    """Greedy argmax of each row of a 2-D fp32 CUDA tensor into an int32 CUDA tensor,
    with no device allocation (see include/mfs.h); enqueued on `stream` (default:
    torch's current stream)."""
    import torch
    assert logits.is_cuda and logits.dtype == torch.float32 and logits.dim() == 2 and logits.stride(1) == 1
    assert out.is_cuda and out.dtype == torch.int32 and out.is_contiguous() and out.numel() >= logits.shape[0]
    rows, cols = logits.shape
    st = _current_stream() if stream is None else ctypes.c_void_p(stream)
    rc = _lib.mfs_argmax_rows_noalloc(logits.data_ptr(), rows, cols, logits.stride(0), out.data_ptr(), st)
    _check(None, rc)


def mfs_rvq_encode(z_sem, z_ac, codebooks, codes, stream=None) -> None:
    """Mimi split RVQ encode on CUDA tensors: z_sem, z_ac [T, D] fp32, codebooks [8, Cb, D]
    fp32 -> codes [T, 8] int32 (see include/mfs.h); enqueued on `stream`."""
    import torch
    for t in (z_sem, z_ac, codebooks):
        assert t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
    assert codes.is_cuda and codes.dtype == torch.int32 and codes.is_contiguous()
    T, D = z_sem.shape
    st = _current_stream() if stream is None else ctypes.c_void_p(stream)
    rc = _lib.mfs_rvq_encode(z_sem.data_ptr(), z_ac.data_ptr(), T, D, codebooks.data_ptr(), codebooks.shape[1],
                             codes.data_ptr(), st)
    _check(None, rc)
