"""Whole-sequence, teacher-forced float64 forward of the Moshi-shaped LM, built from
torch library routines (F.rms_norm, F.linear, F.scaled_dot_product_attention,
F.silu, complex rotation).  Test-only pin for the CPU oracle.

It computes the same model as the oracle by a different route: every frame of a
fully forced token sequence at once, with a causal sliding-window mask over
absolute positions instead of a ring of cached keys; the depformer runs all 16
substeps of all frames at once with a causal mask, per-substep weights applied
by einsum.  Agreement with the oracle's step-by-step results (to fp64 rounding)
pins the oracle's indexing, masking, rotation and wiring.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

import synth


def _t(arr: np.ndarray, dtype: str) -> torch.Tensor:
    if arr.dtype == np.uint16:
        arr = synth.bf16_to_f32(arr)
    return torch.from_numpy(np.asarray(arr, np.float64))


def input_rows(s, tokens: np.ndarray) -> np.ndarray:
    """Embedding row read by stream k at frame p: the token of frame p-1-delay[k], or INIT."""
    T = tokens.shape[0]
    X = np.empty((T, 17), np.int64)
    for p in range(T):
        for k in range(17):
            f = p - 1 - s.delays[k]
            X[p, k] = tokens[f, k] if f >= 0 else (s.text_vocab if k == 0 else s.card)
    return X


def rotate(x: torch.Tensor, theta: float) -> torch.Tensor:
    """x [T, H, hd]: interleaved pairs as complex numbers times exp(i p theta^(-2i/hd))."""
    T, H, hd = x.shape
    i = torch.arange(hd // 2, dtype=torch.float64)
    freq = theta ** (-2.0 * i / hd)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * freq[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    z = torch.view_as_complex(x.reshape(T, H, hd // 2, 2).contiguous())
    return torch.view_as_real(z * rot).reshape(T, H, hd)


def forward(s, w, tokens: np.ndarray):
    """tokens [T, 17], every entry >= 0.  Returns (text_logits [T,V], dep_logits [T,16,C])."""
    T = tokens.shape[0]
    d, H, hd, Fw = s.d, s.n_heads, s.head_dim, s.ffn
    W = {k: _t(v, s.weight_dtype) for k, v in w.items()}
    X = torch.from_numpy(input_rows(s, tokens))
    x = W["emb.text"][X[:, 0]].clone()
    for k in range(1, 17):
        x = x + W["emb.audio"][k - 1][X[:, k]]
    pos = torch.arange(T)
    mask = (pos[None, :] <= pos[:, None]) & (pos[None, :] >= pos[:, None] - s.window + 1)
    for l in range(s.n_layers):
        a = F.rms_norm(x, (d,), W[f"layers.{l}.attn_norm"], s.eps)
        q, k, v = F.linear(a, W[f"layers.{l}.wqkv"]).split(d, dim=1)
        q = rotate(q.reshape(T, H, hd), s.rope_theta).transpose(0, 1)
        k = rotate(k.reshape(T, H, hd), s.rope_theta).transpose(0, 1)
        v = v.reshape(T, H, hd).transpose(0, 1)
        if s.kv_dtype == "bf16":  # the cache holds rotated keys and values in bf16
            k = k.to(torch.bfloat16).to(torch.float64)
            v = v.to(torch.bfloat16).to(torch.float64)
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask)
        x = x + F.linear(o.transpose(0, 1).reshape(T, d), W[f"layers.{l}.wo"])
        a = F.rms_norm(x, (d,), W[f"layers.{l}.ffn_norm"], s.eps)
        gate, up = F.linear(a, W[f"layers.{l}.wgu"]).split(Fw, dim=1)
        x = x + F.linear(F.silu(gate) * up, W[f"layers.{l}.wdown"])
    h = F.rms_norm(x, (d,), W["out_norm"], s.eps)
    text_logits = F.linear(h, W["text_head"])

    # depformer over all frames: chain inputs are the forced tokens where the target
    # frame exists, else the previous substep's argmax, found by iterating to the
    # fixed point (substep j is final after j+1 passes, by causality).
    S, dd, dH, dhd, dF = s.dep_steps, s.dep_d, s.dep_heads, s.dep_head_dim, s.dep_ffn
    base = torch.einsum("jnk,tk->tjn", W["dep.in"], h)            # [T, S, dd]
    prev = np.zeros((T, S), np.int64)
    known = np.zeros((T, S), bool)
    for p in range(T):
        prev[p, 0], known[p, 0] = tokens[p, 0], True
        for j in range(1, S):
            f = p - s.delays[j]
            if f >= 0:
                prev[p, j], known[p, j] = tokens[f, j], True
    logits = None
    for _ in range(S + 1):
        u = base.clone()
        u[:, 0] += W["dep.emb.text"][torch.from_numpy(prev[:, 0])]
        for j in range(1, S):
            u[:, j] += W["dep.emb.audio"][j - 1][torch.from_numpy(prev[:, j])]
        for l in range(s.dep_layers):
            a = F.rms_norm(u, (dd,), W[f"dep.layers.{l}.attn_norm"], s.eps)
            qkv = torch.einsum("jnk,tjk->tjn", W[f"dep.layers.{l}.wqkv"], a)
            q, k, v = (t.reshape(T, S, dH, dhd).transpose(1, 2) for t in qkv.split(dd, dim=2))
            o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
            o = o.transpose(1, 2).reshape(T, S, dd)
            u = u + torch.einsum("jnk,tjk->tjn", W[f"dep.layers.{l}.wo"], o)
            a = F.rms_norm(u, (dd,), W[f"dep.layers.{l}.ffn_norm"], s.eps)
            gate, up = torch.einsum("jnk,tjk->tjn", W[f"dep.layers.{l}.wgu"], a).split(dF, dim=2)
            u = u + torch.einsum("jnk,tjk->tjn", W[f"dep.layers.{l}.wdown"], F.silu(gate) * up)
        z = F.rms_norm(u, (dd,), W["dep.out_norm"], s.eps)
        logits = torch.einsum("jnk,tjk->tjn", W["dep.head"], z)
        am = logits.argmax(dim=2).numpy()
        new = prev.copy()
        for p in range(T):
            for j in range(1, S):
                if not known[p, j]:
                    new[p, j] = am[p, j - 1]
        if np.array_equal(new, prev):
            break
        prev = new
    return text_logits.numpy(), logits.numpy()
