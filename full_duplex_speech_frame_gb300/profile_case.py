"""A small case of the frame step for hardware-counter captures.

    python -m full_duplex_speech_frame_gb300.profile_case [--layers L] [--dep-layers DL] [--steps N]

The full PersonaPlex widths (4096-d temporal, 32 x 128 heads, FFN 11264,
32000-word text head, 1024-d depformer with 16 per-substep weight sets) with
fewer layers, so that a multi-pass profiler capture holds about 1.5 GB on the
device instead of 17 GB, while the streamed weights (about 1.4 GB per step)
still exceed the L2 cache and DRAM counters keep their meaning.  Launch order:
8 prompt frames (one launch each), then N decode steps.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from full_duplex_speech_frame_gb300 import mfs  # noqa: E402

PROMPT = 8


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--dep-layers", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4)
    a = ap.parse_args()
    import torch
    torch.cuda.set_stream(torch.cuda.Stream())
    s = synth.FULL.replace(n_layers=a.layers, dep_layers=a.dep_layers, max_slots=1)
    cfg = mfs.make_config(d=s.d, n_layers=s.n_layers, n_heads=s.n_heads, head_dim=s.head_dim, ffn=s.ffn,
                          text_vocab=s.text_vocab, card=s.card, window=s.window, max_pos=s.max_pos,
                          dep_d=s.dep_d, dep_layers=s.dep_layers, dep_heads=s.dep_heads,
                          dep_head_dim=s.dep_head_dim, dep_ffn=s.dep_ffn, delays=s.delays,
                          rope_theta=s.rope_theta, eps=s.eps, weight_dtype=s.weight_dtype,
                          kv_dtype=s.kv_dtype, max_slots=1, n_q=s.n_q, dep_steps=s.dep_steps)
    ctx = mfs.mfs_create(cfg)
    for name, arr in synth.make_weights(s, 0).items():
        mfs.mfs_load_weights(ctx, name, arr)
    mfs.mfs_prefill(ctx, [0], synth.forced_frames(s, 1, synth.STREAM_PROMPT, PROMPT, 1).transpose(1, 0, 2))
    u = synth.user_frames(s, 1, a.steps, 1)
    for p in range(a.steps):
        text, codes = mfs.mfs_step(ctx, [0], u[p])
    print(f"profile case: {a.layers} temporal / {a.dep_layers} depformer layers, {PROMPT} prompt launches, "
          f"{a.steps} steps; last text token {int(text[0])}")


if __name__ == "__main__":
    main()
