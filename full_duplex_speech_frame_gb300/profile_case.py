"""A small case of the frame step for hardware-counter captures.

    python -m full_duplex_speech_frame_gb300.profile_case [--layers L] [--dep-layers DL] [--steps N] [--batch B]
    python -m full_duplex_speech_frame_gb300.profile_case --rvq

--rvq instead runs the Mimi RVQ encode of 2432 frames (D 256, 8 codebooks of
2048, seeded normal latents and codebooks) N times.

The full PersonaPlex widths (4096-d temporal, 32 x 128 heads, FFN 11264,
32000-word text head, 1024-d depformer with 16 per-substep weight sets) with
fewer layers, so that a multi-pass profiler capture holds about 1.5 GB on the
device instead of 17 GB, while the streamed weights (about 1.4 GB per step)
still exceed the L2 cache and DRAM counters keep their meaning.  Launch order:
the prompt (8 frames of every slot: one launch for B = 1 or B >= 5 with the
tensor-core pass, whose prompt chunks take up to 32 rows; more otherwise; none
with --full-rings), then N decode steps of the B slots (B >= 5: the tensor-core
pass; up to 8 slots, the depformer in a second launch on the CUDA-core pass).
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
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--full-rings", action="store_true",
                    help="start every slot from a synthetic state with a full ring (positions past the window)")
    ap.add_argument("--rvq", action="store_true", help="run the Mimi RVQ encode instead of frame steps")
    a = ap.parse_args()
    import torch
    torch.cuda.set_stream(torch.cuda.Stream())
    if a.rvq:
        T, D, C = 2432, 256, 2048
        z = torch.from_numpy(synth.normal_f32(0, 501, 2 * T * D).reshape(2, T, D)).cuda()
        cb = torch.from_numpy(synth.normal_f32(0, 503, 8 * C * D).reshape(8, C, D)).cuda()
        codes = torch.empty(T, 8, dtype=torch.int32, device="cuda")
        for _ in range(a.steps):
            mfs.mfs_rvq_encode(z[0], z[1], cb, codes)
        torch.cuda.synchronize()
        print(f"profile case: RVQ encode of {T} frames x {a.steps}; code of frame 0 {codes[0].tolist()}")
        return
    B = a.batch
    s = synth.FULL.replace(n_layers=a.layers, dep_layers=a.dep_layers, max_slots=B)
    ctx = mfs.context_with_weights(s, synth.make_weights(s, 0))
    slots = list(range(B))
    if a.full_rings:
        import numpy as np
        st = synth.slot_state(s, 1, 300, 0)
        for i in slots:
            st[4:8] = np.frombuffer(np.int32(s.window + 7 * i).tobytes(), np.uint8)
            mfs.mfs_import_slot(ctx, i, st)
    else:
        mfs.mfs_prefill(ctx, slots, synth.forced_frames(s, 1, synth.STREAM_PROMPT, PROMPT, B).transpose(1, 0, 2))
    u = synth.user_frames(s, 1, a.steps, B)
    for p in range(a.steps):
        text, codes = mfs.mfs_step(ctx, slots, u[p])
    start = "full rings" if a.full_rings else f"{PROMPT}-frame prompt"
    print(f"profile case: {a.layers} temporal / {a.dep_layers} depformer layers, B = {B}, {start}, "
          f"{a.steps} steps; last text token {int(text[0])}")


if __name__ == "__main__":
    main()
