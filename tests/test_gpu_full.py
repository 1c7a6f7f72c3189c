"""CUDA path against the oracle at the full PersonaPlex shape (bf16 weights)."""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mfs():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from full_duplex_speech_frame_gb300 import mfs as m
    return m


@pytest.fixture(scope="module")
def full_weights():
    return synth.make_weights(synth.FULL, 0)


def test_full_b1_prompt_then_decode(mfs, full_weights):
    """Full shape, B = 1: a 250-frame forced prompt, then decode frames with the user rows
    supplied and the agent rows generated; the first frames are compared with the oracle."""
    s = synth.FULL.replace(max_slots=1)
    w = full_weights
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    prompt = synth.forced_frames(s, 1, synth.STREAM_PROMPT, 250, 1)[:, 0]
    mfs.mfs_prefill(ctx, [0], prompt[None])
    orc.prefill(0, prompt)
    assert mfs.mfs_position(ctx, 0) == orc.position(0) == 250
    u = synth.user_frames(s, 1, 4, 1)
    flips = 0
    for p in range(4):
        text, codes = mfs.mfs_step(ctx, [0], u[p])
        dbg = mfs.mfs_read_debug(ctx)
        ref = orc.step([0], u[p], want_logits=True)
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {250 + p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {250 + p}")
        flips += H.check_argmax(dbg["text_argmax"], ref["text_logits"], "text argmax")
        flips += H.check_argmax(dbg["code_argmax"], ref["dep_logits"], "code argmax")
        if not (np.array_equal(text, ref["text"]) and np.array_equal(codes, ref["codes"])):
            break


def test_full_teacher_forced_wrap(mfs, full_weights):
    """Full model dimensions with the ring shortened to 24 frames: 40 forced frames wrap it."""
    s = synth.FULL.replace(max_slots=2, window=24)
    w = full_weights
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    prompt = synth.forced_frames(s, 3, synth.STREAM_PROMPT, 36, 1)[:, 0]
    mfs.mfs_prefill(ctx, [1], prompt[None])
    orc.prefill(1, prompt)
    z = synth.forced_frames(s, 3, synth.STREAM_FORCED, 3, 1)
    for p in range(3):
        text, codes = mfs.mfs_step(ctx, [1], z[p])
        dbg = mfs.mfs_read_debug(ctx)
        ref = orc.step([1], z[p], want_logits=True)
        np.testing.assert_array_equal(codes, ref["codes"])
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {36 + p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {36 + p}")
        H.check_argmax(dbg["code_argmax"], ref["dep_logits"], "code argmax")
