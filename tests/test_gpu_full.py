"""CUDA path against the oracle at the full PersonaPlex shape (bf16 weights), over
the five workloads' stated run lengths.  The oracle follows the GPU's chosen
tokens (follow mode), so a legal flip at a near tie (top-2 margin below 0.1)
does not end the comparison: every frame of every sampled slot is compared
(logits within 2e-2 x RMS elementwise, greedy tokens equal unless the oracle's
margin is below 0.1, outputs bit for bit).  The pages' own gate for this model
is greedy agreement over at least 100 frames (SGLang-Omni cookbook,
PersonaPlex, "Reference parity")."""
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


def step_followed(mfs, ctx, slots, frames_p, orc, rows, orc_slots, tally, label):
    """One GPU step of `slots`; then the oracle steps its slots `orc_slots` (GPU rows
    `rows`) following the GPU's chosen tokens.  Outputs compared bit for bit."""
    text, codes = mfs.mfs_step(ctx, list(slots), frames_p)
    dbg = mfs.mfs_read_debug(ctx)
    if rows:
        fol = H.follow_tokens(text[rows], codes[rows], dbg["code_argmax"][rows])
        ref = orc.step(list(orc_slots), frames_p[rows], want_logits=True, follow=fol)
        np.testing.assert_array_equal(text[rows], ref["text"], err_msg=label)
        np.testing.assert_array_equal(codes[rows], ref["codes"], err_msg=label)
        tally.step(dbg, rows, ref, label)
    return text, codes, dbg


def test_full_b1_prompt_then_125_decode_frames(mfs, full_weights):
    """Config 2: B = 1, a 250-frame forced prompt, then 125 decode frames (10 s) with the
    user rows supplied and the agent rows generated; every frame compared."""
    s = synth.FULL.replace(max_slots=1)
    w = full_weights
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    prompt = synth.forced_frames(s, 1, synth.STREAM_PROMPT, 250, 1)[:, 0]
    mfs.mfs_prefill(ctx, [0], prompt[None])
    orc.prefill(0, prompt)
    assert mfs.mfs_position(ctx, 0) == orc.position(0) == 250
    u = synth.user_frames(s, 1, 125, 1)
    tally = H.Tally("config 2 (B=1, 250-frame prompt, 125 decode frames)")
    for p in range(125):
        step_followed(mfs, ctx, [0], u[p], orc, [0], [0], tally, f"frame {250 + p}")
    print(tally.report())
    assert tally.frames == 125


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


def test_full_b8_mixed_windows_125_frames(mfs, full_weights):
    """Config 3: B = 8, per-slot ring lengths uniform in [0, 3000] (synthetic states imported
    into both sides, NaN in every ring row outside the window), 125 decode frames for all eight slots in one call (the tensor-core
    pass).  The slots with the shortest and the longest window are followed by the oracle
    over all 125 frames.  Isolation: a copy of a sampled slot stepped in another batch of
    eight, beside other slots, gives bit-identical results.  A ninth slot two frames below
    max_pos reaches the RoPE range end, then gets MFS_E_RANGE."""
    s = synth.FULL.replace(max_slots=17)
    ctx = H.gpu_context(s, full_weights)
    lens = synth.prefill_lengths(1, 8, 0, 3000)
    states = {}
    for i in range(8):
        # ring rows the window never reaches hold NaN: any read of one would show
        st = H.nan_stale_rows(synth.slot_state(s, 1, i, int(lens[i])), s, int(lens[i]))
        mfs.mfs_import_slot(ctx, i, st)
        if i in (int(np.argmin(lens)), int(np.argmax(lens))):
            states[i] = st
        else:
            del st
    sampled = sorted(states)
    assert np.array_equal(mfs.mfs_export_slot(ctx, sampled[0]), states[sampled[0]])  # bit-exact round trip
    mfs.mfs_import_slot(ctx, 8, states[sampled[1]])      # a copy, stepped in the other batch
    for i in range(9, 16):                                # its neighbours there
        mfs.mfs_import_slot(ctx, i, synth.slot_state(s, 2, i, int(lens[i - 8]) // 2))
    mfs.mfs_import_slot(ctx, 16, synth.slot_state(s, 3, 16, s.max_pos - 2))
    orc = oracle.Oracle(s.replace(max_slots=2), full_weights)
    for k, i in enumerate(sampled):
        orc.import_slot(k, states[i])
    del states
    u = synth.user_frames(s, 1, 125, 8)
    other = synth.user_frames(s, 2, 4, 8)
    tally = H.Tally("config 3 (B=8, windows U[0,3000], 125 frames)")
    for p in range(125):
        text, codes, dbg = step_followed(mfs, ctx, list(range(8)), u[p], orc, sampled, [0, 1], tally,
                                         f"B=8 frame {p}")
        if p < 4:
            row = sampled[1]
            batch = [8] + list(range(9, 16))
            inp = other[p].copy()
            inp[0] = u[p][row]
            t1, c1 = mfs.mfs_step(ctx, batch, inp)
            d1 = mfs.mfs_read_debug(ctx)
            assert t1[0] == text[row] and np.array_equal(c1[0], codes[row])
            assert np.array_equal(d1["text_logits"][0], dbg["text_logits"][row])
            assert np.array_equal(d1["dep_logits"][0], dbg["dep_logits"][row])
    print(tally.report())
    assert tally.frames == 250
    # the RoPE range end: two frames, then MFS_E_RANGE with the state unchanged
    for p in range(2):
        mfs.mfs_step(ctx, [16], u[p][:1])
    assert mfs.mfs_position(ctx, 16) == s.max_pos
    with pytest.raises(mfs.MfsError) as e:
        mfs.mfs_step(ctx, [16], u[0][:1])
    assert e.value.status == "MFS_E_RANGE" and mfs.mfs_position(ctx, 16) == s.max_pos


def test_full_b32_full_rings_with_churn_250_frames(mfs, full_weights):
    """Config 4: B = 32, every ring full (positions past 3000, so every step wraps), 250
    frames; every 20 frames four seeded slots leave, are reset and rejoin empty.  The
    oracle follows one slot that never leaves through all 250 frames, and one slot
    reset at frame 200 (and not again) from its rejoin to the end."""
    s = synth.FULL.replace(max_slots=32)
    ctx = H.gpu_context(s, full_weights)
    pos = 3000 + synth.uniform_int(1, synth.STREAM_LENGTHS + 1, 32, 0, 2000)
    events = {20 * e: synth.churn_slots(1, e - 1, 32, 4) for e in range(1, 13)}  # frames 20, 40, .., 240
    churned = set(int(i) for ev in events.values() for i in ev)
    keep = [i for i in range(32) if i not in churned]
    assert keep, "some slot must stay for the whole run"
    late = [int(i) for i in events[200] if all(i not in events[f] for f in (220, 240))][0]
    stay = keep[0]
    shared = synth.slot_state(s, 1, 100, 0)
    orc = oracle.Oracle(s.replace(max_slots=2), full_weights)
    for i in range(32):
        if i == stay:
            st = synth.slot_state(s, 1, 200 + i, int(pos[i]))
            orc.import_slot(0, st)
        else:
            st = shared
            st[4:8] = np.frombuffer(np.int32(pos[i]).tobytes(), np.uint8)  # same ring, own position
        mfs.mfs_import_slot(ctx, i, st)
        del st
    del shared
    u = synth.user_frames(s, 1, 250, 32)
    tally = H.Tally("config 4 (B=32, full rings, churn every 20 frames, 250 frames)")
    late_on = False
    for p in range(250):
        if p in events:
            for i in events[p]:
                mfs.mfs_reset_slot(ctx, int(i))
            if p == 200:
                orc.reset_slot(1)
                late_on = True
        rows, oslots = [stay], [0]
        if late_on:
            rows, oslots = [stay, late], [0, 1]
        step_followed(mfs, ctx, list(range(32)), u[p], orc, rows, oslots, tally, f"B=32 frame {p}")
    print(tally.report())
    assert tally.frames == 250 + 50
    assert mfs.mfs_position(ctx, late) == 50


def test_full_b16_prompts_then_500_decode_frames(mfs, full_weights):
    """Config 5: B = 16, every slot prefills a 250-frame prompt of random text and code
    tokens in one call (the tensor-core pass), then decodes 500 frames, reaching position
    750 of the 8192-position RoPE range.  A slot's state after the batched prompt equals
    the same prompt run in another batch of 16 beside other prompts, bit for bit; one slot
    is followed by the oracle (its own prompt path) over all 500 decode frames."""
    s = synth.FULL.replace(max_slots=32)
    ctx = H.gpu_context(s, full_weights)
    prompt = synth.forced_frames(s, 1, synth.STREAM_PROMPT, 250, 16)  # [T, B, 17]
    mfs.mfs_prefill(ctx, list(range(16)), prompt.transpose(1, 0, 2))
    other = synth.forced_frames(s, 4, synth.STREAM_PROMPT, 250, 16)
    other[:, 0] = prompt[:, 5]
    mfs.mfs_prefill(ctx, list(range(16, 32)), other.transpose(1, 0, 2))
    assert np.array_equal(mfs.mfs_export_slot(ctx, 5), mfs.mfs_export_slot(ctx, 16))
    orc = oracle.Oracle(s.replace(max_slots=1), full_weights)
    orc.prefill(0, prompt[:, 5])
    u = synth.user_frames(s, 1, 500, 16)
    tally = H.Tally("config 5 (B=16, 250-frame prompts, 500 decode frames)")
    for p in range(500):
        step_followed(mfs, ctx, list(range(16)), u[p], orc, [5], [0], tally, f"B=16 frame {250 + p}")
    print(tally.report())
    assert tally.frames == 500 and mfs.mfs_position(ctx, 5) == 750


def test_full_sampling_heads_draw_from_gpu_logits(mfs, full_weights):
    """Full shape, B = 2 sampled slots (32000-word text head, top-25; audio top-250): every
    generated token is the oracle sampler's draw from the GPU's own logits with the same
    uniform, except at a CDF boundary where fp32 and fp64 may part."""
    from tests.test_gpu_tiny import _near_cdf_boundary
    s = synth.FULL.replace(max_slots=2)
    ctx = H.gpu_context(s, full_weights)
    mfs.mfs_prefill(ctx, [0, 1], synth.forced_frames(s, 5, synth.STREAM_PROMPT, 12, 2).transpose(1, 0, 2))
    for slot in (0, 1):
        mfs.mfs_set_sampling(ctx, slot, 0.7, 25, 0.8, 250)
    u = synth.user_frames(s, 5, 3, 2)
    unif = ((synth.uniform_int(5, 98, 3 * 2 * 17, 0, 1 << 24).reshape(3, 2, 17)) + 0.5) / float(1 << 24)
    checked = 0
    for p in range(3):
        text, codes = mfs.mfs_step_sampled(ctx, [0, 1], u[p], unif[p])
        dbg = mfs.mfs_read_debug(ctx)
        for i in range(2):
            for k in range(9):
                if p == 0 and s.delays[k] == 1:
                    continue  # frame p - 1 belongs to the prompt: its token was supplied, not drawn
                lg = dbg["text_logits"][i] if k == 0 else dbg["dep_logits"][i][k - 1]
                temp, topk = (0.7, 25) if k == 0 else (0.8, 250)
                got = text[i] if k == 0 else codes[i][k - 1]
                want = oracle.sample_topk(lg, temp, topk, unif[p][i][k])
                if got != want:
                    assert _near_cdf_boundary(lg, temp, topk, unif[p][i][k]), (p, i, k, got, want)
                checked += 1
    assert checked == 40
