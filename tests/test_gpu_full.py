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


def _compare_rows(dbg, rows, ref, what):
    """Logits and raw argmaxes of step rows `rows` against oracle results `ref`
    (stacked in the same order).  Returns True while every token agrees."""
    H.check_logits(dbg["text_logits"][rows], ref["text_logits"], f"{what} text logits")
    H.check_logits(dbg["dep_logits"][rows], ref["dep_logits"], f"{what} depformer logits")
    H.check_argmax(dbg["text_argmax"][rows], ref["text_logits"], f"{what} text argmax")
    H.check_argmax(dbg["code_argmax"][rows], ref["dep_logits"], f"{what} code argmax")
    return True


def test_full_b8_mixed_windows(mfs, full_weights):
    """Full shape, B = 8: per-slot ring lengths uniform in [0, 3000] (synthetic states
    imported into both sides), decode steps for all eight slots in one call; the
    slots with the shortest and longest windows are checked against the oracle, one
    more slot sits two frames below max_pos (RoPE range end, then MFS_E_RANGE), and a
    copy of a sampled slot stepped alone gives bit-identical results (isolation)."""
    s = synth.FULL.replace(max_slots=9)
    ctx = H.gpu_context(s, full_weights)
    lens = synth.prefill_lengths(1, 8, 0, 3000)
    lens[3] = s.max_pos - 2
    states = {}
    for i in range(8):
        st = synth.slot_state(s, 1, i, int(lens[i]))
        mfs.mfs_import_slot(ctx, i, st)
        if i in (int(np.argmin(lens)), int(np.argmax(np.where(lens < s.max_pos - 2, lens, -1)))):
            states[i] = st
        else:
            del st
    sampled = sorted(states)
    # a bit-exact round trip of the state
    assert np.array_equal(mfs.mfs_export_slot(ctx, sampled[0]), states[sampled[0]])
    mfs.mfs_import_slot(ctx, 8, states[sampled[1]])  # a copy, stepped alone below
    orc = oracle.Oracle(s.replace(max_slots=2), full_weights)
    for k, i in enumerate(sampled):
        orc.import_slot(k, states[i])
    u = synth.user_frames(s, 1, 2, 8)
    alive = [True, True]
    for p in range(2):
        text, codes = mfs.mfs_step(ctx, list(range(8)), u[p])
        dbg = mfs.mfs_read_debug(ctx)
        for k, i in enumerate(sampled):
            if not alive[k]:
                continue
            ref = orc.step([k], u[p][i:i + 1], want_logits=True)
            _compare_rows(dbg, [i], ref, f"B=8 slot {i} (window {min(int(lens[i]) + p + 1, s.window)})")
            alive[k] = bool(text[i] == ref["text"][0] and np.array_equal(codes[i], ref["codes"][0]))
        if p == 0:
            row = sampled[1]
            t1, c1 = mfs.mfs_step(ctx, [8], u[p][row:row + 1])
            d1 = mfs.mfs_read_debug(ctx)
            assert t1[0] == text[row] and np.array_equal(c1[0], codes[row])
            assert np.array_equal(d1["text_logits"][0], dbg["text_logits"][row])
            assert np.array_equal(d1["dep_logits"][0], dbg["dep_logits"][row])
    assert mfs.mfs_position(ctx, 3) == s.max_pos
    with pytest.raises(mfs.MfsError) as e:
        mfs.mfs_step(ctx, [3], u[0][3:4])
    assert e.value.status == "MFS_E_RANGE" and mfs.mfs_position(ctx, 3) == s.max_pos


def test_full_b32_full_rings_with_churn(mfs, full_weights):
    """Full shape, B = 32, every ring full (positions past 3000, so every step wraps);
    after three steps four seeded slots leave, are reset and rejoin empty.  Two of the
    reset slots and two others are followed by the oracle through all six steps."""
    s = synth.FULL.replace(max_slots=32)
    ctx = H.gpu_context(s, full_weights)
    pos = 3000 + synth.uniform_int(1, synth.STREAM_LENGTHS + 1, 32, 0, 2000)
    churn = synth.churn_slots(1, 0, 32, 4)
    keep = [i for i in range(32) if i not in churn]
    sampled = [int(churn[0]), int(churn[1]), keep[0], keep[-1]]
    shared = synth.slot_state(s, 1, 100, 0)
    orc = oracle.Oracle(s.replace(max_slots=4), full_weights)
    for i in range(32):
        if i in sampled:
            st = synth.slot_state(s, 1, 200 + i, int(pos[i]))
            orc.import_slot(sampled.index(i), st)
        else:
            st = shared
            st[4:8] = np.frombuffer(np.int32(pos[i]).tobytes(), np.uint8)  # same ring, own position
        mfs.mfs_import_slot(ctx, i, st)
        del st
    del shared
    u = synth.user_frames(s, 1, 6, 32)
    alive = [True] * 4
    for p in range(6):
        if p == 3:
            for i in churn:
                mfs.mfs_reset_slot(ctx, int(i))
                if i in sampled:
                    orc.reset_slot(sampled.index(int(i)))
                    alive[sampled.index(int(i))] = True
        text, codes = mfs.mfs_step(ctx, list(range(32)), u[p])
        dbg = mfs.mfs_read_debug(ctx)
        for k, i in enumerate(sampled):
            if not alive[k]:
                continue
            ref = orc.step([k], u[p][i:i + 1], want_logits=True)
            _compare_rows(dbg, [i], ref, f"B=32 slot {i} step {p}")
            alive[k] = bool(text[i] == ref["text"][0] and np.array_equal(codes[i], ref["codes"][0]))
    for i in churn:
        assert mfs.mfs_position(ctx, int(i)) == 3


def test_full_b16_prompts_then_decode(mfs, full_weights):
    """Full shape, B = 16: every slot prefills a 250-frame prompt in one call, then decodes.
    A slot's state after the batched prompt equals the same prompt run alone, bit for bit;
    two slots continue against the oracle from their exported states."""
    s = synth.FULL.replace(max_slots=17)
    ctx = H.gpu_context(s, full_weights)
    prompt = synth.forced_frames(s, 1, synth.STREAM_PROMPT, 250, 16)  # [T, B, 17]
    mfs.mfs_prefill(ctx, list(range(16)), prompt.transpose(1, 0, 2))
    mfs.mfs_prefill(ctx, [16], prompt[:, 5:6].transpose(1, 0, 2))
    st5 = mfs.mfs_export_slot(ctx, 5)
    assert np.array_equal(st5, mfs.mfs_export_slot(ctx, 16))
    sampled = [5, 12]
    orc = oracle.Oracle(s.replace(max_slots=2), full_weights)
    orc.import_slot(0, st5)
    del st5
    orc.import_slot(1, mfs.mfs_export_slot(ctx, 12))
    u = synth.user_frames(s, 1, 2, 16)
    alive = [True, True]
    for p in range(2):
        text, codes = mfs.mfs_step(ctx, list(range(16)), u[p])
        dbg = mfs.mfs_read_debug(ctx)
        for k, i in enumerate(sampled):
            if not alive[k]:
                continue
            ref = orc.step([k], u[p][i:i + 1], want_logits=True)
            _compare_rows(dbg, [i], ref, f"B=16 slot {i} frame {250 + p}")
            alive[k] = bool(text[i] == ref["text"][0] and np.array_equal(codes[i], ref["codes"][0]))


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
