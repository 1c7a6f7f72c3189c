"""CUDA path against the oracle on the tiny Moshi-shaped LM (fp32 weights), plus
the integer invariants (isolation, reset, prompt path, errors) bit for bit."""
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


def tiny(**kw):
    return synth.TINY.replace(**kw)


def lockstep(mfs, s, w, frames, slots=(0,), ctx=None, orc=None):
    """Run GPU and oracle side by side over frames [T, n, 17]; returns per-step records."""
    ctx = ctx or H.gpu_context(s, w)
    orc = orc or oracle.Oracle(s, w)
    recs = []
    for p in range(frames.shape[0]):
        text, codes = mfs.mfs_step(ctx, list(slots), frames[p])
        dbg = mfs.mfs_read_debug(ctx)
        ref = orc.step(list(slots), frames[p], want_logits=True)
        recs.append((text, codes, dbg, ref))
    return recs, ctx, orc


@pytest.mark.parametrize("gain_std", [0.0, 0.1])
def test_tiny_teacher_forced_parity(mfs, gain_std):
    s = tiny()
    w = synth.make_weights(s, 0, gain_std=gain_std)
    z = synth.forced_frames(s, 0, synth.STREAM_FORCED, 32, 1)
    recs, _, _ = lockstep(mfs, s, w, z)
    for p, (text, codes, dbg, ref) in enumerate(recs):
        np.testing.assert_array_equal(text, ref["text"])
        np.testing.assert_array_equal(codes, ref["codes"])
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")
        H.check_argmax(dbg["text_argmax"], ref["text_logits"], f"text argmax, frame {p}")
        H.check_argmax(dbg["code_argmax"], ref["dep_logits"], f"code argmax, frame {p}")


def test_tiny_free_running_config(mfs):
    """The tiny workload as specified: seed 0, B=1, 32 frames, user rows random, rest generated."""
    s = tiny()
    w = synth.make_weights(s, 0)
    u = synth.user_frames(s, 0, 32, 1)
    recs, _, _ = lockstep(mfs, s, w, u)
    compared = 0
    for p, (text, codes, dbg, ref) in enumerate(recs):
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")
        H.check_argmax(dbg["text_argmax"], ref["text_logits"], f"text argmax, frame {p}")
        H.check_argmax(dbg["code_argmax"], ref["dep_logits"], f"code argmax, frame {p}")
        if not (np.array_equal(text, ref["text"]) and np.array_equal(codes, ref["codes"])):
            break   # a legal flip (checked above): histories diverge from here on
        compared += 1
    assert compared >= 16, f"only {compared} frames matched token for token"


def test_tiny_long_window_split_attention(mfs):
    """W = 200 with two slots at different positions (a 150-frame prompt on one): windows
    of more than 64 keys are split into chunks and merged; one slot wraps a W = 200 ring
    after a 190-frame prompt.  Compared with the oracle, and slot 1 alone is bit-identical."""
    s = tiny(window=200, max_slots=3)
    w = synth.make_weights(s, 6, gain_std=0.1)
    ctx = H.gpu_context(s, w)
    orc = oracle.Oracle(s, w)
    pr0 = synth.forced_frames(s, 6, synth.STREAM_PROMPT, 150, 1)[:, 0]
    pr1 = synth.forced_frames(s, 7, synth.STREAM_PROMPT, 190, 1)[:, 0]
    mfs.mfs_prefill(ctx, [0], pr0[None])
    mfs.mfs_prefill(ctx, [1], pr1[None])
    mfs.mfs_prefill(ctx, [2], pr1[None])
    orc.prefill(0, pr0)
    orc.prefill(1, pr1)
    z = synth.forced_frames(s, 8, synth.STREAM_FORCED, 16, 2)
    for p in range(16):
        text, codes = mfs.mfs_step(ctx, [0, 1], z[p])
        dbg = mfs.mfs_read_debug(ctx)
        ref = orc.step([0, 1], z[p], want_logits=True)
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")
        np.testing.assert_array_equal(codes, ref["codes"])
        t2, c2 = mfs.mfs_step(ctx, [2], z[p][1:2])
        d2 = mfs.mfs_read_debug(ctx)
        assert np.array_equal(d2["text_logits"][0], dbg["text_logits"][1])
        assert np.array_equal(d2["dep_logits"][0], dbg["dep_logits"][1])


def test_tiny_ring_wraps(mfs):
    """W = 8 over 40 frames: every step after the 8th wraps the ring."""
    s = tiny(window=8)
    w = synth.make_weights(s, 2, gain_std=0.1)
    z = synth.forced_frames(s, 2, synth.STREAM_FORCED, 40, 1)
    recs, _, _ = lockstep(mfs, s, w, z)
    for p, (text, codes, dbg, ref) in enumerate(recs):
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")


def test_tiny_batch_of_four_mixed_lengths(mfs):
    """Four slots at different positions (prompts of 0, 3, 9, 70 frames; W = 64) in one batch."""
    s = tiny()
    w = synth.make_weights(s, 3, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    for slot, T in enumerate([0, 3, 9, 70]):
        if T:
            pr = synth.forced_frames(s, 10 + slot, synth.STREAM_PROMPT, T, 1)[:, 0]
            mfs.mfs_prefill(ctx, [slot], pr[None])
            orc.prefill(slot, pr)
    order = [2, 0, 3, 1]
    frames = synth.forced_frames(s, 4, synth.STREAM_FORCED, 6, 4)
    recs, _, _ = lockstep(mfs, s, w, frames, slots=order, ctx=ctx, orc=orc)
    for p, (text, codes, dbg, ref) in enumerate(recs):
        np.testing.assert_array_equal(codes, ref["codes"])
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")
        H.check_argmax(dbg["code_argmax"], ref["dep_logits"], f"code argmax, frame {p}")


def test_persistent_and_per_phase_launches_bit_identical(mfs):
    s = tiny(window=16)
    w = synth.make_weights(s, 5, gain_std=0.1)
    u = synth.user_frames(s, 5, 20, 2)
    a, b = H.gpu_context(s, w), H.gpu_context(s, w)
    mfs.mfs_set_mode(b, 1)
    for p in range(20):
        ta, ca = mfs.mfs_step(a, [0, 1], u[p])
        tb, cb = mfs.mfs_step(b, [0, 1], u[p])
        assert mfs.mfs_launches_per_step(a) == 1 and mfs.mfs_launches_per_step(b) > 100
        np.testing.assert_array_equal(ta, tb)
        np.testing.assert_array_equal(ca, cb)
        da, db = mfs.mfs_read_debug(a), mfs.mfs_read_debug(b)
        for k in da:
            np.testing.assert_array_equal(da[k], db[k])


def test_slot_isolation_bit_exact(mfs):
    """A slot's outputs are bit-identical alone, or batched with any other slots' contents."""
    s = tiny(max_slots=4)
    w = synth.make_weights(s, 6, gain_std=0.1)
    T = 12
    mine = synth.user_frames(s, 60, T, 1)[:, 0]
    others = [synth.user_frames(s, 61 + k, T, 3) for k in range(2)]
    runs = []
    for mode in range(3):
        ctx = H.gpu_context(s, w)
        outs = []
        for p in range(T):
            if mode == 0:
                slots, fr = [1], mine[p][None]
            elif mode == 1:
                slots, fr = [3, 1], np.stack([others[0][p, 0], mine[p]])
            else:
                slots, fr = [0, 2, 1, 3], np.stack([others[1][p, 0], others[1][p, 1], mine[p], others[1][p, 2]])
            text, codes = mfs.mfs_step(ctx, slots, fr)
            dbg = mfs.mfs_read_debug(ctx)
            i = slots.index(1)
            outs.append((text[i], codes[i].copy(), dbg["text_logits"][i].copy(), dbg["dep_logits"][i].copy()))
        runs.append(outs)
    for p in range(T):
        for r in runs[1:]:
            assert runs[0][p][0] == r[p][0]
            for k in (1, 2, 3):
                np.testing.assert_array_equal(runs[0][p][k], r[p][k])


def test_reset_equals_fresh(mfs):
    s = tiny()
    w = synth.make_weights(s, 7)
    u = synth.user_frames(s, 70, 8, 1)
    ctx = H.gpu_context(s, w)
    for p in range(5):
        mfs.mfs_step(ctx, [2], synth.user_frames(s, 71, 5, 1)[p])
    mfs.mfs_reset_slot(ctx, 2)
    assert mfs.mfs_position(ctx, 2) == 0
    fresh = H.gpu_context(s, w)
    for p in range(8):
        a = mfs.mfs_step(ctx, [2], u[p])
        da = mfs.mfs_read_debug(ctx)
        b = mfs.mfs_step(fresh, [2], u[p])
        db = mfs.mfs_read_debug(fresh)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])
        np.testing.assert_array_equal(da["dep_logits"], db["dep_logits"])


def test_prompt_path_equals_forced_steps(mfs):
    """The prompt path takes the first 16 frames of both slots as one chunk of 32 rows
    (earlier frames of a slot read from the chunk's own rows), the rest one frame per
    launch; it equals 30 forced steps bit for bit."""
    s = tiny(window=16)
    w = synth.make_weights(s, 8, gain_std=0.1)
    z = synth.forced_frames(s, 80, synth.STREAM_PROMPT, 30, 2)
    nxt = synth.user_frames(s, 81, 4, 2)
    a, b = H.gpu_context(s, w), H.gpu_context(s, w)
    mfs.mfs_prefill(a, [0, 1], z.transpose(1, 0, 2))
    for p in range(30):
        mfs.mfs_step(b, [0, 1], z[p])
    assert mfs.mfs_position(a, 0) == mfs.mfs_position(b, 1) == 30
    for p in range(4):
        ta, ca = mfs.mfs_step(a, [0, 1], nxt[p])
        da = mfs.mfs_read_debug(a)
        tb, cb = mfs.mfs_step(b, [0, 1], nxt[p])
        db = mfs.mfs_read_debug(b)
        np.testing.assert_array_equal(ta, tb)
        np.testing.assert_array_equal(ca, cb)
        np.testing.assert_array_equal(da["text_logits"], db["text_logits"])


def test_errors_are_rejected_before_launch(mfs):
    s = tiny(max_pos=6, max_slots=2)
    w = synth.make_weights(s, 9)
    ctx = H.gpu_context(s, w)
    good = synth.user_frames(s, 90, 8, 2)
    mfs.mfs_step(ctx, [0], good[0, :1])
    ref = mfs.mfs_read_debug(ctx)

    def expect(status, fn, *a):
        with pytest.raises(mfs.MfsError) as e:
            fn(*a)
        assert e.value.status == status, str(e.value)

    bad = good[1, :1].copy()
    bad[0, 5] = s.card
    expect("MFS_E_TOKEN", mfs.mfs_step, ctx, [0], bad)
    bad = good[1, :1].copy()
    bad[0, 0] = -2
    expect("MFS_E_TOKEN", mfs.mfs_step, ctx, [0], bad)
    expect("MFS_E_SLOT", mfs.mfs_step, ctx, [2], good[1, :1])
    expect("MFS_E_ARG", mfs.mfs_step, ctx, [1, 1], good[1])
    expect("MFS_E_TOKEN", mfs.mfs_prefill, ctx, [1], good[1:3, :1].transpose(1, 0, 2))  # -1 in a prompt
    assert mfs.mfs_position(ctx, 0) == 1 and mfs.mfs_position(ctx, 1) == 0
    # nothing ran: the last step's diagnostics are still those of the first step
    np.testing.assert_array_equal(mfs.mfs_read_debug(ctx)["text_logits"], ref["text_logits"])
    for p in range(1, 6):
        mfs.mfs_step(ctx, [0], good[p, :1])
    expect("MFS_E_RANGE", mfs.mfs_step, ctx, [0], good[6, :1])
    assert mfs.mfs_position(ctx, 0) == 6
    # a context whose weights are incomplete refuses to step
    empty = mfs.mfs_create(H.config_of(s))
    expect("MFS_E_STATE", mfs.mfs_step, empty, [0], good[0, :1])
    expect("MFS_E_STATE", mfs.mfs_load_weights, empty, "layers.0.wqkv", w["layers.0.wo"])
    expect("MFS_E_STATE", mfs.mfs_load_weights, empty, "no.such.tensor", w["layers.0.wo"])


def test_device_resident_step_and_deferred_token_error(mfs):
    import torch
    s = tiny()
    w = synth.make_weights(s, 11)
    u = synth.user_frames(s, 110, 6, 2)
    a, b = H.gpu_context(s, w), H.gpu_context(s, w)
    dcodes = torch.from_numpy(u).cuda()
    dtext = torch.empty(2, dtype=torch.int32, device="cuda")
    dco = torch.empty(2, 16, dtype=torch.int32, device="cuda")
    for p in range(4):
        mfs.mfs_step_device(a, [1, 0], dcodes[p], dtext, dco)
        mfs.mfs_sync(a)
        tb, cb = mfs.mfs_step(b, [1, 0], u[p])
        np.testing.assert_array_equal(dtext.cpu().numpy(), tb)
        np.testing.assert_array_equal(dco.cpu().numpy(), cb)
    # an out-of-range device token turns that step and the next into no-ops
    bad = dcodes[4].clone()
    bad[0, 3] = s.card + 5
    mfs.mfs_step_device(a, [1, 0], bad, dtext, dco)
    mfs.mfs_step_device(a, [1, 0], dcodes[5], dtext, dco)
    with pytest.raises(mfs.MfsError) as e:
        mfs.mfs_sync(a)
    assert e.value.status == "MFS_E_TOKEN"
    assert mfs.mfs_position(a, 0) == 4 and mfs.mfs_position(a, 1) == 4
    # and the context carries on exactly like one that never saw the bad step
    for p in (4, 5):
        ta, ca = mfs.mfs_step(a, [1, 0], u[p])
        tb, cb = mfs.mfs_step(b, [1, 0], u[p])
        np.testing.assert_array_equal(ta, tb)
        np.testing.assert_array_equal(ca, cb)


def test_tiny_skip_settled_substeps(mfs):
    """With trailing settled substeps skipped (user streams supplied in decode: substeps 8..15),
    every output and the logits of the substeps that run are bit-identical to the full run;
    a fully supplied frame skips the whole depformer.  The full run is checked against the oracle."""
    s = tiny(max_slots=2)
    w = synth.make_weights(s, 9, gain_std=0.1)
    a, b = H.gpu_context(s, w), H.gpu_context(s, w)
    mfs.mfs_set_skip_settled(b, True)
    orc = oracle.Oracle(s, w)
    u = synth.user_frames(s, 9, 12, 2)
    z = synth.forced_frames(s, 9, synth.STREAM_FORCED, 3, 2)
    frames = np.concatenate([u, z, u[:3]], axis=0)
    for p in range(frames.shape[0]):
        ta, ca = mfs.mfs_step(a, [0, 1], frames[p])
        da = mfs.mfs_read_debug(a)
        tb, cb = mfs.mfs_step(b, [0, 1], frames[p])
        db = mfs.mfs_read_debug(b)
        ref = orc.step([0, 1], frames[p], want_logits=True)
        H.check_logits(da["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")
        np.testing.assert_array_equal(ta, tb)
        np.testing.assert_array_equal(ca, cb)
        np.testing.assert_array_equal(da["text_logits"], db["text_logits"])
        ran = db["code_argmax"][0] >= 0
        # stream k is settled when its token for frame p - delay[k] was supplied (or that frame is < 0)
        settled = [all((frames[p][i][k] >= 0) if s.delays[k] == 0 else (p == 0 or frames[p - 1][i][k] >= 0)
                       for i in range(2)) for k in range(17)]
        jend = 16
        while jend > 0 and settled[jend]:
            jend -= 1
        assert np.array_equal(ran, np.arange(16) < jend), f"frame {p}: substeps run {np.flatnonzero(ran)}, want < {jend}"
        np.testing.assert_array_equal(da["dep_logits"][:, ran], db["dep_logits"][:, ran])
        np.testing.assert_array_equal(da["code_argmax"][:, ran], db["code_argmax"][:, ran])


def _near_cdf_boundary(lg, temp, k, u, tol=1e-4):
    """True when u * total lies within tol * total of a candidate's cumulative weight
    (index order), where an fp32 and an fp64 evaluation may legitimately disagree."""
    lg = np.asarray(lg, np.float64)
    k = min(k, lg.size)
    cand = sorted(sorted(range(lg.size), key=lambda i: (-lg[i], i))[:k])
    wts = np.exp((lg[cand] - lg.max()) / temp)
    cum = np.cumsum(wts)
    return bool(np.min(np.abs(cum - u * cum[-1])) < tol * cum[-1])


def test_tiny_sampling_heads(mfs):
    """Two sampled slots (text 0.7 / top-25, audio 0.8 / top-250; and top-k past the
    vocabularies, which keeps every candidate).  Every generated token equals the oracle's
    sampler applied to the GPU's own logits with the same uniform (an fp32/fp64
    disagreement is allowed only at a CDF boundary); logits follow the oracle, which
    samples with the same uniforms, until a legal divergence."""
    s = tiny(max_slots=2)
    w = synth.make_weights(s, 11, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    cfg = {0: (0.7, 25, 0.8, 250), 1: (1.0, 5000, 1.3, 2048)}
    for slot, c in cfg.items():
        mfs.mfs_set_sampling(ctx, slot, *c)
        orc.set_sampling(slot, *c)
    T = 16
    u = synth.user_frames(s, 11, T, 2)
    unif = ((synth.uniform_int(11, 99, T * 2 * 17, 0, 1 << 24).reshape(T, 2, 17)) + 0.5) / float(1 << 24)
    checked = compared = 0
    for p in range(T):
        text, codes = mfs.mfs_step_sampled(ctx, [0, 1], u[p], unif[p])
        dbg = mfs.mfs_read_debug(ctx)
        ref = orc.step([0, 1], u[p], want_logits=True, uniforms=unif[p])
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")
        for i in range(2):
            tt, tk, at, ak = cfg[i]
            for k in range(9):  # text and agent streams 1..8 are generated
                f = p - s.delays[k]
                if f < 0:
                    continue
                lg = dbg["text_logits"][i] if k == 0 else dbg["dep_logits"][i][k - 1]
                temp, topk = (tt, tk) if k == 0 else (at, ak)
                got = text[i] if k == 0 else codes[i][k - 1]
                want = oracle.sample_topk(lg, temp, topk, unif[p][i][k])
                if got != want:
                    assert _near_cdf_boundary(lg, temp, topk, unif[p][i][k]), (p, i, k, got, want)
                checked += 1
        compared += 1
        if not (np.array_equal(text, ref["text"]) and np.array_equal(codes, ref["codes"])):
            break  # a draw at a CDF boundary went the other way: histories diverge from here
    assert checked >= 60 and compared >= 4, (checked, compared)
    with pytest.raises(mfs.MfsError):
        bad = unif[0].copy()
        bad[0][3] = 1.0
        mfs.mfs_step_sampled(ctx, [0, 1], u[0], bad)


def test_tiny_device_wait_gives_up_and_context_recovers(mfs):
    """A phase launched without its input waits, gives up after the (shortened) limit and
    reports MFS_E_DEVICE with the wait site; the context then runs normal steps that match
    the oracle (the stalled slot is reset first)."""
    s = tiny(max_slots=2)
    w = synth.make_weights(s, 12, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    mfs.mfs_set_wait_limit(ctx, 50)
    u = synth.user_frames(s, 12, 6, 2)
    mfs.mfs_step(ctx, [0, 1], u[0])
    orc.step([0, 1], u[0])
    with pytest.raises(mfs.MfsError) as e:
        mfs.mfs_debug_stall(ctx, 0)
    assert e.value.status == "MFS_E_DEVICE" and "gave up" in str(e.value)
    mfs.mfs_reset_slot(ctx, 0)
    orc.reset_slot(0)
    for p in range(1, 6):
        text, codes = mfs.mfs_step(ctx, [0, 1], u[p])
        dbg = mfs.mfs_read_debug(ctx)
        ref = orc.step([0, 1], u[p], want_logits=True)
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")


def test_tiny_session_priming(mfs):
    """Priming (voice prompt, silence, persona text, silence) through the prompt path on the
    GPU, then decode: logits follow the oracle primed with the same frames."""
    from full_duplex_speech_frame_gb300.priming import priming_frames, prime_slot
    s = tiny(max_slots=2)
    w = synth.make_weights(s, 13, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    voice = synth.uniform_int(13, 401, 6 * 8, 0, s.card).reshape(6, 8)
    persona = synth.uniform_int(13, 402, 5, 0, s.text_vocab)
    f = priming_frames(voice, persona, text_pad=3, agent_silence=[7] * 8, user_fill=[11] * 8,
                       silence_after_voice=2, silence_after_persona=2)
    prime_slot(ctx, 1, f)
    orc.prefill(1, f)
    assert mfs.mfs_position(ctx, 1) == orc.position(1) == f.shape[0]
    u = synth.user_frames(s, 13, 4, 1)
    for p in range(4):
        text, codes = mfs.mfs_step(ctx, [1], u[p])
        dbg = mfs.mfs_read_debug(ctx)
        ref = orc.step([1], u[p], want_logits=True)
        H.check_logits(dbg["text_logits"], ref["text_logits"], f"text logits, frame {p}")
        H.check_logits(dbg["dep_logits"], ref["dep_logits"], f"depformer logits, frame {p}")
        if not (np.array_equal(text, ref["text"]) and np.array_equal(codes, ref["codes"])):
            break


def test_tiny_sampling_with_skipped_substeps(mfs):
    """Sampling and skipped settled substeps together: every output equals a sampled run
    without skipping (same uniforms), bit for bit."""
    s = tiny(max_slots=2)
    w = synth.make_weights(s, 14, gain_std=0.1)
    a, b = H.gpu_context(s, w), H.gpu_context(s, w)
    for ctx in (a, b):
        for slot in (0, 1):
            mfs.mfs_set_sampling(ctx, slot, 0.7, 25, 0.8, 250)
    mfs.mfs_set_skip_settled(b, True)
    u = synth.user_frames(s, 14, 8, 2)
    unif = ((synth.uniform_int(14, 97, 8 * 2 * 17, 0, 1 << 24).reshape(8, 2, 17)) + 0.5) / float(1 << 24)
    for p in range(8):
        ta, ca = mfs.mfs_step_sampled(a, [0, 1], u[p], unif[p])
        tb, cb = mfs.mfs_step_sampled(b, [0, 1], u[p], unif[p])
        np.testing.assert_array_equal(ta, tb)
        np.testing.assert_array_equal(ca, cb)


def test_tiny_slot_state_import_rejects_bad_headers(mfs):
    """Import checks the header against the context before touching the slot."""
    s = tiny(max_slots=2, weight_dtype="bf16", kv_dtype="bf16", window=8)
    w = synth.make_weights(s, 15, gain_std=0.1)
    ctx = H.gpu_context(s, w)
    good = synth.slot_state(s, 15, 0, 5)
    mfs.mfs_import_slot(ctx, 1, good)
    assert mfs.mfs_position(ctx, 1) == 5
    cases = {"window": (8, 12), "dtype": (12, 16), "position": (4, 8)}
    for what, (lo, hi) in cases.items():
        bad = good.copy()
        bad[lo:hi] = np.frombuffer(np.int32(99999).tobytes(), np.uint8)
        with pytest.raises(mfs.MfsError) as e:
            mfs.mfs_import_slot(ctx, 0, bad)
        assert e.value.status == "MFS_E_ARG", what
    bad = good.copy()
    bad[16:20] = np.frombuffer(np.int32(s.text_vocab).tobytes(), np.uint8)  # history token out of range
    with pytest.raises(mfs.MfsError):
        mfs.mfs_import_slot(ctx, 0, bad)
    with pytest.raises(mfs.MfsError):
        mfs.mfs_import_slot(ctx, 0, good[:-16])
    assert mfs.mfs_position(ctx, 0) == 0  # untouched
    np.testing.assert_array_equal(mfs.mfs_export_slot(ctx, 1), good)
