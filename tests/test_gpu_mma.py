"""Tensor-core weight pass (batches of 5..32 slots, bf16 weights) against the
oracle on the tiny Moshi-shaped LM with bf16 weights and key/value cache.  The
tiny matrices are a few tiles, so most tiles are shared by several CTAs
(partial sums handed to the tile's owner), and the last tiles of the text
head, the depformer gate/up and the depformer down projection are ragged in
rows or in K."""
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


def tiny_bf16(**kw):
    return synth.TINY.replace(weight_dtype="bf16", kv_dtype="bf16", **kw)


def followed_run(mfs, s, w, frames, slots, ctx, orc, tally, label):
    """GPU steps of every slot in `slots`; the oracle follows the GPU's chosen tokens
    (a legal flip at a near tie does not end the comparison).  Outputs bit for bit."""
    for p in range(frames.shape[0]):
        text, codes = mfs.mfs_step(ctx, list(slots), frames[p])
        dbg = mfs.mfs_read_debug(ctx)
        fol = H.follow_tokens(text, codes, dbg["code_argmax"])
        ref = orc.step(list(slots), frames[p], want_logits=True, follow=fol)
        np.testing.assert_array_equal(text, ref["text"])
        np.testing.assert_array_equal(codes, ref["codes"])
        tally.step(dbg, list(range(len(slots))), ref, f"{label} frame {p}")


@pytest.mark.parametrize("n", [5, 8, 13, 32])
def test_mma_batch_mixed_positions(mfs, n):
    """n slots at different positions (prompts of up to 40 frames, W = 24 so some wrap),
    free-running agent streams, followed by the oracle for 10 frames."""
    s = tiny_bf16(window=24, max_slots=n)
    w = synth.make_weights(s, 40 + n, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    lens = synth.prefill_lengths(40 + n, n, 0, 40)
    for slot in range(n):
        if lens[slot]:
            pr = synth.forced_frames(s, 100 + slot, synth.STREAM_PROMPT, int(lens[slot]), 1)[:, 0]
            mfs.mfs_prefill(ctx, [slot], pr[None])
            orc.prefill(slot, pr)
    order = list(np.random.default_rng(n).permutation(n))
    u = synth.user_frames(s, 40 + n, 10, n)
    tally = H.Tally(f"tensor-core pass, tiny bf16, B={n}")
    followed_run(mfs, s, w, u, order, ctx, orc, tally, f"B={n}")
    print(tally.report())
    assert tally.frames == 10 * n


def test_mma_batched_prompt_then_decode(mfs):
    """Eight slots prefill a 20-frame prompt in one call (the tensor-core pass per
    frame), then decode; the oracle runs its own prompt path."""
    s = tiny_bf16(window=16, max_slots=8)
    w = synth.make_weights(s, 50, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    pr = synth.forced_frames(s, 50, synth.STREAM_PROMPT, 20, 8)  # [T, B, 17]
    mfs.mfs_prefill(ctx, list(range(8)), pr.transpose(1, 0, 2))
    for slot in range(8):
        orc.prefill(slot, pr[:, slot])
    u = synth.user_frames(s, 51, 6, 8)
    tally = H.Tally("tensor-core prompt path, tiny bf16, B=8")
    followed_run(mfs, s, w, u, list(range(8)), ctx, orc, tally, "prompt B=8")
    print(tally.report())


@pytest.mark.parametrize("n,T", [(1, 40), (3, 21), (16, 5)])
def test_mma_prompt_chunks(mfs, n, T):
    """Prompt chunks of up to 32 rows through the tensor-core pass: 1 slot takes 32 frames
    per launch, 3 slots 10, 16 slots 2 (the last frames of a short prompt run one per
    launch).  Against the oracle's prompt path, then 6 decode frames followed."""
    s = tiny_bf16(window=48, max_slots=n)
    w = synth.make_weights(s, 70 + n, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    pr = synth.forced_frames(s, 70 + n, synth.STREAM_PROMPT, T, n)  # [T, n, 17]
    mfs.mfs_prefill(ctx, list(range(n)), pr.transpose(1, 0, 2))
    for slot in range(n):
        orc.prefill(slot, pr[:, slot])
        assert mfs.mfs_position(ctx, slot) == T
    u = synth.user_frames(s, 71 + n, 6, n)
    tally = H.Tally(f"tensor-core prompt chunks, {n} slots x {T} frames")
    followed_run(mfs, s, w, u, list(range(n)), ctx, orc, tally, f"prompt {n}x{T}")
    print(tally.report())


def test_mma_slot_isolation_bit_exact(mfs):
    """A slot's outputs and logits are bit-identical whatever the other slots of the
    batch hold (same batch size, other slots with other histories and tokens)."""
    s = tiny_bf16(window=16, max_slots=16)
    w = synth.make_weights(s, 52, gain_std=0.1)
    a, b = H.gpu_context(s, w), H.gpu_context(s, w)
    pa = synth.forced_frames(s, 52, synth.STREAM_PROMPT, 9, 8)
    pb = synth.forced_frames(s, 53, synth.STREAM_PROMPT, 9, 8)
    pb[:, 3] = pa[:, 3]  # slot 3 is the same in both contexts
    mfs.mfs_prefill(a, list(range(8)), pa.transpose(1, 0, 2))
    mfs.mfs_prefill(b, list(range(8)), pb.transpose(1, 0, 2))
    ua = synth.user_frames(s, 54, 5, 8)
    ub = synth.user_frames(s, 55, 5, 8)
    ub[:, 3] = ua[:, 3]
    for p in range(5):
        ta, ca = mfs.mfs_step(a, list(range(8)), ua[p])
        da = mfs.mfs_read_debug(a)
        tb, cb = mfs.mfs_step(b, list(range(8)), ub[p])
        db = mfs.mfs_read_debug(b)
        assert ta[3] == tb[3] and np.array_equal(ca[3], cb[3])
        assert np.array_equal(da["text_logits"][3], db["text_logits"][3])
        assert np.array_equal(da["dep_logits"][3], db["dep_logits"][3])
        assert not np.array_equal(da["text_logits"][2], db["text_logits"][2])


def test_mma_persistent_and_per_phase_launches_bit_identical(mfs):
    s = tiny_bf16(window=16, max_slots=6)
    w = synth.make_weights(s, 56, gain_std=0.1)
    u = synth.user_frames(s, 56, 8, 6)
    a, b = H.gpu_context(s, w), H.gpu_context(s, w)
    mfs.mfs_set_mode(b, 1)
    for p in range(8):
        ta, ca = mfs.mfs_step(a, list(range(6)), u[p])
        da = mfs.mfs_read_debug(a)
        tb, cb = mfs.mfs_step(b, list(range(6)), u[p])
        db = mfs.mfs_read_debug(b)
        assert np.array_equal(ta, tb) and np.array_equal(ca, cb)
        assert np.array_equal(da["text_logits"], db["text_logits"])
        assert np.array_equal(da["dep_logits"], db["dep_logits"])


def test_mma_sampling_and_skipped_substeps(mfs):
    """Sampling heads through the tensor-core pass (draws equal the oracle sampler on the
    GPU's own logits), and skipped settled substeps leave every output unchanged."""
    from tests.test_gpu_tiny import _near_cdf_boundary
    s = tiny_bf16(window=16, max_slots=9)
    w = synth.make_weights(s, 57, gain_std=0.1)
    ctx = H.gpu_context(s, w)
    for slot in range(9):
        mfs.mfs_set_sampling(ctx, slot, 0.7, 25, 0.8, 250)
    u = synth.user_frames(s, 57, 4, 9)
    unif = ((synth.uniform_int(57, 99, 4 * 9 * 17, 0, 1 << 24).reshape(4, 9, 17)) + 0.5) / float(1 << 24)
    checked = 0
    for p in range(4):
        text, codes = mfs.mfs_step_sampled(ctx, list(range(9)), u[p], unif[p])
        dbg = mfs.mfs_read_debug(ctx)
        for i in range(9):
            for k in range(9):
                if p == 0 and s.delays[k] == 1:
                    continue
                lg = dbg["text_logits"][i] if k == 0 else dbg["dep_logits"][i][k - 1]
                temp, topk = (0.7, 25) if k == 0 else (0.8, 250)
                got = text[i] if k == 0 else codes[i][k - 1]
                want = oracle.sample_topk(lg, temp, topk, unif[p][i][k])
                if got != want:
                    assert _near_cdf_boundary(lg, temp, topk, unif[p][i][k]), (p, i, k, got, want)
                checked += 1
    assert checked == 4 * 9 * 9 - 9 * 7
    # skipped settled substeps: the user streams are supplied, so substeps 8..15 only
    # reproduce supplied outputs
    a, b = H.gpu_context(s, w), H.gpu_context(s, w)
    mfs.mfs_set_skip_settled(b, True)
    for p in range(4):
        ta, ca = mfs.mfs_step(a, list(range(9)), u[p])
        tb, cb = mfs.mfs_step(b, list(range(9)), u[p])
        assert np.array_equal(ta, tb) and np.array_equal(ca, cb)


@pytest.mark.parametrize("n", [2, 5])
def test_tag_period_wrap_is_invisible(mfs, n):
    """Phases hand values over as words tagged (sequence << 10) | phase, which repeat every
    2^22 steps; the library resets its tagged buffers before the step that starts a period.
    Steps across that point (sequence numbers 2^22 - 3 .. 2^22 + 4, on the CUDA-core pass
    for 2 slots and the tensor-core pass for 5) give outputs and logits bit-identical to the
    same steps at small sequence numbers."""
    s = tiny_bf16(window=24, max_slots=n)
    w = synth.make_weights(s, 77, gain_std=0.1)
    pr = synth.forced_frames(s, 78, synth.STREAM_PROMPT, 6, n).transpose(1, 0, 2)
    u = synth.user_frames(s, 79, 7, n)
    runs = []
    for start in (None, (1 << 22) - 4):
        ctx = H.gpu_context(s, w)
        mfs.mfs_prefill(ctx, list(range(n)), pr)
        if start is not None:
            mfs.mfs_debug_set_seq(ctx, start)
        res = []
        for p in range(u.shape[0]):
            text, codes = mfs.mfs_step(ctx, list(range(n)), u[p])
            dbg = mfs.mfs_read_debug(ctx)
            res.append([text.copy(), codes.copy(), dbg["text_logits"], dbg["dep_logits"]])
        runs.append(res)
    for a, b in zip(*runs):
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("n", [2, 6])
def test_ring_mask_oldest(mfs, n):
    """The masked-oldest-slot window (W - 1 keys once the ring of capacity W is full), on the
    CUDA-core pass (2 slots) and the tensor-core pass (6 slots), W = 8, 20 steps from
    position 0 (two wraps): the oracle with the same flag follows the GPU, and the GPU
    matches, bit for bit, a context with a plain window of 7."""
    s = tiny_bf16(window=8, max_slots=n)
    w = synth.make_weights(s, 90 + n, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w, mask_oldest=True)
    mfs.mfs_set_ring_mask_oldest(ctx, True)
    ctx7 = H.gpu_context(s.replace(window=7), w)
    u = synth.user_frames(s, 91 + n, 20, n)
    tally = H.Tally(f"masked oldest ring slot, W=8, B={n}")
    slots = list(range(n))
    for p in range(u.shape[0]):
        text, codes = mfs.mfs_step(ctx, slots, u[p])
        dbg = mfs.mfs_read_debug(ctx)
        text7, codes7 = mfs.mfs_step(ctx7, slots, u[p])
        dbg7 = mfs.mfs_read_debug(ctx7)
        np.testing.assert_array_equal(text, text7)
        np.testing.assert_array_equal(codes, codes7)
        np.testing.assert_array_equal(dbg["text_logits"], dbg7["text_logits"])
        np.testing.assert_array_equal(dbg["dep_logits"], dbg7["dep_logits"])
        fol = H.follow_tokens(text, codes, dbg["code_argmax"])
        ref = orc.step(slots, u[p], want_logits=True, follow=fol)
        np.testing.assert_array_equal(text, ref["text"])
        np.testing.assert_array_equal(codes, ref["codes"])
        tally.step(dbg, slots, ref, f"frame {p}")
    print(tally.report())


def test_ring_mask_oldest_rejects_bad_flag(mfs):
    s = tiny_bf16(window=8, max_slots=2)
    ctx = H.gpu_context(s, synth.make_weights(s, 5, gain_std=0.1))
    with pytest.raises(mfs.MfsError):
        mfs._check(ctx, mfs._lib.mfs_set_ring_mask_oldest(ctx.handle, 2))
