"""Pins of the CPU oracle to things other than itself (closed forms, invariants,
brute force, library routines, the pages' printed constants).  CPU only."""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from tests import _seqref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_shape(**kw):
    base = synth.TINY.replace(window=8, max_slots=3)
    return base.replace(**kw)


@pytest.fixture(scope="module")
def tiny_w8():
    s = small_shape()
    w = synth.make_weights(s, seed=3, gain_std=0.1)
    return s, w


# ----------------------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    n, c, eps = 64, -0.37, 1e-8
    g = synth.normal_f32(5, 0, n, 1.0, 0.2)
    out = oracle.rmsnorm(np.full(n, c), g, eps)
    expect = c / np.sqrt(c * c + eps) * g.astype(np.float64)
    np.testing.assert_allclose(out, expect, rtol=1e-14, atol=0)
    # sign of the constant times the gain, to within eps
    np.testing.assert_allclose(out, -g.astype(np.float64), rtol=1e-6)


def test_rmsnorm_scale_invariance_and_library():
    x = synth.normal_f32(6, 0, 300).astype(np.float64)
    g = synth.normal_f32(6, 1, 300, 1.0, 0.3)
    a = oracle.rmsnorm(x, g, 1e-8)
    b = oracle.rmsnorm(17.0 * x, g, 1e-8)
    np.testing.assert_allclose(a, b, rtol=1e-8)   # differs by ~eps/2 relative
    ref = F.rms_norm(torch.from_numpy(x), (300,), torch.from_numpy(g.astype(np.float64)), 1e-8)
    np.testing.assert_allclose(a, ref.numpy(), rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------- RoPE

@pytest.mark.parametrize("hd", [64, 128])
def test_rope_complex_closed_form(hd):
    v = synth.normal_f32(7, hd, hd).astype(np.float64)
    for p in (0, 1, 5, 257, 2999, 8191):
        out = oracle.rope(v, p)
        z = v[0::2] + 1j * v[1::2]
        i = np.arange(hd // 2)
        z = z * np.exp(1j * p * 10000.0 ** (-2.0 * i / hd))
        np.testing.assert_allclose(out[0::2], z.real, rtol=0, atol=1e-12)
        np.testing.assert_allclose(out[1::2], z.imag, rtol=0, atol=1e-12)


def test_rope_invariants():
    hd = 128
    q = synth.normal_f32(8, 0, hd).astype(np.float64)
    k = synth.normal_f32(8, 1, hd).astype(np.float64)
    np.testing.assert_array_equal(oracle.rope(q, 0), q)                      # R(0) = I
    for p in (3, 100, 4000):
        assert abs(np.linalg.norm(oracle.rope(q, p)) - np.linalg.norm(q)) < 1e-12  # rotation
    # <R(p) q, R(p') k> depends only on p - p'
    a = oracle.rope(q, 1000) @ oracle.rope(k, 990)
    b = oracle.rope(q, 10) @ oracle.rope(k, 0)
    c = oracle.rope(q, 7010) @ oracle.rope(k, 7000)
    assert abs(a - b) < 1e-9 and abs(c - b) < 1e-9


# ----------------------------------------------------------------------------- attention

def test_attention_single_key_returns_value():
    q = synth.normal_f32(9, 0, 64).astype(np.float64)
    K = synth.normal_f32(9, 1, 64).astype(np.float64).reshape(1, 64)
    V = synth.normal_f32(9, 2, 64).astype(np.float64).reshape(1, 64)
    np.testing.assert_allclose(oracle.attention(q, K, V), V[0], rtol=0, atol=1e-15)


def test_attention_equal_keys_average_values():
    q = synth.normal_f32(10, 0, 64).astype(np.float64)
    K = np.tile(synth.normal_f32(10, 1, 64).astype(np.float64), (7, 1))
    V = synth.normal_f32(10, 2, 7 * 64).astype(np.float64).reshape(7, 64)
    np.testing.assert_allclose(oracle.attention(q, K, V), V.mean(0), rtol=1e-13, atol=1e-15)


def test_attention_matches_library_sdpa():
    for n in (1, 2, 16, 300):
        q = synth.normal_f32(11, n, 128, 0.0, 2.0).astype(np.float64)
        K = synth.normal_f32(12, n, n * 128, 0.0, 2.0).astype(np.float64).reshape(n, 128)
        V = synth.normal_f32(13, n, n * 128).astype(np.float64).reshape(n, 128)
        ref = F.scaled_dot_product_attention(torch.from_numpy(q)[None, None, None],
                                             torch.from_numpy(K)[None, None],
                                             torch.from_numpy(V)[None, None])[0, 0, 0].numpy()
        np.testing.assert_allclose(oracle.attention(q, K, V), ref, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------- stream layout

def test_golden_stream_layout_matches_workload_constants():
    g = json.load(open(os.path.join(GOLDEN, "stream_layout.json")))
    assert tuple(g["delays"]) == synth.DELAYS
    assert g["n_streams"] == synth.N_STREAMS == 1 + synth.FULL.n_q
    assert [synth.DELAYS[k] for k in g["semantic_rows"]] == [0, 0]
    assert g["frame_ms"] * (1 + g["acoustic_delay_frames"]) == g["theoretical_latency_ms"]


def test_golden_bitrate_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "mimi_bitrate.json")))
    bits = g["frame_rate_hz"] * g["codebooks_per_side"] * np.log2(g["card"])
    assert bits == pytest.approx(g["bitrate_kbps"] * 1000)
    assert g["sample_rate_hz"] / g["frame_rate_hz"] == g["samples_per_frame"]
    assert synth.FULL.card == g["card"] and synth.FULL.n_q == 2 * g["codebooks_per_side"]


# ----------------------------------------------------------------------------- delay schedule

def expected_rows(s, chosen):
    """brute force: row read by stream k at step p is chosen[p-1-delay[k]][k] or INIT."""
    T = chosen.shape[0]
    X = np.empty((T, 17), np.int64)
    for p in range(T):
        for k in range(17):
            f = p - 1 - s.delays[k]
            X[p, k] = chosen[f, k] if f >= 0 else (s.text_vocab if k == 0 else s.card)
    return X


def test_delay_schedule_forced_bit_exact(tiny_w8):
    s, w = tiny_w8
    T = 12
    z = synth.forced_frames(s, 21, synth.STREAM_FORCED, T, 1)[:, 0]
    o = oracle.Oracle(s, w)
    rows, outs = [], []
    for p in range(T):
        r = o.step([0], z[p:p + 1], want_tokens=True)
        rows.append(r["x_tokens"][0])
        outs.append(r)
    np.testing.assert_array_equal(np.array(rows), expected_rows(s, z))
    # every (stream, frame) comes out exactly once, at step frame + delay
    for p, r in enumerate(outs):
        assert r["text"][0] == z[p, 0]
        for k in range(1, 17):
            f = p - s.delays[k]
            assert r["codes"][0, k - 1] == (z[f, k] if f >= 0 else -1)


def test_delay_schedule_free_running(tiny_w8):
    """Generated rows: the input column at step p is the column chosen at earlier steps."""
    s, w = tiny_w8
    T = 10
    inp = synth.user_frames(s, 22, T, 1)[:, 0]
    o = oracle.Oracle(s, w)
    res = [o.step([0], inp[p:p + 1], want_tokens=True) for p in range(T)]
    chosen = np.full((T, 17), -7, np.int64)
    for p, r in enumerate(res):
        chosen[p, 0] = r["text"][0]
        for k in range(1, 17):
            f = p - s.delays[k]
            if f >= 0:
                chosen[f, k] = r["codes"][0, k - 1]
    # user rows come out as supplied
    for p in range(T):
        for k in range(9, 17):
            f = p - s.delays[k]
            if f >= 0:
                assert chosen[f, k] == inp[f, k]
    X = np.array([r["x_tokens"][0] for r in res])
    exp = expected_rows(s, chosen)
    np.testing.assert_array_equal(X, exp)
    assert (X >= 0).all()


def _chosen_as_follow(s, r):
    """Follow-mode input from one step's results: the chosen token of every stream,
    and for a frame before 0 (output -1) the raw argmax the substep chain used."""
    f = np.empty((len(r["text"]), 17), np.int32)
    f[:, 0] = r["text"]
    f[:, 1:] = np.where(r["codes"] >= 0, r["codes"], r["code_argmax"])
    return f


def test_follow_with_own_choices_changes_nothing(tiny_w8):
    """Follow mode fed the oracle's own chosen tokens reproduces every output and
    logit bit for bit (it only replaces a choice by the same choice)."""
    s, w = tiny_w8
    T = 8
    inp = synth.user_frames(s, 23, T, 2)
    a, b = oracle.Oracle(s, w), oracle.Oracle(s, w)
    for p in range(T):
        ra = a.step([0, 1], inp[p], want_logits=True, want_tokens=True)
        rb = b.step([0, 1], inp[p], want_logits=True, want_tokens=True, follow=_chosen_as_follow(s, ra))
        for key in ra:
            np.testing.assert_array_equal(ra[key], rb[key])


def test_follow_equals_forcing_the_same_frame(tiny_w8):
    """Adopting token v for a generated stream k is the same as the caller supplying v
    for that stream's frame: at the same step for a stream without delay, at the step
    before for a delayed one.  Outputs, logits and embedding rows agree bit for bit."""
    s, w = tiny_w8
    T = 9
    inp = synth.user_frames(s, 24, T, 1)[:, 0]
    toks = synth.uniform_int(24, 90, T * 17, 0, 1000).reshape(T, 17)
    fol = np.full((T, 17), -1, np.int32)
    forced = inp.copy()
    for p in range(1, T - 1):
        for k in (0, 1, 2, 5, 8):  # text, an undelayed and three delayed agent streams (generated)
            v = int(toks[p, k]) % (s.text_vocab if k == 0 else s.card)
            forced[p, k] = v                       # the caller supplies frame p
            fol[p + s.delays[k], k] = v            # follow mode adopts it when frame p is generated
    a, b, plain = oracle.Oracle(s, w), oracle.Oracle(s, w), oracle.Oracle(s, w)
    changed = 0
    for p in range(T):
        ra = a.step([0], inp[p:p + 1], want_logits=True, want_tokens=True, follow=fol[p:p + 1])
        rb = b.step([0], forced[p:p + 1], want_logits=True, want_tokens=True)
        rp = plain.step([0], inp[p:p + 1], want_logits=True)
        for key in ("text", "codes", "text_logits", "dep_logits", "x_tokens", "text_argmax", "code_argmax"):
            np.testing.assert_array_equal(ra[key], rb[key], err_msg=f"step {p} {key}")
        changed += int(not np.array_equal(ra["dep_logits"], rp["dep_logits"]))
    assert changed >= T - 2  # the adopted tokens really changed the run (not a vacuous pin)


def test_follow_rejects_out_of_range_tokens(tiny_w8):
    s, w = tiny_w8
    o = oracle.Oracle(s, w)
    fol = np.full((1, 17), -1, np.int32)
    fol[0, 4] = s.card
    with pytest.raises(ValueError):
        o.step([0], synth.user_frames(s, 25, 1, 1)[0], follow=fol)
    assert o.position(0) == 0


# ----------------------------------------------------------------------------- model

@pytest.mark.parametrize("T", [20])
def test_oracle_matches_whole_sequence_library_forward(tiny_w8, T):
    """Step-by-step oracle (ring of W=8) == whole-sequence masked forward, in fp64."""
    s, w = tiny_w8
    z = synth.forced_frames(s, 31, synth.STREAM_FORCED, T, 1)[:, 0]
    o = oracle.Oracle(s, w)
    tl, dl = [], []
    for p in range(T):
        r = o.step([0], z[p:p + 1], want_logits=True)
        tl.append(r["text_logits"][0])
        dl.append(r["dep_logits"][0])
    ref_t, ref_d = _seqref.forward(s, w, z)
    tl, dl = np.array(tl), np.array(dl)
    np.testing.assert_allclose(tl, ref_t, rtol=0, atol=1e-10 * np.abs(ref_t).max())
    np.testing.assert_allclose(dl, ref_d, rtol=0, atol=1e-10 * np.abs(ref_d).max())


@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
def test_oracle_matches_library_forward_bf16_weights(kv_dtype):
    """bf16 weights; with a bf16 cache the library forward rounds rotated keys and values
    with torch's own bf16 conversion, which pins the oracle's rounding and where it applies."""
    s = small_shape(weight_dtype="bf16", kv_dtype=kv_dtype, window=5)
    w = synth.make_weights(s, seed=4, gain_std=0.1)
    T = 9
    z = synth.forced_frames(s, 32, synth.STREAM_FORCED, T, 1)[:, 0]
    o = oracle.Oracle(s, w)
    res = [o.step([0], z[p:p + 1], want_logits=True) for p in range(T)]
    ref_t, ref_d = _seqref.forward(s, w, z)
    tl = np.array([r["text_logits"][0] for r in res])
    dl = np.array([r["dep_logits"][0] for r in res])
    np.testing.assert_allclose(tl, ref_t, rtol=0, atol=1e-10 * np.abs(ref_t).max())
    np.testing.assert_allclose(dl, ref_d, rtol=0, atol=1e-10 * np.abs(ref_d).max())


def test_ring_equals_brute_force_history(tiny_w8):
    """Ring storage at position mod W == every position kept and masked to the last W."""
    s, w = tiny_w8
    T = 40
    inp = synth.user_frames(s, 23, T, 1)[:, 0]
    a, b = oracle.Oracle(s, w), oracle.Oracle(s, w, brute_force=True)
    for p in range(T):
        ra = a.step([0], inp[p:p + 1], want_logits=True)
        rb = b.step([0], inp[p:p + 1], want_logits=True)
        for key in ra:
            np.testing.assert_array_equal(ra[key], rb[key])


def test_masked_oldest_slot_is_a_window_of_w_minus_1(tiny_w8):
    """The masked-oldest-slot variant (a ring of capacity W whose oldest slot is masked once
    full) attends exactly like the plain window of W - 1: same outputs and logits at every
    step, including the steps before the ring fills and after it wraps; with the flag off
    it differs once the ring holds W positions."""
    s, w = tiny_w8
    T = 3 * s.window + 5
    inp = synth.user_frames(s, 24, T, 1)[:, 0]
    a = oracle.Oracle(s, w, mask_oldest=True)
    b = oracle.Oracle(s.replace(window=s.window - 1), w)
    c = oracle.Oracle(s, w)
    differs = False
    for p in range(T):
        ra = a.step([0], inp[p:p + 1], want_logits=True)
        rb = b.step([0], inp[p:p + 1], want_logits=True)
        rc = c.step([0], inp[p:p + 1], want_logits=True)
        for key in ra:
            np.testing.assert_array_equal(ra[key], rb[key])
        if p < s.window - 1:
            np.testing.assert_array_equal(ra["text_logits"], rc["text_logits"])
        differs |= not np.array_equal(ra["text_logits"], rc["text_logits"])
    assert differs


def test_window_actually_limits_context(tiny_w8):
    """Tokens older than the window (through every layer) cannot change the output."""
    s, w = tiny_w8
    reach = 2 + s.n_layers * (s.window - 1)   # frame 0 enters positions 1..2; each layer
    T = reach + 4                             # widens the receptive field by W - 1
    z1 = synth.forced_frames(s, 41, synth.STREAM_FORCED, T, 1)[:, 0]
    z2 = z1.copy()
    z2[0] = synth.forced_frames(s, 42, synth.STREAM_FORCED, 1, 1)[0, 0]   # change frame 0 only
    outs = []
    for z in (z1, z2):
        o = oracle.Oracle(s, w)
        outs.append([o.step([0], z[p:p + 1], want_logits=True)["text_logits"][0] for p in range(T)])
    assert not np.array_equal(outs[0][3], outs[1][3])
    assert not np.array_equal(outs[0][reach], outs[1][reach])
    for p in range(reach + 1, T):
        np.testing.assert_array_equal(outs[0][p], outs[1][p])


def test_depformer_causality(tiny_w8):
    """Changing the supplied code of stream j changes substeps >= j only."""
    s, w = tiny_w8
    z = synth.forced_frames(s, 43, synth.STREAM_FORCED, 3, 1)[:, 0]
    base = oracle.Oracle(s, w)
    for p in range(2):
        base.step([0], z[p:p + 1])
    ref = base.step([0], z[2:3], want_logits=True)["dep_logits"][0]
    j = 9                                 # user semantic stream, delay 0: read by substep 9
    z2 = z.copy()
    z2[2, j] = (z2[2, j] + 1) % s.card
    o = oracle.Oracle(s, w)
    for p in range(2):
        o.step([0], z2[p:p + 1])
    alt = o.step([0], z2[2:3], want_logits=True)["dep_logits"][0]
    np.testing.assert_array_equal(alt[:j], ref[:j])
    assert not np.array_equal(alt[j], ref[j])


def test_argmax_lowest_index_on_ties():
    s = small_shape()
    w = synth.make_weights(s, seed=5)
    head = np.zeros_like(w["text_head"])
    r = synth.normal_f32(44, 0, s.d, 0.0, 0.02)
    head[5], head[9], head[2] = r, r, -r
    w["text_head"] = head
    o = oracle.Oracle(s, w)
    res = o.step([0], synth.user_frames(s, 45, 1, 1)[0], want_logits=True)
    lg = res["text_logits"][0]
    a = lg[5]
    assert lg[9] == a and lg[2] == -a
    assert res["text_argmax"][0] == (5 if a > 0 else 2 if a < 0 else 0)
    w["text_head"] = np.zeros_like(head)              # all logits 0 -> index 0
    o = oracle.Oracle(s, w)
    assert o.step([0], synth.user_frames(s, 45, 1, 1)[0])["text_argmax"][0] == 0


def test_slot_isolation_and_reset(tiny_w8):
    s, w = tiny_w8
    T = 6
    a = synth.user_frames(s, 46, T, 3)
    solo, multi = oracle.Oracle(s, w), oracle.Oracle(s, w)
    for p in range(T):
        r1 = solo.step([1], a[p, 1:2], want_logits=True)
        r3 = multi.step([2, 1, 0], a[p, [2, 1, 0]], want_logits=True)
        for key in r1:
            np.testing.assert_array_equal(r1[key][0], r3[key][1])
    # a reset slot behaves as a fresh one
    multi.reset_slot(1)
    fresh = oracle.Oracle(s, w)
    for p in range(3):
        ra = multi.step([1], a[p, 1:2], want_logits=True)
        rb = fresh.step([1], a[p, 1:2], want_logits=True)
        for key in ra:
            np.testing.assert_array_equal(ra[key], rb[key])


def test_prefill_equals_forced_steps(tiny_w8):
    s, w = tiny_w8
    T = 11
    z = synth.forced_frames(s, 47, synth.STREAM_FORCED, T, 1)[:, 0]
    nxt = synth.user_frames(s, 48, 3, 1)[:, 0]
    a, b = oracle.Oracle(s, w), oracle.Oracle(s, w)
    a.prefill(0, z)
    for p in range(T):
        b.step([0], z[p:p + 1])
    assert a.position(0) == b.position(0) == T
    for p in range(3):
        ra = a.step([0], nxt[p:p + 1], want_logits=True)
        rb = b.step([0], nxt[p:p + 1], want_logits=True)
        for key in ra:
            np.testing.assert_array_equal(ra[key], rb[key])


def test_oracle_rejects_bad_input(tiny_w8):
    s, w = tiny_w8
    o = oracle.Oracle(s, w)
    bad = synth.user_frames(s, 49, 1, 1)[0]
    bad[0, 3] = s.card
    with pytest.raises(ValueError):
        o.step([0], bad)
    with pytest.raises(ValueError):
        o.step([3], synth.user_frames(s, 49, 1, 1)[0])
    assert o.position(0) == 0


def test_slot_state_import_continues_exactly():
    """A bf16-cache slot exported after some steps and imported into another slot of a
    fresh oracle continues bit for bit like the original (position, history and every
    ring row carried over; the ring wraps at W = 5 within the run)."""
    s = small_shape(weight_dtype="bf16", kv_dtype="bf16", window=5)
    w = synth.make_weights(s, seed=8, gain_std=0.1)
    z = synth.user_frames(s, 41, 14, 1)
    a, b = oracle.Oracle(s, w), oracle.Oracle(s, w)
    for p in range(9):
        a.step([0], z[p])
    b.import_slot(2, a.export_slot(0))
    assert b.position(2) == a.position(0) == 9
    for p in range(9, 14):
        ra = a.step([0], z[p], want_logits=True)
        rb = b.step([2], z[p], want_logits=True)
        for key in ra:
            np.testing.assert_array_equal(ra[key], rb[key], err_msg=key)
    bad = a.export_slot(0)
    bad[4:8] = np.frombuffer(np.int32(s.max_pos + 1).tobytes(), np.uint8)
    with pytest.raises(ValueError):
        b.import_slot(1, bad)


# ---------------------------------------------------------------- sampling heads

def _topk_probs(lg, temp, k):
    """Closed form: the k largest logits (ties to the lower index), softmax of logit / temp."""
    order = sorted(range(len(lg)), key=lambda i: (-lg[i], i))[:k]
    z = np.array([lg[i] for i in order]) / temp
    p = np.exp(z - z.max())
    return dict(zip(order, p / p.sum()))


def test_sampler_greedy_limits():
    rng = np.random.default_rng(1)
    lg = rng.standard_normal(300)
    for u in (0.0, 0.3, 0.999):
        assert oracle.sample_topk(lg, 0.7, 1, u) == int(np.argmax(lg))
        assert oracle.sample_topk(lg, 0.0, 25, u) == int(np.argmax(lg))
        assert oracle.sample_topk(lg, 1e-9, 25, u) == int(np.argmax(lg))


def test_sampler_equal_logits_ties_to_lower_indices():
    lg = np.zeros(50)
    for m in range(10):
        assert oracle.sample_topk(lg, 0.8, 10, (m + 0.5) / 10) == m


def test_sampler_matches_the_closed_form_distribution():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal(40) * 2.0
    lg[7] = lg[11]  # a tie inside the candidate set
    for temp, k in ((0.8, 7), (0.7, 25), (1.3, 40)):
        exact = _topk_probs(lg, temp, k)
        grid = 20000
        counts = {}
        for g in range(grid):
            t = oracle.sample_topk(lg, temp, k, (g + 0.5) / grid)
            counts[t] = counts.get(t, 0) + 1
        assert set(counts) <= set(exact)
        for i, p in exact.items():
            assert abs(counts.get(i, 0) / grid - p) <= 2.0 / grid, (temp, k, i)


def test_sampler_temperature_scales_logits():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal(200)
    for u in np.linspace(0.01, 0.99, 60):
        assert oracle.sample_topk(lg, 2.0, 30, u) == oracle.sample_topk(lg / 2.0, 1.0, 30, u)


def test_sampled_step_draws_from_its_own_logits(tiny_w8):
    """A sampled oracle step picks the text token and each generated code with the sampler
    applied to that step's logits and the row's uniforms; k = 1 is the greedy step."""
    s, w = tiny_w8
    u = synth.user_frames(s, 51, 6, 1)
    unif = (synth.uniform_int(51, 77, 6 * 17, 0, 1 << 24).reshape(6, 1, 17) + 0.5) / float(1 << 24)
    a, b = oracle.Oracle(s, w), oracle.Oracle(s, w)
    a.set_sampling(0, 0.7, 25, 0.8, 250)
    b.set_sampling(0, 0.7, 1, 0.8, 1)
    g = oracle.Oracle(s, w)
    for p in range(6):
        r = a.step([0], u[p], want_logits=True, uniforms=unif[p])
        assert r["text"][0] == oracle.sample_topk(r["text_logits"][0], 0.7, 25, unif[p][0][0])
        # substep 0 yields stream 1 (delay 0): drawn from its logits with stream 1's uniform
        assert r["codes"][0][0] == oracle.sample_topk(r["dep_logits"][0][0], 0.8, 250, unif[p][0][1])
        rb = b.step([0], u[p], want_logits=True, uniforms=unif[p])
        rg = g.step([0], u[p], want_logits=True)
        for key in ("text", "codes", "text_logits", "dep_logits"):
            np.testing.assert_array_equal(rb[key], rg[key])


# ---------------------------------------------------------------- Mimi split RVQ encode

def test_rvq_matches_library_nearest_neighbours():
    """Each stage is the library's nearest neighbour (scipy cdist + argmin) on the residual
    left by the stage before; the semantic codebook sees its own latent."""
    cdist = pytest.importorskip("scipy.spatial.distance").cdist
    rng = np.random.default_rng(5)
    T, D, Cb = 12, 16, 64
    zs, za = rng.standard_normal((T, D)).astype(np.float32), rng.standard_normal((T, D)).astype(np.float32)
    cb = rng.standard_normal((8, Cb, D)).astype(np.float32)
    codes, gap = oracle.rvq_encode(zs, za, cb)
    assert (gap >= 0).all()
    np.testing.assert_array_equal(codes[:, 0], np.argmin(cdist(zs.astype(np.float64), cb[0].astype(np.float64), "sqeuclidean"), axis=1))
    r = za.astype(np.float64)
    for q in range(1, 8):
        want = np.argmin(cdist(r, cb[q].astype(np.float64), "sqeuclidean"), axis=1)
        np.testing.assert_array_equal(codes[:, q], want)
        r = r - cb[q][want].astype(np.float64)


def test_rvq_exact_codewords_and_ties():
    """A latent equal to a codeword picks it; a zero residual then picks the codeword of
    least norm, the lower index on a tie."""
    D, Cb = 8, 16
    cb = np.zeros((8, Cb, D), np.float32)
    rng = np.random.default_rng(6)
    cb[:, 1:] = rng.standard_normal((8, Cb - 1, D)).astype(np.float32)
    cb[:, 0] = 0.0
    cb[:, 5] = 0.0  # same (zero) codeword at 0 and 5: the tie goes to 0
    zs = cb[0, 9][None].copy()
    za = cb[1, 7][None].copy()
    codes, _ = oracle.rvq_encode(zs, za, cb)
    assert codes[0, 0] == 9 and codes[0, 1] == 7
    assert (codes[0, 2:] == 0).all()


def test_synthetic_slot_state_round_trips_through_the_oracle():
    """The synthetic state generator writes the documented slot-state layout: the oracle
    reads it and writes back the same bytes (position, history, every ring row)."""
    s = small_shape(weight_dtype="bf16", kv_dtype="bf16", window=6)
    w = synth.make_weights(s, 9)
    o = oracle.Oracle(s, w)
    for pos in (0, 4, 23):
        st = synth.slot_state(s, 9, pos, pos)
        o.import_slot(1, st)
        assert o.position(1) == pos
        np.testing.assert_array_equal(o.export_slot(1), st)
