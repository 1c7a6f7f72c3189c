"""Session priming frames (voice prompt, silence, persona text, silence) and their
effect on the oracle: priming through the prompt path equals stepping the same
supplied frames one by one."""
import numpy as np
import pytest

import oracle
import synth
from full_duplex_speech_frame_gb300.priming import priming_frames


def _frames(s):
    voice = synth.uniform_int(3, 301, 5 * 8, 0, s.card).reshape(5, 8)
    persona = synth.uniform_int(3, 302, 4, 0, s.text_vocab)
    return voice, persona, priming_frames(voice, persona, text_pad=3, agent_silence=[7] * 8, user_fill=[11] * 8,
                                          silence_after_voice=2, silence_after_persona=3)


def test_priming_layout_follows_the_four_phases():
    s = synth.TINY
    voice, persona, f = _frames(s)
    assert f.shape == (5 + 2 + 4 + 3, 17) and f.dtype == np.int32 and (f >= 0).all()
    np.testing.assert_array_equal(f[:5, 1:9], voice)           # voice: agent rows
    assert (f[:5, 0] == 3).all()                                # text pad while the voice plays
    assert (f[5:7, 1:9] == 7).all() and (f[5:7, 0] == 3).all()  # silence
    np.testing.assert_array_equal(f[7:11, 0], persona)          # persona on the text row
    assert (f[7:11, 1:9] == 7).all()
    assert (f[11:, 1:9] == 7).all() and (f[11:, 0] == 3).all()  # silence
    assert (f[:, 9:] == 11).all()                               # user rows: the fill throughout
    with pytest.raises(ValueError):
        priming_frames(voice, [-1], text_pad=3, agent_silence=[7] * 8, user_fill=[11] * 8,
                       silence_after_voice=0, silence_after_persona=0)


def test_priming_by_prompt_path_equals_stepping_the_frames():
    s = synth.TINY.replace(window=8, max_slots=2)
    w = synth.make_weights(s, 4, gain_std=0.1)
    _, _, f = _frames(s)
    a, b = oracle.Oracle(s, w), oracle.Oracle(s, w)
    a.prefill(0, f)
    for t in range(f.shape[0]):
        b.step([0], f[t:t + 1])
    u = synth.user_frames(s, 4, 3, 1)
    for p in range(3):
        ra = a.step([0], u[p], want_logits=True)
        rb = b.step([0], u[p], want_logits=True)
        np.testing.assert_allclose(ra["text_logits"], rb["text_logits"], rtol=0, atol=1e-9)
        np.testing.assert_array_equal(ra["codes"], rb["codes"])
