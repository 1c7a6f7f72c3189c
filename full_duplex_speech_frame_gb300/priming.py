"""Session priming: the persona and voice a session starts with, as supplied frames.

PersonaPlex conditions the assistant before the conversation in four phases run
through the ordinary lockstep step with every token supplied (mobius PR #368,
commit note on persona and voice priming: voice prompt, silence, persona text,
silence; vLLM-Omni PersonaPlex recipe, "Architecture": the voice clone forces the
agent audio rows from the reference audio's Mimi codes, the persona forces the
text row from ``<system> ... <system>`` tokens).  With every row supplied the
library's prompt path (``mfs_prefill``) runs the temporal stack only, which is
exactly what those frames change.

The token values themselves (the text pad token, the codes of silence, the user
rows' fill, the tokenizer and the Mimi encoder) belong to the trained model and
are the caller's: this module only lays them out.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

N_STREAMS = 17
AGENT = slice(1, 9)   # rows 1..8: agent audio codebooks
USER = slice(9, 17)   # rows 9..16: user audio codebooks


def priming_frames(voice_codes, persona_tokens: Sequence[int], *, text_pad: int, agent_silence: Sequence[int],
                   user_fill: Sequence[int], silence_after_voice: int, silence_after_persona: int) -> np.ndarray:
    """Frames [T, 17] (int32, every entry supplied) for the four priming phases, in order:

    1. voice: one frame per row of ``voice_codes`` [Tv, 8]; agent rows = that row, text = pad;
    2. ``silence_after_voice`` frames: agent rows = ``agent_silence``, text = pad;
    3. persona: one frame per token; text = the token, agent rows = ``agent_silence``;
    4. ``silence_after_persona`` frames as in 2.

    The user rows hold ``user_fill`` throughout.
    """
    voice = np.asarray(voice_codes, dtype=np.int64).reshape(-1, 8)
    persona = np.asarray(list(persona_tokens), dtype=np.int64).reshape(-1)
    sil = np.asarray(agent_silence, dtype=np.int64).reshape(8)
    fill = np.asarray(user_fill, dtype=np.int64).reshape(8)
    if silence_after_voice < 0 or silence_after_persona < 0:
        raise ValueError("silence lengths must be >= 0")
    T = voice.shape[0] + silence_after_voice + persona.size + silence_after_persona
    out = np.empty((T, N_STREAMS), np.int64)
    out[:, 0] = text_pad
    out[:, AGENT] = sil
    out[:, USER] = fill
    t = 0
    out[t:t + voice.shape[0], AGENT] = voice
    t += voice.shape[0] + silence_after_voice
    out[t:t + persona.size, 0] = persona
    if (out < 0).any():
        raise ValueError("priming tokens must be >= 0 (every entry is supplied)")
    return out.astype(np.int32)


def prime_slot(ctx, slot: int, frames: np.ndarray) -> None:
    """Start ``slot`` afresh and run the priming frames through the prompt path."""
    from full_duplex_speech_frame_gb300 import mfs
    mfs.mfs_reset_slot(ctx, slot)
    if len(frames):
        mfs.mfs_prefill(ctx, [slot], np.asarray(frames, np.int32)[None])
