"""Key/value ring rows outside a slot's window are never read: imported states hold
NaN in every row the next steps must not read (positions never written, the row
of the position that just left the window after a wrap), and reset slots keep a
ring full of NaN.  Every output stays finite and matches the oracle, on the
CUDA-core path (2 slots) and the tensor-core path (6 slots)."""
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


@pytest.mark.parametrize("n", [2, 6])
def test_stale_rows_never_read(mfs, n):
    s = synth.TINY.replace(weight_dtype="bf16", kv_dtype="bf16", window=16, max_slots=n)
    w = synth.make_weights(s, 60 + n, gain_std=0.1)
    ctx, orc = H.gpu_context(s, w), oracle.Oracle(s, w)
    # positions: early (rows above p unused), just below, at and just past a wrap, far past it
    pos = [3, 15, 16, 17, 40, 9][:n]
    reset = n - 1  # this slot gets a NaN ring, then a reset: it restarts at frame 0 over NaN rows
    for i in range(n):
        st = synth.slot_state(s, 60 + n, i, pos[i])
        H.nan_stale_rows(st, s, pos[i], all_rows=(i == reset))
        mfs.mfs_import_slot(ctx, i, st)
        orc.import_slot(i, st)
    mfs.mfs_reset_slot(ctx, reset)
    orc.reset_slot(reset)
    u = synth.user_frames(s, 60 + n, 12, n)
    tally = H.Tally(f"NaN stale rows, {n} slots")
    for p in range(12):
        text, codes = mfs.mfs_step(ctx, list(range(n)), u[p])
        dbg = mfs.mfs_read_debug(ctx)
        assert np.isfinite(dbg["text_logits"]).all() and np.isfinite(dbg["dep_logits"]).all(), f"frame {p}"
        fol = H.follow_tokens(text, codes, dbg["code_argmax"])
        ref = orc.step(list(range(n)), u[p], want_logits=True, follow=fol)
        np.testing.assert_array_equal(codes, ref["codes"])
        tally.step(dbg, list(range(n)), ref, f"frame {p}")
    print(tally.report())
