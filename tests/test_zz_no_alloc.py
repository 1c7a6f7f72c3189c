"""The argmax entry point that allocates no device memory (mfs_argmax_rows_noalloc).

Callers that cannot call cudaMalloc when they pick tokens (a serving engine
whose allocator already holds the free device memory, a real-time loop that
must not block on the allocator) use this call; its scratch is a fixed array
inside the library.  Here it is checked against the frame step's own text and
code argmax (mfs_step, read back with mfs_read_debug) on the logits of two
frames in a row, so that the second call runs on the scratch the first left.
"""
import ctypes

import numpy as np
import pytest

import synth
from tests import _harness as H


@pytest.fixture(scope="module")
def mfs():
    from full_duplex_speech_frame_gb300 import mfs as m
    return m


def test_noalloc_rejects_sizes_beyond_its_scratch(mfs):
    """Host-side checks only: nothing is launched, the pointers are never touched."""
    fake = ctypes.c_void_p(16)
    lib = mfs._lib
    rc = lib.mfs_argmax_rows_noalloc(fake, 4097, 10, 10, fake, None)
    assert rc == -4 and "exceed the fixed scratch" in mfs.mfs_last_error(None)
    rc = lib.mfs_argmax_rows_noalloc(fake, 17, 65536 * 4096 // 16, 65536 * 4096 // 16, fake, None)
    assert rc == -4
    assert lib.mfs_argmax_rows_noalloc(fake, 4, 10, 9, fake, None) == -1
    assert lib.mfs_argmax_rows_noalloc(None, 4, 10, 10, fake, None) == -1
    assert lib.mfs_argmax_rows_noalloc(None, 0, 10, 10, None, None) == 0


@pytest.mark.gpu
def test_noalloc_argmax_matches_the_step(mfs):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    s = synth.TINY.replace(max_slots=2, window=8)
    w = synth.make_weights(s, 5, gain_std=0.1)
    ctx = H.gpu_context(s, w)
    u = synth.user_frames(s, 5, 2, 2)
    stream = torch.cuda.current_stream()
    for p in range(2):  # two frames, two calls each, back to back on one stream
        mfs.mfs_step(ctx, [0, 1], u[p])
        dbg = mfs.mfs_read_debug(ctx)
        tl = torch.from_numpy(dbg["text_logits"]).cuda()
        dl = torch.from_numpy(dbg["dep_logits"].reshape(-1, s.card)).cuda()
        t_out = torch.full((2,), -7, dtype=torch.int32, device="cuda")
        c_out = torch.full((32,), -7, dtype=torch.int32, device="cuda")
        mfs.mfs_argmax_rows_noalloc(tl, t_out, stream.cuda_stream)
        mfs.mfs_argmax_rows_noalloc(dl, c_out, stream.cuda_stream)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(t_out.cpu().numpy(), dbg["text_argmax"])
        np.testing.assert_array_equal(c_out.cpu().numpy().reshape(2, 16), dbg["code_argmax"])


@pytest.mark.gpu
def test_noalloc_argmax_many_column_blocks(mfs):
    """Rows of 32000 columns (8 blocks each, the text head's width), with ties planted
    across block boundaries and strided rows: lowest index of the maximum, as numpy."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(7)
    rows, cols, ld = 64, 32000, 32008
    x = rng.standard_normal((rows, ld)).astype(np.float32)
    x[:, cols:] = 100.0  # padding beyond cols must be ignored
    for r in range(0, rows, 3):
        a, b = sorted(rng.choice(cols, 2, replace=False))
        x[r, a] = x[r, b] = 9.0  # tie: the lower column wins
    x[5, :cols] = -np.inf
    x[6, :cols] = np.nan
    x[6, 31999] = 1.0
    dev = torch.from_numpy(x).cuda()[:, :cols]
    out = torch.empty(rows, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out.fill_(-7)
        mfs.mfs_argmax_rows_noalloc(dev, out, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        want = np.argmax(np.where(np.isnan(x[:, :cols]), -np.inf, x[:, :cols]), axis=1)
        np.testing.assert_array_equal(out.cpu().numpy(), want)
