"""Mimi split RVQ encode on the GPU (mfs_rvq_encode) against the oracle's quantizer."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

GAP = 0.05  # distances within this of each other may rank differently in fp32 and fp64


@pytest.fixture(scope="module")
def mfs():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from full_duplex_speech_frame_gb300 import mfs as m
    return m


def _case(T, D, Cb, seed):
    zs = synth.normal_f32(seed, 501, T * D).reshape(T, D)
    za = synth.normal_f32(seed, 502, T * D).reshape(T, D)
    cb = synth.normal_f32(seed, 503, 8 * Cb * D).reshape(8, Cb, D)
    return zs, za, cb


def _encode(mfs, zs, za, cb):
    import torch
    codes = torch.full((zs.shape[0], 8), -7, dtype=torch.int32, device="cuda")
    mfs.mfs_rvq_encode(torch.from_numpy(zs).cuda(), torch.from_numpy(za).cuda(), torch.from_numpy(cb).cuda(), codes)
    torch.cuda.synchronize()
    return codes.cpu().numpy()


@pytest.mark.parametrize("T,D,Cb", [(37, 256, 2048), (1, 1024, 300), (16, 8, 5)])
def test_rvq_matches_oracle(mfs, T, D, Cb):
    """Codes equal the oracle's; a frame's chain is compared up to a stage whose best two
    distances lie within GAP (there fp32 may rank them the other way; later residuals differ)."""
    zs, za, cb = _case(T, D, Cb, T + D)
    got = _encode(mfs, zs, za, cb)
    want, gap = oracle.rvq_encode(zs, za, cb)
    compared = 0
    for t in range(T):
        if got[t, 0] != want[t, 0]:
            assert gap[t, 0] < GAP, (t, 0)
        for q in range(1, 8):
            if got[t, q] != want[t, q]:
                assert gap[t, q] < GAP, (t, q, gap[t, q])
                break
            compared += 1
    assert compared >= 6 * T


def test_rvq_rejects_bad_sizes(mfs):
    import torch
    z = torch.zeros(4, 6, device="cuda")
    with pytest.raises(mfs.MfsError):
        mfs.mfs_rvq_encode(z, z, torch.zeros(8, 4, 6, device="cuda"), torch.zeros(4, 8, dtype=torch.int32, device="cuda"))
