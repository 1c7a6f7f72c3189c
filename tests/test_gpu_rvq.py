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


def _compare(got, want, gap, T):
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


# D a multiple of 8 runs on the tensor cores (approximate scores, fp32 re-rank of the candidates
# near the best score): CTA pairs of 32 frames up to D = 520, one CTA per 16 frames for D = 1024;
# D = 12 and D = 36 on the CUDA cores (every distance exact).  2432 x 256 x 2048 is the timed
# workload; 2472 frames take two launches of CTA pairs; Cb = 300, 130 and 5 leave ragged codeword
# tiles (Cb = 5: the second CTA of a pair has no tile), T = 37 a ragged frame group.
@pytest.mark.parametrize("T,D,Cb", [(37, 256, 2048), (1, 1024, 300), (16, 8, 5), (2432, 256, 2048),
                                    (23, 12, 100), (5, 36, 7), (40, 520, 130), (2472, 64, 300)])
def test_rvq_matches_oracle(mfs, T, D, Cb):
    """Codes equal the oracle's; a frame's chain is compared up to a stage whose best two
    distances lie within GAP (there fp32 may rank them the other way; later residuals differ)."""
    zs, za, cb = _case(T, D, Cb, T + D)
    got = _encode(mfs, zs, za, cb)
    want, gap = oracle.rvq_encode(zs, za, cb)
    _compare(got, want, gap, T)
    if T == 2432:  # no internal wait ran into its limit (that costs about 2 s and leaves codes -1)
        import torch
        z0, z1, c = (torch.from_numpy(a).cuda() for a in (zs, za, cb))
        out = torch.empty(T, 8, dtype=torch.int32, device="cuda")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        mfs.mfs_rvq_encode(z0, z1, c, out)
        e0.record()
        mfs.mfs_rvq_encode(z0, z1, c, out)
        e1.record()
        torch.cuda.synchronize()
        assert e0.elapsed_time(e1) < 100.0
        assert (out.cpu().numpy() == got).all()


def test_rvq_clustered_codebooks(mfs):
    """Codebooks of 64 clusters of 48 close codewords (member m of cluster g at index 64 m + g:
    a cluster spans every codeword tile but lies in one class of indices mod 8), latents near
    cluster centres: the nearest codeword has 47 close rivals in its own class, of which the
    tensor-core path keeps the best 2 by its approximate score, yet it must still be found."""
    T, D, G, M = 64, 256, 64, 48
    Cb = G * M
    centre = synth.normal_f32(7, 511, 8 * G * D).reshape(8, 1, G, D)
    member = 0.3 * synth.normal_f32(7, 512, 8 * M * G * D).reshape(8, M, G, D)
    cb = np.ascontiguousarray((centre + member).reshape(8, Cb, D), np.float32)
    pick = (np.arange(T) * 37) % G
    zs = np.ascontiguousarray(centre[0, 0, pick] + 0.05 * synth.normal_f32(7, 513, T * D).reshape(T, D), np.float32)
    za = np.ascontiguousarray(centre[1, 0, pick[::-1]] + 0.05 * synth.normal_f32(7, 514, T * D).reshape(T, D),
                              np.float32)
    got = _encode(mfs, zs, za, cb)
    want, gap = oracle.rvq_encode(zs, za, cb)
    assert (got[:, 0] % G == pick).all() and (got[:, 1] % G == pick[::-1]).all()
    _compare(got, want, gap, T)


def test_rvq_rejects_bad_sizes(mfs):
    import torch
    z = torch.zeros(4, 6, device="cuda")
    with pytest.raises(mfs.MfsError):
        mfs.mfs_rvq_encode(z, z, torch.zeros(8, 4, 6, device="cuda"), torch.zeros(4, 8, dtype=torch.int32, device="cuda"))
