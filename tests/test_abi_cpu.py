"""The C-ABI library builds, loads and exports every entry point that
include/mfs.h declares; the binding's config struct matches the header's
layout.  No GPU needed (no compute calls)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mfs.h")


@pytest.fixture(scope="module")
def lib():
    from full_duplex_speech_frame_gb300.build import build
    build()
    from full_duplex_speech_frame_gb300 import mfs
    return mfs


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mfs_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 15
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, missing
    nm = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (mfs_\w+)", nm))
    assert set(names) <= exported


def test_config_struct_layout_matches_header(lib, tmp_path):
    src = tmp_path / "probe.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "mfs.h"\nint main(void){'
                   'printf("%zu %zu %zu %zu %zu\\n", sizeof(mfs_config), offsetof(mfs_config, delays),'
                   ' offsetof(mfs_config, rope_theta), offsetof(mfs_config, weight_dtype),'
                   ' offsetof(mfs_config, max_slots)); return 0;}\n')
    exe = tmp_path / "probe"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    C = lib.mfs_config
    assert got == [ctypes.sizeof(C), C.delays.offset, C.rope_theta.offset, C.weight_dtype.offset,
                   C.max_slots.offset]


def test_create_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import synth
    from tests import _harness as H
    with pytest.raises(lib.MfsError) as e:
        lib.mfs_create(H.config_of(synth.TINY))
    assert e.value.status == "MFS_E_CUDA"
    assert lib.mfs_last_error(None)


def test_bad_config_is_rejected_with_reason(lib):
    import synth
    from tests import _harness as H
    cfg = H.config_of(synth.TINY.replace(head_dim=48))
    with pytest.raises(lib.MfsError) as e:
        lib.mfs_create(cfg)
    # without a GPU the device query fails first; with one, the shape check does
    assert e.value.status in ("MFS_E_ARG", "MFS_E_CUDA")
