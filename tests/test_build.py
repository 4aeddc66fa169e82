"""The in-tree build's freshness check: a library is reused only when it is newer than every
source and was compiled with the same extra flags (a flagged diagnostic build must not be
mistaken for the product build, or the other way round)."""
import os

from mla_latent_kv_78_b300 import build as B


def _lib(tmp_path, flags=None, mtime=100.0):
    lib = tmp_path / "libx.so"
    lib.write_bytes(b"\0")
    os.utime(lib, (mtime, mtime))
    if flags is not None:
        (tmp_path / "libx.so.flags").write_text(flags)
    return str(lib)


def test_current_when_newer_and_same_flags(tmp_path):
    lib = _lib(tmp_path, flags="")
    assert B.is_current(lib, 99.0, "")
    assert B.is_current(lib, 100.0, "")


def test_stale_when_a_source_is_newer(tmp_path):
    lib = _lib(tmp_path, flags="")
    assert not B.is_current(lib, 101.0, "")


def test_stale_when_the_flags_differ(tmp_path):
    lib = _lib(tmp_path, flags="-DMLA_TC_TRACE")
    assert not B.is_current(lib, 99.0, "")
    lib = _lib(tmp_path, flags="")
    assert not B.is_current(lib, 99.0, "-DMLA_TC_TRACE")


def test_stale_without_a_stamp_or_a_library(tmp_path):
    lib = _lib(tmp_path, flags=None)
    assert not B.is_current(lib, 99.0, "")
    assert not B.is_current(str(tmp_path / "missing.so"), 0.0, "")
