"""The in-tree build is keyed on the sources' contents, the flags and the host
architecture, not on modification times: a library copied from another machine or built
from other sources is rebuilt even when it looks newer than every source."""
import os
import platform

from mixed_precision_tensor_gb300 import _build


def test_newer_library_with_another_key_is_stale(tmp_path):
    lib = tmp_path / "libtcg.so"
    lib.write_bytes(b"not this build")
    key = _build.source_key()
    assert not _build.up_to_date(str(lib), key)             # no stamp at all
    (tmp_path / "libtcg.so.key").write_text("0" * 64 + "\n")
    future = os.path.getmtime(_build.CSRC) + 10 ** 6
    os.utime(lib, (future, future))                           # newer than every source
    assert not _build.up_to_date(str(lib), key)
    (tmp_path / "libtcg.so.key").write_text(key + "\n")
    assert _build.up_to_date(str(lib), key)


def test_key_covers_contents_and_architecture(tmp_path, monkeypatch):
    a = tmp_path / "a.cu"
    a.write_text("kernel one\n")
    k1 = _build.source_key([str(a)])
    a.write_text("kernel two\n")
    k2 = _build.source_key([str(a)])
    assert k1 != k2
    a.write_text("kernel one\n")
    os.utime(a, (1, 1))                                        # mtime does not matter
    assert _build.source_key([str(a)]) == k1
    other = "aarch64" if platform.machine() != "aarch64" else "x86_64"
    monkeypatch.setattr(_build.platform, "machine", lambda: other)
    assert _build.source_key([str(a)]) != k1
