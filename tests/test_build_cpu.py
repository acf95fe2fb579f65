"""The build's dependency rule: an edit to any header under csrc/ or include/
recompiles every translation unit (so a stale library is never shipped), and
an up-to-date tree recompiles nothing.  Checked on a scratch copy of the file
layout, without running nvcc."""
import os
import shutil
import time

from quantization_mxfp4_cast_gb300 import build


def make_tree(tmp_path):
    csrc, inc, bld = tmp_path / "csrc", tmp_path / "include", tmp_path / "_build"
    for d in (csrc, inc, bld):
        d.mkdir()
    for f in os.listdir(build.CSRC):
        if f.endswith((".cu", ".cuh", ".h")):
            shutil.copy(os.path.join(build.CSRC, f), csrc / f)
    shutil.copy(os.path.join(build.INCLUDE, "mxfp4.h"), inc / "mxfp4.h")
    old = time.time() - 100
    for f in list(csrc.iterdir()) + list(inc.iterdir()):
        os.utime(f, (old, old))
    for src in build.SOURCES:
        (bld / src.replace(".cu", ".o")).write_bytes(b"")  # objects newer than the sources
    return csrc, inc, bld


def test_every_header_is_a_dependency(tmp_path):
    csrc, inc, bld = make_tree(tmp_path)
    names = {os.path.basename(h) for h in build.headers(str(csrc), str(inc))}
    assert {"ptx.cuh", "quant.cuh", "internal.h", "mxfp4.h"} <= names
    assert build.stale_sources(str(csrc), str(inc), str(bld)) == []
    for n, h in enumerate(build.headers(str(csrc), str(inc))):
        t = time.time() + 100 * (n + 1)
        os.utime(h, (t, t))
        assert build.stale_sources(str(csrc), str(inc), str(bld)) == build.SOURCES, os.path.basename(h)
        for o in bld.iterdir():
            os.utime(o, (t + 1, t + 1))
        assert build.stale_sources(str(csrc), str(inc), str(bld)) == []


def test_a_source_edit_rebuilds_that_object_only(tmp_path):
    csrc, inc, bld = make_tree(tmp_path)
    t = time.time() + 100
    os.utime(csrc / "cast.cu", (t, t))
    assert build.stale_sources(str(csrc), str(inc), str(bld)) == ["cast.cu"]
    assert build.stale_sources(str(csrc), str(inc), str(bld), force=True) == build.SOURCES
