"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
declared symbol, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import glob
import os
import re

import pytest

import non_cartesian_mri_gather_gb300 as fhd
from non_cartesian_mri_gather_gb300 import build as fhd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fhd_build.build()
    return fhd.load()


def declared_functions():
    names = []
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        src = "\n".join(l for l in src.splitlines() if not l.strip().startswith("#"))
        names += re.findall(r"\b([A-Za-z_]\w*)\s*\(", src)
    return sorted(set(names))


def test_headers_declare_the_operators():
    names = declared_functions()
    for n in ("fhd_compute", "fwd_compute", "fhfrho_apply", "fhd_workspace_bytes", "fhd_workspace_status",
              "fhd_status_string"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in fhd.SIGNATURES, f"binding lacks {name}"


def test_version_and_strings(lib):
    assert fhd.fhd_version() == 100
    for s in range(8):
        assert len(fhd.fhd_status_string(s)) >= 2
    assert fhd.fhd_status_string(99) == "unknown status"


# Fake, never-dereferenced addresses: validation must reject these calls on the host.
A = 0x10000000


def call_fhd(lib, M=10, N=10, ptrs=None, out=None, mode=0, ws=A + 0x100000, wsb=1 << 30):
    p = ptrs if ptrs is not None else [A + 0x1000 * i for i in range(8)]
    o = out if out is not None else [A + 0x20000, A + 0x30000]
    return lib.fhd_compute(M, p[0], p[1], p[2], p[3], p[4], N, p[5], p[6], p[7], o[0], o[1], mode, ws, wsb, None)


def test_rejects_negative_sizes(lib):
    assert call_fhd(lib, M=-1) == 1
    assert call_fhd(lib, N=-5) == 1
    assert lib.fwd_compute(-1, *[A] * 5, 3, *[A] * 5, 0, A, 1 << 20, None) == 1
    assert lib.fhfrho_apply(3, *[A] * 5, -2, *[A] * 5, 0, A, 1 << 20, None) == 1


def test_rejects_bad_mode(lib):
    assert call_fhd(lib, mode=7) == 1
    assert call_fhd(lib, mode=4) == 1


def test_rejects_null(lib):
    p = [A + 0x1000 * i for i in range(8)]
    p[3] = None
    assert call_fhd(lib, ptrs=p) == 1
    assert call_fhd(lib, out=[A + 0x20000, None]) == 1


def test_rejects_misaligned(lib):
    p = [A + 0x1000 * i for i in range(8)]
    p[6] += 2
    assert call_fhd(lib, ptrs=p) == 2
    assert call_fhd(lib, ws=A + 0x100000 + 64) == 2


def test_rejects_aliasing(lib):
    # output overlaps an input
    assert call_fhd(lib, out=[A + 0x1000 * 5 + 8, A + 0x30000]) == 3
    # the two outputs overlap each other
    assert call_fhd(lib, out=[A + 0x20000, A + 0x20000 + 4]) == 3


def test_rejects_missing_workspace(lib):
    assert call_fhd(lib, ws=None) == 4


def test_empty_problems_are_noops(lib):
    # N == 0: nothing to write, no pointer is needed and no CUDA call is made
    assert lib.fhd_compute(10, None, None, None, None, None, 0, None, None, None, None, None, 0, None, 0, None) == 0
    assert lib.fwd_compute(10, None, None, None, None, None, 0, None, None, None, None, None, 1, None, 0, None) == 0
    assert lib.fhfrho_apply(0, None, None, None, None, None, 10, None, None, None, None, None, 0, None, 0, None) == 0


def test_workspace_bytes_without_device(lib):
    # no GPU here: the query fails cleanly with 0
    assert fhd.fhd_workspace_bytes(fhd.OP_FHD, 100, 100, 0) >= 0
    assert lib.fhd_workspace_bytes(9, 1, 1, 0) == 0
    assert lib.fhd_workspace_bytes(0, -1, 1, 0) == 0


def test_binding_requires_library(tmp_path, monkeypatch):
    import importlib

    mod = importlib.import_module("non_cartesian_mri_gather_gb300")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        mod.load()


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 152, 304, 1000])
def test_schedule_replay(lib, ctas):
    """Host replay of the gather/fix-up schedule: every block finished once, fix-ups complete."""
    TB, T = 2048, 128
    cases = [(1, 1), (1, 5000), (1024, 2048), (2049, 129), (262144, 16384), (2097152, 262144),
             (16777216, 100000), (262144, 2097152), (3 * TB + 5, 3 * T + 7), (100, 200000), (5000000, 3)]
    for nt, ns in cases:
        assert lib.fhd_test_schedule(nt, ns, ctas) == 0, (nt, ns, ctas)


def test_schedule_rejects_empty(lib):
    assert lib.fhd_test_schedule(0, 10, 4) != 0
    assert lib.fhd_test_schedule(10, 0, 4) != 0


def test_set_path_hook(lib):
    prev = lib.fhd_test_set_path(0)
    assert prev in (0, 1, 2)
    assert lib.fhd_test_set_path(3) == -1
    assert lib.fhd_test_set_path(-1) == -1
    assert lib.fhd_test_set_path(2) == 0
    assert lib.fhd_test_set_path(prev) == 2
    prev = lib.fhd_test_set_step_records(1)
    assert prev in (0, 1)
    assert lib.fhd_test_set_step_records(2) == -1
    assert lib.fhd_test_set_step_records(0) == 1
    assert lib.fhd_test_set_step_records(prev) == 0


# Partial rows of a workspace on a 152-SM device: 2 slots per CTA of
# 2 x 8192 floats.
_PARTIAL = 2 * 152 * 2 * 8192 * 4


@pytest.mark.parametrize("nt,ns", [(1, 1), (1, 100000), (1024, 2048), (2049, 1000), (300, 31), (20000, 777),
                                   (320000, 40), (311296, 5), (100, 40000), (8192, 2048)])
def test_split_shape_covers_sources(lib, nt, ns):
    """Slices cover the sources once and their partial rows fit the workspace."""
    import ctypes

    k, ln = ctypes.c_int(0), ctypes.c_int64(0)
    assert lib.fhd_test_split_shape(nt, ns, 152, 152, _PARTIAL, ctypes.byref(k), ctypes.byref(ln)) in (0, 1)
    assert 1 <= k.value <= 65535 and ln.value >= 1
    assert k.value * ln.value >= ns and (k.value - 1) * ln.value < ns
    if k.value > 1:
        assert 2 * 4 * nt * k.value <= _PARTIAL
        assert ln.value >= 32 or ns < 64


def test_split_shape_choice(lib):
    """The benchmark workloads: 32^2 x 2048 is split; the 3D ones are not."""
    for nt, ns, want in [(1024, 2048, 1), (262144, 16384, 0), (2097152, 262144, 0), (16777216, 100000, 0),
                         (262144, 2097152, 0), (1, 1, 1), (65536, 4096, 0), (5000, 2000, 1)]:
        assert lib.fhd_test_split_shape(nt, ns, 152, 152, _PARTIAL, None, None) == want, (nt, ns)
    assert lib.fhd_test_split_shape(0, 1, 152, 152, _PARTIAL, None, None) == -1
