"""The C-ABI library builds, loads without a GPU and exports every symbol include/*.h declares.
Host-side validation is exercised through calls that must fail before any launch."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", src):
            name = m.group(1)
            if name.startswith("spec_"):
                names.add(name)
    return names


@pytest.fixture(scope="module")
def cuda_lib():
    from draft_sampling_verification_markov_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_every_declared_symbol_is_exported(cuda_lib):
    names = _declared_functions()
    assert {"spec_markov_propose", "spec_verify_greedy", "spec_verify_rejection",
            "spec_tv_confidence", "spec_schedule_prefix"} <= names
    missing = [n for n in sorted(names) if not hasattr(cuda_lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_host_only_entry_points(cuda_lib):
    cuda_lib.spec_abi_version.restype = ctypes.c_int
    assert cuda_lib.spec_abi_version() == 1
    cuda_lib.spec_status_string.restype = ctypes.c_char_p
    cuda_lib.spec_status_string.argtypes = [ctypes.c_int]
    assert cuda_lib.spec_status_string(0) == b"ok"
    assert b"workspace" in cuda_lib.spec_status_string(-3)
    f = cuda_lib.spec_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 5
    a = f(0, 256, 7, 129280, 256)
    assert a > 256 and a % 256 == 0
    assert f(7, 256, 7, 129280, 256) >= max(f(op, 256, 7, 129280, 256) for op in range(7))
    assert f(0, -1, 7, 10, 0) == 0          # invalid sizes report 0
    assert f(99, 1, 1, 1, 0) == 0


def test_validation_rejects_before_launch(cuda_lib):
    """Bad arguments return error codes without touching the device (null workspace,
    negative sizes, unknown dtype, bad temperature)."""
    vp = ctypes.c_void_p
    fn = cuda_lib.spec_markov_propose
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_float,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, ctypes.c_size_t, vp]
    bogus = vp(0x1000)
    # negative R
    assert fn(bogus, 1, None, None, 1, 0, None, None, 0.0, -1, 2, 8, bogus, None, None, bogus,
              1 << 20, None) == -1
    # unknown dtype
    assert fn(bogus, 7, None, None, 1, 0, None, None, 0.0, 1, 2, 8, bogus, None, None, bogus,
              1 << 20, None) == -2
    # negative temperature
    assert fn(bogus, 1, None, None, 1, 0, None, None, -1.0, 1, 2, 8, bogus, None, None, bogus,
              1 << 20, None) == -1
    # misaligned workspace
    assert fn(bogus, 1, None, None, 1, 0, None, None, 0.0, 1, 2, 8, bogus, None, None,
              vp(0x1010), 1 << 20, None) == -1
    # workspace too small
    assert fn(bogus, 1, None, None, 1, 0, None, None, 0.0, 1, 2, 8, bogus, None, None, bogus,
              16, None) == -3
    # rank > 0 without weights
    assert fn(bogus, 1, None, None, 1, 64, None, None, 0.0, 1, 2, 8, bogus, None, None, bogus,
              1 << 20, None) == -1
    sched = cuda_lib.spec_schedule_prefix
    sched.restype = ctypes.c_int
    sched.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp,
                      ctypes.c_size_t, vp]
    # Bmax < R, and too many candidates
    assert sched(bogus, bogus, 3, 4, 2, bogus, bogus, bogus, bogus, 1024, None) == -1
    assert sched(bogus, bogus, 1 << 20, 2048, 16, bogus, bogus, bogus, bogus, 1024, None) == -1
    topk = cuda_lib.spec_schedule_topk
    topk.restype = ctypes.c_int
    topk.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                     ctypes.c_size_t, vp]
    # no capacity, then Bmax < R
    assert topk(bogus, bogus, 8, 4, 2, None, bogus, bogus, bogus, None, bogus, 1024, None) == -1
    assert topk(bogus, bogus, 3, 4, 2, bogus, bogus, bogus, bogus, None, bogus, 1024, None) == -1
    # flattened batch: lengths and offsets are required
    fl = cuda_lib.spec_flat_layout
    fl.restype = ctypes.c_int
    fl.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, ctypes.c_size_t, vp]
    assert fl(None, 4, 3, bogus, None, None, bogus, 1024, None) == -1
    assert fl(bogus, 4, 3, None, None, None, bogus, 1024, None) == -1
    gf = cuda_lib.spec_verify_greedy_flat
    gf.restype = ctypes.c_int
    gf.argtypes = [vp, ctypes.c_int, vp, vp, vp] + [ctypes.c_int] * 3 + [vp] * 4 + [
        ctypes.c_size_t, vp]
    assert gf(bogus, 1, bogus, bogus, None, 4, 3, 8, bogus, None, None, bogus, 1 << 20,
              None) == -1
    # packing rows into the flattened layout: a row width that is not a multiple of 4 bytes,
    # missing lengths, a misaligned destination
    fp = cuda_lib.spec_flat_pack
    fp.restype = ctypes.c_int
    fp.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp,
                   ctypes.c_size_t, vp]
    assert fp(bogus, 6, bogus, bogus, 4, 3, bogus, bogus, 1024, None) == -1
    assert fp(bogus, 8, None, bogus, 4, 3, bogus, bogus, 1024, None) == -1
    assert fp(bogus, 8, bogus, bogus, 4, 3, vp(0x1002), bogus, 1024, None) == -1
    # the MTP greedy step: a bad dtype, no target, a workspace too small, no draft logits
    mg = cuda_lib.spec_mtp_greedy
    mg.restype = ctypes.c_int
    mg.argtypes = [vp, vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp,
                   vp, vp, vp, ctypes.c_size_t, vp]
    assert mg(bogus, bogus, 5, None, 4, 3, 64, bogus, bogus, None, None, bogus, 1 << 20,
              None) == -2
    assert mg(bogus, None, 1, None, 4, 3, 64, bogus, bogus, None, None, bogus, 1 << 20,
              None) == -1
    assert mg(bogus, bogus, 1, None, 4, 3, 64, bogus, bogus, None, None, bogus, 16, None) == -3
    assert mg(None, bogus, 1, None, 4, 3, 64, bogus, bogus, None, None, bogus, 1 << 20,
              None) == -1
    # the no-allocation greedy verify: beyond its fixed scratch, then a bad dtype
    na = cuda_lib.spec_verify_greedy_noalloc
    na.restype = ctypes.c_int
    na.argtypes = [vp, ctypes.c_int, vp, vp] + [ctypes.c_int] * 3 + [vp] * 5
    assert na(bogus, 0, bogus, None, 16385, 3, 8, bogus, bogus, bogus, None, None) == -7
    assert na(bogus, 9, bogus, None, 4, 3, 8, bogus, bogus, bogus, None, None) == -2


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from draft_sampling_verification_markov_gb300 import build, spec
    monkeypatch.setattr(build, "SO", str(tmp_path / "missing.so"))
    monkeypatch.setattr(spec, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        spec.lib()
