"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/dspark.h declares, sizes its workspace, and rejects
bad arguments before touching the device."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "dspark_build", os.path.join(ROOT, "verify_markov_head_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return C.CDLL(b.build())


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(dspark_[a-z_0-9]+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"dspark_draft_markov", "dspark_confidence_sts", "dspark_schedule", "dspark_verify"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    lib.dspark_status_string.restype = C.c_char_p
    assert lib.dspark_version() >= 100
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.dspark_status_string(code)


def test_workspace_sizes(lib):
    lib.dspark_workspace_bytes.restype = C.c_size_t
    assert lib.dspark_workspace_bytes(64, 7, 151936, 256) > 0
    assert lib.dspark_workspace_bytes(4, 7, 1024, 32) > 0
    assert lib.dspark_workspace_bytes(0, 7, 1024, 32) == 0        # B < 1
    assert lib.dspark_workspace_bytes(4, 17, 1024, 32) == 0       # gamma above the limit
    assert lib.dspark_workspace_bytes(4, 7, 1020, 32) == 0        # V not a multiple of 8
    lib.dspark_sts_workspace_bytes.restype = C.c_size_t
    assert lib.dspark_sts_workspace_bytes(7, 256, 15) >= 7 * 256 * 15 * 8   # int64 bin totals
    assert lib.dspark_sts_workspace_bytes(7, 65537, 15) == 0      # grid above the limit
    assert lib.dspark_sts_workspace_bytes(7, 256, 65) == 0        # bins above the limit
    assert lib.dspark_sts_workspace_bytes(0, 256, 15) == 0        # gamma < 1


def test_null_pointers_are_rejected_without_a_device(lib):
    vp = C.c_void_p
    lib.dspark_draft_markov.argtypes = [vp, C.c_int, vp, vp, C.c_int, vp, C.c_int, C.c_int, C.c_int, C.c_int,
                                        C.c_int, C.c_float, C.c_uint64, C.c_uint64, vp, vp, vp, vp, vp,
                                        C.c_size_t, vp]
    st = lib.dspark_draft_markov(None, 0, None, None, 0, None, 4, 7, 1024, 32, 0, 1.0, 0, 0,
                                 None, None, None, None, None, 0, None)
    assert st == -1
    st = lib.dspark_draft_markov(None, 0, None, None, 0, None, 4, 7, 1024, 32, 0, -1.0, 0, 0,
                                 None, None, None, None, None, 0, None)
    assert st == -1
    lib.dspark_schedule.argtypes = [vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp, vp, vp,
                                    C.c_size_t, vp]
    assert lib.dspark_schedule(None, None, None, 32, 4, 7, 1, None, None, None, None, 0, None) == -1
    assert lib.dspark_schedule(None, None, None, 32, 1000, 7, 1, None, None, None, None, 0, None) == -1
    assert lib.dspark_schedule(None, None, None, 32, 4, 7, 9, None, None, None, None, 0, None) == -1


def test_target_stream_and_full_prefix_verify_reject_bad_arguments(lib):
    """dspark_draft_markov_target and a full-prefix dspark_verify (K = NULL)
    check their arguments on the host: null or host pointers, a bad
    temperature or an unknown target type return before any launch."""
    vp = C.c_void_p
    lib.dspark_draft_markov_target.argtypes = [vp, C.c_int, vp, vp, C.c_int, vp, C.c_int, vp, C.c_int, C.c_int,
                                               C.c_int, C.c_int, C.c_int, C.c_float, C.c_uint64, C.c_uint64,
                                               vp, vp, vp, vp, vp, C.c_size_t, vp]
    args = [None, 0, None, None, 1, None, 0, None, 4, 7, 1024, 64, 0, 1.0, 0, 0, None, None, None, None, None, 0,
            None]
    assert lib.dspark_draft_markov_target(*args) == -1          # null pointers
    host = (C.c_float * 64)()
    args_host = list(args)
    for i in (0, 2, 3, 5, 7, 16, 17, 18, 20):
        args_host[i] = C.cast(host, vp)
    assert lib.dspark_draft_markov_target(*args_host) == -1     # host memory is not device memory
    bad_tau = list(args)
    bad_tau[13] = 0.0
    assert lib.dspark_draft_markov_target(*bad_tau) == -1
    bad_type = list(args)
    bad_type[6] = 7
    assert lib.dspark_draft_markov_target(*bad_type) == -4      # unknown target type: unsupported
    lib.dspark_verify.argtypes = [vp, C.c_int, vp, C.c_int, vp, vp, C.c_int, vp, vp, vp, vp, vp,
                                  C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_float, C.c_uint64, C.c_uint64,
                                  vp, vp, vp, vp, vp, vp, vp, vp, vp, C.c_size_t, vp]
    st = lib.dspark_verify(None, 0, None, 0, None, None, 1, None, None, None, None, None,   # K = NULL
                           4, 7, 1024, 64, 0, 1.0, 0, 0, None, None, None, None, None, None, None, None, None,
                           0, None)
    assert st == -1


def test_noalloc_draft_rejects_host_pointers_and_large_batches(lib):
    """dspark_draft_markov_noalloc checks its arguments as dspark_draft_markov
    does: host memory is not device memory (DSPARK_ERR_INVALID, before any
    launch), and a batch beyond its fixed array is unsupported."""
    vp = C.c_void_p
    lib.dspark_draft_markov_noalloc.argtypes = [vp, C.c_int, vp, vp, C.c_int, vp, C.c_int, C.c_int, C.c_int,
                                                C.c_int, C.c_int, C.c_float, C.c_uint64, C.c_uint64,
                                                vp, vp, vp, vp, vp]
    host = (C.c_float * 64)()
    h = C.cast(host, vp)
    args = [h, 0, h, h, 1, h, 4, 7, 1024, 64, 0, 1.0, 0, 0, h, h, h, None, None]
    assert lib.dspark_draft_markov_noalloc(*args) == -1          # host pointers
    args_null = list(args)
    args_null[0] = None
    assert lib.dspark_draft_markov_noalloc(*args_null) == -1
    bad_tau = list(args)
    bad_tau[11] = float("nan")
    assert lib.dspark_draft_markov_noalloc(*bad_tau) == -1


def test_package_imports_and_fails_loudly_without_library(tmp_path):
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r); import verify_markov_head_gb300 as vm; "
            "print(vm.dspark_version())" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert r.returncode == 0 and int(r.stdout.strip()) >= 100
