"""The C-ABI library loads, exports every symbol include/*.h declares, and rejects bad arguments on
the host before touching a GPU (no compute call is made here)."""
import ctypes
import glob
import os
import re
import threading

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[\w ]+?\s*\*?\s*(mamba_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def ms():
    import sequence_scan_selective_b300 as m
    return m


def test_header_declares_entry_points():
    assert {"mamba_scan_fwd", "mamba_state_step", "mamba_scan_last_error", "mamba_scan_version",
            "mamba_scan_launch_count", "mamba_scan_device_status"} <= _declared()


def test_library_exports_every_declared_symbol(ms):
    lib = ctypes.CDLL(ms.LIB_PATH)
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing
    assert set(ms.EXPORTED) >= _declared()


def test_version(ms):
    hdr = open(os.path.join(ROOT, "include", "mamba_scan.h")).read()
    v = int(re.search(r"#define MAMBA_SCAN_VERSION (\d+)", hdr).group(1))
    assert ms.version() == v


def _shape(ms, **kw):
    s = dict(batch=1, dim=4, dstate=16, seqlen=8, in_dtype=0)
    s.update(kw)
    return ms.Shape(**s)


def test_host_argument_checks(ms):
    lib = ms.lib()
    P = ctypes.c_void_p
    dummy = P(256)  # never dereferenced: every case below fails validation first
    assert lib.mamba_scan_fwd(None, dummy, dummy, dummy, dummy, dummy, None, None, None, 1, P(4096), None, None) == -1
    assert b"NULL" in lib.mamba_scan_last_error()
    for bad in (dict(batch=0), dict(dim=-1), dict(dstate=0), dict(dstate=65), dict(seqlen=-1), dict(in_dtype=2)):
        s = _shape(ms, **bad)
        rc = lib.mamba_scan_fwd(ctypes.byref(s), dummy, dummy, dummy, dummy, dummy, None, None, None, 1, P(1 << 40),
                                None, None)
        assert rc == -1, bad
        assert lib.mamba_scan_last_error()
    s = _shape(ms)
    assert lib.mamba_scan_fwd(ctypes.byref(s), None, dummy, dummy, dummy, dummy, None, None, None, 1, P(1 << 40),
                              None, None) == -1
    # y overlapping u
    assert lib.mamba_scan_fwd(ctypes.byref(s), P(1 << 20), P(1 << 30), dummy, P(1 << 31), P(1 << 32), None, None,
                              None, 1, P((1 << 20) + 8), None, None) == -1
    assert b"overlap" in lib.mamba_scan_last_error()
    assert lib.mamba_state_step(ctypes.byref(s), None, dummy, dummy, dummy, dummy, dummy, None, None, None, 1,
                                dummy, None) == -1
    assert lib.mamba_state_step(ctypes.byref(_shape(ms, dstate=100)), dummy, dummy, dummy, dummy, dummy, dummy,
                                None, None, None, 1, dummy, None) == -1


def test_error_message_is_thread_local(ms):
    lib = ms.lib()
    lib.mamba_scan_fwd(None, None, None, None, None, None, None, None, None, 1, None, None, None)
    seen = []
    t = threading.Thread(target=lambda: seen.append(lib.mamba_scan_last_error()))
    t.start()
    t.join()
    assert seen == [b""]
    assert lib.mamba_scan_last_error() != b""


def test_launch_counter_starts_without_gpu_work(ms):
    assert ms.launch_count() >= 0


def test_product_package_does_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "sequence_scan_selective_b300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if os.path.isfile(path) and path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            text = open(path, errors="replace").read()
            assert "oracle" not in text.lower(), path


def _prototypes():
    """name -> number of parameters, from the comment-stripped header."""
    out = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"(mamba_\w+)\s*\(([^)]*)\)\s*;", text):
            params = m.group(2).strip()
            out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_counts_match_header(ms):
    lib = ms.lib()
    protos = _prototypes()
    assert protos
    for name, n in protos.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)


def test_bwd_host_argument_checks(ms):
    lib = ms.lib()
    P = ctypes.c_void_p
    d = P(256)  # never dereferenced: every case below fails validation first
    args = lambda s, disc=0, z=None, dz=None, A=d: (ctypes.byref(s), disc, d, d, A, d, d, None, z, None, 1, None, d,
                                                   None, d, d, dz, d, d, d, None, None, None, None)
    assert lib.mamba_scan_bwd(*args(_shape(ms, dstate=65))) == -1
    assert b"dstate" in lib.mamba_scan_last_error()
    assert lib.mamba_scan_bwd(*args(_shape(ms), disc=7)) == -1
    assert lib.mamba_scan_bwd(*args(_shape(ms), dz=d)) == -1
    assert b"dz" in lib.mamba_scan_last_error()
    assert lib.mamba_scan_bwd(*args(_shape(ms), A=None)) == -1
    assert lib.mamba_scan_bwd(*args(_shape(ms, seqlen=-3))) == -1


def test_discretisation_and_conv_host_checks(ms):
    lib = ms.lib()
    P = ctypes.c_void_p
    d = P(256)  # never dereferenced: every case below fails validation first
    s = _shape(ms)
    # unknown discretisation
    assert lib.mamba_scan_fwd_ex(ctypes.byref(s), 5, d, d, d, d, d, None, None, None, 1, None, P(1 << 40), None,
                                 None) == -1
    assert b"discretization" in lib.mamba_scan_last_error()
    assert lib.mamba_state_step_ex(ctypes.byref(s), -1, d, d, d, d, d, d, None, None, None, 1, d, None) == -1
    # convolution: weights required, width 1..4
    conv = lambda w, k: lib.mamba_scan_fwd_conv(ctypes.byref(s), 0, d, w, None, k, 1, None, d, d, d, d, None, None,
                                                None, 1, None, P(1 << 40), None, None)
    assert conv(None, 4) == -1 and b"conv_w" in lib.mamba_scan_last_error()
    assert conv(d, 0) == -1 and b"conv_k" in lib.mamba_scan_last_error()
    assert conv(d, 5) == -1 and b"conv_k" in lib.mamba_scan_last_error()


def test_bench_byte_counts():
    """The algorithmic byte formulas the roofline divides by, against a hand count of one shape."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    import synth
    cfg = synth.CONFIGS["m130"]
    b, d, n, L = 8, 1536, 16, 2048
    # forward: u, delta, z read and y written (fp32), B and C read, A/D/bias, last_state
    assert bench.scan_bytes(cfg) == 4 * 4 * b * d * L + 2 * 4 * b * n * L + 4 * d * (n + 2) + 4 * b * d * n
    assert bench.scan_bytes(cfg) == 405647360
    # backward: u, delta, z, dy read, du, ddelta, dz written; B, C read, dB, dC written (fp32);
    # A, D, bias read and their gradients written; h0, dlast read, dh0 written
    assert bench.bwd_bytes(cfg) == (7 * 4 * b * d * L + 4 * 4 * b * n * L + 2 * 4 * d * (n + 2)
                                    + 3 * 4 * b * d * n)


def test_block_bwd_host_argument_checks(ms):
    """mamba_scan_bwd_conv refuses a missing kernel, a width outside 1..4 and a bad shape before
    touching the device."""
    lib = ms.lib()
    P = ctypes.c_void_p
    d = P(256)  # never dereferenced: every case below fails validation first
    args = lambda s, w=d, k=4: (ctypes.byref(s), 0, d, w, None, k, 1, None, d, d, d, d, None, None, None, 1, None,
                                d, None, d, d, None, d, d, d, None, None, d, None, None, None, None)
    assert lib.mamba_scan_bwd_conv(*args(_shape(ms), w=None)) == -1
    assert b"conv_w" in lib.mamba_scan_last_error()
    assert lib.mamba_scan_bwd_conv(*args(_shape(ms), k=5)) == -1
    assert b"conv_k" in lib.mamba_scan_last_error()
    assert lib.mamba_scan_bwd_conv(*args(_shape(ms), k=0)) == -1
    assert lib.mamba_scan_bwd_conv(*args(_shape(ms, dstate=65))) == -1
    assert lib.mamba_scan_bwd_conv(*args(_shape(ms, seqlen=-1))) == -1


def test_train_checkpoint_host_argument_checks(ms):
    lib = ms.lib()
    P = ctypes.c_void_p
    d = P(256)  # never dereferenced: every case below fails validation first
    written = ctypes.c_int(7)
    fwd = lambda s, ck, y=P(1 << 40): lib.mamba_scan_fwd_train(ctypes.byref(s), 0, d, d, d, d, d, None, None, None,
                                                               1, None, y, None, ck, ctypes.byref(written), None)
    assert fwd(_shape(ms), None) == -1
    assert b"ckpt" in lib.mamba_scan_last_error() and written.value == 0
    assert fwd(_shape(ms, dstate=17), P(1 << 41)) == -1
    assert b"dstate" in lib.mamba_scan_last_error() and written.value == 0
    assert fwd(_shape(ms), P((1 << 41) + 4)) == -1
    assert b"aligned" in lib.mamba_scan_last_error()
    assert fwd(_shape(ms), P(1 << 41), y=P((1 << 41) + 64)) == -1  # ckpt overlapping y
    assert b"overlap" in lib.mamba_scan_last_error()
    bwd = lambda s, ck, du=d: lib.mamba_scan_bwd_ckpt(ctypes.byref(s), 0, d, d, d, d, d, None, None, None, 1, None,
                                                      d, None, ck, du, d, None, d, d, d, None, None, None, None)
    assert bwd(_shape(ms), P((1 << 41) + 8)) == -1
    assert b"aligned" in lib.mamba_scan_last_error()
    assert bwd(_shape(ms), P(1 << 41), du=P((1 << 41) + 32)) == -1
    assert b"overlap" in lib.mamba_scan_last_error()
    assert bwd(_shape(ms, dstate=65), P(1 << 41)) == -1


def test_train_checkpoint_bytes_host_query(ms, monkeypatch):
    """The size query runs the forward planners on the host (148 SMs when no device answers):
    checkpoints for the layer shapes, none for the million-token shape (split along L), none for
    N > 16 or L = 0."""
    lib = ms.lib()
    q = lambda **kw: (lambda n: (lib.mamba_scan_fwd_train_ckpt_bytes(ctypes.byref(_shape(ms, **kw)),
                                                                     ctypes.byref(n)), n.value))(ctypes.c_size_t(9))
    assert lib.mamba_scan_fwd_train_ckpt_bytes(ctypes.byref(_shape(ms)), None) == -1
    assert q(batch=4, dim=4096, dstate=16, seqlen=2048, in_dtype=1) == (0, 4 * 256 * 4096 * 64)
    assert q(batch=8, dim=1536, dstate=16, seqlen=2048) == (0, 8 * 256 * 1536 * 64)
    assert q(batch=1, dim=1536, dstate=16, seqlen=1 << 20) == (0, 0)
    assert q(batch=2, dim=64, dstate=17, seqlen=100) == (0, 0)
    assert q(batch=2, dim=64, dstate=16, seqlen=0) == (0, 0)
    assert q(batch=2, dim=64, dstate=16, seqlen=-1)[0] == -1
    monkeypatch.setenv("MAMBA_SCAN_NSEG", "1")  # read by the planners at every call
    assert q(batch=1, dim=1536, dstate=16, seqlen=1 << 20) == (0, 1536 * (1 << 17) * 64)


def test_plain_c_client(ms, tmp_path):
    """The header and library serve a C99 program with no Python or torch in between: version,
    the checkpoint size query at the 1.4B layer shape, an argument error and its message, and no
    kernel launched."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    inc = os.path.join(os.path.dirname(here), "include")
    libdir = os.path.dirname(ms.LIB_PATH)
    exe = str(tmp_path / "c_client")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", inc, os.path.join(here, "c_client.c"),
                    "-L", libdir, "-lmambascan", f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split("\n")
    assert out[0] == f"version {ms.lib().mamba_scan_version()} {ms.lib().mamba_scan_version()}"
    assert out[1] == f"ckpt_bytes 0 {4 * 256 * 4096 * 64}"
    assert out[2].startswith("bad_shape -1 ") and "dstate" in out[2]
    assert out[3] == "null_shape -1"
    assert out[4] == "launches 0"


def test_header_is_valid_cxx(tmp_path):
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no C++ compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    hdr = os.path.join(os.path.dirname(here), "include", "mamba_scan.h")
    subprocess.run([gxx, "-std=c++17", "-Wall", "-Werror", "-fsyntax-only", "-x", "c++", hdr], check=True)
