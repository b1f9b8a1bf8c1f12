"""The C ABI library loads and exports what include/*.h declares (no GPU)."""

import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding
    return binding


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(inc, f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(s2\w*)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_the_boundary():
    names = declared_functions()
    for n in ("s2_create", "s2_prefill", "s2_decode_frames", "s2_destroy", "s2_release",
              "s2_stats", "s2_strerror"):
        assert n in names, n
    assert len(names) >= 15


def test_library_exports_every_declared_symbol(lib):
    import ctypes
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_status_names(lib):
    assert lib.strerror(0) == "ok"
    assert "invalid" in lib.strerror(lib.S2_EINVAL)
    assert "KV" in lib.strerror(lib.S2_ENOMEM)
    assert lib.strerror(12345) == "unknown status"


def test_argument_validation_before_any_device_call(lib):
    L = lib.LIB
    assert L.s2op_gemv(None, 1, 10, 8, None, 8, 1, None, 1e-6, None, 10, 0, 0, None) == lib.S2_EINVAL
    assert L.s2op_gemv(1, 1, 10, 8, 1, 8, 9, None, 1e-6, 1, 10, 0, 0, None) == lib.S2_EINVAL  # B > 8
    assert L.s2_prefill(None, 0, None, 4, None, None, None) == lib.S2_EINVAL
    assert L.s2_decode_frames(None, None, 1, 1, None) == lib.S2_EINVAL
    import ctypes
    h = ctypes.c_void_p()
    assert L.s2_create(b"/nonexistent/weights.s2w", None, ctypes.byref(h)) == lib.S2_EBADFILE


def test_bad_weight_file_is_rejected(lib, tmp_path):
    import ctypes
    p = tmp_path / "bad.s2w"
    p.write_bytes(b"NOTDUALAR" + b"\0" * 200)
    h = ctypes.c_void_p()
    assert lib.LIB.s2_create(str(p).encode(), None, ctypes.byref(h)) == lib.S2_EBADFILE


def _create_status(lib, path):
    import ctypes
    h = ctypes.c_void_p()
    st = lib.LIB.s2_create(str(path).encode(), None, ctypes.byref(h))
    if st == 0:                      # a GPU machine loaded it: let go of it
        lib.LIB.s2_destroy(h)
    return st


# (field, byte offset, struct format, value): one header field changed per case
_HEADER_FAULTS = [
    ("magic", 0, "<8s", b"S2DUALAX"),
    ("version", 8, "<I", 2),
    ("weight dtype", 12, "<I", 7),
    ("kv heads not dividing q heads", 16 + 2 * 4, "<i", 3),
    ("head dim without a kernel (32, group 2)", 16 + 3 * 4, "<i", 32),
    ("d not a multiple of 8", 16 + 0 * 4, "<i", 252),
    ("codebooks != 10", 16 + 9 * 4, "<i", 9),
    ("semantic range not ending at the vocabulary", 16 + 8 * 4, "<i", 447),
    ("no tensors", 68, "<I", 0),
    ("absurd tensor count", 68, "<I", 200000),
]


@pytest.mark.parametrize("field,off,fmt,val", _HEADER_FAULTS, ids=[f[0] for f in _HEADER_FAULTS])
def test_malformed_header_is_rejected_before_any_device_work(lib, tiny_path, tmp_path, field, off, fmt,
                                                              val):
    """The loader checks the header on the host first; every malformed field
    gives S2_EBADFILE (no crash, no device call needed to find out)."""
    import struct
    raw = bytearray(open(tiny_path, "rb").read(4096))
    struct.pack_into(fmt, raw, off, val)
    p = tmp_path / "bad.s2w"
    p.write_bytes(bytes(raw))
    assert _create_status(lib, p) == lib.S2_EBADFILE, field


@pytest.mark.parametrize("keep", [0, 100, 128 + 64])
def test_truncated_file_is_rejected(lib, tiny_path, tmp_path, keep):
    p = tmp_path / "short.s2w"
    p.write_bytes(open(tiny_path, "rb").read(keep))
    assert _create_status(lib, p) == lib.S2_EBADFILE


def test_intact_header_passes_the_host_checks(lib, tiny_path):
    """Control for the cases above: the unmodified file is not rejected as a
    bad file (without a GPU the next step, creating a stream, fails instead)."""
    assert _create_status(lib, tiny_path) != lib.S2_EBADFILE


def test_rope_table_matches_oracle_bit_for_bit(lib):
    """The library's host-side RoPE table equals the oracle's bf16 table."""
    import oracle
    for hd, theta in ((128, 1e6), (64, 1e6)):
        cs, sn = lib.s2op_rope_table(1800, hd, theta)
        oc, osn = oracle.rope_table(1800, hd, theta)
        np.testing.assert_array_equal(cs, oc)
        np.testing.assert_array_equal(sn, osn)


def test_workspace_size_queries(lib):
    assert lib.s2op_argmax_workspace_bytes(8) >= 8 * 152 * 8
    assert lib.s2op_attn_decode_workspace_bytes(4, 1, 32, 8, 128, 16) >= 4 * 32 * 16 * 130 * 4
    assert lib.s2op_tc_gemm_tickets(2560, 1024) == 20 * 4


def test_vocoder_host_side_refusals(tmp_path):
    """The vocoder entry points refuse bad arguments and malformed files on
    the host (no GPU needed): a well-formed file parses and only then fails
    at the first device allocation (ECUDA here, with no device)."""
    import ctypes as C
    from serving_dual_ar_gb300 import binding as b
    from s2_inputs.vocoder import DAC_MICRO, ensure_vocoder
    h = C.c_void_p()
    assert b.LIB.s2_vocoder_create(b"/nonexistent.s2v", 1, 1, None, C.byref(h)) == b.S2_EBADFILE
    path = ensure_vocoder(DAC_MICRO, str(tmp_path))
    assert b.LIB.s2_vocoder_create(path.encode(), 0, 1, None, C.byref(h)) == b.S2_EINVAL
    assert b.LIB.s2_vocoder_create(path.encode(), 1, 0, None, C.byref(h)) == b.S2_EINVAL
    assert b.LIB.s2_vocoder_create(path.encode(), 1, 1, None, None) == b.S2_EINVAL
    bad = tmp_path / "bad.s2v"
    raw = bytearray(open(path, "rb").read())
    raw[0:8] = b"NOTAVOCO"
    bad.write_bytes(bytes(raw))
    assert b.LIB.s2_vocoder_create(str(bad).encode(), 1, 1, None, C.byref(h)) == b.S2_EBADFILE
    trunc = tmp_path / "trunc.s2v"
    trunc.write_bytes(open(path, "rb").read()[:-4096])
    assert b.LIB.s2_vocoder_create(str(trunc).encode(), 1, 1, None, C.byref(h)) == b.S2_EBADFILE
    st = b.LIB.s2_vocoder_create(path.encode(), 1, 1, None, C.byref(h))
    assert st in (b.S2_ECUDA, b.S2_ENOMEM) and not h.value
    assert b.LIB.s2_vocoder_decode(None, None, 1, 1, None) == b.S2_EINVAL
    assert b.LIB.s2_vocoder_hop(None) == 0
    assert b.LIB.s2_vocoder_read_stage(None, 0, None, 0) == b.S2_EINVAL
