"""The allocation-free decode attention entry point.

Some callers cannot allocate device memory: a real-time audio thread (an
allocation may block on the driver or synchronise the device mid-frame) or a
host whose device memory belongs to another allocator.  For them the library
offers s2op_attn_decode_noalloc, which keeps its scratch in a fixed array
inside the library.  This file checks it through the C ABI against the
workspace-taking entry point, on two calls in a row (the shared array keeps
the previous call's contents).  It is named to run after every other test
file, and it also passes on its own in a fresh process.
"""

import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding
    L = binding.LIB
    vp, i32, f32 = C.c_void_p, C.c_int32, C.c_float
    L.s2op_attn_decode_noalloc.restype = i32
    L.s2op_attn_decode_noalloc.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, f32, vp, vp,
                                          vp, vp, i32, vp, i32, vp, i32, i32, vp]
    L.s2op_attn_decode_noalloc_max_bytes.restype = C.c_size_t
    L.s2op_attn_decode_noalloc_max_bytes.argtypes = []
    return binding


def _inputs(B=5, H=32, Hkv=8, hd=128, seed=7):
    rng = np.random.default_rng(seed)
    pos = np.array([3, 16, 40, 95, 130][:B], np.int32)
    P, n_pages, tld = 16, 64, 12
    perm = rng.permutation(n_pages)
    table = np.stack([perm[i * tld:(i + 1) * tld] for i in range(B)]).astype(np.int32)
    pool = rng.standard_normal((n_pages, 2, Hkv, P, hd), dtype=np.float32)
    qkv = rng.standard_normal((B, (H + 2 * Hkv) * hd), dtype=np.float32)
    qg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    kg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    cos, sin = oracle.rope_table(256, hd, 1e6)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    return dict(B=B, H=H, Hkv=Hkv, hd=hd, pos=d(pos), table=d(table), tld=tld,
                pool=d(pool).to(torch.bfloat16), qkv=d(qkv), qg=d(qg), kg=d(kg),
                cos=d(cos), sin=d(sin))


def _call_noalloc(lib, x, o, nsplit, B=None):
    B = x["B"] if B is None else B
    p = lib.ptr
    return lib.LIB.s2op_attn_decode_noalloc(
        p(x["qkv"]), x["qkv"].shape[1], B, 1, x["H"], x["Hkv"], x["hd"], p(x["qg"]), p(x["kg"]),
        1e-6, p(x["cos"]), p(x["sin"]), p(x["pos"]), p(x["pool"]), 1, p(x["table"]), x["tld"],
        p(o), o.shape[1], nsplit, None)


@pytest.mark.parametrize("nsplit", [1, 4, 16])
def test_noalloc_matches_workspace_entry_point_twice(lib, nsplit):
    x = _inputs()
    qd = x["H"] * x["hd"]
    ref = torch.zeros((x["B"], qd), dtype=torch.float32, device="cuda")
    ws = torch.zeros(lib.s2op_attn_decode_workspace_bytes(x["B"], 1, x["H"], x["Hkv"], x["hd"], nsplit),
                     dtype=torch.uint8, device="cuda")
    lib.s2op_attn_decode(x["qkv"], x["qkv"].shape[1], x["B"], 1, x["H"], x["Hkv"], x["hd"], x["qg"],
                         x["kg"], 1e-6, x["cos"], x["sin"], x["pos"], x["pool"], 1, x["table"],
                         x["tld"], ref, qd, nsplit=nsplit, workspace=ws)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full((x["B"], qd), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_noalloc(lib, x, out, nsplit) == 0
        torch.cuda.synchronize()
        # same kernel, same split order, same merge: bit-identical results,
        # so a wrong scratch or ticket offset cannot hide in a tolerance
        assert torch.equal(out, ref)


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    x = _inputs()
    limit = lib.LIB.s2op_attn_decode_noalloc_max_bytes()
    assert limit == 8 << 20
    out = torch.zeros((x["B"], x["H"] * x["hd"]), dtype=torch.float32, device="cuda")
    # 5 sequences x 32 heads x 130 floats x 4 B = 83 KB per split: 128 splits exceed 8 MiB
    assert _call_noalloc(lib, x, out, 128) == lib.S2_EINVAL
