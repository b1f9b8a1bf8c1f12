"""The tensor-core GEMM's launch planner, called in the library on the CPU.

The planner is host code: the token-column tile width from the row count, and
the K split -- the most splits whose CTAs still fit one wave (one CTA per SM)
while every split keeps at least 4 of the 64-wide k-tiles.  It is reached
through its exported C++ symbol (Itanium mangling, as gcc emits on x86-64 and
aarch64)."""
import ctypes

import pytest

BM, BK = 128, 64


@pytest.fixture(scope="module")
def plan():
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding
    f = getattr(binding.LIB, "_ZN2s212tc_gemm_planEiiiiPiS0_b")
    f.restype = None
    f.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_int)] * 2 + [ctypes.c_bool]
    ws = getattr(binding.LIB, "_ZN2s217tc_gemm_ws_floatsEiiib")
    ws.restype = ctypes.c_size_t
    ws.argtypes = [ctypes.c_int] * 3 + [ctypes.c_bool]

    def call(N, K, T, sms=152, two=False):
        tn, sk = ctypes.c_int(), ctypes.c_int()
        f(N, K, T, sms, ctypes.byref(tn), ctypes.byref(sk), two)
        return tn.value, sk.value

    call.ws_floats = lambda N, T, sk, two=False: ws(N, T, sk, two)
    return call


def test_s2_projection_plans_at_32_rows(plan):
    # (N, K) of the S2 projections; grid = row tiles x column tiles x splits
    assert plan(6144, 2560, 32) == (32, 3)      # 48 tiles x 3 = 144 CTAs
    assert plan(2560, 4096, 32) == (32, 7)      # 20 x 7 = 140
    assert plan(19456, 2560, 32) == (32, 1)     # 152 tiles fill the SMs alone
    assert plan(2560, 9728, 32) == (32, 7)      # 20 x 7 = 140


@pytest.mark.parametrize("T,two,tn", [(1, False, 32), (32, False, 32), (33, False, 64), (64, False, 64),
                                      (65, False, 128), (128, False, 128), (129, False, 256),
                                      (940, False, 256), (940, True, 128)])
def test_column_tile_width(plan, T, two, tn):
    assert plan(2560, 2560, T, two=two)[0] == tn


@pytest.mark.parametrize("N", [128, 2560, 6144, 19456])
@pytest.mark.parametrize("K", [256, 1024, 2560, 4096, 9728])
@pytest.mark.parametrize("T", [1, 32, 64, 200, 940])
@pytest.mark.parametrize("sms", [148, 152])
def test_split_is_the_largest_that_fits_one_wave(plan, N, K, T, sms):
    tn, s = plan(N, K, T, sms)
    tiles = (N // BM) * -(-T // tn)
    kt = K // BK
    assert s >= 1
    if s > 1:
        assert tiles * s <= sms and kt // s >= 4
    # one more split would break a rule
    assert tiles * (s + 1) > sms or kt // (s + 1) < 4 or s + 1 > kt // 4
    # the split-K workspace holds one fp32 partial tile per split, none unsplit
    want = s * tiles * tn * BM if s > 1 else 0
    assert plan.ws_floats(N, T, s) == want
