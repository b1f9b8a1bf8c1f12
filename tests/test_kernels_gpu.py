"""Kernel-level parity: each CUDA kernel, called through the C ABI
(include/s2_ops.h), against the oracle's operations on the same seeded
inputs.  Sizes span several CTAs/tiles and ragged tails."""

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding
    return binding


def dev(a, dt=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dt is not None:
        t = t.to(dt)
    return t.cuda()


def bf16_values(a):
    """The bf16 values a rounds to, as float64 (what the device sees)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).double().numpy()


# --------------------------------------------------------------------- K1 GEMV

GEMV_CASES = [
    # N, K, B, mode, norm
    (6144, 2560, 1, 0, True),      # S2 fused q/k/v projection with the pre-attention norm
    (2560, 4096, 1, 1, False),     # output projection + residual
    (19456, 2560, 1, 2, True),     # gate/up + SwiGLU
    (2560, 9728, 1, 1, False),     # down projection + residual
    (2560, 9728, 2, 1, False),
    (6144, 2560, 3, 0, True),
    (4096, 2560, 8, 0, True),
    (300, 264, 5, 0, False),       # ragged: rows not a multiple of the row group
    (17, 2560, 1, 0, True),        # fewer rows than SMs
    (512, 256, 8, 2, True),
]


@pytest.mark.parametrize("wdt", ["bf16", "f32"])
@pytest.mark.parametrize("N,K,B,mode,norm", GEMV_CASES)
def test_gemv_matches_oracle(b, wdt, N, K, B, mode, norm):
    rng = np.random.default_rng(N * 7 + K + B)
    W = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    X = rng.standard_normal((B, K), dtype=np.float32)
    g = rng.uniform(0.5, 1.5, K).astype(np.float32) if norm else None
    Wd = dev(W, torch.bfloat16) if wdt == "bf16" else dev(W)
    W64 = bf16_values(W) if wdt == "bf16" else W.astype(np.float64)
    out_cols = N // 2 if mode == 2 else N
    Y0 = rng.standard_normal((B, out_cols), dtype=np.float32)
    Yd = dev(Y0)
    b.s2op_gemv(Wd, N, K, dev(X), K, B, Yd, out_cols, mode=mode, gain=None if g is None else dev(g),
                w_bf16=(wdt == "bf16"))
    torch.cuda.synchronize()
    a = oracle.rms_norm(X.astype(np.float64), g.astype(np.float64), 1e-6) if norm else X.astype(np.float64)
    y = a @ W64.T
    if mode == 1:
        ref = Y0 + y
    elif mode == 2:
        ref = oracle.swiglu(y[:, 0::2], y[:, 1::2])
    else:
        ref = y
    got = Yd.cpu().numpy()
    np.testing.assert_allclose(got, ref, rtol=2e-4, atol=2e-4)


@pytest.mark.parametrize("B", [1, 3, 8])
def test_argmax_head_matches_oracle(b, B):
    N, K = 4096, 2560
    rng = np.random.default_rng(100 + B)
    W = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    X = rng.standard_normal((B, K), dtype=np.float32)
    g = np.ones(K, np.float32)
    ws = torch.zeros(b.s2op_argmax_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    codes = torch.zeros(B, dtype=torch.int32, device="cuda")
    logits = torch.zeros((B, N), dtype=torch.float32, device="cuda")
    b.s2op_gemv_argmax(dev(W, torch.bfloat16), N, K, dev(X), K, B, codes, ws, logits=logits, gain=dev(g))
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    ref = oracle.rms_norm(X.astype(np.float64), g.astype(np.float64), 1e-6) @ bf16_values(W).T
    np.testing.assert_allclose(lg, ref, rtol=1e-4, atol=1e-4)
    c = codes.cpu().numpy()
    # the pick is the arg-max of the kernel's own logits, lowest index on ties
    np.testing.assert_array_equal(c, np.argmax(lg, axis=1))
    srt = np.sort(ref, axis=1)
    clear = (srt[:, -1] - srt[:, -2]) > 1e-3
    np.testing.assert_array_equal(c[clear], np.argmax(ref, axis=1)[clear])
    assert int(ws[:4].view(torch.int32)[0].item()) == 0


def test_argmax_ties_go_to_lowest_index(b):
    N, K, B = 4096, 256, 2
    rng = np.random.default_rng(5)
    W = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    X = rng.standard_normal((B, K), dtype=np.float32)
    # rows 3001 and 99 (different CTAs) and 2048 identical, aligned with x
    xn = X[0] / np.linalg.norm(X[0])
    for r in (3001, 99, 2048):
        W[r] = xn
    ws = torch.zeros(b.s2op_argmax_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    codes = torch.zeros(B, dtype=torch.int32, device="cuda")
    b.s2op_gemv_argmax(dev(W), N, K, dev(X), K, B, codes, ws, w_bf16=False)
    torch.cuda.synchronize()
    assert codes.cpu().numpy()[0] == 99


# --------------------------------------------------------------------- K2 tcgen05 GEMM

TC_CASES = [
    # N, K, T, epi, split_k
    (128, 64, 1, 0, 0),
    (256, 256, 17, 0, 0),
    (2560, 2560, 32, 0, 0),
    (6144, 2560, 41, 0, 0),
    (2560, 4096, 64, 1, 0),
    (2560, 9728, 128, 1, 0),
    (19456, 2560, 200, 2, 0),
    (2560, 2560, 1024, 0, 0),
    (1024, 2560, 300, 1, 2),
    (512, 1024, 96, 0, 4),
    (2560, 4096, 32, 1, 7),     # splits that do not divide the 64 k-tiles
    (2560, 9728, 32, 0, 7),     # 152 k-tiles over 7 splits
]


@pytest.mark.parametrize("N,K,T,epi,split_k", TC_CASES)
def test_tc_gemm_matches_oracle(b, N, K, T, epi, split_k):
    rng = np.random.default_rng(N + 3 * K + 7 * T)
    A = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    Bm = rng.standard_normal((T, K), dtype=np.float32)
    A64, B64 = bf16_values(A), bf16_values(Bm)
    y = B64 @ A64.T                                          # [T, N]
    ws_bytes = b.s2op_tc_gemm_workspace_bytes(N, K, T, split_k)
    ws = torch.zeros(max(ws_bytes, 16) // 4, dtype=torch.float32, device="cuda")
    tk = torch.zeros(b.s2op_tc_gemm_tickets(N, T) + 4, dtype=torch.int32, device="cuda")
    Ad, Bd = dev(A, torch.bfloat16), dev(Bm, torch.bfloat16)
    if epi == 2:
        Y16 = torch.zeros((T, N // 2), dtype=torch.bfloat16, device="cuda")
        b.s2op_tc_gemm(Ad, N, K, Bd, T, K, Y16=Y16, ldy16=N // 2, epi=2, split_k=split_k,
                       workspace=ws, tickets=tk)
        torch.cuda.synchronize()
        ref = oracle.swiglu(y[:, 0::2], y[:, 1::2])
        got = Y16.double().cpu().numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-2, atol=1e-2)   # bf16 output
    else:
        Y0 = rng.standard_normal((T, N), dtype=np.float32)
        Yd = dev(Y0)
        b.s2op_tc_gemm(Ad, N, K, Bd, T, K, Y=Yd, ldy=N, epi=epi, split_k=split_k,
                       workspace=ws, tickets=tk)
        torch.cuda.synchronize()
        ref = y + (Y0 if epi == 1 else 0)
        tol = 2e-5 * np.sqrt(K) + 1e-5
        np.testing.assert_allclose(Yd.cpu().numpy(), ref, rtol=1e-4, atol=tol)
    assert int(tk.abs().sum().item()) == 0


@pytest.mark.parametrize("N,K,T,epi,two", [(2560, 4096, 32, 1, True), (2560, 9728, 32, 0, True),
                                            (6144, 2560, 32, 0, True), (4096, 2560, 32, 0, False),
                                            (19456, 2560, 17, 2, True)])
def test_tc_gemm_cluster_reduction_equals_workspace_reduction(b, N, K, T, epi, two):
    """With automatic splits the K-splits of a tile form one cluster and sum
    their partials through distributed shared memory; with the same split
    count forced explicitly they go through the global workspace.  Same
    partials, same order (split 0, 1, ...): the automatic result must equal
    one of the explicit ones bit for bit (the 32-row decode shapes: O, down,
    QKV, the head, and an unsplit gate/up)."""
    rng = np.random.default_rng(N + K + T)
    A = dev(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02), torch.bfloat16)
    X = rng.standard_normal((T, K), dtype=np.float32)
    hi = torch.from_numpy(X).to(torch.bfloat16)
    lo = (torch.from_numpy(X) - hi.float()).to(torch.bfloat16)
    Y0 = rng.standard_normal((T, N), dtype=np.float32)
    nbytes = max(b.s2op_tc_gemm2_workspace_bytes(N, K, T, s) for s in range(1, 9))
    ws = torch.zeros(max(nbytes, 16) // 4, dtype=torch.float32, device="cuda")
    tk = torch.zeros(b.s2op_tc_gemm2_tickets(N, T) + 4, dtype=torch.int32, device="cuda")

    def run(split):
        if epi == 2:
            Yh = torch.zeros((T, N // 2), dtype=torch.bfloat16, device="cuda")
            if two:
                b.s2op_tc_gemm2(A, N, K, hi.cuda(), lo.cuda(), T, K, Y16=Yh, ldy16=N // 2, epi=2,
                                split_k=split, workspace=ws, tickets=tk)
            else:
                b.s2op_tc_gemm(A, N, K, hi.cuda(), T, K, Y16=Yh, ldy16=N // 2, epi=2, split_k=split,
                               workspace=ws, tickets=tk)
            torch.cuda.synchronize()
            return Yh.float().cpu().numpy()
        Yd = dev(Y0)
        if two:
            b.s2op_tc_gemm2(A, N, K, hi.cuda(), lo.cuda(), T, K, Y=Yd, ldy=N, epi=epi, split_k=split,
                            workspace=ws, tickets=tk)
        else:
            b.s2op_tc_gemm(A, N, K, hi.cuda(), T, K, Y=Yd, ldy=N, epi=epi, split_k=split, workspace=ws,
                           tickets=tk)
        torch.cuda.synchronize()
        return Yd.cpu().numpy()

    auto = run(0)
    explicit = [run(s) for s in range(1, 9) if s <= K // 64]
    assert any(np.array_equal(auto, e) for e in explicit)
    assert int(tk.abs().sum().item()) == 0
    # and the result is right: against the fp64 product of the operands
    ref = (hi.double() + (lo.double() if two else 0)).numpy() @ A.double().cpu().numpy().T
    if epi == 2:
        np.testing.assert_allclose(auto, oracle.swiglu(ref[:, 0::2], ref[:, 1::2]), rtol=1e-2, atol=1e-2)
    else:
        np.testing.assert_allclose(auto, ref + (Y0 if epi == 1 else 0), rtol=1e-4,
                                   atol=2e-5 * np.sqrt(K) + 1e-5)


TC2_CASES = [
    (2560, 2560, 32, 0), (6144, 2560, 41, 0), (2560, 9728, 128, 1), (19456, 2560, 200, 2),
    (2560, 4096, 1024, 1), (512, 256, 7, 2),
]


@pytest.mark.parametrize("N,K,T,epi", TC2_CASES)
def test_tc_gemm_two_plane_matches_fp32_activations(b, N, K, T, epi):
    """With the activations split into bf16 hi + lo planes, the tensor-core
    product matches fp32 activations (not only their bf16 rounding)."""
    rng = np.random.default_rng(N + 5 * K + 11 * T)
    A = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    X = rng.standard_normal((T, K), dtype=np.float32)
    Xt = torch.from_numpy(X)
    hi = Xt.to(torch.bfloat16)
    lo = (Xt - hi.float()).to(torch.bfloat16)
    y = X.astype(np.float64) @ bf16_values(A).T
    ws = torch.zeros(max(b.s2op_tc_gemm2_workspace_bytes(N, K, T), 16) // 4, dtype=torch.float32,
                     device="cuda")
    tk = torch.zeros(b.s2op_tc_gemm2_tickets(N, T) + 4, dtype=torch.int32, device="cuda")
    Ad = dev(A, torch.bfloat16)
    if epi == 2:
        Yh = torch.zeros((T, N // 2), dtype=torch.bfloat16, device="cuda")
        Yl = torch.zeros((T, N // 2), dtype=torch.bfloat16, device="cuda")
        b.s2op_tc_gemm2(Ad, N, K, hi.cuda(), lo.cuda(), T, K, Y16=Yh, Y16lo=Yl, ldy16=N // 2, epi=2,
                        workspace=ws, tickets=tk)
        torch.cuda.synchronize()
        got = Yh.double().cpu().numpy() + Yl.double().cpu().numpy()
        ref = oracle.swiglu(y[:, 0::2], y[:, 1::2])
        np.testing.assert_allclose(got, ref, rtol=1e-4, atol=1e-4)
    else:
        Y0 = rng.standard_normal((T, N), dtype=np.float32)
        Yd = dev(Y0)
        b.s2op_tc_gemm2(Ad, N, K, hi.cuda(), lo.cuda(), T, K, Y=Yd, ldy=N, epi=epi, workspace=ws,
                        tickets=tk)
        torch.cuda.synchronize()
        ref = y + (Y0 if epi == 1 else 0)
        np.testing.assert_allclose(Yd.cpu().numpy(), ref, rtol=1e-4, atol=2e-5 * np.sqrt(K) + 1e-5)
    assert int(tk.abs().sum().item()) == 0


# --------------------------------------------------------------------- K3+K4 decode attention

def _rope(n, hd):
    return oracle.rope_table(n, hd, 1e6)


@pytest.mark.parametrize("H,Hkv,hd,kv_bf16", [(32, 8, 128, True), (32, 8, 128, False), (4, 2, 64, False)])
@pytest.mark.parametrize("m", [1, 2])
@pytest.mark.parametrize("nsplit", [1, 3, 16])
def test_decode_attention_matches_oracle(b, H, Hkv, hd, kv_bf16, m, nsplit):
    pos = np.array([0, 15, 16, 77, 130], np.int32)[:4 if m == 2 else 5]
    check_decode_attention(b, H, Hkv, hd, kv_bf16, m, nsplit, pos, H + hd + m * 10 + nsplit)


@pytest.mark.parametrize("m", [1, 2])
@pytest.mark.parametrize("nsplit", [3, 16])
def test_decode_attention_around_the_one_split_range(b, m, nsplit):
    """Key ranges (cached keys plus the new rows) just inside and just outside
    the range one split attends alone (64 keys): 64 keys (one split writes the
    rows), 65 (the splits' partial slots merged), 128 and 129."""
    pos = np.array([63, 64, 127, 128], np.int32) - (m - 1)
    check_decode_attention(b, 32, 8, 128, False, m, nsplit, pos, 77 + m + nsplit)


def check_decode_attention(b, H, Hkv, hd, kv_bf16, m, nsplit, pos, seed):
    rng = np.random.default_rng(seed)
    B = len(pos)
    P = 16
    n_pages = 96
    tld = 12
    perm = rng.permutation(n_pages)
    table = np.zeros((B, tld), np.int32)
    for i in range(B):
        table[i] = perm[i * tld:(i + 1) * tld]
    pool = np.zeros((n_pages, 2, Hkv, P, hd), np.float32)
    hist = []
    for i in range(B):
        K = rng.standard_normal((Hkv, pos[i], hd), dtype=np.float32)
        V = rng.standard_normal((Hkv, pos[i], hd), dtype=np.float32)
        if kv_bf16:
            K, V = bf16_values(K).astype(np.float32), bf16_values(V).astype(np.float32)
        hist.append((K, V))
        for p in range(pos[i]):
            pool[table[i, p // P], 0, :, p % P] = K[:, p]
            pool[table[i, p // P], 1, :, p % P] = V[:, p]
    qd, kvd = H * hd, Hkv * hd
    qkv = rng.standard_normal((B * m, qd + 2 * kvd), dtype=np.float32)
    qg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    kg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    cos, sin = _rope(256, hd)
    pool_d = dev(pool, torch.bfloat16) if kv_bf16 else dev(pool)
    o = torch.zeros((B * m, qd), dtype=torch.float32, device="cuda")
    wsb = b.s2op_attn_decode_workspace_bytes(B, m, H, Hkv, hd, nsplit)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    b.s2op_attn_decode(dev(qkv), qkv.shape[1], B, m, H, Hkv, hd, dev(qg), dev(kg), 1e-6, dev(cos),
                       dev(sin), dev(pos), pool_d, kv_bf16, dev(table), tld, o, qd, nsplit=nsplit,
                       workspace=ws)
    torch.cuda.synchronize()
    got = o.cpu().numpy()
    pool_after = pool_d.float().cpu().numpy()
    for i in range(B):
        rows = qkv[i * m:(i + 1) * m].astype(np.float64)
        p = pos[i] + np.arange(m)
        q = oracle.rms_norm(rows[:, :qd].reshape(m, H, hd), qg.astype(np.float64), 1e-6)
        k = oracle.rms_norm(rows[:, qd:qd + kvd].reshape(m, Hkv, hd), kg.astype(np.float64), 1e-6)
        v = rows[:, qd + kvd:].reshape(m, Hkv, hd)
        q = oracle.apply_rope(q, cos[p][:, None], sin[p][:, None])
        k = oracle.apply_rope(k, cos[p][:, None], sin[p][:, None])
        Kall = np.concatenate([hist[i][0].astype(np.float64), k.transpose(1, 0, 2)], axis=1)
        Vall = np.concatenate([hist[i][1].astype(np.float64), v.transpose(1, 0, 2)], axis=1)
        ref = oracle.gqa_attention(q, Kall, Vall, p).reshape(m, qd)
        np.testing.assert_allclose(got[i * m:(i + 1) * m], ref, rtol=2e-4, atol=2e-4)
        for j in range(m):
            pp = p[j]
            stored_k = pool_after[table[i, pp // P], 0, :, pp % P]
            stored_v = pool_after[table[i, pp // P], 1, :, pp % P]
            tol = 8e-3 if kv_bf16 else 1e-5
            np.testing.assert_allclose(stored_k, k[j], rtol=tol, atol=tol)
            np.testing.assert_allclose(stored_v, v[j], rtol=tol, atol=tol)
    # untouched pages stay untouched
    used = set()
    for i in range(B):
        for p in range(pos[i] + m):
            used.add((table[i, p // P], p % P))
    for pg in range(n_pages):
        for s in range(P):
            if (pg, s) not in used:
                assert not pool_after[pg, :, :, s].any()
    assert int(ws.sum().item()) == 0 or nsplit > 1  # tickets reset (partials may remain)


# Split counts the runtime picks (CTAs for twice the 152 SMs, at most 16
# splits): 16 at batch 1, 2 at batch 32, 1 at batch 128.
@pytest.mark.parametrize("kv_bf16", [False, True])
@pytest.mark.parametrize("nsplit", [16, 2, 1])
def test_decode_attention_long_context_matches_oracle(b, kv_bf16, nsplit):
    """1,000 / 1,699 / 1,700 cached keys (1,001, 1,700 and 1,701 with the new
    row): the batch-128 workload's contexts reach ~1,700 keys.  Pages are
    scattered over a pool; every output row is compared with the oracle's
    attention over the full key list in float64."""
    H, Hkv, hd, m = 32, 8, 128, 1
    rng = np.random.default_rng(4242 + nsplit + 7 * kv_bf16)
    pos = np.array([1000, 1699, 1700], np.int32)
    B, P = len(pos), 16
    tld = (int(pos.max()) + m + P - 1) // P
    n_pages = B * tld + 5
    table = rng.permutation(n_pages)[:B * tld].astype(np.int32).reshape(B, tld)
    pool = np.zeros((n_pages, 2, Hkv, P, hd), np.float32)
    hist = []
    for i in range(B):
        K = rng.standard_normal((Hkv, pos[i], hd), dtype=np.float32)
        V = rng.standard_normal((Hkv, pos[i], hd), dtype=np.float32)
        if kv_bf16:
            K, V = bf16_values(K).astype(np.float32), bf16_values(V).astype(np.float32)
        hist.append((K, V))
        pg = table[i, np.arange(pos[i]) // P]
        sl = np.arange(pos[i]) % P
        pool[pg, 0, :, sl] = K.transpose(1, 0, 2)
        pool[pg, 1, :, sl] = V.transpose(1, 0, 2)
    qd, kvd = H * hd, Hkv * hd
    qkv = rng.standard_normal((B * m, qd + 2 * kvd), dtype=np.float32)
    qg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    kg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    cos, sin = _rope(1800, hd)
    pool_d = dev(pool, torch.bfloat16) if kv_bf16 else dev(pool)
    o = torch.zeros((B * m, qd), dtype=torch.float32, device="cuda")
    ws = torch.zeros(b.s2op_attn_decode_workspace_bytes(B, m, H, Hkv, hd, nsplit), dtype=torch.uint8,
                     device="cuda")
    b.s2op_attn_decode(dev(qkv), qkv.shape[1], B, m, H, Hkv, hd, dev(qg), dev(kg), 1e-6, dev(cos),
                       dev(sin), dev(pos), pool_d, kv_bf16, dev(table), tld, o, qd, nsplit=nsplit,
                       workspace=ws)
    torch.cuda.synchronize()
    got = o.cpu().numpy()
    for i in range(B):
        row = qkv[i].astype(np.float64)
        p = pos[i] + np.arange(m)
        q = oracle.rms_norm(row[None, :qd].reshape(m, H, hd), qg.astype(np.float64), 1e-6)
        k = oracle.rms_norm(row[None, qd:qd + kvd].reshape(m, Hkv, hd), kg.astype(np.float64), 1e-6)
        v = row[None, qd + kvd:].reshape(m, Hkv, hd)
        q = oracle.apply_rope(q, cos[p][:, None], sin[p][:, None])
        k = oracle.apply_rope(k, cos[p][:, None], sin[p][:, None])
        Kall = np.concatenate([hist[i][0].astype(np.float64), k.transpose(1, 0, 2)], axis=1)
        Vall = np.concatenate([hist[i][1].astype(np.float64), v.transpose(1, 0, 2)], axis=1)
        ref = oracle.gqa_attention(q, Kall, Vall, p).reshape(m, qd)
        np.testing.assert_allclose(got[i * m:(i + 1) * m], ref, rtol=2e-4, atol=2e-4)


# ------------------------------------------------- K11 shared-prefix attention

@pytest.mark.parametrize("B,P,nsplit,kv_bf16", [(32, 896, 2, False), (32, 896, 2, True), (5, 80, 1, False),
                                                (17, 64, 3, False), (40, 128, 1, False), (32, 896, 1, False),
                                                (3, 16, 2, False), (32, 1152, 2, False), (9, 2048, 4, True),
                                                (33, 1040, 2, False)])
def test_shared_prefix_attention_matches_oracle(b, B, P, nsplit, kv_bf16):
    """B sequences whose tables begin with the same P keys (shared pages)
    followed by private pages of different lengths: the split-KV attention
    over the private keys plus the tensor-core prefix attention (clusters of
    8 CTAs, 128-key chunks) give the oracle's attention over each sequence's
    full key list.  Cases: the batch-32 workload's 896 shared keys (7 of the
    8 CTAs busy; one private split, so the split-KV launch must still leave
    a partial); a ragged last chunk (80, 1,040 keys); one 16-key chunk; more
    chunks than CTAs (1,152 and 2,048 keys: the CTA's chunks combined in
    registers); 40 and 33 sequences = two 128-row query tiles, the second
    ragged."""
    H, Hkv, hd, Pg = 32, 8, 128, 16
    rng = np.random.default_rng(B * 1000 + P + nsplit + 7 * kv_bf16)
    priv = rng.integers(1, 200, B)                   # private cached keys per sequence
    pos = (P + priv).astype(np.int32)                # the new row's position
    tld = (int(pos.max()) + 1 + Pg - 1) // Pg
    n_shared = P // Pg
    n_pages = n_shared + B * (tld - n_shared) + 3
    perm = rng.permutation(n_pages)
    table = np.zeros((B, tld), np.int32)
    table[:, :n_shared] = perm[:n_shared]
    for i in range(B):
        table[i, n_shared:] = perm[n_shared + i * (tld - n_shared): n_shared + (i + 1) * (tld - n_shared)]
    pool = np.zeros((n_pages, 2, Hkv, Pg, hd), np.float32)
    Ks = rng.standard_normal((Hkv, P, hd), dtype=np.float32)
    Vs = rng.standard_normal((Hkv, P, hd), dtype=np.float32)
    if kv_bf16:
        Ks, Vs = bf16_values(Ks).astype(np.float32), bf16_values(Vs).astype(np.float32)
    hist = []
    for i in range(B):
        Kp = rng.standard_normal((Hkv, priv[i], hd), dtype=np.float32)
        Vp = rng.standard_normal((Hkv, priv[i], hd), dtype=np.float32)
        if kv_bf16:
            Kp, Vp = bf16_values(Kp).astype(np.float32), bf16_values(Vp).astype(np.float32)
        K = np.concatenate([Ks, Kp], axis=1)
        V = np.concatenate([Vs, Vp], axis=1)
        hist.append((K, V))
        pg = table[i, np.arange(pos[i]) // Pg]
        sl = np.arange(pos[i]) % Pg
        pool[pg, 0, :, sl] = K.transpose(1, 0, 2)
        pool[pg, 1, :, sl] = V.transpose(1, 0, 2)
    qd, kvd = H * hd, Hkv * hd
    qkv = rng.standard_normal((B, qd + 2 * kvd), dtype=np.float32)
    qg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    kg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    max_keys = int(pos.max()) + 1
    cos, sin = _rope(max_keys, hd)
    pool_d = dev(pool, torch.bfloat16) if kv_bf16 else dev(pool)
    o = torch.zeros((B, qd), dtype=torch.float32, device="cuda")
    ws = torch.zeros(b.s2op_attn_decode_prefix_workspace_bytes(B, H, Hkv, hd, nsplit, max_keys),
                     dtype=torch.uint8, device="cuda")
    b.s2op_attn_prefix_planes(pool_d, kv_bf16, dev(table), Hkv, hd, P, max_keys, ws)
    b.s2op_attn_decode_shared_prefix(dev(qkv), qkv.shape[1], B, H, Hkv, hd, dev(qg), dev(kg), 1e-6,
                                     dev(cos), dev(sin), dev(pos), pool_d, kv_bf16, dev(table), tld, P,
                                     max_keys, o, qd, nsplit=nsplit, workspace=ws)
    torch.cuda.synchronize()
    got = o.cpu().numpy()
    for i in range(B):
        row = qkv[i].astype(np.float64)
        p_ = pos[i] + np.arange(1)
        q = oracle.rms_norm(row[None, :qd].reshape(1, H, hd), qg.astype(np.float64), 1e-6)
        k = oracle.rms_norm(row[None, qd:qd + kvd].reshape(1, Hkv, hd), kg.astype(np.float64), 1e-6)
        v = row[None, qd + kvd:].reshape(1, Hkv, hd)
        q = oracle.apply_rope(q, cos[p_][:, None], sin[p_][:, None])
        k = oracle.apply_rope(k, cos[p_][:, None], sin[p_][:, None])
        Kall = np.concatenate([hist[i][0].astype(np.float64), k.transpose(1, 0, 2)], axis=1)
        Vall = np.concatenate([hist[i][1].astype(np.float64), v.transpose(1, 0, 2)], axis=1)
        ref = oracle.gqa_attention(q, Kall, Vall, p_).reshape(qd)
        np.testing.assert_allclose(got[i], ref, rtol=2e-4, atol=2e-4, err_msg=f"sequence {i}")
    # the new rows' keys were appended to the private pages, the shared pages untouched
    after = pool_d.float().cpu().numpy()
    np.testing.assert_array_equal(after[perm[:n_shared]], pool[perm[:n_shared]])
    # again on the same workspace (tickets back at zero, same partial order):
    # the same outputs bit for bit; the appended keys are rewritten with the
    # same values, so the pool is restored first only for clarity
    pool_d.copy_(dev(pool, torch.bfloat16) if kv_bf16 else dev(pool))
    o2 = torch.zeros_like(o)
    b.s2op_attn_decode_shared_prefix(dev(qkv), qkv.shape[1], B, H, Hkv, hd, dev(qg), dev(kg), 1e-6,
                                     dev(cos), dev(sin), dev(pos), pool_d, kv_bf16, dev(table), tld, P,
                                     max_keys, o2, qd, nsplit=nsplit, workspace=ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o2.cpu().numpy(), got)


# --------------------------------------------------------------------- K9 prefill attention

@pytest.mark.parametrize("H,Hkv,hd,kv_bf16,T,pos0", [
    (32, 8, 128, True, 70, 32),     # suffix after a cached 2-page prefix
    (32, 8, 128, True, 130, 0),     # cold, ragged last query tile
    (4, 2, 64, False, 16, 0),       # tiny model
    (8, 2, 128, False, 45, 96),
    (32, 8, 128, False, 44, 896),   # a batch-32 suffix over the 896 radix-cached keys
    (32, 8, 128, False, 1024, 0),   # the voice-clone prompt: 16 key chunks per query tile
    (32, 8, 128, True, 600, 64),    # long suffix after 4 cached pages, ragged last tile
])
def test_prefill_attention_matches_oracle(b, H, Hkv, hd, kv_bf16, T, pos0):
    """Prompts long enough to cover the SMs with 32-token tiles (hd 128, 4
    heads per kv head: 1,024 and 600 rows) run the tcgen05 kernel, the others
    the CUDA-core one; both against the oracle's causal attention."""
    rng = np.random.default_rng(T + pos0 + hd)
    P = 16
    n_pages = max(40, -(-(pos0 + T) // P) + 8)
    npg = -(-(pos0 + T) // P)
    table = rng.permutation(n_pages)[:npg].astype(np.int32)
    pool = np.zeros((n_pages, 2, Hkv, P, hd), np.float32)
    K0 = rng.standard_normal((Hkv, pos0, hd), dtype=np.float32)
    V0 = rng.standard_normal((Hkv, pos0, hd), dtype=np.float32)
    if kv_bf16:
        K0, V0 = bf16_values(K0).astype(np.float32), bf16_values(V0).astype(np.float32)
    for p in range(pos0):
        pool[table[p // P], 0, :, p % P] = K0[:, p]
        pool[table[p // P], 1, :, p % P] = V0[:, p]
    qd, kvd = H * hd, Hkv * hd
    qkv = rng.standard_normal((T, qd + 2 * kvd), dtype=np.float32)
    qg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    kg = rng.uniform(0.5, 1.5, hd).astype(np.float32)
    cos, sin = _rope(max(512, pos0 + T), hd)
    pool_d = dev(pool, torch.bfloat16) if kv_bf16 else dev(pool)
    qs = torch.zeros((T, qd), dtype=torch.float32, device="cuda")
    o = torch.zeros((T, qd), dtype=torch.float32, device="cuda")
    b.s2op_attn_prefill(dev(qkv), qkv.shape[1], T, pos0, H, Hkv, hd, dev(qg), dev(kg), 1e-6, dev(cos),
                        dev(sin), pool_d, kv_bf16, dev(table), qs, o, qd)
    torch.cuda.synchronize()
    rows = qkv.astype(np.float64)
    p = pos0 + np.arange(T)
    q = oracle.rms_norm(rows[:, :qd].reshape(T, H, hd), qg.astype(np.float64), 1e-6)
    k = oracle.rms_norm(rows[:, qd:qd + kvd].reshape(T, Hkv, hd), kg.astype(np.float64), 1e-6)
    v = rows[:, qd + kvd:].reshape(T, Hkv, hd)
    q = oracle.apply_rope(q, cos[p][:, None], sin[p][:, None])
    k = oracle.apply_rope(k, cos[p][:, None], sin[p][:, None])
    kn, vn = k.transpose(1, 0, 2), v.transpose(1, 0, 2)
    if kv_bf16:   # new keys/values are read back from the bf16 pages
        kn, vn = bf16_values(kn), bf16_values(vn)
    Kall = np.concatenate([K0.astype(np.float64), kn], axis=1)
    Vall = np.concatenate([V0.astype(np.float64), vn], axis=1)
    ref = oracle.gqa_attention(q, Kall, Vall, p).reshape(T, qd)
    tol = 3e-3 if kv_bf16 else 2e-4
    np.testing.assert_allclose(o.cpu().numpy(), ref, rtol=tol, atol=tol)


# ----------------------------------------------------------- read calibration

@pytest.mark.parametrize("mode,barrier", [(0, 0), (1, 0), (1, 1)])
def test_stream_read_calibration_runs_clean(b, mode, barrier):
    """The calibration streams (plain loads; the bulk-copy ring with and
    without the consumers' grid barrier) read a ragged list of buffers,
    including ones smaller than one chunk per CTA, without a failed wait."""
    sizes = [16, 4096 * 16 + 48, 3 << 20, (37 << 20) + 160, 1 << 16]
    bufs = [torch.zeros(n // 2, dtype=torch.bfloat16, device="cuda") for n in sizes]
    scratch = torch.zeros(b.s2op_stream_read_scratch_bytes(len(bufs)), dtype=torch.uint8, device="cuda")
    for reps, chunk, stages in [(1, 16384, 12), (3, 8192, 24), (2, 1024, 2)]:
        err = b.s2op_stream_read(bufs, sizes, scratch, reps=reps, mode=mode, chunk_bytes=chunk,
                                 stages=stages, barrier=barrier)
        torch.cuda.synchronize()
        assert err == 0
    with pytest.raises(b.S2Error):
        b.s2op_stream_read(bufs, sizes, scratch, mode=1, chunk_bytes=65536, stages=4)   # > 200 KB ring
