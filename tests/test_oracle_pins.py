"""Pins of the oracle against things other than itself (CPU only).

Each test checks the oracle against a number printed on the pages, a closed
form, a mathematical invariant, brute-force recomputation, or an independent
library routine (PyTorch CPU, SciPy), so that a dropped term, a wrong sign or
index or a transposed operand in the oracle fails one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import (DualAROracle, OracleWeights, rms_norm, rope_table,
                    apply_rope, softmax, gqa_attention, silu, bf16_round,
                    embed_prompt, feedback_embedding)
from s2_inputs import (S2, TINY, MICRO, param_counts, make_workload,
                       random_prompt, WeightFile)

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "page_numbers.json")))


# ---------------------------------------------------------------- page numbers

def test_param_counts_match_pages():
    """Shapes of the S2 model against the pages' parameter figures."""
    c = param_counts(S2)
    assert c["layer"] == 100_925_440
    time_axis = c["slow_layers"] + c["tok_emb"]
    depth_axis = c["fast_layers"]
    g = GOLDEN["params_time_axis"]
    assert abs(time_axis / g["value"] - 1) < g["rel_tol"], time_axis
    g = GOLDEN["params_depth_axis"]
    assert abs(depth_axis / g["value"] - 1) < g["rel_tol"], depth_axis
    # read per frame at batch 1: slow stack + the full tied head + 9 fast
    # passes, each reading the 4 fast layers and one head slice
    per_frame = (c["slow_layers"] + c["tok_emb"]
                 + 9 * (c["fast_layers"] + c["fast_head_slice"]))
    g = GOLDEN["params_read_per_frame_batch1"]
    assert abs(per_frame / g["value"] - 1) < g["rel_tol"], per_frame
    # 10 passes instead of 9 would miss the printed figure by > 5%
    wrong = per_frame + c["fast_layers"] + c["fast_head_slice"]
    assert abs(wrong / g["value"] - 1) > 0.04
    assert S2.n_slow == GOLDEN["slow_layers"]["value"]
    assert S2.n_fast == GOLDEN["fast_layers"]["value"]
    assert S2.n_codebooks == GOLDEN["codebooks"]["value"]
    assert S2.n_codebooks - 1 == GOLDEN["residual_codes_per_frame"]["value"]


def test_frame_rate_arithmetic():
    spf = GOLDEN["samples_per_frame"]["value"]
    sr = GOLDEN["sample_rate_hz"]["value"]
    ms = 1000.0 * spf / sr
    assert abs(ms - GOLDEN["frame_ms"]["value"]) < GOLDEN["frame_ms"]["abs_tol"]
    hz = sr / spf
    assert abs(hz - GOLDEN["frame_rate_hz"]["value"]) < GOLDEN["frame_rate_hz"]["abs_tol"]
    # tok/s x RTF = audio frames per second of audio: 63.3 * 0.34 ~ 21.5 Hz,
    # so the page's "tok/s" counts frames
    g = GOLDEN["h200_rtf_and_tok_s"]
    assert abs(g["tok_s"] * g["rtf"] - hz) < 0.2


# ------------------------------------------------------------- elementary ops

def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000) * 10 ** rng.uniform(-8, 8, 10000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 3.0e38]])
    x = x.astype(np.float32)
    # exact ties: the halfway points between consecutive bf16 values
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32) * np.float32(1.0)
    x = np.concatenate([x, ties, -ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(bf16_round(x), ref)


def test_rope_table_is_bf16_of_cos_sin():
    cos, sin = rope_table(300, 128, 1e6)
    i = torch.arange(64, dtype=torch.float64)
    ang = torch.arange(300, dtype=torch.float64)[:, None] * (1e6 ** (-2 * i / 128))[None, :]
    ref_c = torch.cos(ang).to(torch.float32).to(torch.bfloat16).to(torch.float32).numpy()
    ref_s = torch.sin(ang).to(torch.float32).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(cos, ref_c)
    np.testing.assert_array_equal(sin, ref_s)


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(1)
    hd = 64
    cos, sin = rope_table(64, hd, 1e6, to_bf16=False)
    x = rng.standard_normal((hd,))
    # position 0 is the identity
    np.testing.assert_allclose(apply_rope(x, cos[0], sin[0]), x, atol=1e-15)
    # a rotation preserves the norm
    for p in (1, 7, 63):
        assert abs(np.linalg.norm(apply_rope(x, cos[p], sin[p])) - np.linalg.norm(x)) < 1e-12
    # q(p) . k(r) depends only on p - r
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    d1 = apply_rope(q, cos[10], sin[10]) @ apply_rope(k, cos[3], sin[3])
    d2 = apply_rope(q, cos[40], sin[40]) @ apply_rope(k, cos[33], sin[33])
    assert abs(d1 - d2) < 1e-12
    # the bf16 table keeps the norm to within its rounding
    cb, sb = rope_table(64, hd, 1e6)
    for p in (5, 50):
        r = np.linalg.norm(apply_rope(x, cb[p], sb[p])) / np.linalg.norm(x)
        assert abs(r - 1) < 2 ** -7


def test_rope_matches_complex_rotation():
    """Rotate-half RoPE equals multiplying z_i = x_i + i x_{i+hd/2} by e^{i a}."""
    rng = np.random.default_rng(2)
    hd = 32
    cos, sin = rope_table(20, hd, 1e4, to_bf16=False)
    i = np.arange(hd // 2)
    x = rng.standard_normal((5, hd))
    p = 17
    z = (x[:, :hd // 2] + 1j * x[:, hd // 2:]) * np.exp(1j * p * 1e4 ** (-2.0 * i / hd))
    ref = np.concatenate([z.real, z.imag], axis=-1)
    np.testing.assert_allclose(apply_rope(x, cos[p], sin[p]), ref, atol=1e-12)


def test_rms_norm_matches_torch_and_constant_case():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 96))
    g = rng.standard_normal(96)
    ref = F.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(rms_norm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-12)
    # a constant vector c*1 normalises to sign(c) * g (up to eps)
    for c in (3.5, -0.25):
        y = rms_norm(np.full(96, c), g, 1e-6)
        np.testing.assert_allclose(y, np.sign(c) * g, rtol=1e-5)


def test_softmax_rows_sum_to_one_and_match_scipy():
    from scipy.special import softmax as sp_softmax
    rng = np.random.default_rng(4)
    s = rng.standard_normal((9, 33)).astype(np.float32) * 20
    p = softmax(s)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-6)
    np.testing.assert_allclose(p, sp_softmax(s, axis=-1), rtol=1e-5, atol=1e-7)


def test_silu_matches_torch():
    z = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-12, atol=1e-300)


def _sdpa(q, K, V, causal_pos):
    """Torch SDPA with GQA, for q [m,H,hd] at positions causal_pos over K,V [Hkv,n,hd]."""
    m, H, hd = q.shape
    n = K.shape[1]
    mask = torch.from_numpy(np.arange(n)[None, :] <= np.asarray(causal_pos)[:, None])
    out = F.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2)[None], torch.from_numpy(K)[None],
        torch.from_numpy(V)[None], attn_mask=mask, enable_gqa=True)
    return out[0].permute(1, 0, 2).numpy()


def test_gqa_attention_matches_torch_sdpa():
    rng = np.random.default_rng(5)
    for H, Hkv, hd, n, m in ((8, 2, 16, 23, 5), (4, 4, 8, 9, 9), (32, 8, 128, 40, 3)):
        q = rng.standard_normal((m, H, hd))
        K = rng.standard_normal((Hkv, n, hd))
        V = rng.standard_normal((Hkv, n, hd))
        pos = np.sort(rng.choice(n, m, replace=False))
        pos[-1] = n - 1
        np.testing.assert_allclose(gqa_attention(q, K, V, pos), _sdpa(q, K, V, pos),
                                   rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 4, 8))
    K = rng.standard_normal((2, 1, 8))
    V = rng.standard_normal((2, 1, 8))
    # context of one key: the output is that value
    o = gqa_attention(q, K, V, [0])
    np.testing.assert_allclose(o[0, :2], np.repeat(V[0], 2, axis=0), atol=1e-15)
    np.testing.assert_allclose(o[0, 2:], np.repeat(V[1], 2, axis=0), atol=1e-15)
    # GQA equals MHA with each kv head repeated for its group of q heads
    K = rng.standard_normal((2, 6, 8))
    V = rng.standard_normal((2, 6, 8))
    q = rng.standard_normal((6, 4, 8))
    pos = np.arange(6)
    a = gqa_attention(q, K, V, pos)
    b = gqa_attention(q, np.repeat(K, 2, axis=0), np.repeat(V, 2, axis=0), pos)
    np.testing.assert_allclose(a, b, atol=1e-14)
    # probabilities: rows sum to one, nothing above the diagonal
    _, p = gqa_attention(q, K, V, pos, return_probs=True)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    assert np.all(p[:, np.triu_indices(6, 1)[0], np.triu_indices(6, 1)[1]] == 0)


# ---------------------------------------------------------------- the model

@pytest.fixture(scope="module")
def micro64(micro_path):
    return OracleWeights(micro_path, dtype=np.float64)


@pytest.fixture(scope="module")
def micro32(micro_path):
    return OracleWeights(micro_path, dtype=np.float32)


def test_layer_matches_torch_composition(micro64):
    """One Slow AR block against the same block composed from torch library
    routines (F.linear, F.rms_norm, SDPA with GQA, F.silu) in float64."""
    w = micro64
    cfg = w.cfg
    o = DualAROracle(w, paged=False)
    rng = np.random.default_rng(7)
    T = 11
    x = rng.standard_normal((T, cfg.d))
    from oracle.model import ContiguousKV
    kv = ContiguousKV(cfg.n_slow, cfg.n_kv, cfg.head_dim, np.float64)
    y = o._layer(w.layer("slow", 0), x, np.arange(T), [kv] * T, 0)

    t = {k: torch.from_numpy(np.asarray(v)) for k, v in w.layer("slow", 0).items()}
    X = torch.from_numpy(x)
    H, Hkv, hd = cfg.n_heads, cfg.n_kv, cfg.head_dim
    a = F.rms_norm(X, (cfg.d,), t["attn_norm"], eps=cfg.eps)
    q = F.linear(a, t["wq"]).view(T, H, hd)
    k = F.linear(a, t["wk"]).view(T, Hkv, hd)
    v = F.linear(a, t["wv"]).view(T, Hkv, hd)
    q = F.rms_norm(q, (hd,), t["q_norm"], eps=cfg.eps)
    k = F.rms_norm(k, (hd,), t["k_norm"], eps=cfg.eps)
    cos, sin = rope_table(T, hd, cfg.rope_theta)
    c = torch.from_numpy(np.concatenate([cos, cos], -1).astype(np.float64))[:, None, :]
    s = torch.from_numpy(np.concatenate([sin, sin], -1).astype(np.float64))[:, None, :]

    def rot(z):
        return torch.cat([-z[..., hd // 2:], z[..., :hd // 2]], dim=-1)
    q = q * c + rot(q) * s
    k = k * c + rot(k) * s
    att = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None],
                                         v.permute(1, 0, 2)[None], is_causal=True,
                                         enable_gqa=True)[0].permute(1, 0, 2).reshape(T, H * hd)
    X = X + F.linear(att, t["wo"])
    m = F.rms_norm(X, (cfg.d,), t["mlp_norm"], eps=cfg.eps)
    X = X + F.linear(F.silu(F.linear(m, t["wg"])) * F.linear(m, t["wu"]), t["wd"])
    np.testing.assert_allclose(y, X.numpy(), rtol=1e-10, atol=1e-10)


def _decode_with_log(w, prompt, n, **kw):
    o = DualAROracle(w, record=True, **kw)
    o.prefill(0, prompt.tokens, prompt.codes, prompt.mask)
    codes = o.decode_frames([0], n)[0]
    return o, codes


def test_cached_decode_equals_full_recompute(micro64):
    """Slow AR: each frame's hidden equals a no-cache causal pass over the
    whole sequence; Fast AR: each frame's logits equal a full recompute."""
    w = micro64
    cfg = w.cfg
    p = random_prompt(cfg, 21, 7, seed=11)
    o, codes = _decode_with_log(w, p, 6, paged=True, pool_pages=16)
    inputs = [embed_prompt(w, p.tokens, p.codes, p.mask)]
    inputs += [feedback_embedding(w, codes[f])[None] for f in range(5)]
    Hfull = o.forward_full(np.concatenate(inputs))
    for f, rec in enumerate(o.log):
        np.testing.assert_allclose(rec["h"], Hfull[p.T - 1 + f], rtol=1e-10, atol=1e-10)
        lg = o.fast_full(rec["h"], codes[f])
        np.testing.assert_allclose(np.stack(rec["logits"][1:]), lg, rtol=1e-9, atol=1e-10)
        assert list(np.argmax(lg, -1)) == list(codes[f, 1:])


def test_paged_equals_contiguous(micro32):
    w = micro32
    p = random_prompt(w.cfg, 37, 12, seed=12)
    _, a = _decode_with_log(w, p, 5, paged=False)
    o, b = _decode_with_log(w, p, 5, paged=True, pool_pages=64, perm_seed=3)
    np.testing.assert_array_equal(a, b)
    # pages really were scattered
    st = o.seqs[0]
    assert st.table != sorted(st.table)


@pytest.mark.parametrize("dt", ["f32", "f64"])
def test_prefix_hit_equals_cold(micro32, micro64, dt):
    """A prompt sharing a 32-position prefix with an earlier one decodes to
    the same codes and hiddens as a cold run, and reuses exactly 2 pages.
    (BLAS blocks a GEMM by its height, so row results depend on how many rows
    a call holds: equal to rounding, bitwise only per row.)"""
    w = micro32 if dt == "f32" else micro64
    tol = 1e-5 if dt == "f32" else 1e-12
    cfg = w.cfg
    base = random_prompt(cfg, 40, 20, seed=13, masked_positions=np.arange(20))
    other = random_prompt(cfg, 45, 0, seed=14)
    tok = np.concatenate([base.tokens[:35], other.tokens[:10]])
    cod = np.concatenate([base.codes[:, :35], other.codes[:, :10]], axis=1)
    msk = np.concatenate([base.mask[:35], other.mask[:10]])
    o = DualAROracle(w, paged=True, pool_pages=64, radix=True, record=True)
    assert o.prefill(0, base.tokens, base.codes, base.mask) == 0
    assert o.prefill(1, tok, cod, msk) == 32
    hot = o.decode_frames([1], 4)[0]
    h_hot = [r["h"] for r in o.log]
    cold_o = DualAROracle(w, paged=True, pool_pages=64, radix=False, record=True)
    cold_o.prefill(1, tok, cod, msk)
    cold = cold_o.decode_frames([1], 4)[0]
    np.testing.assert_array_equal(hot, cold)
    for a, b in zip(h_hot, [r["h"] for r in cold_o.log]):
        np.testing.assert_allclose(a, b, rtol=tol, atol=tol)


def test_radix_key_includes_codes(micro32):
    """Same semantic ids but a different residual code must not share KV."""
    w = micro32
    cfg = w.cfg
    a = random_prompt(cfg, 40, 40, seed=15, masked_positions=np.arange(40))
    b_codes = a.codes.copy()
    b_codes[5, 20] = (b_codes[5, 20] + 1) % cfg.codebook_size   # page 1, codebook 5
    o = DualAROracle(w, paged=True, pool_pages=64)
    o.prefill(0, a.tokens, a.codes, a.mask)
    assert o.prefill(1, a.tokens, b_codes, a.mask) == 16        # only page 0 shared


def test_closed_form_with_zero_output_projections(micro_path):
    """With W_o = W_d = 0 every block leaves the residual unchanged, so the
    slow hidden is RMSNorm of the input embedding and the semantic logits
    are its product with the semantic rows of the tied embedding."""
    base = OracleWeights(micro_path, dtype=np.float64)
    cfg = base.cfg
    ov = {}
    for l in range(cfg.n_slow):
        ov[f"slow.{l}.wo"] = np.zeros_like(base.t[f"slow.{l}.wo"])
        ov[f"slow.{l}.wd"] = np.zeros_like(base.t[f"slow.{l}.wd"])
    w = OracleWeights(micro_path, dtype=np.float64, overrides=ov)
    p = random_prompt(cfg, 9, 3, seed=16)
    o = DualAROracle(w, paged=False)
    o.prefill(0, p.tokens, p.codes, p.mask)
    t = p.T - 1
    e = torch.from_numpy(w.t["tok_emb"][p.tokens[t]].copy())
    if p.mask[t]:
        for k in range(cfg.n_codebooks):
            e = e + torch.from_numpy(w.t["vq_emb"][k, p.codes[k, t]])
    h = F.rms_norm(e, (cfg.d,), torch.from_numpy(w.t["slow.final_norm"]), eps=cfg.eps)
    np.testing.assert_allclose(o.seqs[0].h_last, h.numpy(), rtol=1e-12)
    s, code0, lg = o.slow_head(o.seqs[0].h_last)
    ref = torch.from_numpy(w.t["tok_emb"][cfg.sem_begin:]) @ h
    np.testing.assert_allclose(lg, ref.numpy(), rtol=1e-12)
    assert code0 == int(torch.argmax(ref))


def _feedback_run(path, ov, T=9, n=3):
    """Greedy decode of an unmasked prompt (no VQ table enters frame 0's
    input) on the micro model with weight overrides; returns the codes and
    the per-frame slow hiddens."""
    w = OracleWeights(path, dtype=np.float64, overrides=ov)
    p = random_prompt(w.cfg, T, 0, seed=21)
    o = DualAROracle(w, paged=False, record=True)
    o.prefill(0, p.tokens, p.codes, p.mask)
    codes = o.decode_frames([0], n)[0]
    return w, p, codes, [r["h"] for r in o.log]


def test_frame_feedback_closed_form(micro_path):
    """Frame feedback ("SGLang Day-0 Support for FishAudio S2", Background and
    Motivation: the VQ codebook embeddings are interleaved into the token
    stream during decoding).  With W_o = W_d = 0 in every slow block the
    residual stream stays at the block input, so the slow hidden that makes
    frame f >= 1 is RMSNorm of the embedding frame f-1 re-entered with:
    the tied-embedding row of its semantic id sem_begin + c0 plus one row of
    each of the 10 VQ tables.  The expected row is built here by hand from
    the weight tables in torch; the plausible mis-wirings (offset dropped,
    token row missing, the Fast AR input tables summed instead, a codebook
    left out) are each shown to give a different hidden."""
    base = OracleWeights(micro_path, dtype=np.float64)
    cfg = base.cfg
    ov = {}
    for l in range(cfg.n_slow):
        ov[f"slow.{l}.wo"] = np.zeros_like(base.t[f"slow.{l}.wo"])
        ov[f"slow.{l}.wd"] = np.zeros_like(base.t[f"slow.{l}.wd"])
    w, p, codes, hs = _feedback_run(micro_path, ov, n=4)
    tok = torch.from_numpy(w.t["tok_emb"])
    vq = torch.from_numpy(w.t["vq_emb"])
    fin = torch.from_numpy(w.t["fast.in_emb"])
    g = torch.from_numpy(w.t["slow.final_norm"])

    def norm(e):
        return F.rms_norm(e, (cfg.d,), g, eps=cfg.eps).numpy()

    for f in range(1, 4):
        c = [int(x) for x in codes[f - 1]]
        vq_sum = sum(vq[k, c[k]] for k in range(cfg.n_codebooks))
        expect = norm(tok[cfg.sem_begin + c[0]] + vq_sum)
        np.testing.assert_allclose(hs[f], expect, rtol=1e-12, atol=1e-12)
        wrong = {
            "offset dropped": norm(tok[c[0]] + vq_sum),
            "token row missing": norm(vq_sum),
            "fast input tables": norm(tok[cfg.sem_begin + c[0]]
                                      + sum(fin[k, c[k]] for k in range(cfg.n_codebooks))),
            "codebook 9 missing": norm(tok[cfg.sem_begin + c[0]] + vq_sum - vq[9, c[9]]),
        }
        for name, h in wrong.items():
            assert np.max(np.abs(h - hs[f])) > 1e-3, name


def test_frame_feedback_table_perturbations(micro_path):
    """Which tables the frame feedback reads, by perturbation (full model,
    no zeroed blocks): doubling any one VQ table changes the hidden of
    frame 1 but not frame 0 (the prompt has no VQ positions); moving the
    tied-embedding row sem_begin + c0 orthogonally to frame 0's hidden (its
    logit, hence frame 0, unchanged) changes frame 1; the row c0 without the
    offset and the unused Fast AR input table 9 change nothing."""
    base, p, codes, hs = _feedback_run(micro_path, {}, n=2)
    cfg = base.cfg
    c0 = int(codes[0, 0])
    for k in range(cfg.n_codebooks):
        vq = base.t["vq_emb"].copy()
        vq[k] *= 2.0
        _, _, ck, hk = _feedback_run(micro_path, {"vq_emb": vq}, n=2)
        np.testing.assert_array_equal(ck[0], codes[0])
        np.testing.assert_array_equal(hk[0], hs[0])
        assert np.max(np.abs(hk[1] - hs[1])) > 1e-6, k
    tok = base.t["tok_emb"].copy()
    h0 = hs[0]
    delta = np.random.default_rng(5).standard_normal(cfg.d) * 0.05
    delta -= (delta @ h0) / (h0 @ h0) * h0                # no change to frame 0's logits
    tok[cfg.sem_begin + c0] += delta
    _, _, ct, ht = _feedback_run(micro_path, {"tok_emb": tok}, n=2)
    np.testing.assert_array_equal(ct[0], codes[0])
    assert np.max(np.abs(ht[1] - hs[1])) > 1e-6
    assert c0 not in set(int(x) for x in p.tokens)        # row c0 is read by nothing else
    tok = base.t["tok_emb"].copy()
    tok[c0] *= 3.0
    _, _, cn, hn = _feedback_run(micro_path, {"tok_emb": tok}, n=2)
    np.testing.assert_array_equal(cn, codes)
    np.testing.assert_array_equal(hn[1], hs[1])
    fin = base.t["fast.in_emb"].copy()
    fin[9] *= 3.0
    _, _, cf, hf = _feedback_run(micro_path, {"fast.in_emb": fin}, n=2)
    np.testing.assert_array_equal(cf, codes)
    np.testing.assert_array_equal(hf[1], hs[1])


def test_vq_sum_uses_all_codebooks(micro_path):
    """Every one of the 10 codebook tables enters masked positions; none
    enters text positions."""
    w = OracleWeights(micro_path, dtype=np.float64)
    cfg = w.cfg
    p = random_prompt(cfg, 12, 4, seed=17)
    e0 = embed_prompt(w, p.tokens, p.codes, p.mask)
    for k in range(cfg.n_codebooks):
        vq = w.t["vq_emb"].copy()
        vq[k] *= 2.0
        w2 = OracleWeights(micro_path, dtype=np.float64, overrides={"vq_emb": vq})
        e1 = embed_prompt(w2, p.tokens, p.codes, p.mask)
        changed = np.any(e1 != e0, axis=1)
        np.testing.assert_array_equal(changed, p.mask.astype(bool))


def test_fast_ar_table_and_head_indexing(micro_path):
    """Code j depends on head slice j and on input tables 0..j-1 only; input
    table 9 and head slice 0 are never read."""
    base = OracleWeights(micro_path, dtype=np.float64)
    cfg = base.cfg
    p = random_prompt(cfg, 10, 2, seed=18)

    def run(ov):
        w = OracleWeights(micro_path, dtype=np.float64, overrides=ov)
        o = DualAROracle(w, paged=False, record=True)
        o.prefill(0, p.tokens, p.codes, p.mask)
        c = o.decode_frames([0], 1)[0, 0]
        return c, o.log[0]["logits"]

    c0, lg0 = run({})
    emb, head = base.t["fast.in_emb"].copy(), base.t["fast.head"].copy()
    emb[9] = 0
    head[0] = 0
    c1, lg1 = run({"fast.in_emb": emb, "fast.head": head})
    np.testing.assert_array_equal(c0, c1)
    for a, b in zip(lg0, lg1):
        np.testing.assert_array_equal(a, b)
    for j in range(1, cfg.n_codebooks):
        head = base.t["fast.head"].copy()
        head[j] = -head[j]
        _, lgj = run({"fast.head": head})
        for i in range(j):                    # earlier codes untouched
            np.testing.assert_array_equal(lg0[i], lgj[i])
        np.testing.assert_allclose(lgj[j], -lg0[j], rtol=1e-12)
    for j in range(cfg.n_codebooks - 1):
        emb = base.t["fast.in_emb"].copy()
        emb[j] = emb[j] * 1.5
        _, lgj = run({"fast.in_emb": emb})
        for i in range(j + 1):                # codes 0..j do not see table j
            np.testing.assert_array_equal(lg0[i], lgj[i])
        assert np.any(lgj[j + 1] != lg0[j + 1])


def test_constrained_heads_stay_in_range(micro32):
    w = micro32
    cfg = w.cfg
    p = random_prompt(cfg, 30, 10, seed=19)
    o = DualAROracle(w, paged=True, pool_pages=32)
    o.prefill(0, p.tokens, p.codes, p.mask)
    c = o.decode_frames([0], 8)[0]
    assert c.min() >= 0 and c.max() < cfg.codebook_size
    # the full-vocabulary masked argmax equals argmax over the semantic slice
    h = o.seqs[0].h_last
    s, code0, lg = o.slow_head(h)
    assert s == cfg.sem_begin + code0 == cfg.sem_begin + int(np.argmax(lg))


def test_teacher_forced_reproduces_free_running(micro32):
    w = micro32
    p = random_prompt(w.cfg, 25, 9, seed=20)
    o, codes = _decode_with_log(w, p, 7, paged=True, pool_pages=32)
    tf = o.teacher_forced(p.tokens, p.codes, p.mask, codes)
    np.testing.assert_array_equal(tf["pred"], codes)
    for f, rec in enumerate(o.log):
        np.testing.assert_allclose(tf["h"][f], rec["h"], rtol=2e-5, atol=2e-5)
        np.testing.assert_allclose(tf["logits"][f], np.stack(rec["logits"]), rtol=2e-4, atol=2e-4)


def test_tiny_workload_free_running_margins(tiny_path):
    """The tiny workload decodes 4 frames; the oracle's top-2 margins are
    far above float32 rounding, so bit-exact code parity is meaningful."""
    w = OracleWeights(tiny_path, dtype=np.float32)
    wl = make_workload(0)
    p = wl.prompts[0]
    o, codes = _decode_with_log(w, p, wl.n_frames, paged=True, pool_pages=wl.pool_pages)
    assert codes.shape == (4, 10)
    tf = o.teacher_forced(p.tokens, p.codes, p.mask, codes)
    np.testing.assert_array_equal(tf["pred"], codes)
    assert tf["margin"].min() > 1e-4, tf["margin"].min()
    # float64 gives the same codes
    w64 = OracleWeights(tiny_path, dtype=np.float64)
    _, c64 = _decode_with_log(w64, p, wl.n_frames, paged=True, pool_pages=wl.pool_pages)
    np.testing.assert_array_equal(codes, c64)


# ---------------------------------------------------------------- INT8 weights

def test_int8_quantisation_properties():
    """Per-row symmetric INT8: the largest |w| of a row maps to +-127, the
    rounding error is at most half a step, and a row of exact multiples of
    its step is reproduced exactly."""
    from oracle import quantize_rows_int8, dequantize_rows_int8
    rng = np.random.default_rng(30)
    w = (rng.standard_normal((64, 200)) * 0.02).astype(np.float32)
    w[5] = 0.0
    q, s = quantize_rows_int8(w)
    assert q.dtype == np.int8 and s.dtype == np.float32
    assert np.all(np.abs(q.astype(int)) <= 127)
    rows = [r for r in range(64) if r != 5]
    assert np.all(np.abs(q[rows]).max(axis=1) == 127)
    assert s[5] == 1.0 and not q[5].any()
    err = np.abs(dequantize_rows_int8(q, s) - w)
    assert np.all(err <= s[:, None] * 0.5 * (1 + 1e-6))
    # exact multiples survive unchanged
    k = rng.integers(-127, 128, (3, 50)).astype(np.float32)
    k[:, 0] = 127
    step = np.float32(0.25)
    q2, s2 = quantize_rows_int8(k * step)
    np.testing.assert_array_equal(s2, step)
    np.testing.assert_array_equal(q2, k.astype(np.int8))


def test_int8_round_half_even_matches_torch():
    """Ties of w/scale round to even, as torch.round does."""
    from oracle import quantize_rows_int8
    w = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.5, 126.5]], np.float32)
    q, s = quantize_rows_int8(w)
    assert s[0] == 1.0
    ref = torch.round(torch.from_numpy(w)).to(torch.int8).numpy()
    np.testing.assert_array_equal(q, ref)


def test_int8_oracle_decodes_and_stays_close(micro_path):
    """The INT8 model is a different model; on the micro config its frames
    mostly agree with the unquantised one and its cached decode still equals
    the full recompute."""
    w8 = OracleWeights(micro_path, dtype=np.float64, quant="int8")
    p = random_prompt(w8.cfg, 20, 6, seed=31)
    o, codes = _decode_with_log(w8, p, 5, paged=True, pool_pages=16)
    tf = o.teacher_forced(p.tokens, p.codes, p.mask, codes)
    np.testing.assert_array_equal(tf["pred"], codes)
    for f, rec in enumerate(o.log):
        np.testing.assert_allclose(tf["h"][f], rec["h"], rtol=1e-9, atol=1e-9)
