"""Pins of the vocoder oracle (oracle/dac.py) against things other than itself.

CPU only.  Convolutions against PyTorch's CPU routines and NumPy's textbook
correlation, the transposed convolution against its adjoint, Snake against
closed-form values, the block and residual structure against special cases
that reduce it to a closed form, and the whole decoder against the pages'
samples per frame, locality and time-shift equivariance.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle.dac import (DacWeights, snake, conv1d, conv_transpose1d, residual_unit,
                        decoder_block, rvq_decode, dac_decode, dac_stages)
from s2_inputs.vocoder import (DAC_S2, DAC_MINI, DAC_MICRO, ensure_vocoder, random_codes,
                               tensor_specs, VocoderFile)

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


@pytest.fixture(scope="module")
def micro(weights_dir):
    return DacWeights(ensure_vocoder(DAC_MICRO, weights_dir))


@pytest.fixture(scope="module")
def mini(weights_dir):
    return DacWeights(ensure_vocoder(DAC_MINI, weights_dir))


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ shapes

def test_full_decoder_hop_is_the_pages_samples_per_frame():
    """2,048 samples per frame at 44.1 kHz ('s2pro-native', What happens to a
    sentence): the upsampling rates multiply to the hop, and 44,100 / 2,048
    is the ~21 Hz frame rate of the codec."""
    assert DAC_S2.hop == GOLDEN["samples_per_frame"]["value"]
    fr = GOLDEN["sample_rate_hz"]["value"] / DAC_S2.hop
    assert abs(fr - GOLDEN["frame_rate_hz"]["value"]) <= GOLDEN["frame_rate_hz"]["abs_tol"]
    assert abs(1000 * DAC_S2.hop / GOLDEN["sample_rate_hz"]["value"] -
               GOLDEN["frame_ms"]["value"]) <= GOLDEN["frame_ms"]["abs_tol"]
    assert DAC_S2.n_codebooks == GOLDEN["codebooks"]["value"]


def test_full_decoder_parameter_count():
    """Tensor shapes of the full decoder add up to its layer-by-layer count
    (each block: transposed conv c*(c/2)*2s + three units of 8*(c/2)^2,
    plus biases and alphas)."""
    n = sum(int(np.prod(s)) for _, s, _ in tensor_specs(DAC_S2))
    L, D = DAC_S2.latent, DAC_S2.dim
    want = 10 * 4096 * 8 + 10 * L * 8 + 10 * L + D * L * 7 + D
    c = D
    for s in DAC_S2.rates:
        h = c // 2
        want += c + c * h * 2 * s + h + 3 * (h + h * h * 7 + h + h + h * h + h)
        c = h
    want += c + c * 7 + 1
    assert n == want
    assert 50e6 < n < 60e6


# ------------------------------------------------------------------ Snake

def test_snake_closed_forms():
    """sin^2 vanishes at multiples of pi/alpha (Snake is the identity
    there), is 1 at odd multiples of pi/(2 alpha), and Snake(0) = 0."""
    alpha = np.array([0.5, 1.0, 1.37])
    k = np.arange(-3, 4, dtype=np.float64)
    x0 = k[None, :] * np.pi / alpha[:, None]
    np.testing.assert_allclose(snake(x0, alpha), x0, atol=1e-12)
    x1 = (k[None, :] + 0.5) * np.pi / alpha[:, None]
    np.testing.assert_allclose(snake(x1, alpha), x1 + 1.0 / (alpha[:, None] + 1e-9), rtol=1e-12)
    assert not snake(np.zeros((3, 5)), alpha).any()


def test_snake_is_channelwise():
    """Each channel uses its own alpha: swapping two channels' alphas swaps
    exactly those rows of the output."""
    x = _rng(1).standard_normal((4, 9))
    a = np.array([0.6, 0.9, 1.2, 1.4])
    b = a[[0, 2, 1, 3]]
    ya, yb = snake(x, a), snake(x, b)
    np.testing.assert_array_equal(ya[[0, 3]], yb[[0, 3]])
    assert not np.allclose(ya[1:3], yb[1:3])


# ------------------------------------------------------------------ convolutions

@pytest.mark.parametrize("cin,cout,k,dil,pad,T", [(3, 5, 7, 1, 3, 20), (4, 4, 7, 3, 9, 33),
                                                  (6, 2, 7, 9, 27, 64), (5, 7, 1, 1, 0, 11)])
def test_conv1d_matches_torch(cin, cout, k, dil, pad, T):
    r = _rng(cin * 100 + k + dil)
    x, w, b = r.standard_normal((cin, T)), r.standard_normal((cout, cin, k)), r.standard_normal(cout)
    ref = F.conv1d(torch.from_numpy(x)[None], torch.from_numpy(w), torch.from_numpy(b),
                   padding=pad, dilation=dil)[0].numpy()
    np.testing.assert_allclose(conv1d(x, w, b, dil, pad), ref, rtol=1e-12, atol=1e-12)


def test_conv1d_single_channel_is_numpy_correlation():
    """One channel in and out: the textbook correlation of the zero-padded
    signal with the kernel dilated by zero-stuffing."""
    r = _rng(7)
    x, w = r.standard_normal(40), r.standard_normal(7)
    for dil in (1, 3, 9):
        wd = np.zeros(6 * dil + 1)
        wd[::dil] = w
        ref = np.correlate(np.pad(x, 3 * dil), wd, mode="valid")
        got = conv1d(x[None], w[None, None], np.zeros(1), dil, 3 * dil)[0]
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("s", [2, 4, 8])
def test_conv_transpose_matches_torch(s):
    r = _rng(s)
    cin, cout, T = 6, 3, 13
    x, w, b = r.standard_normal((cin, T)), r.standard_normal((cin, cout, 2 * s)), r.standard_normal(cout)
    ref = F.conv_transpose1d(torch.from_numpy(x)[None], torch.from_numpy(w), torch.from_numpy(b),
                             stride=s, padding=s // 2)[0].numpy()
    got = conv_transpose1d(x, w, b, s, s // 2)
    assert got.shape == (cout, T * s)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("s", [2, 4, 8])
def test_conv_transpose_is_the_adjoint_of_the_strided_conv(s):
    """<convT(x; W), y> = <x, conv(y; W, stride s)>: the transposed
    convolution is the adjoint of the strided convolution with the same
    weights and padding (no bias)."""
    r = _rng(10 + s)
    cin, cout, T = 5, 4, 11
    w = r.standard_normal((cin, cout, 2 * s))
    x = r.standard_normal((cin, T))
    y = r.standard_normal((cout, T * s))
    lhs = np.sum(conv_transpose1d(x, w, np.zeros(cout), s, s // 2) * y)
    # strided conv: out[i, t] = sum_{o,j} w[i, o, j] y[o, t*s + j - s/2]
    ypad = np.pad(y, ((0, 0), (s // 2, s // 2 + s)))
    cy = np.zeros((cin, T))
    for t in range(T):
        cy[:, t] = np.einsum("ioj,oj->i", w, ypad[:, t * s:t * s + 2 * s])
    assert abs(lhs - np.sum(x * cy)) < 1e-9 * max(1.0, abs(lhs))


# ------------------------------------------------------------------ structure

def _unit_params(c, r, zero_conv2=False):
    p = {"alpha1": r.random(c) + 0.5, "alpha2": r.random(c) + 0.5,
         "conv1.w": r.standard_normal((c, c, 7)) / 5, "conv1.b": r.standard_normal(c) * 0.1,
         "conv2.w": r.standard_normal((c, c, 1)) / 3, "conv2.b": r.standard_normal(c) * 0.1}
    if zero_conv2:
        p["conv2.w"] = np.zeros((c, c, 1))
        p["conv2.b"] = np.zeros(c)
    return p


def test_residual_unit_with_zero_output_conv_is_identity():
    r = _rng(21)
    x = r.standard_normal((4, 30))
    np.testing.assert_array_equal(residual_unit(x, _unit_params(4, r, True), 3), x)


def test_residual_unit_with_constant_inner_conv_closed_form():
    """conv1 = 0 with bias c: the inner activation is Snake(c) at every time
    (the padding does not reach it: padding enters only through conv1's
    input), so the unit adds conv2.w @ Snake(c) + conv2.b to x."""
    r = _rng(22)
    p = _unit_params(5, r)
    p["conv1.w"] = np.zeros((5, 5, 7))
    x = r.standard_normal((5, 17))
    inner = snake(p["conv1.b"][:, None], p["alpha2"])[:, 0]
    want = x + (p["conv2.w"][:, :, 0] @ inner + p["conv2.b"])[:, None]
    np.testing.assert_allclose(residual_unit(x, p, 9), want, rtol=1e-12, atol=1e-12)


def test_residual_unit_matches_torch_composition():
    r = _rng(23)
    p = _unit_params(6, r)
    x = r.standard_normal((6, 50))
    t = {k: torch.from_numpy(v) for k, v in p.items()}
    X = torch.from_numpy(x)[None]

    def sn(v, a):
        a = a[None, :, None]
        return v + torch.sin(a * v).pow(2) / (a + 1e-9)

    Y = F.conv1d(sn(X, t["alpha1"]), t["conv1.w"], t["conv1.b"], padding=9, dilation=3)
    Y = F.conv1d(sn(Y, t["alpha2"]), t["conv2.w"], t["conv2.b"])
    np.testing.assert_allclose(residual_unit(x, p, 3), (X + Y)[0].numpy(), rtol=1e-12, atol=1e-12)


def test_decoder_block_without_residual_branches_is_snake_then_upsample():
    """All residual units' output convs zero: the block is Snake followed by
    the transposed convolution alone (checked against torch)."""
    r = _rng(24)
    c, s = 6, 4
    p = {"alpha": r.random(c) + 0.5, "up.w": r.standard_normal((c, c // 2, 2 * s)),
         "up.b": r.standard_normal(c // 2)}
    for j in range(3):
        for k, v in _unit_params(c // 2, r, True).items():
            p[f"res.{j}.{k}"] = v
    x = r.standard_normal((c, 9))
    want = F.conv_transpose1d(torch.from_numpy(snake(x, p["alpha"]))[None], torch.from_numpy(p["up.w"]),
                              torch.from_numpy(p["up.b"]), stride=s, padding=s // 2)[0].numpy()
    np.testing.assert_allclose(decoder_block(x, p, s), want, rtol=1e-12, atol=1e-12)


def test_decoder_block_dilation_order():
    """The three units run with dilations 1, 3, 9 in that order: running the
    units by hand in another order gives a different result, the stated
    order the same one."""
    r = _rng(25)
    c, s = 4, 2
    p = {"alpha": r.random(c) + 0.5, "up.w": r.standard_normal((c, c // 2, 2 * s)) / 3,
         "up.b": np.zeros(c // 2)}
    units = [_unit_params(c // 2, r) for _ in range(3)]
    for j, u in enumerate(units):
        for k, v in u.items():
            p[f"res.{j}.{k}"] = v
    x = r.standard_normal((c, 40))
    y = conv_transpose1d(snake(x, p["alpha"]), p["up.w"], p["up.b"], s, s // 2)
    want = residual_unit(residual_unit(residual_unit(y, units[0], 1), units[1], 3), units[2], 9)
    other = residual_unit(residual_unit(residual_unit(y, units[0], 9), units[1], 3), units[2], 1)
    got = decoder_block(x, p, s)
    np.testing.assert_array_equal(got, want)
    assert not np.allclose(got, other)


def test_rvq_decode_against_embedding_and_pointwise_conv(micro):
    """Sum over codebooks of a table lookup and a 1x1 projection, recomputed
    with torch's embedding and conv1d."""
    codes = random_codes(DAC_MICRO, 1, 12, 31)[0].T          # [n_cb, T]
    cb = torch.from_numpy(micro.t["rvq.codebook"])
    pw = torch.from_numpy(micro.t["rvq.proj_w"])
    pb = torch.from_numpy(micro.t["rvq.proj_b"])
    z = 0
    for k in range(codes.shape[0]):
        e = F.embedding(torch.from_numpy(codes[k]).long(), cb[k]).T[None]    # [1, cb_dim, T]
        z = z + F.conv1d(e, pw[k][:, :, None], pb[k])[0]
    np.testing.assert_allclose(rvq_decode(codes, micro), z.numpy(), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ whole decoder

def _torch_decode(codes, wt):
    """The decoder as a composition of torch's CPU routines (fp64)."""
    t = {k: torch.from_numpy(v) for k, v in wt.t.items()}

    def sn(v, a):
        a = a[None, :, None]
        return v + torch.sin(a * v).pow(2) / (a + 1e-9)

    z = 0
    for k in range(codes.shape[1]):
        e = F.embedding(torch.from_numpy(codes[:, k]).long(), t["rvq.codebook"][k]).T[None]
        z = z + F.conv1d(e, t["rvq.proj_w"][k][:, :, None], t["rvq.proj_b"][k])
    x = F.conv1d(z, t["conv_in.w"], t["conv_in.b"], padding=3)
    for i, s in enumerate(wt.cfg.rates):
        p = f"block.{i}."
        x = F.conv_transpose1d(sn(x, t[p + "alpha"]), t[p + "up.w"], t[p + "up.b"], stride=s,
                               padding=s // 2)
        for j, dil in enumerate((1, 3, 9)):
            q = f"{p}res.{j}."
            y = F.conv1d(sn(x, t[q + "alpha1"]), t[q + "conv1.w"], t[q + "conv1.b"], padding=3 * dil,
                         dilation=dil)
            x = x + F.conv1d(sn(y, t[q + "alpha2"]), t[q + "conv2.w"], t[q + "conv2.b"])
    y = F.conv1d(sn(x, t["out.alpha"]), t["out.w"], t["out.b"], padding=3)
    return torch.tanh(y)[0, 0].numpy()


@pytest.mark.parametrize("which", ["micro", "mini"])
def test_decode_matches_torch_composition(which, micro, mini):
    wt = micro if which == "micro" else mini
    codes = random_codes(wt.cfg, 1, 9, 41)[0]
    got = dac_decode(codes, wt)
    assert got.shape == (9 * wt.cfg.hop,)
    np.testing.assert_allclose(got, _torch_decode(codes, wt), rtol=0, atol=1e-12)
    assert np.all(np.abs(got) < 1)
    assert got.std() > 0.05           # the random decoder is not saturated or silent


def _receptive_frames(cfg):
    """Frames of context on each side that can reach an output sample:
    input conv 3 frames; block i (rate s at the block's input rate, hop h_i
    samples of the block's output per frame) adds one input sample of the
    transposed conv and 3*(1+3+9) output samples of its units; output conv 3
    samples."""
    r = 3.0
    h = 1
    for s in cfg.rates:
        r += 1.0 / h                    # the transposed conv reads input t and t +- 1
        h *= s
        r += 3 * (1 + 3 + 9) / h
    r += 3.0 / h
    return int(math.ceil(r))


def test_decode_is_local(mini):
    """Changing the codes of the last frame leaves every sample outside its
    receptive field bit-identical, and changes samples inside it."""
    cfg = mini.cfg
    T = 24
    codes = random_codes(cfg, 1, T, 42)[0]
    alt = codes.copy()
    alt[-1] = (alt[-1] + 1) % cfg.codebook_size
    a, b = dac_decode(codes, mini), dac_decode(alt, mini)
    first = (T - 1 - _receptive_frames(cfg)) * cfg.hop
    assert first > 0
    np.testing.assert_array_equal(a[:first], b[:first])
    assert not np.allclose(a[-cfg.hop:], b[-cfg.hop:])


def test_decode_is_time_shift_equivariant(mini):
    """Dropping the first frame shifts the waveform by one hop away from the
    edges (zero padding is the only position dependence)."""
    cfg = mini.cfg
    T = 24
    codes = random_codes(cfg, 1, T, 43)[0]
    a, b = dac_decode(codes, mini), dac_decode(codes[1:], mini)
    m = (_receptive_frames(cfg) + 1) * cfg.hop
    np.testing.assert_allclose(a[cfg.hop + m:-m], b[m:-m], rtol=0, atol=1e-12)


def test_stages_have_the_stated_shapes(mini):
    cfg = mini.cfg
    st = dict(dac_stages(random_codes(cfg, 1, 5, 44)[0], mini))
    assert st["latent"].shape == (cfg.latent, 5)
    assert st["conv_in"].shape == (cfg.dim, 5)
    h = 1
    for i, s in enumerate(cfg.rates):
        h *= s
        assert st[f"block.{i}"].shape == (cfg.channels(i), 5 * h)
    assert st["audio"].shape == (5 * cfg.hop,)


def test_vocoder_file_round_trip(mini):
    """The stored bf16 conv weights widen to the float32 draws rounded to
    bf16; alphas lie in [0.5, 1.5)."""
    vf = VocoderFile(mini_path := ensure_vocoder(DAC_MINI))
    assert vf.config("dac_mini") == DAC_MINI
    for name, (dt, shape, _, _) in vf.entries.items():
        a = mini.t[name]
        assert a.shape == tuple(shape)
        if name.endswith("alpha") or name.endswith("alpha1") or name.endswith("alpha2"):
            assert a.min() >= 0.5 and a.max() < 1.5
        if dt == 1:
            assert np.all(a.astype(np.float32).view(np.uint32) & 0xFFFF == 0)
    del mini_path
