"""DAC vocoder decode: plain fp64 CPU oracle (codes -> waveform).

TEST INFRASTRUCTURE ONLY (as the rest of this package): nothing on the
product path imports or runs it.

What the pages fix: the residual codebook indices the Dual-AR emits are
decoded into a waveform by a DAC codec ("SGLang Day-0 Support for FishAudio
S2", Architecture, Stage 3), 2,048 audio samples per frame at 44.1 kHz
("s2pro-native", What happens to a sentence), 10 codebooks at about 21 Hz
("Fish Audio Abre Codigo do S2", Arquitetura Dual-AR).  The pages print no
decoder layers; the reading taken is the published DAC decoder (Kumar et al.
2023, "High-Fidelity Audio Compression with Improved RVQGAN"), written here
from its description:

  * residual codebook lookup: every codebook k maps its code to a cb_dim
    vector, a 1x1 projection with bias lifts it to the latent width, and the
    codebooks' contributions are summed;
  * a k=7 convolution to the decoder width;
  * per upsampling block of rate s: Snake, a transposed convolution of
    kernel 2s and stride s with s/2 samples cropped from both ends (exactly
    s output samples per input sample), then three residual units with
    dilations 1, 3, 9, each x + conv_k1(Snake(conv_k7,dil(Snake(x)))) with
    "same" padding 3*dil;
  * Snake, a k=7 convolution to one channel, tanh.

Snake(x) = x + sin^2(alpha x) / (alpha + 1e-9), alpha per channel.  Every
convolution pads with zeros.  Activations are [channels, time]; weights are
the stored bf16 / f32 values widened exactly to float64.
"""

import numpy as np

from s2_inputs.vocoder import VocoderFile, DILATIONS


def _widen(raw, is_bf16):
    if is_bf16:
        return (np.asarray(raw, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
            np.float32).astype(np.float64)
    return np.asarray(raw, dtype=np.float32).astype(np.float64)


class DacWeights:
    """Every tensor of a vocoder file, widened exactly to float64."""

    def __init__(self, src):
        vf = src if isinstance(src, VocoderFile) else VocoderFile(src)
        self.cfg = vf.config()
        self.t = {name: _widen(vf.raw(name), vf.is_bf16(name)) for name in vf.entries}

    def sub(self, prefix):
        n = len(prefix)
        return {k[n:]: v for k, v in self.t.items() if k.startswith(prefix)}


def snake(x, alpha):
    """Snake activation, channel-wise: x + sin(alpha x)^2 / (alpha + 1e-9)."""
    a = np.asarray(alpha, dtype=np.float64)[:, None]
    return x + np.sin(a * x) ** 2 / (a + 1e-9)


def conv1d(x, w, b, dilation=1, padding=0):
    """y[o, t] = b[o] + sum_{i, j} w[o, i, j] x[i, t + j*dilation - padding],
    x read as zero outside [0, T).  x [Cin, T], w [Cout, Cin, k]."""
    cin, T = x.shape
    cout, cin_w, k = w.shape
    assert cin == cin_w
    xp = np.zeros((cin, T + 2 * padding), dtype=np.float64)
    xp[:, padding:padding + T] = x
    tout = T + 2 * padding - dilation * (k - 1)
    y = np.repeat(np.asarray(b, dtype=np.float64)[:, None], tout, axis=1)
    for j in range(k):
        y += w[:, :, j] @ xp[:, j * dilation:j * dilation + tout]
    return y


def conv_transpose1d(x, w, b, stride, padding):
    """Transposed convolution: input sample t adds w[:, :, j]^T x[:, t] to
    output position t*stride + j of the uncropped output, then `padding`
    samples are dropped at both ends.  x [Cin, T], w [Cin, Cout, k]."""
    cin, T = x.shape
    cin_w, cout, k = w.shape
    assert cin == cin_w
    full = np.zeros((cout, (T - 1) * stride + k), dtype=np.float64)
    for j in range(k):
        full[:, j:j + stride * (T - 1) + 1:stride] += w[:, :, j].T @ x
    tout = (T - 1) * stride + k - 2 * padding
    return full[:, padding:padding + tout] + np.asarray(b, dtype=np.float64)[:, None]


def residual_unit(x, p, dilation):
    """x + conv_k1(Snake(conv_k7,dilation(Snake(x))))."""
    y = conv1d(snake(x, p["alpha1"]), p["conv1.w"], p["conv1.b"], dilation, 3 * dilation)
    y = conv1d(snake(y, p["alpha2"]), p["conv2.w"], p["conv2.b"])
    return x + y


def decoder_block(x, p, stride):
    """Snake -> transposed conv (kernel 2*stride, stride) -> residual units."""
    assert stride % 2 == 0
    y = conv_transpose1d(snake(x, p["alpha"]), p["up.w"], p["up.b"], stride, stride // 2)
    for j, dil in enumerate(DILATIONS):
        y = residual_unit(y, {k[len(f"res.{j}."):]: v for k, v in p.items()
                              if k.startswith(f"res.{j}.")}, dil)
    return y


def rvq_decode(codes, wt):
    """codes [n_codebooks, T] -> latent [latent, T]: the sum over codebooks
    of proj_w[k] @ codebook[k][codes[k]] + proj_b[k]."""
    cb, pw, pb = wt.t["rvq.codebook"], wt.t["rvq.proj_w"], wt.t["rvq.proj_b"]
    n_cb, T = codes.shape
    z = np.zeros((pw.shape[1], T), dtype=np.float64)
    for k in range(n_cb):
        z += pw[k] @ cb[k][codes[k]].T + pb[k][:, None]
    return z


def dac_stages(codes, wt):
    """All intermediate activations of one sequence: codes [T, n_codebooks]
    -> list of (name, array); the last is the waveform [T * hop]."""
    codes = np.asarray(codes)
    out = []
    z = rvq_decode(codes.T, wt)
    out.append(("latent", z))
    x = conv1d(z, wt.t["conv_in.w"], wt.t["conv_in.b"], 1, 3)
    out.append(("conv_in", x))
    for i, s in enumerate(wt.cfg.rates):
        x = decoder_block(x, wt.sub(f"block.{i}."), s)
        out.append((f"block.{i}", x))
    y = conv1d(snake(x, wt.t["out.alpha"]), wt.t["out.w"], wt.t["out.b"], 1, 3)
    out.append(("audio", np.tanh(y[0])))
    return out


def dac_decode(codes, wt):
    """Waveform [T * hop] of one sequence's codes [T, n_codebooks]."""
    return dac_stages(codes, wt)[-1][1]


def dac_decode_batch(codes, wt):
    """codes [B, T, n_codebooks] -> waveforms [B, T * hop] (sequences are
    independent)."""
    return np.stack([dac_decode(c, wt) for c in np.asarray(codes)])
