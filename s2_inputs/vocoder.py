"""Random-init DAC vocoder weights: configuration, file format, writer, reader.

Data only: shapes, seeded random numbers and the byte layout.  The decode
arithmetic lives in the oracle and in the CUDA path, each on its own.

The decoder shape is a DAC-style convolutional decoder (codes -> residual
codebook lookup -> 1x1 projections summed -> conv -> upsampling blocks ->
conv -> tanh).  Per codebook: an embedding table [C, cb_dim] and a 1x1
projection cb_dim -> latent with bias.  Each upsampling block of rate s maps
c -> c/2 channels: Snake, transposed conv (kernel 2s, stride s), then three
residual units with dilations 1, 3, 9 (Snake, conv k=7, Snake, conv k=1,
residual add).  The output stage is Snake, conv c_last -> 1 (k=7), tanh.

File format (little-endian):

  offset 0   char[8]  magic "S2DACVOC"
         8   u32      version (1)
        12   u32      n_blocks
        16   i32[5]   latent, dim, cb_dim, n_codebooks, codebook_size
        36   i32[8]   rates (n_blocks used)
        68   u32      n_tensors
        72   u32      seed
        76   u64      data offset
       128   entries  n_tensors x 128 bytes (same entry layout as the Dual-AR
                      weight file: char name[64], u32 dtype (0 f32, 1 bf16),
                      u32 ndim, u64 shape[4], u64 offset, u64 nbytes, u64 0)
  Tensors start on 4096-byte boundaries, row-major.  Conv weights are
  [c_out, c_in, k]; transposed-conv weights [c_in, c_out, k] (the usual
  framework layouts).

Values (one ``numpy.random.default_rng([seed, index])`` stream per tensor in
file order, float32):
  * conv and transposed-conv weights N(0, 1/fan_in), fan_in = c_in * k
    (c_in * 2 for a transposed conv: two taps reach each output sample),
    except the residual units' 1x1 output convs, N(0, 1/(16 fan_in)), so
    that the activations stay of order one through the stack; all rounded
    to nearest-even bf16 and stored as bf16;
  * biases N(0, 0.02^2), float32;
  * Snake alphas uniform on [0.5, 1.5), float32 (one per channel);
  * codebooks N(0, 1), projections N(0, 1/(n_codebooks cb_dim)), float32.
"""

import os
import struct
from dataclasses import dataclass

import numpy as np

from .weights import _f32_to_bf16_bits

MAGIC = b"S2DACVOC"
HEADER = 128
ENTRY = 128
ALIGN = 4096
DILATIONS = (1, 3, 9)
MAX_BLOCKS = 8


@dataclass(frozen=True)
class VocoderConfig:
    name: str
    latent: int
    dim: int
    rates: tuple
    cb_dim: int = 8
    n_codebooks: int = 10
    codebook_size: int = 4096
    seed: int = 2

    @property
    def hop(self):
        h = 1
        for r in self.rates:
            h *= r
        return h

    def channels(self, i):
        """Channels at the output of block i (i = -1: the input conv)."""
        return self.dim >> (i + 1)


# Full-size decoder: 2,048 samples per frame at 44.1 kHz (rates 8*8*4*4*2),
# latent 1024, decoder width 1536 halving per block down to 48 channels,
# 10 codebooks of 4,096 entries (the codes the Fast AR emits).
DAC_S2 = VocoderConfig(name="dac_s2", latent=1024, dim=1536, rates=(8, 8, 4, 4, 2))

# Small decoder for oracle pins and quick parity (hop 32; channels 256 ->
# 128, 64, 32: the last is not a multiple of 64).
DAC_MINI = VocoderConfig(name="dac_mini", latent=128, dim=256, rates=(4, 4, 2),
                         codebook_size=512, seed=5)

# Micro decoder for fp64 brute-force pins on the CPU (hop 8).
DAC_MICRO = VocoderConfig(name="dac_micro", latent=12, dim=16, rates=(2, 4),
                          cb_dim=4, codebook_size=16, seed=9)

VOCODERS = {v.name: v for v in (DAC_S2, DAC_MINI, DAC_MICRO)}


def tensor_specs(cfg: VocoderConfig):
    """(name, shape, kind) in file order; kind in {'conv', 'conv_res',
    'convT', 'bias', 'alpha', 'codebook', 'proj'}."""
    L, D = cfg.latent, cfg.dim
    specs = [("rvq.codebook", (cfg.n_codebooks, cfg.codebook_size, cfg.cb_dim), "codebook"),
             ("rvq.proj_w", (cfg.n_codebooks, L, cfg.cb_dim), "proj"),
             ("rvq.proj_b", (cfg.n_codebooks, L), "bias"),
             ("conv_in.w", (D, L, 7), "conv"),
             ("conv_in.b", (D,), "bias")]
    for i, s in enumerate(cfg.rates):
        ci, co = cfg.channels(i - 1), cfg.channels(i)
        p = f"block.{i}."
        specs += [(p + "alpha", (ci,), "alpha"),
                  (p + "up.w", (ci, co, 2 * s), "convT"),
                  (p + "up.b", (co,), "bias")]
        for j in range(len(DILATIONS)):
            q = f"{p}res.{j}."
            specs += [(q + "alpha1", (co,), "alpha"),
                      (q + "conv1.w", (co, co, 7), "conv"),
                      (q + "conv1.b", (co,), "bias"),
                      (q + "alpha2", (co,), "alpha"),
                      (q + "conv2.w", (co, co, 1), "conv_res"),
                      (q + "conv2.b", (co,), "bias")]
    cl = cfg.channels(len(cfg.rates) - 1)
    specs += [("out.alpha", (cl,), "alpha"),
              ("out.w", (1, cl, 7), "conv"),
              ("out.b", (1,), "bias")]
    return specs


def _layout(cfg):
    specs = tensor_specs(cfg)
    off = HEADER + ENTRY * len(specs)
    off = (off + ALIGN - 1) // ALIGN * ALIGN
    data0 = off
    table = []
    for name, shape, kind in specs:
        n = int(np.prod(shape))
        dt = 1 if kind in ("conv", "conv_res", "convT") else 0
        nbytes = n * (2 if dt == 1 else 4)
        table.append((name, shape, kind, dt, off, nbytes))
        off = (off + nbytes + ALIGN - 1) // ALIGN * ALIGN
    return data0, table, off


def _gen(cfg, index, shape, kind):
    rng = np.random.default_rng([cfg.seed, index])
    if kind == "alpha":
        return (rng.random(size=shape, dtype=np.float32) + np.float32(0.5)).astype(np.float32)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    gain = 1.0
    if kind in ("conv", "conv_res"):
        fan_in = shape[1] * shape[2]
        if kind == "conv_res":
            gain = 0.25
    elif kind == "convT":
        fan_in = shape[0] * 2          # each output sample sees 2 taps of every input channel
    elif kind == "proj":
        fan_in = shape[2] * shape[0]   # the codebooks' sum has unit variance
    elif kind == "bias":
        return x * np.float32(0.02)
    else:                              # codebook
        return x
    return x * np.float32(gain / np.sqrt(fan_in))


def write_vocoder(cfg: VocoderConfig, path: str):
    data0, table, total = _layout(cfg)
    tmp = path + ".tmp"
    with open(tmp, "wb") as f:
        hdr = bytearray(HEADER)
        struct.pack_into("<8sII", hdr, 0, MAGIC, 1, len(cfg.rates))
        struct.pack_into("<5i", hdr, 16, cfg.latent, cfg.dim, cfg.cb_dim, cfg.n_codebooks,
                         cfg.codebook_size)
        rates = list(cfg.rates) + [0] * (MAX_BLOCKS - len(cfg.rates))
        struct.pack_into("<8i", hdr, 36, *rates)
        struct.pack_into("<IIQ", hdr, 68, len(table), cfg.seed, data0)
        f.write(hdr)
        for name, shape, kind, dt, off, nbytes in table:
            e = bytearray(ENTRY)
            shp = list(shape) + [0] * (4 - len(shape))
            struct.pack_into("<64sII4QQQQ", e, 0, name.encode(), dt, len(shape), *shp, off, nbytes, 0)
            f.write(e)
        f.truncate(total)
    mm = np.memmap(tmp, dtype=np.uint8, mode="r+")
    for i, (name, shape, kind, dt, off, nbytes) in enumerate(table):
        a = _gen(cfg, i, shape, kind)
        b = _f32_to_bf16_bits(a).reshape(-1).view(np.uint8) if dt == 1 else a.reshape(-1).view(np.uint8)
        mm[off:off + nbytes] = b
    mm.flush()
    del mm
    os.replace(tmp, path)
    return path


def vocoder_path(cfg: VocoderConfig, root: str = None):
    root = root or os.environ.get("S2_WEIGHTS_DIR") or os.path.join(
        os.environ.get("TMPDIR", "/tmp"), "s2_weights")
    os.makedirs(root, exist_ok=True)
    return os.path.join(root, f"{cfg.name}_seed{cfg.seed}.s2v")


def ensure_vocoder(cfg: VocoderConfig, root: str = None):
    path = vocoder_path(cfg, root)
    if os.path.exists(path) and os.path.getsize(path) == _layout(cfg)[2]:
        try:
            if VocoderFile(path).config(cfg.name) == cfg:
                return path
        except Exception:
            pass
    return write_vocoder(cfg, path)


class VocoderFile:
    """Read-only view of a vocoder weight file (memory-mapped)."""

    def __init__(self, path):
        self.path = path
        with open(path, "rb") as f:
            hdr = f.read(HEADER)
            magic, ver, nb = struct.unpack_from("<8sII", hdr, 0)
            if magic != MAGIC or ver != 1 or not 1 <= nb <= MAX_BLOCKS:
                raise ValueError(f"{path}: not a vocoder weight file")
            (self.latent, self.dim, self.cb_dim, self.n_codebooks,
             self.codebook_size) = struct.unpack_from("<5i", hdr, 16)
            self.rates = tuple(struct.unpack_from("<8i", hdr, 36)[:nb])
            n, self.seed, self.data0 = struct.unpack_from("<IIQ", hdr, 68)
            self.entries = {}
            for i in range(n):
                nm, dt, nd, s0, s1, s2, s3, off, nbytes, _ = struct.unpack_from(
                    "<64sII4QQQQ", f.read(ENTRY), 0)
                self.entries[nm.rstrip(b"\0").decode()] = (dt, (s0, s1, s2, s3)[:nd], off, nbytes)

    def config(self, name="file"):
        return VocoderConfig(name=name, latent=self.latent, dim=self.dim, rates=self.rates,
                             cb_dim=self.cb_dim, n_codebooks=self.n_codebooks,
                             codebook_size=self.codebook_size, seed=self.seed)

    def raw(self, name):
        """Stored values: float32 array, or uint16 bf16 bit patterns."""
        dt, shape, off, nbytes = self.entries[name]
        return np.memmap(self.path, dtype=np.uint16 if dt == 1 else np.float32, mode="r",
                         offset=off, shape=tuple(shape))

    def is_bf16(self, name):
        return self.entries[name][0] == 1


def random_codes(cfg: VocoderConfig, batch: int, frames: int, seed: int):
    """Codes [batch, frames, n_codebooks], uniform over [0, codebook_size)."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, cfg.codebook_size, size=(batch, frames, cfg.n_codebooks), dtype=np.int32)
