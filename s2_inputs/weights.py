"""Random-init weight file: format, writer and reader.

Format (little-endian), shared by the oracle reader below and the C++ loader
of the CUDA path, which parses it on its own:

  offset 0   char[8]  magic "S2DUALAR"
         8   u32      version (1)
        12   u32      weight dtype: 0 = f32, 1 = bf16 (matrices and tables;
                      norm gains are always f32)
        16   i32[11]  d, n_heads, n_kv, head_dim, ffn, n_slow, n_fast, vocab,
                      sem_begin, n_codebooks, codebook_size
        60   f32[2]   rms eps, rope theta
        68   u32      n_tensors
        72   u32      seed
        76   u64      data offset (start of the first tensor)
       128   entries  n_tensors x 128 bytes:
                      char name[64], u32 dtype (0 f32, 1 bf16), u32 ndim,
                      u64 shape[4], u64 offset, u64 nbytes, u64 reserved
  Tensors start on 4096-byte boundaries, row-major.

Values: matrices and tables are N(0, 0.02) drawn with
``numpy.random.default_rng([seed, index])`` (PCG64), one stream per tensor in
file order, as float32 and rounded to nearest-even bf16 for bf16 files; norm
gains are 1.0.
"""

import os
import struct
import multiprocessing as mp

import numpy as np

from .config import ModelConfig

MAGIC = b"S2DUALAR"
HEADER = 128
ENTRY = 128
ALIGN = 4096


def tensor_specs(cfg: ModelConfig):
    """List of (name, shape, kind) in file order; kind is 'mat' or 'gain'."""
    d, F, hd = cfg.d, cfg.ffn, cfg.head_dim
    specs = [("tok_emb", (cfg.vocab, d), "mat"),
             ("vq_emb", (cfg.n_codebooks, cfg.codebook_size, d), "mat")]

    def layer(prefix):
        return [(prefix + "attn_norm", (d,), "gain"),
                (prefix + "wq", (cfg.q_dim, d), "mat"),
                (prefix + "wk", (cfg.kv_dim, d), "mat"),
                (prefix + "wv", (cfg.kv_dim, d), "mat"),
                (prefix + "q_norm", (hd,), "gain"),
                (prefix + "k_norm", (hd,), "gain"),
                (prefix + "wo", (d, cfg.q_dim), "mat"),
                (prefix + "mlp_norm", (d,), "gain"),
                (prefix + "wg", (F, d), "mat"),
                (prefix + "wu", (F, d), "mat"),
                (prefix + "wd", (d, F), "mat")]

    for l in range(cfg.n_slow):
        specs += layer(f"slow.{l}.")
    specs.append(("slow.final_norm", (d,), "gain"))
    for l in range(cfg.n_fast):
        specs += layer(f"fast.{l}.")
    specs.append(("fast.final_norm", (d,), "gain"))
    specs.append(("fast.in_emb", (cfg.n_codebooks, cfg.codebook_size, d), "mat"))
    specs.append(("fast.head", (cfg.n_codebooks, cfg.codebook_size, d), "mat"))
    return specs


def _layout(cfg):
    specs = tensor_specs(cfg)
    wbytes = 2 if cfg.wdtype == "bf16" else 4
    off = HEADER + ENTRY * len(specs)
    off = (off + ALIGN - 1) // ALIGN * ALIGN
    data0 = off
    table = []
    for name, shape, kind in specs:
        n = int(np.prod(shape))
        dt = 1 if (kind == "mat" and cfg.wdtype == "bf16") else 0
        nbytes = n * (2 if dt == 1 else 4)
        table.append((name, shape, kind, dt, off, nbytes))
        off = (off + nbytes + ALIGN - 1) // ALIGN * ALIGN
    del wbytes
    return data0, table, off


def _f32_to_bf16_bits(a):
    """Nearest-even rounding of float32 to bf16, returned as uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (r >> np.uint32(16)).astype(np.uint16)


def _gen_tensor(cfg, index, shape, kind):
    if kind == "gain":
        return np.ones(shape, dtype=np.float32)
    rng = np.random.default_rng([cfg.seed, index])
    return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(cfg.init_std)


def _write_one(args):
    path, cfg, index, shape, kind, dt, off, nbytes = args
    a = _gen_tensor(cfg, index, shape, kind)
    mm = np.memmap(path, dtype=np.uint8, mode="r+", offset=off, shape=(nbytes,))
    if dt == 1:
        mm[:] = _f32_to_bf16_bits(a).reshape(-1).view(np.uint8)
    else:
        mm[:] = a.reshape(-1).view(np.uint8)
    mm.flush()
    del mm
    return index


def write_weights(cfg: ModelConfig, path: str, workers: int = 0):
    """Write the random-init weight file of ``cfg`` to ``path``.

    Tensors are generated independently (one seeded stream each), so the
    work is spread over a spawn-started process pool when ``workers`` > 1.
    """
    data0, table, total = _layout(cfg)
    tmp = path + ".tmp"
    with open(tmp, "wb") as f:
        hdr = bytearray(HEADER)
        struct.pack_into("<8sII", hdr, 0, MAGIC, 1, 1 if cfg.wdtype == "bf16" else 0)
        struct.pack_into("<11i", hdr, 16, cfg.d, cfg.n_heads, cfg.n_kv,
                         cfg.head_dim, cfg.ffn, cfg.n_slow, cfg.n_fast,
                         cfg.vocab, cfg.sem_begin, cfg.n_codebooks,
                         cfg.codebook_size)
        struct.pack_into("<ff", hdr, 60, cfg.eps, cfg.rope_theta)
        struct.pack_into("<IIQ", hdr, 68, len(table), cfg.seed, data0)
        f.write(hdr)
        for name, shape, kind, dt, off, nbytes in table:
            e = bytearray(ENTRY)
            nm = name.encode()
            assert len(nm) < 64
            shp = list(shape) + [0] * (4 - len(shape))
            struct.pack_into("<64sII4QQQQ", e, 0, nm, dt, len(shape), *shp,
                             off, nbytes, 0)
            f.write(e)
        f.truncate(total)
    jobs = [(tmp, cfg, i, shape, kind, dt, off, nbytes)
            for i, (name, shape, kind, dt, off, nbytes) in enumerate(table)]
    if workers is None or workers <= 1:
        for j in jobs:
            _write_one(j)
    else:
        ctx = mp.get_context("spawn")
        # biggest tensors first for load balance
        jobs.sort(key=lambda j: -j[7])
        with ctx.Pool(workers) as pool:
            for _ in pool.imap_unordered(_write_one, jobs, chunksize=1):
                pass
    os.replace(tmp, path)
    return path


def weights_path(cfg: ModelConfig, root: str = None):
    root = root or os.environ.get("S2_WEIGHTS_DIR") or os.path.join(
        os.environ.get("TMPDIR", "/tmp"), "s2_weights")
    os.makedirs(root, exist_ok=True)
    return os.path.join(root, f"{cfg.name}_seed{cfg.seed}_{cfg.wdtype}.s2w")


def ensure_weights(cfg: ModelConfig, root: str = None, workers: int = None):
    """Path of the weight file of ``cfg``, writing it first if absent or stale."""
    path = weights_path(cfg, root)
    data0, table, total = _layout(cfg)
    if os.path.exists(path) and os.path.getsize(path) == total:
        try:
            wf = WeightFile(path)
            if wf.cfg_tuple() == _cfg_tuple(cfg):
                return path
        except Exception:
            pass
    if workers is None:
        workers = min(16, os.cpu_count() or 1) if total > (64 << 20) else 1
    return write_weights(cfg, path, workers)


def _cfg_tuple(cfg):
    return (cfg.d, cfg.n_heads, cfg.n_kv, cfg.head_dim, cfg.ffn, cfg.n_slow,
            cfg.n_fast, cfg.vocab, cfg.sem_begin, cfg.n_codebooks,
            cfg.codebook_size, cfg.seed, 1 if cfg.wdtype == "bf16" else 0)


class WeightFile:
    """Read-only view of a weight file (memory-mapped)."""

    def __init__(self, path):
        self.path = path
        with open(path, "rb") as f:
            hdr = f.read(HEADER)
            magic, ver, wdt = struct.unpack_from("<8sII", hdr, 0)
            if magic != MAGIC or ver != 1:
                raise ValueError(f"{path}: not a Dual-AR weight file")
            dims = struct.unpack_from("<11i", hdr, 16)
            self.eps, self.rope_theta = struct.unpack_from("<ff", hdr, 60)
            n, self.seed, self.data0 = struct.unpack_from("<IIQ", hdr, 68)
            (self.d, self.n_heads, self.n_kv, self.head_dim, self.ffn,
             self.n_slow, self.n_fast, self.vocab, self.sem_begin,
             self.n_codebooks, self.codebook_size) = dims
            self.wdtype = "bf16" if wdt == 1 else "f32"
            self.entries = {}
            for i in range(n):
                e = f.read(ENTRY)
                nm, dt, nd, s0, s1, s2, s3, off, nbytes, _ = struct.unpack_from(
                    "<64sII4QQQQ", e, 0)
                name = nm.rstrip(b"\0").decode()
                self.entries[name] = (dt, (s0, s1, s2, s3)[:nd], off, nbytes, i)

    def cfg_tuple(self):
        return (self.d, self.n_heads, self.n_kv, self.head_dim, self.ffn,
                self.n_slow, self.n_fast, self.vocab, self.sem_begin,
                self.n_codebooks, self.codebook_size, self.seed,
                1 if self.wdtype == "bf16" else 0)

    def config(self, name="file"):
        return ModelConfig(name=name, d=self.d, n_heads=self.n_heads,
                           n_kv=self.n_kv, head_dim=self.head_dim, ffn=self.ffn,
                           n_slow=self.n_slow, n_fast=self.n_fast,
                           vocab=self.vocab, sem_begin=self.sem_begin,
                           n_codebooks=self.n_codebooks,
                           codebook_size=self.codebook_size,
                           wdtype=self.wdtype, seed=self.seed,
                           eps=float(self.eps), rope_theta=float(self.rope_theta))

    def raw(self, name):
        """Stored values: float32 array, or uint16 bf16 bit patterns."""
        dt, shape, off, nbytes, _ = self.entries[name]
        return np.memmap(self.path, dtype=np.uint16 if dt == 1 else np.float32,
                         mode="r", offset=off, shape=tuple(shape))

    def is_bf16(self, name):
        return self.entries[name][0] == 1

    def names(self):
        return list(self.entries)
