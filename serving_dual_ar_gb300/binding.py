"""ctypes binding of libs2.so: the C ABI of include/s2.h, include/s2_ops.h
and include/s2_dac.h under the same names.  Argument marshalling only -- every step of the
Dual-AR path runs in the library's CUDA kernels.  There is no fallback: if
the library is missing or fails to load, importing raises.

Array arguments may be numpy arrays (host memory) or torch tensors (host or
CUDA); they are passed by pointer.  Torch CUDA tensors stay on the device.
"""

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("S2_LIB") or os.path.join(HERE, "libs2.so")

S2_OK, S2_EINVAL, S2_ENOMEM, S2_ECUDA, S2_ETIMEOUT, S2_EBADFILE, S2_ESTATE = 0, -1, -2, -3, -4, -5, -6
S2_FLAG_NO_GRAPH, S2_FLAG_NO_TC, S2_FLAG_NO_PDL, S2_FLAG_NO_RADIX, S2_FLAG_INT8 = 1, 2, 4, 8, 16
S2_FLAG_KV_BF16 = 64
S2_FLAG_PERSIST = 128
S2_FLAG_STREAM = 256
S2_FLAG_NO_PREFIX_TC = 512
S2_CODE_EOS = -1


class S2Error(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})")


class s2_opts(C.Structure):
    _fields_ = [("max_seqs", C.c_int32), ("max_batch", C.c_int32),
                ("kv_pool_pages", C.c_int32), ("page_size", C.c_int32),
                ("max_ctx", C.c_int32), ("max_prompt", C.c_int32),
                ("page_perm_seed", C.c_uint64), ("cuda_stream", C.c_void_p),
                ("flags", C.c_int32), ("prefill_rows", C.c_int32), ("reserved", C.c_int32 * 6)]


class s2_stats_t(C.Structure):
    _fields_ = [("prefill_tokens", C.c_int64), ("cached_tokens", C.c_int64),
                ("frames_decoded", C.c_int64), ("pages_used", C.c_int32),
                ("pages_total", C.c_int32), ("radix_pages", C.c_int32),
                ("last_error", C.c_int32), ("device_error", C.c_int32),
                ("num_sms", C.c_int32), ("weight_bytes", C.c_int64),
                ("kernel_launches", C.c_int64), ("evicted_pages", C.c_int64),
                ("reserved", C.c_int64 * 4)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libs2.so not built ({LIB_PATH}); run serving_dual_ar_gb300.build.build()")
    lib = C.CDLL(LIB_PATH, mode=C.RTLD_GLOBAL)
    vp, i32, i64, f32, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t
    sig = {
        "s2_create": (i32, [C.c_char_p, C.POINTER(s2_opts), C.POINTER(vp)]),
        "s2_destroy": (None, [vp]),
        "s2_prefill": (i32, [vp, i32, vp, i32, vp, vp, vp]),
        "s2_prefill_batch": (i32, [vp, i32, vp, vp, vp, vp, vp, vp]),
        "s2_decode_frames": (i32, [vp, vp, i32, i32, vp]),
        "s2_release": (i32, [vp, i32]),
        "s2_radix_clear": (i32, [vp]),
        "s2_stats": (i32, [vp, C.POINTER(s2_stats_t)]),
        "s2_strerror": (C.c_char_p, [i32]),
        "s2_set_debug_sinks": (i32, [vp, vp, vp, vp, i32]),
        "s2_model_dims": (i32, [vp, vp]),
        "s2_set_sampling": (i32, [vp, f32, f32, C.c_uint64]),
        "s2_set_top_p": (i32, [vp, f32, f32]),
        "s2_set_stop": (i32, [vp, i32]),
        "s2op_gemv": (i32, [vp, i32, i32, i32, vp, i32, i32, vp, f32, vp, i32, i32, i32, vp]),
        "s2op_argmax_workspace_bytes": (sz, [i32]),
        "s2op_gemv_argmax": (i32, [vp, i32, i32, i32, vp, i32, i32, vp, f32, vp, vp, vp, vp]),
        "s2op_tc_gemm_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "s2op_tc_gemm_tickets": (sz, [i32, i32]),
        "s2op_tc_gemm": (i32, [vp, i32, i32, vp, i32, i32, vp, i32, vp, i32, i32, i32, vp, vp, vp]),
        "s2op_tc_set_trace": (i32, [vp, i32]),
        "s2op_tc_gemm2_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "s2op_tc_gemm2_tickets": (sz, [i32, i32]),
        "s2op_tc_gemm2": (i32, [vp, i32, i32, vp, vp, i32, i32, vp, i32, vp, vp, i32, i32, i32, vp, vp,
                                vp]),
        "s2op_attn_decode_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "s2op_attn_decode_pick_split": (i32, [i32, i32, i32, i32, i32]),
        "s2op_attn_decode": (i32, [vp, i32, i32, i32, i32, i32, i32, vp, vp, f32, vp, vp, vp, vp,
                                   i32, vp, i32, vp, i32, i32, vp, vp]),
        "s2op_attn_decode_prefix_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "s2op_attn_decode_shared_prefix": (i32, [vp, i32, i32, i32, i32, i32, vp, vp, f32, vp, vp, vp, vp,
                                                 i32, vp, i32, i32, i32, vp, i32, i32, vp, vp]),
        "s2op_attn_prefix_planes": (i32, [vp, i32, vp, i32, i32, i32, i32, vp, vp]),
        "s2op_attn_prefix_set_trace": (i32, [vp, i32]),
        "s2op_attn_prefill": (i32, [vp, i32, i32, i32, i32, i32, i32, vp, vp, f32, vp, vp, vp, i32,
                                    vp, vp, vp, i32, vp]),
        "s2op_rope_table": (i32, [i32, i32, f32, vp, vp]),
        "s2op_stream_read_scratch_bytes": (sz, [i32]),
        "s2op_stream_read": (i32, [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]),
        "s2_vocoder_create": (i32, [C.c_char_p, i32, i32, vp, C.POINTER(vp)]),
        "s2_vocoder_destroy": (None, [vp]),
        "s2_vocoder_hop": (i32, [vp]),
        "s2_vocoder_decode": (i32, [vp, vp, i32, i32, vp]),
        "s2_vocoder_read_stage": (i32, [vp, i32, vp, sz]),
        "s2_vocoder_last_launches": (i64, [vp]),
        "s2_vocoder_set_profile": (i32, [vp, i32]),
        "s2_vocoder_profile": (i32, [vp, vp, i32]),
        "s2op_attn_decode_noalloc_max_bytes": (sz, []),
        "s2op_attn_decode_noalloc": (i32, [vp, i32, i32, i32, i32, i32, i32, vp, vp, f32, vp, vp, vp,
                                           vp, i32, vp, i32, vp, i32, i32, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()
EXPORTED = sorted(n for n in dir(LIB) if n.startswith("s2"))


def strerror(status):
    return LIB.s2_strerror(int(status)).decode()


def ptr(a):
    """Raw pointer of a numpy array / torch tensor (None -> NULL)."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be C-contiguous")
        return a.ctypes.data
    raise TypeError(f"cannot pass {type(a)} by pointer")


def _check(s, what):
    if s != S2_OK:
        raise S2Error(s, what)
    return s


def _stream(stream):
    if stream is None:
        return None
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


# ---------------------------------------------------------------- model ABI

def s2_create(weights_path, max_seqs=64, max_batch=128, kv_pool_pages=0, max_ctx=2048,
              max_prompt=0, page_perm_seed=0, stream=None, flags=0, prefill_rows=0):
    o = s2_opts()
    o.max_seqs, o.max_batch, o.kv_pool_pages, o.page_size = max_seqs, max_batch, kv_pool_pages, 16
    o.max_ctx, o.max_prompt, o.page_perm_seed = max_ctx, max_prompt, page_perm_seed
    o.prefill_rows = prefill_rows
    o.cuda_stream, o.flags = _stream(stream), flags
    h = C.c_void_p()
    _check(LIB.s2_create(os.fsencode(weights_path), C.byref(o), C.byref(h)), "s2_create")
    return h.value


def s2_destroy(ctx):
    LIB.s2_destroy(ctx)


def s2_prefill(ctx, seq, tokens, vq_codes=None, vq_mask=None):
    """tokens int32 [T]; vq_codes int32 [10, T]; vq_mask uint8 [T]. Returns cached length."""
    T = int(tokens.shape[0])
    cached = C.c_int32(0)
    _check(LIB.s2_prefill(ctx, int(seq), ptr(tokens), T, ptr(vq_codes), ptr(vq_mask),
                          C.addressof(cached)), "s2_prefill")
    return cached.value


def s2_prefill_batch(ctx, seqs, prompts):
    """Prefill several free sequences in one call.  ``prompts``: list of
    (tokens, vq_codes [n_codebooks, T] or None, vq_mask [T] or None) host
    arrays, one per sequence.  Returns the cached positions per prompt."""
    n = len(seqs)
    lens = np.array([len(p[0]) for p in prompts], np.int32)
    toks = np.ascontiguousarray(np.concatenate([np.asarray(p[0], np.int32) for p in prompts]))
    any_mask = any(p[2] is not None for p in prompts)
    codes = mask = None
    if any_mask:
        nc = next(np.asarray(p[1]).shape[0] for p in prompts if p[1] is not None)
        blocks, masks = [], []
        for (t, c, m) in prompts:
            T = len(t)
            blocks.append(np.asarray(c, np.int32).reshape(nc, T) if c is not None else np.zeros((nc, T), np.int32))
            masks.append(np.asarray(m, np.uint8) if m is not None else np.zeros(T, np.uint8))
        codes = np.ascontiguousarray(np.concatenate([b.reshape(-1) for b in blocks]))
        mask = np.ascontiguousarray(np.concatenate(masks))
    cached = np.zeros(n, np.int32)
    _check(LIB.s2_prefill_batch(ctx, n, ptr(np.ascontiguousarray(seqs, dtype=np.int32)), ptr(toks), ptr(lens),
                                ptr(codes), ptr(mask), ptr(cached)), "s2_prefill_batch")
    return cached


def s2_decode_frames(ctx, seqs, n, out=None):
    """Decode n frames for each sequence id in ``seqs``; returns int32 [B, n, 10]."""
    seqs = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32)) if not hasattr(seqs, "data_ptr") else seqs
    B = int(seqs.shape[0])
    if out is None:
        out = np.zeros((B, n, 10), np.int32)
    _check(LIB.s2_decode_frames(ctx, ptr(seqs), B, int(n), ptr(out)), "s2_decode_frames")
    return out


def s2_release(ctx, seq):
    _check(LIB.s2_release(ctx, int(seq)), "s2_release")


def s2_radix_clear(ctx):
    _check(LIB.s2_radix_clear(ctx), "s2_radix_clear")


def s2_stats(ctx):
    st = s2_stats_t()
    _check(LIB.s2_stats(ctx, C.byref(st)), "s2_stats")
    return {f: getattr(st, f) for f, _ in s2_stats_t._fields_ if f != "reserved"}


def s2_set_debug_sinks(ctx, logits=None, hidden=None, layers=None, max_frames=0):
    _check(LIB.s2_set_debug_sinks(ctx, ptr(logits), ptr(hidden), ptr(layers), int(max_frames)),
           "s2_set_debug_sinks")


def s2_set_sampling(ctx, temperature_slow=0.0, temperature_fast=0.0, seed=0):
    _check(LIB.s2_set_sampling(ctx, float(temperature_slow), float(temperature_fast), int(seed)),
           "s2_set_sampling")


def s2_set_top_p(ctx, top_p_slow=1.0, top_p_fast=1.0):
    _check(LIB.s2_set_top_p(ctx, float(top_p_slow), float(top_p_fast)), "s2_set_top_p")


def s2_set_stop(ctx, eos_token=-1):
    _check(LIB.s2_set_stop(ctx, int(eos_token)), "s2_set_stop")


def s2_model_dims(ctx):
    d = np.zeros(12, np.int32)
    _check(LIB.s2_model_dims(ctx, ptr(d)), "s2_model_dims")
    keys = ["d", "n_heads", "n_kv", "head_dim", "ffn", "n_slow", "n_fast", "vocab",
            "sem_begin", "n_codebooks", "codebook_size", "wbf16"]
    return dict(zip(keys, d.tolist()))


# ---------------------------------------------------------------- op ABI

def s2op_gemv(W, N, K, X, ldx, B, Y, ldy, mode=0, gain=None, eps=1e-6, w_bf16=True, grid=0,
              stream=None):
    _check(LIB.s2op_gemv(ptr(W), int(w_bf16), N, K, ptr(X), ldx, B, ptr(gain), eps, ptr(Y), ldy,
                         mode, grid, _stream(stream)), "s2op_gemv")


def s2op_argmax_workspace_bytes(B):
    return LIB.s2op_argmax_workspace_bytes(B)


def s2op_gemv_argmax(W, N, K, X, ldx, B, codes, workspace, logits=None, gain=None, eps=1e-6,
                     w_bf16=True, stream=None):
    _check(LIB.s2op_gemv_argmax(ptr(W), int(w_bf16), N, K, ptr(X), ldx, B, ptr(gain), eps,
                                ptr(codes), ptr(logits), ptr(workspace), _stream(stream)),
           "s2op_gemv_argmax")


def s2op_tc_gemm_workspace_bytes(N, K, T, split_k=0):
    return LIB.s2op_tc_gemm_workspace_bytes(N, K, T, split_k)


def s2op_tc_gemm_tickets(N, T):
    return LIB.s2op_tc_gemm_tickets(N, T)


def s2op_tc_gemm(A, N, K, Bm, T, ldb, Y=None, ldy=0, Y16=None, ldy16=0, epi=0, split_k=0,
                 workspace=None, tickets=None, stream=None):
    _check(LIB.s2op_tc_gemm(ptr(A), N, K, ptr(Bm), T, ldb, ptr(Y), ldy, ptr(Y16), ldy16, epi,
                            split_k, ptr(workspace), ptr(tickets), _stream(stream)), "s2op_tc_gemm")


def s2op_tc_gemm2_workspace_bytes(N, K, T, split_k=0):
    return LIB.s2op_tc_gemm2_workspace_bytes(N, K, T, split_k)


def s2op_tc_gemm2_tickets(N, T):
    return LIB.s2op_tc_gemm2_tickets(N, T)


def s2op_tc_gemm2(A, N, K, Bhi, Blo, T, ldb, Y=None, ldy=0, Y16=None, Y16lo=None, ldy16=0, epi=0,
                  split_k=0, workspace=None, tickets=None, stream=None):
    _check(LIB.s2op_tc_gemm2(ptr(A), N, K, ptr(Bhi), ptr(Blo), T, ldb, ptr(Y), ldy, ptr(Y16),
                             ptr(Y16lo), ldy16, epi, split_k, ptr(workspace), ptr(tickets),
                             _stream(stream)), "s2op_tc_gemm2")


def s2op_tc_set_trace(buf, max_ctas):
    """K2 phase trace into ``buf`` (device uint64 [max_ctas, 6]); 0 turns it off."""
    _check(LIB.s2op_tc_set_trace(ptr(buf), max_ctas), "s2op_tc_set_trace")


def s2op_attn_decode_pick_split(B, H, Hkv, hd, kv_bf16=False):
    n = LIB.s2op_attn_decode_pick_split(B, H, Hkv, hd, int(kv_bf16))
    if n < 1:
        raise S2Error(n, "s2op_attn_decode_pick_split")
    return n


def s2op_attn_decode_workspace_bytes(B, m, H, Hkv, hd, nsplit):
    return LIB.s2op_attn_decode_workspace_bytes(B, m, H, Hkv, hd, nsplit)


def s2op_attn_decode(qkv, qkv_ld, B, m, H, Hkv, hd, q_gain, k_gain, eps, rope_cos, rope_sin, pos,
                     kv, kv_bf16, table, table_ld, o, o_ld, nsplit=1, workspace=None, stream=None):
    _check(LIB.s2op_attn_decode(ptr(qkv), qkv_ld, B, m, H, Hkv, hd, ptr(q_gain), ptr(k_gain), eps,
                                ptr(rope_cos), ptr(rope_sin), ptr(pos), ptr(kv), int(kv_bf16),
                                ptr(table), table_ld, ptr(o), o_ld, nsplit, ptr(workspace),
                                _stream(stream)), "s2op_attn_decode")


def s2op_attn_decode_prefix_workspace_bytes(B, H, Hkv, hd, nsplit, max_keys):
    return LIB.s2op_attn_decode_prefix_workspace_bytes(B, H, Hkv, hd, nsplit, max_keys)


def s2op_attn_decode_shared_prefix(qkv, qkv_ld, B, H, Hkv, hd, q_gain, k_gain, eps, rope_cos, rope_sin,
                                   pos, kv, kv_bf16, table, table_ld, shared_len, max_keys, o, o_ld,
                                   nsplit=1, workspace=None, stream=None):
    _check(LIB.s2op_attn_decode_shared_prefix(ptr(qkv), qkv_ld, B, H, Hkv, hd, ptr(q_gain), ptr(k_gain), eps,
                                              ptr(rope_cos), ptr(rope_sin), ptr(pos), ptr(kv), int(kv_bf16),
                                              ptr(table), table_ld, shared_len, max_keys, ptr(o), o_ld,
                                              nsplit, ptr(workspace), _stream(stream)),
           "s2op_attn_decode_shared_prefix")


def s2op_attn_prefix_set_trace(buf, max_ctas):
    _check(LIB.s2op_attn_prefix_set_trace(ptr(buf), max_ctas), "s2op_attn_prefix_set_trace")


def s2op_attn_prefix_planes(kv, kv_bf16, table, Hkv, hd, shared_len, max_keys, workspace, stream=None):
    _check(LIB.s2op_attn_prefix_planes(ptr(kv), int(kv_bf16), ptr(table), Hkv, hd, shared_len, max_keys,
                                       ptr(workspace), _stream(stream)), "s2op_attn_prefix_planes")


def s2op_attn_prefill(qkv, qkv_ld, T, pos0, H, Hkv, hd, q_gain, k_gain, eps, rope_cos, rope_sin,
                      kv, kv_bf16, table, q_scratch, o, o_ld, stream=None):
    _check(LIB.s2op_attn_prefill(ptr(qkv), qkv_ld, T, pos0, H, Hkv, hd, ptr(q_gain), ptr(k_gain),
                                 eps, ptr(rope_cos), ptr(rope_sin), ptr(kv), int(kv_bf16),
                                 ptr(table), ptr(q_scratch), ptr(o), o_ld, _stream(stream)),
           "s2op_attn_prefill")


def s2op_stream_read_scratch_bytes(n_ops):
    return LIB.s2op_stream_read_scratch_bytes(n_ops)


def s2op_stream_read(bufs, nbytes, scratch, reps=1, mode=0, chunk_bytes=16384, stages=12, barrier=0,
                     stream=None):
    """Read-bandwidth calibration stream over device buffers; returns the
    kernel's error word for mode 1 (synchronising), else 0."""
    n = len(bufs)
    pa = (C.c_void_p * n)(*[ptr(x) for x in bufs])
    ba = (C.c_ulonglong * n)(*[int(x) for x in nbytes])
    err = C.c_int(0)
    _check(LIB.s2op_stream_read(pa, ba, n, reps, mode, chunk_bytes, stages, barrier, ptr(scratch),
                                C.byref(err) if mode == 1 else None, _stream(stream)),
           "s2op_stream_read")
    return err.value


def s2op_rope_table(n_pos, hd, theta):
    cs = np.zeros((n_pos, hd // 2), np.float32)
    sn = np.zeros((n_pos, hd // 2), np.float32)
    _check(LIB.s2op_rope_table(n_pos, hd, theta, ptr(cs), ptr(sn)), "s2op_rope_table")
    return cs, sn


# ---------------------------------------------------------------- vocoder ABI (s2_dac.h)

def s2_vocoder_create(path, max_seqs, max_frames, stream=None):
    h = C.c_void_p()
    _check(LIB.s2_vocoder_create(os.fsencode(path), max_seqs, max_frames, _stream(stream), C.byref(h)),
           "s2_vocoder_create")
    return h


def s2_vocoder_destroy(v):
    LIB.s2_vocoder_destroy(v)


def s2_vocoder_hop(v):
    return LIB.s2_vocoder_hop(v)


def s2_vocoder_decode(v, codes, out=None):
    """codes int32 [batch, n, n_codebooks] (numpy or torch, host or CUDA) ->
    waveform float32 [batch, n * hop] (``out`` if given, else a new numpy
    array)."""
    if isinstance(codes, np.ndarray):
        codes = np.ascontiguousarray(codes, dtype=np.int32)
    B, n = int(codes.shape[0]), int(codes.shape[1])
    if out is None:
        out = np.zeros((B, n * s2_vocoder_hop(v)), np.float32)
    _check(LIB.s2_vocoder_decode(v, ptr(codes), B, n, ptr(out)), "s2_vocoder_decode")
    return out


def s2_vocoder_read_stage(v, stage, batch, T, channels):
    """Intermediate activation of the last decode as float32 [batch, T, channels]."""
    a = np.zeros((batch, T, channels), np.float32)
    _check(LIB.s2_vocoder_read_stage(v, stage, ptr(a), a.nbytes), "s2_vocoder_read_stage")
    return a


def s2_vocoder_last_launches(v):
    return LIB.s2_vocoder_last_launches(v)


def s2_vocoder_set_profile(v, on=True):
    _check(LIB.s2_vocoder_set_profile(v, int(bool(on))), "s2_vocoder_set_profile")


def s2_vocoder_profile(v, max_launches=256):
    """Per-launch durations (ms) of the last decode, in launch order."""
    a = np.zeros(max_launches, np.float32)
    n = LIB.s2_vocoder_profile(v, ptr(a), max_launches)
    if n < 0:
        raise S2Error(n, "s2_vocoder_profile")
    return a[:n].copy()
