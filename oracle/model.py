"""Dual-AR oracle: the plain definition of prefill and greedy frame decode.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain NumPy, in the
floating type the caller picks (float32 as the benchmark asks for the
full-size runs, float64 for the small brute-force pins).  No blocking or
fusion: every step is the textbook operation, in the order the pages give.

What is computed, per frame (see "s2pro-native", What happens to a sentence:
a 36-layer backbone picks one semantic token, a 4-layer decoder then emits
the residual codes greedily; "Fish Audio Abre Código do S2", Arquitetura
Dual-AR: the Slow AR runs along time and predicts the semantic codebook, the
Fast AR emits the 9 residual codebooks of each time step):

  1. Slow AR step on the previous frame's input embedding (the first frame
     after a prefill uses the prefill's last hidden state instead).
  2. Final RMSNorm -> h; logits over the tied embedding, restricted to the
     semantic ids ("constrained decoding", SGLang page, Background); the
     argmax s gives code 0 = s - sem_begin.
  3. Fast AR over depth positions 0..9: position 0 is h, position j (1..9)
     is the Fast AR input table j-1 at code j-1; the output at position j,
     after the fast final RMSNorm, is read by head slice j; its argmax is
     code j.  KV is fresh every frame.
  4. The next Slow AR input is E_tok[s] + sum_k E_vq[k, code_k] (SGLang
     page, Background: VQ codebook embeddings are interleaved into the token
     stream during decoding; Architecture: VQ embeddings are added to the
     input embedding at masked positions).

Readings where the pages are silent:
  * Layer: Qwen3-style pre-norm GQA block -- RMSNorm, q/k/v projections,
    per-head RMSNorm of q and k with gains shared across heads, RoPE
    (rotate-half pairing, theta 1e6), causal softmax attention with scale
    1/sqrt(head_dim) where q head h reads kv head h // (H / Hkv), output
    projection and residual; RMSNorm, SwiGLU MLP (silu(gate) * up, then down)
    and residual.  No biases.  RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g.
  * RoPE table: angle p * theta^(-2i/hd) in float64, cos/sin rounded to
    float32 and then to bf16 (nearest even) and used as float32 (SGLang
    page, Engineering Appendix "BF16 RoPE Precision Mismatch": the model was
    trained with bf16 RoPE, and the fix casts the float32 cos/sin cache to
    bf16 and back).
  * Fast AR input tables and heads are per codebook: in_emb[10, C, d] (input
    of position j uses table j-1) and head[10, C, d] (code j uses slice j;
    slice 0 and table 9 are never read).
  * Greedy ties go to the lowest index (NumPy argmax).
"""

import math

import numpy as np

from s2_inputs import WeightFile
from .radix import RadixCache, position_keys
from .sampling import sample, pick

TEST_ONLY = True


# --------------------------------------------------------------------------
# Elementary operations


def bf16_round(a):
    """Round to float32, then to the nearest bf16 value (ties to even).

    Returns float32 values that are exactly representable in bf16.  Follows
    the bf16 cast of the SGLang page's RoPE fix (Engineering Appendix).
    """
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).reshape(f.shape)


def rms_norm(x, g, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g."""
    dt = x.dtype
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return (x / np.sqrt(ms + dt.type(eps))) * g.astype(dt)


def rope_table(n_pos, head_dim, theta, to_bf16=True):
    """cos and sin tables [n_pos, head_dim/2] for rotate-half RoPE.

    Angles p * theta^(-2i/head_dim) in float64.  With ``to_bf16`` the values
    go float64 -> float32 -> bf16, as the SGLang page's appendix prescribes
    for S2; otherwise they stay float64 (used by the exactness pins).
    """
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    c, s = np.cos(ang), np.sin(ang)
    if to_bf16:
        return bf16_round(c), bf16_round(s)
    return c, s


def apply_rope(x, cos, sin):
    """Rotate-half RoPE: pairs (x[i], x[i + hd/2]) rotate by the angle of i.

    ``cos``/``sin`` broadcast against x[..., :hd/2].
    """
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    c = cos.astype(x.dtype)
    s = sin.astype(x.dtype)
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(s, axis=-1):
    """exp(s - max) / sum; -inf entries get probability 0."""
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def gqa_attention(q, K, V, q_pos, return_probs=False):
    """Causal grouped-query attention.

    q [m, H, hd] at absolute positions q_pos [m]; K, V [Hkv, n, hd] hold keys
    at positions 0..n-1.  Query head h reads kv head h // (H / Hkv); query i
    sees keys j <= q_pos[i].  Scores are scaled by 1/sqrt(hd).
    """
    m, H, hd = q.shape
    Hkv, n, _ = K.shape
    group = H // Hkv
    scale = q.dtype.type(1.0 / math.sqrt(hd))
    visible = np.arange(n)[None, :] <= np.asarray(q_pos)[:, None]     # [m, n]
    out = np.empty_like(q)
    probs = np.empty((H, m, n), dtype=q.dtype) if return_probs else None
    for h in range(H):
        g = h // group
        s = (q[:, h, :] @ K[g].T) * scale                               # [m, n]
        s = np.where(visible, s, -np.inf)
        p = softmax(s, axis=-1)
        out[:, h, :] = p @ V[g]
        if return_probs:
            probs[h] = p
    return (out, probs) if return_probs else out


def silu(z):
    """z * sigmoid(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (z.dtype.type(1.0) + np.exp(-z))


def swiglu(gate, up):
    """SwiGLU activation: silu(gate) * up."""
    return silu(gate) * up


def masked_argmax(logits, allowed):
    """Greedy pick among allowed entries; ties -> lowest index."""
    return int(np.argmax(np.where(allowed, logits, -np.inf)))


# --------------------------------------------------------------------------
# Weights


def _widen(raw, is_bf16, dtype):
    if is_bf16:
        a = (np.asarray(raw).astype(np.uint32) << np.uint32(16)).view(np.float32)
        return a.astype(dtype, copy=False)
    return np.asarray(raw, dtype=np.float32).astype(dtype)


def quantize_rows_int8(w):
    """Symmetric per-output-channel INT8 ("s2pro-native", The gate that says
    no: INT8 with per-channel weight scales is the 8-bit candidate).

    For each row n: scale_n = max_k |w[n,k]| / 127 (float32; 1 for an all-zero
    row), q[n,k] = round-half-even(w[n,k] / scale_n) clipped to [-127, 127].
    Returns (q int8 [N, K], scale float32 [N]).
    """
    w = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w), axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
    q = np.clip(np.rint(w / scale[..., None]), -127, 127).astype(np.int8)
    return q, scale


def dequantize_rows_int8(q, scale):
    return q.astype(np.float32) * scale[..., None]


class OracleWeights:
    """All tensors of a weight file, widened exactly to ``dtype``.

    With ``quant="int8"`` every matrix the decode streams -- the layer
    projections of both stacks, the semantic slice of the tied embedding used
    as the head and the Fast AR head slices -- is replaced by its per-row INT8
    quantisation (dequantised values); gathered tables stay as stored.
    """

    LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
                  "mlp_norm", "wg", "wu", "wd")
    MATS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")

    def __init__(self, src, dtype=np.float32, overrides=None, quant=None):
        wf = src if isinstance(src, WeightFile) else WeightFile(src)
        self.cfg = wf.config()
        self.dtype = dtype
        self.quant = quant
        self.t = {}
        for name in wf.names():
            self.t[name] = _widen(wf.raw(name), wf.is_bf16(name), dtype)
        for k, v in (overrides or {}).items():
            self.t[k] = np.asarray(v, dtype=dtype)
        self.sem_head = None
        if quant == "int8":
            cfg = self.cfg
            for stack, n in (("slow", cfg.n_slow), ("fast", cfg.n_fast)):
                for l in range(n):
                    for m in self.MATS:
                        k = f"{stack}.{l}.{m}"
                        self.t[k] = dequantize_rows_int8(*quantize_rows_int8(self.t[k])).astype(dtype)
            self.t["fast.head"] = dequantize_rows_int8(
                *quantize_rows_int8(self.t["fast.head"])).astype(dtype)
            self.sem_head = dequantize_rows_int8(
                *quantize_rows_int8(self.t["tok_emb"][cfg.sem_begin:])).astype(dtype)
        elif quant is not None:
            raise ValueError(f"unknown quantisation {quant}")

    def head_rows(self):
        """The semantic rows the slow head reads."""
        if self.sem_head is not None:
            return self.sem_head
        return self.t["tok_emb"][self.cfg.sem_begin:]

    def layer(self, stack, l):
        return {k: self.t[f"{stack}.{l}.{k}"] for k in self.LAYER_KEYS}


# --------------------------------------------------------------------------
# KV stores


class ContiguousKV:
    """Per-sequence KV as growing arrays [Hkv, n, hd] per layer."""

    def __init__(self, n_layers, n_kv, hd, dtype, cap=64):
        self.K = [np.zeros((n_kv, cap, hd), dtype) for _ in range(n_layers)]
        self.V = [np.zeros((n_kv, cap, hd), dtype) for _ in range(n_layers)]

    def _grow(self, l, n):
        cap = self.K[l].shape[1]
        if n <= cap:
            return
        new = max(n, 2 * cap)
        for arrs in (self.K, self.V):
            a = arrs[l]
            b = np.zeros((a.shape[0], new, a.shape[2]), a.dtype)
            b[:, :cap] = a
            arrs[l] = b

    def write(self, l, pos, k, v):
        pos = np.asarray(pos)
        self._grow(l, int(pos.max()) + 1)
        self.K[l][:, pos, :] = np.transpose(k, (1, 0, 2))
        self.V[l][:, pos, :] = np.transpose(v, (1, 0, 2))

    def read(self, l, n):
        return self.K[l][:, :n], self.V[l][:, :n]


class PagedKV:
    """A shared pool of fixed-size pages [L][pages][2][Hkv][P][hd].

    Free physical pages are handed out in a seeded random order when
    ``perm_seed`` is given (scattered pages), else in ascending order.
    Pages carry reference counts (sequences and the radix tree).
    """

    def __init__(self, n_layers, n_kv, hd, n_pages, dtype, page=16, perm_seed=None):
        self.P = page
        self.pool = np.zeros((n_layers, n_pages, 2, n_kv, page, hd), dtype)
        order = (np.random.default_rng(perm_seed).permutation(n_pages)
                 if perm_seed is not None else np.arange(n_pages))
        self.free = [int(p) for p in order[::-1]]          # pop() from the end
        self.ref = np.zeros(n_pages, np.int64)

    def alloc(self):
        if not self.free:
            raise MemoryError("KV pool exhausted")
        p = self.free.pop()
        self.ref[p] = 1
        return p

    def incref(self, p):
        self.ref[p] += 1

    def decref(self, p):
        self.ref[p] -= 1
        if self.ref[p] == 0:
            self.free.append(int(p))

    def view(self, table):
        return _PageView(self, table)


class _PageView:
    """One sequence's view of a PagedKV through its page table."""

    def __init__(self, kv, table):
        self.kv, self.table = kv, table

    def write(self, l, pos, k, v):
        P = self.kv.P
        for i, p in enumerate(np.asarray(pos).tolist()):
            page = self.table[p // P]
            self.kv.pool[l, page, 0, :, p % P, :] = k[i]
            self.kv.pool[l, page, 1, :, p % P, :] = v[i]

    def read(self, l, n):
        P = self.kv.P
        pages = self.table[: -(-n // P)]
        blk = self.kv.pool[l, pages]                        # [np, 2, Hkv, P, hd]
        K = np.concatenate(list(blk[:, 0]), axis=1)[:, :n]
        V = np.concatenate(list(blk[:, 1]), axis=1)[:, :n]
        return K, V


# --------------------------------------------------------------------------
# Embeddings


def embed_prompt(w, tokens, codes, mask):
    """Input embedding of prompt positions.

    e_t = E_tok[tok_t] + mask_t * sum_{k<10} E_vq[k, codes[k, t]]
    (SGLang page, Architecture: VQ embeddings are injected into the input
    embedding at masked positions.)
    """
    cfg = w.cfg
    e = w.t["tok_emb"][np.asarray(tokens)].copy()
    if mask is not None:
        for t in np.nonzero(np.asarray(mask))[0]:
            for k in range(cfg.n_codebooks):
                e[t] += w.t["vq_emb"][k, int(codes[k, t])]
    return e


def feedback_embedding(w, frame_codes):
    """Slow AR input for the step after a frame: the frame re-enters the
    stream as a VQ position whose token is the semantic id sem_begin + code 0
    (SGLang page, Background: VQ codebook embeddings are interleaved into the
    token stream during decoding)."""
    cfg = w.cfg
    e = w.t["tok_emb"][cfg.sem_begin + int(frame_codes[0])].copy()
    for k in range(cfg.n_codebooks):
        e += w.t["vq_emb"][k, int(frame_codes[k])]
    return e


# --------------------------------------------------------------------------
# The model


class _Seq:
    __slots__ = ("table", "length", "h_last", "last", "kv", "finished")

    def __init__(self):
        self.table, self.length, self.h_last, self.last, self.kv = [], 0, None, None, None
        self.finished = False


class DualAROracle:
    """Prefill + greedy Dual-AR decode over a paged (or contiguous) KV cache.

    ``paged`` selects the page pool (with optional scattered page order and
    radix prefix sharing) or one contiguous KV per sequence.
    """

    def __init__(self, weights, paged=True, pool_pages=256, page=16,
                 perm_seed=None, radix=True, record=False, sampling=None, eos=None):
        # sampling: None (greedy) or (temperature_slow, temperature_fast, seed)
        # with optional (top_p_slow, top_p_fast) appended (1.0 = no filter).
        # eos: None, or the token id whose tied-embedding row joins the Slow
        # head's constrained set; a frame that picks it ends the sequence.
        self.sampling = sampling
        self.eos = eos
        self.w = weights
        self.cfg = weights.cfg
        self.dt = weights.dtype
        self.paged = paged
        self.page = page
        cfg = self.cfg
        if paged:
            self.kv = PagedKV(cfg.n_slow, cfg.n_kv, cfg.head_dim, pool_pages,
                              self.dt, page, perm_seed)
        self.radix = RadixCache(page) if (paged and radix) else None
        self.seqs = {}
        self.record = record
        self.log = []                      # per-frame records when ``record``
        self._rope_n = 0
        self._grow_rope(2048)

    # ---- helpers -----------------------------------------------------------

    def _grow_rope(self, n):
        if n <= self._rope_n:
            return
        n = max(n, 2 * self._rope_n)
        self.cos, self.sin = rope_table(n, self.cfg.head_dim, self.cfg.rope_theta)
        self._rope_n = n

    def _layer(self, lw, x, pos, views, l):
        """One transformer block on rows x [m, d]; row i sits at position
        pos[i] of the sequence whose KV view is views[i]."""
        cfg, dt = self.cfg, self.dt
        m = x.shape[0]
        H, Hkv, hd = cfg.n_heads, cfg.n_kv, cfg.head_dim
        pos = np.asarray(pos)
        self._grow_rope(int(pos.max()) + 1)
        a = rms_norm(x, lw["attn_norm"], cfg.eps)
        q = (a @ lw["wq"].T).reshape(m, H, hd)
        k = (a @ lw["wk"].T).reshape(m, Hkv, hd)
        v = (a @ lw["wv"].T).reshape(m, Hkv, hd)
        q = rms_norm(q, lw["q_norm"], cfg.eps)
        k = rms_norm(k, lw["k_norm"], cfg.eps)
        c, s = self.cos[pos][:, None, :], self.sin[pos][:, None, :]
        q = apply_rope(q, c, s)
        k = apply_rope(k, c, s)
        # store this call's keys and values, then attend per sequence
        groups = {}
        for i, vw in enumerate(views):
            groups.setdefault(id(vw), (vw, []))[1].append(i)
        for vw, rows in groups.values():
            vw.write(l, pos[rows], k[rows], v[rows])
        o = np.empty_like(q)
        for vw, rows in groups.values():
            K, V = vw.read(l, int(pos[rows].max()) + 1)
            o[rows] = gqa_attention(q[rows], K, V, pos[rows])
        x = x + o.reshape(m, H * hd) @ lw["wo"].T
        h = rms_norm(x, lw["mlp_norm"], cfg.eps)
        x = x + swiglu(h @ lw["wg"].T, h @ lw["wu"].T) @ lw["wd"].T
        return x

    def slow_forward(self, x, pos, views, capture=None):
        for l in range(self.cfg.n_slow):
            x = self._layer(self.w.layer("slow", l), x, pos, views, l)
            if capture is not None:
                capture.append(x.copy())
        return x

    def slow_head(self, h):
        """Tied-embedding logits over the full vocabulary, restricted to the
        semantic ids; returns (semantic id, code 0, semantic-slice logits)."""
        cfg = self.cfg
        if self.w.sem_head is not None:        # INT8 head: only the semantic rows exist
            logits = np.full(cfg.vocab, -np.inf, dtype=self.dt)
            logits[cfg.sem_begin:] = self.w.sem_head @ h
        else:
            logits = self.w.t["tok_emb"] @ h
        allowed = np.arange(cfg.vocab) >= cfg.sem_begin
        s = masked_argmax(logits, allowed)
        return s, s - cfg.sem_begin, logits[cfg.sem_begin:]

    def _pick(self, logits, codebook, seq, pos):
        if self.sampling is None:
            return int(np.argmax(logits))
        t_slow, t_fast, seed = self.sampling[:3]
        p_slow, p_fast = self.sampling[3:5] if len(self.sampling) >= 5 else (1.0, 1.0)
        if codebook == 0:
            return pick(logits, t_slow, p_slow, seed, seq, pos, 0)
        return pick(logits, t_fast, p_fast, seed, seq, pos, codebook)

    def eos_logit(self, h):
        """Logit of the end-of-speech row (bf16 tied embedding row . h)."""
        return np.float32(self.w.t["tok_emb"][self.eos] @ h)

    def fast_frame(self, h, code0, seq=0, pos=0):
        """The Fast AR depth loop for one frame, with its own fresh KV."""
        cfg = self.cfg
        kv = ContiguousKV(cfg.n_fast, cfg.n_kv, cfg.head_dim, self.dt, cap=16)
        views = [kv]
        x = h[None, :].astype(self.dt)
        for l in range(cfg.n_fast):                     # position 0: h
            x = self._layer(self.w.layer("fast", l), x, [0], views, l)
        codes, logits = [code0], []
        for j in range(1, cfg.n_codebooks):             # positions 1..9
            x = self.w.t["fast.in_emb"][j - 1, codes[j - 1]][None, :].copy()
            for l in range(cfg.n_fast):
                x = self._layer(self.w.layer("fast", l), x, [j], views, l)
            y = rms_norm(x[0], self.w.t["fast.final_norm"], cfg.eps)
            lg = self.w.t["fast.head"][j] @ y
            codes.append(self._pick(lg, j, seq, pos))
            logits.append(lg)
        return codes, logits

    # ---- sequence API ------------------------------------------------------

    def _ensure_pages(self, st, n_positions):
        while len(st.table) * self.page < n_positions:
            st.table.append(self.kv.alloc())

    def prefill(self, seq, tokens, codes, mask):
        """Prefill a prompt; returns the number of positions reused from the
        radix cache (a multiple of the page size, at most T-1)."""
        cfg = self.cfg
        T = len(tokens)
        st = _Seq()
        P = 0
        keys = None
        if self.paged:
            if self.radix is not None:
                keys = position_keys(tokens, codes, mask)
                hit = self.radix.match(keys, (T - 1) // self.page)
                for p in hit:
                    self.kv.incref(p)
                st.table = list(hit)
                P = len(hit) * self.page
            self._ensure_pages(st, T)
            st.kv = self.kv.view(st.table)
        else:
            st.kv = ContiguousKV(cfg.n_slow, cfg.n_kv, cfg.head_dim, self.dt)
        e = embed_prompt(self.w, tokens[P:], None if codes is None else codes[:, P:],
                         None if mask is None else mask[P:])
        x = self.slow_forward(e, np.arange(P, T), [st.kv] * (T - P))
        st.h_last = rms_norm(x[-1], self.w.t["slow.final_norm"], cfg.eps)
        st.length = T
        if self.radix is not None:
            for p in self.radix.insert(keys, st.table):
                self.kv.incref(p)
        self.seqs[seq] = st
        return P

    def release(self, seq):
        st = self.seqs.pop(seq)
        if self.paged:
            for p in st.table:
                self.kv.decref(p)

    def decode_frames(self, seqs, n):
        """n frames for each sequence; returns int32 [B, n, 10].  A sequence
        that picked EOS emits -1 codes from that frame on (it is finished)."""
        cfg = self.cfg
        B = len(seqs)
        out = np.zeros((B, n, cfg.n_codebooks), np.int32)
        for f in range(n):
            sts = [self.seqs[s] for s in seqs]
            # slow step for sequences that already emitted a frame
            rows = [b for b, st in enumerate(sts) if st.last is not None and not st.finished]
            hs = [st.h_last for st in sts]
            if rows:
                e = np.stack([feedback_embedding(self.w, sts[b].last) for b in rows])
                pos = np.array([sts[b].length for b in rows])
                for b in rows:
                    if self.paged:
                        self._ensure_pages(sts[b], sts[b].length + 1)
                x = self.slow_forward(e, pos, [sts[b].kv for b in rows])
                for i, b in enumerate(rows):
                    sts[b].length += 1
                    hs[b] = rms_norm(x[i], self.w.t["slow.final_norm"], cfg.eps)
            for b, st in enumerate(sts):
                if st.finished:
                    out[b, f] = -1
                    continue
                s, code0, lg0 = self.slow_head(hs[b])
                pos = st.length - 1          # the position whose hidden made this frame
                if self.eos is not None:     # candidates: C semantic codes, then EOS
                    cand = np.append(np.asarray(lg0, np.float32), self.eos_logit(hs[b]))
                    code0 = self._pick(cand, 0, seqs[b], pos)
                    if code0 == cfg.codebook_size:
                        st.finished = True
                        out[b, f] = -1
                        continue
                else:
                    code0 = self._pick(lg0, 0, seqs[b], pos)
                codes, lgs = self.fast_frame(hs[b], code0, seqs[b], pos)
                st.last = np.array(codes, np.int32)
                st.h_last = hs[b]
                out[b, f] = codes
                if self.record:
                    self.log.append({"seq": seqs[b], "frame": f, "h": hs[b],
                                     "logits": [lg0] + lgs})
        return out

    # ---- brute force and teacher forcing ----------------------------------

    def forward_full(self, inputs, capture=None):
        """All positions of one sequence recomputed with no cache: a causal
        pass over the input embeddings [T, d]; returns the slow hidden states
        after the final RMSNorm [T, d]."""
        cfg = self.cfg
        T = inputs.shape[0]
        kv = ContiguousKV(cfg.n_slow, cfg.n_kv, cfg.head_dim, self.dt, cap=T)
        x = self.slow_forward(inputs.astype(self.dt), np.arange(T), [kv] * T, capture)
        return rms_norm(x, self.w.t["slow.final_norm"], cfg.eps)

    def fast_full(self, h, frame_codes):
        """Fast AR logits of one frame by full recompute: a causal pass over
        positions [h, in_emb[0][c0], ..., in_emb[8][c8]]; returns logits of
        codes 1..9 [9, C]."""
        return self.fast_block(h[None, :], np.asarray(frame_codes)[None, :])[0]

    def fast_block(self, H, frames):
        """Teacher-forced Fast AR for many frames at once.

        H [n, d] slow hiddens, frames [n, 10] the codes fed at positions
        1..9.  Each frame is its own 10-position causal sequence.  Returns
        logits [n, 9, C] for codes 1..9.
        """
        cfg, dt = self.cfg, self.dt
        n = H.shape[0]
        NC = cfg.n_codebooks
        U = np.empty((n, NC, cfg.d), dt)
        U[:, 0] = H
        for j in range(1, NC):
            U[:, j] = self.w.t["fast.in_emb"][j - 1][frames[:, j - 1]]
        x = U.reshape(n * NC, cfg.d)
        pos = np.tile(np.arange(NC), n)
        kvs = [ContiguousKV(cfg.n_fast, cfg.n_kv, cfg.head_dim, dt, cap=NC)
               for _ in range(n)]
        views = [kvs[i // NC] for i in range(n * NC)]
        for l in range(cfg.n_fast):
            x = self._layer(self.w.layer("fast", l), x, pos, views, l)
        y = rms_norm(x.reshape(n, NC, cfg.d), self.w.t["fast.final_norm"], cfg.eps)
        out = np.empty((n, NC - 1, cfg.codebook_size), dt)
        for j in range(1, NC):
            out[:, j - 1] = y[:, j] @ self.w.t["fast.head"][j].T
        return out

    def teacher_forced(self, tokens, codes, mask, frames, capture_rows=None, seq=0):
        """Score a decoded frame stream by one causal full-sequence pass.

        The slow inputs are the prompt followed by the feedback embeddings of
        frames 0..n-2; frame f's hidden is the final-normed output at
        position T-1+f.  Returns per-frame slow hiddens [n, d], the oracle's
        argmax codes [n, 10], the top-2 margins [n, 10] and the logits
        (semantic slice [n, C] and fast [n, 9, C]).  ``capture_rows`` lists
        sequence positions whose per-layer residuals are returned.
        """
        cfg = self.cfg
        T = len(tokens)
        frames = np.asarray(frames)
        n = frames.shape[0]
        e = [embed_prompt(self.w, tokens, codes, mask)]
        if n > 1:
            e.append(np.stack([feedback_embedding(self.w, frames[f]) for f in range(n - 1)]))
        inputs = np.concatenate(e, axis=0)
        cap = [] if capture_rows is not None else None
        Hs = self.forward_full(inputs, cap)[T - 1:]
        sem = self.w.head_rows()
        lg0 = Hs @ sem.T                                  # [n, C]
        lgf = self.fast_block(Hs, frames)                 # [n, 9, C]
        logits = np.concatenate([lg0[:, None, :], lgf], axis=1)   # [n, 10, C]
        if self.sampling is None:
            pred = np.argmax(logits, axis=-1).astype(np.int32)
        else:
            pred = np.array([[self._pick(logits[f, k], k, seq, T - 1 + f)
                              for k in range(cfg.n_codebooks)] for f in range(n)], np.int32)
        top2 = np.sort(logits, axis=-1)[..., -2:]
        margin = top2[..., 1] - top2[..., 0]
        res = {"h": Hs, "pred": pred, "margin": margin, "logits": logits}
        if cap is not None:
            res["layers"] = np.stack([c[np.asarray(capture_rows)] for c in cap])
        return res
