// Host runtime behind the C ABI of include/s2.h: weight loading, the KV page
// pool and radix tree, sequence state, prefill and the per-frame launch
// sequence (captured in CUDA graphs, kernels chained with programmatic
// dependent launch).
#include "s2.h"
#include "s2_kernels.h"
#include "s2_radix.h"

#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <vector>

namespace s2 {

struct Dims {
  int d, H, Hkv, hd, F, Ls, Lf, V, sem, NC, C;
  float eps, theta;
  int wbf16;
  int qd() const { return H * hd; }
  int kvd() const { return Hkv * hd; }
  int qkvd() const { return qd() + 2 * kvd(); }
};

struct QMat {
  int8_t* q = nullptr;  // INT8 copy of a streamed matrix
  float* s = nullptr;   // per-row scales
};

struct LayerW {
  QMat qqkv, qo, qgu, qdn;  // INT8 copies (INT8 mode)
  void* qkv = nullptr;  // [q + 2 kv, d]: wq rows, then wk, then wv
  void* o = nullptr;    // [d, q]
  void* gu = nullptr;   // [2F, d]: gate row i at 2i, up row i at 2i+1
  void* dn = nullptr;   // [d, F]
  float* attn_norm = nullptr;
  float* q_norm = nullptr;
  float* k_norm = nullptr;
  float* mlp_norm = nullptr;
};

struct SeqState {
  bool live = false;
  bool primed = false;
  bool finished = false;   // picked the end-of-speech row (decode no longer allowed)
  int length = 0;
  std::vector<int> pages;
};

// S2_SYNC_CHECK=1 (debugging): synchronise after every library call and
// report the first one that failed; graphs are then disabled.
static const bool g_sync_check = [] {
  const char* e = std::getenv("S2_SYNC_CHECK");
  return e && e[0] == '1';
}();

#define CK(x)                                                               \
  do {                                                                      \
    cudaError_t e_ = (x);                                                   \
    if (e_ == cudaSuccess && g_sync_check) e_ = cudaDeviceSynchronize();    \
    if (e_ != cudaSuccess) {                                                \
      std::fprintf(stderr, "s2: %s failed: %s (%s:%d)\n", #x,               \
                   cudaGetErrorString(e_), __FILE__, __LINE__);             \
      return S2_ECUDA;                                                      \
    }                                                                       \
  } while (0)

}  // namespace s2

using namespace s2;

struct s2_ctx {
  Dims D{};
  s2_opts opt{};
  cudaStream_t st = nullptr;
  bool own_stream = false;
  int num_sms = 0;
  bool pdl = true, graphs = true, use_tc = true, use_radix = true, int8 = false;
  size_t wsz = 2;
  int kv_bf16 = 1;      // slow KV pool element type
  size_t kvsz = 2;

  // weights
  char* wbuf = nullptr;
  size_t wbytes = 0;
  void* tok_emb = nullptr;
  void* vq_emb = nullptr;
  void* fast_in = nullptr;
  void* fast_head = nullptr;
  float* slow_final = nullptr;
  float* fast_final = nullptr;
  std::vector<LayerW> slow, fast;
  char* qbuf = nullptr;  // INT8 weights (INT8 mode)
  QMat q_sem, q_fhead;   // semantic head slice [C, d], Fast AR heads [10 C, d]
  float* rope_cos = nullptr;
  float* rope_sin = nullptr;

  // KV
  void* pool = nullptr;
  long long page_elems = 0;
  size_t layer_elems = 0;
  int max_pages_seq = 0;
  PagePool pages;
  RadixTree radix{16};
  std::vector<SeqState> seqs;

  // device buffers (decode)
  char* dbuf = nullptr;
  float* seq_x = nullptr;     // [max_seqs][d]
  int* seq_codes = nullptr;   // [max_seqs][10]
  float* x_slow = nullptr;    // [B][d]
  float* qkv = nullptr;       // [2B][qkvd]
  float* attn_o = nullptr;    // [2B][qd]
  float* hff = nullptr;       // [2B][F]
  float* h_slow = nullptr;    // [B][d]
  float* x_fast = nullptr;    // [2B][d]
  void* fast_kv = nullptr;    // [Lf][B][page]
  int* last_codes = nullptr;  // [B][10]
  int* codes_all = nullptr;   // [B][max_frames][10]
  int max_frames = 0;
  int* table_b = nullptr;     // [B][max_pages_seq]
  int* pos_base = nullptr;    // [B]
  int* slots = nullptr;       // [B]
  int* frame_ctr = nullptr;
  float* part_val = nullptr;  // [8][gemv_max_grid]: per-CTA arg-max partials
  int* part_idx = nullptr;
  unsigned* ticket = nullptr;
  float* attn_part = nullptr;
  unsigned* attn_tickets = nullptr;
  unsigned* pf_tickets = nullptr;   // prefill attention key split: [query tiles][H]
  size_t attn_part_floats = 0;
  int attn_max_split = 16;
  // tensor-core attention over a prefix every row of a decode batch shares
  // (radix pages): whether this call uses it, the shared length (device
  // word and host copy, set per decode call), and the prefix keys of every
  // Slow AR layer as the MMAs' operand images (written once per call,
  // px_stride keys per (layer, kv head))
  bool use_prefix_tc = true;
  bool prefix_on = false;
  int* shared_len = nullptr;
  int shared_host = 0;
  void* px_planes = nullptr;
  uint8_t* q_img = nullptr;   // the query tiles of the prefix attention (one layer at a time)
  int px_stride = 0;
  size_t px_layer_bytes = 0;
  int tc_min_rows = 16;       // decode rows at which projections move to tcgen05
  int* err = nullptr;
  // bf16 operands of the tensor-core path
  __nv_bfloat16* a16 = nullptr;   // [rows][max(d, qd)]
  __nv_bfloat16* h16 = nullptr;   // [rows][F]
  __nv_bfloat16* a16lo = nullptr; // remainder planes (x ~= hi + lo)
  __nv_bfloat16* h16lo = nullptr;
  float* tc_ws = nullptr;
  size_t tc_ws_floats = 0;
  unsigned* tc_tickets = nullptr;
  size_t tc_n_tickets = 0;
  float* logits_b = nullptr;      // [B][C] (batched heads)
  // prefill buffers
  float* px = nullptr;
  float* pqkv = nullptr;
  float* pq = nullptr;
  float* po = nullptr;
  float* ph = nullptr;
  int* ptok = nullptr;
  int* pcodes = nullptr;
  uint8_t* pmask = nullptr;
  int* ptable = nullptr;
  // batched prefill: segment table [max_batch][5], row / query-tile -> segment,
  // page tables [max_batch][max_pages_seq]
  int* pf_info = nullptr;
  int* pf_row_seg = nullptr;
  int* pf_tile_seg = nullptr;
  int* pf_tables = nullptr;
  // host staging (pinned)
  int* hstage = nullptr;
  size_t hstage_ints = 0;

  // debug sinks
  float* dbg_logits = nullptr;   // device sinks the kernels write
  float* dbg_hidden = nullptr;
  float* dbg_layers = nullptr;
  int dbg_frames = 0;
  // host sinks: the caller's host buffers, filled from library-owned device
  // shadows (dbg_* above) at the end of every decode call
  float* dbg_host[3] = {nullptr, nullptr, nullptr};  // logits, hidden, layers
  float* dbg_shadow[3] = {nullptr, nullptr, nullptr};

  float temp_slow = 0.f, temp_fast = 0.f;  // sampling temperatures (0: greedy)
  float top_p_slow = 1.f, top_p_fast = 1.f; // nucleus filters of the sampled heads (1: off)
  int eos = -1;                              // end-of-speech token (-1: no stopping)
  int* done = nullptr;                       // [B] rows that picked EOS in this call
  unsigned long long seed = 0;
  std::map<std::pair<int, int>, cudaGraphExec_t> graph;
  std::map<std::pair<int, int>, long long> graph_launches;  // kernels per replay

  // persistent decode: the recorded frame per batch size (ok = false: the
  // frame has an operation the persistent kernel does not run)
  struct PersistProg {
    bool ok = false;
    PersistOp* ops = nullptr;  // device copy
    int n_ops = 0, maxb = 0, grid = 0;
    size_t smem = 0;
  };
  bool persist = false;
  std::map<int, PersistProg> persist_progs;
  // streaming decode (batch 1-2): the same recorded frame with its stream plan
  struct StreamProg {
    bool ok = false;
    PersistOp* ops = nullptr;   // device copies
    StreamPlan* plan = nullptr;
    int n_ops = 0, maxb = 0, grid = 0;
    StreamLayout L;
  };
  bool stream = false;
  std::map<int, StreamProg> stream_progs;
  // host-side fault injection (test hooks read at creation):
  // S2_FAULT_ALLOC_AT=n fails the context's n-th device allocation;
  // S2_FAULT_BARRIER=1 makes CTA 0 of the persistent kernel skip its arrival at
  // the barrier before the program's first attention operation (nothing in
  // flight there) with a 50 ms budget, so the other CTAs' waits run out
  // S2_FRAME_TRACE=<file> (measurement): every GEMV and decode-attention
  // launch of a captured frame gets a slot of per-CTA timestamps; after each
  // decode call the last frame's stamps are written to the file
  std::string ftrace_path;
  unsigned long long* ftrace = nullptr;   // [kFtLaunches][kFrameTraceCtas][4]
  int ft_next = 0;
  bool ft_in_frame = false;   // slots are handed out only while a frame is enqueued
  std::vector<std::string> ft_kind;
  std::vector<int> ft_ctas;   // CTAs of the launch in each slot
  int alloc_count = 0;
  int fault_alloc_at = 0;
  bool fault_barrier = false;
  unsigned* pwords = nullptr;  // [64]: barrier counter at 0, abort flag at 32

  s2_stats_t stats{};
};

namespace {

int fail(s2_ctx* c, int s) {
  if (c && s) c->stats.last_error = s;
  return s;
}

// Every device allocation of a context goes through here: with
// S2_FAULT_ALLOC_AT=n the context's n-th allocation fails as if the device
// were out of memory (no cudaMalloc is made).
template <typename T>
cudaError_t dev_alloc(s2_ctx* c, T** p, size_t bytes) {
  ++c->alloc_count;
  if (c->fault_alloc_at > 0 && c->alloc_count == c->fault_alloc_at) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(reinterpret_cast<void**>(p), bytes);
}

bool is_device_ptr(const void* p) {
  if (!p) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// ---------------------------------------------------------------- weight file

struct Entry {
  std::string name;
  uint32_t dtype, ndim;
  uint64_t shape[4], offset, nbytes;
};

int read_header(int fd, Dims& D, std::vector<Entry>& ents) {
  unsigned char hdr[128];
  if (pread(fd, hdr, 128, 0) != 128) return S2_EBADFILE;
  if (std::memcmp(hdr, "S2DUALAR", 8) != 0) return S2_EBADFILE;
  uint32_t ver, wdt, n;
  std::memcpy(&ver, hdr + 8, 4);
  std::memcpy(&wdt, hdr + 12, 4);
  if (ver != 1 || wdt > 1) return S2_EBADFILE;
  int32_t dims[11];
  std::memcpy(dims, hdr + 16, 44);
  float ft[2];
  std::memcpy(ft, hdr + 60, 8);
  std::memcpy(&n, hdr + 68, 4);
  D.d = dims[0]; D.H = dims[1]; D.Hkv = dims[2]; D.hd = dims[3]; D.F = dims[4];
  D.Ls = dims[5]; D.Lf = dims[6]; D.V = dims[7]; D.sem = dims[8]; D.NC = dims[9]; D.C = dims[10];
  D.eps = ft[0]; D.theta = ft[1];
  D.wbf16 = (int)wdt;
  if (D.d <= 0 || D.H <= 0 || D.Hkv <= 0 || D.H % D.Hkv || D.NC != 10 || D.sem + D.C != D.V ||
      n == 0 || n > 100000)
    return S2_EBADFILE;
  std::vector<unsigned char> tab((size_t)n * 128);
  if (pread(fd, tab.data(), tab.size(), 128) != (ssize_t)tab.size()) return S2_EBADFILE;
  ents.resize(n);
  for (uint32_t i = 0; i < n; ++i) {
    const unsigned char* e = tab.data() + (size_t)i * 128;
    char nm[65] = {0};
    std::memcpy(nm, e, 64);
    ents[i].name = nm;
    std::memcpy(&ents[i].dtype, e + 64, 4);
    std::memcpy(&ents[i].ndim, e + 68, 4);
    std::memcpy(ents[i].shape, e + 72, 32);
    std::memcpy(&ents[i].offset, e + 104, 8);
    std::memcpy(&ents[i].nbytes, e + 112, 8);
  }
  return S2_OK;
}

struct Loader {
  int fd;
  cudaStream_t st;
  char* pin[2] = {nullptr, nullptr};
  cudaEvent_t ev[2];
  size_t cap = 64u << 20;
  int cur = 0;
  int init() {
    for (int i = 0; i < 2; ++i) {
      if (cudaMallocHost(&pin[i], cap) != cudaSuccess) return S2_ENOMEM;
      cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
      cudaEventRecord(ev[i], st);
    }
    return S2_OK;
  }
  void fini() {
    cudaStreamSynchronize(st);
    for (int i = 0; i < 2; ++i) {
      if (pin[i]) cudaFreeHost(pin[i]);
      cudaEventDestroy(ev[i]);
    }
  }
  // Copy rows of ``row_bytes`` from the file to dst with a destination pitch.
  int rows(uint64_t off, size_t row_bytes, size_t n_rows, char* dst, size_t dpitch) {
    const size_t per = std::max<size_t>(1, cap / row_bytes);
    for (size_t r0 = 0; r0 < n_rows; r0 += per) {
      const size_t nr = std::min(per, n_rows - r0);
      cudaEventSynchronize(ev[cur]);
      size_t want = nr * row_bytes, got = 0;
      while (got < want) {
        ssize_t k = pread(fd, pin[cur] + got, want - got, off + r0 * row_bytes + got);
        if (k <= 0) return S2_EBADFILE;
        got += (size_t)k;
      }
      if (cudaMemcpy2DAsync(dst + r0 * dpitch, dpitch, pin[cur], row_bytes, row_bytes, nr,
                            cudaMemcpyHostToDevice, st) != cudaSuccess)
        return S2_ECUDA;
      cudaEventRecord(ev[cur], st);
      cur ^= 1;
    }
    return S2_OK;
  }
};

template <typename T>
T* carve(char*& p, size_t n) {
  T* r = reinterpret_cast<T*>(p);
  p += (n * sizeof(T) + 255) / 256 * 256;
  return r;
}

// RoPE table of the blocks (bf16-rounded cos/sin, see rope_fill).
int build_rope(s2_ctx* c, int n_pos) {
  const int half = c->D.hd / 2;
  std::vector<float> cs((size_t)n_pos * half), sn((size_t)n_pos * half);
  rope_fill(n_pos, c->D.hd, c->D.theta, cs.data(), sn.data());
  CK(cudaMemcpy(c->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(c->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice));
  return S2_OK;
}

// ---------------------------------------------------------------- launches

struct Rows {
  const float* X;
  int ldx;
  int rows;
};

// GEMV over any number of rows (chunks of 8).
constexpr int kFtLaunches = 1024;

// The next frame-timeline slot (null when tracing is off or the slots ran out);
// ``kind`` builds the launch's label only when a slot is handed out.
template <class Kind>
unsigned long long* ft_slot(s2_ctx* c, Kind&& kind, int ctas) {
  if (!c->ftrace || !c->ft_in_frame || c->ft_next >= kFtLaunches) return nullptr;
  if ((int)c->ft_kind.size() <= c->ft_next) {
    c->ft_kind.resize(c->ft_next + 1);
    c->ft_ctas.resize(c->ft_next + 1);
  }
  c->ft_kind[c->ft_next] = kind();
  c->ft_ctas[c->ft_next] = std::min(ctas, kFrameTraceCtas);
  return c->ftrace + (size_t)(c->ft_next++) * kFrameTraceCtas * 4;
}

int gemv(s2_ctx* c, GemvArgs a, int rows) {
  const int grid = gemv_grid(a, c->num_sms);
  if (grid > gemv_max_grid(c->num_sms)) return S2_EINVAL;  // arg-max partials are sized for this
  for (int r0 = 0; r0 < rows; r0 += 8) {
    GemvArgs b = a;
    b.B = std::min(8, rows - r0);
    b.X = a.X + (size_t)r0 * a.ldx;
    if (a.Y) b.Y = a.Y + (size_t)r0 * a.ldy;
    if (a.normed_out) b.normed_out = a.normed_out + (size_t)r0 * a.normed_ld;
    if (a.mode == GEMV_ARGMAX) {
      if (a.codes) b.codes = a.codes + (size_t)r0 * a.codes_ld;
      if (a.last_codes) b.last_codes = a.last_codes + (size_t)r0 * a.codes_per_frame;
      if (a.logits) b.logits = a.logits + (size_t)r0 * a.logits_ld;
      if (a.copy_src) b.copy_src = a.copy_src + (size_t)r0 * a.copy_src_ld;
      if (a.copy_dst) b.copy_dst = a.copy_dst + (size_t)r0 * a.copy_dst_ld;
      if (a.emb_dst) b.emb_dst = a.emb_dst + (size_t)r0 * a.emb_dst_ld;
      if (a.samp_seq) b.samp_seq = a.samp_seq + r0;
      if (a.samp_pos) b.samp_pos = a.samp_pos + r0;
      if (r0 + 8 < rows) b.frame_inc = nullptr;  // only the last chunk advances the frame
    }
    b.trace = ft_slot(c, [&] {
      return "gemv " + std::to_string(a.N) + "x" + std::to_string(a.K) + " mode " + std::to_string(a.mode) +
             " rows " + std::to_string(b.B) + " grid " + std::to_string(grid);
    }, grid);
    CK(launch_gemv(b, c->st, c->pdl, grid));
  }
  return S2_OK;
}

GemvArgs gv(s2_ctx* c, const void* W, int N, int K, const float* X, int ldx, float* Y, int ldy,
            int mode, const float* gain = nullptr, const QMat* qm = nullptr) {
  GemvArgs a;
  a.W = W;
  a.w_is_bf16 = c->D.wbf16;
  if (c->int8 && qm && qm->q) {
    a.W = qm->q;
    a.w_int8 = 1;
    a.wscale = qm->s;
  }
  a.N = N;
  a.K = K;
  a.unit = mode == GEMV_SWIGLU ? 2 : 1;
  a.X = X;
  a.ldx = ldx;
  a.gain = gain;
  a.eps = c->D.eps;
  a.Y = Y;
  a.ldy = ldy;
  a.mode = mode;
  a.err = c->err;
  return a;
}

int tc(s2_ctx* c, const void* W, int N, int K, const __nv_bfloat16* Bm, int T, int ldb, float* Y,
       int ldy, __nv_bfloat16* Y16, int ldy16, int epi) {
  // the remainder plane sits at the same offset in the matching *lo buffer
  auto lo_of = [&](const __nv_bfloat16* hi) -> __nv_bfloat16* {
    if (!hi) return nullptr;
    if (hi >= c->a16 && hi < c->h16) return c->a16lo + (hi - c->a16);
    return c->h16lo + (hi - c->h16);
  };
  TcGemmArgs g;
  g.A = static_cast<const __nv_bfloat16*>(W);
  g.N = N;
  g.K = K;
  g.Bm = Bm;
  g.Blo = lo_of(Bm);
  g.Y16lo = lo_of(Y16);
  g.T = T;
  g.ldb = ldb;
  g.Y = Y;
  g.ldy = ldy;
  g.Y16 = Y16;
  g.ldy16 = ldy16;
  g.epi = epi;
  g.split_k = 0;
  g.ws = c->tc_ws;
  g.ws_floats = c->tc_ws_floats;
  g.tickets = c->tc_tickets;
  g.n_tickets = c->tc_n_tickets;
  g.err = c->err;
  if (c->ftrace) {
    int tn, sk;
    tc_gemm_plan(N, K, T, c->num_sms, &tn, &sk, true);
    g.trace = ft_slot(c, [&] {
      return "tc " + std::to_string(N) + "x" + std::to_string(K) + " epi " + std::to_string(epi) + " rows " +
             std::to_string(T);
    }, (N / 128) * ((T + tn - 1) / tn) * sk);
  }
  CK(launch_tc_gemm(g, c->st, c->pdl, c->num_sms));
  return S2_OK;
}

int rms16(s2_ctx* c, const float* X, int ldx, int rows, const float* gain, float* out = nullptr,
          int out_ld = 0) {
  RmsRowsArgs r;
  r.x = X;
  r.ldx = ldx;
  r.rows = rows;
  r.d = c->D.d;
  r.gain = gain;
  r.eps = c->D.eps;
  r.out = out;
  r.out_ld = out_ld;
  r.out16 = c->a16;
  r.out16lo = c->a16lo;
  r.out16_ld = c->D.d;
  r.trace = ft_slot(c, [&] { return "rms rows " + std::to_string(rows); }, rows);
  CK(launch_rms_rows(r, c->st, c->pdl));
  return S2_OK;
}

bool tc_rows(s2_ctx* c, int rows) { return c->use_tc && rows >= c->tc_min_rows; }

int attn_split(s2_ctx* c, int B) {
  return attn_pick_split(B, c->D.Hkv, c->num_sms,
                         attn_decode_ctas_per_sm(c->D.hd, c->D.H / c->D.Hkv, c->kv_bf16), c->attn_max_split);
}

// One transformer block over ``rows`` rows at X (decode: new rows per
// sequence m, positions from pos_base/frame/pos_off).
int layer_decode(s2_ctx* c, const LayerW& w, float* X, int ldx, int B, int m, void* kv,
                 const int* table, const int* pos_base, const int* frame, int pos_off, int nsplit,
                 bool kv_bf16, const void* px = nullptr) {
  const Dims& D = c->D;
  const int rows = B * m;
  const bool tcp = tc_rows(c, rows);
  int s;
  if (tcp) {
    if ((s = rms16(c, X, ldx, rows, w.attn_norm))) return s;
    if ((s = tc(c, w.qkv, D.qkvd(), D.d, c->a16, rows, D.d, c->qkv, D.qkvd(), nullptr, 0, TC_STORE)))
      return s;
  } else if ((s = gemv(c, gv(c, w.qkv, D.qkvd(), D.d, X, ldx, c->qkv, D.qkvd(), GEMV_STORE, w.attn_norm,
                               &w.qqkv),
                       rows))) {
    return s;
  }
  AttnDecodeArgs a;
  a.qkv = c->qkv;
  a.qkv_ld = D.qkvd();
  a.B = B;
  a.m = m;
  a.H = D.H;
  a.Hkv = D.Hkv;
  a.hd = D.hd;
  a.q_gain = w.q_norm;
  a.k_gain = w.k_norm;
  a.eps = D.eps;
  a.rope_cos = c->rope_cos;
  a.rope_sin = c->rope_sin;
  a.pos_base = pos_base;
  a.frame = frame;
  a.pos_off = pos_off;
  a.kv = kv;
  a.kv_bf16 = kv_bf16;
  a.page_elems = c->page_elems;
  a.table = table;
  a.table_ld = c->max_pages_seq;
  if (tcp) {
    a.o16 = c->a16;
    a.o16lo = c->a16lo;
    a.o16_ld = D.qd();
  } else {
    a.o = c->attn_o;
    a.o_ld = D.qd();
  }
  a.nsplit = nsplit;
  a.part = c->attn_part;
  a.tickets = c->attn_tickets;
  a.err = c->err;
  if (tcp && table && m == 1 && c->prefix_on && px) {
    // the private keys (key_begin..) by the split-KV attention, which only
    // leaves its partial slots; then the batch's shared prefix on the tensor
    // cores, whose cluster merges its partials with those slots
    a.key_begin = c->shared_len;
    a.part_base = 0;
    a.merge_later = 1;
    a.q_img = c->q_img;
    a.trace = ft_slot(c, [&] {
      return "attn B " + std::to_string(B) + " m " + std::to_string(m) + " splits " + std::to_string(nsplit) +
             " private";
    }, B * D.Hkv * nsplit);
    CK(launch_attn_decode(a, c->st, c->pdl));
    a.trace = nullptr;
    CK(launch_attn_prefix_cl(a, px, c->px_stride, c->st, c->pdl));
  } else {
    a.trace = ft_slot(c, [&] {
      return "attn B " + std::to_string(B) + " m " + std::to_string(m) + " splits " + std::to_string(nsplit);
    }, B * D.Hkv * nsplit);
    CK(launch_attn_decode(a, c->st, c->pdl));
  }
  if (tcp) {
    if ((s = tc(c, w.o, D.d, D.qd(), c->a16, rows, D.qd(), X, ldx, nullptr, 0, TC_ADD))) return s;
    if ((s = rms16(c, X, ldx, rows, w.mlp_norm))) return s;
    if ((s = tc(c, w.gu, 2 * D.F, D.d, c->a16, rows, D.d, nullptr, 0, c->h16, D.F, TC_SWIGLU_BF16)))
      return s;
    return tc(c, w.dn, D.d, D.F, c->h16, rows, D.F, X, ldx, nullptr, 0, TC_ADD);
  }
  if ((s = gemv(c, gv(c, w.o, D.d, D.qd(), c->attn_o, D.qd(), X, ldx, GEMV_ADD, nullptr, &w.qo), rows)))
    return s;
  if ((s = gemv(c, gv(c, w.gu, 2 * D.F, D.d, X, ldx, c->hff, D.F, GEMV_SWIGLU, w.mlp_norm, &w.qgu), rows)))
    return s;
  if ((s = gemv(c, gv(c, w.dn, D.d, D.F, c->hff, D.F, X, ldx, GEMV_ADD, nullptr, &w.qdn), rows))) return s;
  return S2_OK;
}

const void* rowptr(s2_ctx* c, const void* base, size_t row) {
  return static_cast<const char*>(base) + row * (size_t)c->D.d * c->wsz;
}

// The constrained head of code ``j`` (0: semantic slice of the tied
// embedding; j >= 1: Fast AR head slice j), with its greedy pick and the
// gather of the next Fast AR input.
int head_pick(s2_ctx* c, int j, int B, int f_dbg);

int head_tc(s2_ctx* c, int j, int B, int f_dbg) {
  const Dims& D = c->D;
  int s;
  const float* X = j == 0 ? c->x_slow : c->x_fast + D.d;
  const int ldx = j == 0 ? D.d : 2 * D.d;
  if ((s = rms16(c, X, ldx, B, j == 0 ? c->slow_final : c->fast_final, j == 0 ? c->h_slow : nullptr, D.d)))
    return s;
  const void* W = j == 0 ? rowptr(c, c->tok_emb, D.sem) : rowptr(c, c->fast_head, (size_t)j * D.C);
  if ((s = tc(c, W, D.C, D.d, c->a16, B, D.d, c->logits_b, D.C, nullptr, 0, TC_STORE))) return s;
  return head_pick(c, j, B, f_dbg);
}

// The CUDA-core logits of head j (RMSNorm prologue; the semantic head also
// writes the normalised slow hidden to h_slow) into logits_b.
int head_logits_gemv(s2_ctx* c, int j, int B) {
  const Dims& D = c->D;
  QMat q{};
  if (c->int8) {
    if (j == 0) q = c->q_sem;
    else {
      q.q = c->q_fhead.q + (size_t)j * D.C * D.d;
      q.s = c->q_fhead.s + (size_t)j * D.C;
    }
  }
  const void* W = j == 0 ? rowptr(c, c->tok_emb, D.sem) : rowptr(c, c->fast_head, (size_t)j * D.C);
  GemvArgs a = gv(c, W, D.C, D.d, j == 0 ? c->x_slow : c->x_fast + D.d, j == 0 ? D.d : 2 * D.d,
                  c->logits_b, D.C, GEMV_STORE, j == 0 ? c->slow_final : c->fast_final, &q);
  if (j == 0) {
    a.normed_out = c->h_slow;
    a.normed_ld = D.d;
  }
  return gemv(c, a, B);
}

// Select kernel over logits_b for head j and the frame tail.
int head_pick(s2_ctx* c, int j, int B, int f_dbg) {
  const Dims& D = c->D;
  ArgmaxRowsArgs a;
  a.top_p = j == 0 ? c->top_p_slow : c->top_p_fast;
  a.done = c->eos >= 0 ? c->done : nullptr;
  if (j == 0 && c->eos >= 0) {
    a.eos_row = rowptr(c, c->tok_emb, (size_t)c->eos);
    a.eos_bf16 = D.wbf16;
    a.h = c->h_slow;
    a.h_ld = D.d;
  }
  a.temperature = j == 0 ? c->temp_slow : c->temp_fast;
  a.seed = c->seed;
  a.samp_seq = c->slots;
  a.samp_pos = c->pos_base;
  a.logits = c->logits_b;
  a.ld = D.C;
  a.rows = B;
  a.C = D.C;
  if (c->dbg_logits && f_dbg >= 0) {
    a.sink = c->dbg_logits + ((size_t)f_dbg * D.NC + j) * D.C;
    a.sink_ld = c->dbg_frames * D.NC * D.C;
  }
  a.codes = c->codes_all;
  a.codes_ld = c->max_frames * D.NC;
  a.codes_per_frame = D.NC;
  a.code_slot = j;
  a.frame = c->frame_ctr;
  a.last_codes = c->last_codes;
  a.ticket = c->ticket + 1;
  a.d = D.d;
  a.emb_is_bf16 = D.wbf16;
  if (j == 0) {
    a.copy_src = c->h_slow;
    a.copy_src_ld = D.d;
    a.copy_dst = c->x_fast;
    a.copy_dst_ld = 2 * D.d;
    a.emb_next = c->fast_in;
  } else if (j < D.NC - 1) {
    a.emb_next = rowptr(c, c->fast_in, (size_t)j * D.C);
  }
  a.emb_dst = c->x_fast + D.d;
  a.emb_dst_ld = 2 * D.d;
  if (j == D.NC - 1) a.frame_inc = c->frame_ctr;
  CK(launch_argmax_rows(a, c->st, c->pdl));
  return S2_OK;
}

// Whether head j goes through logits + the select kernel (end-of-speech
// stopping, or a top-p filtered draw) instead of the GEMV's own arg-max.
bool head_select(s2_ctx* c, int j) {
  if (c->eos >= 0) return true;
  const float t = j == 0 ? c->temp_slow : c->temp_fast;
  const float p = j == 0 ? c->top_p_slow : c->top_p_fast;
  return t > 0.f && p < 1.f;
}

int head(s2_ctx* c, int j, int B, int f_dbg) {
  if (tc_rows(c, B) && c->D.C % 128 == 0) return head_tc(c, j, B, f_dbg);
  if (head_select(c, j)) {
    const int s = head_logits_gemv(c, j, B);
    return s ? s : head_pick(c, j, B, f_dbg);
  }
  const Dims& D = c->D;
  GemvArgs a;
  a.temperature = j == 0 ? c->temp_slow : c->temp_fast;
  a.seed = c->seed;
  a.samp_seq = c->slots;
  a.samp_pos = c->pos_base;
  a.w_is_bf16 = D.wbf16;
  a.N = D.C;
  a.K = D.d;
  a.unit = 1;
  a.eps = D.eps;
  a.mode = GEMV_ARGMAX;
  a.part_val = c->part_val;
  a.part_idx = c->part_idx;
  a.ticket = c->ticket;
  a.codes = c->codes_all;
  a.codes_ld = c->max_frames * D.NC;
  a.codes_per_frame = D.NC;
  a.code_slot = j;
  a.frame = c->frame_ctr;
  a.last_codes = c->last_codes;
  a.tail_d = D.d;
  a.emb_is_bf16 = D.wbf16;
  a.err = c->err;
  if (c->dbg_logits && f_dbg >= 0) {
    a.logits = c->dbg_logits + ((size_t)f_dbg * D.NC + j) * D.C;
    a.logits_ld = c->dbg_frames * D.NC * D.C;
  }
  if (c->int8) {
    a.w_int8 = 1;
    a.wscale = j == 0 ? c->q_sem.s : c->q_fhead.s + (size_t)j * D.C;
  }
  if (j == 0) {
    a.W = c->int8 ? (const void*)c->q_sem.q : rowptr(c, c->tok_emb, D.sem);
    a.X = c->x_slow;
    a.ldx = D.d;
    a.gain = c->slow_final;
    a.normed_out = c->h_slow;
    a.normed_ld = D.d;
    a.copy_src = c->h_slow;
    a.copy_src_ld = D.d;
    a.copy_dst = c->x_fast;
    a.copy_dst_ld = 2 * D.d;
    a.emb_next = c->fast_in;
    a.emb_dst = c->x_fast + D.d;
    a.emb_dst_ld = 2 * D.d;
  } else {
    a.W = c->int8 ? (const void*)(c->q_fhead.q + (size_t)j * D.C * D.d) : rowptr(c, c->fast_head, (size_t)j * D.C);
    a.X = c->x_fast + D.d;
    a.ldx = 2 * D.d;
    a.gain = c->fast_final;
    if (j < D.NC - 1) {
      a.emb_next = rowptr(c, c->fast_in, (size_t)j * D.C);
      a.emb_dst = c->x_fast + D.d;
      a.emb_dst_ld = 2 * D.d;
    }
    if (j == D.NC - 1) a.frame_inc = c->frame_ctr;
  }
  return gemv(c, a, B);
}


enum FrameMode { FRAME_SLOW = 1, FRAME_HEADFAST = 2, FRAME_FULL = 3 };

// One frame on rows [0, B): [slow step] -> semantic head -> Fast AR passes
// 1..9.  Row b's slow step writes position pos_base[b] + frame.
int enqueue_frame_body(s2_ctx* c, int B, int mode, int f_dbg);

int enqueue_frame(s2_ctx* c, int B, int mode, int f_dbg) {
  c->ft_next = 0;
  c->ft_in_frame = true;
  const int s = enqueue_frame_body(c, B, mode, f_dbg);
  c->ft_in_frame = false;
  return s;
}

int enqueue_frame_body(s2_ctx* c, int B, int mode, int f_dbg) {
  const Dims& D = c->D;
  int s;
  if (mode & FRAME_SLOW) {
    EmbedArgs e;
    e.tok_emb = c->tok_emb;
    e.vq_emb = c->vq_emb;
    e.w_bf16 = D.wbf16;
    e.d = D.d;
    e.n_codebooks = D.NC;
    e.codebook_size = D.C;
    e.sem_begin = D.sem;
    e.rows = B;
    e.fb = c->last_codes;
    e.out = c->x_slow;
    e.out_ld = D.d;
    CK(launch_embed(e, c->st, c->pdl));
    const int ns = attn_split(c, B);
    for (int l = 0; l < D.Ls; ++l) {
      void* kv = static_cast<char*>(c->pool) + (size_t)l * c->layer_elems * c->kvsz;
      const void* px = c->prefix_on ? static_cast<char*>(c->px_planes) + l * c->px_layer_bytes : nullptr;
      if ((s = layer_decode(c, c->slow[l], c->x_slow, D.d, B, 1, kv, c->table_b, c->pos_base,
                            c->frame_ctr, 0, ns, c->kv_bf16, px)))
        return s;
      if (c->dbg_layers && f_dbg >= 0)
        CK(cudaMemcpyAsync(c->dbg_layers + ((size_t)f_dbg * D.Ls + l) * B * D.d, c->x_slow,
                           (size_t)B * D.d * 4, cudaMemcpyDeviceToDevice, c->st));
    }
  }
  if (!(mode & FRAME_HEADFAST)) return S2_OK;
  if ((s = head(c, 0, B, f_dbg))) return s;
  if (c->dbg_hidden && f_dbg >= 0)
    CK(cudaMemcpy2DAsync(c->dbg_hidden + (size_t)f_dbg * D.d, (size_t)c->dbg_frames * D.d * 4,
                         c->h_slow, (size_t)D.d * 4, (size_t)D.d * 4, B, cudaMemcpyDeviceToDevice,
                         c->st));
  const size_t fkv_layer = (size_t)B * c->page_elems;
  for (int j = 1; j < D.NC; ++j) {
    const bool first = j == 1;
    float* X = first ? c->x_fast : c->x_fast + D.d;
    const int ldx = first ? D.d : 2 * D.d;
    for (int l = 0; l < D.Lf; ++l) {
      void* kv = static_cast<char*>(c->fast_kv) + (size_t)l * fkv_layer * sizeof(float);
      if ((s = layer_decode(c, c->fast[l], X, ldx, B, first ? 2 : 1, kv, nullptr, nullptr, nullptr,
                            first ? 0 : j, 1, false)))
        return s;
    }
    if ((s = head(c, j, B, f_dbg))) return s;
  }
  return S2_OK;
}

}  // namespace

// ====================================================================== ABI

extern "C" const char* s2_strerror(int s) {
  switch (s) {
    case S2_OK: return "ok";
    case S2_EINVAL: return "invalid argument";
    case S2_ENOMEM: return "out of KV pages or device memory";
    case S2_ECUDA: return "CUDA error";
    case S2_ETIMEOUT: return "device wait timed out";
    case S2_EBADFILE: return "bad weight file";
    case S2_ESTATE: return "sequence in the wrong state";
    default: return "unknown status";
  }
}

extern "C" int s2_create(const char* path, const s2_opts* o, s2_ctx** out) {
  if (!path || !out) return S2_EINVAL;
  *out = nullptr;
  s2_opts opt{};
  if (o) opt = *o;
  if (opt.max_seqs <= 0) opt.max_seqs = 64;
  if (opt.max_batch <= 0) opt.max_batch = opt.max_seqs;
  if (opt.page_size <= 0) opt.page_size = 16;
  if (opt.max_ctx <= 0) opt.max_ctx = 2048;
  if (opt.max_prompt <= 0) opt.max_prompt = std::min(opt.max_ctx, 2048);
  if (opt.kv_pool_pages <= 0) opt.kv_pool_pages = opt.max_seqs * ((opt.max_ctx + 15) / 16);
  if (opt.prefill_rows < opt.max_prompt) opt.prefill_rows = opt.max_prompt;
  if (opt.page_size != 16 || opt.max_batch > opt.max_seqs || opt.max_prompt > opt.max_ctx)
    return S2_EINVAL;

  int fd = open(path, O_RDONLY);
  if (fd < 0) return S2_EBADFILE;
  Dims D;
  std::vector<Entry> ents;
  int s = read_header(fd, D, ents);
  if (s) {
    close(fd);
    return s;
  }
  if (!((D.hd == 128 && D.H / D.Hkv == 4) || (D.hd == 64 && D.H / D.Hkv == 2)) || D.d % 8 ||
      D.F % 8) {
    close(fd);
    return S2_EBADFILE;
  }
  s2_ctx* c = new s2_ctx();
  c->D = D;
  c->opt = opt;
  c->st = static_cast<cudaStream_t>(opt.cuda_stream);
  if (!c->st) {
    // graphs cannot be captured on the legacy default stream: use a blocking
    // stream of our own (it still synchronises with the default stream)
    if (cudaStreamCreate(&c->st) != cudaSuccess) {
      close(fd);
      delete c;
      return S2_ECUDA;
    }
    c->own_stream = true;
  }
  c->pdl = !(opt.flags & S2_FLAG_NO_PDL);
  c->graphs = !(opt.flags & S2_FLAG_NO_GRAPH) && !g_sync_check;
  c->persist = (opt.flags & S2_FLAG_PERSIST) && !g_sync_check;
  c->stream = (opt.flags & S2_FLAG_STREAM) && !g_sync_check;
  c->use_prefix_tc = !(opt.flags & S2_FLAG_NO_PREFIX_TC) && D.hd == 128 && D.H == 4 * D.Hkv &&
                     opt.max_batch >= 2;
  if (const char* e = std::getenv("S2_FAULT_ALLOC_AT")) c->fault_alloc_at = std::atoi(e);
  if (const char* e = std::getenv("S2_FAULT_BARRIER")) c->fault_barrier = std::atoi(e) != 0;
  if (const char* e = std::getenv("S2_FRAME_TRACE")) {
    // measurement only: outside the counted allocations (no fault index)
    c->ftrace_path = e;
    if (cudaMalloc(&c->ftrace, (size_t)kFtLaunches * kFrameTraceCtas * 4 * 8) != cudaSuccess ||
        cudaMemset(c->ftrace, 0, (size_t)kFtLaunches * kFrameTraceCtas * 4 * 8) != cudaSuccess) {
      cudaGetLastError();
      if (c->ftrace) cudaFree(c->ftrace);
      c->ftrace = nullptr;
    }
  }
  c->use_tc = !(opt.flags & S2_FLAG_NO_TC) && D.wbf16;
  c->use_radix = !(opt.flags & S2_FLAG_NO_RADIX);
  c->int8 = (opt.flags & S2_FLAG_INT8) != 0;
  if (c->int8) c->use_tc = false;
  c->wsz = D.wbf16 ? 2 : 4;
  c->kv_bf16 = D.wbf16 && (opt.flags & S2_FLAG_KV_BF16);
  c->kvsz = c->kv_bf16 ? 2 : 4;
  int dev;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  c->stats.num_sms = c->num_sms;
  c->seqs.resize(opt.max_seqs);

  auto cleanup = [&](int st) {
    close(fd);
    s2_destroy(c);
    return st;
  };

  // ---- weights: one device allocation
  const size_t ws = c->wsz;
  const size_t d = D.d, F = D.F;
  auto al = [](size_t b) { return (b + 255) / 256 * 256; };
  size_t per_layer = al((size_t)D.qkvd() * d * ws) + al(d * D.qd() * ws) + al(2 * F * d * ws) +
                     al(d * F * ws) + al(d * 4) * 2 + al((size_t)D.hd * 4) * 2;
  size_t table = al((size_t)D.NC * D.C * d * ws);
  c->wbytes = al((size_t)D.V * d * ws) + 3 * table + (size_t)(D.Ls + D.Lf) * per_layer + 2 * al(d * 4);
  if (dev_alloc(c, &c->wbuf, c->wbytes) != cudaSuccess) return cleanup(S2_ENOMEM);
  c->stats.weight_bytes = (int64_t)c->wbytes;
  char* p = c->wbuf;
  c->tok_emb = carve<char>(p, (size_t)D.V * d * ws);
  c->vq_emb = carve<char>(p, (size_t)D.NC * D.C * d * ws);
  c->fast_in = carve<char>(p, (size_t)D.NC * D.C * d * ws);
  c->fast_head = carve<char>(p, (size_t)D.NC * D.C * d * ws);
  c->slow_final = carve<float>(p, d);
  c->fast_final = carve<float>(p, d);
  auto mk = [&](std::vector<LayerW>& v, int n) {
    v.resize(n);
    for (auto& w : v) {
      w.qkv = carve<char>(p, (size_t)D.qkvd() * d * ws);
      w.o = carve<char>(p, d * D.qd() * ws);
      w.gu = carve<char>(p, 2 * F * d * ws);
      w.dn = carve<char>(p, d * F * ws);
      w.attn_norm = carve<float>(p, d);
      w.mlp_norm = carve<float>(p, d);
      w.q_norm = carve<float>(p, D.hd);
      w.k_norm = carve<float>(p, D.hd);
    }
  };
  mk(c->slow, D.Ls);
  mk(c->fast, D.Lf);

  Loader ld;
  ld.fd = fd;
  ld.st = c->st;
  if ((s = ld.init())) {
    ld.fini();
    return cleanup(s);
  }
  int loaded = 0;
  for (const Entry& e : ents) {
    const size_t esz = e.dtype == 1 ? 2 : 4;
    const bool is_gain = e.ndim == 1;
    if (!is_gain && esz != ws) { ld.fini(); return cleanup(S2_EBADFILE); }
    size_t rows = e.ndim >= 1 ? e.shape[0] : 1;
    for (uint32_t k = 1; k + 1 < e.ndim; ++k) rows *= e.shape[k];
    const size_t rb = (e.ndim >= 2 ? e.shape[e.ndim - 1] : e.shape[0]) * esz;
    if (e.ndim == 1) rows = 1;
    if (rows * rb != e.nbytes) { ld.fini(); return cleanup(S2_EBADFILE); }
    char* dst = nullptr;
    size_t pitch = rb;
    const std::string& n = e.name;
    auto layer_of = [&](const char* pre, std::vector<LayerW>& v, LayerW*& w, std::string& key) {
      const size_t lp = std::strlen(pre);
      if (n.compare(0, lp, pre) != 0) return false;
      const size_t dot = n.find('.', lp);
      if (dot == std::string::npos) return false;
      const int l = std::atoi(n.substr(lp, dot - lp).c_str());
      if (l < 0 || l >= (int)v.size()) return false;
      w = &v[l];
      key = n.substr(dot + 1);
      return true;
    };
    LayerW* w = nullptr;
    std::string key;
    if (n == "tok_emb") dst = (char*)c->tok_emb;
    else if (n == "vq_emb") dst = (char*)c->vq_emb;
    else if (n == "fast.in_emb") dst = (char*)c->fast_in;
    else if (n == "fast.head") dst = (char*)c->fast_head;
    else if (n == "slow.final_norm") dst = (char*)c->slow_final;
    else if (n == "fast.final_norm") dst = (char*)c->fast_final;
    else if (layer_of("slow.", c->slow, w, key) || layer_of("fast.", c->fast, w, key)) {
      if (key == "wq") dst = (char*)w->qkv;
      else if (key == "wk") dst = (char*)w->qkv + (size_t)D.qd() * d * ws;
      else if (key == "wv") dst = (char*)w->qkv + (size_t)(D.qd() + D.kvd()) * d * ws;
      else if (key == "wo") dst = (char*)w->o;
      else if (key == "wg") { dst = (char*)w->gu; pitch = 2 * rb; }
      else if (key == "wu") { dst = (char*)w->gu + rb; pitch = 2 * rb; }
      else if (key == "wd") dst = (char*)w->dn;
      else if (key == "attn_norm") dst = (char*)w->attn_norm;
      else if (key == "mlp_norm") dst = (char*)w->mlp_norm;
      else if (key == "q_norm") dst = (char*)w->q_norm;
      else if (key == "k_norm") dst = (char*)w->k_norm;
    }
    if (!dst) continue;
    if ((s = ld.rows(e.offset, rb, rows, dst, pitch))) { ld.fini(); return cleanup(s); }
    ++loaded;
  }
  ld.fini();
  const int want = 6 + (D.Ls + D.Lf) * 11;
  if (loaded != want) return cleanup(S2_EBADFILE);
  close(fd);
  fd = -1;
  auto cleanup2 = [&](int st) {
    s2_destroy(c);
    return st;
  };

  // ---- INT8 copies of every streamed matrix
  if (c->int8) {
    size_t qb = 0;
    auto qsz = [&](size_t N, size_t K) { return al(N * K) + al(N * 4); };
    for (int l = 0; l < D.Ls + D.Lf; ++l)
      qb += qsz(D.qkvd(), d) + qsz(d, D.qd()) + qsz(2 * F, d) + qsz(d, F);
    qb += qsz(D.C, d) + qsz((size_t)D.NC * D.C, d);
    if (dev_alloc(c, &c->qbuf, qb) != cudaSuccess) return cleanup2(S2_ENOMEM);
    char* q = c->qbuf;
    auto mkq = [&](QMat& m, const void* W, size_t N, size_t K) {
      m.q = carve<int8_t>(q, N * K);
      m.s = carve<float>(q, N);
      return launch_quantize_rows(W, D.wbf16, (int)N, (int)K, m.q, m.s, c->st);
    };
    cudaError_t e = cudaSuccess;
    for (auto* v : {&c->slow, &c->fast})
      for (LayerW& w : *v) {
        if (!e) e = mkq(w.qqkv, w.qkv, D.qkvd(), d);
        if (!e) e = mkq(w.qo, w.o, d, D.qd());
        if (!e) e = mkq(w.qgu, w.gu, 2 * F, d);
        if (!e) e = mkq(w.qdn, w.dn, d, F);
      }
    if (!e) e = mkq(c->q_sem, static_cast<char*>(c->tok_emb) + (size_t)D.sem * d * ws, D.C, d);
    if (!e) e = mkq(c->q_fhead, c->fast_head, (size_t)D.NC * D.C, d);
    if (e != cudaSuccess) return cleanup2(S2_ECUDA);
  }

  // ---- KV pool
  c->page_elems = 2LL * D.Hkv * 16 * D.hd;
  c->layer_elems = (size_t)opt.kv_pool_pages * c->page_elems;
  c->max_pages_seq = (opt.max_ctx + 15) / 16;
  if (dev_alloc(c, &c->pool, c->layer_elems * D.Ls * c->kvsz) != cudaSuccess) return cleanup2(S2_ENOMEM);
  c->pages.init(opt.kv_pool_pages, opt.page_perm_seed);
  if (c->use_prefix_tc && c->use_tc) {
    c->px_stride = attn_prefix_plane_stride(opt.max_ctx);
    c->px_layer_bytes = attn_prefix_plane_bytes(D.Hkv, D.hd, c->px_stride, 1);
    if (dev_alloc(c, &c->px_planes, c->px_layer_bytes * D.Ls) != cudaSuccess) return cleanup2(S2_ENOMEM);
  }

  // ---- work buffers
  // T: rows of one prefill pass (a prompt's uncached rows, or a batched pass)
  const int B = opt.max_batch, B2 = 2 * opt.max_batch, T = opt.prefill_rows;
  c->max_frames = 1024;
  const int rows16 = std::max(T, B2);
  const size_t wide = std::max<size_t>(d, D.qd());
  size_t tcws = 0, tct = 0;
  if (c->use_tc) {
    // largest split-K workspace over the projections at the largest row count
    const int Ns[4] = {D.qkvd(), (int)d, 2 * D.F, (int)d};
    const int Ks[4] = {(int)d, D.qd(), (int)d, D.F};
    for (int i = 0; i < 4; ++i)
      for (int r : {B, B2, T}) {
        int tn, sk;
        tc_gemm_plan(Ns[i], Ks[i], r, c->num_sms, &tn, &sk, true);
        tcws = std::max(tcws, tc_gemm_ws_floats(Ns[i], r, sk, true));
        tct = std::max(tct, tc_gemm_tickets(Ns[i], r, true));
      }
    int tn, sk;
    tc_gemm_plan(D.C, (int)d, B, c->num_sms, &tn, &sk, true);
    tcws = std::max(tcws, tc_gemm_ws_floats(D.C, B, sk, true));
    tct = std::max(tct, tc_gemm_tickets(D.C, B, true));
  }
  c->tc_ws_floats = tcws;
  c->tc_n_tickets = tct;
  // two passes over the same carve sequence: sizes, then pointers
  auto carve_all = [&](char* base) {
    char* p = base;
    c->seq_x = carve<float>(p, (size_t)opt.max_seqs * d);
    c->seq_codes = carve<int>(p, (size_t)opt.max_seqs * D.NC);
    c->x_slow = carve<float>(p, (size_t)B * d);
    c->qkv = carve<float>(p, (size_t)B2 * D.qkvd());
    c->attn_o = carve<float>(p, (size_t)B2 * D.qd());
    c->hff = carve<float>(p, (size_t)B2 * F);
    c->h_slow = carve<float>(p, (size_t)B * d);
    c->x_fast = carve<float>(p, (size_t)B2 * d);
    c->fast_kv = carve<float>(p, (size_t)D.Lf * B * c->page_elems);
    c->last_codes = carve<int>(p, (size_t)B * D.NC);
    c->done = carve<int>(p, B);
    c->codes_all = carve<int>(p, (size_t)B * c->max_frames * D.NC);
    c->table_b = carve<int>(p, (size_t)B * c->max_pages_seq);
    c->pos_base = carve<int>(p, B);
    c->slots = carve<int>(p, B);
    c->frame_ctr = carve<int>(p, 16);
    c->part_val = carve<float>(p, (size_t)8 * gemv_max_grid(c->num_sms));
    c->part_idx = carve<int>(p, (size_t)8 * gemv_max_grid(c->num_sms));
    c->ticket = carve<unsigned>(p, 16);
    c->attn_part_floats = attn_decode_scratch_floats(B2, 1, D.H, D.hd, c->attn_max_split);
    c->attn_part = carve<float>(p, c->attn_part_floats);
    c->attn_tickets = carve<unsigned>(p, (size_t)B * D.Hkv + 16);
    c->pf_tickets = carve<unsigned>(p, (size_t)((T + 63) / 64) * D.H + 16);
    c->err = carve<int>(p, 16);
    c->pwords = carve<unsigned>(p, 64);
    c->shared_len = carve<int>(p, 16);
    c->q_img = c->use_prefix_tc ? carve<uint8_t>(p, attn_prefix_qimg_bytes(B, D.Hkv)) : nullptr;
    c->a16 = carve<__nv_bfloat16>(p, (size_t)rows16 * wide);
    c->h16 = carve<__nv_bfloat16>(p, (size_t)rows16 * F);
    c->a16lo = carve<__nv_bfloat16>(p, (size_t)rows16 * wide);
    c->h16lo = carve<__nv_bfloat16>(p, (size_t)rows16 * F);
    c->tc_ws = carve<float>(p, tcws);
    c->tc_tickets = carve<unsigned>(p, tct + 16);
    c->logits_b = carve<float>(p, (size_t)B * D.C);
    c->px = carve<float>(p, (size_t)T * d);
    c->pqkv = carve<float>(p, (size_t)T * D.qkvd());
    c->pq = carve<float>(p, (size_t)T * D.qd());
    c->po = carve<float>(p, (size_t)T * D.qd());
    c->ph = carve<float>(p, (size_t)T * F);
    c->ptok = carve<int>(p, T);
    c->pcodes = carve<int>(p, (size_t)D.NC * T);
    c->pmask = carve<uint8_t>(p, T);
    c->ptable = carve<int>(p, c->max_pages_seq);
    c->pf_info = carve<int>(p, (size_t)5 * B + 16);
    c->pf_row_seg = carve<int>(p, (size_t)T + 16);
    c->pf_tile_seg = carve<int>(p, (size_t)T / 32 + B + 16);
    c->pf_tables = carve<int>(p, (size_t)B * c->max_pages_seq);
    return (size_t)(p - base);
  };
  char* const fake = reinterpret_cast<char*>((uintptr_t)256);  // sizing pass: any base works
  const size_t need = carve_all(fake);
  if (dev_alloc(c, &c->dbuf, need) != cudaSuccess) return cleanup2(S2_ENOMEM);
  cudaMemset(c->dbuf, 0, need);
  if (carve_all(c->dbuf) != need) return cleanup2(S2_ECUDA);
  c->hstage_ints = (size_t)B * c->max_pages_seq + 4 * (size_t)B + (size_t)(D.NC + 2) * T + 64;
  if (cudaMallocHost(&c->hstage, c->hstage_ints * 4) != cudaSuccess) return cleanup2(S2_ENOMEM);

  if (dev_alloc(c, &c->rope_cos, (size_t)opt.max_ctx * D.hd / 2 * 4) != cudaSuccess ||
      dev_alloc(c, &c->rope_sin, (size_t)opt.max_ctx * D.hd / 2 * 4) != cudaSuccess)
    return cleanup2(S2_ENOMEM);
  if ((s = build_rope(c, opt.max_ctx))) return cleanup2(s);
  if (cudaStreamSynchronize(c->st) != cudaSuccess) return cleanup2(S2_ECUDA);
  c->stats.pages_total = opt.kv_pool_pages;
  *out = c;
  return S2_OK;
}

static void free_debug_shadows(s2_ctx* c) {
  for (int i = 0; i < 3; ++i) {
    if (c->dbg_shadow[i]) cudaFree(c->dbg_shadow[i]);
    c->dbg_shadow[i] = nullptr;
    c->dbg_host[i] = nullptr;
  }
}

// Floats of debug sink i (0 logits, 1 hidden, 2 layers) for a decode call of
// B rows.
static size_t debug_sink_floats(const s2_ctx* c, int i, int B) {
  const Dims& D = c->D;
  const size_t f = (size_t)c->dbg_frames;
  if (i == 0) return (size_t)B * f * D.NC * D.C;
  if (i == 1) return (size_t)B * f * D.d;
  return f * D.Ls * (size_t)B * D.d;
}

extern "C" void s2_destroy(s2_ctx* c) {
  if (!c) return;
  cudaStreamSynchronize(c->st);
  for (auto& kv : c->graph) cudaGraphExecDestroy(kv.second);
  for (auto& kv : c->persist_progs)
    if (kv.second.ops) cudaFree(kv.second.ops);
  for (auto& kv : c->stream_progs) {
    if (kv.second.ops) cudaFree(kv.second.ops);
    if (kv.second.plan) cudaFree(kv.second.plan);
  }
  for (int i = 0; i < 3; ++i)
    if (c->dbg_shadow[i]) cudaFree(c->dbg_shadow[i]);
  if (c->wbuf) cudaFree(c->wbuf);
  if (c->qbuf) cudaFree(c->qbuf);
  if (c->pool) cudaFree(c->pool);
  if (c->px_planes) cudaFree(c->px_planes);
  if (c->ftrace) cudaFree(c->ftrace);
  if (c->dbuf) cudaFree(c->dbuf);
  if (c->rope_cos) cudaFree(c->rope_cos);
  if (c->rope_sin) cudaFree(c->rope_sin);
  if (c->hstage) cudaFreeHost(c->hstage);
  if (c->own_stream) cudaStreamDestroy(c->st);
  delete c;
}

namespace {

// Prefill compute for rows P..T-1 of one sequence whose table is in ptable.
int prefill_compute(s2_ctx* c, int P, int T) {
  const Dims& D = c->D;
  const int R = T - P;
  int s;
  EmbedArgs e;
  e.tok_emb = c->tok_emb;
  e.vq_emb = c->vq_emb;
  e.w_bf16 = D.wbf16;
  e.d = D.d;
  e.n_codebooks = D.NC;
  e.codebook_size = D.C;
  e.sem_begin = D.sem;
  e.rows = R;
  e.tokens = c->ptok + P;
  e.codes = c->pcodes + P;
  e.codes_ld = T;
  e.mask = c->pmask + P;
  e.out = c->px;
  e.out_ld = D.d;
  CK(launch_embed(e, c->st, c->pdl));
  const bool tcp = c->use_tc && R >= 16;
  for (int l = 0; l < D.Ls; ++l) {
    const LayerW& w = c->slow[l];
    void* kv = static_cast<char*>(c->pool) + (size_t)l * c->layer_elems * c->kvsz;
    if (tcp) {
      RmsRowsArgs r;
      r.x = c->px; r.ldx = D.d; r.rows = R; r.d = D.d; r.gain = w.attn_norm; r.eps = D.eps;
      r.out16 = c->a16; r.out16lo = c->a16lo; r.out16_ld = D.d;
      CK(launch_rms_rows(r, c->st, c->pdl));
      if ((s = tc(c, w.qkv, D.qkvd(), D.d, c->a16, R, D.d, c->pqkv, D.qkvd(), nullptr, 0, TC_STORE)))
        return s;
    } else {
      if ((s = gemv(c, gv(c, w.qkv, D.qkvd(), D.d, c->px, D.d, c->pqkv, D.qkvd(), GEMV_STORE, w.attn_norm,
                          &w.qqkv), R)))
        return s;
    }
    QkRopeArgs q;
    q.qkv = c->pqkv; q.qkv_ld = D.qkvd(); q.T = R; q.pos0 = P;
    q.H = D.H; q.Hkv = D.Hkv; q.hd = D.hd; q.q_gain = w.q_norm; q.k_gain = w.k_norm; q.eps = D.eps;
    q.rope_cos = c->rope_cos; q.rope_sin = c->rope_sin;
    q.kv = kv; q.kv_bf16 = c->kv_bf16; q.page_elems = c->page_elems; q.table = c->ptable; q.q_out = c->pq;
    CK(launch_qk_rope_append(q, c->st, c->pdl));
    AttnPrefillArgs a;
    a.q = c->pq; a.T = R; a.pos0 = P; a.H = D.H; a.Hkv = D.Hkv; a.hd = D.hd;
    a.kv = kv; a.kv_bf16 = c->kv_bf16; a.page_elems = c->page_elems; a.table = c->ptable;
    if (tcp) { a.o16 = c->a16; a.o16lo = c->a16lo; a.o16_ld = D.qd(); }
    else { a.o = c->po; a.o_ld = D.qd(); }
    a.err = c->err;
    a.tc = c->use_tc ? 1 : 0;
    {
      // few query tiles over a long context (a short suffix after a radix
      // hit): split the keys so that the CTAs cover the SMs twice, at least
      // two 64-key tiles per split, within the shared split-KV scratch
      const int ctas = (R + 63) / 64 * D.H;
      const int kt_n = (P + R + 63) / 64;
      int ks = std::min({(2 * c->num_sms + ctas - 1) / ctas, kt_n / 2, 16});
      while (ks > 1 && attn_prefill_part_floats(R, D.H, D.hd, ks) > c->attn_part_floats) --ks;
      if (ks > 1) {
        a.ksplit = ks;
        a.part = c->attn_part;
        a.tickets = c->pf_tickets;
      }
    }
    CK(launch_attn_prefill(a, c->st, c->pdl));
    if (tcp) {
      if ((s = tc(c, w.o, D.d, D.qd(), c->a16, R, D.qd(), c->px, D.d, nullptr, 0, TC_ADD))) return s;
      if ((s = rms16(c, c->px, D.d, R, w.mlp_norm))) return s;
      if ((s = tc(c, w.gu, 2 * D.F, D.d, c->a16, R, D.d, nullptr, 0, c->h16, D.F, TC_SWIGLU_BF16)))
        return s;
      if ((s = tc(c, w.dn, D.d, D.F, c->h16, R, D.F, c->px, D.d, nullptr, 0, TC_ADD))) return s;
    } else {
      if ((s = gemv(c, gv(c, w.o, D.d, D.qd(), c->po, D.qd(), c->px, D.d, GEMV_ADD, nullptr, &w.qo), R)))
        return s;
      if ((s = gemv(c, gv(c, w.gu, 2 * D.F, D.d, c->px, D.d, c->ph, D.F, GEMV_SWIGLU, w.mlp_norm, &w.qgu),
                    R)))
        return s;
      if ((s = gemv(c, gv(c, w.dn, D.d, D.F, c->ph, D.F, c->px, D.d, GEMV_ADD, nullptr, &w.qdn), R)))
        return s;
    }
  }
  return S2_OK;
}

// One segment of a batched prefill: the uncached rows of one sequence.
struct PfSeg {
  int seq, row0, R, P, tab_off, tile0;
};

// The Slow AR over several sequences' uncached rows at once (their rows
// concatenated, staged at ptok / pcodes [NC][R_total] / pmask, the segment
// tables at pf_info / pf_row_seg / pf_tile_seg / pf_tables): one pass of the
// row-wise kernels over all rows; RoPE / KV append per row's sequence; the
// causal attention per segment (one tcgen05 launch over every segment's
// query tiles, else one launch per segment).
int prefill_compute_segs(s2_ctx* c, const std::vector<PfSeg>& segs, int R_total, int n_tiles) {
  const Dims& D = c->D;
  int s;
  EmbedArgs e;
  e.tok_emb = c->tok_emb;
  e.vq_emb = c->vq_emb;
  e.w_bf16 = D.wbf16;
  e.d = D.d;
  e.n_codebooks = D.NC;
  e.codebook_size = D.C;
  e.sem_begin = D.sem;
  e.rows = R_total;
  e.tokens = c->ptok;
  e.codes = c->pcodes;
  e.codes_ld = R_total;
  e.mask = c->pmask;
  e.out = c->px;
  e.out_ld = D.d;
  CK(launch_embed(e, c->st, c->pdl));
  PrefillSegs sg;
  sg.info = c->pf_info;
  sg.row_seg = c->pf_row_seg;
  sg.tile_seg = c->pf_tile_seg;
  sg.tables = c->pf_tables;
  sg.n_tiles = n_tiles;
  const bool tcp = c->use_tc && R_total >= 16;
  for (int l = 0; l < D.Ls; ++l) {
    const LayerW& w = c->slow[l];
    void* kv = static_cast<char*>(c->pool) + (size_t)l * c->layer_elems * c->kvsz;
    if (tcp) {
      if ((s = rms16(c, c->px, D.d, R_total, w.attn_norm))) return s;
      if ((s = tc(c, w.qkv, D.qkvd(), D.d, c->a16, R_total, D.d, c->pqkv, D.qkvd(), nullptr, 0, TC_STORE)))
        return s;
    } else if ((s = gemv(c, gv(c, w.qkv, D.qkvd(), D.d, c->px, D.d, c->pqkv, D.qkvd(), GEMV_STORE, w.attn_norm,
                                 &w.qqkv),
                         R_total))) {
      return s;
    }
    QkRopeArgs q;
    q.qkv = c->pqkv; q.qkv_ld = D.qkvd(); q.T = R_total; q.pos0 = 0;
    q.H = D.H; q.Hkv = D.Hkv; q.hd = D.hd; q.q_gain = w.q_norm; q.k_gain = w.k_norm; q.eps = D.eps;
    q.rope_cos = c->rope_cos; q.rope_sin = c->rope_sin;
    q.kv = kv; q.kv_bf16 = c->kv_bf16; q.page_elems = c->page_elems; q.q_out = c->pq; q.segs = sg;
    CK(launch_qk_rope_append(q, c->st, c->pdl));
    AttnPrefillArgs a;
    a.q = c->pq; a.T = R_total; a.H = D.H; a.Hkv = D.Hkv; a.hd = D.hd;
    a.kv = kv; a.kv_bf16 = c->kv_bf16; a.page_elems = c->page_elems;
    if (tcp) { a.o16 = c->a16; a.o16lo = c->a16lo; a.o16_ld = D.qd(); }
    else { a.o = c->po; a.o_ld = D.qd(); }
    a.err = c->err;
    a.tc = c->use_tc ? 1 : 0;
    a.segs = sg;
    cudaError_t ae = cudaErrorNotSupported;
    if (segs.size() > 1 && D.Hkv * n_tiles >= 128) ae = launch_attn_prefill_segs(a, c->st, c->pdl);
    if (ae == cudaErrorNotSupported) {
      // segment by segment through the single-sequence launcher
      for (const PfSeg& g : segs) {
        AttnPrefillArgs b = a;
        b.segs = PrefillSegs();
        b.q = c->pq + (size_t)g.row0 * D.qd();
        b.T = g.R;
        b.pos0 = g.P;
        b.table = c->pf_tables + g.tab_off;
        if (tcp) { b.o16 = c->a16 + (size_t)g.row0 * D.qd(); b.o16lo = c->a16lo + (size_t)g.row0 * D.qd(); }
        else b.o = c->po + (size_t)g.row0 * D.qd();
        const int ctas = (g.R + 63) / 64 * D.H;
        const int kt_n = (g.P + g.R + 63) / 64;
        int ks = std::min({(2 * c->num_sms + ctas - 1) / ctas, kt_n / 2, 16});
        while (ks > 1 && attn_prefill_part_floats(g.R, D.H, D.hd, ks) > c->attn_part_floats) --ks;
        if (ks > 1) {
          b.ksplit = ks;
          b.part = c->attn_part;
          b.tickets = c->pf_tickets;
        }
        CK(launch_attn_prefill(b, c->st, c->pdl));
      }
    } else {
      CK(ae);
    }
    if (tcp) {
      if ((s = tc(c, w.o, D.d, D.qd(), c->a16, R_total, D.qd(), c->px, D.d, nullptr, 0, TC_ADD))) return s;
      if ((s = rms16(c, c->px, D.d, R_total, w.mlp_norm))) return s;
      if ((s = tc(c, w.gu, 2 * D.F, D.d, c->a16, R_total, D.d, nullptr, 0, c->h16, D.F, TC_SWIGLU_BF16)))
        return s;
      if ((s = tc(c, w.dn, D.d, D.F, c->h16, R_total, D.F, c->px, D.d, nullptr, 0, TC_ADD))) return s;
    } else {
      if ((s = gemv(c, gv(c, w.o, D.d, D.qd(), c->po, D.qd(), c->px, D.d, GEMV_ADD, nullptr, &w.qo), R_total)))
        return s;
      if ((s = gemv(c, gv(c, w.gu, 2 * D.F, D.d, c->px, D.d, c->ph, D.F, GEMV_SWIGLU, w.mlp_norm, &w.qgu),
                    R_total)))
        return s;
      if ((s = gemv(c, gv(c, w.dn, D.d, D.F, c->ph, D.F, c->px, D.d, GEMV_ADD, nullptr, &w.qdn), R_total)))
        return s;
    }
  }
  return S2_OK;
}

}  // namespace

extern "C" int s2_prefill(s2_ctx* c, int32_t seq, const int32_t* tokens, int32_t T,
                          const int32_t* vq_codes, const uint8_t* vq_mask, int32_t* cached_out) {
  if (!c) return S2_EINVAL;
  const Dims& D = c->D;
  if (seq < 0 || seq >= c->opt.max_seqs || !tokens || T < 1 || T > c->opt.max_prompt)
    return fail(c, S2_EINVAL);
  if (c->seqs[seq].live) return fail(c, S2_ESTATE);
  // host copies of the prompt (for validation and radix keys)
  std::vector<int32_t> tok(T), codes;
  std::vector<uint8_t> mask;
  auto fetch = [&](void* dst, const void* src, size_t bytes) {
    if (is_device_ptr(src)) return cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost) == cudaSuccess;
    std::memcpy(dst, src, bytes);
    return true;
  };
  if (!fetch(tok.data(), tokens, (size_t)T * 4)) return fail(c, S2_ECUDA);
  if (vq_mask) {
    mask.resize(T);
    if (!fetch(mask.data(), vq_mask, T)) return fail(c, S2_ECUDA);
  }
  bool any_mask = false;
  for (int t = 0; t < T; ++t) any_mask |= (!mask.empty() && mask[t]);
  codes.assign((size_t)D.NC * T, 0);
  if (any_mask) {
    if (!vq_codes) return fail(c, S2_EINVAL);
    if (!fetch(codes.data(), vq_codes, codes.size() * 4)) return fail(c, S2_ECUDA);
  }
  for (int t = 0; t < T; ++t) {
    if (tok[t] < 0 || tok[t] >= D.V) return fail(c, S2_EINVAL);
    if (any_mask && mask[t])
      for (int k = 0; k < D.NC; ++k) {
        const int v = codes[(size_t)k * T + t];
        if (v < 0 || v >= D.C) return fail(c, S2_EINVAL);
      }
  }
  std::vector<int32_t> keys;
  position_keys(tok.data(), codes.data(), mask.empty() ? nullptr : mask.data(), T, D.NC, keys);
  std::vector<int> table;
  int dropped = 0;
  const int P = admit_prompt(c->pages, c->use_radix ? &c->radix : nullptr, keys, T, table, &dropped);
  c->stats.evicted_pages += dropped;
  if (P < 0) return fail(c, S2_ENOMEM);
  SeqState& S = c->seqs[seq];
  S = SeqState();
  S.live = true;
  S.pages = std::move(table);
  // stage prompt + table
  int* h = c->hstage;
  std::memcpy(h, tok.data(), (size_t)T * 4);
  std::memcpy(h + T, codes.data(), codes.size() * 4);
  std::memcpy(h + T + D.NC * T, S.pages.data(), S.pages.size() * 4);
  CK(cudaMemcpyAsync(c->ptok, h, (size_t)T * 4, cudaMemcpyHostToDevice, c->st));
  CK(cudaMemcpyAsync(c->pcodes, h + T, codes.size() * 4, cudaMemcpyHostToDevice, c->st));
  CK(cudaMemcpyAsync(c->ptable, h + T + D.NC * T, S.pages.size() * 4, cudaMemcpyHostToDevice, c->st));
  if (!mask.empty()) CK(cudaMemcpyAsync(c->pmask, mask.data(), T, cudaMemcpyHostToDevice, c->st));
  else CK(cudaMemsetAsync(c->pmask, 0, T, c->st));
  const long long g0 = g_launch_count;
  int s = prefill_compute(c, P, T);
  c->stats.kernel_launches += g_launch_count - g0;
  if (s) return fail(c, s);
  // the prompt's last residual row primes the first frame
  CK(cudaMemcpyAsync(c->seq_x + (size_t)seq * D.d, c->px + (size_t)(T - P - 1) * D.d, (size_t)D.d * 4,
                     cudaMemcpyDeviceToDevice, c->st));
  // staging buffers are reused by the next call: finish the copies first
  CK(cudaStreamSynchronize(c->st));
  if (c->use_radix)
    for (int pg : c->radix.insert(keys, T, S.pages)) c->pages.incref(pg);
  S.length = T;
  S.primed = true;
  S.finished = false;
  c->stats.prefill_tokens += T - P;
  c->stats.cached_tokens += P;
  if (cached_out) {
    if (is_device_ptr(cached_out)) CK(cudaMemcpy(cached_out, &P, 4, cudaMemcpyHostToDevice));
    else *cached_out = P;
  }
  return S2_OK;
}

extern "C" int s2_prefill_batch(s2_ctx* c, int32_t n, const int32_t* seqs_in, const int32_t* tokens,
                                const int32_t* lengths, const int32_t* vq_codes, const uint8_t* vq_mask,
                                int32_t* cached_out) {
  if (!c) return S2_EINVAL;
  const Dims& D = c->D;
  if (n < 1 || !seqs_in || !tokens || !lengths) return fail(c, S2_EINVAL);
  auto fetch = [&](void* dst, const void* src, size_t bytes) {
    if (is_device_ptr(src)) return cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost) == cudaSuccess;
    std::memcpy(dst, src, bytes);
    return true;
  };
  std::vector<int32_t> seqs(n), lens(n);
  if (!fetch(seqs.data(), seqs_in, (size_t)n * 4) || !fetch(lens.data(), lengths, (size_t)n * 4))
    return fail(c, S2_ECUDA);
  std::vector<size_t> off(n + 1, 0);
  std::vector<char> seen(c->opt.max_seqs, 0);
  for (int i = 0; i < n; ++i) {
    if (seqs[i] < 0 || seqs[i] >= c->opt.max_seqs || lens[i] < 1 || lens[i] > c->opt.max_prompt)
      return fail(c, S2_EINVAL);
    if (seen[seqs[i]]) return fail(c, S2_EINVAL);
    seen[seqs[i]] = 1;
    if (c->seqs[seqs[i]].live) return fail(c, S2_ESTATE);
    off[i + 1] = off[i] + lens[i];
  }
  const size_t total = off[n];
  std::vector<int32_t> tok(total), codes((size_t)D.NC * total, 0);
  std::vector<uint8_t> mask;
  if (!fetch(tok.data(), tokens, total * 4)) return fail(c, S2_ECUDA);
  if (vq_mask) {
    mask.resize(total);
    if (!fetch(mask.data(), vq_mask, total)) return fail(c, S2_ECUDA);
  }
  bool any_mask = false;
  for (size_t t = 0; t < mask.size(); ++t) any_mask |= mask[t] != 0;
  if (any_mask) {
    if (!vq_codes) return fail(c, S2_EINVAL);
    if (!fetch(codes.data(), vq_codes, codes.size() * 4)) return fail(c, S2_ECUDA);
  }
  // sequence i: tokens at off[i], codes block [NC][T_i] at NC * off[i]
  std::vector<std::vector<int32_t>> keys(n);
  for (int i = 0; i < n; ++i) {
    const int T = lens[i];
    const int32_t* ci = codes.data() + (size_t)D.NC * off[i];
    for (int t = 0; t < T; ++t) {
      const size_t g = off[i] + t;
      if (tok[g] < 0 || tok[g] >= D.V) return fail(c, S2_EINVAL);
      if (any_mask && mask[g])
        for (int k = 0; k < D.NC; ++k)
          if (ci[(size_t)k * T + t] < 0 || ci[(size_t)k * T + t] >= D.C) return fail(c, S2_EINVAL);
    }
    position_keys(tok.data() + off[i], ci, mask.empty() ? nullptr : mask.data() + off[i], T, D.NC, keys[i]);
  }

  std::vector<int32_t> cached(n, -1);
  auto report = [&]() {
    if (!cached_out) return true;
    if (is_device_ptr(cached_out))
      return cudaMemcpy(cached_out, cached.data(), (size_t)n * 4, cudaMemcpyHostToDevice) == cudaSuccess;
    std::memcpy(cached_out, cached.data(), (size_t)n * 4);
    return true;
  };
  struct Member {
    int i, P;
  };
  std::vector<Member> group;
  // compute the admitted group: chunks of at most prefill_rows rows and
  // max_batch sequences, each one pass of the Slow AR over their uncached rows
  auto flush = [&]() -> int {
    size_t g0 = 0;
    while (g0 < group.size()) {
      size_t g1 = g0;
      int R_total = 0;
      while (g1 < group.size() && (int)(g1 - g0) < c->opt.max_batch &&
             R_total + lens[group[g1].i] - group[g1].P <= c->opt.prefill_rows) {
        R_total += lens[group[g1].i] - group[g1].P;
        ++g1;
      }
      const int cnt = (int)(g1 - g0);
      std::vector<PfSeg> segs(cnt);
      std::vector<int32_t> ctok(R_total), ccodes((size_t)D.NC * R_total), rseg(R_total), tseg, info(5 * cnt);
      std::vector<uint8_t> cmask(R_total, 0);
      std::vector<int32_t> tables((size_t)cnt * c->max_pages_seq, 0);
      int row = 0, tiles = 0;
      for (int k = 0; k < cnt; ++k) {
        const Member& m = group[g0 + k];
        const int T = lens[m.i], R = T - m.P;
        const int32_t* ci = codes.data() + (size_t)D.NC * off[m.i];
        for (int t = 0; t < R; ++t) {
          const size_t src = off[m.i] + m.P + t;
          ctok[row + t] = tok[src];
          if (!mask.empty()) cmask[row + t] = mask[src];
          for (int q = 0; q < D.NC; ++q) ccodes[(size_t)q * R_total + row + t] = ci[(size_t)q * T + m.P + t];
          rseg[row + t] = k;
        }
        const std::vector<int>& pg = c->seqs[seqs[m.i]].pages;
        std::copy(pg.begin(), pg.end(), tables.begin() + (size_t)k * c->max_pages_seq);
        segs[k] = PfSeg{seqs[m.i], row, R, m.P, k * c->max_pages_seq, tiles};
        const int nt = (R + 31) / 32;
        for (int q = 0; q < nt; ++q) tseg.push_back(k);
        info[5 * k + 0] = row;
        info[5 * k + 1] = R;
        info[5 * k + 2] = m.P;
        info[5 * k + 3] = k * c->max_pages_seq;
        info[5 * k + 4] = tiles;
        row += R;
        tiles += nt;
      }
      CK(cudaMemcpyAsync(c->ptok, ctok.data(), (size_t)R_total * 4, cudaMemcpyHostToDevice, c->st));
      CK(cudaMemcpyAsync(c->pcodes, ccodes.data(), ccodes.size() * 4, cudaMemcpyHostToDevice, c->st));
      CK(cudaMemcpyAsync(c->pmask, cmask.data(), (size_t)R_total, cudaMemcpyHostToDevice, c->st));
      CK(cudaMemcpyAsync(c->pf_row_seg, rseg.data(), (size_t)R_total * 4, cudaMemcpyHostToDevice, c->st));
      CK(cudaMemcpyAsync(c->pf_tile_seg, tseg.data(), tseg.size() * 4, cudaMemcpyHostToDevice, c->st));
      CK(cudaMemcpyAsync(c->pf_info, info.data(), info.size() * 4, cudaMemcpyHostToDevice, c->st));
      CK(cudaMemcpyAsync(c->pf_tables, tables.data(), tables.size() * 4, cudaMemcpyHostToDevice, c->st));
      const long long l0 = g_launch_count;
      int st = prefill_compute_segs(c, segs, R_total, tiles);
      c->stats.kernel_launches += g_launch_count - l0;
      if (st) return st;
      // each prompt's last residual row primes its first frame
      for (const PfSeg& g : segs)
        CK(cudaMemcpyAsync(c->seq_x + (size_t)g.seq * D.d, c->px + (size_t)(g.row0 + g.R - 1) * D.d,
                           (size_t)D.d * 4, cudaMemcpyDeviceToDevice, c->st));
      // the host staging vectors die with this chunk: finish the copies first
      CK(cudaStreamSynchronize(c->st));
      for (int k = 0; k < cnt; ++k) {
        const Member& m = group[g0 + k];
        SeqState& S = c->seqs[seqs[m.i]];
        if (c->use_radix)
          for (int pgid : c->radix.insert(keys[m.i], lens[m.i], S.pages)) c->pages.incref(pgid);
        S.length = lens[m.i];
        S.primed = true;
        S.finished = false;
        c->stats.prefill_tokens += lens[m.i] - m.P;
        c->stats.cached_tokens += m.P;
        cached[m.i] = m.P;
      }
      g0 = g1;
    }
    group.clear();
    return S2_OK;
  };

  for (int i = 0; i < n; ++i) {
    const int T = lens[i];
    // a prompt that would reuse pages a pending one of this group is about to
    // insert waits for the next group (the same hits as calls one by one)
    if (c->use_radix && !group.empty()) {
      const int kPage = c->radix.page();
      const int maxp = (T - 1) / kPage;
      const int tree_hit = (int)c->radix.match(keys[i], T, maxp).size();
      bool dep = false;
      for (const Member& m : group) {
        const int lim = std::min(maxp, lens[m.i] / kPage);
        int common = 0;
        while (common < lim &&
               std::equal(keys[i].begin() + (size_t)common * kPage * kKeyInts,
                          keys[i].begin() + (size_t)(common + 1) * kPage * kKeyInts,
                          keys[m.i].begin() + (size_t)common * kPage * kKeyInts))
          ++common;
        dep |= common > tree_hit;
      }
      if (dep) {
        const int st = flush();
        if (st) {
          report();
          return fail(c, st);
        }
      }
    }
    std::vector<int> table;
    int dropped = 0;
    const int P = admit_prompt(c->pages, c->use_radix ? &c->radix : nullptr, keys[i], T, table, &dropped);
    c->stats.evicted_pages += dropped;
    if (P < 0) {
      const int st = flush();   // the prompts before this one are prefilled, as by separate calls
      report();
      return fail(c, st ? st : S2_ENOMEM);
    }
    SeqState& S = c->seqs[seqs[i]];
    S = SeqState();
    S.live = true;
    S.pages = std::move(table);
    group.push_back(Member{i, P});
  }
  const int st = flush();
  if (!report()) return fail(c, S2_ECUDA);
  return st ? fail(c, st) : S2_OK;
}

extern "C" int s2_release(s2_ctx* c, int32_t seq) {
  if (!c || seq < 0 || seq >= c->opt.max_seqs) return fail(c, S2_EINVAL);
  SeqState& S = c->seqs[seq];
  if (!S.live) return fail(c, S2_ESTATE);
  for (int pg : S.pages) c->pages.decref(pg);
  S = SeqState();
  return S2_OK;
}

namespace {

int run_one(s2_ctx* c, int B, int mode, int f_dbg) {
  if (f_dbg >= 0 || !c->graphs) {
    const long long g0 = g_launch_count;
    int s = enqueue_frame(c, B, mode, f_dbg);
    c->stats.kernel_launches += g_launch_count - g0;
    return s;
  }
  auto key = std::make_pair(B, mode | (c->prefix_on ? 8 : 0));
  auto it = c->graph.find(key);
  if (it == c->graph.end()) {
    cudaGraph_t g;
    CK(cudaStreamBeginCapture(c->st, cudaStreamCaptureModeThreadLocal));
    const long long g0 = g_launch_count;
    int s = enqueue_frame(c, B, mode, -1);
    c->graph_launches[key] = g_launch_count - g0;
    cudaError_t e = cudaStreamEndCapture(c->st, &g);
    if (s) return s;
    if (e != cudaSuccess) return S2_ECUDA;
    cudaGraphExec_t ex;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return S2_ECUDA;
    it = c->graph.emplace(key, ex).first;
  }
  CK(cudaGraphLaunch(it->second, c->st));
  c->stats.kernel_launches += c->graph_launches[key];
  return S2_OK;
}

// The persistent program of a FRAME_FULL frame on B rows: the frame's
// launches recorded (not run), every GEMV re-planned for one batch instance,
// uploaded once.  Null when the frame has an operation the persistent kernel
// does not run (INT8 or fp32 weights, tensor-core projections) or the kernel
// does not fit one CTA per SM.
s2_ctx::PersistProg* persist_prog(s2_ctx* c, int B) {
  auto it = c->persist_progs.find(B);
  if (it != c->persist_progs.end()) return it->second.ok ? &it->second : nullptr;
  s2_ctx::PersistProg& P = c->persist_progs[B];
  OpRecorder rec;
  rec.max_grid = c->num_sms;
  g_recorder = &rec;
  const int s = enqueue_frame(c, B, FRAME_FULL, -1);
  g_recorder = nullptr;
  if (s || !rec.ok || rec.ops.empty()) return nullptr;
  int rows = 1;
  for (const PersistOp& op : rec.ops)
    if (op.kind == PK_GEMV) rows = std::max(rows, op.g.B);
  const int maxb = rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : 8;
  for (PersistOp& op : rec.ops)
    if (op.kind == PK_GEMV && !gemv_persist_layout(op, maxb)) return nullptr;
  const size_t smem = persist_smem_bytes(rec.ops);
  const int grid = persist_grid(c->num_sms, maxb, smem);
  if (grid != c->num_sms) return nullptr;
  const size_t bytes = rec.ops.size() * sizeof(PersistOp);
  if (dev_alloc(c, &P.ops, bytes) != cudaSuccess) {
    P.ops = nullptr;
    cudaGetLastError();
    return nullptr;
  }
  if (cudaMemcpy(P.ops, rec.ops.data(), bytes, cudaMemcpyHostToDevice) != cudaSuccess) return nullptr;
  P.n_ops = (int)rec.ops.size();
  P.maxb = maxb;
  P.grid = grid;
  P.smem = smem;
  P.ok = true;
  return &P;
}

// The streaming program of a FRAME_FULL frame on B rows: the frame's
// launches recorded (not run) and planned for the streaming kernel, uploaded
// once.  Null when the frame has an operation the streaming kernel does not
// run or its shared memory does not fit one CTA per SM.
s2_ctx::StreamProg* stream_prog(s2_ctx* c, int B) {
  auto it = c->stream_progs.find(B);
  if (it != c->stream_progs.end()) return it->second.ok ? &it->second : nullptr;
  s2_ctx::StreamProg& P = c->stream_progs[B];
  if (B > 2) return nullptr;
  OpRecorder rec;
  rec.max_grid = c->num_sms;
  g_recorder = &rec;
  const int s = enqueue_frame(c, B, FRAME_FULL, -1);
  g_recorder = nullptr;
  if (s || !rec.ok || rec.ops.empty()) return nullptr;
  std::vector<StreamPlan> plan;
  StreamLayout L;
  int maxb = 0;
  if (!stream_plan(rec.ops, c->num_sms, plan, L, maxb)) return nullptr;
  if (!stream_fits(maxb, stream_smem_bytes(L))) return nullptr;
  const size_t ob = rec.ops.size() * sizeof(PersistOp), pb = plan.size() * sizeof(StreamPlan);
  if (dev_alloc(c, &P.ops, ob) != cudaSuccess || dev_alloc(c, &P.plan, pb) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (cudaMemcpy(P.ops, rec.ops.data(), ob, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(P.plan, plan.data(), pb, cudaMemcpyHostToDevice) != cudaSuccess)
    return nullptr;
  P.n_ops = (int)rec.ops.size();
  P.maxb = maxb;
  P.grid = c->num_sms;
  P.L = L;
  P.ok = true;
  return &P;
}

// n frames for rows [0, B); on the first frame of a call only rows [0, Bc)
// (the continuing sequences) run a slow step, the primed ones already hold
// their prompt's last hidden state.  With S2_FLAG_PERSIST the full frames
// run in one persistent kernel when the frame allows it; otherwise frame by
// frame from CUDA graphs.
int run_frames(s2_ctx* c, int B, int Bc, int n, bool first_chunk) {
  const bool dbg = c->dbg_logits || c->dbg_hidden || c->dbg_layers;
  auto go = [&](int b, int mode, int fdbg) {
    if (dbg) {
      const long long g0 = g_launch_count;
      int s = enqueue_frame(c, b, mode, fdbg);
      c->stats.kernel_launches += g_launch_count - g0;
      return s;
    }
    return run_one(c, b, mode, -1);
  };
  int f = 0, s;
  if (first_chunk && Bc < B) {
    const int fdbg = dbg && c->dbg_frames > 0 ? 0 : -1;
    if (Bc > 0 && (s = go(Bc, FRAME_SLOW, fdbg))) return s;
    if ((s = go(B, FRAME_HEADFAST, fdbg))) return s;
    f = 1;
  }
  if (f < n && !dbg && c->stream && !c->persist) {
    if (s2_ctx::StreamProg* P = stream_prog(c, B)) {
      // barrier counter, abort flag and the tickets start at zero
      CK(cudaMemsetAsync(c->pwords, 0, 64 * sizeof(unsigned), c->st));
      CK(cudaMemsetAsync(c->ticket, 0, 16 * sizeof(unsigned), c->st));
      CK(cudaMemsetAsync(c->attn_tickets, 0, ((size_t)c->opt.max_batch * c->D.Hkv + 16) * sizeof(unsigned),
                         c->st));
      // S2_STREAM_TRACE=<file>: CTA 0's per-operation timing of one frame
      // (a profiling aid; synchronises the stream)
      const char* trace_path = std::getenv("S2_STREAM_TRACE");
      constexpr int kTW = 6;   // words per operation (see k_stream.cu)
      unsigned long long* trace = nullptr;
      if (trace_path && cudaMalloc(&trace, (size_t)P->n_ops * kTW * 8) != cudaSuccess) trace = nullptr;
      if (trace) CK(cudaMemsetAsync(trace, 0, (size_t)P->n_ops * kTW * 8, c->st));
      const long long g0 = g_launch_count;
      const cudaError_t e = launch_stream(P->ops, P->plan, P->n_ops, n - f, P->maxb, P->L, c->pwords,
                                          reinterpret_cast<int*>(c->pwords + 32), c->err, P->grid, c->st,
                                          trace);
      c->stats.kernel_launches += g_launch_count - g0;
      if (trace) {
        std::vector<unsigned long long> h((size_t)P->n_ops * kTW);
        std::vector<PersistOp> ops(P->n_ops);
        cudaStreamSynchronize(c->st);
        cudaMemcpy(h.data(), trace, h.size() * 8, cudaMemcpyDeviceToHost);
        cudaMemcpy(ops.data(), P->ops, ops.size() * sizeof(PersistOp), cudaMemcpyDeviceToHost);
        cudaFree(trace);
        if (FILE* fp = std::fopen(trace_path, "w")) {
          std::fprintf(fp, "# op kind N K rows barrier_us body_us prologue_us first_slot_us last_slot_us\n");
          for (int i = 0; i < P->n_ops; ++i) {
            const PersistOp& op = ops[i];
            const unsigned long long* w = &h[(size_t)i * kTW];
            const char* kind = op.kind == PK_GEMV ? "gemv" : op.kind == PK_ATTN ? "attn" : "embed";
            const int N = op.kind == PK_GEMV ? op.g.N : 0, K = op.kind == PK_GEMV ? op.g.K : 0;
            const int rows = op.kind == PK_GEMV ? op.g.B : op.kind == PK_ATTN ? op.at.B * op.at.m : op.e.rows;
            auto us = [&](int a, int b) { return w[a] && w[b] ? (double)(w[b] - w[a]) * 1e-3 : 0.0; };
            std::fprintf(fp, "%d %s %d %d %d %.3f %.3f %.3f %.3f %.3f\n", i, kind, N, K, rows, us(0, 1),
                         us(1, 5), us(1, 2), us(1, 3), us(1, 4));
          }
          std::fclose(fp);
        }
      }
      CK(e);
      return S2_OK;
    }
  }
  if (f < n && !dbg && c->persist) {
    if (s2_ctx::PersistProg* P = persist_prog(c, B)) {
      // barrier counter, abort flag and the tickets start at zero
      CK(cudaMemsetAsync(c->pwords, 0, 64 * sizeof(unsigned), c->st));
      CK(cudaMemsetAsync(c->ticket, 0, 16 * sizeof(unsigned), c->st));
      CK(cudaMemsetAsync(c->attn_tickets, 0, ((size_t)c->opt.max_batch * c->D.Hkv + 16) * sizeof(unsigned),
                         c->st));
      // S2_PERSIST_TRACE=<file>: write CTA 0's per-operation timing of one
      // frame (a profiling aid; synchronises the stream)
      const char* trace_path = std::getenv("S2_PERSIST_TRACE");
      unsigned long long* trace = nullptr;
      if (trace_path && cudaMalloc(&trace, (size_t)P->n_ops * 3 * 8) != cudaSuccess) trace = nullptr;
      const long long g0 = g_launch_count;
      // fault injection: the barrier before the first attention operation
      // (no copies are in flight there: the preceding GEMV consumed all it
      // issued, and attention prefetches nothing before its wait)
      int fault_op = -1;
      if (c->fault_barrier) {
        std::vector<PersistOp> ops(P->n_ops);
        CK(cudaMemcpy(ops.data(), P->ops, ops.size() * sizeof(PersistOp), cudaMemcpyDeviceToHost));
        for (int i = 1; i < P->n_ops && fault_op < 0; ++i)
          if (ops[i].kind == PK_ATTN) fault_op = i;
      }
      const cudaError_t e = launch_persist(P->ops, P->n_ops, n - f, P->maxb, c->pwords,
                                           reinterpret_cast<int*>(c->pwords + 32), c->err, P->grid,
                                           P->smem, c->st, trace, fault_op,
                                           fault_op >= 0 ? 50000000ull : 0ull);
      c->stats.kernel_launches += g_launch_count - g0;
      if (trace) {
        std::vector<unsigned long long> h((size_t)P->n_ops * 3);
        std::vector<PersistOp> ops(P->n_ops);
        cudaStreamSynchronize(c->st);
        cudaMemcpy(h.data(), trace, h.size() * 8, cudaMemcpyDeviceToHost);
        cudaMemcpy(ops.data(), P->ops, ops.size() * sizeof(PersistOp), cudaMemcpyDeviceToHost);
        cudaFree(trace);
        if (FILE* fp = std::fopen(trace_path, "w")) {
          std::fprintf(fp, "# op kind N K rows barrier_us body_us\n");
          for (int i = 0; i < P->n_ops; ++i) {
            const PersistOp& op = ops[i];
            const char* kind = op.kind == PK_GEMV ? "gemv" : op.kind == PK_ATTN ? "attn" : "embed";
            const int N = op.kind == PK_GEMV ? op.g.N : 0, K = op.kind == PK_GEMV ? op.g.K : 0;
            const int rows = op.kind == PK_GEMV ? op.g.B : op.kind == PK_ATTN ? op.at.B * op.at.m : op.e.rows;
            std::fprintf(fp, "%d %s %d %d %d %.3f %.3f\n", i, kind, N, K, rows,
                         (double)(h[i * 3 + 1] - h[i * 3]) * 1e-3, (double)(h[i * 3 + 2] - h[i * 3 + 1]) * 1e-3);
          }
          std::fclose(fp);
        }
      }
      CK(e);
      return S2_OK;
    }
  }
  for (; f < n; ++f)
    if ((s = go(B, FRAME_FULL, dbg && f < c->dbg_frames ? f : -1))) return s;
  return S2_OK;
}

}  // namespace

extern "C" int s2_decode_frames(s2_ctx* c, const int32_t* seqs_in, int32_t B, int32_t n,
                                int32_t* out) {
  if (!c || !seqs_in || !out || B < 1 || B > c->opt.max_batch || n < 1) return fail(c, S2_EINVAL);
  const Dims& D = c->D;
  std::vector<int32_t> seqs(B);
  if (is_device_ptr(seqs_in)) {
    if (cudaMemcpy(seqs.data(), seqs_in, (size_t)B * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
      return fail(c, S2_ECUDA);
  } else {
    std::memcpy(seqs.data(), seqs_in, (size_t)B * 4);
  }
  std::vector<char> seen(c->opt.max_seqs, 0);
  for (int b = 0; b < B; ++b) {
    const int q = seqs[b];
    if (q < 0 || q >= c->opt.max_seqs || seen[q]) return fail(c, S2_EINVAL);
    seen[q] = 1;
    if (!c->seqs[q].live || c->seqs[q].finished) return fail(c, S2_ESTATE);
  }
  // internal row order: continuing sequences first, then the freshly primed ones
  std::vector<int> perm;  // internal row -> caller index
  for (int b = 0; b < B; ++b)
    if (!c->seqs[seqs[b]].primed) perm.push_back(b);
  const int Bc = (int)perm.size();
  for (int b = 0; b < B; ++b)
    if (c->seqs[seqs[b]].primed) perm.push_back(b);
  bool identity = true;
  for (int r = 0; r < B; ++r) identity &= perm[r] == r;
  // reserve pages for every slow step of the call (primed rows skip frame 0's)
  auto slow_steps = [&](int b) { return n - (c->seqs[seqs[b]].primed ? 1 : 0); };
  std::vector<std::vector<int>*> tables(B);
  std::vector<int> want(B);
  for (int b = 0; b < B; ++b) {
    SeqState& S = c->seqs[seqs[b]];
    want[b] = S.length + slow_steps(b);
    if (want[b] > c->opt.max_ctx) return fail(c, S2_EINVAL);
    tables[b] = &S.pages;
  }
  int dropped = 0;
  const bool reserved =
      reserve_pages(c->pages, c->use_radix ? &c->radix : nullptr, tables, want, 16, &dropped);
  c->stats.evicted_pages += dropped;
  if (!reserved) return fail(c, S2_ENOMEM);
  // the leading pages every row's table holds in common (radix-shared
  // prompt pages): their keys go to the tensor-core prefix attention
  {
    int common = 0;
    if (c->use_prefix_tc && B >= 2 && tc_rows(c, B)) {
      size_t np = tables[0]->size();
      for (int b = 1; b < B; ++b) np = std::min(np, tables[b]->size());
      while ((size_t)common < np) {
        const int pg = (*tables[0])[common];
        bool same = true;
        for (int b = 1; b < B && same; ++b) same = (*tables[b])[common] == pg;
        if (!same) break;
        ++common;
      }
    }
    const int shared = common * 16;
    c->prefix_on = shared >= 64 && c->px_planes && shared <= c->px_stride;
    c->shared_host = c->prefix_on ? shared : 0;
    if (c->prefix_on) {
      c->hstage[0] = shared;
      CK(cudaMemcpyAsync(c->shared_len, c->hstage, 4, cudaMemcpyHostToDevice, c->st));
      CK(cudaStreamSynchronize(c->st));   // the staging word is reused below
    }
  }
  const bool out_dev = is_device_ptr(out);
  bool first_chunk = true;
  if (c->eos >= 0) CK(cudaMemsetAsync(c->done, 0, (size_t)B * sizeof(int), c->st));
  for (int f0 = 0; f0 < n; f0 += c->max_frames) {
    const int nn = std::min(c->max_frames, n - f0);
    // per-call metadata in internal row order: page tables, position bases, slots
    int* h = c->hstage;
    const int mp = c->max_pages_seq;
    for (int r = 0; r < B; ++r) {
      const SeqState& S = c->seqs[seqs[perm[r]]];
      const int fsf = (first_chunk && S.primed) ? 1 : 0;
      std::memcpy(h + (size_t)r * mp, S.pages.data(), S.pages.size() * 4);
      h[(size_t)B * mp + r] = S.length - fsf;
      h[(size_t)B * mp + B + r] = seqs[perm[r]];
    }
    CK(cudaMemcpyAsync(c->table_b, h, (size_t)B * mp * 4, cudaMemcpyHostToDevice, c->st));
    CK(cudaMemcpyAsync(c->pos_base, h + (size_t)B * mp, (size_t)B * 4, cudaMemcpyHostToDevice, c->st));
    CK(cudaMemcpyAsync(c->slots, h + (size_t)B * mp + B, (size_t)B * 4, cudaMemcpyHostToDevice, c->st));
    if (first_chunk && c->prefix_on) {
      // the shared prefix's keys of every Slow AR layer as operand images
      // (the pages do not change while the rows share them)
      PrefixPlanesArgs pp;
      pp.kv = c->pool;
      pp.layer_bytes = (long long)(c->layer_elems * c->kvsz);
      pp.kv_bf16 = c->kv_bf16 ? 1 : 0;
      pp.page_elems = c->page_elems;
      pp.table = c->table_b;
      pp.Hkv = D.Hkv;
      pp.hd = D.hd;
      pp.layers = D.Ls;
      pp.P = c->shared_host;
      pp.stride = c->px_stride;
      pp.planes = c->px_planes;
      CK(launch_attn_prefix_planes(pp, c->st));
      c->stats.kernel_launches += 1;
    }
    if (first_chunk) {
      // primed rows start from their prompt's last residual, continuing rows
      // from their last frame's codes (each row only reads its own kind)
      c->stats.kernel_launches += 2;
      CK(launch_gather_rows(c->x_slow, D.d, c->seq_x, D.d, c->slots, B, D.d, c->st, false));
      CK(launch_gather_rows_i32(c->last_codes, D.NC, c->seq_codes, D.NC, c->slots, B, D.NC, c->st, false));
    }
    CK(cudaMemsetAsync(c->frame_ctr, 0, 4, c->st));
    int s = run_frames(c, B, first_chunk ? Bc : B, nn, first_chunk);
    if (s) return fail(c, s);
    const cudaMemcpyKind kind = out_dev ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost;
    if (identity) {
      CK(cudaMemcpy2DAsync(out + (size_t)f0 * D.NC, (size_t)n * D.NC * 4, c->codes_all,
                           (size_t)c->max_frames * D.NC * 4, (size_t)nn * D.NC * 4, B, kind, c->st));
    } else {
      for (int r = 0; r < B; ++r)
        CK(cudaMemcpyAsync(out + ((size_t)perm[r] * n + f0) * D.NC,
                           c->codes_all + (size_t)r * c->max_frames * D.NC, (size_t)nn * D.NC * 4,
                           kind, c->st));
    }
    // staging is reused: wait for the uploads of this chunk
    CK(cudaStreamSynchronize(c->st));
    if (c->eos >= 0) {
      // rows that picked the end-of-speech row: their sequences are finished
      CK(cudaMemcpy(c->hstage, c->done, (size_t)B * sizeof(int), cudaMemcpyDeviceToHost));
      for (int r = 0; r < B; ++r)
        if (c->hstage[r]) c->seqs[seqs[perm[r]]].finished = true;
    }
    for (int b = 0; b < B; ++b) {
      SeqState& S = c->seqs[seqs[b]];
      S.length += nn - ((first_chunk && S.primed) ? 1 : 0);
      S.primed = false;
    }
    first_chunk = false;
  }
  CK(launch_scatter_rows_i32(c->seq_codes, D.NC, c->last_codes, D.NC, c->slots, B, D.NC, c->st, false));
  c->stats.kernel_launches += 1;
  c->stats.frames_decoded += (int64_t)B * n;
  if (c->ftrace && c->ft_next > 0) {
    // the last frame's timeline: "id kind" lines, then "id cta entry wait prologue exit"
    std::vector<unsigned long long> h((size_t)c->ft_next * kFrameTraceCtas * 4);
    CK(cudaStreamSynchronize(c->st));
    CK(cudaMemcpy(h.data(), c->ftrace, h.size() * 8, cudaMemcpyDeviceToHost));
    if (FILE* fp = std::fopen(c->ftrace_path.c_str(), "w")) {
      for (int i = 0; i < c->ft_next; ++i) std::fprintf(fp, "launch %d %s\n", i, c->ft_kind[i].c_str());
      for (int i = 0; i < c->ft_next; ++i)
        for (int k = 0; k < c->ft_ctas[i]; ++k) {
          const unsigned long long* t = &h[((size_t)i * kFrameTraceCtas + k) * 4];
          if (t[0]) std::fprintf(fp, "%d %d %llu %llu %llu %llu\n", i, k, t[0], t[1], t[2], t[3]);
        }
      std::fclose(fp);
    }
  }
  // host debug sinks: copy the shadows the kernels wrote
  for (int i = 0; i < 3; ++i)
    if (c->dbg_host[i])
      CK(cudaMemcpyAsync(c->dbg_host[i], c->dbg_shadow[i], debug_sink_floats(c, i, B) * sizeof(float),
                         cudaMemcpyDeviceToHost, c->st));
  if (!out_dev || c->dbg_host[0] || c->dbg_host[1] || c->dbg_host[2]) CK(cudaStreamSynchronize(c->st));
  return S2_OK;
}

extern "C" int s2_radix_clear(s2_ctx* c) {
  if (!c) return S2_EINVAL;
  for (int pg : c->radix.clear()) c->pages.decref(pg);
  return S2_OK;
}

extern "C" int s2_stats(s2_ctx* c, s2_stats_t* out) {
  if (!c || !out) return S2_EINVAL;
  int e = 0;
  cudaStreamSynchronize(c->st);
  cudaMemcpy(&e, c->err, 4, cudaMemcpyDeviceToHost);
  c->stats.device_error = e;
  c->stats.pages_used = c->pages.n_total() - c->pages.n_free();
  c->stats.radix_pages = c->radix.held();
  *out = c->stats;
  return S2_OK;
}

extern "C" int s2_set_debug_sinks(s2_ctx* c, float* logits, float* hidden, float* layers,
                                  int32_t max_frames) {
  if (!c || max_frames < 0) return S2_EINVAL;
  cudaStreamSynchronize(c->st);
  free_debug_shadows(c);
  c->dbg_frames = max_frames;
  float* in[3] = {logits, hidden, layers};
  float* dev[3] = {nullptr, nullptr, nullptr};
  for (int i = 0; i < 3; ++i) {
    if (!in[i]) continue;
    if (is_device_ptr(in[i])) {
      dev[i] = in[i];
      continue;
    }
    // host buffer: the kernels write a device shadow sized for the largest batch
    const size_t bytes = debug_sink_floats(c, i, c->opt.max_batch) * sizeof(float);
    if (bytes && dev_alloc(c, &c->dbg_shadow[i], bytes) != cudaSuccess) {
      cudaGetLastError();
      free_debug_shadows(c);
      c->dbg_logits = c->dbg_hidden = c->dbg_layers = nullptr;
      return fail(c, S2_ENOMEM);
    }
    c->dbg_host[i] = in[i];
    dev[i] = c->dbg_shadow[i];
  }
  c->dbg_logits = dev[0];
  c->dbg_hidden = dev[1];
  c->dbg_layers = dev[2];
  return S2_OK;
}

// Captured frames carry the head configuration: drop them.
static void drop_frames(s2_ctx* c) {
  for (auto& kv : c->graph) cudaGraphExecDestroy(kv.second);
  c->graph.clear();
  c->graph_launches.clear();
  cudaStreamSynchronize(c->st);
  for (auto& kv : c->persist_progs)
    if (kv.second.ops) cudaFree(kv.second.ops);
  c->persist_progs.clear();
  for (auto& kv : c->stream_progs) {
    if (kv.second.ops) cudaFree(kv.second.ops);
    if (kv.second.plan) cudaFree(kv.second.plan);
  }
  c->stream_progs.clear();
}

extern "C" int s2_set_stop(s2_ctx* c, int32_t eos_token) {
  if (!c) return S2_EINVAL;
  if (eos_token >= 0 && (eos_token >= c->D.V || eos_token >= c->D.sem)) return S2_EINVAL;
  c->eos = eos_token < 0 ? -1 : eos_token;
  drop_frames(c);
  return S2_OK;
}

extern "C" int s2_set_top_p(s2_ctx* c, float top_p_slow, float top_p_fast) {
  if (!c || !(top_p_slow > 0.f && top_p_slow <= 1.f) || !(top_p_fast > 0.f && top_p_fast <= 1.f))
    return S2_EINVAL;
  c->top_p_slow = top_p_slow;
  c->top_p_fast = top_p_fast;
  drop_frames(c);
  return S2_OK;
}

extern "C" int s2_set_sampling(s2_ctx* c, float temperature_slow, float temperature_fast,
                               uint64_t seed) {
  if (!c || !(temperature_slow >= 0.f) || !(temperature_fast >= 0.f)) return S2_EINVAL;
  c->temp_slow = temperature_slow;
  c->temp_fast = temperature_fast;
  c->seed = seed;
  drop_frames(c);  // the captured frames carry the old parameters
  return S2_OK;
}

extern "C" int s2_model_dims(s2_ctx* c, int32_t* d) {
  if (!c || !d) return S2_EINVAL;
  const Dims& D = c->D;
  int32_t v[12] = {D.d, D.H, D.Hkv, D.hd, D.F, D.Ls, D.Lf, D.V, D.sem, D.NC, D.C, D.wbf16};
  std::memcpy(d, v, sizeof v);
  return S2_OK;
}
