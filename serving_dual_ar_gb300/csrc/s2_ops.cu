// Per-kernel C ABI (include/s2_ops.h): thin marshalling onto the launchers.
#include "s2.h"
#include "s2_ops.h"
#include "s2_kernels.h"

#include <cmath>
#include <cstring>

namespace s2 {

thread_local long long g_launch_count = 0;

static int num_sms_current() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

static int status(cudaError_t e) {
  if (e == cudaSuccess) return S2_OK;
  if (e == cudaErrorInvalidValue) {
    cudaGetLastError();
    return S2_EINVAL;
  }
  return S2_ECUDA;
}

static float bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  float r;
  std::memcpy(&r, &u, 4);
  return r;
}

// cos/sin of p * theta^(-2i/hd) in double, rounded to float, then to bf16
// with ties to even, kept as float.
void rope_fill(int n_pos, int hd, float theta, float* cs, float* sn) {
  const int half = hd / 2;
  for (int p = 0; p < n_pos; ++p)
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow((double)theta, -2.0 * i / (double)hd);
      const double a = (double)p * inv;
      cs[(size_t)p * half + i] = bf16_rne((float)std::cos(a));
      sn[(size_t)p * half + i] = bf16_rne((float)std::sin(a));
    }
}

}  // namespace s2

using namespace s2;

extern "C" int s2op_gemv(const void* W, int w_bf16, int N, int K, const float* X, int ldx, int B,
                         const float* gain, float eps, float* Y, int ldy, int mode, int grid_ctas,
                         void* stream) {
  if (!W || !X || !Y || N <= 0 || K <= 0 || B < 1 || B > 8 || mode < 0 || mode > 2) return S2_EINVAL;
  GemvArgs a;
  a.W = W;
  a.w_is_bf16 = w_bf16 ? 1 : 0;
  a.N = N;
  a.K = K;
  a.unit = mode == GEMV_SWIGLU ? 2 : 1;
  a.X = X;
  a.ldx = ldx;
  a.B = B;
  a.gain = gain;
  a.eps = eps;
  a.Y = Y;
  a.ldy = ldy;
  a.mode = mode;
  if (N % a.unit) return S2_EINVAL;
  int grid = grid_ctas > 0 ? grid_ctas : gemv_grid(a, num_sms_current());
  if (grid > N / a.unit) grid = N / a.unit;
  return status(launch_gemv(a, static_cast<cudaStream_t>(stream), false, grid));
}

extern "C" size_t s2op_argmax_workspace_bytes(int B) {
  return (size_t)(B > 0 ? B : 1) * 2048 * 8 + 256;
}

extern "C" int s2op_gemv_argmax(const void* W, int w_bf16, int N, int K, const float* X, int ldx,
                                int B, const float* gain, float eps, int32_t* codes, float* logits,
                                void* workspace, void* stream) {
  if (!W || !X || !codes || !workspace || N <= 0 || B < 1 || B > 8) return S2_EINVAL;
  GemvArgs a;
  a.W = W;
  a.w_is_bf16 = w_bf16 ? 1 : 0;
  a.N = N;
  a.K = K;
  a.X = X;
  a.ldx = ldx;
  a.B = B;
  a.gain = gain;
  a.eps = eps;
  a.mode = GEMV_ARGMAX;
  int grid = gemv_grid(a, num_sms_current());
  if (grid > 2048) grid = 2048;
  char* ws = static_cast<char*>(workspace);
  a.ticket = reinterpret_cast<unsigned*>(ws);
  a.part_val = reinterpret_cast<float*>(ws + 256);
  a.part_idx = reinterpret_cast<int*>(ws + 256 + (size_t)B * 2048 * 4);
  a.codes = codes;
  a.codes_ld = 1;
  a.codes_per_frame = 1;
  a.code_slot = 0;
  a.logits = logits;
  a.logits_ld = N;
  a.tail_d = K;
  return status(launch_gemv(a, static_cast<cudaStream_t>(stream), false, grid));
}

extern "C" size_t s2op_tc_gemm_workspace_bytes(int N, int K, int T, int split_k) {
  int tn, sk;
  tc_gemm_plan(N, K, T, num_sms_current(), &tn, &sk);
  if (split_k > 0) sk = split_k;
  return tc_gemm_ws_floats(N, T, sk) * 4;
}

extern "C" size_t s2op_tc_gemm_tickets(int N, int T) { return tc_gemm_tickets(N, T); }

extern "C" int s2op_tc_gemm(const void* A, int N, int K, const void* Bm, int T, int ldb, float* Y,
                            int ldy, void* Y16, int ldy16, int epi, int split_k, float* workspace,
                            uint32_t* tickets, void* stream) {
  if (epi < 0 || epi > 2 || split_k < 0) return S2_EINVAL;
  TcGemmArgs a;
  a.A = static_cast<const __nv_bfloat16*>(A);
  a.N = N;
  a.K = K;
  a.Bm = static_cast<const __nv_bfloat16*>(Bm);
  a.T = T;
  a.ldb = ldb;
  a.Y = Y;
  a.ldy = ldy;
  a.Y16 = static_cast<__nv_bfloat16*>(Y16);
  a.ldy16 = ldy16;
  a.epi = epi;
  a.split_k = split_k;
  a.ws = workspace;
  a.tickets = tickets;
  return status(launch_tc_gemm(a, static_cast<cudaStream_t>(stream), false, num_sms_current()));
}

extern "C" size_t s2op_tc_gemm2_workspace_bytes(int N, int K, int T, int split_k) {
  int tn, sk;
  tc_gemm_plan(N, K, T, num_sms_current(), &tn, &sk, true);
  if (split_k > 0) sk = split_k;
  return tc_gemm_ws_floats(N, T, sk, true) * 4;
}

extern "C" size_t s2op_tc_gemm2_tickets(int N, int T) { return tc_gemm_tickets(N, T, true); }

extern "C" int s2op_tc_gemm2(const void* A, int N, int K, const void* Bhi, const void* Blo, int T,
                             int ldb, float* Y, int ldy, void* Y16, void* Y16lo, int ldy16, int epi,
                             int split_k, float* workspace, uint32_t* tickets, void* stream) {
  if (epi < 0 || epi > 2 || split_k < 0 || !Blo) return S2_EINVAL;
  TcGemmArgs a;
  a.A = static_cast<const __nv_bfloat16*>(A);
  a.N = N;
  a.K = K;
  a.Bm = static_cast<const __nv_bfloat16*>(Bhi);
  a.Blo = static_cast<const __nv_bfloat16*>(Blo);
  a.T = T;
  a.ldb = ldb;
  a.Y = Y;
  a.ldy = ldy;
  a.Y16 = static_cast<__nv_bfloat16*>(Y16);
  a.Y16lo = static_cast<__nv_bfloat16*>(Y16lo);
  a.ldy16 = ldy16;
  a.epi = epi;
  a.split_k = split_k;
  a.ws = workspace;
  a.tickets = tickets;
  return status(launch_tc_gemm(a, static_cast<cudaStream_t>(stream), false, num_sms_current()));
}

extern "C" int s2op_tc_set_trace(void* buf, int max_ctas) {
  if (max_ctas < 0 || (max_ctas > 0 && !buf)) return S2_EINVAL;
  tc_set_trace(static_cast<unsigned long long*>(buf), max_ctas);
  return S2_OK;
}

extern "C" int s2op_attn_prefix_set_trace(void* buf, int max_ctas) {
  if (max_ctas < 0 || (max_ctas > 0 && !buf)) return S2_EINVAL;
  attn_prefix_set_trace(static_cast<unsigned long long*>(buf), max_ctas);
  return S2_OK;
}

extern "C" int s2op_attn_decode_pick_split(int B, int H, int Hkv, int hd, int kv_bf16) {
  if (B < 1 || Hkv < 1 || H % Hkv) return S2_EINVAL;
  return attn_pick_split(B, Hkv, num_sms_current(), attn_decode_ctas_per_sm(hd, H / Hkv, kv_bf16 != 0), 16);
}

extern "C" size_t s2op_attn_decode_workspace_bytes(int B, int m, int H, int Hkv, int hd, int nsplit) {
  return attn_decode_scratch_floats(B, m, H, hd, nsplit) * 4 + 256 + (size_t)B * Hkv * 4;
}

extern "C" int s2op_attn_decode(const float* qkv, int qkv_ld, int B, int m, int H, int Hkv, int hd,
                                const float* q_gain, const float* k_gain, float eps,
                                const float* rope_cos, const float* rope_sin, const int32_t* pos,
                                void* kv, int kv_bf16, const int32_t* table, int table_ld, float* o,
                                int o_ld, int nsplit, void* workspace, void* stream) {
  if (!qkv || !pos || !kv || !table || !o || !q_gain || !k_gain || !rope_cos || !rope_sin)
    return S2_EINVAL;
  if (B < 1 || m < 1 || m > 2 || nsplit < 1 || Hkv < 1 || H % Hkv) return S2_EINVAL;
  if (nsplit > 1 && !workspace) return S2_EINVAL;
  AttnDecodeArgs a;
  a.qkv = qkv;
  a.qkv_ld = qkv_ld;
  a.B = B;
  a.m = m;
  a.H = H;
  a.Hkv = Hkv;
  a.hd = hd;
  a.q_gain = q_gain;
  a.k_gain = k_gain;
  a.eps = eps;
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.pos_base = pos;
  a.kv = kv;
  a.kv_bf16 = kv_bf16 ? 1 : 0;
  a.page_elems = 2LL * Hkv * 16 * hd;
  a.table = table;
  a.table_ld = table_ld;
  a.o = o;
  a.o_ld = o_ld;
  a.nsplit = nsplit;
  if (workspace) {
    const size_t pf = attn_decode_scratch_floats(B, m, H, hd, nsplit);
    a.part = static_cast<float*>(workspace);
    a.tickets = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + (pf * 4 + 255) / 256 * 256);
  }
  return status(launch_attn_decode(a, static_cast<cudaStream_t>(stream), false));
}

// Workspace of the shared-prefix ops: the prefix keys' operand images, the
// query tiles, the shared length (one device word in 256 bytes), the
// split-KV partial slots and their tickets.
static size_t prefix_plane_region(int Hkv, int hd, int max_keys) {
  return (attn_prefix_plane_bytes(Hkv, hd, attn_prefix_plane_stride(max_keys > 0 ? max_keys : 1), 1) + 255) /
         256 * 256;
}

extern "C" size_t s2op_attn_decode_prefix_workspace_bytes(int B, int H, int Hkv, int hd, int nsplit,
                                                         int max_keys) {
  const size_t pf = attn_decode_scratch_floats(B, 1, H, hd, nsplit > 0 ? nsplit : 1);
  return prefix_plane_region(Hkv, hd, max_keys) + attn_prefix_qimg_bytes(B > 0 ? B : 1, Hkv) + 256 +
         (pf * 4 + 255) / 256 * 256 + (size_t)B * Hkv * 4;
}

extern "C" int s2op_attn_prefix_planes(const void* kv, int kv_bf16, const int32_t* table, int Hkv, int hd,
                                       int shared_len, int max_keys, void* workspace, void* stream) {
  if (!kv || !table || !workspace || Hkv < 1 || hd != 128 || shared_len < 16 || shared_len % 16 ||
      shared_len > max_keys)
    return S2_EINVAL;
  PrefixPlanesArgs p;
  p.kv = kv;
  p.layer_bytes = 0;
  p.kv_bf16 = kv_bf16 ? 1 : 0;
  p.page_elems = 2LL * Hkv * 16 * hd;
  p.table = table;
  p.Hkv = Hkv;
  p.hd = hd;
  p.layers = 1;
  p.P = shared_len;
  p.stride = attn_prefix_plane_stride(max_keys);
  p.planes = workspace;
  return status(launch_attn_prefix_planes(p, static_cast<cudaStream_t>(stream)));
}

extern "C" int s2op_attn_decode_shared_prefix(const float* qkv, int qkv_ld, int B, int H, int Hkv, int hd,
                                              const float* q_gain, const float* k_gain, float eps,
                                              const float* rope_cos, const float* rope_sin,
                                              const int32_t* pos, void* kv, int kv_bf16,
                                              const int32_t* table, int table_ld, int shared_len,
                                              int max_keys, float* o, int o_ld, int nsplit,
                                              void* workspace, void* stream) {
  if (!qkv || !pos || !kv || !table || !o || !q_gain || !k_gain || !rope_cos || !rope_sin || !workspace)
    return S2_EINVAL;
  if (B < 1 || nsplit < 1 || Hkv < 1 || H != 4 * Hkv || hd != 128 || shared_len < 0 || shared_len % 16 ||
      shared_len > max_keys)
    return S2_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const void* planes = ws;
  ws += prefix_plane_region(Hkv, hd, max_keys);
  uint8_t* q_img = reinterpret_cast<uint8_t*>(ws);
  ws += attn_prefix_qimg_bytes(B, Hkv);
  const size_t pf = attn_decode_scratch_floats(B, 1, H, hd, nsplit);
  int* len = reinterpret_cast<int*>(ws);
  if (cudaMemcpyAsync(len, &shared_len, 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)   // the host word is a local
    return S2_ECUDA;
  AttnDecodeArgs a;
  a.qkv = qkv;
  a.qkv_ld = qkv_ld;
  a.B = B;
  a.m = 1;
  a.H = H;
  a.Hkv = Hkv;
  a.hd = hd;
  a.q_gain = q_gain;
  a.k_gain = k_gain;
  a.eps = eps;
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.pos_base = pos;
  a.kv = kv;
  a.kv_bf16 = kv_bf16 ? 1 : 0;
  a.page_elems = 2LL * Hkv * 16 * hd;
  a.table = table;
  a.table_ld = table_ld;
  a.o = o;
  a.o_ld = o_ld;
  a.nsplit = nsplit;
  a.part = reinterpret_cast<float*>(ws + 256);
  a.tickets = reinterpret_cast<unsigned*>(ws + 256 + (pf * 4 + 255) / 256 * 256);
  a.key_begin = len;
  a.part_base = 0;
  a.merge_later = 1;
  a.q_img = q_img;
  // the private keys' split-KV partials (and the query tiles), then the
  // prefix's cluster merges them
  cudaError_t e = launch_attn_decode(a, st, false);
  if (e == cudaSuccess) e = launch_attn_prefix_cl(a, planes, attn_prefix_plane_stride(max_keys), st, true);
  return status(e);
}

extern "C" int s2op_attn_prefill(const float* qkv, int qkv_ld, int T, int pos0, int H, int Hkv, int hd,
                                 const float* q_gain, const float* k_gain, float eps,
                                 const float* rope_cos, const float* rope_sin, void* kv, int kv_bf16,
                                 const int32_t* table, float* q_scratch, float* o, int o_ld,
                                 void* stream) {
  if (!qkv || !kv || !table || !q_scratch || !o || T < 1 || pos0 < 0 || Hkv < 1 || H % Hkv)
    return S2_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  QkRopeArgs q;
  q.qkv = qkv;
  q.qkv_ld = qkv_ld;
  q.T = T;
  q.pos0 = pos0;
  q.H = H;
  q.Hkv = Hkv;
  q.hd = hd;
  q.q_gain = q_gain;
  q.k_gain = k_gain;
  q.eps = eps;
  q.rope_cos = rope_cos;
  q.rope_sin = rope_sin;
  q.kv = kv;
  q.kv_bf16 = kv_bf16 ? 1 : 0;
  q.page_elems = 2LL * Hkv * 16 * hd;
  q.table = table;
  q.q_out = q_scratch;
  int s = status(launch_qk_rope_append(q, st, false));
  if (s) return s;
  AttnPrefillArgs a;
  a.q = q_scratch;
  a.T = T;
  a.pos0 = pos0;
  a.H = H;
  a.Hkv = Hkv;
  a.hd = hd;
  a.kv = kv;
  a.kv_bf16 = q.kv_bf16;
  a.page_elems = q.page_elems;
  a.table = table;
  a.o = o;
  a.o_ld = o_ld;
  return status(launch_attn_prefill(a, st, false));
}

extern "C" int s2op_rope_table(int n_pos, int hd, float theta, float* cos_out, float* sin_out) {
  if (n_pos < 1 || hd < 2 || hd % 2 || !cos_out || !sin_out) return S2_EINVAL;
  rope_fill(n_pos, hd, theta, cos_out, sin_out);
  return S2_OK;
}
