// DAC vocoder runtime behind include/s2_dac.h: weight-file loading and
// repacking, activation buffers, tensor maps and the decode sequence.
//
// Decode of `batch` sequences of n frames (codec stage: "SGLang Day-0
// Support for FishAudio S2", Architecture, Stage 3; 2,048 samples per frame:
// "s2pro-native", What happens to a sentence):
//   1. clear the halo rows of every bf16 plane buffer (the convolutions' zero
//      padding: the sequence length sets where the halos are);
//   2. codebook lookup + projections -> latent (fp32 and planes);
//   3. input convolution (k=7) -> level 1, planes hold Snake(x) for block 0;
//   4. per upsampling block: the transposed convolution (one launch, both
//      phase groups), then per residual unit conv k=7 (planes P = Snake of
//      its output) and conv k=1 (+ residual into the fp32 stream; planes X =
//      Snake of the result for whatever reads it next);
//   5. output convolution to one channel + tanh (CUDA cores).
// Every convolution is one launch of the tcgen05 implicit-GEMM kernel.
#include "s2.h"
#include "s2_dac.h"
#include "s2_kernels.h"
#include "dac.h"
#include "tma_map.h"

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

using namespace s2;

namespace {

constexpr int kCh = 64;            // channel padding (one TMA box width)
constexpr int kSlackRows = 1024;   // rows past the last sequence (reads of masked tail rows)

int pad64(int c) { return (c + kCh - 1) / kCh * kCh; }

struct VEntry {
  uint32_t dtype, ndim;
  uint64_t shape[4], off, nbytes;
};

struct Level {
  int C = 0, Cp = 0;
  long long up = 1;            // samples of this level per frame
  long long cap_rows = 0;
  float* F = nullptr;          // fp32 value (residual stream / stage output)
  __nv_bfloat16 *Xh = nullptr, *Xl = nullptr;   // planes read by the next convolution
  __nv_bfloat16 *Ph = nullptr, *Pl = nullptr;   // residual units' inner planes
  CUtensorMap mXh, mXl, mPh, mPl;
};

struct Conv {
  int in_lv = 0;
  bool in_P = false;
  int out_lv = 0;
  bool out_F = false, out_P = false, resid = false;
  int groups = 1, taps = 1, n_group = 0, phases = 1, up = 1, nt = 64, kchunks = 1, cout_pad = 0;
  int tap_off[2][kDacMaxTaps] = {};
  size_t w_off = 0;            // element offset in the packed weights
  int w_rows = 0;
  size_t bias_off = 0;         // float offsets in the parameter buffer
  long long alpha_off = -1, inv_off = -1;
  CUtensorMap mW;
};

int pick_nt(int n_group) {
  for (int nt : {256, 192, 128, 64})
    if (n_group % nt == 0) return nt;
  return 0;
}

float bf16_to_f(uint16_t u) {
  uint32_t v = (uint32_t)u << 16;
  float f;
  std::memcpy(&f, &v, 4);
  return f;
}

}  // namespace

struct s2_vocoder {
  int latent = 0, dim = 0, cbd = 0, ncb = 0, csize = 0, nb = 0;
  int rates[8] = {};
  int hop = 1;
  int max_seqs = 0, max_frames = 0;
  cudaStream_t st = nullptr;
  __nv_bfloat16* wbuf = nullptr;
  float* pbuf = nullptr;
  size_t cb_off = 0, pw_off = 0, pb_off = 0, outw_off = 0, outb_off = 0;
  std::vector<Level> lv;       // lv[0] latent, lv[1] input conv, lv[2 + i] block i
  std::vector<Conv> convs;
  int32_t* codes_dev = nullptr;
  float* audio_dev = nullptr;
  float* tables = nullptr;     // projected codebook tables [ncb, csize, latent]
  int* err = nullptr;
  int last_B = 0, last_n = 0;
  long long last_launches = 0;
  std::vector<void*> allocs;
  // per-launch timing (s2_vocoder_set_profile): an event before every launch
  // and one after the last, on the vocoder's stream
  bool profile = false;
  std::vector<cudaEvent_t> ev;
  int n_ev = 0;
};

namespace {

cudaError_t valloc(s2_vocoder* v, void** p, size_t bytes) {
  cudaError_t e = cudaMalloc(p, bytes);
  if (e == cudaSuccess) v->allocs.push_back(*p);
  return e;
}

// S2_ENOMEM when the device is out of memory, S2_ECUDA for any other failure
// (no device, a sticky error)
int alloc_status(cudaError_t e) { return e == cudaErrorMemoryAllocation ? S2_ENOMEM : S2_ECUDA; }

void vfree(s2_vocoder* v) {
  for (void* p : v->allocs) cudaFree(p);
  v->allocs.clear();
}

bool is_dev(const void* p) {
  cudaPointerAttributes at;
  if (!p || cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

struct FileData {
  std::map<std::string, VEntry> e;
  std::vector<uint8_t> bytes;   // the whole file
  const VEntry* get(const std::string& n, std::initializer_list<uint64_t> shape, uint32_t dtype) const {
    auto it = e.find(n);
    if (it == e.end() || it->second.dtype != dtype || it->second.ndim != shape.size()) return nullptr;
    int i = 0;
    for (uint64_t s : shape)
      if (it->second.shape[i++] != s) return nullptr;
    const uint64_t el = dtype == 1 ? 2 : 4;
    uint64_t n_el = 1;
    for (uint64_t s : shape) n_el *= s;
    if (it->second.nbytes != n_el * el || it->second.off + it->second.nbytes > bytes.size()) return nullptr;
    return &it->second;
  }
  const float* f32(const VEntry* x) const { return reinterpret_cast<const float*>(bytes.data() + x->off); }
  const uint16_t* b16(const VEntry* x) const { return reinterpret_cast<const uint16_t*>(bytes.data() + x->off); }
};

int read_file(const char* path, FileData& fd, s2_vocoder* v) {
  FILE* f = std::fopen(path, "rb");
  if (!f) return S2_EBADFILE;
  std::fseek(f, 0, SEEK_END);
  const long sz = std::ftell(f);
  std::fseek(f, 0, SEEK_SET);
  if (sz < 128) {
    std::fclose(f);
    return S2_EBADFILE;
  }
  fd.bytes.resize((size_t)sz);
  const size_t got = std::fread(fd.bytes.data(), 1, (size_t)sz, f);
  std::fclose(f);
  if (got != (size_t)sz) return S2_EBADFILE;
  const uint8_t* h = fd.bytes.data();
  uint32_t ver, nb, ntens;
  int32_t dims[5], rates[8];
  uint64_t data0;
  if (std::memcmp(h, "S2DACVOC", 8)) return S2_EBADFILE;
  std::memcpy(&ver, h + 8, 4);
  std::memcpy(&nb, h + 12, 4);
  std::memcpy(dims, h + 16, 20);
  std::memcpy(rates, h + 36, 32);
  std::memcpy(&ntens, h + 68, 4);
  std::memcpy(&data0, h + 76, 8);
  if (ver != 1 || nb < 1 || nb > 8 || ntens > 4096 || 128 + (size_t)ntens * 128 > (size_t)sz) return S2_EBADFILE;
  v->latent = dims[0];
  v->dim = dims[1];
  v->cbd = dims[2];
  v->ncb = dims[3];
  v->csize = dims[4];
  v->nb = (int)nb;
  for (int i = 0; i < 8; ++i) v->rates[i] = i < (int)nb ? rates[i] : 0;
  for (uint32_t i = 0; i < ntens; ++i) {
    const uint8_t* p = h + 128 + (size_t)i * 128;
    char name[65] = {};
    std::memcpy(name, p, 64);
    VEntry x;
    std::memcpy(&x.dtype, p + 64, 4);
    std::memcpy(&x.ndim, p + 68, 4);
    std::memcpy(x.shape, p + 72, 32);
    std::memcpy(&x.off, p + 104, 8);
    std::memcpy(&x.nbytes, p + 112, 8);
    if (x.ndim > 4) return S2_EBADFILE;
    fd.e[name] = x;
  }
  return S2_OK;
}

int create_impl(s2_vocoder* v, const char* path, int max_seqs, int max_frames) {
  FileData fd;
  int rc = read_file(path, fd, v);
  if (rc) return rc;
  if (v->latent <= 0 || v->dim <= 0 || v->cbd < 1 || v->cbd > 16 || v->ncb < 1 || v->ncb > 16 || v->csize < 1)
    return S2_EINVAL;
  v->hop = 1;
  for (int i = 0; i < v->nb; ++i) {
    if (v->rates[i] < 2 || v->rates[i] % 2 || v->rates[i] > 64) return S2_EINVAL;
    v->hop *= v->rates[i];
  }
  if (v->dim % (1 << v->nb) || (v->dim >> v->nb) > 96) return S2_EINVAL;
  v->max_seqs = max_seqs;
  v->max_frames = max_frames;

  // ---- levels
  v->lv.resize(2 + v->nb);
  v->lv[0].C = v->latent;
  v->lv[1].C = v->dim;
  long long up = 1;
  for (int i = 0; i < v->nb; ++i) {
    up *= v->rates[i];
    v->lv[2 + i].C = v->dim >> (i + 1);
    v->lv[2 + i].up = up;
  }
  for (Level& L : v->lv) {
    L.Cp = pad64(L.C);
    L.cap_rows = (long long)max_seqs * (max_frames * L.up + 2 * kDacHalo) + kSlackRows;
  }

  // ---- parameters (f32) and packed weights (bf16), built on the host
  std::vector<float> P;
  std::vector<uint16_t> W;
  auto push_f = [&](const float* src, int n, int npad, float fill) {
    const size_t o = P.size();
    for (int i = 0; i < npad; ++i) P.push_back(i < n ? src[i] : fill);
    while (P.size() % 8) P.push_back(0.f);   // 32-byte aligned vectors
    return o;
  };
  auto push_alpha = [&](const VEntry* a, int n, int npad, Conv& c) {
    const float* s = fd.f32(a);
    c.alpha_off = (long long)push_f(s, n, npad, 1.f);
    std::vector<float> inv(n);
    for (int i = 0; i < n; ++i) inv[i] = (float)(1.0 / ((double)s[i] + 1e-9));
    c.inv_off = (long long)push_f(inv.data(), n, npad, 1.f);
  };
  const int L = v->latent, D = v->dim;
  const VEntry* cb = fd.get("rvq.codebook", {(uint64_t)v->ncb, (uint64_t)v->csize, (uint64_t)v->cbd}, 0);
  const VEntry* pw = fd.get("rvq.proj_w", {(uint64_t)v->ncb, (uint64_t)L, (uint64_t)v->cbd}, 0);
  const VEntry* pb = fd.get("rvq.proj_b", {(uint64_t)v->ncb, (uint64_t)L}, 0);
  if (!cb || !pw || !pb) return S2_EBADFILE;
  v->cb_off = push_f(fd.f32(cb), (int)(cb->nbytes / 4), (int)(cb->nbytes / 4), 0.f);
  v->pw_off = push_f(fd.f32(pw), (int)(pw->nbytes / 4), (int)(pw->nbytes / 4), 0.f);
  v->pb_off = push_f(fd.f32(pb), (int)(pb->nbytes / 4), (int)(pb->nbytes / 4), 0.f);

  // plain convolution w [cout, cin, k] -> packed [k][cout_pad][cin_pad]
  auto add_conv = [&](const std::string& pre, int cin, int cout, int k, int dil, int in_lv, bool in_P, int out_lv,
                      bool out_F, bool out_P, bool resid, const VEntry* alpha_next) -> bool {
    const VEntry* w = fd.get(pre + ".w", {(uint64_t)cout, (uint64_t)cin, (uint64_t)k}, 1);
    const VEntry* bb = fd.get(pre + ".b", {(uint64_t)cout}, 0);
    if (!w || !bb) return false;
    Conv c;
    c.in_lv = in_lv; c.in_P = in_P; c.out_lv = out_lv; c.out_F = out_F; c.out_P = out_P; c.resid = resid;
    const int cip = pad64(cin), cop = pad64(cout);
    c.groups = 1; c.taps = k; c.n_group = cop; c.phases = 1; c.up = 1; c.kchunks = cip / kCh; c.cout_pad = cop;
    for (int j = 0; j < k; ++j) c.tap_off[0][j] = c.tap_off[1][j] = j * dil - (k / 2) * dil;
    c.nt = pick_nt(cop);
    c.w_off = W.size();
    c.w_rows = k * cop;
    W.resize(W.size() + (size_t)k * cop * cip, 0);
    const uint16_t* src = fd.b16(w);
    for (int j = 0; j < k; ++j)
      for (int o = 0; o < cout; ++o)
        for (int i = 0; i < cin; ++i)
          W[c.w_off + ((size_t)j * cop + o) * cip + i] = src[((size_t)o * cin + i) * k + j];
    c.bias_off = push_f(fd.f32(bb), cout, cop, 0.f);
    if (alpha_next) push_alpha(alpha_next, cout, cop, c);
    v->convs.push_back(c);
    return true;
  };
  // transposed convolution w [cin, cout, 2s], stride s, crop s/2: phases
  // r < s/2 (group 0) read x[q] (k = r + s/2) and x[q-1] (k = r + 3s/2);
  // phases r >= s/2 (group 1) read x[q+1] (k = r - s/2) and x[q] (k = r + s/2)
  auto add_convT = [&](const std::string& pre, int cin, int cout, int s, int in_lv, int out_lv,
                       const VEntry* alpha_next) -> bool {
    const VEntry* w = fd.get(pre + ".w", {(uint64_t)cin, (uint64_t)cout, (uint64_t)(2 * s)}, 1);
    const VEntry* bb = fd.get(pre + ".b", {(uint64_t)cout}, 0);
    if (!w || !bb) return false;
    Conv c;
    c.in_lv = in_lv; c.out_lv = out_lv; c.out_F = true;
    const int cip = pad64(cin), cop = pad64(cout), h = s / 2;
    c.groups = 2; c.taps = 2; c.phases = h; c.n_group = h * cop; c.up = s; c.kchunks = cip / kCh; c.cout_pad = cop;
    c.tap_off[0][0] = 0; c.tap_off[0][1] = -1;
    c.tap_off[1][0] = 1; c.tap_off[1][1] = 0;
    c.nt = pick_nt(c.n_group);
    c.w_off = W.size();
    c.w_rows = 2 * 2 * c.n_group;
    W.resize(W.size() + (size_t)c.w_rows * cip, 0);
    const uint16_t* src = fd.b16(w);
    for (int g = 0; g < 2; ++g)
      for (int tap = 0; tap < 2; ++tap)
        for (int rl = 0; rl < h; ++rl) {
          const int r = g * h + rl;
          const int kk = g == 0 ? (tap == 0 ? r + h : r + 3 * h) : (tap == 0 ? r - h : r + h);
          for (int o = 0; o < cout; ++o)
            for (int i = 0; i < cin; ++i)
              W[c.w_off + (((size_t)(g * 2 + tap) * c.n_group) + (size_t)rl * cop + o) * cip + i] =
                  src[((size_t)i * cout + o) * (2 * s) + kk];
        }
    c.bias_off = push_f(fd.f32(bb), cout, cop, 0.f);
    push_alpha(alpha_next, cout, cop, c);
    v->convs.push_back(c);
    return true;
  };

  auto alpha = [&](const std::string& n, int c) { return fd.get(n, {(uint64_t)c}, 0); };
  const int clast = v->dim >> v->nb;
  if (!alpha("block.0.alpha", D)) return S2_EBADFILE;
  if (!add_conv("conv_in", L, D, 7, 1, 0, false, 1, true, false, false, alpha("block.0.alpha", D)))
    return S2_EBADFILE;
  for (int i = 0; i < v->nb; ++i) {
    const int ci = v->dim >> i, co = v->dim >> (i + 1), lo = 2 + i;
    const std::string p = "block." + std::to_string(i) + ".";
    const VEntry* a1 = alpha(p + "res.0.alpha1", co);
    if (!a1 || !add_convT(p + "up", ci, co, v->rates[i], lo - 1, lo, a1)) return S2_EBADFILE;
    for (int j = 0; j < 3; ++j) {
      const std::string q = p + "res." + std::to_string(j) + ".";
      const int dil = j == 0 ? 1 : j == 1 ? 3 : 9;
      const VEntry* a2 = alpha(q + "alpha2", co);
      const VEntry* nxt = j < 2 ? alpha(p + "res." + std::to_string(j + 1) + ".alpha1", co)
                                : i + 1 < v->nb ? alpha("block." + std::to_string(i + 1) + ".alpha", co)
                                                : alpha("out.alpha", co);
      if (!a2 || !nxt) return S2_EBADFILE;
      if (!add_conv(q + "conv1", co, co, 7, dil, lo, false, lo, false, true, false, a2)) return S2_EBADFILE;
      if (!add_conv(q + "conv2", co, co, 1, 1, lo, true, lo, true, false, true, nxt)) return S2_EBADFILE;
    }
  }
  const VEntry* ow = fd.get("out.w", {1, (uint64_t)clast, 7}, 1);
  const VEntry* ob = fd.get("out.b", {1}, 0);
  if (!ow || !ob) return S2_EBADFILE;
  {
    // [7][c8] with the channels padded to a multiple of 8 by zeros (the
    // planes' padding channels are 0 as well)
    const int c8 = (clast + 7) / 8 * 8;
    std::vector<float> wt(7 * c8, 0.f);
    for (int j = 0; j < 7; ++j)
      for (int c = 0; c < clast; ++c) wt[j * c8 + c] = bf16_to_f(fd.b16(ow)[c * 7 + j]);
    v->outw_off = push_f(wt.data(), 7 * c8, 7 * c8, 0.f);
    v->outb_off = push_f(fd.f32(ob), 1, 1, 0.f);
  }
  for (const Conv& c : v->convs)
    if (!c.nt) return S2_EINVAL;

  // ---- device memory
  if (cudaError_t e = valloc(v, reinterpret_cast<void**>(&v->wbuf), W.size() * 2)) return alloc_status(e);
  if (cudaError_t e = valloc(v, reinterpret_cast<void**>(&v->pbuf), P.size() * 4)) return alloc_status(e);
  if (cudaMemcpy(v->wbuf, W.data(), W.size() * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(v->pbuf, P.data(), P.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return S2_ECUDA;
  for (size_t i = 0; i < v->lv.size(); ++i) {
    Level& Lv = v->lv[i];
    const size_t n = (size_t)Lv.cap_rows * Lv.Cp;
    void *F, *xh, *xl;
    if (cudaError_t e = valloc(v, &F, n * 4)) return alloc_status(e);
    if (cudaError_t e = valloc(v, &xh, n * 2)) return alloc_status(e);
    if (cudaError_t e = valloc(v, &xl, n * 2)) return alloc_status(e);
    Lv.F = static_cast<float*>(F);
    Lv.Xh = static_cast<__nv_bfloat16*>(xh);
    Lv.Xl = static_cast<__nv_bfloat16*>(xl);
    if (cudaMemset(F, 0, n * 4) || cudaMemset(xh, 0, n * 2) || cudaMemset(xl, 0, n * 2)) return S2_ECUDA;
    if (!tma_map_bf16_2d(&Lv.mXh, xh, Lv.cap_rows, Lv.Cp, Lv.Cp, 128) ||
        !tma_map_bf16_2d(&Lv.mXl, xl, Lv.cap_rows, Lv.Cp, Lv.Cp, 128))
      return S2_ECUDA;
    if (i >= 2) {
      void *ph, *pl;
      if (cudaError_t e = valloc(v, &ph, n * 2)) return alloc_status(e);
      if (cudaError_t e = valloc(v, &pl, n * 2)) return alloc_status(e);
      Lv.Ph = static_cast<__nv_bfloat16*>(ph);
      Lv.Pl = static_cast<__nv_bfloat16*>(pl);
      if (cudaMemset(ph, 0, n * 2) || cudaMemset(pl, 0, n * 2)) return S2_ECUDA;
      if (!tma_map_bf16_2d(&Lv.mPh, ph, Lv.cap_rows, Lv.Cp, Lv.Cp, 128) ||
          !tma_map_bf16_2d(&Lv.mPl, pl, Lv.cap_rows, Lv.Cp, Lv.Cp, 128))
        return S2_ECUDA;
    }
  }
  for (Conv& c : v->convs) {
    const int cip = c.kchunks * kCh;
    if (!tma_map_bf16_2d(&c.mW, v->wbuf + c.w_off, c.w_rows, cip, cip, c.nt)) return S2_ECUDA;
  }
  if (cudaError_t e = valloc(v, reinterpret_cast<void**>(&v->codes_dev), (size_t)max_seqs * max_frames * v->ncb * 4))
    return alloc_status(e);
  if (cudaError_t e = valloc(v, reinterpret_cast<void**>(&v->audio_dev), (size_t)max_seqs * max_frames * v->hop * 4))
    return alloc_status(e);
  if (cudaError_t e = valloc(v, reinterpret_cast<void**>(&v->err), 64)) return alloc_status(e);
  if (cudaMemset(v->err, 0, 64)) return S2_ECUDA;
  if (v->latent % 4) return S2_EINVAL;
  if (cudaError_t e = valloc(v, reinterpret_cast<void**>(&v->tables), (size_t)v->ncb * v->csize * v->latent * 4))
    return alloc_status(e);
  if (launch_dac_project(v->ncb, v->csize, v->cbd, v->latent, v->pbuf + v->cb_off, v->pbuf + v->pw_off,
                         v->pbuf + v->pb_off, v->tables, nullptr) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    return S2_ECUDA;
  return S2_OK;
}

// Event before the next launch (profiling only).
cudaError_t mark(s2_vocoder* v) {
  if (!v->profile) return cudaSuccess;
  if (v->n_ev == (int)v->ev.size()) {
    cudaEvent_t e;
    cudaError_t r = cudaEventCreate(&e);
    if (r) return r;
    v->ev.push_back(e);
  }
  return cudaEventRecord(v->ev[v->n_ev++], v->st);
}

cudaError_t run_decode(s2_vocoder* v, const int32_t* codes, int B, int n, float* audio) {
  const long long T0 = n;
  v->n_ev = 0;
  auto S_of = [&](const Level& L) { return (int)(T0 * L.up + 2 * kDacHalo); };
  auto T_of = [&](const Level& L) { return (int)(T0 * L.up); };
  DacHaloJobs jobs = {};
  for (size_t i = 0; i < v->lv.size(); ++i) {
    const Level& L = v->lv[i];
    jobs.job[jobs.n++] = {L.Xh, L.Xl, L.Cp, S_of(L), T_of(L)};
    if (L.Ph) jobs.job[jobs.n++] = {L.Ph, L.Pl, L.Cp, S_of(L), T_of(L)};
  }
  cudaError_t e = mark(v);
  if (!e) e = launch_dac_zero_halos(jobs, B, v->st);
  if (!e) e = mark(v);
  if (e) return e;
  const Level& Z = v->lv[0];
  e = launch_dac_rvq(codes, B, n, v->ncb, v->csize, v->latent, v->tables, Z.F, Z.Xh, Z.Xl, Z.Cp, S_of(Z), v->err,
                     v->st);
  if (e) return e;
  for (const Conv& c : v->convs) {
    const Level& I = v->lv[c.in_lv];
    Level& O = v->lv[c.out_lv];
    DacConvParams p = {};
    p.taps = c.taps;
    std::memcpy(p.tap_off, c.tap_off, sizeof(p.tap_off));
    p.kchunks = c.kchunks;
    p.n_group = c.n_group;
    p.phases = c.phases;
    p.cphase = c.cout_pad;
    p.up = c.up;
    p.T_in = T_of(I);
    p.S_in = S_of(I);
    p.S_out = S_of(O);
    p.tiles_per_seq = (p.T_in + 127) / 128;
    p.bias = v->pbuf + c.bias_off;
    p.alpha = c.alpha_off >= 0 ? v->pbuf + c.alpha_off : nullptr;
    p.inv_alpha = c.inv_off >= 0 ? v->pbuf + c.inv_off : nullptr;
    p.resid = c.resid ? O.F : nullptr;
    p.out_f32 = c.out_F ? O.F : nullptr;
    p.out_hi = c.out_P ? O.Ph : O.Xh;
    p.out_lo = c.out_P ? O.Pl : O.Xl;
    p.err = v->err;
    e = mark(v);
    if (!e) e = launch_dac_conv(c.in_P ? I.mPh : I.mXh, c.in_P ? I.mPl : I.mXl, c.mW, p, c.groups, c.nt, B, v->st);
    if (e) return e;
  }
  const Level& last = v->lv.back();
  e = mark(v);
  if (!e) e = launch_dac_out(last.Xh, last.Xl, last.Cp, (last.C + 7) / 8 * 8, v->pbuf + v->outw_off,
                             v->pbuf + v->outb_off, B, T_of(last), S_of(last), audio, v->st);
  if (!e) e = mark(v);
  return e;
}

}  // namespace

extern "C" int s2_vocoder_create(const char* path, int32_t max_seqs, int32_t max_frames, void* cuda_stream,
                                 s2_vocoder** out) {
  if (!out) return S2_EINVAL;
  *out = nullptr;
  if (!path || max_seqs <= 0 || max_frames <= 0 || (long long)max_seqs * max_frames > (1LL << 24)) return S2_EINVAL;
  s2_vocoder* v = new s2_vocoder();
  v->st = static_cast<cudaStream_t>(cuda_stream);
  const int rc = create_impl(v, path, max_seqs, max_frames);
  if (rc) {
    vfree(v);
    cudaGetLastError();
    delete v;
    return rc;
  }
  *out = v;
  return S2_OK;
}

extern "C" void s2_vocoder_destroy(s2_vocoder* v) {
  if (!v) return;
  cudaStreamSynchronize(v->st);
  for (cudaEvent_t e : v->ev) cudaEventDestroy(e);
  vfree(v);
  delete v;
}

extern "C" int32_t s2_vocoder_hop(const s2_vocoder* v) { return v ? v->hop : 0; }

extern "C" int64_t s2_vocoder_last_launches(const s2_vocoder* v) { return v ? v->last_launches : 0; }

extern "C" int s2_vocoder_decode(s2_vocoder* v, const int32_t* codes, int32_t batch, int32_t n, float* audio) {
  if (!v || !codes || !audio || batch < 1 || batch > v->max_seqs || n < 1 || n > v->max_frames) return S2_EINVAL;
  const size_t ncodes = (size_t)batch * n * v->ncb;
  const size_t nsamp = (size_t)batch * n * v->hop;
  const bool codes_dev = is_dev(codes), audio_dev = is_dev(audio);
  if (!codes_dev)
    for (size_t i = 0; i < ncodes; ++i)
      if (codes[i] < 0 || codes[i] >= v->csize) return S2_EINVAL;
  const long long l0 = g_launch_count;
  cudaError_t e = cudaSuccess;
  const int32_t* cd = codes;
  if (!codes_dev) {
    e = cudaMemcpyAsync(v->codes_dev, codes, ncodes * 4, cudaMemcpyHostToDevice, v->st);
    cd = v->codes_dev;
  }
  float* ad = audio_dev ? audio : v->audio_dev;
  if (!e) e = cudaMemsetAsync(v->err, 0, 4, v->st);
  if (!e) e = run_decode(v, cd, batch, n, ad);
  if (!e && !audio_dev) e = cudaMemcpyAsync(audio, ad, nsamp * 4, cudaMemcpyDeviceToHost, v->st);
  int herr = 0;
  if (!e) e = cudaMemcpyAsync(&herr, v->err, 4, cudaMemcpyDeviceToHost, v->st);
  if (!e) e = cudaStreamSynchronize(v->st);
  v->last_launches = g_launch_count - l0;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return S2_ECUDA;
  }
  v->last_B = batch;
  v->last_n = n;
  if (herr == 4) return S2_EINVAL;
  if (herr) return S2_ETIMEOUT;
  return S2_OK;
}

extern "C" int s2_vocoder_read_stage(s2_vocoder* v, int32_t stage, float* dst, size_t bytes) {
  if (!v || !dst || !v->last_B || stage < -1 || stage > v->nb) return S2_EINVAL;
  const Level& L = v->lv[stage + 1];
  const int T = (int)(v->last_n * L.up), S = T + 2 * kDacHalo;
  if (bytes < (size_t)v->last_B * T * L.C * 4) return S2_EINVAL;
  for (int b = 0; b < v->last_B; ++b)
    if (cudaMemcpy2D(dst + (size_t)b * T * L.C, (size_t)L.C * 4, L.F + ((size_t)b * S + kDacHalo) * L.Cp,
                     (size_t)L.Cp * 4, (size_t)L.C * 4, (size_t)T, cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      return S2_ECUDA;
    }
  return S2_OK;
}

extern "C" int s2_vocoder_set_profile(s2_vocoder* v, int32_t on) {
  if (!v) return S2_EINVAL;
  v->profile = on != 0;
  return S2_OK;
}

extern "C" int32_t s2_vocoder_profile(s2_vocoder* v, float* ms, int32_t max) {
  if (!v || !v->profile || v->n_ev < 2) return 0;
  const int n = v->n_ev - 1 < max ? v->n_ev - 1 : max;
  for (int i = 0; i < n; ++i)
    if (!ms || cudaEventElapsedTime(&ms[i], v->ev[i], v->ev[i + 1]) != cudaSuccess) {
      cudaGetLastError();
      return S2_ECUDA;
    }
  return n;
}
