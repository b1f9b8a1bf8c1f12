// Decode attention with library-owned scratch: the variant of
// s2op_attn_decode for callers that cannot allocate device memory.
//
// The split-KV partials and the per-(sequence, kv head) tickets live in one
// file-scope __device__ array of a fixed size.  The array exists on every GPU
// that loads this library, for as long as the library stays loaded.  Host
// code never uses the array's name as a device address: the address comes
// from cudaGetSymbolAddress, fetched once per device, with that device
// current, on the first call made on it.
#include "s2.h"
#include "s2_ops.h"
#include "s2_kernels.h"

#include <mutex>

namespace {

__device__ __align__(256) unsigned char g_attn_scratch[S2_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up once).
int scratch_for_current_device(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return S2_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return S2_ECUDA;
    }
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_ptr[dev];
  return S2_OK;
}

}  // namespace

extern "C" size_t s2op_attn_decode_noalloc_max_bytes(void) { return S2_NOALLOC_SCRATCH_BYTES; }

extern "C" int s2op_attn_decode_noalloc(const float* qkv, int qkv_ld, int B, int m, int H, int Hkv,
                                        int hd, const float* q_gain, const float* k_gain, float eps,
                                        const float* rope_cos, const float* rope_sin,
                                        const int32_t* pos, void* kv, int kv_bf16,
                                        const int32_t* table, int table_ld, float* o, int o_ld,
                                        int nsplit, void* stream) {
  using namespace s2;
  if (!qkv || !pos || !kv || !table || !o || !q_gain || !k_gain || !rope_cos || !rope_sin)
    return S2_EINVAL;
  if (B < 1 || m < 1 || m > 2 || nsplit < 1 || Hkv < 1 || H % Hkv) return S2_EINVAL;
  // partials, then the tickets on a 256-byte boundary
  const size_t part_bytes = attn_decode_scratch_floats(B, m, H, hd, nsplit) * 4;
  const size_t tick_off = (part_bytes + 255) / 256 * 256;
  const size_t tick_bytes = (size_t)B * Hkv * 4;
  if (tick_off + tick_bytes > S2_NOALLOC_SCRATCH_BYTES) return S2_EINVAL;
  unsigned char* scratch = nullptr;
  int s = scratch_for_current_device(&scratch);
  if (s) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the tickets must start at zero
  if (cudaMemsetAsync(scratch + tick_off, 0, tick_bytes, st) != cudaSuccess) return S2_ECUDA;
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
  a.part = reinterpret_cast<float*>(scratch);
  a.tickets = reinterpret_cast<unsigned*>(scratch + tick_off);
  cudaError_t e = launch_attn_decode(a, st, false);
  if (e == cudaErrorInvalidValue) {
    cudaGetLastError();
    return S2_EINVAL;
  }
  return e == cudaSuccess ? S2_OK : S2_ECUDA;
}
