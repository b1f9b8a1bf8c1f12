// Staging helpers of the tensor-core attention kernels: fp32 values as two
// bf16 planes (hi = bf16(x), lo = bf16(x - hi): ~16 mantissa bits between
// them) packed into 16-byte units of the 128-byte swizzled K-major layout, and
// 8-element loads of fp32 or bf16 KV-cache rows.
#pragma once

#include "s2_common.cuh"

namespace s2 {

// 8 floats as two 16-byte units of bf16: hi = bf16(x), lo = bf16(x - hi),
// both rounded to nearest even; each pair converted by one packed convert
// (element 2e in the low 16 bits of word e)
S2_DEV void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    const float2 hf = __bfloat1622float2(h2);
    const __nv_bfloat162 l2 = __floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
    h[e] = *reinterpret_cast<const uint32_t*>(&h2);
    l[e] = *reinterpret_cast<const uint32_t*>(&l2);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
S2_DEV void st_shared16(uint8_t* base, uint32_t off, const uint4& v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}
S2_DEV void st_shared_bf16(uint8_t* base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
}

template <typename KT>
S2_DEV void load8kv(const KT* p, float (&v)[8]);
template <>
S2_DEV void load8kv<float>(const float* p, float (&v)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(p + 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
S2_DEV void load8kv<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldcg(reinterpret_cast<const uint4*>(p));
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}

}  // namespace s2
