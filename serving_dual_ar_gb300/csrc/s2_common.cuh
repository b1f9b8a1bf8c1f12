// Shared device helpers for the sm_103a kernels: bf16 conversion, warp
// reductions, mbarrier / bulk-copy (TMA) wrappers and programmatic dependent
// launch (PDL) controls, all as inline PTX.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "s2_kernels.h"

#define S2_DEV __device__ __forceinline__

namespace s2 {

constexpr int kWarp = 32;

// ---------------------------------------------------------------- numerics

S2_DEV float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
S2_DEV float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

template <typename T> struct Vec8;   // 8 consecutive weights as floats

// Load 8 values starting at p (16-byte aligned for bf16, 32 for float).
S2_DEV void load8(const __nv_bfloat16* p, float (&v)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}
S2_DEV void load8(const float* p, float (&v)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// Read-only global path for activations (kept in L1).
S2_DEV void ldg8(const float* p, float (&v)[8]) {
  float4 a = __ldg(reinterpret_cast<const float4*>(p));
  float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

S2_DEV float to_f(float x) { return x; }
S2_DEV float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> S2_DEV T from_f(float x);
template <> S2_DEV float from_f<float>(float x) { return x; }
template <> S2_DEV __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Store v as bf16 "hi" and, when lo is given, the bf16 of the remainder
// v - hi: hi + lo carries ~16 mantissa bits, so a tensor-core product taken
// as A*hi + A*lo is nearly as exact as with fp32 operands.
S2_DEV void st_bf16_split(__nv_bfloat16* hi, __nv_bfloat16* lo, size_t i, float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  hi[i] = h;
  if (lo) lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
}

S2_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
S2_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// (value, index) arg-max with ties to the lowest index.
S2_DEV bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}
S2_DEV void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// ---------------------------------------------------------------- sampling noise

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11): counter c, key (k0, k1).
S2_DEV uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Gumbel noise -ln(-ln U) for code index i of codebook k at position pos of
// sequence seq: U from word i % 4 of Philox(counter (i/4, k, pos, seq), seed),
// as an odd multiple of 2^-24 in (0, 1).
S2_DEV float gumbel_noise(unsigned long long seed, int seq, int pos, int codebook, int i) {
  const uint4 r = philox4x32_10(make_uint4((uint32_t)(i >> 2), (uint32_t)codebook, (uint32_t)pos,
                                           (uint32_t)seq),
                                (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t w = (i & 3) == 0 ? r.x : (i & 3) == 1 ? r.y : (i & 3) == 2 ? r.z : r.w;
  const float u = (float)(((w >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
  return -logf(-logf(u));
}

// Frame timeline stamp: thread 0 of CTA ``cta`` writes the global timer into
// slot i of its four (no-op without a trace buffer).
S2_DEV void frame_stamp(unsigned long long* trace, int cta, int i) {
  if (trace && threadIdx.x == 0 && cta < kFrameTraceCtas) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    trace[cta * 4 + i] = t;
  }
}

// ---------------------------------------------------------------- PDL

// Wait until the grids this launch depends on have completed and their
// memory is visible (no-op when launched without a programmatic edge).
S2_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to start launching its CTAs.
S2_DEV void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Synchronisation hooks of a kernel body: arrive() as the body starts,
// before it issues loads that do not depend on earlier work; wait() before
// its first read of anything earlier work writes.  A stand-alone kernel
// waits for the previous grid (PDL); the persistent decode kernel splits its
// grid barrier into the two halves.
struct PdlSync {
  S2_DEV void arrive() const {}
  S2_DEV void wait() const {
    pdl_launch_next();
    pdl_wait();
  }
};

// ---------------------------------------------------------------- mbarrier

S2_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
S2_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
S2_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
S2_DEV void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
S2_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
               :: "r"(smem_u32(bar)) : "memory");
}
S2_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
S2_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait: spins at most ``limit`` polls (each try_wait itself blocks
// for a hardware-defined time slice).  On expiry sets *err (if given) and
// returns false; the caller then skips the dependent work and exits, so a
// lost completion can never hang the GPU.
S2_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, uint32_t limit = 2000000u) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  if (err) atomicExch(err, 1);
  return false;
}

// ---------------------------------------------------------------- bulk copy

// 1-D bulk copy global -> shared (TMA engine), completing on ``bar`` with a
// transaction count of ``bytes``.  dst, src 16-byte aligned; bytes % 16 == 0.
S2_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// Same, with an L2 eviction-first hint (streamed weights are read once per pass).
S2_DEV void bulk_g2s_evict_first(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}
// Per-thread 16-byte async copies global -> shared (bypassing L1); they
// complete in commit groups (cp_async_commit / cp_async_wait_group).  dst and
// src 16-byte aligned.  The _hint form carries an L2 cache-policy operand.
S2_DEV void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
S2_DEV void cp_async16_hint(void* dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;"
               :: "r"(smem_u32(dst)), "l"(src), "l"(policy) : "memory");
}
S2_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's most recent groups are pending.
template <int N>
S2_DEV void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }
S2_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

S2_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

}  // namespace s2
