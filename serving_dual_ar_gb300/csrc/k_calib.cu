// HBM read-bandwidth calibration kernels (s2op_stream_read).
//
// The decode frame is a read-only weight stream ("s2pro-native", Where it
// stands: bandwidth, not arithmetic), so the ceiling that matters is what a
// plain read stream reaches on this part, at the sizes the frame reads: one
// projection is 21-100 MB, one frame ~14.7 GB in ~370 dependent pieces.
// Two ways of reading a list of buffers ("operations"), each a pure stream
// whose loaded values only feed a checksum:
//   mode 0 (ldg):  one launch per operation; every thread issues eight
//       16-byte non-coherent loads (L1 no-allocate) before using any;
//   mode 1 (ring): one persistent launch, one CTA per SM.  A producer thread
//       walks all operations in order and streams the CTA's contiguous share
//       of each through a ring of shared-memory chunks with bulk copies (TMA
//       engine, completion on an mbarrier per chunk); consumer warps read each
//       chunk and release it.  The producer never waits for anything but a
//       free chunk, so the stream runs across operation boundaries.  With
//       ``barrier`` set the consumers pass a grid barrier before each
//       operation, as a dependent chain of operations must; the producer does
//       not, so the next operation's bytes are already arriving while the
//       barrier resolves.
// Every wait is bounded; after a failed wait the CTA stops issuing, waits
// (bounded) for the copies it has issued, and sets the error word.
#include "s2.h"
#include "s2_ops.h"
#include "s2_kernels.h"
#include "s2_common.cuh"

namespace s2 {

namespace {

constexpr int kCalConsumerWarps = 8;
constexpr int kCalThreads = 32 * (kCalConsumerWarps + 1);
constexpr int kCalMaxStages = 32;
constexpr uint32_t kCalWaitLimit = 4000000u;

struct CalOp {
  const uint8_t* base;
  unsigned long long bytes;
};

// The CTA's contiguous share [lo, hi) of an operation, in 16-byte units.
S2_DEV void cal_slice(unsigned long long bytes, int c, int n, unsigned long long& lo,
                      unsigned long long& hi) {
  const unsigned long long u = bytes / 16;
  lo = u * (unsigned long long)c / (unsigned long long)n * 16ull;
  hi = u * (unsigned long long)(c + 1) / (unsigned long long)n * 16ull;
}

S2_DEV uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

S2_DEV float sum16(const uint4& u) {
  return bf16lo(u.x) + bf16hi(u.x) + bf16lo(u.y) + bf16hi(u.y) + bf16lo(u.z) + bf16hi(u.z) +
         bf16lo(u.w) + bf16hi(u.w);
}

__global__ void __launch_bounds__(256)
stream_ldg_kernel(const uint8_t* base, unsigned long long bytes, float* sink) {
  const uint4* p = reinterpret_cast<const uint4*>(base);
  const unsigned long long n = bytes / 16;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  float acc = 0.f;
  for (; i + 7 * stride < n; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = ld_stream16(p + i + j * stride);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc += sum16(v[j]);
  }
  for (; i < n; i += stride) acc += sum16(ld_stream16(p + i));
  if (acc == 1234.5f) sink[0] = acc;  // keeps the loads; practically never true
}

S2_DEV unsigned cal_ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(kCalThreads, 1)
stream_ring_kernel(const CalOp* __restrict__ ops, int n_ops, int reps, int chunk, int stages,
                   int barrier, unsigned* bar, int* err, float* sink) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kCalMaxStages], empty[kCalMaxStages], op_done, go;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCalConsumerWarps);
    }
    mbar_init(&op_done, kCalConsumerWarps);
    mbar_init(&go, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int total = n_ops * reps;
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      long long k = 0;  // chunks issued
      bool ok = true;
      for (int t = 0; t < total && ok; ++t) {
        const CalOp op = ops[t % n_ops];
        unsigned long long lo, hi;
        cal_slice(op.bytes, blockIdx.x, gridDim.x, lo, hi);
        for (unsigned long long off = lo; off < hi; off += (unsigned)chunk, ++k) {
          const int s = (int)(k % stages);
          if (k >= stages && !mbar_wait(&empty[s], (uint32_t)((k / stages - 1) & 1), err, kCalWaitLimit)) {
            ok = false;
            break;
          }
          if (*reinterpret_cast<volatile int*>(&s_abort)) { ok = false; break; }
          const unsigned long long left = hi - off;
          const uint32_t nb = left < (unsigned long long)chunk ? (uint32_t)left : (uint32_t)chunk;
          mbar_arrive_expect_tx(&full[s], nb);
          bulk_g2s_evict_first(smem + (size_t)s * chunk, op.base + off, nb, &full[s], pol);
        }
      }
      if (!ok) s_abort = 1;
      // every copy issued must have landed before this CTA may exit
      for (long long j = k > stages ? k - stages : 0; j < k; ++j)
        mbar_wait(&full[j % stages], (uint32_t)((j / stages) & 1), nullptr, kCalWaitLimit);
    }
  } else {
    const int cw = warp - 1;
    long long k = 0;
    float acc = 0.f;
    unsigned target = 0;
    bool ok = true;
    for (int t = 0; t < total && ok; ++t) {
      if (barrier && t > 0) {
        // every consumer warp done with operation t-1 (op_done), then one
        // thread takes the grid barrier and releases the others (go); all
        // waits bounded
        const uint32_t ph = (uint32_t)((t - 1) & 1);
        __syncwarp();
        if (lane == 0) mbar_arrive(&op_done);
        if (cw == 0 && lane == 0) {
          bool good = mbar_wait(&op_done, ph, err, kCalWaitLimit);
          if (good) {
            target += gridDim.x;
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(bar) : "memory");
            uint32_t it = 0;
            while (cal_ld_acquire(bar) < target) {
              if (++it > (1u << 26) || *reinterpret_cast<volatile int*>(err)) {
                atomicExch(err, 2);
                good = false;
                break;
              }
            }
          }
          if (!good) *reinterpret_cast<volatile int*>(&s_abort) = 1;
          mbar_arrive(&go);
        }
        if (!mbar_wait(&go, ph, err, kCalWaitLimit) || *reinterpret_cast<volatile int*>(&s_abort)) break;
      }
      const CalOp op = ops[t % n_ops];
      unsigned long long lo, hi;
      cal_slice(op.bytes, blockIdx.x, gridDim.x, lo, hi);
      for (unsigned long long off = lo; off < hi; off += (unsigned)chunk, ++k) {
        const int s = (int)(k % stages);
        if (!mbar_wait(&full[s], (uint32_t)((k / stages) & 1), err, kCalWaitLimit)) {
          s_abort = 1;
          ok = false;
          break;
        }
        const unsigned long long left = hi - off;
        const int nv = (int)((left < (unsigned long long)chunk ? left : (unsigned long long)chunk) / 16);
        const uint4* p = reinterpret_cast<const uint4*>(smem + (size_t)s * chunk);
        for (int v = cw * 32 + lane; v < nv; v += kCalConsumerWarps * 32) acc += sum16(p[v]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
    if (acc == 1234.5f) sink[0] = acc;
  }
}

}  // namespace

}  // namespace s2

using namespace s2;

// Scratch layout: [0] barrier counter, [1] error word, [2] sink, ops from byte 256.
extern "C" size_t s2op_stream_read_scratch_bytes(int n_ops) {
  return 256 + (size_t)(n_ops > 0 ? n_ops : 1) * sizeof(CalOp);
}

extern "C" int s2op_stream_read(const void* const* bufs, const unsigned long long* bytes, int n_ops,
                                int reps, int mode, int chunk_bytes, int stages, int barrier,
                                void* scratch, int* err_out, void* stream) {
  if (!bufs || !bytes || n_ops < 1 || reps < 1 || !scratch) return S2_EINVAL;
  for (int i = 0; i < n_ops; ++i)
    if (!bufs[i] || (reinterpret_cast<uintptr_t>(bufs[i]) & 15) || bytes[i] % 16) return S2_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return S2_ECUDA;
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  unsigned* bar = reinterpret_cast<unsigned*>(sc);
  int* err = reinterpret_cast<int*>(sc + 4);
  float* sink = reinterpret_cast<float*>(sc + 8);
  if (mode == 0) {
    const int grid = sms * 8;
    for (int r = 0; r < reps; ++r)
      for (int i = 0; i < n_ops; ++i) {
        stream_ldg_kernel<<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(bufs[i]), bytes[i], sink);
        ++g_launch_count;
      }
    return cudaGetLastError() == cudaSuccess ? S2_OK : S2_ECUDA;
  }
  if (mode != 1) return S2_EINVAL;
  if (chunk_bytes < 1024 || chunk_bytes % 16 || stages < 2 || stages > kCalMaxStages ||
      (size_t)chunk_bytes * stages > 200 * 1024)
    return S2_EINVAL;
  std::vector<CalOp> host(n_ops);
  for (int i = 0; i < n_ops; ++i) host[i] = {static_cast<const uint8_t*>(bufs[i]), bytes[i]};
  CalOp* dops = reinterpret_cast<CalOp*>(sc + 256);
  if (cudaMemsetAsync(sc, 0, 256, st) != cudaSuccess ||
      cudaMemcpyAsync(dops, host.data(), n_ops * sizeof(CalOp), cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return S2_ECUDA;
  const int smem = chunk_bytes * stages;
  if (cudaFuncSetAttribute(stream_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return S2_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kCalThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the consumers' grid barrier needs co-residency
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (s2_launch(&cfg, stream_ring_kernel, (const CalOp*)dops, n_ops, reps, chunk_bytes, stages,
                barrier, bar, err, sink) != cudaSuccess)
    return S2_ECUDA;
  if (err_out) {
    if (cudaMemcpyAsync(err_out, err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return S2_ECUDA;
  }
  return S2_OK;
}
