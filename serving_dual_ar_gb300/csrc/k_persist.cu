// Persistent decode kernel (S2_FLAG_PERSIST): whole Dual-AR decode frames in
// one cooperative launch.
//
// At batch 1 a frame is ~380 dependent operations (per Slow AR layer: QKV
// GEMV, attention, O GEMV, gate/up GEMV, down GEMV; the semantic head; nine
// Fast AR passes of four layers and a head), most of them a 20-100 MB weight
// stream.  Here one CTA of 16 warps per SM stays resident for all frames and
// walks the recorded operation list:
//   * a GEMV arrives at the grid barrier, issues the first three segments of
//     its weight range into its shared-memory ring (~192 KB per SM in
//     flight), and only then waits for the operation that produces its input,
//     so the stream does not stop at an operation boundary;
//   * attention runs up to four 128-thread units side by side per CTA, each
//     on its own named barrier and shared-memory area;
//   * the operation descriptors are double-buffered in shared memory, the
//     next one fetched with cp.async while the current one runs.
// Every operation is the same device code, with the same arguments and the
// same split of the work over CTAs and warps, as the stand-alone kernel the
// per-frame CUDA graph launches, so both paths give bit-identical results.
// Activations are read through the coherent path (no read-only cache): the
// barrier's release/acquire pair makes the previous operation's writes
// visible.
// Measured on the S2 batch-1 frame it is slower than the CUDA-graph path
// (7.4 against 4.65 ms per frame): the grid barriers, waiting for the slowest
// of 152 CTAs, cost more than graph launches with programmatic dependent
// launch, and the attention units run slower than the stand-alone kernel.
// It stays as an option and as a second, independent execution of the frame.
#include "gemv_body.cuh"
#include "attn_body.cuh"
#include "embed_body.cuh"


namespace s2 {

thread_local OpRecorder* g_recorder = nullptr;

namespace {

using Attn = AttnSmem<128, 4>;

S2_DEV unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
S2_DEV unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr unsigned long long kBarrierTimeoutNs = 2000000000ull;  // 2 s
constexpr unsigned kBarrierMaxPolls = 1u << 26;

// Per-CTA barrier state (shared memory).
struct PersistState {
  unsigned target;  // arrivals the next barrier waits for (thread 0)
  int ok;           // result of the last barrier (CTA-uniform)
  unsigned long long t_pass;  // when thread 0 passed the last barrier (trace)
};

// Grid barrier, in two halves.  grid_arrive: once this CTA's work of the
// previous operation is done, thread 0 adds one arrival (release).  The CTA
// then issues the loads of the next operation that depend on nothing (its
// weight stream), and grid_wait polls (acquire) until the counter reaches this
// barrier's target (targets grow by the grid size per barrier; the counter
// starts at zero).  Arriving before those loads keeps them from delaying the
// arrival.  Bounded: after 2 s, 2^26 polls, or once another CTA has given up
// (*abort set), st->ok turns 0 and a timeout is recorded in *err (2).
S2_DEV void grid_arrive(unsigned* bar, PersistState* st, int* abort_flag, bool skip) {
  __syncthreads();
  if (threadIdx.x == 0) {
    st->target += gridDim.x;
    if (!skip && !*reinterpret_cast<volatile int*>(abort_flag))
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(bar) : "memory");
  }
}
S2_DEV void grid_wait(unsigned* bar, PersistState* st, int* abort_flag, int* err,
                      unsigned long long budget_ns) {
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned long long t0 = global_ns();
    for (unsigned it = 0; ld_acquire(bar) < st->target; ++it) {
      if ((it & 255u) == 255u) {
        if (*reinterpret_cast<volatile int*>(abort_flag)) { ok = 0; break; }
        if (it > kBarrierMaxPolls || global_ns() - t0 > budget_ns) {
          atomicExch(abort_flag, 1);
          if (err) atomicExch(err, 2);
          ok = 0;
          break;
        }
      }
    }
    st->ok = ok;
    st->t_pass = global_ns();
  }
  __syncthreads();
}

// The sync hooks of an operation: the two barrier halves, except for the
// launch's first operation (nothing inside the launch precedes it).
// ``skip_arrival`` (fault injection only): this CTA does not arrive, so every
// CTA's wait at this barrier runs out after ``budget_ns``.
struct PersistSync {
  unsigned* bar;
  int* abort_flag;
  int* err;
  PersistState* st;
  bool skip;
  bool skip_arrival;
  unsigned long long budget_ns;
  S2_DEV void arrive() const {
    if (!skip) grid_arrive(bar, st, abort_flag, skip_arrival);
  }
  S2_DEV void wait() const {
    if (!skip) grid_wait(bar, st, abort_flag, err, budget_ns);
  }
};

// Dynamic shared memory: two descriptor slots, then the phases' work area.
// Each phase function addresses it through this symbol (not a pointer
// argument), so the compiler knows every access is a shared-memory one.
extern __shared__ __align__(128) uint8_t g_psmem[];
constexpr size_t kSlotBytes = (sizeof(PersistOp) + 127) / 128 * 128;
S2_DEV const PersistOp& slot_op(int slot) {
  return *reinterpret_cast<const PersistOp*>(g_psmem + slot * kSlotBytes);
}
S2_DEV uint8_t* work_area() { return g_psmem + 2 * kSlotBytes; }

// The phases.  ptxas allocates registers per function; where each phase is
// compiled (inlined into the kernel or called) decides where it spills, so
// the kernel comes in three arrangements V (kPersistVariant selects one):
//   0: GEMV inlined, attention and embedding called;
//   1: every phase called;
//   2: every phase inlined.
template <int MAXB>
S2_DEV void gemv_phase(int slot, PersistSync w) {
  const PersistOp& op = slot_op(slot);
  if ((int)blockIdx.x < op.grid)
    gemv_body<__nv_bfloat16, MAXB, true, kPersistVmax, false, persist_adepth(MAXB)>(
        op.g, op.L, blockIdx.x, op.grid, work_area(), w);
  else {
    w.arrive();
    w.wait();
  }
}

S2_DEV void attn_phase(int slot_i, PersistSync w) {
  const PersistOp& op = slot_op(slot_i);
  uint8_t* work = work_area();
  w.arrive();
  w.wait();
  const AttnDecodeArgs& a = op.at;
  const int units = a.B * a.Hkv * a.nsplit;
  const int tid = threadIdx.x, slot = tid >> 7;
  Attn& S = reinterpret_cast<Attn*>(work)[slot];
  auto none = [] {};
  for (int u = blockIdx.x + gridDim.x * slot; u < units; u += gridDim.x * kPersistAttnUnits) {
    const int b = u % a.B, g = (u / a.B) % a.Hkv, split = u / (a.B * a.Hkv);
    if (a.kv_bf16)
      attn_body<__nv_bfloat16, 128, 4, false>(a, b, g, split, tid & 127, 1 + slot, S, none);
    else
      attn_body<float, 128, 4, false>(a, b, g, split, tid & 127, 1 + slot, S, none);
  }
}

S2_DEV void embed_phase(int slot, PersistSync w) {
  const PersistOp& op = slot_op(slot);
  w.arrive();
  w.wait();
  // work items (row, 512 columns) over the CTAs
  const int nb = (op.e.d + kPersistThreads - 1) / kPersistThreads;
  for (int u = blockIdx.x; u < op.e.rows * nb; u += gridDim.x)
    embed_body<__nv_bfloat16>(op.e, u / nb, (u % nb) * kPersistThreads, op.e.d, threadIdx.x, [] {});
}

template <int MAXB>
__device__ __noinline__ void gemv_call(int slot, PersistSync w) { gemv_phase<MAXB>(slot, w); }
__device__ __noinline__ void attn_call(int slot, PersistSync w) { attn_phase(slot, w); }
__device__ __noinline__ void embed_call(int slot, PersistSync w) { embed_phase(slot, w); }

template <int MAXB, int V>
__global__ void __launch_bounds__(kPersistThreads, 1)
persist_decode_kernel(const PersistOp* __restrict__ ops, int n_ops, int n_frames, unsigned* bar,
                      int* abort_flag, int* err, unsigned long long* trace, int fault_op,
                      unsigned long long budget_ns) {
  uint8_t* smem = g_psmem;
  __shared__ PersistState st;
  const int tid = threadIdx.x;
  auto fetch = [&](int t) {  // descriptor of step t into slot t & 1
    const uint8_t* src = reinterpret_cast<const uint8_t*>(ops + t % n_ops);
    uint8_t* dst = smem + (t & 1) * kSlotBytes;
    for (int o = tid * 16; o < (int)sizeof(PersistOp); o += kPersistThreads * 16)
      cp_async16(dst + o, src + o);
    cp_async_commit();
  };
  if (tid == 0) {
    st.target = 0;
    st.ok = 1;
    st.t_pass = 0;
  }
  const int total = n_ops * n_frames;
  // trace (optional): CTA 0's clock around each operation of one frame
  const int trace_frame = n_frames > 1 ? 1 : 0;
  const bool tracer = trace && blockIdx.x == 0 && tid == 0;
  if (total > 0) fetch(0);
  for (int t = 0; t < total; ++t) {
    cp_async_wait_all();
    __syncthreads();
    if (!st.ok) break;
    const PersistOp& op = slot_op(t & 1);
    if (t + 1 < total) fetch(t + 1);
    const bool traced = tracer && t / n_ops == trace_frame;
    if (traced) trace[(t % n_ops) * 3] = global_ns();
    const PersistSync w{bar, abort_flag, err, &st, t == 0, t == fault_op && blockIdx.x == 0, budget_ns};
    switch (op.kind) {
      case PK_GEMV:
        if (V == 1) gemv_call<MAXB>(t & 1, w);
        else gemv_phase<MAXB>(t & 1, w);
        break;
      case PK_ATTN:
        if (V == 2) attn_phase(t & 1, w);
        else attn_call(t & 1, w);
        break;
      case PK_EMBED:
        if (V == 2) embed_phase(t & 1, w);
        else embed_call(t & 1, w);
        break;
      default: break;
    }
    if (traced) {
      trace[(t % n_ops) * 3 + 1] = st.t_pass;
      trace[(t % n_ops) * 3 + 2] = global_ns();
    }
  }
  cp_async_wait_all();
}

}  // namespace

using PersistKernel = void (*)(const PersistOp*, int, int, unsigned*, int*, int*, unsigned long long*, int,
                               unsigned long long);
template <int V>
static PersistKernel kernel_v(int maxb) {
  switch (maxb) {
    case 1: return persist_decode_kernel<1, V>;
    case 2: return persist_decode_kernel<2, V>;
    case 4: return persist_decode_kernel<4, V>;
    case 8: return persist_decode_kernel<8, V>;
    default: return nullptr;
  }
}
// Arrangement 0 (GEMV inlined, attention and embedding called): the
// fastest of the three when measured.
constexpr int kPersistVariant = 0;
static PersistKernel persist_kernel_for(int maxb) {
  switch (kPersistVariant) {
    case 1: return kernel_v<1>(maxb);
    case 2: return kernel_v<2>(maxb);
    default: return kernel_v<0>(maxb);
  }
}

size_t persist_smem_bytes(const std::vector<PersistOp>& ops) {
  size_t need = 0;
  for (const PersistOp& op : ops) {
    if (op.kind == PK_GEMV) need = std::max(need, (size_t)op.L.smem);
    if (op.kind == PK_ATTN) need = std::max(need, kPersistAttnUnits * sizeof(Attn));
  }
  return 2 * kSlotBytes + need;
}

int persist_grid(int num_sms, int maxb, size_t smem) {
  PersistKernel k = persist_kernel_for(maxb);
  if (!k || smem > 227 * 1024) return 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kPersistThreads, smem) != cudaSuccess ||
      per_sm < 1)
    return 0;
  return num_sms;
}

cudaError_t launch_persist(const PersistOp* ops, int n_ops, int n_frames, int maxb, unsigned* bar,
                           int* abort_flag, int* err, int grid, size_t smem, cudaStream_t st,
                           unsigned long long* trace, int fault_op, unsigned long long budget_ns) {
  PersistKernel k = persist_kernel_for(maxb);
  if (!k || !ops || n_ops < 1 || n_frames < 1 || !bar || !abort_flag || grid < 1)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPersistThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the barrier cannot deadlock
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return s2_launch(&cfg, k, ops, n_ops, n_frames, bar, abort_flag, err, trace, fault_op,
                   budget_ns ? budget_ns : kBarrierTimeoutNs);
}

}  // namespace s2
