// Thin inline-PTX wrappers for the sm_103a features the attention kernels use:
// mbarriers, TMA tensor loads and bulk reductions, and the 5th-generation
// tensor core (tcgen05: TMEM allocation, MMA, commit, TMEM loads/stores).
//
// Every wait here is bounded: past a time limit it records FA_ERR_TIMEOUT in
// the library's device status word, raises the CTA's abort flag and returns
// false, so a lost arrival ends the kernel with an error instead of a hang.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

// ----------------------------------------------------------------------------
// Status word of the kernels in this translation unit (0 = ok). Static
// storage, one per translation unit; the host reads it in check mode.
// ----------------------------------------------------------------------------
static __device__ int g_fa_status;

// Test hooks of this translation unit, set from the host only when the
// FA_TEST_* environment variables ask for them: the bound on every wait, and
// a switch that makes the TMA producer issue no loads (so the waits run out).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
static __device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;
static __device__ int g_test_drop_loads = 0;

constexpr int kStatusTimeout = -4;  // == FA_ERR_TIMEOUT

// Host side, for this translation unit's copies of the above: set the test
// hooks (synchronises `stream`: the values are copied from the host stack),
// and read-and-clear the status word (-3 when the read itself fails).
static inline cudaError_t set_test_hooks_here(unsigned long long wait_limit_ns, int drop_loads,
                                              cudaStream_t stream) {
  cudaError_t e = cudaMemcpyToSymbolAsync(g_wait_limit_ns, &wait_limit_ns, sizeof(wait_limit_ns), 0,
                                          cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_test_drop_loads, &drop_loads, sizeof(drop_loads), 0, cudaMemcpyHostToDevice,
                                stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

static inline int take_status_here() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(int)) != cudaSuccess) return -3;
  cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(int));
  return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start before the previous kernel on its stream has
// finished; griddep_wait() blocks until that kernel has completed and its
// memory operations are visible (nothing before it may read what that kernel
// writes). griddep_launch_dependents() lets the next such kernel launch once
// every CTA of this grid has called it or exited (it does not make this
// grid's later writes visible early: the dependent still waits).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for completion of the phase with the given parity. Returns false on
// timeout or when the CTA has already aborted (``abort_flag`` != 0).
// The bound (g_wait_limit_ns, 2 s by default) is far above the longest
// legitimate wait of these kernels (a full kernel runs for milliseconds).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (*(volatile int*)&g_fa_status != 0) {  // another CTA already gave up
        *abort_flag = 1;
        return false;
      }
      const uint64_t now = global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > *(volatile unsigned long long*)&g_wait_limit_ns) {
        atomicExch(&g_fa_status, kStatusTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Wait for an operation this CTA issued (a copy, an MMA) to complete, also
// after an abort: a CTA must not exit or free TMEM with work in flight. Bounded
// by the same time limit, read every 256 polls like mbar_wait (reading the
// timer on every poll made the spinning thread slow its CTA's other warps).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      const uint64_t now = global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > *(volatile unsigned long long*)&g_wait_limit_ns) {
        atomicExch(&g_fa_status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Barrier among ``count`` threads (a multiple of 32) of the CTA, id 1..15.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier among ``count`` threads that also returns the AND of ``pred`` over
// them, so a group can take a uniform decision (e.g. after a bounded wait).
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// ----------------------------------------------------------------------------
// Proxy fences
// ----------------------------------------------------------------------------
// Generic-proxy shared-memory writes -> visible to the async proxy (TMA, MMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy global accesses with its async-proxy
// (bulk copy / bulk reduction) global accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ----------------------------------------------------------------------------
// Counters in global memory that order work between CTAs
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until *counter == want (acquire), bounded like mbar_wait. The caller
// only ever waits for counters that CTAs already running will advance, so the
// bound is reached only if something is broken.
__device__ __forceinline__ bool counter_wait_eq(const uint32_t* counter, uint32_t want, volatile int* abort_flag) {
  if (ld_acquire_gpu(counter) == want) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(counter) == want) return true;
    if (*abort_flag) return false;
    if (*(volatile int*)&g_fa_status != 0) {
      *abort_flag = 1;
      return false;
    }
    if (global_timer_ns() - t0 > *(volatile unsigned long long*)&g_wait_limit_ns) {
      atomicExch(&g_fa_status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// ----------------------------------------------------------------------------
// TMA (tensor map driven bulk copies)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 3-D tiled load global -> shared, completion signalled on ``bar`` (tx bytes).
// x (innermost coordinate) must be a multiple of 8 for 16-bit data.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Contiguous global -> shared bulk copy (no tensor map), completion on ``bar``.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Contiguous shared -> global fp32 add-reduction (bulk, async). Both addresses
// 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory
// ----------------------------------------------------------------------------
// Warp-wide. Writes the TMEM base address of ``ncols`` columns to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// MMA issue from a whole warp: every lane of the issuing warp runs the
// issuing loop (its waits made warp-uniform with __all_sync), so the operand
// descriptors and addresses are warp-uniform values, and one lane chosen by
// elect.sync issues each instruction. Measured on the forward against one
// lane in a divergent branch issuing: 5652 against 6298 us on N = 65536,
// 205.7 against 220.3 on the padded N = 4096 batch. All 32 lanes must reach
// these together.

// Arrive once on ``bar`` when all tcgen05 ops issued so far by the issuing
// lane finish.
__device__ __forceinline__ void tc_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc] (bf16 or f16 operands, fp32 D).
__device__ __forceinline__ void tc_mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc].
__device__ __forceinline__ void tc_mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same two products with 8-bit operands (kind::f8f6f4; both E4M3 here):
// one instruction covers K = 32 elements (32 bytes of a row).
__device__ __forceinline__ void tc_mma_ss_f8_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_mma_ts_f8_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::f16 with fp32 accumulate.
// Bits: [4,6) D format (1 = f32), [7,10) A format (0 = f16, 1 = bf16), [10,13)
// B format, 15 A major (1 = MN), 16 B major (1 = MN), [17,23) N>>3, [24,29) M>>4.
// A and B always share one input type.
__host__ __device__ constexpr uint32_t idesc_f32acc(int M, int N, bool a_mn_major, bool b_mn_major, bool bf16) {
  return (1u << 4) | (static_cast<uint32_t>(bf16) << 7) | (static_cast<uint32_t>(bf16) << 10) |
         (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return idesc_f32acc(M, N, a_mn_major, b_mn_major, true);
}
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return idesc_f32acc(M, N, a_mn_major, b_mn_major, false);
}
// kind::f8f6f4 uses the same layout; format code 0 in the A and B fields is
// E4M3. Both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return idesc_f32acc(M, N, false, false, false);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
// Bits: [0,14) start>>4, [16,30) leading byte offset>>4, [32,46) stride byte
// offset>>4, [46,48) = 1 (descriptor version), [61,64) layout (2 = 128B swizzle).
//  K-major operand: rows of 128 B (64 bf16 along K), 8-row atoms of 1024 B;
//    SBO = 1024 (next 8 rows), LBO unused. Advancing K by 16 elements inside
//    the 128 B row adds 32 B to the start address.
//  MN-major operand: 128 B runs along M/N, consecutive K at 128 B stride;
//    SBO = 1024 (next 8 K), LBO = distance between 64-element M/N chunks.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// The descriptor of the same operand layout starting ``bytes`` further on (a
// multiple of 16): only the start-address field moves, and it cannot carry
// into the next field because shared-memory addresses stay below 256 KB.
// Building each operand's descriptor once and advancing it per k-step keeps
// the issuing thread's work per MMA to a 64-bit add. Measured on GB300 with a
// lone issuing thread: about 61 clocks per tcgen05.mma issue this way against
// about 110 with the full encoding in the loop, while a 128x128x16 bf16
// product occupies the tensor pipe for 64 clocks.
__device__ __forceinline__ uint64_t sdesc_advance(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// ---- TMEM <-> registers (one warp = 32 lanes; 32x32b: thread i <-> lane i) ----
#define FA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                 "=r"(r[i + 6]), "=r"(r[i + 7])
#define FA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                 "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive 32-bit columns starting at taddr, for this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      FA_W8(0), FA_W8(8)
      : "memory");
}
// 64 consecutive 32-bit columns as fp32, plus their maximum (one value per
// lane: the row maximum of the columns loaded; tcgen05.ld.red, sm_103a).
__device__ __forceinline__ void tmem_ld64_max(uint32_t taddr, uint32_t (&r)[64], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x64.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
      "%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,"
      "%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, %64, [%65];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24), FA_R8(32), FA_R8(40), FA_R8(48), FA_R8(56), "=f"(mx)
      : "r"(taddr)
      : "memory");
}

#undef FA_R8
#undef FA_W8

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------
// Arithmetic helpers
// ----------------------------------------------------------------------------
// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> packed bf16x2, round to nearest even; ``lo`` in bits [0,16).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- Packed fp32 pairs (one 64-bit register, ``lo`` in the low half): the
// f32x2 add/sub/mul/fma forms do two fp32 operations per instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Two fp32 -> packed f16x2, round to nearest even; ``lo`` in bits [0,16).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four floats -> four E4M3 codes (round to nearest even, saturating at
// +-448), element k in byte k.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Packed bf16x2 -> packed f16x2 (exact for |x| in [2^-14, 65504]; smaller
// magnitudes round to the f16 subnormal grid, error < 2^-25).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  return pack_f16x2(lo, hi);
}

}  // namespace fa
