// common.cuh -- device helpers shared by the i8kv kernels (sm_103a).
//
// Inline PTX for the pieces the kernels are built from: mbarrier pipelines fed
// by bulk (TMA) copies, ldmatrix, the INT8 and BF16 warp-level MMAs, and the
// bounded waits every spin loop in this library goes through.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace i8kv {

// Device error word: 0 = fine; the first failure wins.
//   1 = a pipeline wait ran past its time limit
//   2 = a block-table entry, slot or length out of range (the access was skipped)
// The library is built without relocatable device code, so every translation
// unit has its own word; each one exports a host accessor (below) and
// i8kv_device_error() reads them all.
static __device__ int g_device_error = 0;

// Defines `cudaError_t fn(int* value)`: reads this unit's error word into
// *value and clears it.
#define I8KV_DEFINE_ERROR_ACCESSOR(fn)                                              \
  cudaError_t fn(int* value) {                                                      \
    int zero = 0;                                                                   \
    cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));       \
    if (e != cudaSuccess) return e;                                                 \
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));                  \
  }

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_device_error, 0, code); }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A wait gives up after this long (the kernels move at most a few hundred KB
// per wait, so a healthy wait ends within microseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity (never suspends).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same test, but a thread whose phase is not complete yet may be suspended (it
// issues nothing) until the phase completes or suspend_ns have passed.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// (and records error 1) if it did not complete within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(1);
      return false;
    }
  }
  return true;
}

// Bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 policy that lets the streamed lines go first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// 4-byte asynchronous copy global -> shared (cp.async); src_bytes = 0 writes
// zeros without reading src.  Both addresses 4-byte aligned.
__device__ __forceinline__ void cp_async_4(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

// The mbarrier's current phase also waits for every cp.async this thread has
// issued so far (the pending count is raised by one now and lowered when the
// copies land, so the barrier's expected arrival count is unchanged).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream is still
// running; griddep_wait() blocks until that kernel has finished and its memory
// is visible (a no-op for an ordinary launch).  griddep_launch_dependents()
// lets the next kernel on the stream start its own launch early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier among `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ----------------------------------------------------------------- fragments
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row_addr)));
}

// D = A(16x32 s8, row) * B(32x8 s8, col) + C, int32 accumulate.
__device__ __forceinline__ void mma_s8_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with unsigned 8-bit B (codes 0..255): s8 x u8 -> exact s32.
__device__ __forceinline__ void mma_s8u8_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.u8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ----------------------------------------------------------------- exact INT8 on the f16 tensor path
// Four int8 codes (little-endian) -> f16x2 {c0, c1} and {c2, c3}, exactly:
// byte b becomes the f16 1024 + (b ^ 0x80) = 1152 + c, then 1152 is subtracted.
__device__ __forceinline__ void s8x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = x ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x5140);
  hi = __byte_perm(u, 0x64646464u, 0x7362);
  const uint32_t bias = 0x64806480u;  // f16x2 (1152, 1152)
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(bias));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(bias));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One exact INT8 m16n8k32 step on the f16 tensor path.  The s8 A fragment
// (rows g / g+8 x k 4t..4t+3 and 16+4t..16+4t+3, as ldmatrix delivers it) is
// split into two k16 MMAs over k {0..15} and {16..31}; inside each the f16
// fragment order pairs logical k (2t, 2t+1 | 2t+8, 2t+9) with physical k
// (4t, 4t+1 | 4t+2, 4t+3).  b[0..3] is B in the matching f16 form (b[0], b[1]
// for k 0..15, b[2], b[3] for k 16..31).  The same permutation on both
// operands leaves the sum unchanged.
__device__ __forceinline__ void mma_s8a_f16b(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[4]) {
  uint32_t a0l, a0h, a1l, a1h, a2l, a2h, a3l, a3h;
  s8x4_to_f16(a[0], a0l, a0h);
  s8x4_to_f16(a[1], a1l, a1h);
  s8x4_to_f16(a[2], a2l, a2h);
  s8x4_to_f16(a[3], a3l, a3h);
  mma_f16_16816(d, a0l, a1l, a0h, a1h, b[0], b[1]);
  mma_f16_16816(d, a2l, a3l, a2h, a3h, b[2], b[3]);
}

// Two small integers (|x| <= 2048) as an exact f16x2 {lo, hi}.
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// s8 B fragment (k 4t..4t+3 and 16+4t..16+4t+3 of column g) -> the f16 form above.
__device__ __forceinline__ void s8b_to_f16(uint32_t x0, uint32_t x1, uint32_t (&b)[4]) {
  s8x4_to_f16(x0, b[0], b[1]);
  s8x4_to_f16(x1, b[2], b[3]);
}


// ----------------------------------------------------------------- 5th-generation tensor cores
// tcgen05: MMAs issued by one thread, operands in shared memory (described by
// 64-bit matrix descriptors), the fp32 accumulator in tensor memory (TMEM:
// 128 lanes x 512 columns of 32 bits per SM; lane = row of the M = 128 tile).

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// `swz` bytes (128 or 64), 16-byte chunks XOR-swizzled by the row within each
// 8-row group (SWIZZLE_128B / SWIZZLE_64B); 8-row groups are 8 * swz bytes
// apart.  The tile must start on an 8 * swz byte boundary; a K offset inside a
// row is added to `saddr` in bytes.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, int swz) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;                            // leading offset (unused by swizzled K-major)
  d |= (uint64_t)((8 * swz) >> 4) << 32;             // stride offset: one 8-row group
  d |= (uint64_t)1 << 46;                            // descriptor version
  d |= (uint64_t)(swz == 128 ? 2 : 4) << 61;         // SWIZZLE_128B = 2, SWIZZLE_64B = 4
  return d;
}

// Instruction descriptor, kind::f16: f16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The same with bf16 A and B (A and B types sit in bits 7-9 and 10-12).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return umma_idesc_f16(M, N) | (1u << 7) | (1u << 10);
}

// D[tmem] (+)= A * B^T, one K = 16 step (cta_group::1).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// The same with A in tensor memory: row m of A in TMEM lane m, two 16-bit
// elements per 32-bit column (the even one in the low half), so one K = 16
// step reads 8 columns starting at a_tmem.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// The mbarrier receives one arrival when every tcgen05 operation this thread
// issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Whole warp: allocate `cols` TMEM columns (a power of two >= 32); the base
// address is written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Whole warp: lane i reads columns [col, col + 16) (or 32) of TMEM lane
// (warp % 4) * 32 + i; `taddr` = base + (lane offset << 16) + col.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Whole warp: lane i writes columns [col, col + 32) of TMEM lane (warp % 4) * 32
// + i; taddr as for tmem_ld32.  tmem_wait_st() waits for this thread's stores.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Generic-proxy shared-memory writes made visible to the tensor cores.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Register budget of the executing warpgroup (all four of its warps execute
// it, with the same count); ptxas allocates the code that follows within it.
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ----------------------------------------------------------------- numerics
// x / s correctly rounded (the IEEE quotient) for one divisor s shared by many
// x, by Markstein's method: with y = RN(1/s), q = RN(x * y) and the exact
// residual r = x - s * q (one FMA), RN(q + r * y) is the correctly rounded
// quotient while nothing overflows or underflows (s >= 2^-100 here).
__device__ __forceinline__ float div_markstein(float x, float s, float y) {
  const float q = __fmul_rn(x, y);
  const float r = __fmaf_rn(-s, q, x);
  return __fmaf_rn(r, y, q);
}
constexpr float kTinyDivisor = 7.8886091e-31f;  // 2^-100

// x[i] / s, correctly rounded, for the N values of one row sharing the divisor
// s > 0, by Markstein's step.  Below 2^-100 both operands are first scaled by
// 2^100 (exact: x <= 127.5 s < 2^-93 cannot overflow, a subnormal keeps its
// bits, and the quotient does not change), which keeps every intermediate of
// the step in the normal range; so no IEEE division routine is inlined at any
// call site (those made the kernels' code far larger than their hot loops).
// The test on s is made once for the row, and the N quotients are independent
// chains of FMA-pipe operations.  y = RN(1/s) is passed in when the caller has
// it; for s below 2^-100 it is recomputed for the scaled divisor.
template <int N>
__device__ __forceinline__ void div_row(float (&x)[N], float s, float y) {
  if (s < kTinyDivisor) {
    const float s2 = __fmul_rn(s, 0x1p100f), y2 = __frcp_rn(s2);
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = div_markstein(__fmul_rn(x[i], 0x1p100f), s2, y2);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = div_markstein(x[i], s, y);
  }
}

// a / 127 correctly rounded below 2^-100 (the rare tiny-absmax case of div127),
// kept out of line so its division routine is compiled once per kernel.
static __device__ __noinline__ float div127_tiny(float a) { return __fdiv_rn(a, 127.0f); }

// 2^x by the hardware approximation (ex2.approx: relative error about 2^-22;
// -inf gives 0).  The kernels keep softmax scores in log2 units (their scale
// folds in log2 e), so every exponential of the softmax is one ex2.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// round-half-even(x) for |x| < 2^21, as the low bits of the fp32 sum
// x + 1.5 * 2^23 (whose unit in the last place is 1): the low byte is the
// integer's two's-complement byte.
__device__ __forceinline__ uint32_t rne_bits(float x) { return __float_as_uint(__fadd_rn(x, 12582912.0f)); }

// Packed fp32 pairs for the f32x2 instructions of sm_100-class GPUs: two
// lanes in one 64-bit register pair, each lane an IEEE round-to-nearest
// operation, so each result equals two scalar __fmul_rn / __fadd_rn /
// __fmaf_rn calls bit for bit at half the instruction count.  One exception,
// measured: ptxas fuses add2(mul2(a, b), c) into one multiply-add (the
// product's rounding is lost), so where a product's rounding is part of the
// definition its sum is taken with scalar __fadd_rn instead.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// The bits of RN(x[i] / s + bias) for the N (even) values of one row: div_row's
// quotient, then one add, on packed pairs.  With bias = 1.5 * 2^23 the low byte
// is round-half-even(x / s) (rne_bits); the same results as div_row followed by
// the scalar add, element by element.
template <int N>
__device__ __forceinline__ void div_rne_row(const float (&x)[N], float s, float y, uint32_t (&q)[N],
                                            float bias = 12582912.0f) {
  if (s < kTinyDivisor) {
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = x[i];
    div_row(t, s, y);
#pragma unroll
    for (int i = 0; i < N; ++i) q[i] = __float_as_uint(__fadd_rn(t[i], bias));
    return;
  }
  const uint64_t y2 = f2(y, y), ns2 = f2(-s, -s), c2 = f2(bias, bias);
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const uint64_t v = f2(x[2 * i], x[2 * i + 1]);
    const uint64_t qq = mul2(v, y2);
    const uint64_t r = fma2(ns2, qq, v);
    float lo, hi;
    f2_split(add2(fma2(r, y2, qq), c2), lo, hi);
    q[2 * i] = __float_as_uint(lo);
    q[2 * i + 1] = __float_as_uint(hi);
  }
}

// a / 127 correctly rounded, by the same method with the constant RN(1/127).
// Checked exhaustively against IEEE division for every float of [1, 2), of the
// top binade [2^127, 2^128) and of [2^-100, 2^-98): scaling a by a power of
// two scales the product, the residual and the corrected quotient exactly, so
// every normal binade between repeats the pattern of [1, 2), and the top and
// bottom binades are where overflow or underflow could break it.  Inputs below
// 2^-100 use the plain division.
__device__ __forceinline__ float div127(float a) {
  if (a < kTinyDivisor) return div127_tiny(a);
  const float y = 0.0078740157f;  // RN(1/127)
  const float q = __fmul_rn(a, y);
  const float r = __fmaf_rn(-127.0f, q, a);
  return __fmaf_rn(r, y, q);
}

// a / 255 correctly rounded, the same method with RN(1/255) (the UINT8
// probability scale); the same exhaustive check covers it.
static __device__ __noinline__ float div255_tiny(float a) { return __fdiv_rn(a, 255.0f); }
__device__ __forceinline__ float div255(float a) {
  if (a < kTinyDivisor) return div255_tiny(a);
  const float y = 0x1.010102p-8f;  // RN(1/255)
  const float q = __fmul_rn(a, y);
  const float r = __fmaf_rn(-255.0f, q, a);
  return __fmaf_rn(r, y, q);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Two fp32 values rounded to nearest-even bf16, packed {lo, hi} (cvt.rn.bf16x2).
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Attention outputs are fp32 or, when out_bf16 is set, the same fp32 values
// rounded to nearest-even bf16 (the pages' decode writes BF16 after the
// partition merge).  `i` is an element index into [rows, D].
__device__ __forceinline__ void store_out1(void* out, int out_bf16, size_t i, float v) {
  if (out_bf16)
    static_cast<uint16_t*>(out)[i] = (uint16_t)(bf16x2_rn(v, 0.f) & 0xffffu);
  else
    static_cast<float*>(out)[i] = v;
}
// Four consecutive elements, i a multiple of 4 (16-byte fp32 or 8-byte bf16 store).
__device__ __forceinline__ void store_out4(void* out, int out_bf16, size_t i, float4 v) {
  if (out_bf16)
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + i) = make_uint2(bf16x2_rn(v.x, v.y), bf16x2_rn(v.z, v.w));
  else
    *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = v;
}

// Host: launch `kernel` with programmatic stream serialization allowed, so its
// launch overlaps the tail of the previous kernel on `stream` (the kernel must
// call griddep_wait() before it touches memory the previous kernel writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace i8kv
