// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM allocation, MMA, commit, TMEM loads) and the proxy fences between them.
//
// Every wait here is bounded: it polls with mbarrier.try_wait and gives up after a limit
// measured on %globaltimer, records the failure in the device error word and returns
// false, so that a protocol mistake ends the kernel instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace b2b {

// ------------------------------------------------------------------------------------
// device error word: {code, kernel id, wait site, tile}; the first error wins.
// ------------------------------------------------------------------------------------
enum : uint32_t { ERR_CODE_TIMEOUT = 6 };

__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code, uint32_t kernel,
                                             uint32_t site, uint32_t tile) {
  if (err == nullptr) return;
  if (atomicCAS(&err[0], 0u, code) == 0u) {
    err[1] = kernel;
    err[2] = site;
    err[3] = tile;
    __threadfence();
  }
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_if(uint32_t pred, uint32_t bar,
                                                         uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%1], %2;\n\t}" ::"r"(pred),
      "r"(bar), "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the hardware park the warp for up to `hint_ns` (it resumes as soon
// as the phase completes), so that waiting warps take no issue slots from the warps that
// share their scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  `abort_flag` (shared
// memory, may be null) lets one role that gave up stop the others quickly.  Between
// checks of the limit the warp sleeps in try_wait (at most 100 us at a time).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          volatile uint32_t* abort_flag, uint32_t* err,
                                          uint32_t kernel, uint32_t site, uint32_t tile) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if (abort_flag != nullptr && *abort_flag != 0u) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      record_error(err, ERR_CODE_TIMEOUT, kernel, site, tile);
      if (abort_flag != nullptr) *abort_flag = 1u;
      return false;
    }
  }
}

// ------------------------------------------------------------------------------------
// warp-converged issue
// ------------------------------------------------------------------------------------
// Returns 1 in exactly one lane of the (fully converged) warp.  The producer and MMA
// roles run as whole warps and predicate their single-thread instructions on this value,
// so their loop state stays warp-uniform and the issue path stays short.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t is_leader;
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, e;\n\t}"
      : "=r"(is_leader));
  return is_leader;
}

// ------------------------------------------------------------------------------------
// fences
// ------------------------------------------------------------------------------------
// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// reads (tcgen05.mma operands, TMA stores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of the stream
// (launched with programmatic stream serialisation) be scheduled while this grid still
// runs; dependency_wait blocks until every prerequisite grid has completed and its memory
// is visible, and returns at once when the kernel was launched without a prerequisite.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// TMA
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// TMA tile loads into shared memory, completing on `bar`; issued only where pred != 0.
__device__ __forceinline__ void tma_load_2d(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                            uint32_t bar, int32_t c0, int32_t c1, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%1], [%2, {%4, %5}], [%3], %6;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                            uint32_t bar, int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%1], [%2, {%4, %5, %6}], [%3], %7;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                            uint32_t bar, int32_t c0, int32_t c1, int32_t c2,
                                            int32_t c3, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%1], [%2, {%4, %5, %6, %7}], [%3], %8;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "l"(policy)
      : "memory");
}

// L2 prefetch of `bytes` contiguous bytes at a 16-byte aligned global address (bytes a
// multiple of 16): no shared memory, no barrier; it only warms L2 for later loads.
__device__ __forceinline__ void bulk_prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(ptr)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

// As tma_store_2d, with an L2 cache policy (createpolicy) for the written lines.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int32_t c0,
                                                  int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::
          "l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until all committed bulk stores have finished READING shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}


// ------------------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor-core MMA
// ------------------------------------------------------------------------------------
// Allocates `ncols` TMEM columns (power of two >= 32); the base address is written to
// shared memory at `dst`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
//   K-major operand (rows of 128 B along K): lbo unused (16), sbo = 1024 (8-row groups).
//   MN-major operand (rows of 128 B along M/N, one row per k): lbo = byte distance between
//   64-element M/N blocks, sbo = 1024 (groups of 8 k-rows).
// Fields: start>>4 [0,14), lbo>>4 [16,30), sbo>>4 [32,46), version 1 [46,48),
// base offset 0 [49,52), layout 2 = SWIZZLE_128B [61,64).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor, kind::f16 with fp32 accumulation.
//   [4,6) D format 1 = f32; [7,10) A format; [10,13) B format (0 = f16, 1 = bf16);
//   bit 15 A major (0 = K); bit 16 B major (1 = MN); [17,23) N>>3; [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t is_bf16, uint32_t b_mn_major,
                                                     uint32_t M, uint32_t N) {
  return (1u << 4) | (is_bf16 << 7) | (is_bf16 << 10) | (b_mn_major << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] x B[smem]; issued only where pred != 0 (one lane).
__device__ __forceinline__ void mma_f16_ss(uint32_t pred, uint32_t d_tmem, uint64_t a_desc,
                                           uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 q, %0, 0;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %3, %4, p;\n\t}" ::"r"(pred),
      "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four consecutive K steps of one 64-wide K chunk in one asm block: the descriptors of
// step j are a + j * astep and b + j * bstep (16-byte units); the first step accumulates
// when `accumulate` != 0, the others always.  One predicate setup and no compiler-visible
// boundaries between the four issues: the issuing thread is otherwise the bottleneck for
// N <= 64, whose MMAs the tensor core finishes in ~48 cycles.
__device__ __forceinline__ void mma_f16_ss_x4(uint32_t pred, uint32_t d_tmem, uint64_t a,
                                              uint64_t b, uint64_t astep, uint64_t bstep,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred q, p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 q, %0, 0;\n\t"
      "setp.ne.b32 p, %7, 0;\n\t"
      "setp.eq.b32 t, %0, %0;\n\t"
      "add.s64 a1, %2, %4;\n\t"
      "add.s64 b1, %3, %5;\n\t"
      "add.s64 a2, a1, %4;\n\t"
      "add.s64 b2, b1, %5;\n\t"
      "add.s64 a3, a2, %4;\n\t"
      "add.s64 b3, b2, %5;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %3, %6, p;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%1], a1, b1, %6, t;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%1], a2, b2, %6, t;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%1], a3, b3, %6, t;\n\t}" ::"r"(pred),
      "r"(d_tmem), "l"(a), "l"(b), "l"(astep), "l"(bstep), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] x B[smem] ("TS" form): A is 128 lanes (rows) x 16 K elements packed
// two per 32-bit column, 8 columns per K step.  Issued only where pred != 0.
__device__ __forceinline__ void mma_f16_ts(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem,
                                           uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 q, %0, 0;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %3, %4, p;\n\t}" ::"r"(pred),
      "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives (once) on `bar` when every tcgen05.mma previously issued by this thread is done;
// issued only where pred != 0 (the lane that issued the MMAs).
__device__ __forceinline__ void mma_commit(uint32_t pred, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}" ::
          "r"(pred),
      "r"(bar)
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp gets lane (base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 32 lanes x 32 bits, 64 consecutive columns in one instruction.
__device__ __forceinline__ void tmem_ld64x(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}

// 32 lanes x 32 bits, 32 consecutive columns from registers in one instruction.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// 32 lanes x 32 bits, 8 consecutive columns from registers (thread t -> lane base + t).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// wait::ld that also threads the loaded registers through the asm statement, so that no
// use of them can be scheduled before the wait completes.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Four consecutive fp32 words of shared memory at a 16-byte aligned address.
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// 32 consecutive columns in two x16 loads (the second only if `two`).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, bool two, uint32_t (&r)[16],
                                          uint32_t (&s)[16]) {
  tmem_ld16(taddr, r);
  if (two) tmem_ld16(taddr + 16, s);
}

__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16], uint32_t (&s)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(s[0]), "+r"(s[1]),
                 "+r"(s[2]), "+r"(s[3]), "+r"(s[4]), "+r"(s[5]), "+r"(s[6]), "+r"(s[7]),
                 "+r"(s[8]), "+r"(s[9]), "+r"(s[10]), "+r"(s[11]), "+r"(s[12]), "+r"(s[13]),
                 "+r"(s[14]), "+r"(s[15])
               :
               : "memory");
}

// ------------------------------------------------------------------------------------
// CTA pairs (a cluster of two CTAs, tcgen05 .cta_group::2).  One MMA of M = 256 rows spans
// both SMs: each CTA's shared memory holds its 128 rows of A and its half of B's N
// columns, and each CTA's TMEM receives its 128 rows of D.  Every tcgen05 allocation,
// MMA and commit of a pair kernel carries .cta_group::2.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// All threads of both CTAs of the cluster; orders each side's earlier memory operations
// (barrier initialisation, remote arrives) before the other side's later ones.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier anywhere in the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Arrive on an mbarrier anywhere in the cluster, release at CTA scope: the signal of a
// thread whose tcgen05 operations are complete and fenced (tcgen05.wait::ld / wait::st,
// tcgen05.fence::before_thread_sync) to the peer CTA's MMA issuer, which acquires the
// barrier and fences with tcgen05.fence::after_thread_sync.  A release at cluster scope
// would also wait for this thread's earlier global stores to be performed cluster-wide.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Bounded wait with acquire at cluster scope (for phases completed by the peer CTA's
// arrives or by the pair's MMA commits); otherwise as mbar_wait.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  volatile uint32_t* abort_flag, uint32_t* err,
                                                  uint32_t kernel, uint32_t site, uint32_t tile) {
  if (mbar_try_wait_cluster(bar, parity, 0u)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity, 100000u)) return true;
    if (abort_flag != nullptr && *abort_flag != 0u) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      record_error(err, ERR_CODE_TIMEOUT, kernel, site, tile);
      if (abort_flag != nullptr) *abort_flag = 1u;
      return false;
    }
  }
}

// TMA loads of a pair kernel: the data lands in this CTA's shared memory and completes
// on `bar_cluster`, a barrier in either CTA of the pair (the leader's, which counts both
// CTAs' bytes before its MMA reads them).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%1], [%2, {%4, %5}], [%3], %6;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 int32_t c2, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%1], [%2, {%4, %5, %6}], [%3], %7;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 int32_t c2, int32_t c3, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%1], [%2, {%4, %5, %6, %7}], [%3], %8;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "l"(policy)
      : "memory");
}

// TMEM allocation for the pair: one warp in EACH CTA executes it, and both get the same
// columns.  Whole warp.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D (+)= A . B over the pair (M = 256 in the instruction descriptor); issued by one lane of
// the leader CTA only.
__device__ __forceinline__ void mma_pair_ss(uint32_t pred, uint32_t d_tmem, uint64_t a_desc,
                                            uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 q, %0, 0;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%1], %2, %3, %4, p;\n\t}" ::"r"(pred),
      "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four K steps of mma_pair_ss in one block (as mma_f16_ss_x4): the first accumulates when
// `accumulate` != 0, the others always.
__device__ __forceinline__ void mma_pair_ss_x4(uint32_t pred, uint32_t d_tmem, uint64_t a,
                                               uint64_t b, uint64_t astep, uint64_t bstep,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred q, p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 q, %0, 0;\n\t"
      "setp.ne.b32 p, %7, 0;\n\t"
      "setp.eq.b32 t, %0, %0;\n\t"
      "add.s64 a1, %2, %4;\n\t"
      "add.s64 b1, %3, %5;\n\t"
      "add.s64 a2, a1, %4;\n\t"
      "add.s64 b2, b1, %5;\n\t"
      "add.s64 a3, a2, %4;\n\t"
      "add.s64 b3, b2, %5;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%1], %2, %3, %6, p;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%1], a1, b1, %6, t;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%1], a2, b2, %6, t;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%1], a3, b3, %6, t;\n\t}" ::"r"(pred),
      "r"(d_tmem), "l"(a), "l"(b), "l"(astep), "l"(bstep), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The TS form over the pair: A from each CTA's TMEM (its 128 rows), B from shared memory.
__device__ __forceinline__ void mma_pair_ts(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem,
                                            uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 q, %0, 0;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%1], [%2], %3, %4, p;\n\t}" ::"r"(pred),
      "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the barrier at `bar` (a CTA-local offset) in every CTA of `cta_mask`
// when all tcgen05.mma previously issued by this thread are done.
__device__ __forceinline__ void mma_commit_pair(uint32_t pred, uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%1], %2;\n\t}" ::"r"(pred),
      "r"(bar), "h"(cta_mask)
      : "memory");
}

}  // namespace b2b
