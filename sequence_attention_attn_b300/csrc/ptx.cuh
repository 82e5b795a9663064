// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers with bounded
// waits, TMA tensor loads, tcgen05 (TMEM allocation, MMA, loads/stores,
// fences) and the shared-memory / instruction descriptors of kind::f16 MMAs.
//
// Every wait on an mbarrier is bounded: after ~1 s of device time it records a
// code in the device status word and returns false, so that a logic error
// ends the kernel with an error status instead of hanging the GPU.  Once the
// status word is non-zero every later main-loop wait gives up soon after.
// Drain waits -- the ones a CTA makes before it frees TMEM or exits, on its
// own TMA loads and MMAs in flight -- ignore the status word and honour only
// their own time limit: those operations complete by themselves, and a CTA
// must not release memory they still write.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace ditk {

// Device status word (one per device; read and cleared by the host).
__device__ unsigned int g_status;
// The value the last status read took out of g_status (see status_take_kernel).
__device__ unsigned int g_status_taken;

constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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

// Waits until the phase with the given parity has completed.  Returns false
// (and sets the status word) if that takes longer than kWaitLimitNs.  With
// kHonourStatus it also returns false once another wait anywhere on the
// device has given up (main-loop waits); without it only its own time limit
// ends it (drain waits).
template <bool kHonourStatus>
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (kHonourStatus && *reinterpret_cast<volatile unsigned int *>(&g_status) != 0u) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow<true>(bar, parity);
}

// A wait on the CTA's own asynchronous work before it exits or frees TMEM.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow<false>(bar, parity);
}

// Warp-uniform wait: every lane polls, and the warp proceeds only if all did.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool mbar_wait_drain_warp(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait_drain(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// One thread waits on a barrier that never completes: the bounded wait must
// give up, set the status word and return.
__global__ void selftest_wait_kernel() {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  mbar_wait(b, 0);
}

// Reads and clears the status word in one atomic exchange, so that a timeout
// recorded by a kernel on another stream is either taken here or left for the
// next read, never lost between a read and a separate clear.
__global__ void status_take_kernel() { g_status_taken = atomicExch(&g_status, 0u); }

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream is still
// running: launch_dependents lets the next kernel launch once every CTA of
// this grid has issued it (or exited), and wait blocks until the previous
// grid has completed and its memory operations are visible.  Without the
// launch attribute both are no-ops.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------- TMA
// 3-D tiled load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(cache_hint)
      : "memory");
}

// 3-D tiled store shared -> global in a bulk group; parts of the box past the
// tensor map's extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 eviction-priority policies for the cache_hint operand.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// MMA and commit, warp-wide: every lane of the warp executes the call with
// the same (warp-uniform) operands and one elected lane issues the
// instruction, so the operand arithmetic stays on the uniform datapath.  The
// elected lane is the same on every call of a converged warp, which the
// commit relies on: it arrives on `bar` once every tcgen05 operation that
// lane issued so far has completed.  Shared-memory descriptors are passed as
// their low and high words (see desc_lo / desc_hi).
//   umma_ss_e: D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, one CTA.
//   umma_ts_e: D[tmem] (+)= A[tmem] * B[smem],   kind::f16, one CTA.
__device__ __forceinline__ void umma_ss_e(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                          uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_ts_e(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 db;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Four K = 16 steps of D[tmem] (+)= A[smem] * B[smem]^T in one block, one
// elected lane (the same one as every other call of a converged warp): both
// descriptors advance by 32 bytes a step (2 in the start-address field); the
// first step accumulates only if acc0 != 0, the others always.
__device__ __forceinline__ void umma_ss4_e(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred e, p0, p1;\n\t.reg .b64 da, db;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\t"
      "setp.eq.b32 p1, %3, %3;\n\t"
      "mov.b64 da, %1;\n\tmov.b64 db, %2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p0;\n\t"
      "add.s64 da, da, 2;\n\tadd.s64 db, db, 2;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, da, 2;\n\tadd.s64 db, db, 2;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, da, 2;\n\tadd.s64 db, db, 2;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc0)
      : "memory");
}
// Eight K = 16 steps of D[tmem] (+)= A[tmem] * B[smem] in one block: A
// advances 8 TMEM columns a step, B's descriptor 2048 bytes (128 in the
// start-address field); the first step accumulates only if acc0 != 0.
__device__ __forceinline__ void umma_ts8_e(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred e, p0, p1;\n\t.reg .b64 db;\n\t.reg .b32 ta;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\t"
      "setp.eq.b32 p1, %3, %3;\n\t"
      "mov.b32 ta, %1;\n\tmov.b64 db, %2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p0;\n\t"
      "add.u32 ta, ta, 8;\n\tadd.s64 db, db, 128;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, ta, 8;\n\tadd.s64 db, db, 128;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, ta, 8;\n\tadd.s64 db, db, 128;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, ta, 8;\n\tadd.s64 db, db, 128;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, ta, 8;\n\tadd.s64 db, db, 128;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, ta, 8;\n\tadd.s64 db, db, 128;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, ta, 8;\n\tadd.s64 db, db, 128;\n\t" "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc0)
      : "memory");
}
__device__ __forceinline__ uint64_t desc64(uint32_t lo, uint32_t hi) {
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ void umma_commit_e(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM -> 32 registers per thread, waited
// inside the same asm block so no use of the registers can be scheduled
// before the data has landed.
#define DITK_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), \
                   "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : DITK_R8(0), DITK_R8(8), DITK_R8(16), DITK_R8(24)
      : "r"(taddr)
      : "memory");
}

// 128 columns in four x32 reducing loads (tcgen05.ld.red, sm_103a), one wait:
// besides the values, each load returns the max of its 32 columns in this
// thread's lane; mx is the max of the four.
__device__ __forceinline__ void tmem_ld128_max_wait(uint32_t taddr, uint32_t (&r)[128], float &mx) {
  float m0, m1, m2, m3;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %128, [%132];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, %129, [%133];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, %130, [%134];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, %131, [%135];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : DITK_R8(0), DITK_R8(8), DITK_R8(16), DITK_R8(24), DITK_R8(32), DITK_R8(40), DITK_R8(48), DITK_R8(56),
        DITK_R8(64), DITK_R8(72), DITK_R8(80), DITK_R8(88), DITK_R8(96), DITK_R8(104), DITK_R8(112), DITK_R8(120),
        "=f"(m0), "=f"(m1), "=f"(m2), "=f"(m3)
      : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
      : "memory");
  mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// 128 columns in four x32 loads, one wait.
__device__ __forceinline__ void tmem_ld128_wait(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : DITK_R8(0), DITK_R8(8), DITK_R8(16), DITK_R8(24), DITK_R8(32), DITK_R8(40),
        DITK_R8(48), DITK_R8(56), DITK_R8(64), DITK_R8(72), DITK_R8(80), DITK_R8(88),
        DITK_R8(96), DITK_R8(104), DITK_R8(112), DITK_R8(120)
      : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : DITK_R8(0), DITK_R8(8)
      : "r"(taddr)
      : "memory");
}
#undef DITK_R8

#define DITK_W8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), \
                   "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])
// 32 registers -> 32 lanes x 32 columns (not waited; see tmem_st_wait).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      DITK_W8(0), DITK_W8(8), DITK_W8(16), DITK_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      DITK_W8(0), DITK_W8(8)
      : "memory");
}
#undef DITK_W8
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor (tcgen05 form) as its two 32-bit words.
// Low word: start address >> 4 in bits 0-13 and the leading byte offset >> 4
// in bits 16-29; shared-memory addresses are below 2^18, so adding a multiple
// of 16 bytes to the start address never carries into the offset field.  High
// word: stride byte offset >> 4 in bits 0-13, descriptor version 1 at bit 14,
// swizzle mode in bits 29-31 (bits 32-45, 46 and 61-63 of the descriptor).
constexpr uint32_t kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6;

__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return (saddr >> 4) | ((lbo_bytes >> 4) << 16);
}
__host__ __device__ constexpr uint32_t desc_hi(uint32_t sbo_bytes, uint32_t swizzle) {
  return (sbo_bytes >> 4) | (1u << 14) | (swizzle << 29);
}

// Instruction descriptor for kind::f16 with bf16 A and B, fp32 accumulator.
// A is K-major; B is K-major (b_mn_major = false) or MN-major (true).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn_major) {
  return (1u << 4)                                  // D format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// ----------------------------------------------------------------- math
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pair arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rd;\n\t"
      "mov.b64 rd, {%0, %1};\n\tmov.b64 ra, {%2, %3};\n\t"
      "add.rn.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace ditk
