// Device-side building blocks for sm_103a: mbarriers with bounded waits, TMA tile loads,
// tcgen05 (TMEM allocation, UMMA issue, commit, TMEM loads) and programmatic dependent
// launch controls.  Inline PTX only; no library kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define KLT_DEV __device__ __forceinline__

namespace klt {

// Sticky device error bits, OR-ed into the handle's error word.
enum : int { DEV_ERR_TIMEOUT = 1 };

KLT_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ PDL
KLT_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
KLT_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ mbarrier
KLT_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
KLT_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
KLT_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
KLT_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
KLT_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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
// As mbar_try_wait, but the thread is suspended (without taking issue slots from the warps
// sharing its scheduler) until the phase completes or about `hint_ns` elapse.
KLT_DEV bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`, giving up after `timeout` SM cycles or as soon as the
// CTA's abort flag is raised.  On expiry raises the abort flag and the device error bit.
// Returns false when the wait did not complete.  Waiting threads sleep in hardware between
// checks so they do not steal issue slots from the MMA and copy threads.
KLT_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                       int* err_word, long long timeout) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 2000)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > timeout) {
      *abort_flag = 1;
      atomicOr(err_word, DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// As mbar_wait, for the latency-critical hand-offs of the tensor pipeline: polls without a
// suspend-time hint so the waiter resumes as soon as the phase completes.
KLT_DEV bool mbar_wait_spin(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                            int* err_word, long long timeout) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > timeout) {
      *abort_flag = 1;
      atomicOr(err_word, DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// ------------------------------------------------------------------ TMA
KLT_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled load of the box at (c0 = inner element index, c1 = row) into shared memory,
// completing `bytes` of transaction count on `bar`.
KLT_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
// 1-D bulk copy of `bytes` contiguous bytes (16-byte aligned, multiple of 16) into shared
// memory, completing the transaction count on `bar`.
KLT_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                       uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Asks L2 to fetch `bytes` (a multiple of 16) contiguous bytes from global memory
// (16-byte aligned); no shared memory and no completion tracking.
KLT_DEV void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)),
               "r"(bytes)
               : "memory");
}
// This CTA's share of [p.pf_ptr, p.pf_ptr + p.pf_bytes), in 64 KB requests.
template <typename P>
KLT_DEV void prefetch_share_l2(const P& p) {
  if (p.pf_ptr == nullptr || p.pf_bytes <= 0) return;
  const long long per = ((p.pf_bytes + gridDim.x - 1) / gridDim.x + 15) & ~15ll;
  const long long lo = per * blockIdx.x;
  const long long hi = lo + per < p.pf_bytes ? lo + per : p.pf_bytes;
  for (long long o = lo; o < hi; o += 65536) {
    const long long n = hi - o < 65536 ? hi - o : 65536;
    bulk_prefetch_l2(p.pf_ptr + o, static_cast<uint32_t>(n));
  }
}
KLT_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
KLT_DEV uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
KLT_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ tcgen05
// Shared-memory matrix descriptor for a K-major operand tile stored with the 128-byte
// swizzle: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart, tile base 1024-aligned.
KLT_DEV uint64_t sdesc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |  // start address
         (static_cast<uint64_t>(1) << 16) |                 // leading offset (unused here)
         (static_cast<uint64_t>(1024 >> 4) << 32) |         // stride between 8-row atoms
         (static_cast<uint64_t>(1) << 46) |                 // descriptor version
         (static_cast<uint64_t>(2) << 61);                  // 128-byte swizzle
}

// Instruction descriptor: fp32 accumulator, A and B of the same format, both K-major,
// shape M x N.  Formats: kind::f16 -> 1 = bf16; kind::f8f6f4 -> 0 = e4m3.
__host__ __device__ constexpr uint32_t idesc_make(uint32_t ab_fmt, int m, int n) {
  return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

KLT_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
KLT_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
KLT_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
KLT_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
KLT_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
KLT_DEV void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

KLT_DEV void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
KLT_DEV void mma_fp8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled FP8 MMA (kind::mxf8f6f4, one UE8M0 scale per 32 K-elements, applied by the
// tensor core): K = 32 per instruction.  The scales are read from TMEM: row m of A at lane m,
// column sfa + m/32; column n of B at lane n%32, column sfb + n/32; the byte within the
// 32-bit word is the instruction descriptor's scale id (bits 29-30 for A, 4-5 for B).
KLT_DEV void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                    uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// D (+)= A * B^T with e2m1 operands (two per byte) and one e4m3 scale per 16 K-elements
// of each row (kind::mxf4nvf4, scale vector 4X): K = 64 per MMA (32 bytes of a row).  The
// scales of A row m are the four bytes of TMEM lane m, column sfa_tmem + m / 32 (byte j
// scales K-elements [16j, 16j + 16)); those of B row n are at lane n % 32, column
// sfb_tmem + n / 32 -- the layout tcgen05.cp 32x128b.warpx4 makes of 512-byte tiles whose
// byte (r % 32) * 16 + 4 * (r / 32) + j holds scale j of row r.
KLT_DEV void mma_nv4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                     uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Instruction descriptor of kind::mxf4nvf4 with e2m1 A and B (format 1), e4m3 scales
// (scale format 0), fp32 accumulation, both operands K-major, shape M x N, K = 64.
__host__ __device__ constexpr uint32_t idesc_nv4(int m, int n) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}
// Instruction descriptor of kind::mxf8f6f4 with e4m3 A and B, UE8M0 scales, fp32
// accumulation, both operands K-major, shape M x N, scale ids for A and B.
__host__ __device__ constexpr uint32_t idesc_mx(int m, int n, uint32_t a_sf_id,
                                                uint32_t b_sf_id) {
  return (b_sf_id << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(m >> 4) << 24) | (a_sf_id << 29);
}
// Copies a 32-row x 16-byte shared-memory tile (row r at +16r) into TMEM columns
// taddr .. taddr+3, lane r of every lane quadrant (tcgen05.cp 32x128b, warpx4).
KLT_DEV void tmem_cp_32x128b_x4(uint32_t taddr, uint32_t saddr) {
  const uint64_t desc = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
                        (static_cast<uint64_t>(128 >> 4) << 16) |
                        (static_cast<uint64_t>(128 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

// The four MMAs of one 128-byte K block (K = 4 x 32 bytes) into one accumulator, issued
// from a single asm block: the first accumulates iff `accumulate`, the rest always do.
// `kind` is the tcgen05.mma kind string (kind::f16 or kind::f8f6f4).
#define KLT_MMA4(KIND)                                                                    \
  asm volatile(                                                                           \
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"        \
      "tcgen05.mma.cta_group::1." KIND " [%0], %1, %2, %3, p;\n\t"                         \
      "tcgen05.mma.cta_group::1." KIND " [%0], %5, %6, %3, q;\n\t"                         \
      "tcgen05.mma.cta_group::1." KIND " [%0], %7, %8, %3, q;\n\t"                         \
      "tcgen05.mma.cta_group::1." KIND " [%0], %9, %10, %3, q;\n\t}" ::"r"(d),             \
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate), "l"(da + 2), "l"(db + 2), "l"(da + 4),  \
      "l"(db + 4), "l"(da + 6), "l"(db + 6)                                                \
      : "memory")
// Gate and up of one K block (eight MMAs, two accumulators `d` and `d + n_off`) in one
// asm block.
#define KLT_MMA8(KIND)                                                                    \
  asm volatile(                                                                           \
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"        \
      "tcgen05.mma.cta_group::1." KIND " [%0], %2, %4, %6, p;\n\t"                         \
      "tcgen05.mma.cta_group::1." KIND " [%1], %3, %4, %6, p;\n\t"                         \
      "tcgen05.mma.cta_group::1." KIND " [%0], %7, %8, %6, q;\n\t"                         \
      "tcgen05.mma.cta_group::1." KIND " [%1], %9, %8, %6, q;\n\t"                         \
      "tcgen05.mma.cta_group::1." KIND " [%0], %10, %11, %6, q;\n\t"                       \
      "tcgen05.mma.cta_group::1." KIND " [%1], %12, %11, %6, q;\n\t"                       \
      "tcgen05.mma.cta_group::1." KIND " [%0], %13, %14, %6, q;\n\t"                       \
      "tcgen05.mma.cta_group::1." KIND " [%1], %15, %14, %6, q;\n\t}" ::"r"(d),            \
      "r"(d + n_off), "l"(da), "l"(du), "l"(db), "r"(accumulate), "r"(idesc), "l"(da + 2), \
      "l"(db + 2), "l"(du + 2), "l"(da + 4), "l"(db + 4), "l"(du + 4), "l"(da + 6),        \
      "l"(db + 6), "l"(du + 6)                                                             \
      : "memory")
KLT_DEV void mma8_bf16(uint32_t d, uint64_t da, uint64_t du, uint64_t db, uint32_t idesc,
                       uint32_t accumulate, uint32_t n_off) {
  KLT_MMA8("kind::f16");
}
KLT_DEV void mma8_fp8(uint32_t d, uint64_t da, uint64_t du, uint64_t db, uint32_t idesc,
                      uint32_t accumulate, uint32_t n_off) {
  KLT_MMA8("kind::f8f6f4");
}
#undef KLT_MMA8

KLT_DEV void mma4_bf16(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc,
                       uint32_t accumulate) {
  KLT_MMA4("kind::f16");
}
KLT_DEV void mma4_fp8(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc,
                      uint32_t accumulate) {
  KLT_MMA4("kind::f8f6f4");
}
#undef KLT_MMA4

// Load 16 consecutive fp32 columns of this thread's TMEM lane and wait for them (the
// wait is in the same asm statement so no use of the registers can move above it).
KLT_DEV void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 16-column loads (e.g. gate and up of one pair) under one wait.
KLT_DEV void tmem_ld16x2(uint32_t ta, uint32_t tb, float* va, float* vb) {
  uint32_t a[16], b[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
        "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]),
        "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]),
        "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]),
        "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    va[i] = __uint_as_float(a[i]);
    vb[i] = __uint_as_float(b[i]);
  }
}

// Four 16-column loads under one wait.
KLT_DEV void tmem_ld16x4(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3, float* v0,
                         float* v1, float* v2, float* v3) {
  uint32_t a[16], b[16], c[16], d[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%65];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%66];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%67];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
        "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]),
        "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]),
        "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]),
        "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]),
        "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3]), "=r"(c[4]), "=r"(c[5]), "=r"(c[6]),
        "=r"(c[7]), "=r"(c[8]), "=r"(c[9]), "=r"(c[10]), "=r"(c[11]), "=r"(c[12]),
        "=r"(c[13]), "=r"(c[14]), "=r"(c[15]), "=r"(d[0]), "=r"(d[1]), "=r"(d[2]),
        "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]), "=r"(d[8]), "=r"(d[9]),
        "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15])
      : "r"(t0), "r"(t1), "r"(t2), "r"(t3)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v0[i] = __uint_as_float(a[i]);
    v1[i] = __uint_as_float(b[i]);
    v2[i] = __uint_as_float(c[i]);
    v3[i] = __uint_as_float(d[i]);
  }
}

// Store 16 consecutive fp32 columns of this thread's TMEM lane and wait for the store.
KLT_DEV void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
KLT_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ misc
// SiLU g / (1 + e^-g) with the fast exponential and the fast divide (each within 2 ulp).
// The exponent is clamped at 80 so the divisor stays inside the fast divide's range; for
// g < -80 the result is below 1e-32 either way.
KLT_DEV float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-fmaxf(g, -80.0f))); }

// Correctly rounded fp32 quotient x / s from inv = 1/s (itself correctly rounded), by one
// residual correction (Markstein's method: q0 = x*inv, r = x - q0*s exactly by FMA,
// q = q0 + r*inv); valid while x / s and the residual stay in the normal range, as for the
// e4m3 requantisation (|x / s| <= 448).  Three FMA-pipe operations instead of a full-range
// division per element.
KLT_DEV float quot_rn(float x, float s, float inv) {
  const float q0 = x * inv;
  const float r = fmaf(-q0, s, x);
  return fmaf(r, inv, q0);
}
// 1/s for normal s: the fast reciprocal refined by one Newton step (error well below
// 1 ulp), for quot_rn when s differs from element to element.
KLT_DEV float rcp_nr(float s) {
  const float y0 = __fdividef(1.0f, s);
  return fmaf(fmaf(-s, y0, 1.0f), y0, y0);
}

// MX (OCP Microscaling, e4m3 elements) shared exponent of a block whose largest magnitude
// is amax: floor(log2 amax) - 8, clamped to the UE8M0 range [-127, 127]; 0 for amax == 0.
// Read from the IEEE fields (a subnormal amax has floor(log2 amax) <= -127).
KLT_DEV int mx_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b == 0) return 0;
  const int f = static_cast<int>(b >> 23);  // biased exponent field
  if (f == 0) return -127;
  const int e = f - 127 - 8;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}
// 2^n as an fp32 value, exact for -127 <= n <= 127 (2^-127 is the subnormal 0x00400000).
KLT_DEV float pow2_exact(int n) {
  return n >= -126 ? __int_as_float((n + 127) << 23) : __int_as_float(0x00400000);
}

// Four consecutive fp32 atomically added to global memory (16-byte aligned), one request.
KLT_DEV void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Per-warpgroup register budget changes (all four warps of the warpgroup execute them).
template <int N>
KLT_DEV void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
KLT_DEV void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// e4m3 code -> fp32 (exact).
KLT_DEV float e4m3_to_f32(uint8_t c) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(h));
}
// e2m1 code (low 4 bits) -> fp32: values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives.
KLT_DEV float e2m1_to_f32(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float mag = e == 0 ? 0.5f * static_cast<float>(m)
                           : __int_as_float(static_cast<int>((126u + e) << 23 | (m << 22)));
  return (c & 8u) ? -mag : mag;
}

// fp32 -> e2m1 code (4 bits): nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6, a tie going to the
// even code (the midpoints 0.25, 1.25, 2.5 and 5 round down, 0.75, 1.75 and 3.5 up),
// saturating at 6; the sign bit only for a non-zero magnitude.
KLT_DEV uint32_t f32_to_e2m1(float v) {
  const float a = fabsf(v);
  const uint32_t c = static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) +
                     static_cast<uint32_t>(a > 1.25f) + static_cast<uint32_t>(a >= 1.75f) +
                     static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) +
                     static_cast<uint32_t>(a > 5.0f);
  return (v < 0.f && c != 0u) ? (c | 8u) : c;
}

// A code whose magnitude bits are zero loses its sign bit (eight 4-bit codes in a word):
// bit 3 of ((m & 7) + 7) is set exactly when the magnitude m is non-zero.
KLT_DEV uint32_t e2m1x8_drop_negative_zero(uint32_t x) {
  const uint32_t nz = ((x & 0x77777777u) + 0x77777777u) & 0x88888888u;
  return x & (nz | 0x77777777u);
}
// Eight fp32 values -> eight e2m1 codes in one word, v[0] in bits 0-3, v[1] in bits 4-7,
// and so on (the even element in the low nibble of each byte): the tensor-core format
// conversion (nearest even on the e2m1 grid, saturating at 6, as f32_to_e2m1), then the
// sign dropped from zero magnitudes.
KLT_DEV uint32_t f32x8_to_e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5,
                                 float v6, float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return e2m1x8_drop_negative_zero(r);
}

// fp32 -> e4m3 code, round to nearest even, saturating to +-448.
KLT_DEV uint8_t f32_to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
// Two values in one conversion: `lo` in bits 0-7, `hi` in bits 8-15.
KLT_DEV uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

KLT_DEV int lane_id() { return threadIdx.x & 31; }

// Cross-CTA signalling inside one launch: writers publish with a release add after their
// data (and a proxy fence when the data is later read by TMA); readers acquire.
KLT_DEV int ld_acquire_gpu(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
KLT_DEV void red_release_gpu_add(int* ptr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
// Orders this thread's generic-proxy global accesses with its async-proxy (TMA) accesses.
KLT_DEV void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

KLT_DEV long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

KLT_DEV void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace klt
