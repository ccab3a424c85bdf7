// kda_tc_common.cuh -- PTX wrappers and shared-memory operand layouts used by
// the tensor-core kernels (tcgen05 MMAs with TMEM accumulators, TMA and bulk
// copies, mbarriers).  Internal to libkda.
//
// Operand layouts (no swizzle; checked against the hardware by a standalone
// probe before the kernels used them):
//   K-major  element (row, k): (row%8)*16 + (row/8)*(Kd*16) + (k/8)*128 + (k%8)*2
//   MN-major element (mn, k):  (mn/8)*(Kd*16) + (k/8)*128 + (k%8)*16 + (mn%8)*2
// Both use the descriptor LBO = 128 B (next 8 K-rows / core matrix along K)
// and SBO = Kd*16 B (next 8 rows or 8 MN elements); an MMA step over K = 16
// advances the start address by 256 bytes.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {
namespace tc {

// Byte offset of element (row, k) in a K-major no-swizzle operand with Kd
// columns: 8x8 core matrices of 16-byte rows; core matrices along K are 128
// bytes apart (LBO), groups of 8 rows are Kd*16 bytes apart (SBO).
__device__ __forceinline__ uint32_t op_off(int row, int k, int Kd) {
  return (uint32_t)((row & 7) * 16 + (row >> 3) * (Kd * 16) + (k >> 3) * 128 +
                    (k & 7) * 2);
}

// Byte offset of element (mn, k) in an MN-major no-swizzle operand: a core
// matrix holds 8 K-rows of 8 consecutive MN elements (16 bytes each); the
// same LBO (128 B, next 8 K-rows) and SBO (Kd*16 B, next 8 MN elements) as
// the K-major layout, so one descriptor form serves both.
__device__ __forceinline__ uint32_t mn_off(int mn, int k, int Kd) {
  return (uint32_t)((mn >> 3) * (Kd * 16) + (k >> 3) * 128 + (k & 7) * 16 +
                    (mn & 7) * 2);
}

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                   bar),
               "r"(bytes)
               : "memory");
}

// Plain arrive (count 1) on a CTA-local mbarrier; release semantics at CTA
// scope, so the caller's prior writes are visible to a thread that observes
// the phase completing.
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

// Bounded wait: gives up after `limit` SM clocks (default about one second).
constexpr long long kWaitLimit = 2ll << 30;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          long long limit = kWaitLimit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map,
                                            int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 1-D bulk copy global -> shared (size a multiple of 16, both 16-B aligned).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Bring `bytes` (a multiple of 16, 16-B aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                   reinterpret_cast<uint64_t>(src)),
               "r"(bytes)
               : "memory");
}

// Bring one box of a tiled tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          slot),
      "r"(ncols)
      : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(ncols)
               : "memory");
}

// Shared-memory matrix descriptor: start address, LBO = 128 B (next core
// matrix along K), SBO (next group of 8 rows), fixed field 0b001 at bit 46,
// no swizzle, base offset 0.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((128u >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B,
// A / B transposed (MN-major) when ta / tb, N >> 3 at bit 17, M >> 4 at 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int ta, int tb) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)ta << 15) |
         ((uint32_t)tb << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b,
                                         uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
          "r"(bar)
      : "memory");
}

// D (M = 128) += A (128 x Kd) * B (N x Kd)^T, Kd / 16 instructions.
__device__ __forceinline__ void mma_group(uint32_t d_tmem, uint32_t a_addr,
                                          uint32_t b_addr, int Kd, int N,
                                          bool accumulate, int ta, int tb) {
  const uint32_t id = idesc_bf16(128, N, ta, tb);
  const uint32_t sbo = (uint32_t)Kd * 16u;
  for (int s = 0; s < Kd / 16; ++s) {
    mma_bf16(d_tmem, smem_desc(a_addr + 256u * s, sbo),
             smem_desc(b_addr + 256u * s, sbo), id,
             (accumulate || s > 0) ? 1u : 0u);
  }
}

// An operand in shared memory with explicit strides, for layouts other than
// the two above: `lbo` is the byte stride between core matrices along K and
// `sbo` between groups of 8 rows (K-major) or 8 MN elements (MN-major).  A
// K-major tile stored with op_off(row, k, Kd), read with lbo = Kd*16,
// sbo = 128 and the transpose bit, is the operand whose MN index is `k`
// and whose K index is `row` (its transpose); the 64-row TMA boxes of 8
// columns ([column group][row][8]) are a K-major operand over rows with
// lbo = 1024, sbo = 128.
struct Opnd {
  uint32_t addr, lbo, sbo;
};

__device__ __forceinline__ uint64_t smem_desc_ls(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// D (M = 128, N columns) (+)= A B^T over `ksteps` steps of K = 16; each step
// moves both operands two core matrices along K.  ta / tb: MN-major.
__device__ __forceinline__ void mma_k(uint32_t d_tmem, Opnd a, int ta, Opnd b, int tb,
                                      int ksteps, int N, bool accumulate) {
  const uint32_t id = idesc_bf16(128, N, ta, tb);
  for (int s = 0; s < ksteps; ++s)
    mma_bf16(d_tmem, smem_desc_ls(a.addr + 2u * a.lbo * (uint32_t)s, a.lbo, a.sbo),
             smem_desc_ls(b.addr + 2u * b.lbo * (uint32_t)s, b.lbo, b.sbo), id,
             (accumulate || s > 0) ? 1u : 0u);
}

// 8 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 16-column loads, one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t t0, uint32_t t1, float (&v)[16],
                                            float (&w)[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(t0), "r"(t1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = __uint_as_float(r[i]);
    w[i] = __uint_as_float(r[16 + i]);
  }
}

// 8 consecutive fp32 columns without waiting: a batch of these is followed
// by one tmem_wait_ld(), then reg_fence8() on each result so no use of the
// registers is scheduled before the wait.
__device__ __forceinline__ void tmem_ld8_nw(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void reg_fence8(uint32_t (&r)[8]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
               "+r"(r[6]), "+r"(r[7]));
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  float a[16], b[16];
  tmem_ld16x2(taddr, taddr + 16, a, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = a[i];
    v[16 + i] = b[i];
  }
}

// 2^x on the special function unit (flushes results below FLT_MIN to 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void st_bf16x8(unsigned char *smem, uint32_t off,
                                          const float (&v)[8]) {
  uint4 w;
  w.x = pack_bf16(v[0], v[1]);
  w.y = pack_bf16(v[2], v[3]);
  w.z = pack_bf16(v[4], v[5]);
  w.w = pack_bf16(v[6], v[7]);
  *reinterpret_cast<uint4 *>(smem + off) = w;
}

__device__ __forceinline__ void ld_bf16x8(const unsigned char *p, float (&v)[8]) {
  const uint4 w = *reinterpret_cast<const uint4 *>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&u[i]);
    v[2 * i] = __low2float(h);
    v[2 * i + 1] = __high2float(h);
  }
}


}  // namespace tc
}  // namespace kda
