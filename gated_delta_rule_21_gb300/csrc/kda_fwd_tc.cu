// kda_fwd_tc.cu -- chunked KDA forward on the 5th-generation tensor cores
// (tcgen05 MMAs with TMEM accumulators, TMA tile staging), bf16 q/k/v,
// K = V = 128, chunks of 64 tokens.
//
// The method (page "feat(kda): integrate KDA attention with tokamax backend
// and CP support", section "Delta Rule formulation") in the chunk form the
// SIMT kernel also uses.  Per unit = (run, head, 32-column value tile) and per
// chunk of C = 64 rows entering with state S0 (K x 32, fp32 in registers):
//
//   G      = cumsum of g (per channel); block decays D_b = e^{E_b - P_b}
//   X      = [K e1 ; Q e1]                       (128 x 128, A operand)
//   Y_b    = K_{0..16b+15} * e^{P_b - G}         (B operands, one per block)
//   D_b    = X Y_b^T  -> rows of block b: A_kk (k rows), A_qk (q rows)
//   T      = (I + beta * strict(A_kk))^-1        (fp32, blocked, CUDA cores)
//   [w|u]  = [T ; A_qk] [beta K e^{G} | beta V]  (one MMA, N = 160)
//   D1     = [w ; Q e^{G}] S0                    (M = 128: w S0 and Q e^G S0)
//   U      = u - w S0                            (CUDA cores, bf16 operand)
//   D1    += [T ; A_qk] U                        (rows 64..127: O / scale)
//   D2     = (K e^{G_C - G})^T U ;  S1 = e^{G_C} S0 + D2
//
// with e1 = e^{G - P_b}, P_b = G before 16-row block b, E_b = G at its last
// row.  Every factor stays inside bf16/fp32 range for g in [-5, 0]: the
// same-block factor e^{P_b - G} <= e^80, all others <= 1.
//
// All MMAs are tcgen05.mma.cta_group::1.kind::f16 with M = 128, bf16
// operands in shared memory (K-major, no swizzle, 8x16-byte core matrices:
// row groups of 8 rows are contiguous blocks of Kd*16 bytes, the core
// matrices of a row group follow each other every 128 bytes), fp32
// accumulators in TMEM.  One thread issues the MMAs and commits them to an
// mbarrier; every mbarrier wait is bounded and reports a timeout through
// the workspace status word instead of hanging.
//
// Phases run one after another inside the CTA (no warp specialisation); the
// raw tiles of the next chunk are fetched by TMA while the current chunk
// finishes.  256 threads, one CTA per SM (about 219 KB of shared memory),
// all 512 TMEM columns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int C = kChunk;  // 64
constexpr int KD = 128;    // key dim
constexpr int VT = 32;     // value columns per CTA

// ---- shared memory map (byte offsets from a 1024-aligned base) -----------
constexpr uint32_t RAW_Q = 0;                 // 64 x 128 bf16, 256-byte rows
constexpr uint32_t RAW_K = RAW_Q + 16384;
constexpr uint32_t RAW_G = RAW_K + 16384;     // 64 x 128 fp32, 512-byte rows
constexpr uint32_t RAW_V = RAW_G + 32768;     // 64 x 32 bf16, 64-byte rows
constexpr uint32_t RAW_TX_BYTES = 16384 + 16384 + 32768 + 4096;
constexpr uint32_t X_OFF = RAW_V + 4096;      // X: 128 rows x Kd 128
constexpr uint32_t Y_OFF = X_OFF + 32768;     // Y_0..Y_3: 16/32/48/64 rows x 128
constexpr uint32_t ST_OFF = Y_OFF + 160 * 256;  // S^T: 32 rows x Kd 128
constexpr uint32_t WQ_OFF = ST_OFF + 8192;    // [w ; Q e^G]: 128 x 128
constexpr uint32_t KHT_OFF = WQ_OFF + 32768;  // (K e^{G_C-G})^T: 128 x Kd 64
constexpr uint32_t RHST_OFF = KHT_OFF + 16384;  // [beta K e^G | beta V]^T: 160 x 64
constexpr uint32_t MISC_OFF = RHST_OFF + 20480;
constexpr uint32_t BETA_OFF = MISC_OFF;           // 64 fp32
constexpr uint32_t DBLK_OFF = MISC_OFF + 256;     // 4 x 128 fp32 block decays
constexpr uint32_t BAR_OFF = MISC_OFF + 2304;     // two mbarriers
constexpr uint32_t TMEMSLOT_OFF = BAR_OFF + 16;   // u32 TMEM base
constexpr uint32_t ABORT_OFF = TMEMSLOT_OFF + 4;  // u32 abort flag
constexpr uint32_t SMEM_BYTES = ABORT_OFF + 12;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for alignment
// Reused after the intra-chunk MMAs are done with X and Y:
constexpr int LDF = C + 1;                        // padded fp32 row stride
constexpr uint32_t AKK_OFF = X_OFF;               // fp32 64 x 65: beta A_kk
constexpr uint32_t TF_OFF = AKK_OFF + 64 * LDF * 4;  // fp32 64 x 65: T
constexpr uint32_t TAQ_OFF = TF_OFF + 64 * LDF * 4;  // [T ; A_qk]: 128 x Kd 64
constexpr uint32_t UT_OFF = TAQ_OFF + 16384;      // U^T: 32 x Kd 64
constexpr uint32_t SCR_OFF = UT_OFF + 4096;       // 3 x 16 x 16 fp32
static_assert(SCR_OFF + 3072 <= ST_OFF, "aliases stay inside X and Y");
static_assert(TAQ_OFF % 16 == 0 && UT_OFF % 16 == 0, "operands 16-byte aligned");
static_assert(SMEM_ALLOC <= 232448, "fits the 227 KB opt-in limit");

// Rows before Y_b (rows of Y_b = 16 (b + 1)).
__device__ __forceinline__ uint32_t y_off(int b) {
  return Y_OFF + 256u * (uint32_t)(8 * b * (b + 1));
}

// ---- TMEM column map (512 columns allocated) ------------------------------
constexpr uint32_t TM_A0 = 0, TM_A1 = 32, TM_A2 = 64, TM_A3 = 128;
constexpr uint32_t TM_TX = 192;  // 160 columns: [w | u]
constexpr uint32_t TM_D1 = 352;  // 32 columns
constexpr uint32_t TM_D2 = 384;  // 32 columns
constexpr uint32_t TMEM_COLS = 512;
static_assert(TM_D2 + 32 <= TMEM_COLS, "TMEM map fits");
__device__ __forceinline__ uint32_t tm_a(int b) {
  return b == 0 ? TM_A0 : b == 1 ? TM_A1 : b == 2 ? TM_A2 : TM_A3;
}

// Byte offset of element (row, k) in a K-major no-swizzle operand with Kd
// columns: 8x8 core matrices of 16-byte rows; core matrices along K are 128
// bytes apart (LBO), groups of 8 rows are Kd*16 bytes apart (SBO).
__device__ __forceinline__ uint32_t op_off(int row, int k, int Kd) {
  return (uint32_t)((row & 7) * 16 + (row >> 3) * (Kd * 16) + (k >> 3) * 128 +
                    (k & 7) * 2);
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

// Bounded wait: gives up after about one second of SM clock.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (2ll << 30)) return false;
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

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
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
                                          bool accumulate) {
  const uint32_t id = idesc_bf16(128, N);
  const uint32_t sbo = (uint32_t)Kd * 16u;
  for (int s = 0; s < Kd / 16; ++s) {
    mma_bf16(d_tmem, smem_desc(a_addr + 256u * s, sbo),
             smem_desc(b_addr + 256u * s, sbo), id,
             (accumulate || s > 0) ? 1u : 0u);
  }
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

__device__ __forceinline__ void st_bf16(unsigned char *smem, uint32_t off,
                                        float v) {
  *reinterpret_cast<__nv_bfloat16 *>(smem + off) = __float2bfloat16_rn(v);
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

// Which 16-column pieces of the intra-chunk products each TMEM lane quadrant
// reads: quadrants 0/2 hold rows 0..31 (blocks 0, 1), 1/3 rows 32..63.
__device__ __forceinline__ int piece_count(int quad) { return (quad & 1) ? 7 : 3; }
__device__ __forceinline__ void piece(int quad, int i, int &b, int &p) {
  if ((quad & 1) == 0) {
    b = i == 0 ? 0 : 1;
    p = i == 0 ? 0 : i - 1;
  } else {
    b = i < 3 ? 2 : 3;
    p = i < 3 ? i : i - 3;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_g,
                  const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  float *sBeta = reinterpret_cast<float *>(smem + BETA_OFF);
  float *sDblk = reinterpret_cast<float *>(smem + DBLK_OFF);
  float *sG = reinterpret_cast<float *>(smem + RAW_G);
  float *sAkk = reinterpret_cast<float *>(smem + AKK_OFF);
  float *sT = reinterpret_cast<float *>(smem + TF_OFF);
  float *sScr = reinterpret_cast<float *>(smem + SCR_OFF);
  volatile uint32_t *sAbort = reinterpret_cast<volatile uint32_t *>(smem + ABORT_OFF);
  const uint32_t tma_bar = sb + BAR_OFF, mma_bar = sb + BAR_OFF + 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int L = 32 * quad + lane;  // this thread's TMEM lane
  const int H = p.H, T = p.T;

  if (warp == 0) tmem_alloc(sb + TMEMSLOT_OFF, TMEM_COLS);
  if (tid == 0) {
    mbar_init(tma_bar, 1);
    mbar_init(mma_bar, 1);
    *sAbort = 0u;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + TMEMSLOT_OFF);
  const uint32_t tq = tmem + ((uint32_t)(32 * quad) << 16);  // lane base of quad
  uint32_t tma_phase = 0, mma_phase = 0;
  // Copies / MMAs issued and not yet seen complete, with the barrier phase
  // parity they will complete (uniform over the CTA).
  bool tma_inflight = false, mma_inflight = false;
  uint32_t tma_pending = 0, mma_pending = 0;

  float S[VT];      // state rows (threads 0..127: key row = tid), fp32
  float u_reg[VT];  // u rows (threads 0..63)
#pragma unroll
  for (int i = 0; i < VT; ++i) S[i] = u_reg[i] = 0.f;

  auto abort_all = [&]() {
    *sAbort = 1u;
    set_status(p.status, KDA_DEVICE_TIMEOUT);
  };

  const uint32_t n_units = total_units(p.runs, p.B, H, p.n_vtiles);
  for (uint32_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit u = decode_unit(p.runs, unit, p.B, T, H, p.n_vtiles);
    const int v0 = u.vt * VT;

    // ---- state entering the run; S^T operand ----
    if (tid < 128) {
      const int c = tid;
#pragma unroll
      for (int i = 0; i < VT; ++i) {
        float s = 0.f;
        if (u.first && p.initial_state)
          s = p.initial_state[(((size_t)u.b * H + u.h) * KD + c) * p.V + v0 + i];
        S[i] = s;
        st_bf16(smem, ST_OFF + op_off(i, c, KD), s);
      }
    }
    float beta_next = 0.f;
    if (tid >= 128 && tid < 192) {
      const int r = tid - 128;
      if (u.start + r < u.end)
        beta_next = p.beta[((size_t)u.b * T + u.start + r) * H + u.h];
    }
    if (tid == 0) {
      const int y = u.b * T + u.start;
      mbar_expect_tx(tma_bar, RAW_TX_BYTES);
      tma_load_2d(sb + RAW_Q, &tm_q, u.h * KD, y, tma_bar);
      tma_load_2d(sb + RAW_K, &tm_k, u.h * KD, y, tma_bar);
      tma_load_2d(sb + RAW_G, &tm_g, u.h * KD, y, tma_bar);
      tma_load_2d(sb + RAW_V, &tm_v, u.h * p.V + v0, y, tma_bar);
    }
    tma_inflight = true;
    tma_pending = tma_phase;

    for (int c0 = u.start; c0 < u.end; c0 += C) {
      const int n = min(C, u.end - c0);
      const bool has_next = c0 + C < u.end;
      const size_t tok0 = (size_t)u.b * T + c0;

      if (tid >= 128 && tid < 192) sBeta[tid - 128] = beta_next;
      if (!mbar_wait(tma_bar, tma_phase)) abort_all();
      else tma_inflight = false;
      tma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;

      // ---- P0: gate cumsum per channel, block decays ----
      if (tid < 128) {
        const int c = tid;
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
          acc += r < n ? sG[r * KD + c] : 0.f;
          sG[r * KD + c] = acc;
        }
        float prev = 0.f;
#pragma unroll
        for (int b = 0; b < kNumSub; ++b) {
          const float e = sG[(b * kSub + kSub - 1) * KD + c];
          sDblk[b * KD + c] = __expf(e - prev);
          prev = e;
        }
      }
      __syncthreads();

      // ---- P1: decay factors and bf16 MMA operands ----
      {
        const int rg = tid >> 4, cg = tid & 15;
        const int r0 = rg * 4, c0c = cg * 8, b = rg >> 2;
        float P[8], E[8], pre[8], suf[8], invD[8], cr1[8], cr2[8], cr3[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = c0c + j;
          P[j] = b > 0 ? sG[(b * kSub - 1) * KD + c] : 0.f;
          E[j] = sG[(b * kSub + kSub - 1) * KD + c];
          // pre = prod_{i<b} D_i, suf = prod_{i>b} D_i, Db = D_b, and the
          // cross factors e^{P_b' - E_b} = prod_{i=b+1}^{b'-1} D_i for
          // b' = b+1 (1), b+2 (D_{b+1}), b+3 (D_{b+1} D_{b+2}).
          float a = 1.f, z = 1.f, Db = 1.f, x2 = 1.f, x3 = 1.f;
#pragma unroll
          for (int i = 0; i < kNumSub; ++i) {
            const float Di = sDblk[i * KD + c];
            if (i < b) a *= Di;
            if (i > b) z *= Di;
            if (i == b) Db = Di;
            if (i == b + 1) { x2 *= Di; x3 *= Di; }
            if (i == b + 2) x3 *= Di;
          }
          pre[j] = a;
          suf[j] = z;
          invD[j] = 1.f / Db;
          cr1[j] = 1.f;
          cr2[j] = x2;
          cr3[j] = x3;
        }
        float kbT[8][4], khT[8][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = r0 + i;
          const bool valid = r < n;
          const float br = sBeta[r];
          float kk[8], qq[8];
          ld_bf16x8(smem + RAW_K + r * 256 + c0c * 2, kk);
          ld_bf16x8(smem + RAW_Q + r * 256 + c0c * 2, qq);
          float xk[8], xq[8], qt[8], yd[8], y1[8], y2[8], y3[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float kv = valid ? kk[j] : 0.f;
            const float qv = valid ? qq[j] : 0.f;
            const float G = sG[r * KD + c0c + j];
            const float e1 = __expf(G - P[j]);
            const float e2 = __expf(E[j] - G);
            xk[j] = kv * e1;
            xq[j] = qv * e1;
            qt[j] = xq[j] * pre[j];
            kbT[j][i] = br * xk[j] * pre[j];
            const float ke2 = kv * e2;
            khT[j][i] = ke2 * suf[j];
            yd[j] = ke2 * invD[j];
            y1[j] = ke2 * cr1[j];
            y2[j] = ke2 * cr2[j];
            y3[j] = ke2 * cr3[j];
          }
          st_bf16x8(smem, X_OFF + op_off(r, c0c, KD), xk);
          st_bf16x8(smem, X_OFF + op_off(64 + r, c0c, KD), xq);
          st_bf16x8(smem, WQ_OFF + op_off(64 + r, c0c, KD), qt);
          st_bf16x8(smem, y_off(b) + op_off(r, c0c, KD), yd);
          if (b + 1 < kNumSub) st_bf16x8(smem, y_off(b + 1) + op_off(r, c0c, KD), y1);
          if (b + 2 < kNumSub) st_bf16x8(smem, y_off(b + 2) + op_off(r, c0c, KD), y2);
          if (b + 3 < kNumSub) st_bf16x8(smem, y_off(b + 3) + op_off(r, c0c, KD), y3);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = c0c + j;
          uint2 w;
          w.x = pack_bf16(kbT[j][0], kbT[j][1]);
          w.y = pack_bf16(kbT[j][2], kbT[j][3]);
          *reinterpret_cast<uint2 *>(smem + RHST_OFF + op_off(c, r0, C)) = w;
          w.x = pack_bf16(khT[j][0], khT[j][1]);
          w.y = pack_bf16(khT[j][2], khT[j][3]);
          *reinterpret_cast<uint2 *>(smem + KHT_OFF + op_off(c, r0, C)) = w;
        }
        // beta V^T rows 128..159 of the TX B operand
        {
          const int v = tid & 31, rr0 = (tid >> 5) * 8;
          float vals[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = rr0 + i;
            const float vv = __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16 *>(smem + RAW_V + r * 64 + v * 2));
            vals[i] = r < n ? sBeta[r] * vv : 0.f;
          }
          st_bf16x8(smem, RHST_OFF + op_off(128 + v, rr0, C), vals);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- P2: intra-chunk products on the tensor cores; next TMA ----
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < kNumSub; ++b)
          mma_group(tmem + tm_a(b), sb + X_OFF, sb + y_off(b), KD, 16 * (b + 1), false);
        mma_commit(mma_bar);
        if (has_next) {
          const int y = (int)(tok0 + C);
          mbar_expect_tx(tma_bar, RAW_TX_BYTES);
          tma_load_2d(sb + RAW_Q, &tm_q, u.h * KD, y, tma_bar);
          tma_load_2d(sb + RAW_K, &tm_k, u.h * KD, y, tma_bar);
          tma_load_2d(sb + RAW_G, &tm_g, u.h * KD, y, tma_bar);
          tma_load_2d(sb + RAW_V, &tm_v, u.h * p.V + v0, y, tma_bar);
        }
      }
      if (has_next) {
        tma_inflight = true;
        tma_pending = tma_phase;
      }
      if (tid >= 128 && tid < 192) {
        const int r = tid - 128;
        beta_next = (has_next && c0 + C + r < u.end)
                        ? p.beta[(tok0 + C + r) * H + u.h] : 0.f;
      }
      mma_inflight = true;
      mma_pending = mma_phase;
      if (!mbar_wait(mma_bar, mma_phase)) abort_all();
      else mma_inflight = false;
      mma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;
      tc_fence_after();

      // ---- P3: A_kk (fp32, beta, strict) and A_qk (bf16, inclusive) ----
      {
        const int r = L & 63;
        const bool is_q = L >= 64;
        const int bme = r >> 4;
        const int np = piece_count(quad);
        for (int pi = half; pi < np; pi += 2) {
          int bb, pp;
          piece(quad, pi, bb, pp);
          float v[16];
          tmem_ld16(tq + tm_a(bb) + 16 * pp, v);
          if (bb == bme) {
            if (!is_q) {
              const float br = sBeta[r];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int j = 16 * pp + i;
                sAkk[r * LDF + j] = j < r ? br * v[i] : 0.f;
              }
            } else {
              float a0[8], a1[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                a0[i] = (16 * pp + i <= r) ? v[i] : 0.f;
                a1[i] = (16 * pp + 8 + i <= r) ? v[8 + i] : 0.f;
              }
              st_bf16x8(smem, TAQ_OFF + op_off(64 + r, 16 * pp, C), a0);
              st_bf16x8(smem, TAQ_OFF + op_off(64 + r, 16 * pp + 8, C), a1);
            }
          }
        }
        if (is_q && half == 0) {
          const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int jj = 16 * (bme + 1); jj < C; jj += 8)
            st_bf16x8(smem, TAQ_OFF + op_off(64 + r, jj, C), z);
        }
      }
      tc_fence_before();
      __syncthreads();

      // ---- P4: T = (I + L)^-1, blocked, fp32 ----
      if (tid < 64) {  // diagonal 16 x 16 blocks by forward substitution
        const int i = tid >> 4, cc = tid & 15, base = 16 * i;
        float x[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          float acc = rr == cc ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < rr; ++m)
            acc = fmaf(-sAkk[(base + rr) * LDF + base + m], x[m], acc);
          x[rr] = rr < cc ? 0.f : acc;
          sT[(base + rr) * LDF + base + cc] = x[rr];
        }
      }
      __syncthreads();
      for (int d = 1; d < kNumSub; ++d) {
        const int nblk = kNumSub - d;
        // M_ij = sum_{m=j}^{i-1} L_im T_mj for blocks (i, j = i - d)
        for (int o = tid; o < nblk * 256; o += kThreads) {
          const int blk = o >> 8, e = o & 255, rr = e >> 4, cc = e & 15;
          const int i = d + blk, j = blk;
          float acc = 0.f;
          for (int m = j; m < i; ++m)
#pragma unroll
            for (int t = 0; t < 16; ++t)
              acc = fmaf(sAkk[(16 * i + rr) * LDF + 16 * m + t],
                         sT[(16 * m + t) * LDF + 16 * j + cc], acc);
          sScr[o] = acc;
        }
        __syncthreads();
        // T_ij = -T_ii M_ij
        for (int o = tid; o < nblk * 256; o += kThreads) {
          const int blk = o >> 8, e = o & 255, rr = e >> 4, cc = e & 15;
          const int i = d + blk, j = blk;
          float acc = 0.f;
#pragma unroll
          for (int t = 0; t < 16; ++t)
            acc = fmaf(sT[(16 * i + rr) * LDF + 16 * i + t], sScr[(blk << 8) + t * 16 + cc], acc);
          sT[(16 * i + rr) * LDF + 16 * j + cc] = -acc;
        }
        __syncthreads();
      }
      {  // T -> bf16 rows 0..63 of [T ; A_qk]
        const int r = tid >> 2, jq = (tid & 3) * 16;
        float t0[8], t1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int j0 = jq + i, j1 = jq + 8 + i;
          t0[i] = (j0 >> 4) > (r >> 4) ? 0.f : sT[r * LDF + j0];
          t1[i] = (j1 >> 4) > (r >> 4) ? 0.f : sT[r * LDF + j1];
        }
        st_bf16x8(smem, TAQ_OFF + op_off(r, jq, C), t0);
        st_bf16x8(smem, TAQ_OFF + op_off(r, jq + 8, C), t1);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- P5: [w | u] = T [beta K e^G | beta V] ----
      if (tid == 0) {
        tc_fence_after();
        mma_group(tmem + TM_TX, sb + TAQ_OFF, sb + RHST_OFF, C, KD + VT, false);
        mma_commit(mma_bar);
      }
      mma_inflight = true;
      mma_pending = mma_phase;
      if (!mbar_wait(mma_bar, mma_phase)) abort_all();
      else mma_inflight = false;
      mma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;
      tc_fence_after();
      if (quad < 2) {  // TMEM lanes 0..63 = chunk rows
        const int r = L;
        if (half == 0) {
          float v[16];
          tmem_ld16(tq + TM_TX + KD, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) u_reg[i] = v[i];
          tmem_ld16(tq + TM_TX + KD + 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) u_reg[16 + i] = v[i];
        }
        for (int pc = half * 4; pc < half * 4 + 4; ++pc) {
          float v[16];
          tmem_ld16(tq + TM_TX + 16 * pc, v);
          float a0[8], a1[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            a0[i] = v[i];
            a1[i] = v[8 + i];
          }
          st_bf16x8(smem, WQ_OFF + op_off(r, 16 * pc, KD), a0);
          st_bf16x8(smem, WQ_OFF + op_off(r, 16 * pc + 8, KD), a1);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- P6: D1 = [w ; Q e^G] S0 ----
      if (tid == 0) {
        tc_fence_after();
        mma_group(tmem + TM_D1, sb + WQ_OFF, sb + ST_OFF, KD, VT, false);
        mma_commit(mma_bar);
      }
      mma_inflight = true;
      mma_pending = mma_phase;
      if (!mbar_wait(mma_bar, mma_phase)) abort_all();
      else mma_inflight = false;
      mma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;
      tc_fence_after();

      // ---- P7: U = u - w S0 -> U^T (bf16) ----
      if (quad < 2 && half == 0) {
        const int r = L;
#pragma unroll
        for (int h16 = 0; h16 < 2; ++h16) {
          float v[16];
          tmem_ld16(tq + TM_D1 + 16 * h16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st_bf16(smem, UT_OFF + op_off(16 * h16 + i, r, C), u_reg[16 * h16 + i] - v[i]);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- P8: D1 += [T ; A_qk] U ; D2 = (K e^{G_C-G})^T U ----
      if (tid == 0) {
        tc_fence_after();
        mma_group(tmem + TM_D1, sb + TAQ_OFF, sb + UT_OFF, C, VT, true);
        mma_group(tmem + TM_D2, sb + KHT_OFF, sb + UT_OFF, C, VT, false);
        mma_commit(mma_bar);
      }
      mma_inflight = true;
      mma_pending = mma_phase;
      if (!mbar_wait(mma_bar, mma_phase)) abort_all();
      else mma_inflight = false;
      mma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;
      tc_fence_after();

      // ---- P9: o rows, state update, S^T for the next chunk ----
      if (half == 0) {
        if (quad >= 2) {
          const int r = L - 64;
          float o[VT];
#pragma unroll
          for (int h16 = 0; h16 < 2; ++h16) {
            float v[16];
            tmem_ld16(tq + TM_D1 + 16 * h16, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[16 * h16 + i] = p.scale * v[i];
          }
          if (r < n) {
            uint4 *dst = reinterpret_cast<uint4 *>(
                static_cast<__nv_bfloat16 *>(p.o) + ((tok0 + r) * H + u.h) * p.V + v0);
#pragma unroll
            for (int q4 = 0; q4 < VT / 8; ++q4) {
              uint4 w;
              w.x = pack_bf16(o[8 * q4 + 0], o[8 * q4 + 1]);
              w.y = pack_bf16(o[8 * q4 + 2], o[8 * q4 + 3]);
              w.z = pack_bf16(o[8 * q4 + 4], o[8 * q4 + 5]);
              w.w = pack_bf16(o[8 * q4 + 6], o[8 * q4 + 7]);
              dst[q4] = w;
            }
          }
        }
        {
          const int c = L;  // key row
          float gam = 1.f;
#pragma unroll
          for (int i = 0; i < kNumSub; ++i) gam *= sDblk[i * KD + c];
#pragma unroll
          for (int h16 = 0; h16 < 2; ++h16) {
            float v[16];
            tmem_ld16(tq + TM_D2 + 16 * h16, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float s = fmaf(gam, S[16 * h16 + i], v[i]);
              S[16 * h16 + i] = s;
              st_bf16(smem, ST_OFF + op_off(16 * h16 + i, c, KD), s);
            }
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
    }

    if (u.last && p.final_state && tid < 128) {
      float4 *dst = reinterpret_cast<float4 *>(
          p.final_state + (((size_t)u.b * H + u.h) * KD + tid) * p.V + v0);
#pragma unroll
      for (int q4 = 0; q4 < VT / 4; ++q4)
        dst[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
    }
  }

done:
  // On a timeout, give what is still in flight one more bounded wait before
  // the shared memory and TMEM are released.
  if (tma_inflight) mbar_wait(tma_bar, tma_pending);
  if (mma_inflight) mbar_wait(mma_bar, mma_pending);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- host side --------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D view [rows, cols] of a row-major tensor, box [64 rows, box_cols].
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt,
              int esize, uint64_t cols, uint64_t rows, uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)esize};
  const cuuint32_t box[2] = {box_cols, (cuuint32_t)C};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fwd_tc_supported(int K, int V, bool bf16, int v_tile) {
  return bf16 && K == KD && V == 128 && (v_tile == 0 || v_tile == VT);
}

cudaError_t launch_fwd_tc(const FwdParams &p_in, cudaStream_t stream) {
  if (!fwd_tc_supported(p_in.K, p_in.V, true, p_in.v_tile)) return cudaErrorNotSupported;
  FwdParams p = p_in;
  p.v_tile = VT;
  p.n_vtiles = p.V / VT;
  const uint64_t rows = (uint64_t)p.B * p.T;
  CUtensorMap mq, mk, mg, mv;
  if (!make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * p.K, rows, KD) ||
      !make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * p.K, rows, KD) ||
      !make_map(&mg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)p.H * p.K, rows, KD) ||
      !make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * p.V, rows, VT))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(
      fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long cap = num_sms();
  long units = p.runs.runs ? (long)p.B * p.T * p.H * p.n_vtiles
                           : (long)p.B * p.H * p.n_vtiles;
  const int grid = (int)(units < cap ? units : cap);
  fwd_tc_kernel<<<grid > 0 ? grid : 1, kThreads, SMEM_ALLOC, stream>>>(p, mq, mk, mg, mv);
  return cudaGetLastError();
}

}  // namespace kda
