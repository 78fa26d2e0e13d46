// bwd_bf16.cu -- exact-attention backward by recomputation, bf16 on sm_103a.
//
// Only O and one statistic per row (LSE = m + ln l) are kept from the
// forward pass; P is recomputed tile by tile from Q, K and LSE
// ("03. FlashAttention", "Backward pass"; "FlashAttention ontleed",
// "Geheugencomplexiteit: van O(N^2) naar O(N)"; Lensa ML "FlashAttention",
// step 5: the backward pass recomputes S from Q and K).  The gradient itself
// is the softmax chain rule:
//   P = exp(scale Q K^T - LSE),  D_i = sum_k dO_ik O_ik,
//   dV = P^T dO,  dS = P * (dO V^T - D),  dK = scale dS^T Q,  dQ = scale dS K.
//
// Three kernels:
//   bwd_pre      -scale D = -scale rowsum(dO * O) and -LSE * log2(e), padded per head
//                to a multiple of 128 rows (so every block copy is aligned
//                and in bounds), and zeroing of the fp32 dQ accumulator.
//   bwd_main     one thread block per (b, h, 128-key block j).  K_j and V_j
//                stay in shared memory; 64-row blocks Q_i, dO_i (with their
//                LSE and D) stream past in a 3-stage TMA ring.  Per block i,
//                in one of two TMEM buffers X = i mod 2:
//                  S^T  = K_j Q_i^T   -> R0_X   (shared-memory operands)
//                  dP^T = V_j dO_i^T  -> R1_X
//                  softmax warps (key row = TMEM lane) form
//                  P^T = exp2(S^T scale log2e - LSE log2e) and
//                  dS^T = scale P^T (dP^T - D) (the softmax scale folded in
//                  here, so dQ and dK need no later multiply), write both as
//                  packed bf16 over the
//                  R0_X columns they were computed from, and dS^T also to
//                  shared memory (double-buffered);
//                  dQ_i^T = K_j^T dS^T -> R1_X    (both operands MN-major)
//                  dV += P^T dO_i, dK += dS^T Q_i  (A operand from TMEM)
//                Block i's softmax overlaps the products of blocks i-1 and
//                i+1.  Three warps issue the products, each on its own SM
//                sub-partition (S^T/dP^T, dV/dK, dQ^T), so the issue slots
//                that the softmax and writer warps take on one do not stall
//                the others.  Eight writer warps add dQ_i into the fp32
//                accumulator with fp32 atomics (one warp instruction covers
//                one query row's 128 contiguous bytes of its quadrant).  dK
//                and dV leave TMEM once.
//   bwd_convert  dQ = bf16(accumulator).
// Causal: query blocks entirely above the key block are skipped; the blocks
// that straddle the diagonal are masked element-wise.
// Grouped query heads ("FlashAttention ontleed", "Interactie met de
// KV-cache"): a thread block owns key block j of key/value head b*Hkv + t and
// streams the query blocks of all g query heads b*Hq + t*g .. + g-1 past it,
// so dK and dV (sums over the group) stay in TMEM until the end.
// Sliding window ("03. FlashAttention", "Variantes et extensions"): key k is
// seen by queries k .. k+w-1, so query blocks past the window of the key
// block are skipped and the blocks that cut through its edge are masked.
// ALiBi (same section): the recomputed P includes the bias -slope_h |i - j|
// (LSE from the forward already does); dS, dQ, dK and dV keep their form.
#include <cfloat>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ int g_status_bwd;

constexpr int HD = 128;
constexpr int BKV = 128;                  // key rows per block (TMEM lanes)
constexpr int BQ = 64;                    // query rows per streamed block
constexpr int PAD = 128;                  // per-head padding of the staged LSE / D
constexpr int STAGES = 3;
constexpr uint32_t TILE = 128 * HD * 2;   // K_j or V_j: 32 KiB
constexpr uint32_t HALF = TILE / 2;       // 128 rows x 64 columns
constexpr uint32_t QTILE = BQ * HD * 2;   // Q_i or dO_i: 16 KiB
constexpr uint32_t QHALF = QTILE / 2;     // 64 rows x 64 columns
constexpr uint32_t STAT = BQ * 4;         // 256 B of -LSE*log2e or -D per block
constexpr uint32_t DS_TILE = BKV * BQ * 2;                   // dS^T [key][query]: 16 KiB

constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + TILE;
constexpr uint32_t OFF_STAGE = OFF_V + TILE;
constexpr uint32_t ST_Q = 0, ST_DO = QTILE, ST_LSE = 2 * QTILE, ST_D = 2 * QTILE + STAT;
constexpr uint32_t STAGE_BYTES = 2 * QTILE + 2048;           // 1024-aligned stages
constexpr uint32_t OFF_DS = OFF_STAGE + STAGES * STAGE_BYTES; // 2 buffers
constexpr uint32_t OFF_BAR = OFF_DS + 2 * DS_TILE;
constexpr int B_KVFULL = 0;
constexpr int B_QFULL = 1;                 // + stage
constexpr int B_QEMPTY = B_QFULL + STAGES; // + stage
constexpr int B_SFULL = B_QEMPTY + STAGES; // + buffer: S^T in TMEM
constexpr int B_DPFULL = B_SFULL + 2;      // + buffer: dP^T in TMEM
constexpr int B_PFULL = B_DPFULL + 2;      // + buffer: P^T, dS^T written (8 warps)
constexpr int B_DQFULL = B_PFULL + 2;      // + buffer
constexpr int B_DQFREE = B_DQFULL + 2;     // + buffer: 8 writer warps read dQ^T
constexpr int B_DKV = B_DQFREE + 2;       // + buffer: dV/dK(i) have read R0_X
constexpr int B_DONE = B_DKV + 2;          // the dV/dK issuer's products completed
constexpr int B_DONE3 = B_DONE + 1;        // dQ issuer's products completed
constexpr int B_EPI = B_DONE3 + 1;          // + (0 dV, 1 dK): staged in shared memory (4 warps)
constexpr int NBAR = B_EPI + 2;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;   // base is 1024-aligned (checked)

constexpr uint32_t TMEM_COLS = 512;
// buffer X: R0 = [128 X, 128 X + 64), R1 = [128 X + 64, 128 X + 128)
constexpr uint32_t TM_DV = 256, TM_DK = 384;

// Warps: 0-7 softmax, then the dQ writers (eight, two per TMEM lane quadrant
// and 32 queries each, when this kernel forms dQ; none otherwise), then the
// producer and the MMA issuers (dV/dK, S^T/dP^T, dQ^T), which land on SM
// sub-partitions 0, 1, 2, 3 either way.  The fp32 reductions of dQ are
// bound by how many a warp keeps in flight (measured on this GPU: ~11 B/clk
// per SM with four warps issuing them, ~18 with eight).
template <bool kDq>
__host__ __device__ constexpr int bwd_writers() { return kDq ? 8 : 0; }
template <bool kDq>
__host__ __device__ constexpr int bwd_threads() { return 32 * (12 + bwd_writers<kDq>()); }
// Key/value heads whose thread blocks are ordered together: 8, fewer when
// the query rows they serve (Q, dO and the fp32 dQ accumulator: 1 KiB per
// row, g query heads per key/value head) pass ~128 MB of L2.
constexpr int kHeadGroupKv = 8;
constexpr long long kHeadGroupBytes = 128ll << 20;
// The deterministic dQ kernel's groups: key/value heads whose K and V fit here.
constexpr long long kDqGroupBytes = 32ll << 20;
constexpr float kLog2e = 1.4426950408889634f;

// S^T = K_j Q_i^T and dP^T = V_j dO_i^T: M = 128 keys, N = 64 queries.
constexpr uint32_t IDESC_ST = idesc_bf16(BKV, BQ, false, false);
// dV += P^T dO_i, dK += dS^T Q_i: A in TMEM, B MN-major; M = 128 keys, N = d.
constexpr uint32_t IDESC_DKV = idesc_bf16(BKV, HD, false, true);
// dQ_i^T = K_j^T dS^T: M = d, N = 64 queries; both operands MN-major.
constexpr uint32_t IDESC_DQ = idesc_bf16(HD, BQ, true, true);

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) {
  return base + OFF_BAR + 8u * static_cast<uint32_t>(i);
}

// One fp32 value added atomically (the result is not needed).
__device__ __forceinline__ void red_add(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

struct Ctx {
  uint32_t sbase;
  volatile int* abort;
  __device__ bool wait(int bar, uint32_t parity) const {
    return mbar_wait(bar_addr(sbase, bar), parity, abort, &g_status_bwd);
  }
};

// ------------------------------------------------------------------ bwd_pre
// Sixteen threads per (padded) row, 16 bytes each: -scale D = -scale sum_k dO_k O_k and
// -LSE * log2(e), zero past the end of the sequence; the row of the dQ
// accumulator is zeroed too.  The padded row count is a multiple of 128, so
// every warp covers two whole rows and every shuffle has all 32 lanes.
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ d_pad, float scale,
                                                      float* __restrict__ lse_pad,
                                                      float* __restrict__ dq_acc, int N,
                                                      int Npad, size_t padded_rows) {
  const size_t prow = static_cast<size_t>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int sub = threadIdx.x & 15;
  if (prow >= padded_rows) return;
  const size_t bh = prow / Npad;
  const int n = static_cast<int>(prow % Npad);
  const bool valid = n < N;
  const size_t row = bh * N + n;
  float s = 0.f;
  if (valid) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * HD + sub * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(dO + row * HD + sub * 8);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fmaf(__uint_as_float(aw[i] << 16), __uint_as_float(bw[i] << 16), s);
      s = fmaf(__uint_as_float(aw[i] & 0xffff0000u), __uint_as_float(bw[i] & 0xffff0000u), s);
    }
    if (dq_acc != nullptr) {
      float4* z = reinterpret_cast<float4*>(dq_acc + row * HD + sub * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (sub == 0) {            // stored negated: the main kernel only adds them
    d_pad[prow] = -s * scale;
    lse_pad[prow] = valid ? -lse[row] * kLog2e : 0.f;
  }
}

// --------------------------------------------------------------- bwd_convert
// Eight accumulator values per thread -> one 16-byte bf16 store.
__global__ void __launch_bounds__(256) bwd_convert_kernel(const float* __restrict__ dq_acc,
                                                          __nv_bfloat16* __restrict__ dq,
                                                          size_t n8) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
  reinterpret_cast<uint4*>(dq)[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                               pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
}

// ------------------------------------------------------------------ bwd_main
// kAlibi: alibi[h] is the ALiBi slope of query head h (h = b*Hq + h' taken
// modulo heads).  kDq: this kernel also forms dQ (fp32 atomics into dq_acc);
// without it only dK and dV are made and dQ is left to bwd_dq_kernel.
template <bool kAlibi, bool kDq>
__global__ void __launch_bounds__(bwd_threads<kDq>(), 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                const float* __restrict__ lse_pad, const float* __restrict__ d_pad,
                float* __restrict__ dq_acc, int BHkv, int N, int Npad, float scale,
                int causal, int qgroup, int window, int head_group,
                const float* __restrict__ alibi, int heads) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {           // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicExch(&g_status_bwd, kStatusLayout);
    return;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const Ctx ctx{sbase, abort_flag};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int WARP_TMA = 8 + bwd_writers<kDq>();
  constexpr int WARP_MMA = WARP_TMA + 1;    // dV/dK
  constexpr int WARP_MMA2 = WARP_TMA + 2;   // S^T/dP^T
  constexpr int WARP_MMA3 = WARP_TMA + 3;   // dQ^T
  // Blocks are ordered by groups of head_group key/value heads, so the few
  // heads in flight keep their dQ accumulator, Q and dO resident in L2;
  // within a group, key blocks go in increasing order (most work first when
  // causal).
  const int nqb = (N + BQ - 1) / BQ;
  const int nkv = (N + BKV - 1) / BKV;
  const int per_group = head_group * nkv;
  const int hgrp = static_cast<int>(blockIdx.x) / per_group;
  const int gsize = min(head_group, BHkv - hgrp * head_group);
  const int rem = static_cast<int>(blockIdx.x) - hgrp * per_group;
  const int j = rem / gsize;                          // key block
  const int bkv = hgrp * head_group + rem % gsize;    // key/value head
  const int i0 = causal ? (j * BKV) / BQ : 0;         // first query block that sees key block j
  // last query block that sees key block j (window: key k is seen up to k+w-1)
  const int i1 = window > 0 ? min(nqb - 1, (j * BKV + BKV - 1 + window - 1) / BQ) : nqb - 1;
  const int nph = i1 - i0 + 1;                        // query blocks per query head
  const int nit = qgroup * nph;                       // over the g query heads of the group
  // Iteration order: query blocks i0..i1 of query head bkv*g, then of the
  // next head of the group, and so on; each loop walks it with a cursor.
  struct Cursor {
    int qi, hq;
    __device__ void next(int lo, int hi) {
      if (++qi > hi) {
        qi = lo;
        ++hq;
      }
    }
  };
  const Cursor first{i0, bkv * qgroup};
  const float scale_log2 = scale * kLog2e;

  if (threadIdx.x == 0) {
    mbar_init(bar_addr(sbase, B_KVFULL), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_addr(sbase, B_QFULL + s), 1);
      mbar_init(bar_addr(sbase, B_QEMPTY + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar_addr(sbase, B_SFULL + x), 1);
      mbar_init(bar_addr(sbase, B_DPFULL + x), 1);
      mbar_init(bar_addr(sbase, B_PFULL + x), 8);
      mbar_init(bar_addr(sbase, B_DQFULL + x), 1);
      mbar_init(bar_addr(sbase, B_DQFREE + x), 8);
      mbar_init(bar_addr(sbase, B_DKV + x), 1);
    }
    mbar_init(bar_addr(sbase, B_DONE), 1);
    mbar_init(bar_addr(sbase, B_DONE3), 1);
    mbar_init(bar_addr(sbase, B_EPI + 0), 4);
    mbar_init(bar_addr(sbase, B_EPI + 1), 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == WARP_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
      prefetch_tmap(&tmdK);
      prefetch_tmap(&tmdV);
      const uint32_t kvf = bar_addr(sbase, B_KVFULL);
      mbar_arrive_expect_tx(kvf, 2 * TILE);
      tma_load_3d(sbase + OFF_K, &tmK, kvf, 0, j * BKV, bkv);
      tma_load_3d(sbase + OFF_K + HALF, &tmK, kvf, 64, j * BKV, bkv);
      tma_load_3d(sbase + OFF_V, &tmV, kvf, 0, j * BKV, bkv);
      tma_load_3d(sbase + OFF_V + HALF, &tmV, kvf, 64, j * BKV, bkv);
      Cursor cur = first;
      for (int it = 0; it < nit; ++it, cur.next(i0, i1)) {
        const int st = it % STAGES;
        const int qb = cur.qi * BQ;
        const int bh = cur.hq;
        if (it >= STAGES && !ctx.wait(B_QEMPTY + st, ((it / STAGES) - 1) & 1)) break;
        const uint32_t qf = bar_addr(sbase, B_QFULL + st);
        const uint32_t sb = sbase + OFF_STAGE + st * STAGE_BYTES;
        mbar_arrive_expect_tx(qf, 2 * QTILE + 2 * STAT);
        tma_load_3d(sb + ST_Q, &tmQ, qf, 0, qb, bh);
        tma_load_3d(sb + ST_Q + QHALF, &tmQ, qf, 64, qb, bh);
        tma_load_3d(sb + ST_DO, &tmdO, qf, 0, qb, bh);
        tma_load_3d(sb + ST_DO + QHALF, &tmdO, qf, 64, qb, bh);
        const size_t srow = static_cast<size_t>(bh) * Npad + qb;
        bulk_load(sb + ST_LSE, lse_pad + srow, STAT, qf);
        bulk_load(sb + ST_D, d_pad + srow, STAT, qf);
      }
    }
    __syncwarp();
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------- gradient issuer
    // Per query block i in buffer X = i mod 2, once its softmax is done:
    //   dV(i) dK(i) [DKV(X): R0_X read]
    // The score products and dQ^T come from two more issuing warps, each on
    // its own SM sub-partition: one thread issuing every product shares its
    // sub-partition's issue slots with the softmax and writer warps there,
    // and loses most of its rate while they are busy.
    if (lane == 0) {
      auto stage = [&](int it) { return sbase + OFF_STAGE + (it % STAGES) * STAGE_BYTES; };
      bool ok = ctx.wait(B_KVFULL, 0);
      for (int it = 0; it < nit && ok; ++it) {
        const int x = it & 1;
        const uint32_t sb = stage(it);
        const uint32_t r0 = tmem + 128u * x;
        if (!(ok = ctx.wait(B_PFULL + x, (it >> 1) & 1))) break;
        tc_fence_after();
        // dV += P^T dO_i, dK += dS^T Q_i.  R0_X holds, per 32-query slice g,
        // P^T packed in columns [32g, 32g+16) and dS^T in [32g+16, 32g+32);
        // 16 queries = 8 packed columns.
        {
          const uint64_t dod = sdesc_sw128(sb + ST_DO, QHALF, 1024);   // dO_i, MN-major
          const uint64_t qd = sdesc_sw128(sb + ST_Q, QHALF, 1024);     // Q_i, MN-major
          uint32_t ap[4], as[4];
          uint64_t bo[4], bq[4];
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            ap[kk] = r0 + 32 * (kk >> 1) + 8 * (kk & 1);
            as[kk] = ap[kk] + 16;
            bo[kk] = dod + ((kk * 2048) >> 4);
            bq[kk] = qd + ((kk * 2048) >> 4);
          }
          const uint32_t acc = it > 0 ? 1u : 0u;
          mma_ts_batch4(tmem + TM_DV, ap, bo, IDESC_DKV, acc);
          mma_ts_batch4(tmem + TM_DK, as, bq, IDESC_DKV, acc);
        }
        mma_commit(bar_addr(sbase, B_DKV + x));
        mma_commit(bar_addr(sbase, B_QEMPTY + it % STAGES));
        // With the ALiBi bias the softmax warps are busier and a third
        // issuer beside them measured slower: dQ^T comes from here then.
        if constexpr (kDq && kAlibi) {
          const uint64_t kd_mn = sdesc_sw128(sbase + OFF_K, HALF, 1024);   // K_j^T, MN-major
          const uint64_t dsd = sdesc_sw128(sbase + OFF_DS + x * DS_TILE, DS_TILE, 1024);
          uint64_t a[8], b[8];
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk) {
            a[kk] = kd_mn + ((kk * 2048) >> 4);
            b[kk] = dsd + ((kk * 2048) >> 4);
          }
          mma_ss_batch8(tmem + 128u * x + 64u, a, b, IDESC_DQ, 0u);
          mma_commit(bar_addr(sbase, B_DQFULL + x));
        }
      }
      // The score products all completed before the last softmax, so this
      // commit covers every product but dQ^T (B_DONE3).
      if (ok) mma_commit(bar_addr(sbase, B_DONE));
    }
    __syncwarp();
  } else if (kDq && !kAlibi && warp == WARP_MMA3) {
    // ------------------------------------------------------------ dQ issuer
    // dQ_i^T = K_j^T dS^T (reduction over the 128 keys) into R1_X, whose
    // dP^T(i) the softmax has read, once P(i) is ready.
    if (lane == 0) {
      const uint64_t kd_mn = sdesc_sw128(sbase + OFF_K, HALF, 1024);   // K_j^T, MN-major
      bool ok = ctx.wait(B_KVFULL, 0);
      for (int it = 0; it < nit && ok; ++it) {
        const int x = it & 1;
        if (!(ok = ctx.wait(B_PFULL + x, (it >> 1) & 1))) break;
        tc_fence_after();
        const uint64_t dsd = sdesc_sw128(sbase + OFF_DS + x * DS_TILE, DS_TILE, 1024);
        uint64_t a[8], b[8];
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          a[kk] = kd_mn + ((kk * 2048) >> 4);
          b[kk] = dsd + ((kk * 2048) >> 4);
        }
        mma_ss_batch8(tmem + 128u * x + 64u, a, b, IDESC_DQ, 0u);
        mma_commit(bar_addr(sbase, B_DQFULL + x));
      }
      if (ok) mma_commit(bar_addr(sbase, B_DONE3));
    }
    __syncwarp();
  } else if (warp == WARP_MMA2) {
    // ---------------------------------------------------------- score issuer
    // S^T(i) and dP^T(i) into buffer X = i mod 2, for i = 0, 1 at once and
    // then i + 2: S^T as soon as dV/dK(i) have read R0_X (DKV), dP^T once
    // the writers have drained dQ^T(i) from R1_X (DQFREE).  Each has its own
    // barrier, so the softmax takes the exponentials while dP^T is still on
    // its way.
    if (lane == 0) {
      const uint32_t kA = sbase + OFF_K, vA = sbase + OFF_V;
      auto stage = [&](int it) { return sbase + OFF_STAGE + (it % STAGES) * STAGE_BYTES; };
      // Descriptors of the key-block operands, fixed for the whole block; a
      // k-step advances the start-address field (units of 16 bytes).
      const uint64_t kd_k = sdesc_sw128(kA, 16, 1024);        // K_j, K-major (S^T)
      const uint64_t vd_k = sdesc_sw128(vA, 16, 1024);        // V_j, K-major (dP^T)
      // S^T (into R0) or dP^T (into R1): reduction over d.
      auto issue_sdp = [&](int it, bool dp) {
        const uint64_t ad = dp ? vd_k : kd_k;
        const uint64_t bd = sdesc_sw128(stage(it) + (dp ? ST_DO : ST_Q), 16, 1024);
        uint64_t a[8], b[8];
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          a[kk] = ad + (((kk >> 2) * HALF + (kk & 3) * 32) >> 4);
          b[kk] = bd + (((kk >> 2) * QHALF + (kk & 3) * 32) >> 4);
        }
        mma_ss_batch8(tmem + 128u * (it & 1) + (dp ? 64u : 0u), a, b, IDESC_ST, 0u);
      };
      auto wait_q = [&](int it) {
        return ctx.wait(B_QFULL + it % STAGES, (it / STAGES) & 1);
      };
      bool ok = ctx.wait(B_KVFULL, 0);
      for (int it = 0; it < 2 && it < nit && ok; ++it) {
        if (!(ok = wait_q(it))) break;
        tc_fence_after();
        issue_sdp(it, false);
        mma_commit(bar_addr(sbase, B_SFULL + (it & 1)));
        issue_sdp(it, true);
        mma_commit(bar_addr(sbase, B_DPFULL + (it & 1)));
      }
      for (int it = 0; it + 2 < nit && ok; ++it) {
        const int x = it & 1;
        if (!(ok = ctx.wait(B_DKV + x, (it >> 1) & 1) && wait_q(it + 2))) break;
        tc_fence_after();
        issue_sdp(it + 2, false);
        mma_commit(bar_addr(sbase, B_SFULL + x));
        if constexpr (kDq) {
          if (!(ok = ctx.wait(B_DQFREE + x, (it >> 1) & 1))) break;
          tc_fence_after();
        }
        issue_sdp(it + 2, true);
        mma_commit(bar_addr(sbase, B_DPFULL + x));
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    // Warp w takes the rows of TMEM lane quadrant w & 3 and the 32-query
    // slice w >> 2 of each 64-query block.
    const int sub = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;                 // key row within block j
    const int kv = j * BKV + row;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const int qlo = causal ? kv : 0;
    const int qhi = window > 0 ? min(N - 1, kv + window - 1) : N - 1;
    const uint32_t qspan = kv < N ? static_cast<uint32_t>(qhi - qlo) : 0u;
    const bool row_valid = kv < N;
    bool ok = true;
    Cursor cur = first;
    for (int it = 0; it < nit; ++it, cur.next(i0, i1)) {
      const int x = it & 1;
      const int st = it % STAGES;
      const int qb = cur.qi * BQ;
      const float slope_log2 = kAlibi ? alibi[cur.hq % heads] * kLog2e : 0.f;
      const float d0 = static_cast<float>(qb + sub * 32 - kv);   // query - key at column 0
      const float* stage_lse =
          reinterpret_cast<const float*>(smem + OFF_STAGE + st * STAGE_BYTES + ST_LSE);
      const float* stage_d =
          reinterpret_cast<const float*>(smem + OFF_STAGE + st * STAGE_BYTES + ST_D);
      // QFULL: the staged LSE / D are visible here; SFULL: S^T in TMEM.
      if (!ctx.wait(B_QFULL + st, (it / STAGES) & 1) ||
          !ctx.wait(B_SFULL + x, (it >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Valid queries for this key row: q in [qlo, qhi] (causal: q >= kv;
      // window: q <= kv + w - 1; past the end of the sequence nothing is
      // valid).  Only blocks on the diagonal, on the window's edge or at a
      // ragged end need it; the test is block-uniform.
      const bool need_mask = (causal && qb < j * BKV + BKV) || (qb + BQ > N) ||
                             (j * BKV + BKV > N) || (window > 0 && qb + BQ > j * BKV + window);
      const int col0 = sub * 32;                      // first query column of this slice
      const uint32_t s_addr = tmem + lane_addr + 128u * x + col0;
      float p[32];
      {
        uint32_t sr[32], pk[16];
        tmem_ld32(s_addr, sr);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          // staged per query: -LSE*log2e (one broadcast 16-byte load)
          float4 l4 = *reinterpret_cast<const float4*>(stage_lse + col0 + e);
          if constexpr (kAlibi) {
            // exponent offset -LSE log2e - slope |i - j| log2e per query column
            if (causal) {
              // every key the mask leaves has key <= query, so |i - j| = i - j:
              // no absolute value, and the offsets on packed pairs
              const uint64_t ns2 = f2pack(-slope_log2, -slope_log2);
              const uint64_t d02 = f2pack(d0, d0);
              const uint64_t de01 = f2add(d02, f2pack(static_cast<float>(e), static_cast<float>(e + 1)));
              const uint64_t de23 = f2add(d02, f2pack(static_cast<float>(e + 2), static_cast<float>(e + 3)));
              f2unpack(f2fma(ns2, de01, f2pack(l4.x, l4.y)), l4.x, l4.y);
              f2unpack(f2fma(ns2, de23, f2pack(l4.z, l4.w)), l4.z, l4.w);
            } else {
              const float de = d0 + static_cast<float>(e);
              l4.x = fmaf(-slope_log2, fabsf(de), l4.x);
              l4.y = fmaf(-slope_log2, fabsf(de + 1.f), l4.y);
              l4.z = fmaf(-slope_log2, fabsf(de + 2.f), l4.z);
              l4.w = fmaf(-slope_log2, fabsf(de + 3.f), l4.w);
            }
          }
          // exponent arguments on packed fp32 pairs
          const uint64_t sc2 = f2pack(scale_log2, scale_log2);
          float a0, a1, a2, a3;
          f2unpack(f2fma(f2pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sc2,
                         f2pack(l4.x, l4.y)), a0, a1);
          f2unpack(f2fma(f2pack(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), sc2,
                         f2pack(l4.z, l4.w)), a2, a3);
          float p0 = fast_exp2(a0), p1 = fast_exp2(a1), p2 = fast_exp2(a2), p3 = fast_exp2(a3);
          if (need_mask) {
            // qlo <= q <= qhi as one unsigned compare per query (the
            // wrap-around of rel + t is the exact difference mod 2^32)
            const uint32_t rel = static_cast<uint32_t>(qb + col0 + e - qlo);
            p0 = (row_valid && rel <= qspan) ? p0 : 0.f;
            p1 = (row_valid && rel + 1 <= qspan) ? p1 : 0.f;
            p2 = (row_valid && rel + 2 <= qspan) ? p2 : 0.f;
            p3 = (row_valid && rel + 3 <= qspan) ? p3 : 0.f;
          }
          p[e] = p0; p[e + 1] = p1; p[e + 2] = p2; p[e + 3] = p3;
          pk[e / 2] = pack_bf16x2(p0, p1);
          pk[e / 2 + 1] = pack_bf16x2(p2, p3);
        }
        // Packed P^T over the first 16 of the 32 columns this thread has just
        // read (no other warp reads them); dS^T takes the other 16.
        tmem_st16(s_addr, pk);
      }
      // DPFULL: dP^T in TMEM.  It is committed after dQ^T(i-2), the last
      // reader of this block's dS^T shared buffer, so the buffer is free too.
      if (!ctx.wait(B_DPFULL + x, (it >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t gk[16];
      {
        uint32_t dr[32];
        tmem_ld32(s_addr + 64, dr);
        const uint64_t s2 = f2pack(scale, scale);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          // staged per query: -scale D (one broadcast 16-byte load);
          // scale dS = P (scale dP - scale D) on packed fp32 pairs
          const float4 d4 = *reinterpret_cast<const float4*>(stage_d + col0 + e);
          float g0, g1, g2, g3;
          f2unpack(f2mul(f2pack(p[e], p[e + 1]),
                         f2fma(f2pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), s2,
                               f2pack(d4.x, d4.y))), g0, g1);
          f2unpack(f2mul(f2pack(p[e + 2], p[e + 3]),
                         f2fma(f2pack(__uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3])), s2,
                               f2pack(d4.z, d4.w))), g2, g3);
          gk[e / 2] = pack_bf16x2(g0, g1);
          gk[e / 2 + 1] = pack_bf16x2(g2, g3);
        }
      }
      tmem_st16(s_addr + 16, gk);
      // dS^T row into this block's shared buffer (MN-major operand of dQ^T).
      if constexpr (kDq) {
        uint8_t* ds_smem = smem + OFF_DS + x * DS_TILE;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint32_t off = sw128_offset(row, sub * 4 + ch);
          *reinterpret_cast<uint4*>(ds_smem + off) =
              make_uint4(gk[4 * ch], gk[4 * ch + 1], gk[4 * ch + 2], gk[4 * ch + 3]);
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_PFULL + x));
    }
    // dV (warps 0-3) and dK (warps 4-7) leave TMEM once, after every
    // product.  K_j and V_j are no longer read then, so each gradient is
    // staged over the tile it belongs to (dV over V_j, dK over K_j) in the
    // same swizzled boxes and leaves with one bulk tensor store, which also
    // drops the rows past N.
    if (ok && nit > 0 && ctx.wait(B_DONE, 0) && (!kDq || kAlibi || ctx.wait(B_DONE3, 0))) {
      tc_fence_after();
      const uint32_t src = tmem + lane_addr + (sub == 0 ? TM_DV : TM_DK);
      const uint32_t stage = sub == 0 ? OFF_V : OFF_K;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(src + c * 32, r);
        uint8_t* box = smem + stage + (c >> 1) * HALF;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(box + sw128_offset(row, (c & 1) * 4 + i)) = make_uint4(
              pack_bf16x2(__uint_as_float(r[8 * i]), __uint_as_float(r[8 * i + 1])),
              pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
              pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
              pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_EPI + sub));
      if (quad == 0 && lane == 0 && ctx.wait(B_EPI + sub, 0)) {
        const CUtensorMap* map = sub == 0 ? &tmdV : &tmdK;
        tma_store_3d(map, sbase + stage, 0, j * BKV, bkv);
        tma_store_3d(map, sbase + stage + HALF, 64, j * BKV, bkv);
        bulk_commit_group();
        bulk_wait_group_read0();   // the block may exit once the tiles have been read
      }
    }
  } else if (kDq && warp < WARP_TMA) {
    // ------------------------------------------------------------ dQ writers
    const int quad = warp & 3;
    const int wq = (warp - 8) >> 2;                  // query half of this writer
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;   // lane = d index
    Cursor cur = first;
    for (int it = 0; it < nit; ++it, cur.next(i0, i1)) {
      const int x = it & 1;
      const int qb = cur.qi * BQ + 32 * wq;          // first query of this writer's half
      const int bh = cur.hq;
      if (!ctx.wait(B_DQFULL + x, (it >> 1) & 1)) break;
      tc_fence_after();
      float g[32];
      {
        uint32_t r[32];
        tmem_ld32(tmem + lane_addr + 128u * x + 64 + 32 * wq, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_DQFREE + x));
      // Lane = head-dimension entry, so one warp instruction adds a query
      // row's 32 entries of this quadrant: 128 contiguous bytes, no shuffles
      // (fewer issue slots taken beside the MMA-issuing warp than the 4x4
      // register transpose that 16-byte vector atomics need).
      const int lim = min(32, N - qb);
      float* base = dq_acc + (static_cast<size_t>(bh) * N + qb) * HD + quad * 32 + lane;
#pragma unroll
      for (int q = 0; q < 32; ++q)
        if (q < lim) red_add(base + static_cast<size_t>(q) * HD, g[q]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ bwd_dq
// Deterministic dQ (the dQ half of the gradient without atomics): one thread
// block per (query head, 128-query block i), K_j / V_j streamed in 128-key
// tiles in increasing key order, dQ_i accumulated in TMEM and written once:
//   S = Q_i K_j^T, dP = dO_i V_j^T            (Q_i, dO_i from TMEM)
//   P = exp2(S scale log2e - LSE log2e [- ALiBi]),  dS = scale P * (dP - D)
//   dQ_i += dS K_j                             (dS from shared memory, K_j MN-major)
// Q_i and dO_i stay for the whole block, so they are copied into tensor
// memory once and the score products take their A operand from there.  The
// softmax copies S and dP into registers as soon as they land, so a single
// TMEM region each suffices: the next tile's S and dP are computed while the
// softmax still works on this one.  dS goes through shared memory to the dQ
// product.  S, dP and dQ are issued by three warps on three SM
// sub-partitions: an issuing warp beside busy softmax warps gets ~80 cycles
// per tcgen05.mma, so 128-key tiles (half the instructions per FLOP of
// 64-key ones) and one product kind per issuer keep issue off the critical
// path.  Each dQ element is summed by one thread block in a fixed order, so
// the result is the same on every run.
constexpr int DQ_BQ = 128;                     // query rows (TMEM lanes)
constexpr int DQ_BK = 128;                     // keys per tile
constexpr int DQ_STAGES = 3;
constexpr uint32_t DQ_TILE = DQ_BQ * HD * 2;   // Q_i, dO_i, K_j or V_j: 32 KiB
constexpr uint32_t DQ_HALF = DQ_TILE / 2;      // 128 rows x 64 columns (one swizzled box)
constexpr uint32_t DQ_STAGE = 2 * DQ_TILE;     // K_j then V_j
constexpr uint32_t DQ_OFF_RING = 0;
// Q_i and dO_i land in the space of ring stage 2; once they have been copied
// into tensor memory, that space joins the K/V ring.
constexpr uint32_t DQ_OFF_Q = 2 * DQ_STAGE;
constexpr uint32_t DQ_OFF_DO = DQ_OFF_Q + DQ_TILE;
constexpr uint32_t DQ_OFF_DS = DQ_STAGES * DQ_STAGE;   // dS [query][key]: two 64-key boxes
constexpr uint32_t DQ_OFF_BAR = DQ_OFF_DS + DQ_TILE;
constexpr int DQB_QFULL = 0;
constexpr int DQB_FULL = 1;                          // + stage
constexpr int DQB_EMPTY = DQB_FULL + DQ_STAGES;      // + stage
constexpr int DQB_SFULL = DQB_EMPTY + DQ_STAGES;     // S(t) in TMEM
constexpr int DQB_DPFULL = DQB_SFULL + 1;            // dP(t) in TMEM
constexpr int DQB_SREAD = DQB_DPFULL + 1;            // the softmax has S(t) in registers (8 warps)
constexpr int DQB_DPREAD = DQB_SREAD + 1;            // ... and dP(t) (8 warps)
constexpr int DQB_PFULL = DQB_DPREAD + 1;            // dS(t) in shared memory (8 warps)
constexpr int DQB_DSFREE = DQB_PFULL + 1;            // dQ(t) has read dS(t)
constexpr int DQB_DONE = DQB_DSFREE + 1;
constexpr int DQB_QTMEM = DQB_DONE + 1;              // Q_i, dO_i copied to TMEM (8 warps)
constexpr int DQ_NBAR = DQB_QTMEM + 1;
constexpr uint32_t DQ_OFF_MISC = DQ_OFF_BAR + DQ_NBAR * 8;
constexpr uint32_t DQ_SMEM = DQ_OFF_MISC + 16 + 1024;   // + 1024-byte alignment slack
static_assert(DQ_SMEM <= 227u * 1024u, "dQ kernel shared memory exceeds the per-block limit");
// 0-15 softmax (four per row, 32 keys each), 16 producer; MMA issuers 17 dQ,
// 18 S, 19 dP
constexpr int DQ_THREADS = 640;
constexpr int DQ_SOFTMAX_WARPS = 16;
constexpr int DQ_WARP_TMA = 16, DQ_WARP_DQ = 17, DQ_WARP_S = 18, DQ_WARP_DP = 19;
constexpr uint32_t DQ_TM_S = 0;                // S: 128 columns
constexpr uint32_t DQ_TM_DP = 128;             // dP: 128 columns
constexpr uint32_t DQ_TM_DQ = 256;             // dQ accumulator: 128 columns
constexpr uint32_t DQ_TM_Q = 384;              // Q_i packed bf16: 64 columns
constexpr uint32_t DQ_TM_DO = 448;             // dO_i packed bf16: 64 columns
// S, dP: M = 128 queries, N = 128 keys, A in TMEM, B K-major.
constexpr uint32_t IDESC_DQ_S = idesc_bf16(DQ_BQ, DQ_BK, false, false);
// dQ += dS K_j: M = 128 queries, N = d; A = dS K-major, B = K_j MN-major.
constexpr uint32_t IDESC_DQ_ACC = idesc_bf16(DQ_BQ, HD, false, true);

template <bool kAlibi>
__global__ void __launch_bounds__(DQ_THREADS, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const float* __restrict__ lse_pad, const float* __restrict__ d_pad,
              __nv_bfloat16* __restrict__ dQ, int BH, int N, int Npad, float scale, int causal,
              int group, int window, const float* __restrict__ alibi, int heads,
              int head_group) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + DQ_OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + DQ_OFF_MISC + 4);
  auto bar = [&](int i) { return sbase + DQ_OFF_BAR + 8u * static_cast<uint32_t>(i); };
  auto wait = [&](int i, uint32_t parity) {
    return mbar_wait(bar(i), parity, abort_flag, &g_status_bwd);
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Blocks are ordered by groups of head_group query heads (whole key/value
  // heads), so the thread blocks in flight share a few heads' K and V and
  // re-read them from L2, not HBM; within a group, query blocks go
  // heavy-first (the last block sees the most keys when causal).
  const int npb = (N + DQ_BQ - 1) / DQ_BQ;
  const int per_group = head_group * npb;
  const int hgrp = static_cast<int>(blockIdx.x) / per_group;
  const int gsize = min(head_group, BH - hgrp * head_group);
  const int rem = static_cast<int>(blockIdx.x) - hgrp * per_group;
  const int qblk = causal ? npb - 1 - rem / gsize : rem / gsize;
  const int bh = hgrp * head_group + rem % gsize;
  const int bkv = bh / group;
  const int q0 = qblk * DQ_BQ;
  // keys seen by some row of the block: [key_lo, key_hi)
  const int key_lo = window > 0 ? max(0, q0 - window + 1) : 0;
  const int key_hi = causal ? min(N, q0 + DQ_BQ) : N;
  const int t_lo = key_lo / DQ_BK;
  const int nt = (key_hi + DQ_BK - 1) / DQ_BK - t_lo;
  auto ring = [&](int t) { return sbase + DQ_OFF_RING + (t % DQ_STAGES) * DQ_STAGE; };
  auto full = [&](int t) { return wait(DQB_FULL + t % DQ_STAGES, (t / DQ_STAGES) & 1); };

  if (threadIdx.x == 0) {
    mbar_init(bar(DQB_QFULL), 1);
    for (int s = 0; s < DQ_STAGES; ++s) {
      mbar_init(bar(DQB_FULL + s), 1);
      mbar_init(bar(DQB_EMPTY + s), 1);
    }
    mbar_init(bar(DQB_SFULL), 1);
    mbar_init(bar(DQB_DPFULL), 1);
    mbar_init(bar(DQB_SREAD), DQ_SOFTMAX_WARPS);
    mbar_init(bar(DQB_DPREAD), DQ_SOFTMAX_WARPS);
    mbar_init(bar(DQB_PFULL), DQ_SOFTMAX_WARPS);
    mbar_init(bar(DQB_DSFREE), 1);
    mbar_init(bar(DQB_DONE), 1);
    mbar_init(bar(DQB_QTMEM), DQ_SOFTMAX_WARPS);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == DQ_WARP_DQ) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == DQ_WARP_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
      const uint32_t qf = bar(DQB_QFULL);
      mbar_arrive_expect_tx(qf, 2 * DQ_TILE);
      tma_load_3d(sbase + DQ_OFF_Q, &tmQ, qf, 0, q0, bh);
      tma_load_3d(sbase + DQ_OFF_Q + DQ_HALF, &tmQ, qf, 64, q0, bh);
      tma_load_3d(sbase + DQ_OFF_DO, &tmdO, qf, 0, q0, bh);
      tma_load_3d(sbase + DQ_OFF_DO + DQ_HALF, &tmdO, qf, 64, q0, bh);
      for (int t = 0; t < nt; ++t) {
        const int st = t % DQ_STAGES;
        if (t >= DQ_STAGES && !wait(DQB_EMPTY + st, ((t / DQ_STAGES) - 1) & 1)) break;
        // stage 2 holds Q_i and dO_i until they are in tensor memory
        if (t == 2 && !wait(DQB_QTMEM, 0)) break;
        const uint32_t fb = bar(DQB_FULL + st);
        const uint32_t dst = ring(t);
        const int key = (t_lo + t) * DQ_BK;
        mbar_arrive_expect_tx(fb, DQ_STAGE);
        tma_load_3d(dst, &tmK, fb, 0, key, bkv);
        tma_load_3d(dst + DQ_HALF, &tmK, fb, 64, key, bkv);
        tma_load_3d(dst + DQ_TILE, &tmV, fb, 0, key, bkv);
        tma_load_3d(dst + DQ_TILE + DQ_HALF, &tmV, fb, 64, key, bkv);
      }
    }
    __syncwarp();
  } else if (warp == DQ_WARP_DQ) {
    // ------------------------------------------------------- dQ issuer
    // dQ += dS K_t once the softmax of tile t has written dS: A = dS from
    // shared memory (K-major: two 64-key boxes), B = K_t MN-major (16 keys =
    // 2048 bytes per step, the two 64-column blocks of d 16 KiB apart).
    if (lane == 0) {
      const uint64_t dsd = sdesc_sw128(sbase + DQ_OFF_DS, 16, 1024);
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        if (!(ok = wait(DQB_PFULL, t & 1))) break;
        tc_fence_after();
        const uint64_t kd = sdesc_sw128(ring(t), DQ_HALF, 1024);
        uint64_t a[8], b[8];
#pragma unroll
        for (int kk = 0; kk < DQ_BK / 16; ++kk) {
          a[kk] = dsd + (((kk >> 2) * DQ_HALF + (kk & 3) * 32) >> 4);
          b[kk] = kd + ((kk * 2048) >> 4);
        }
        mma_ss_batch8(tmem + DQ_TM_DQ, a, b, IDESC_DQ_ACC, t > 0 ? 1u : 0u);
        // S(t) and dP(t) completed before the softmax of tile t wrote dS,
        // so this covers every reader of stage t; and of dS(t).
        mma_commit(bar(DQB_EMPTY + t % DQ_STAGES));
        mma_commit(bar(DQB_DSFREE));
      }
      if (ok) mma_commit(bar(DQB_DONE));
    }
    __syncwarp();
  } else if (warp == DQ_WARP_S || warp == DQ_WARP_DP) {
    // ---------------------------------------------- score issuers (S, dP)
    // S(t) = Q_i K_t^T or dP(t) = dO_i V_t^T (one warp each): A from
    // TMEM (16 elements of d = 8 packed columns per step), B = the K or V
    // tile K-major.  Each waits for the softmax to have copied its previous
    // result into registers.
    const bool dp = warp == DQ_WARP_DP;
    if (lane == 0) {
      bool ok = wait(DQB_QTMEM, 0);
      tc_fence_after();
      for (int t = 0; t < nt && ok; ++t) {
        if (t >= 1 && !(ok = wait(dp ? DQB_DPREAD : DQB_SREAD, (t - 1) & 1))) break;
        if (!(ok = full(t))) break;
        tc_fence_after();
        const uint64_t bd = sdesc_sw128(ring(t) + (dp ? DQ_TILE : 0u), 16, 1024);
        uint32_t a[8];
        uint64_t b[8];
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          a[kk] = tmem + (dp ? DQ_TM_DO : DQ_TM_Q) + 8 * kk;
          b[kk] = bd + (((kk >> 2) * DQ_HALF + (kk & 3) * 32) >> 4);
        }
        mma_ts_batch8(tmem + (dp ? DQ_TM_DP : DQ_TM_S), a, b, IDESC_DQ_S, 0u);
        mma_commit(bar(dp ? DQB_DPFULL : DQB_SFULL));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w: TMEM lane quadrant w & 3 (query rows), key quarter w >> 2 (32
    // of the tile's 128 keys).  Four warps per row: each one's serial work
    // per tile (load, exponentials, dS) is a quarter of a row.
    const int quad = warp & 3, sub = warp >> 2;
    const int row = quad * 32 + lane;
    const int q = q0 + row;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const bool row_valid = q < N;
    const size_t srow = static_cast<size_t>(bh) * Npad + q;      // q < Npad always
    const float nlse = lse_pad[srow];                            // -LSE log2e
    const float nd = d_pad[srow];                                // -scale D
    const float scale_log2 = scale * kLog2e;
    const float slope_log2 = kAlibi ? alibi[bh % heads] * kLog2e : 0.f;
    // keys this row sees: [lo, hi]
    const int lo = window > 0 ? q - window + 1 : 0;
    const int hi = causal ? min(q, N - 1) : N - 1;
    // Q_i (warps 0-7) or dO_i (warps 8-15), row by row, into tensor memory,
    // half a row (one 64-column box) per warp: column c holds elements 2c
    // and 2c+1 of the row (the A-operand layout).
    bool ok = wait(DQB_QFULL, 0);
    if (ok) {
      const uint8_t* tile = smem + (sub < 2 ? DQ_OFF_Q : DQ_OFF_DO);
      const uint32_t col = sub < 2 ? DQ_TM_Q : DQ_TM_DO;
      {
        const int h = sub & 1;
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(tile + h * DQ_HALF +
                                                          sw128_offset(row, c));
          r[4 * c] = v.x;
          r[4 * c + 1] = v.y;
          r[4 * c + 2] = v.z;
          r[4 * c + 3] = v.w;
        }
        tmem_st32(tmem + lane_addr + col + 32 * h, r);
      }
      tmem_wait_st();
      tc_fence_before();
      fence_proxy_async_smem();   // the tiles' space is refilled by TMA next
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DQB_QTMEM));
    }
    const uint32_t s_addr = tmem + lane_addr + DQ_TM_S + 32 * sub;
    const uint32_t dp_addr = tmem + lane_addr + DQ_TM_DP + 32 * sub;
    uint8_t* ds_box = smem + DQ_OFF_DS + (sub >> 1) * DQ_HALF;   // box of this warp's 32 keys
    const uint64_t sc2 = f2pack(scale_log2, scale_log2);
    const uint64_t s2 = f2pack(scale, scale), nd2 = f2pack(nd, nd);
    for (int t = 0; t < nt && ok; ++t) {
      if (!wait(DQB_SFULL, t & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int j0 = (t_lo + t) * DQ_BK + 32 * sub;               // first key of this quarter
      const bool need_mask = !row_valid || j0 < lo || j0 + 31 > hi;
      const float d0 = static_cast<float>(q - j0);
      float p[32];
      {
        uint32_t sr[32];
        tmem_ld32(s_addr, sr);                    // this quarter's 32 scores
        // S(t) is in registers: its columns may take S(t + 1)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(DQB_SREAD));
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int k = e;
          float b0 = nlse, b1 = nlse;
          if constexpr (kAlibi) {
            b0 = fmaf(-slope_log2, fabsf(d0 - static_cast<float>(k)), nlse);
            b1 = fmaf(-slope_log2, fabsf(d0 - static_cast<float>(k + 1)), nlse);
          }
          // exponent arguments on a packed fp32 pair
          float a0, a1;
          f2unpack(f2fma(f2pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sc2,
                         f2pack(b0, b1)), a0, a1);
          float p0 = fast_exp2(a0);
          float p1 = fast_exp2(a1);
          if (need_mask) {
            const bool v0 = row_valid && j0 + k >= lo && j0 + k <= hi;
            const bool v1 = row_valid && j0 + k + 1 >= lo && j0 + k + 1 <= hi;
            p0 = v0 ? p0 : 0.f;
            p1 = v1 ? p1 : 0.f;
          }
          p[k] = p0;
          p[k + 1] = p1;
        }
      }
      if (!wait(DQB_DPFULL, t & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t gk[16];
      {
        uint32_t dr[32];
        tmem_ld32(dp_addr, dr);
        // dP(t) is in registers: its columns may take dP(t + 1)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(DQB_DPREAD));
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int k = e;
          // scale dS = P (scale dP - scale D) on a packed fp32 pair
          float g0, g1;
          f2unpack(f2mul(f2pack(p[k], p[k + 1]),
                         f2fma(f2pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), s2,
                               nd2)), g0, g1);
          gk[k / 2] = pack_bf16x2(g0, g1);
        }
      }
      // dS row into shared memory (the K-major A operand of dQ) once dQ(t-1)
      // has read the previous one
      if (t >= 1 && !wait(DQB_DSFREE, (t - 1) & 1)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(ds_box + sw128_offset(row, 4 * (sub & 1) + c)) =
            make_uint4(gk[4 * c], gk[4 * c + 1], gk[4 * c + 2], gk[4 * c + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DQB_PFULL));
    }
    if (ok && wait(DQB_DONE, 0)) {
      tc_fence_after();
      __nv_bfloat16* out = dQ + (static_cast<size_t>(bh) * N + q) * HD + 32 * sub;
      {
        uint32_t r[32];
        tmem_ld32(tmem + lane_addr + DQ_TM_DQ + 32 * sub, r);
        if (row_valid) {
          uint4* d4 = reinterpret_cast<uint4*>(out);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            d4[i] = make_uint4(
                pack_bf16x2(__uint_as_float(r[8 * i]), __uint_as_float(r[8 * i + 1])),
                pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == DQ_WARP_DQ) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

size_t padded_len(int N) { return (static_cast<size_t>(N) + PAD - 1) / PAD * PAD; }

template <class K>
cudaError_t set_smem(K kernel, uint32_t bytes = SMEM_BYTES) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

}  // namespace

size_t backward_workspace_bytes(int B, int H, int N) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t prow = static_cast<size_t>(B) * H * padded_len(N);
  return align256(rows * HD * sizeof(float)) + 2 * align256(prow * sizeof(float));
}

cudaError_t launch_backward_bf16(const BwdMaps& maps, const void* q, const void* k,
                                 const void* v, const void* o, const float* lse,
                                 const void* dO, void* dq, void* dk, void* dv, int B, int H,
                                 int Hkv, int N, float scale, int causal, int window,
                                 const float* alibi, const BwdMaps* dq_maps, void* ws,
                                 cudaStream_t stream, const TimingEvents& ev) {
  (void)q;   // the tensors behind the maps
  (void)dk;
  (void)dv;
  (void)k;
  (void)v;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    cudaError_t e = set_smem(bwd_main_kernel<false, true>);
    if (e == cudaSuccess) e = set_smem(bwd_main_kernel<true, true>);
    if (e == cudaSuccess) e = set_smem(bwd_main_kernel<false, false>);
    if (e == cudaSuccess) e = set_smem(bwd_main_kernel<true, false>);
    if (e == cudaSuccess) e = set_smem(bwd_dq_kernel<false>, DQ_SMEM);
    if (e == cudaSuccess) e = set_smem(bwd_dq_kernel<true>, DQ_SMEM);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  const int BH = B * H;
  const int Npad = static_cast<int>(padded_len(N));
  const size_t rows = static_cast<size_t>(BH) * N;
  const size_t prows = static_cast<size_t>(BH) * Npad;
  float* dq_acc = static_cast<float*>(ws);
  float* d_pad = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                          align256(rows * HD * sizeof(float)));
  float* lse_pad = reinterpret_cast<float*>(reinterpret_cast<char*>(d_pad) +
                                            align256(prows * sizeof(float)));
  const bool deterministic = dq_maps != nullptr;
  bwd_pre_kernel<<<dim3(static_cast<unsigned>((prows + 15) / 16)), dim3(256), 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, d_pad,
      scale, lse_pad, deterministic ? nullptr : dq_acc, N, Npad, prows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nkv = (N + BKV - 1) / BKV;
  if (ev.before) cudaEventRecord(ev.before, stream);
  const int g = H / Hkv;
  // Blocks go heavy-first (increasing key block) within each group of heads:
  // a longer heavy-first list evens out the end of the grid (grouped query
  // heads make each block g times longer, where it counts most), while the
  // group's rows must stay in L2.
  long long fit = kHeadGroupBytes / (static_cast<long long>(g) * N * 1024);
  fit = fit < 1 ? 1 : (fit > kHeadGroupKv ? kHeadGroupKv : fit);
  const int head_group = static_cast<int>(fit);   // key/value heads per group
  auto kernel = deterministic
                    ? (alibi ? bwd_main_kernel<true, false> : bwd_main_kernel<false, false>)
                    : (alibi ? bwd_main_kernel<true, true> : bwd_main_kernel<false, true>);
  kernel<<<dim3(nkv * B * Hkv), dim3(deterministic ? bwd_threads<false>() : bwd_threads<true>()),
           SMEM_BYTES, stream>>>(
      maps.q, maps.k, maps.v, maps.dO, maps.dk, maps.dv, lse_pad, d_pad, dq_acc, B * Hkv, N,
      Npad, scale, causal, g, window, head_group, alibi, H);
  e = cudaGetLastError();
  if (ev.after) cudaEventRecord(ev.after, stream);
  if (e != cudaSuccess) return e;
  if (deterministic) {
    // dQ by query blocks, in a fixed key order, written once (no atomics)
    const int npb = (N + DQ_BQ - 1) / DQ_BQ;
    // whole key/value heads per group, their K and V (512 B per key row)
    // within ~32 MB of L2
    long long kv_fit = kDqGroupBytes / (static_cast<long long>(N) * 512);
    kv_fit = kv_fit < 1 ? 1 : (kv_fit > kHeadGroupKv ? kHeadGroupKv : kv_fit);
    const int dq_group = static_cast<int>(kv_fit) * g;   // query heads per group
    auto dqk = alibi ? bwd_dq_kernel<true> : bwd_dq_kernel<false>;
    dqk<<<dim3(npb * BH), dim3(DQ_THREADS), DQ_SMEM, stream>>>(
        dq_maps->q, dq_maps->k, dq_maps->v, dq_maps->dO, lse_pad, d_pad,
        static_cast<__nv_bfloat16*>(dq), BH, N, Npad, scale, causal, g, window, alibi, H,
        dq_group);
    return cudaGetLastError();
  }
  const size_t n8 = rows * HD / 8;
  bwd_convert_kernel<<<dim3(static_cast<unsigned>((n8 + 255) / 256)), dim3(256), 0, stream>>>(
      dq_acc, static_cast<__nv_bfloat16*>(dq), n8);
  return cudaGetLastError();
}

int status_backward_bf16(bool clear) {
  int s = 0;
  cudaMemcpyFromSymbol(&s, g_status_bwd, sizeof(int));
  if (clear && s != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_status_bwd, &zero, sizeof(int));
  }
  return s;
}

}  // namespace fa
