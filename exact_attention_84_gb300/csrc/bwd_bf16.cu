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
//   bwd_pre      D = rowsum(dO * O) (fp32) and zeroing of the fp32 dQ
//                accumulator.
//   bwd_main     one thread block per (b, h, 128-key block j).  K_j and V_j
//                stay in shared memory; 64-row blocks Q_i, dO_i stream past
//                in a 2-stage TMA ring.  Per block i the tensor cores form
//                S^T = K_j Q_i^T and dP^T = V_j dO_i^T in TMEM; the softmax
//                warps (one key row per thread) turn them into P^T and dS^T
//                (bf16, swizzled shared memory); the tensor cores then add
//                dV += P^T dO_i and dK += dS^T Q_i in TMEM and form
//                dQ_i^T = K_j^T dS^T, which four writer warps add into the
//                fp32 accumulator with atomics.  dK, dV leave TMEM once.
//   bwd_convert  dQ = bf16(accumulator).
// Causal: query blocks entirely above the key block are skipped; the two
// blocks that straddle the diagonal are masked element-wise.
#include <cfloat>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ int g_status_bwd;

constexpr int HD = 128;
constexpr int BKV = 128;                  // key rows per block (TMEM lanes)
constexpr int BQ = 64;                    // query rows per streamed block
constexpr uint32_t KV_TILE = BKV * HD * 2;        // 32 KiB
constexpr uint32_t KV_HALF = KV_TILE / 2;         // 128 rows x 64 cols
constexpr uint32_t Q_TILE = BQ * HD * 2;          // 16 KiB
constexpr uint32_t Q_HALF = Q_TILE / 2;           // 64 rows x 64 cols
constexpr uint32_t PT_TILE = BKV * BQ * 2;        // 16 KiB, [key][query] bf16

constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + KV_TILE;
constexpr uint32_t OFF_Q = OFF_V + KV_TILE;          // 2 stages
constexpr uint32_t OFF_DO = OFF_Q + 2 * Q_TILE;      // 2 stages
constexpr uint32_t OFF_PT = OFF_DO + 2 * Q_TILE;
constexpr uint32_t OFF_DST = OFF_PT + PT_TILE;
constexpr uint32_t OFF_STAT = OFF_DST + PT_TILE;     // [2 buffers][LSE 64 | D 64] fp32
constexpr uint32_t OFF_BAR = OFF_STAT + 2 * 2 * BQ * 4;
constexpr int B_KVFULL = 0;
constexpr int B_QFULL = 1;     // + stage
constexpr int B_QEMPTY = 3;    // + stage
constexpr int B_SFULL = 5;
constexpr int B_SFREE = 6;
constexpr int B_PFULL = 7;
constexpr int B_PFREE = 8;
constexpr int B_DQFULL = 9;
constexpr int B_DQFREE = 10;
constexpr int B_STAT = 11;     // + buffer: the 128 softmax threads staged LSE / D
constexpr int NBAR = 13;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_DP = 64, TM_DQ = 128, TM_DV = 256, TM_DK = 384;

constexpr int NTHREADS = 320;   // 0 producer, 1 MMA, 2-5 softmax, 6-9 dQ writers
constexpr float kLog2e = 1.4426950408889634f;

// S^T = K_j Q_i^T and dP^T = V_j dO_i^T: M = 128 keys, N = 64 queries.
constexpr uint32_t IDESC_ST = idesc_bf16(BKV, BQ, false, false);
// dV += P^T dO_i, dK += dS^T Q_i: M = 128 keys, N = 128 (d), B MN-major.
constexpr uint32_t IDESC_DKV = idesc_bf16(BKV, HD, false, true);
// dQ_i^T = K_j^T dS^T: M = 128 (d), N = 64 queries; both operands MN-major.
constexpr uint32_t IDESC_DQ = idesc_bf16(HD, BQ, true, true);

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) {
  return base + OFF_BAR + 8u * static_cast<uint32_t>(i);
}

__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, float* out) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// ------------------------------------------------------------------ bwd_pre
// One warp per row: D = sum_k dO_k O_k; the row of the dQ accumulator is
// zeroed at the same time.
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      float* __restrict__ Dvec,
                                                      float* __restrict__ dq_acc,
                                                      size_t rows) {
  const size_t row = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint2 a = *reinterpret_cast<const uint2*>(o + row * HD + lane * 4);
  const uint2 b = *reinterpret_cast<const uint2*>(dO + row * HD + lane * 4);
  float s = __uint_as_float(a.x << 16) * __uint_as_float(b.x << 16);
  s = fmaf(__uint_as_float(a.x & 0xffff0000u), __uint_as_float(b.x & 0xffff0000u), s);
  s = fmaf(__uint_as_float(a.y << 16), __uint_as_float(b.y << 16), s);
  s = fmaf(__uint_as_float(a.y & 0xffff0000u), __uint_as_float(b.y & 0xffff0000u), s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) Dvec[row] = s;
  *reinterpret_cast<float4*>(dq_acc + row * HD + lane * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// --------------------------------------------------------------- bwd_convert
__global__ void __launch_bounds__(256) bwd_convert_kernel(const float* __restrict__ dq_acc,
                                                          __nv_bfloat16* __restrict__ dq,
                                                          size_t n4) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 v = reinterpret_cast<const float4*>(dq_acc)[i];
  reinterpret_cast<uint2*>(dq)[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// ------------------------------------------------------------------ bwd_main
__global__ void __launch_bounds__(NTHREADS, 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const float* __restrict__ LSE, const float* __restrict__ Dvec,
                float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dK,
                __nv_bfloat16* __restrict__ dV, int BH, int N, float scale, int causal) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int j = tile / BH;                  // key block (small j = most work when causal)
  const int bh = tile % BH;
  const int nqb = (N + BQ - 1) / BQ;
  const int i0 = causal ? (j * BKV) / BQ : 0;
  const int nit = nqb - i0;
  const float scale_log2 = scale * kLog2e;

  if (threadIdx.x == 0) {
    mbar_init(bar_addr(sbase, B_KVFULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_addr(sbase, B_QFULL + s), 1);
      mbar_init(bar_addr(sbase, B_QEMPTY + s), 1);
    }
    mbar_init(bar_addr(sbase, B_SFULL), 1);
    mbar_init(bar_addr(sbase, B_SFREE), 4);
    mbar_init(bar_addr(sbase, B_PFULL), 4);
    mbar_init(bar_addr(sbase, B_PFREE), 1);
    mbar_init(bar_addr(sbase, B_DQFULL), 1);
    mbar_init(bar_addr(sbase, B_DQFREE), 4);
    mbar_init(bar_addr(sbase, B_STAT), 128);
    mbar_init(bar_addr(sbase, B_STAT + 1), 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
      const uint32_t kvf = bar_addr(sbase, B_KVFULL);
      mbar_arrive_expect_tx(kvf, 2 * KV_TILE);
      tma_load_3d(sbase + OFF_K, &tmK, kvf, 0, j * BKV, bh);
      tma_load_3d(sbase + OFF_K + KV_HALF, &tmK, kvf, 64, j * BKV, bh);
      tma_load_3d(sbase + OFF_V, &tmV, kvf, 0, j * BKV, bh);
      tma_load_3d(sbase + OFF_V + KV_HALF, &tmV, kvf, 64, j * BKV, bh);
      for (int it = 0; it < nit; ++it) {
        const int st = it & 1;
        const int qb = (i0 + it) * BQ;
        if (it >= 2 && !mbar_wait(bar_addr(sbase, B_QEMPTY + st), ((it >> 1) - 1) & 1,
                                  abort_flag, &g_status_bwd))
          break;
        const uint32_t qf = bar_addr(sbase, B_QFULL + st);
        mbar_arrive_expect_tx(qf, 2 * Q_TILE);
        const uint32_t qs = sbase + OFF_Q + st * Q_TILE;
        const uint32_t ds = sbase + OFF_DO + st * Q_TILE;
        tma_load_3d(qs, &tmQ, qf, 0, qb, bh);
        tma_load_3d(qs + Q_HALF, &tmQ, qf, 64, qb, bh);
        tma_load_3d(ds, &tmdO, qf, 0, qb, bh);
        tma_load_3d(ds + Q_HALF, &tmdO, qf, 64, qb, bh);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(bar_addr(sbase, B_KVFULL), 0, abort_flag, &g_status_bwd);
      for (int it = 0; it < nit && ok; ++it) {
        const int st = it & 1;
        const uint32_t qs = sbase + OFF_Q + st * Q_TILE;
        const uint32_t ds = sbase + OFF_DO + st * Q_TILE;
        ok = mbar_wait(bar_addr(sbase, B_QFULL + st), (it >> 1) & 1, abort_flag, &g_status_bwd);
        if (ok && it > 0)
          ok = mbar_wait(bar_addr(sbase, B_SFREE), (it - 1) & 1, abort_flag, &g_status_bwd);
        if (!ok) break;
        tc_fence_after();
        // S^T = K_j Q_i^T and dP^T = V_j dO_i^T (reduction over d)
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * KV_HALF + (kk & 3) * 32;
          const uint32_t kb = (kk >> 2) * Q_HALF + (kk & 3) * 32;
          mma_ss(tmem + TM_S, sdesc_sw128(sbase + OFF_K + ka, 16, 1024),
                 sdesc_sw128(qs + kb, 16, 1024), IDESC_ST, kk > 0 ? 1u : 0u);
          mma_ss(tmem + TM_DP, sdesc_sw128(sbase + OFF_V + ka, 16, 1024),
                 sdesc_sw128(ds + kb, 16, 1024), IDESC_ST, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_addr(sbase, B_SFULL));
        ok = mbar_wait(bar_addr(sbase, B_PFULL), it & 1, abort_flag, &g_status_bwd);
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO_i and dK += dS^T Q_i (reduction over the 64 queries)
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          mma_ss(tmem + TM_DV, sdesc_sw128(sbase + OFF_PT + kk * 32, 16, 1024),
                 sdesc_sw128(ds + kk * 2048, Q_HALF, 1024), IDESC_DKV, acc);
          mma_ss(tmem + TM_DK, sdesc_sw128(sbase + OFF_DST + kk * 32, 16, 1024),
                 sdesc_sw128(qs + kk * 2048, Q_HALF, 1024), IDESC_DKV, acc);
        }
        if (it > 0)
          ok = mbar_wait(bar_addr(sbase, B_DQFREE), (it - 1) & 1, abort_flag, &g_status_bwd);
        if (!ok) break;
        tc_fence_after();
        // dQ_i^T = K_j^T dS^T (reduction over the 128 keys)
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          mma_ss(tmem + TM_DQ, sdesc_sw128(sbase + OFF_K + kk * 2048, KV_HALF, 1024),
                 sdesc_sw128(sbase + OFF_DST + kk * 2048, PT_TILE, 1024), IDESC_DQ,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_addr(sbase, B_DQFULL));
        mma_commit(bar_addr(sbase, B_PFREE));
        mma_commit(bar_addr(sbase, B_QEMPTY + st));
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int row = quad * 32 + lane;                 // key row within block j
    const int kv = j * BKV + row;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const int gtid = threadIdx.x - 64;                // 0..127 within the group
    float* stat = reinterpret_cast<float*>(smem + OFF_STAT);
    bool ok = true;
    for (int it = 0; it < nit; ++it) {
      const int qb = (i0 + it) * BQ;
      float* st_buf = stat + (it & 1) * (2 * BQ);     // [LSE*log2e | D]
      {
        const int c = gtid & (BQ - 1);
        const int q = qb + c;
        float val = 0.f;
        if (q < N) {
          const size_t idx = static_cast<size_t>(bh) * N + q;
          val = (gtid < BQ) ? LSE[idx] * kLog2e : Dvec[idx];
        }
        st_buf[gtid] = val;
      }
      // All 128 threads have staged their value before anyone reads the
      // buffer; a buffer is rewritten two blocks later, after every thread
      // has arrived here again (so has finished reading it).
      mbar_arrive(bar_addr(sbase, B_STAT + (it & 1)));
      if (!mbar_wait(bar_addr(sbase, B_STAT + (it & 1)), (it >> 1) & 1, abort_flag,
                     &g_status_bwd) ||
          !mbar_wait(bar_addr(sbase, B_SFULL), it & 1, abort_flag, &g_status_bwd)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[BQ], dp[BQ];
      tmem_ld32_sync(tmem + lane_addr + TM_S, s);
      tmem_ld32_sync(tmem + lane_addr + TM_S + 32, s + 32);
      tmem_ld32_sync(tmem + lane_addr + TM_DP, dp);
      tmem_ld32_sync(tmem + lane_addr + TM_DP + 32, dp + 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_SFREE));

      const bool need_mask = (causal && qb < j * BKV + BKV) || (qb + BQ > N) || (kv >= N);
      uint32_t pk[BQ / 2], dk[BQ / 2];
#pragma unroll
      for (int c = 0; c < BQ; c += 2) {
        float p0 = fast_exp2(fmaf(s[c], scale_log2, -st_buf[c]));
        float p1 = fast_exp2(fmaf(s[c + 1], scale_log2, -st_buf[c + 1]));
        if (need_mask) {
          const int q0 = qb + c;
          if (q0 >= N || kv >= N || (causal && q0 < kv)) p0 = 0.f;
          if (q0 + 1 >= N || kv >= N || (causal && q0 + 1 < kv)) p1 = 0.f;
        }
        const float g0 = p0 * (dp[c] - st_buf[BQ + c]);
        const float g1 = p1 * (dp[c + 1] - st_buf[BQ + c + 1]);
        pk[c / 2] = pack_bf16x2(p0, p1);
        dk[c / 2] = pack_bf16x2(g0, g1);
      }
      if (it > 0 && !mbar_wait(bar_addr(sbase, B_PFREE), (it - 1) & 1, abort_flag,
                               &g_status_bwd)) {
        ok = false;
        break;
      }
      uint8_t* pt = smem + OFF_PT;
      uint8_t* dst = smem + OFF_DST;
#pragma unroll
      for (int ch = 0; ch < BQ / 8; ++ch) {
        const uint32_t off = sw128_offset(row, ch);
        *reinterpret_cast<uint4*>(pt + off) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        *reinterpret_cast<uint4*>(dst + off) =
            make_uint4(dk[4 * ch], dk[4 * ch + 1], dk[4 * ch + 2], dk[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_PFULL));
    }
    // dK and dV rows leave TMEM once, after the last block's MMAs.
    if (ok && nit > 0 &&
        mbar_wait(bar_addr(sbase, B_PFREE), (nit - 1) & 1, abort_flag, &g_status_bwd)) {
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        __nv_bfloat16* out = half == 0 ? dV : dK;
        const float mul = half == 0 ? 1.f : scale;
        const uint32_t src = tmem + lane_addr + (half == 0 ? TM_DV : TM_DK);
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          float acc[32];
          tmem_ld32_sync(src + c * 32, acc);
          if (kv < N) {
            uint4* d4 = reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * N + kv) * HD +
                                                 c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(pack_bf16x2(acc[8 * i] * mul, acc[8 * i + 1] * mul),
                                 pack_bf16x2(acc[8 * i + 2] * mul, acc[8 * i + 3] * mul),
                                 pack_bf16x2(acc[8 * i + 4] * mul, acc[8 * i + 5] * mul),
                                 pack_bf16x2(acc[8 * i + 6] * mul, acc[8 * i + 7] * mul));
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ writers
    const int quad = warp & 3;
    const int dcol = quad * 32 + lane;               // head-dimension index (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    for (int it = 0; it < nit; ++it) {
      const int qb = (i0 + it) * BQ;
      if (!mbar_wait(bar_addr(sbase, B_DQFULL), it & 1, abort_flag, &g_status_bwd)) break;
      tc_fence_after();
      float g[BQ];
      tmem_ld32_sync(tmem + lane_addr + TM_DQ, g);
      tmem_ld32_sync(tmem + lane_addr + TM_DQ + 32, g + 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_DQFREE));
      float* base = dq_acc + (static_cast<size_t>(bh) * N + qb) * HD + dcol;
      const int lim = min(BQ, N - qb);
#pragma unroll 8
      for (int c = 0; c < BQ; ++c)
        if (c < lim) red_add_f32(base + static_cast<size_t>(c) * HD, g[c] * scale);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

size_t backward_workspace_bytes(int B, int H, int N) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  return align256(rows * HD * sizeof(float)) + align256(rows * sizeof(float));
}

cudaError_t launch_backward_bf16(const BwdMaps& maps, const void* q, const void* k,
                                 const void* v, const void* o, const float* lse,
                                 const void* dO, void* dq, void* dk, void* dv, int B, int H,
                                 int N, float scale, int causal, void* ws,
                                 cudaStream_t stream, const TimingEvents& ev) {
  (void)q;
  (void)k;
  (void)v;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int BH = B * H;
  const size_t rows = static_cast<size_t>(BH) * N;
  float* dq_acc = static_cast<float*>(ws);
  float* Dvec = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                         align256(rows * HD * sizeof(float)));
  bwd_pre_kernel<<<dim3(static_cast<unsigned>((rows + 7) / 8)), dim3(256), 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), Dvec, dq_acc,
      rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nkv = (N + BKV - 1) / BKV;
  if (ev.before) cudaEventRecord(ev.before, stream);
  bwd_main_kernel<<<dim3(nkv * BH), dim3(NTHREADS), SMEM_BYTES, stream>>>(
      maps.q, maps.k, maps.v, maps.dO, lse, Dvec, dq_acc, static_cast<__nv_bfloat16*>(dk),
      static_cast<__nv_bfloat16*>(dv), BH, N, scale, causal);
  e = cudaGetLastError();
  if (ev.after) cudaEventRecord(ev.after, stream);
  if (e != cudaSuccess) return e;
  const size_t n4 = rows * HD / 4;
  bwd_convert_kernel<<<dim3(static_cast<unsigned>((n4 + 255) / 256)), dim3(256), 0, stream>>>(
      dq_acc, static_cast<__nv_bfloat16*>(dq), n4);
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
