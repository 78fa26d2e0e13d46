// fwd_bf16.cu -- fused exact-attention forward for bf16 on sm_103a.
//
// Method ("FlashAttention ontleed", sections "Tiling en Online Softmax" and
// "Algoritmische kern in pseudocode"; "03. FlashAttention", section
// "FlashAttention v1", "Mecanisme"): one thread block keeps a 128-row block
// Q_i on chip while 128-row K_j / V_j tiles stream past it.  Per tile:
//   S = Q_i K_j^T                  (tensor cores, fp32 accumulator in TMEM)
//   m_new = max(m, rowmax(S*scale)) (softmax warps, registers)
//   P = exp(S*scale - m_new)        (bf16, written to shared memory)
//   l = l e^(m - m_new) + rowsum(P)
//   O = diag(e^(m - m_new)) O + P V_j   (rescale in TMEM, MMA accumulates)
// and after the last tile O / l and LSE = m + ln(l) go to HBM once.  The
// N x N score matrix never leaves the chip (Lensa ML "FlashAttention",
// step 3: 0 B of S written).
//
// GB300 mapping (the pages' A100/H100 designs are prior art only):
//   warp 0      TMA producer: Q once, then K_j and V_j into a 2-stage ring
//               (128-byte swizzled boxes of 64 columns) under mbarriers.
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma from one
//               thread: S_j into one of two TMEM score buffers, then
//               O += P_{j-1} V_{j-1}; completion via tcgen05.commit.
//   warps 2-5   softmax: each thread owns one row (TMEM lane), reads its
//               128 scores, keeps m and l in registers, exponentiates with
//               ex2 on log2(e)-prescaled values, rescales its O row in TMEM
//               when its maximum moved, writes P (bf16) into a swizzled
//               shared-memory tile for the P.V MMA, and runs the epilogue.
// Causal: key tiles above the diagonal are skipped; only the diagonal tile
// (and a ragged last tile) is masked element-wise.  Heavy (late) query
// blocks are scheduled first.
#include <cfloat>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ int g_status_fwd_bf16;

constexpr int BM = 128;                 // query rows per block (TMEM lanes)
constexpr int BN = 128;                 // keys per tile
constexpr int HD = 128;                 // head dimension
constexpr int STAGES = 2;               // K/V ring depth
constexpr uint32_t TILE_BYTES = BM * HD * 2;        // 32 KiB
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;     // 128 rows x 64 columns

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + STAGES * TILE_BYTES;
constexpr uint32_t OFF_P = OFF_V + STAGES * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_P + TILE_BYTES;
// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_KFULL = 1;                 // + stage
constexpr int B_VFULL = B_KFULL + STAGES;  // + stage
constexpr int B_EMPTY = B_VFULL + STAGES;  // + stage
constexpr int B_SFULL = B_EMPTY + STAGES;  // + buffer (2)
constexpr int B_SFREE = B_SFULL + 2;       // + buffer (2)
constexpr int B_PFULL = B_SFREE + 2;
constexpr int B_ODONE = B_PFULL + 1;
constexpr int NBAR = B_ODONE + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256;

constexpr int NTHREADS = 192;
constexpr int SOFTMAX_WARPS = 4;

constexpr float kLn2 = 0.6931471805599453f;

// S = Q K^T: A = Q (K-major), B = K tile (K-major), M = N = 128.
constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
// O += P V: A = P (K-major over keys), B = V tile, whose rows run along the
// reduction (key) axis with d contiguous: MN-major.
constexpr uint32_t IDESC_O = idesc_bf16(BM, HD, false, true);

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) {
  return base + OFF_BAR + 8u * static_cast<uint32_t>(i);
}

__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, float* out) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(NTHREADS, 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                float* __restrict__ LSE, int BH, int N, float scale_log2, int causal) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int nq = (N + BM - 1) / BM;
  const int nkv = (N + BN - 1) / BN;
  const int tile = blockIdx.x;
  const int qi = causal ? (nq - 1 - tile / BH) : (tile / BH);
  const int bh = tile % BH;
  const int nt = causal ? min(qi + 1, nkv) : nkv;

  if (threadIdx.x == 0) {
    mbar_init(bar_addr(sbase, B_QFULL), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_addr(sbase, B_KFULL + s), 1);
      mbar_init(bar_addr(sbase, B_VFULL + s), 1);
      mbar_init(bar_addr(sbase, B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_addr(sbase, B_SFULL + b), 1);
      mbar_init(bar_addr(sbase, B_SFREE + b), SOFTMAX_WARPS);
    }
    mbar_init(bar_addr(sbase, B_PFULL), SOFTMAX_WARPS);
    mbar_init(bar_addr(sbase, B_ODONE), 1);
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
      const uint32_t qf = bar_addr(sbase, B_QFULL);
      mbar_arrive_expect_tx(qf, TILE_BYTES);
      tma_load_3d(sbase + OFF_Q, &tmQ, qf, 0, qi * BM, bh);
      tma_load_3d(sbase + OFF_Q + HALF_BYTES, &tmQ, qf, 64, qi * BM, bh);
      for (int j = 0; j < nt; ++j) {
        const int st = j % STAGES;
        if (j >= STAGES &&
            !mbar_wait(bar_addr(sbase, B_EMPTY + st), ((j / STAGES) - 1) & 1, abort_flag,
                       &g_status_fwd_bf16))
          break;
        const uint32_t kf = bar_addr(sbase, B_KFULL + st);
        const uint32_t vf = bar_addr(sbase, B_VFULL + st);
        const uint32_t ks = sbase + OFF_K + st * TILE_BYTES;
        const uint32_t vs = sbase + OFF_V + st * TILE_BYTES;
        mbar_arrive_expect_tx(kf, TILE_BYTES);
        tma_load_3d(ks, &tmK, kf, 0, j * BN, bh);
        tma_load_3d(ks + HALF_BYTES, &tmK, kf, 64, j * BN, bh);
        mbar_arrive_expect_tx(vf, TILE_BYTES);
        tma_load_3d(vs, &tmV, vf, 0, j * BN, bh);
        tma_load_3d(vs + HALF_BYTES, &tmV, vf, 64, j * BN, bh);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(bar_addr(sbase, B_QFULL), 0, abort_flag, &g_status_fwd_bf16);
      auto issue_pv = [&](int t) -> bool {
        const int st = t % STAGES;
        if (!mbar_wait(bar_addr(sbase, B_PFULL), t & 1, abort_flag, &g_status_fwd_bf16))
          return false;
        if (!mbar_wait(bar_addr(sbase, B_VFULL + st), (t / STAGES) & 1, abort_flag,
                       &g_status_fwd_bf16))
          return false;
        tc_fence_after();
        const uint32_t vs = sbase + OFF_V + st * TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t a = sdesc_sw128(sbase + OFF_P + (kk >> 2) * HALF_BYTES + (kk & 3) * 32,
                                         16, 1024);
          const uint64_t b = sdesc_sw128(vs + kk * 2048, HALF_BYTES, 1024);
          mma_ss(tmem + TM_O, a, b, IDESC_O, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_addr(sbase, B_ODONE));
        mma_commit(bar_addr(sbase, B_EMPTY + st));
        return true;
      };
      if (ok) {
        tc_fence_after();
        for (int j = 0; j < nt && ok; ++j) {
          const int st = j % STAGES;
          const int b = j & 1;
          if (!mbar_wait(bar_addr(sbase, B_KFULL + st), (j / STAGES) & 1, abort_flag,
                         &g_status_fwd_bf16)) {
            ok = false;
            break;
          }
          if (j >= 2 && !mbar_wait(bar_addr(sbase, B_SFREE + b), ((j >> 1) - 1) & 1,
                                   abort_flag, &g_status_fwd_bf16)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ks = sbase + OFF_K + st * TILE_BYTES;
          const uint32_t sd = tmem + (b ? TM_S1 : TM_S0);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
            const uint64_t a = sdesc_sw128(sbase + OFF_Q + off, 16, 1024);
            const uint64_t bd = sdesc_sw128(ks + off, 16, 1024);
            mma_ss(sd, a, bd, IDESC_S, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar_addr(sbase, B_SFULL + b));
          if (j >= 1 && !issue_pv(j - 1)) ok = false;
        }
        if (ok) issue_pv(nt - 1);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;             // row of the Q block
    const int q_row = qi * BM + row;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    float m = -INFINITY;                          // running max, log2 units
    float l = 0.f;                                // running sum
    bool ok = true;
    uint8_t* sP = smem + OFF_P;

    for (int j = 0; j < nt; ++j) {
      const int b = j & 1;
      if (!mbar_wait(bar_addr(sbase, B_SFULL + b), (j >> 1) & 1, abort_flag,
                     &g_status_fwd_bf16)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[BN];
      const uint32_t sd = tmem + lane_addr + (b ? TM_S1 : TM_S0);
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32_sync(sd + c * 32, s + c * 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_SFREE + b));

      // mask: causal diagonal tile, or keys past the end of the sequence
      const bool diag = causal && (j == qi);
      const bool ragged = (j == nkv - 1) && (N % BN != 0);
      if (diag || ragged) {
        const int lim = causal ? min(q_row, N - 1) : (N - 1);
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (j * BN + c > lim) s[c] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m, mx * scale_log2);
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = fast_exp2(m - m_ref);
      float rs = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float p0 = fast_exp2(fmaf(s[2 * c], scale_log2, -m_ref));
        const float p1 = fast_exp2(fmaf(s[2 * c + 1], scale_log2, -m_ref));
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * corr + rs;
      m = m_new;

      if (j > 0) {
        // O and the P buffer are in use by P_{j-1} V_{j-1} until it completes.
        if (!mbar_wait(bar_addr(sbase, B_ODONE), (j - 1) & 1, abort_flag,
                       &g_status_fwd_bf16)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, corr != 1.f)) {
          const uint32_t od = tmem + lane_addr + TM_O;
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(od + c * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
            tmem_st32(od + c * 32, r);
          }
          tmem_wait_st();
        }
      }
      // P row -> shared memory in the 128-byte-swizzled K-major layout
#pragma unroll
      for (int ch = 0; ch < BN / 8; ++ch) {
        const uint32_t off = (ch >> 3) * HALF_BYTES + sw128_offset(row, ch & 7);
        *reinterpret_cast<uint4*>(sP + off) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_PFULL));
    }

    if (ok && mbar_wait(bar_addr(sbase, B_ODONE), (nt - 1) & 1, abort_flag,
                        &g_status_fwd_bf16)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const uint32_t od = tmem + lane_addr + TM_O;
      __nv_bfloat16* orow = O + (static_cast<size_t>(bh) * N + q_row) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float acc[32];
        tmem_ld32_sync(od + c * 32, acc);
        if (q_row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16x2(acc[8 * i] * inv_l, acc[8 * i + 1] * inv_l),
                                pack_bf16x2(acc[8 * i + 2] * inv_l, acc[8 * i + 3] * inv_l),
                                pack_bf16x2(acc[8 * i + 4] * inv_l, acc[8 * i + 5] * inv_l),
                                pack_bf16x2(acc[8 * i + 6] * inv_l, acc[8 * i + 7] * inv_l));
        }
      }
      if (LSE != nullptr && q_row < N)
        LSE[static_cast<size_t>(bh) * N + q_row] = m * kLn2 + logf(l);
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

cudaError_t launch_forward_bf16(const FwdMaps& maps, void* o, float* lse, int B, int H,
                                int N, float scale, int causal, cudaStream_t stream,
                                const TimingEvents& ev) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int BH = B * H;
  const int nq = (N + BM - 1) / BM;
  const float scale_log2 = scale * 1.4426950408889634f;
  if (ev.before) cudaEventRecord(ev.before, stream);
  fwd_bf16_kernel<<<dim3(nq * BH), dim3(NTHREADS), SMEM_BYTES, stream>>>(
      maps.q, maps.k, maps.v, static_cast<__nv_bfloat16*>(o), lse, BH, N, scale_log2, causal);
  cudaError_t e = cudaGetLastError();
  if (ev.after) cudaEventRecord(ev.after, stream);
  return e;
}

int status_forward_bf16(bool clear) {
  int s = 0;
  cudaMemcpyFromSymbol(&s, g_status_fwd_bf16, sizeof(int));
  if (clear && s != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_status_fwd_bf16, &zero, sizeof(int));
  }
  return s;
}

}  // namespace fa
