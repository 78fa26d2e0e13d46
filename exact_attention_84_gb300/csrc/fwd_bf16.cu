// fwd_bf16.cu -- fused exact-attention forward for bf16 on sm_103a.
//
// Method ("FlashAttention ontleed", sections "Tiling en Online Softmax" and
// "Algoritmische kern in pseudocode"; "03. FlashAttention", section
// "FlashAttention v1", "Mecanisme"): Q blocks stay on chip while K_j / V_j
// tiles stream past them.  Per tile and Q block:
//   S = Q K_j^T                      (tensor cores, fp32 accumulator in TMEM)
//   m_new = max(m, rowmax(S*scale))  (softmax warps, registers)
//   P = exp(S*scale - m_new)         (bf16, written back into TMEM)
//   l = l e^(m - m_new) + rowsum(P)
//   O = diag(e^(m - m_new)) O + P V_j   (rescale in TMEM, MMA accumulates)
// and after the last tile O / l and LSE = m + ln(l) go to HBM once.  The
// N x N score matrix never leaves the chip (Lensa ML "FlashAttention",
// step 3: 0 B of S written).
//
// GB300 mapping (the pages' A100/H100 designs are prior art only):
//   * One thread block owns two 128-row Q blocks (A and B) that share every
//     K/V tile.  Tiles are 128 keys; TMA streams K_j and V_j (128-byte
//     swizzled 64-column boxes) into a 4-slot shared-memory ring.
//   * TMEM (512 columns): S_A, S_B (128 each) and O_A, O_B (128 each).  The
//     softmax writes P as packed bf16 over the first 64 columns of its S
//     buffer, and the P.V product takes P straight from TMEM (A operand in
//     tensor memory), so only V is read from shared memory for it.
//   * Warps 0-3 run the softmax of block A, warps 4-7 that of block B (one
//     thread per row = TMEM lane); warp 8 issues TMA; warp 9 allocates TMEM
//     and issues every tcgen05.mma from one thread, interleaving the two
//     blocks: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), ... so one block's
//     softmax overlaps the other block's products.
//   * The arrival of S(j) implies PV(j-1) of the same block has completed
//     (one thread issues them in order and tcgen05.commit tracks all earlier
//     products), so the softmax may rescale O in TMEM right then.  A row's
//     reference maximum is only raised when the new maximum exceeds it by
//     more than 8 (log2 units); otherwise the old reference is kept and the
//     exponentials stay below 2^8.  O / l and LSE = m + ln(l) use the same
//     reference, so the result is unchanged while most O rescales are skipped.
// Causal: key tiles above the diagonal are skipped; only diagonal tiles (and
// a ragged last tile) are masked element-wise.  Heavy (late) Q blocks are
// scheduled first.
// Grouped query heads ("FlashAttention ontleed", "Interactie met de
// KV-cache": several query heads share one key/value head): query head
// b*Hq + h reads key/value head b*Hkv + h/g, which is (b*Hq + h) / g since
// Hq = g*Hkv; consecutive thread blocks take consecutive query heads, so the
// g heads of a group read the same K/V tiles close together in time (L2).
// Sliding window ("03. FlashAttention", "Variantes et extensions": only keys
// inside the window): query i sees keys i-w+1 .. i.  Each Q block starts at
// the first key tile that any of its rows sees; tiles that cut through the
// window's lower edge are masked element-wise like diagonal tiles.
#include <cfloat>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ int g_status_fwd_bf16;

constexpr int BM = 128;                 // query rows per Q block (TMEM lanes)
constexpr int BN = 128;                 // keys per tile
constexpr int HD = 128;                 // head dimension
constexpr int SLOTS = 4;                // K/V ring slots (each one 128x128 bf16 tile)
constexpr uint32_t TILE_BYTES = BM * HD * 2;        // 32 KiB
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;     // 128 rows x 64 columns

constexpr uint32_t OFF_QA = 0;
constexpr uint32_t OFF_QB = OFF_QA + TILE_BYTES;
constexpr uint32_t OFF_SLOT = OFF_QB + TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_SLOT + SLOTS * TILE_BYTES;
// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_FULL = 1;                  // + slot
constexpr int B_EMPTY = B_FULL + SLOTS;    // + slot
constexpr int B_SFULL = B_EMPTY + SLOTS;   // + block (A = 0, B = 1)
constexpr int B_PFULL = B_SFULL + 2;       // + block
constexpr int B_ODONE = B_PFULL + 2;       // + block
constexpr int NBAR = B_ODONE + 2;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;          // + 128 * block
constexpr uint32_t TM_O = 256;        // + 128 * block

constexpr int NTHREADS = 320;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// S = Q K^T: A = Q (K-major), B = K tile (K-major), M = N = 128.
constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
// O += P V: A = P (in TMEM), B = V tile, whose rows run along the reduction
// (key) axis with d contiguous: MN-major.
constexpr uint32_t IDESC_O = idesc_bf16(BM, HD, false, true);

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) {
  return base + OFF_BAR + 8u * static_cast<uint32_t>(i);
}

struct Ctx {
  uint32_t sbase;
  volatile int* abort;
  __device__ bool wait(int bar, uint32_t parity) const {
    return mbar_wait(bar_addr(sbase, bar), parity, abort, &g_status_fwd_bf16);
  }
};

// S = Q K^T for Q block `blk` against the K tile in `kslot`: 8 k-steps of
// 16 along d, both operands K-major (128-byte rows, two 64-column boxes).
__device__ __forceinline__ void issue_s(const Ctx& c, uint32_t tmem, int blk, uint32_t kslot) {
  const uint64_t qd = sdesc_sw128(c.sbase + (blk ? OFF_QB : OFF_QA), 16, 1024);
  const uint64_t kd = sdesc_sw128(c.sbase + OFF_SLOT + kslot * TILE_BYTES, 16, 1024);
  uint64_t a[8], b[8];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint64_t off = ((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4;   // descriptor units
    a[kk] = qd + off;
    b[kk] = kd + off;
  }
  mma_ss_batch8(tmem + TM_S + 128 * blk, a, b, IDESC_S, 0u);
}

// O (+)= P V for Q block `blk`: P packed in TMEM (16 keys = 8 columns per
// step), V tile MN-major (16 key rows = 2048 bytes per step).
__device__ __forceinline__ void issue_pv(const Ctx& c, uint32_t tmem, int blk, uint32_t vslot,
                                         bool first) {
  const uint64_t vd = sdesc_sw128(c.sbase + OFF_SLOT + vslot * TILE_BYTES, HALF_BYTES, 1024);
  uint32_t a[8];
  uint64_t b[8];
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    a[kk] = tmem + TM_S + 128 * blk + kk * 8;
    b[kk] = vd + ((kk * 2048) >> 4);
  }
  mma_ts_batch8(tmem + TM_O + 128 * blk, a, b, IDESC_O, first ? 0u : 1u);
}

// kWindow: a sliding window is applied (window >= 1); the plain instantiation
// carries none of its bookkeeping.
template <bool kWindow>
__global__ void __launch_bounds__(NTHREADS, 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                float* __restrict__ LSE, int BH, int N, float scale_log2, int causal,
                int group, int window) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const Ctx ctx{sbase, abort_flag};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int npair = (N + 2 * BM - 1) / (2 * BM);
  const int nkv = (N + BN - 1) / BN;
  const int pair = causal ? (npair - 1 - static_cast<int>(blockIdx.x) / BH)
                          : (static_cast<int>(blockIdx.x) / BH);
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int bkv = bh / group;                   // key/value head of this query head
  // key tiles [lo, nt) needed by Q block A (tile 2*pair) and B (tile 2*pair + 1)
  const int ntA = causal ? min(2 * pair + 1, nkv) : nkv;
  const int ntB = causal ? min(2 * pair + 2, nkv) : nkv;
  const int loA = kWindow ? max(0, 2 * pair * BM - window + 1) / BN : 0;
  const int loB = kWindow ? min(max(0, (2 * pair + 1) * BM - window + 1) / BN, ntB - 1) : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar_addr(sbase, B_QFULL), 1);
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(bar_addr(sbase, B_FULL + s), 1);
      mbar_init(bar_addr(sbase, B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_addr(sbase, B_SFULL + b), 1);
      mbar_init(bar_addr(sbase, B_PFULL + b), 4);
      mbar_init(bar_addr(sbase, B_ODONE + b), 1);
    }
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
      const uint32_t qf = bar_addr(sbase, B_QFULL);
      const int q0 = pair * 2 * BM;
      mbar_arrive_expect_tx(qf, 2 * TILE_BYTES);
      tma_load_3d(sbase + OFF_QA, &tmQ, qf, 0, q0, bh);
      tma_load_3d(sbase + OFF_QA + HALF_BYTES, &tmQ, qf, 64, q0, bh);
      tma_load_3d(sbase + OFF_QB, &tmQ, qf, 0, q0 + BM, bh);
      tma_load_3d(sbase + OFF_QB + HALF_BYTES, &tmQ, qf, 64, q0 + BM, bh);
      bool ok = true;
      int cnt = 0;
      for (int j = loA; j < ntB && ok; ++j) {
        for (int which = 0; which < 2 && ok; ++which, ++cnt) {
          const int slot = cnt % SLOTS;
          if (cnt >= SLOTS && !ctx.wait(B_EMPTY + slot, ((cnt / SLOTS) - 1) & 1)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_addr(sbase, B_FULL + slot);
          const uint32_t dst = sbase + OFF_SLOT + slot * TILE_BYTES;
          const CUtensorMap* map = which ? &tmV : &tmK;
          mbar_arrive_expect_tx(fb, TILE_BYTES);
          tma_load_3d(dst, map, fb, 0, j * BN, bkv);
          tma_load_3d(dst + HALF_BYTES, map, fb, 64, j * BN, bkv);
        }
      }
    }
    __syncwarp();
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Tiles are numbered from loA: K_j sits in slot (2t) % SLOTS and V_j in
      // (2t+1) % SLOTS with t = j - loA; the n-th fill of a slot completes
      // phase n of its FULL barrier.  Block A works on tiles [loA, ntA) and
      // block B on [loB, ntB), with loB <= loA + 1 and ntB >= ntA, so B takes
      // every tile after the first.
      auto full_k = [&](int j) {
        const int t = j - loA;
        return ctx.wait(B_FULL + (2 * t) % SLOTS, ((2 * t) / SLOTS) & 1);
      };
      auto full_v = [&](int j) {
        const int t = j - loA;
        return ctx.wait(B_FULL + (2 * t + 1) % SLOTS, ((2 * t + 1) / SLOTS) & 1);
      };
      auto active_a = [&](int j) { return j < ntA; };
      auto active_b = [&](int j) { return j >= loB; };
      bool ok = ctx.wait(B_QFULL, 0) && full_k(loA);
      if (ok) {
        tc_fence_after();
        issue_s(ctx, tmem, 0, 0);
        mma_commit(bar_addr(sbase, B_SFULL + 0));
        if (active_b(loA)) {
          issue_s(ctx, tmem, 1, 0);
          mma_commit(bar_addr(sbase, B_SFULL + 1));
        }
        mma_commit(bar_addr(sbase, B_EMPTY + 0));
      }
      for (int j = loA; j < ntB && ok; ++j) {
        const int t = j - loA;
        const int vslot = (2 * t + 1) % SLOTS;
        const int kslot_next = (2 * t + 2) % SLOTS;
        bool v_ready = false, k_next_ready = false;
        if (active_a(j)) {
          ok = ctx.wait(B_PFULL + 0, (j - loA) & 1) && full_v(j);
          if (!ok) break;
          v_ready = true;
          tc_fence_after();
          issue_pv(ctx, tmem, 0, vslot, j == loA);
          if (j == ntA - 1) mma_commit(bar_addr(sbase, B_ODONE + 0));
        }
        if (active_a(j + 1)) {
          ok = full_k(j + 1);
          if (!ok) break;
          k_next_ready = true;
          tc_fence_after();
          issue_s(ctx, tmem, 0, kslot_next);
          mma_commit(bar_addr(sbase, B_SFULL + 0));
        }
        if (active_b(j)) {
          ok = ctx.wait(B_PFULL + 1, (j - loB) & 1) && (v_ready || full_v(j));
          if (!ok) break;
          tc_fence_after();
          issue_pv(ctx, tmem, 1, vslot, j == loB);
          if (j == ntB - 1) mma_commit(bar_addr(sbase, B_ODONE + 1));
        }
        mma_commit(bar_addr(sbase, B_EMPTY + vslot));
        if (j + 1 < ntB) {
          ok = k_next_ready || full_k(j + 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(ctx, tmem, 1, kslot_next);
          mma_commit(bar_addr(sbase, B_SFULL + 1));
          mma_commit(bar_addr(sbase, B_EMPTY + kslot_next));
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int blk = warp >> 2;                    // 0: block A, 1: block B
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;             // row within the Q block
    const int qt = 2 * pair + blk;                // Q tile index (128-row units)
    const int q_row = qt * BM + row;
    const int nt = blk ? ntB : ntA;
    const int lo = blk ? loB : loA;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + TM_S + 128 * blk;
    const uint32_t o_addr = tmem + lane_addr + TM_O + 128 * blk;
    float m = -INFINITY;                          // reference max, log2 units
    float l = 0.f;                                // running sum
    bool ok = true;

    for (int j = lo; j < nt; ++j) {
      if (!ctx.wait(B_SFULL + blk, (j - lo) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[BN];
      {
        uint32_t r[BN];
        tmem_ld128(s_addr, r);                    // the row's 128 scores in one round trip
#pragma unroll
        for (int i = 0; i < BN; ++i) s[i] = __uint_as_float(r[i]);
      }
      // mask: causal diagonal tile, keys past the end of the sequence, or a
      // tile that cuts through the window's lower edge
      const bool diag = causal && (j == qt);
      const bool ragged = (j == nkv - 1) && (N % BN != 0);
      const bool wedge = kWindow && j * BN < qt * BM + BM - window;
      if (diag || ragged || wedge) {
        // keys visible to this row: key_lo <= key <= key_hi, tested as one
        // unsigned compare per key
        const int key_hi = causal ? min(q_row, N - 1) : (N - 1);
        const int key_lo = kWindow ? q_row - window + 1 : 0;
        const uint32_t span = static_cast<uint32_t>(key_hi - key_lo);
        const int rel0 = j * BN - key_lo;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (static_cast<uint32_t>(rel0 + c) > span) s[c] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) mx = fmaxf(mx, s[c]);
      mx *= scale_log2;
      // Raise the reference max only when the new one exceeds it by more
      // than the threshold (always on the first tile, where m = -inf).
      float corr = 1.f;
      if (mx > m + kRescaleThreshold) {
        corr = fast_exp2(m - mx);                 // 0 on the first tile
        m = mx;
      }
      const bool rescale_o = (j > lo) && __any_sync(0xffffffffu, corr != 1.f);
      // A row that has seen no visible key yet (only possible with a window)
      // keeps m = -inf; it uses 0 as the exponent reference so its masked
      // scores give exp2(-inf) = 0, not NaN.
      const float mref = (kWindow && m == -INFINITY) ? 0.f : m;
      float rs = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float p0 = fast_exp2(fmaf(s[2 * c], scale_log2, -mref));
        const float p1 = fast_exp2(fmaf(s[2 * c + 1], scale_log2, -mref));
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * corr + rs;
      // P (packed bf16) over the first 64 columns of this block's S buffer
      tmem_st32(s_addr, *reinterpret_cast<const uint32_t(*)[32]>(pk));
      tmem_st32(s_addr + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
      if (rescale_o) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
          tmem_st32(o_addr + c * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_PFULL + blk));
    }

    if (ok && ctx.wait(B_ODONE + blk, 0)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = O + (static_cast<size_t>(bh) * N + q_row) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(o_addr + c * 32, r);
        if (q_row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(
                pack_bf16x2(__uint_as_float(r[8 * i]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l),
                pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l),
                pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l),
                pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l));
        }
      }
      if (LSE != nullptr && q_row < N)
        LSE[static_cast<size_t>(bh) * N + q_row] = m * kLn2 + logf(l);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_forward_bf16(const FwdMaps& maps, void* o, float* lse, int B, int H,
                                int Hkv, int N, float scale, int causal, int window,
                                cudaStream_t stream, const TimingEvents& ev) {
  static bool attr_set = false;
  if (!attr_set) {
    for (auto fn : {fwd_bf16_kernel<false>, fwd_bf16_kernel<true>}) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(SMEM_BYTES));
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  const int BH = B * H;
  const int npair = (N + 2 * BM - 1) / (2 * BM);
  const float scale_log2 = scale * 1.4426950408889634f;
  if (ev.before) cudaEventRecord(ev.before, stream);
  auto kernel = window > 0 ? fwd_bf16_kernel<true> : fwd_bf16_kernel<false>;
  kernel<<<dim3(npair * BH), dim3(NTHREADS), SMEM_BYTES, stream>>>(
      maps.q, maps.k, maps.v, static_cast<__nv_bfloat16*>(o), lse, BH, N, scale_log2, causal,
      H / Hkv, window);
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
