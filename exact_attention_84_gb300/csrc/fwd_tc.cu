// fwd_tc.cu -- fused exact-attention forward on the tcgen05 tensor cores of
// sm_103a, for bf16 and for fp8 (e4m3) inputs.
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
// ALiBi ("03. FlashAttention", "Variantes et extensions": the linear bias
// fused into the kernel): -slope_h * |i - j| is added to each scaled score
// right after it leaves TMEM, before the mask and the online softmax.
// FP8 ("03. FlashAttention", "FlashAttention v3": the FP8 format as a
// hardware lever): Q, K, V in e4m3 with per-tensor descale factors; the
// same loop runs kind::f8f6f4 products (K = 32 per instruction, twice the
// bf16 rate) with fp32 accumulation.  P is rounded to e4m3 (values <= 2^8
// thanks to the lazy rescale, inside e4m3's range) and kept in TMEM as four
// bytes per column; V is read through a transposed copy so both operands of
// P V are K-major.  scale * q_descale * k_descale multiplies the scores and
// v_descale the output; O is written in bf16.
#include <cfloat>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ int g_status_fwd;

constexpr int BM = 128;                 // query rows per Q block (TMEM lanes)
constexpr int BN = 128;                 // keys per tile
constexpr int HD = 128;                 // head dimension

// Shared-memory layout for one element type: two Q blocks, a ring of K/V
// tile slots, the mbarriers and a few words of control state.
template <uint32_t kTileBytes, int kSlots>
struct FwdLayout {
  static constexpr uint32_t TILE = kTileBytes;   // one 128 x 128 tile
  static constexpr int SLOTS = kSlots;           // K/V ring slots
  static constexpr uint32_t OFF_QA = 0;
  static constexpr uint32_t OFF_QB = OFF_QA + TILE;
  static constexpr uint32_t OFF_SLOT = OFF_QB + TILE;
  static constexpr uint32_t OFF_BAR = OFF_SLOT + SLOTS * TILE;
  // barrier indices
  static constexpr int B_QFULL = 0;
  static constexpr int B_FULL = 1;                  // + slot
  static constexpr int B_EMPTY = B_FULL + SLOTS;    // + slot
  static constexpr int B_SFULL = B_EMPTY + SLOTS;   // + block (A = 0, B = 1)
  static constexpr int B_PFULL = B_SFULL + 2;       // + block
  static constexpr int B_ODONE = B_PFULL + 2;       // + block
  static constexpr int B_OSTG = B_ODONE + 2;        // + block: O staged (softmax warps arrive)
  static constexpr int B_XCHG = B_OSTG + 2;         // + 4 block + quadrant: row parts met
  static constexpr int NBAR = B_XCHG + 8;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // partial row maxima / sums of the two parts of each row (two softmax
  // warps per row): [parity][block][part][row] floats
  static constexpr uint32_t OFF_XCHG = (OFF_MISC + 16 + 15) & ~15u;
  static constexpr uint32_t SMEM_BYTES = OFF_XCHG + 2 * 2 * 2 * 128 * 4 + 1024;   // + alignment slack
  static_assert(SMEM_BYTES <= 227u * 1024u, "forward shared memory exceeds the per-block limit");
};

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;          // + 128 * block
constexpr uint32_t TM_O = 256;        // + 128 * block

// Softmax warps per row: two for the ALiBi variants, whose heavier per-score
// work makes the softmax the longer side of the ping-pong (measured 7%
// faster), one otherwise (two measured 5% slower there: the MMA-issuing warp
// then shares its sub-partition with four softmax warps instead of two).
// Warps: 8 KH softmax, then the TMA producer, then the MMA issuer.
template <bool kAlibi>
__host__ __device__ constexpr int row_warps() { return kAlibi ? 2 : 1; }
template <bool kAlibi>
__host__ __device__ constexpr int fwd_threads() { return 32 * (8 * row_warps<kAlibi>() + 2); }

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// Block order: the K and V of the heads whose blocks run together.
constexpr long long kFwdGroupBytes = 32ll << 20;

// ---- bf16: 128 x 128 tiles as two 64-column (128-byte) swizzled boxes.
struct Bf16 : FwdLayout<BM * HD * 2, 4> {
  static constexpr uint32_t HALF = TILE / 2;        // 128 rows x 64 columns
  // S = Q K^T: A = Q (K-major), B = K tile (K-major), M = N = 128.
  static constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
  // O += P V: A = P (in TMEM), B = V tile, whose rows run along the
  // reduction (key) axis with d contiguous: MN-major.
  static constexpr uint32_t IDESC_O = idesc_bf16(BM, HD, false, true);
  static constexpr int P_COLS = BN / 2;             // packed P: 2 keys per TMEM column
  static constexpr bool kSplitChains = false;       // row max as one chain
  // O leaves through the block's Q tile (same two swizzled boxes) and one
  // bulk tensor store, instead of per-row stores from every thread.
  static constexpr bool kStoreTma = true;

  // a 128-row tile of Q or K (rows `row`.., head `head`)
  __device__ static void load_rows(uint32_t dst, const CUtensorMap* map, uint32_t bar, int row,
                                   int head) {
    tma_load_3d(dst, map, bar, 0, row, head);
    tma_load_3d(dst + HALF, map, bar, 64, row, head);
  }
  // the V tile of keys `key`.. (V itself, [keys][d])
  __device__ static void load_v(uint32_t dst, const CUtensorMap* map, uint32_t bar, int key,
                                int head) {
    load_rows(dst, map, bar, key, head);
  }
  // S = Q K^T: 8 k-steps of 16 along d, both operands K-major.
  __device__ static void issue_s(uint32_t d, uint32_t q_smem, uint32_t k_smem) {
    const uint64_t qd = sdesc_sw128(q_smem, 16, 1024);
    const uint64_t kd = sdesc_sw128(k_smem, 16, 1024);
    uint64_t a[8], b[8];
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const uint64_t off = ((kk >> 2) * HALF + (kk & 3) * 32) >> 4;   // descriptor units
      a[kk] = qd + off;
      b[kk] = kd + off;
    }
    mma_ss_batch8(d, a, b, IDESC_S, 0u);
  }
  // O (+)= P V: P packed in TMEM (16 keys = 8 columns per step), V tile
  // MN-major (16 key rows = 2048 bytes per step).
  __device__ static void issue_pv(uint32_t d, uint32_t p_tmem, uint32_t v_smem, bool first) {
    const uint64_t vd = sdesc_sw128(v_smem, HALF, 1024);
    uint32_t a[8];
    uint64_t b[8];
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
      a[kk] = p_tmem + kk * 8;
      b[kk] = vd + ((kk * 2048) >> 4);
    }
    mma_ts_batch8(d, a, b, IDESC_O, first ? 0u : 1u);
  }
  // four consecutive probabilities into the packed P words
  __device__ static void pack4(uint32_t* pk, int c4, float p0, float p1, float p2, float p3) {
    pk[2 * c4] = pack_bf16x2(p0, p1);
    pk[2 * c4 + 1] = pack_bf16x2(p2, p3);
  }
};

// ---- fp8 (e4m3): a 128 x 128 tile is one 128-byte swizzled box.  V is read
// from a transposed copy V^T [d][keys], so the P V product takes both
// operands K-major (keys contiguous), the layout every 8-bit operand shares.
struct Fp8 : FwdLayout<BM * HD, 8> {
  static constexpr uint32_t IDESC_S = idesc_e4m3(BM, BN);
  static constexpr uint32_t IDESC_O = idesc_e4m3(BM, HD);
  static constexpr int P_COLS = BN / 4;             // packed P: 4 keys per TMEM column
  static constexpr bool kSplitChains = true;        // row max as 8 parallel chains
  static constexpr bool kStoreTma = false;          // a Q tile (16 KB) cannot hold bf16 O

  __device__ static void load_rows(uint32_t dst, const CUtensorMap* map, uint32_t bar, int row,
                                   int head) {
    tma_load_3d(dst, map, bar, 0, row, head);
  }
  // V^T tile: rows = the 128 head-dimension entries, columns = keys `key`..
  __device__ static void load_v(uint32_t dst, const CUtensorMap* map, uint32_t bar, int key,
                                int head) {
    tma_load_3d(dst, map, bar, key, 0, head);
  }
  // S = Q K^T: 4 k-steps of 32 along d (32 bytes each), both K-major.
  __device__ static void issue_s(uint32_t d, uint32_t q_smem, uint32_t k_smem) {
    const uint64_t qd = sdesc_sw128(q_smem, 16, 1024);
    const uint64_t kd = sdesc_sw128(k_smem, 16, 1024);
    uint64_t a[4], b[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      a[kk] = qd + ((kk * 32) >> 4);
      b[kk] = kd + ((kk * 32) >> 4);
    }
    mma_f8_ss_batch4(d, a, b, IDESC_S, 0u);
  }
  // O (+)= P V: P packed in TMEM (32 keys = 8 columns per step), V^T K-major
  // (32 keys = 32 bytes per step).
  __device__ static void issue_pv(uint32_t d, uint32_t p_tmem, uint32_t v_smem, bool first) {
    const uint64_t vd = sdesc_sw128(v_smem, 16, 1024);
    uint32_t a[4];
    uint64_t b[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      a[kk] = p_tmem + kk * 8;
      b[kk] = vd + ((kk * 32) >> 4);
    }
    mma_f8_ts_batch4(d, a, b, IDESC_O, first ? 0u : 1u);
  }
  __device__ static void pack4(uint32_t* pk, int c4, float p0, float p1, float p2, float p3) {
    pk[c4] = pack_e4m3x4(p0, p1, p2, p3);
  }
};

template <class T>
struct Ctx {
  uint32_t sbase;
  volatile int* abort;
  __device__ uint32_t bar(int i) const {
    return sbase + T::OFF_BAR + 8u * static_cast<uint32_t>(i);
  }
  __device__ bool wait(int i, uint32_t parity) const {
    return mbar_wait(bar(i), parity, abort, &g_status_fwd);
  }
};

// The kernel body for element type T.  kWindow: a sliding window is applied
// (window >= 1); kAlibi: the ALiBi bias -slope_h * |i - j| is added to the
// scaled scores (alibi[h] = slope of query head h, h = bh % heads).  The
// plain instantiation carries none of their bookkeeping.  out_scale
// multiplies O at the end (the fp8 V descale; 1 for bf16).
template <class T, bool kWindow, bool kAlibi>
__device__ __forceinline__ void fwd_body(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                         const CUtensorMap* tmV, const CUtensorMap* tmO,
                                         __nv_bfloat16* __restrict__ O,
                                         float* __restrict__ LSE, int BH, int N,
                                         float scale_log2, float out_scale, int causal,
                                         int group, int window, const float* __restrict__ alibi,
                                         int heads, int nsplit, int head_group) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + T::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 4);
  const Ctx<T> ctx{sbase, abort_flag};
  constexpr int SLOTS = T::SLOTS;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int KH = row_warps<kAlibi>();       // softmax warps per row
  constexpr int HC = BN / KH;                   // key columns of a tile per softmax warp
  constexpr int WARP_TMA = 8 * KH;
  constexpr int WARP_MMA = 8 * KH + 1;

  const int npair = (N + 2 * BM - 1) / (2 * BM);
  const int nkv = (N + BN - 1) / BN;
  // Work items are (Q pair, head); the last nsplit items (non-causal only)
  // are split into two thread blocks of one Q tile each, so that a last
  // wave of items that would keep few SMs busy for a whole item runs as
  // twice as many half-length blocks.
  const int nfull = npair * BH - nsplit;
  const int bid = static_cast<int>(blockIdx.x);
  const int item = bid < nfull ? bid : nfull + (bid - nfull) / 2;
  const bool has_b = bid < nfull;                 // this block runs Q block B too
  // Items go in groups of head_group query heads (whole key/value heads), so
  // the blocks in flight share a few heads' K and V and re-read them from L2
  // rather than HBM; within a group Q pairs go heavy-first (causal), heads
  // fastest.
  const int per_group = head_group * npair;
  const int hgrp = item / per_group;
  const int gsize = min(head_group, BH - hgrp * head_group);
  const int rem = item - hgrp * per_group;
  const int pair = causal ? (npair - 1 - rem / gsize) : (rem / gsize);
  const int bh = hgrp * head_group + rem % gsize;
  // Q tile of block A: the pair's first, or for a split item its own tile
  const int qt_a = 2 * pair + (has_b ? 0 : (bid - nfull) & 1);
  const int bkv = bh / group;                   // key/value head of this query head
  // key tiles [lo, nt) needed by Q block A (tile 2*pair) and B (tile 2*pair + 1)
  const int ntA = causal ? min(2 * pair + 1, nkv) : nkv;
  const int ntB = causal ? min(2 * pair + 2, nkv) : nkv;
  const int loA = kWindow ? max(0, 2 * pair * BM - window + 1) / BN : 0;
  const int loB = kWindow ? min(max(0, (2 * pair + 1) * BM - window + 1) / BN, ntB - 1) : 0;

  if (threadIdx.x == 0) {
    mbar_init(ctx.bar(T::B_QFULL), 1);
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(ctx.bar(T::B_FULL + s), 1);
      mbar_init(ctx.bar(T::B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(ctx.bar(T::B_SFULL + b), 1);
      mbar_init(ctx.bar(T::B_PFULL + b), 4 * KH);
      mbar_init(ctx.bar(T::B_ODONE + b), 1);
      mbar_init(ctx.bar(T::B_OSTG + b), 4 * KH);
    }
    for (int x = 0; x < 8; ++x) mbar_init(ctx.bar(T::B_XCHG + x), 2);
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
      prefetch_tmap(tmQ);
      prefetch_tmap(tmK);
      prefetch_tmap(tmV);
      if constexpr (T::kStoreTma) prefetch_tmap(tmO);
      const uint32_t qf = ctx.bar(T::B_QFULL);
      const int q0 = qt_a * BM;
      mbar_arrive_expect_tx(qf, (has_b ? 2 : 1) * T::TILE);
      T::load_rows(sbase + T::OFF_QA, tmQ, qf, q0, bh);
      if (has_b) T::load_rows(sbase + T::OFF_QB, tmQ, qf, q0 + BM, bh);
      bool ok = true;
      int cnt = 0;
      // key tiles in processing order: the last one (the diagonal one when
      // causal) first, down to loA
      for (int j = ntB - 1; j >= loA && ok; --j) {
        for (int which = 0; which < 2 && ok; ++which, ++cnt) {
          const int slot = cnt % SLOTS;
          if (cnt >= SLOTS && !ctx.wait(T::B_EMPTY + slot, ((cnt / SLOTS) - 1) & 1)) {
            ok = false;
            break;
          }
          const uint32_t fb = ctx.bar(T::B_FULL + slot);
          const uint32_t dst = sbase + T::OFF_SLOT + slot * T::TILE;
          mbar_arrive_expect_tx(fb, T::TILE);
          if (which)
            T::load_v(dst, tmV, fb, j * BN, bkv);
          else
            T::load_rows(dst, tmK, fb, j * BN, bkv);
        }
      }
    }
    __syncwarp();
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Key tiles go in decreasing order: step t works on tile ntB - 1 - t,
      // K in slot (2t) % SLOTS and V in (2t+1) % SLOTS; the n-th fill of a
      // slot completes phase n of its FULL barrier.  Block B (the later Q
      // tile) works on steps [0, tB1], block A on [tA0, nsteps): under the
      // causal mask the step that only block B needs (its diagonal tile) is
      // the first one, where the pipeline is filling anyway, and both blocks
      // end together on tile loA instead of block A's softmax idling through
      // block B's last tile.
      const int nsteps = ntB - loA;
      const int tA0 = ntB - ntA;
      const int tB1 = ntB - 1 - loB;
      auto full_k = [&](int t) {
        return ctx.wait(T::B_FULL + (2 * t) % SLOTS, ((2 * t) / SLOTS) & 1);
      };
      auto full_v = [&](int t) {
        return ctx.wait(T::B_FULL + (2 * t + 1) % SLOTS, ((2 * t + 1) / SLOTS) & 1);
      };
      auto active_a = [&](int t) { return t >= tA0 && t < nsteps; };
      auto active_b = [&](int t) { return has_b && t <= tB1; };
      bool ok = ctx.wait(T::B_QFULL, 0) && full_k(0);
      if (ok) {
        tc_fence_after();
        if (active_a(0)) {
          T::issue_s(tmem + TM_S, sbase + T::OFF_QA, sbase + T::OFF_SLOT);
          mma_commit(ctx.bar(T::B_SFULL + 0));
        }
        if (active_b(0)) {
          T::issue_s(tmem + TM_S + 128, sbase + T::OFF_QB, sbase + T::OFF_SLOT);
          mma_commit(ctx.bar(T::B_SFULL + 1));
        }
        mma_commit(ctx.bar(T::B_EMPTY + 0));
      }
      for (int t = 0; t < nsteps && ok; ++t) {
        const int vslot = (2 * t + 1) % SLOTS;
        const int kslot_next = (2 * t + 2) % SLOTS;
        bool v_ready = false, k_next_ready = false;
        if (active_a(t)) {
          ok = ctx.wait(T::B_PFULL + 0, (t - tA0) & 1) && full_v(t);
          if (!ok) break;
          v_ready = true;
          tc_fence_after();
          T::issue_pv(tmem + TM_O, tmem + TM_S, sbase + T::OFF_SLOT + vslot * T::TILE, t == tA0);
          if (t == nsteps - 1) mma_commit(ctx.bar(T::B_ODONE + 0));
        }
        if (active_a(t + 1)) {
          ok = full_k(t + 1);
          if (!ok) break;
          k_next_ready = true;
          tc_fence_after();
          T::issue_s(tmem + TM_S, sbase + T::OFF_QA, sbase + T::OFF_SLOT + kslot_next * T::TILE);
          mma_commit(ctx.bar(T::B_SFULL + 0));
        }
        if (active_b(t)) {
          ok = ctx.wait(T::B_PFULL + 1, t & 1) && (v_ready || full_v(t));
          if (!ok) break;
          tc_fence_after();
          T::issue_pv(tmem + TM_O + 128, tmem + TM_S + 128, sbase + T::OFF_SLOT + vslot * T::TILE, t == 0);
          if (t == tB1) mma_commit(ctx.bar(T::B_ODONE + 1));
        }
        mma_commit(ctx.bar(T::B_EMPTY + vslot));
        if (t + 1 < nsteps) {
          ok = k_next_ready || full_k(t + 1);
          if (!ok) break;
          if (active_b(t + 1)) {
            tc_fence_after();
            T::issue_s(tmem + TM_S + 128, sbase + T::OFF_QB,
                       sbase + T::OFF_SLOT + kslot_next * T::TILE);
            mma_commit(ctx.bar(T::B_SFULL + 1));
          }
          mma_commit(ctx.bar(T::B_EMPTY + kslot_next));
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // KH warps per row: warp w works on block w / (4 KH) (A or B), on key
    // part (w >> 2) % KH of every tile (HC = 128 / KH of its keys) and on
    // the rows of TMEM lane quadrant w & 3.  With two parts the halves of a
    // row share its running maximum (one exchange through shared memory per
    // tile, so they take identical rescaling decisions) and each keeps its
    // own part of the row sum until the end.
    const int blk = warp / (4 * KH);              // 0: block A, 1: block B
    const int half = (warp >> 2) % KH;            // key part of this warp
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;             // row within the Q block
    const bool live = blk == 0 || has_b;          // block B idles in a split item
    const int qt = qt_a + blk;                    // Q tile index (128-row units)
    const int q_row = qt * BM + row;
    const int lo = blk ? loB : loA;
    const int nt = live ? (blk ? ntB : ntA) : lo;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + TM_S + 128 * blk;
    const uint32_t o_addr = tmem + lane_addr + TM_O + 128 * blk;
    constexpr int OC = HD / 32 / KH;              // 32-column chunks of O per warp
    float* xchg = reinterpret_cast<float*>(smem + T::OFF_XCHG);
    auto xslot = [&](int par, int h) { return xchg + ((par * 2 + blk) * 2 + h) * BM + row; };
    const int xbar = T::B_XCHG + blk * 4 + quad;  // the row halves' meeting point
    // Publish this half's value in slot `par`, then read the other half's
    // once both have arrived (phase `phase` of the meeting barrier).
    auto exchange = [&](float mine, int par, int phase, float& theirs) {
      *xslot(par, half) = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(ctx.bar(xbar));
      if (!ctx.wait(xbar, phase & 1)) return false;
      theirs = *xslot(par, half ^ 1);
      return true;
    };
    float m = -INFINITY;                          // reference max, log2 units
    float l = 0.f;                                // running sum (of this key part)
    bool ok = true;
    // ALiBi scales and biases the scores in place; the max and the
    // exponentials then take them as they are.
    const float slope_log2 = kAlibi ? alibi[bh % heads] * 1.4426950408889634f : 0.f;
    const float sl = kAlibi ? 1.f : scale_log2;

    // this block's key tiles, last first (the order the products come in)
    for (int u = 0; u < nt - lo; ++u) {
      const int j = nt - 1 - u;
      if (!ctx.wait(T::B_SFULL + blk, u & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[HC];
      {
        uint32_t r[HC];
        if constexpr (KH == 1)
          tmem_ld128(s_addr, r);                  // the row's 128 scores in one round trip
        else
          tmem_ld64(s_addr + HC * half, r);       // this part's 64 scores
#pragma unroll
        for (int i = 0; i < HC; ++i) s[i] = __uint_as_float(r[i]);
      }
      const int key0 = j * BN + HC * half;        // key of column 0 of this part
      if constexpr (kAlibi) {
        const float d0 = static_cast<float>(key0 - q_row);   // key - query at column 0
        if (causal) {
          // every key the mask leaves has key <= query: -|i - j| = j - i;
          // on packed pairs: s = s scale + (slope c + slope d0)
          const uint64_t base2 = f2pack(slope_log2 * d0, slope_log2 * d0);
          const uint64_t slope2 = f2pack(slope_log2, slope_log2);
          const uint64_t scale2 = f2pack(scale_log2, scale_log2);
#pragma unroll
          for (int c = 0; c < HC; c += 2) {
            const uint64_t bias = f2fma(slope2, f2pack(static_cast<float>(c), static_cast<float>(c + 1)), base2);
            f2unpack(f2fma(f2pack(s[c], s[c + 1]), scale2, bias), s[c], s[c + 1]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < HC; ++c)
            s[c] = fmaf(s[c], scale_log2, -slope_log2 * fabsf(d0 + static_cast<float>(c)));
        }
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
        const int rel0 = key0 - key_lo;
#pragma unroll
        for (int c = 0; c < HC; ++c)
          if (static_cast<uint32_t>(rel0 + c) > span) s[c] = -INFINITY;
      }
      float mx;
      if constexpr (T::kSplitChains) {
        // Row maximum as 8 independent chains: with the faster fp8 products
        // one long chain of dependent max operations leaves the warp waiting
        // on their latency (measured: the bf16 kernel runs faster without).
        float mxp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mxp[k] = s[k];
#pragma unroll
        for (int c = 8; c < HC; c += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k) mxp[k] = fmaxf(mxp[k], s[c + k]);
        mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                   fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
      } else {
        // three-input max: one instruction per two scores (the softmax is
        // bound by instruction issue, so each one saved counts)
        mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < HC; c += 2)
          asm("max.f32 %0, %1, %2, %3;" : "=f"(mx) : "f"(mx), "f"(s[c]), "f"(s[c + 1]));
      }
      if constexpr (KH == 2) {
        float other;
        if (!exchange(mx, u & 1, u, other)) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, other);
      }
      mx *= sl;
      // Raise the reference max only when the new one exceeds it by more
      // than the threshold (always on the first tile, where m = -inf).
      float corr = 1.f;
      if (mx > m + kRescaleThreshold) {
        corr = fast_exp2(m - mx);                 // 0 on the first tile
        m = mx;
      }
      const bool rescale_o = (u > 0) && __any_sync(0xffffffffu, corr != 1.f);
      // A row that has seen no visible key yet (only possible with a window)
      // keeps m = -inf; it uses 0 as the exponent reference so its masked
      // scores give exp2(-inf) = 0, not NaN.
      const float mref = (kWindow && m == -INFINITY) ? 0.f : m;
      // P = exp2(S scale - m) and the row sum
      constexpr int PW = T::P_COLS / KH;          // packed P words of this part
      uint32_t pk[PW];
      // exponent arguments and row sums on packed fp32 pairs: one
      // instruction per two scores (measured +7% on the whole kernel)
      const uint64_t sl2 = f2pack(sl, sl), nm2 = f2pack(-mref, -mref);
      uint64_t acc2 = f2pack(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < HC / 4; ++c) {
        float a0, a1, a2, a3;
        f2unpack(f2fma(f2pack(s[4 * c], s[4 * c + 1]), sl2, nm2), a0, a1);
        f2unpack(f2fma(f2pack(s[4 * c + 2], s[4 * c + 3]), sl2, nm2), a2, a3);
        const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
        const float p2 = fast_exp2(a2), p3 = fast_exp2(a3);
        acc2 = f2add(acc2, f2add(f2pack(p0, p1), f2pack(p2, p3)));
        T::pack4(pk, c, p0, p1, p2, p3);
      }
      float r0, r1;
      f2unpack(acc2, r0, r1);
      l = l * corr + (r0 + r1);
      // Packed P of this part over its share of the first P_COLS columns of
      // the block's S buffer.  With two parts the other one has read its
      // scores from them already: it met this one after its load completed.
      if constexpr (PW >= 32) {
#pragma unroll
        for (int c = 0; c < PW; c += 32)
          tmem_st32(s_addr + PW * half + c, *reinterpret_cast<const uint32_t(*)[32]>(pk + c));
      } else {
        tmem_st16(s_addr + PW * half, pk);
      }
      if (rescale_o) {
#pragma unroll 1
        for (int c = OC * half; c < OC * half + OC; ++c) {
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
      if (lane == 0) mbar_arrive(ctx.bar(T::B_PFULL + blk));
    }

    // With two parts, the row sum of both (one more meeting).
    float l_row = l;
    if constexpr (KH == 2) {
      if (ok && live) {
        float other;
        ok = exchange(l, (nt - lo) & 1, nt - lo, other);
        l_row = l + other;
      }
    }
    if (ok && live && ctx.wait(T::B_ODONE + blk, 0)) {
      tc_fence_after();
      const float inv_l = out_scale / l_row;
      auto pack8 = [&](const uint32_t (&r)[32], int i) {
        return make_uint4(
            pack_bf16x2(__uint_as_float(r[8 * i]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l),
            pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l),
            pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l),
            pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l));
      };
      if constexpr (T::kStoreTma) {
        // Every product of this block has completed, so its Q tile is free:
        // the row goes there in the tile's own swizzled layout (columns
        // 32c.. of the row = 16-byte chunks 4(c&1).. of box c>>1), each warp
        // its OC chunks, and one thread stores both boxes with the bulk
        // tensor engine, which also drops the rows past N.
        const uint32_t stage = blk ? T::OFF_QB : T::OFF_QA;
#pragma unroll 1
        for (int c = OC * half; c < OC * half + OC; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + c * 32, r);
          uint8_t* box = smem + stage + (c >> 1) * T::HALF;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(box + sw128_offset(row, (c & 1) * 4 + i)) = pack8(r, i);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(ctx.bar(T::B_OSTG + blk));
        if (quad == 0 && half == 0 && lane == 0 && ctx.wait(T::B_OSTG + blk, 0)) {
          tma_store_3d(tmO, sbase + stage, 0, qt * BM, bh);
          tma_store_3d(tmO, sbase + stage + T::HALF, 64, qt * BM, bh);
          bulk_commit_group();
          bulk_wait_group_read0();   // the block may exit once the tile has been read
        }
      } else {
        __nv_bfloat16* orow = O + (static_cast<size_t>(bh) * N + q_row) * HD;
#pragma unroll 1
        for (int c = OC * half; c < OC * half + OC; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + c * 32, r);
          if (q_row < N) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = pack8(r, i);
          }
        }
      }
      if (LSE != nullptr && half == 0 && q_row < N)
        LSE[static_cast<size_t>(bh) * N + q_row] = m * kLn2 + logf(l_row);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// kWindow: a sliding window is applied (window >= 1); kAlibi: ALiBi bias.
template <bool kWindow, bool kAlibi>
__global__ void __launch_bounds__(fwd_threads<kAlibi>(), 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                __nv_bfloat16* __restrict__ O, float* __restrict__ LSE, int BH, int N,
                float scale_log2, int causal, int group, int window,
                const float* __restrict__ alibi, int heads, int nsplit, int head_group) {
  fwd_body<Bf16, kWindow, kAlibi>(&tmQ, &tmK, &tmV, &tmO, O, LSE, BH, N, scale_log2, 1.f,
                                  causal, group, window, alibi, heads, nsplit, head_group);
}

// Q, K e4m3 [BH, N, 128]; tmV maps the transposed copy V^T [BH, 128, keys].
template <bool kWindow, bool kAlibi>
__global__ void __launch_bounds__(fwd_threads<kAlibi>(), 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmVt, __nv_bfloat16* __restrict__ O,
               float* __restrict__ LSE, int BH, int N, float scale_log2, float v_descale,
               int causal, int group, int window, const float* __restrict__ alibi, int heads,
               int head_group) {
  fwd_body<Fp8, kWindow, kAlibi>(&tmQ, &tmK, &tmVt, nullptr, O, LSE, BH, N, scale_log2,
                                 v_descale, causal, group, window, alibi, heads, 0, head_group);
}

// V [rows, 128] e4m3 -> V^T [128, ld] per head, 64 keys x 128 columns per
// block.  Rows are staged in shared memory with a 33-word stride; each
// thread then turns 4 keys x 4 columns (four 32-bit words) into 4 words of
// 4 keys each with byte permutes and stores them, 16 threads covering 64
// contiguous bytes of an output row.
__global__ void __launch_bounds__(256) transpose_v_kernel(const uint8_t* __restrict__ v,
                                                          uint8_t* __restrict__ vt, int N,
                                                          int ld) {
  constexpr int KB = 64;                          // keys per block
  constexpr int RW = HD / 4 + 1;                  // shared row stride in words
  __shared__ uint32_t tile[KB * RW];
  const int head = blockIdx.y;
  const int k0 = blockIdx.x * KB;
  const uint8_t* src = v + static_cast<size_t>(head) * N * HD;
  uint8_t* dst = vt + static_cast<size_t>(head) * HD * ld;
  for (int i = threadIdx.x; i < KB * 8; i += blockDim.x) {
    const int r = i >> 3, c = i & 7;              // key row, 16-byte chunk
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + r < N)
      x = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(k0 + r) * HD + c * 16);
    uint32_t* t = tile + r * RW + 4 * c;
    t[0] = x.x;
    t[1] = x.y;
    t[2] = x.z;
    t[3] = x.w;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = lane & 15;                       // 4-key group
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int db = (lane >> 4) + 2 * (warp + 8 * it);   // 4-column group, 0..31
    const uint32_t w0 = tile[(4 * kb + 0) * RW + db];
    const uint32_t w1 = tile[(4 * kb + 1) * RW + db];
    const uint32_t w2 = tile[(4 * kb + 2) * RW + db];
    const uint32_t w3 = tile[(4 * kb + 3) * RW + db];
    // t0 = [w0.b0 w1.b0 w0.b1 w1.b1], t1 = [w0.b2 w1.b2 w0.b3 w1.b3], ...
    const uint32_t t0 = __byte_perm(w0, w1, 0x5140), t1 = __byte_perm(w0, w1, 0x7362);
    const uint32_t t2 = __byte_perm(w2, w3, 0x5140), t3 = __byte_perm(w2, w3, 0x7362);
    const uint32_t col[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                             __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632)};
    const int key = k0 + 4 * kb;
    if (key < ld) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(4 * db + c) * ld + key) = col[c];
    }
  }
}

template <class K>
cudaError_t set_smem(K kernel, uint32_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

// Query heads per group of the block order: whole key/value heads (g query
// heads each) whose K and V (2 N 128 elem_bytes bytes per key/value head)
// stay within kFwdGroupBytes of L2.
int forward_head_group(int BH, int g, int N, int elem_bytes) {
  long long kv = kFwdGroupBytes / (2ll * N * 128 * elem_bytes);
  kv = kv < 1 ? 1 : kv;
  const long long heads = kv * g;
  return static_cast<int>(heads < BH ? heads : BH);
}

}  // namespace

cudaError_t launch_forward_bf16(const FwdMaps& maps, void* o, float* lse, int B, int H,
                                int Hkv, int N, float scale, int causal, int window,
                                const float* alibi, cudaStream_t stream,
                                const TimingEvents& ev) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    cudaError_t e = set_smem(fwd_bf16_kernel<false, false>, Bf16::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(fwd_bf16_kernel<true, false>, Bf16::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(fwd_bf16_kernel<false, true>, Bf16::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(fwd_bf16_kernel<true, true>, Bf16::SMEM_BYTES);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  const int BH = B * H;
  const int npair = (N + 2 * BM - 1) / (2 * BM);
  const float scale_log2 = scale * 1.4426950408889634f;
  auto kernel = alibi ? (window > 0 ? fwd_bf16_kernel<true, true> : fwd_bf16_kernel<false, true>)
                      : (window > 0 ? fwd_bf16_kernel<true, false>
                                    : fwd_bf16_kernel<false, false>);
  // Without the mask every item costs the same, so a last wave of r items on
  // S SMs (r <= S/2) runs as 2r half-length blocks instead.
  int nsplit = 0;
  if (!causal) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        sms > 0) {
      const long long items = static_cast<long long>(npair) * BH;
      const long long r = items % sms;
      if (items > sms && r > 0 && 2 * r <= sms) nsplit = static_cast<int>(r);
    }
  }
  const int head_group = forward_head_group(BH, H / Hkv, N, 2);
  if (ev.before) cudaEventRecord(ev.before, stream);
  kernel<<<dim3(npair * BH + nsplit), dim3(alibi ? fwd_threads<true>() : fwd_threads<false>()),
           Bf16::SMEM_BYTES, stream>>>(
      maps.q, maps.k, maps.v, maps.o, static_cast<__nv_bfloat16*>(o), lse, BH, N, scale_log2,
      causal, H / Hkv, window, alibi, H, nsplit, head_group);
  cudaError_t e = cudaGetLastError();
  if (ev.after) cudaEventRecord(ev.after, stream);
  return e;
}

size_t fp8_vt_ld(int N) { return (static_cast<size_t>(N) + 15) / 16 * 16; }

size_t forward_fp8_workspace_bytes(int B, int Hkv, int N) {
  return align256(static_cast<size_t>(B) * Hkv * HD * fp8_vt_ld(N));
}

cudaError_t launch_transpose_v_fp8(const void* v, void* vt, int B, int Hkv, int N,
                                   cudaStream_t stream) {
  const int ld = static_cast<int>(fp8_vt_ld(N));
  transpose_v_kernel<<<dim3((N + 63) / 64, B * Hkv), dim3(256), 0, stream>>>(
      static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), N, ld);
  return cudaGetLastError();
}

cudaError_t launch_forward_fp8(const FwdMaps& maps, void* o, float* lse, int B, int H, int Hkv,
                               int N, float scale, float q_descale, float k_descale,
                               float v_descale, int causal, int window, const float* alibi,
                               cudaStream_t stream, const TimingEvents& ev) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    cudaError_t e = set_smem(fwd_fp8_kernel<false, false>, Fp8::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(fwd_fp8_kernel<true, false>, Fp8::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(fwd_fp8_kernel<false, true>, Fp8::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(fwd_fp8_kernel<true, true>, Fp8::SMEM_BYTES);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  const int BH = B * H;
  const int npair = (N + 2 * BM - 1) / (2 * BM);
  const float scale_log2 = scale * q_descale * k_descale * 1.4426950408889634f;
  auto kernel = alibi ? (window > 0 ? fwd_fp8_kernel<true, true> : fwd_fp8_kernel<false, true>)
                      : (window > 0 ? fwd_fp8_kernel<true, false> : fwd_fp8_kernel<false, false>);
  const int head_group = forward_head_group(BH, H / Hkv, N, 1);
  if (ev.before) cudaEventRecord(ev.before, stream);
  kernel<<<dim3(npair * BH), dim3(alibi ? fwd_threads<true>() : fwd_threads<false>()),
           Fp8::SMEM_BYTES, stream>>>(
      maps.q, maps.k, maps.v, static_cast<__nv_bfloat16*>(o), lse, BH, N, scale_log2, v_descale,
      causal, H / Hkv, window, alibi, H, head_group);
  cudaError_t e = cudaGetLastError();
  if (ev.after) cudaEventRecord(ev.after, stream);
  return e;
}

int status_forward_bf16(bool clear) {
  int s = 0;
  cudaMemcpyFromSymbol(&s, g_status_fwd, sizeof(int));
  if (clear && s != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_status_fwd, &zero, sizeof(int));
  }
  return s;
}

}  // namespace fa
