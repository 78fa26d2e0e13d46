// decode.cu -- split-KV attention for one new query token per sequence.
//
// FlashDecoding ("FlashAttention ontleed", "Interactie met de KV-cache";
// "03. FlashAttention", "Variantes et extensions"; Lensa ML FAQ on decoding):
// with one query row the cost is reading the KV cache, so the Lkv rows of
// each (batch, head) are cut into num_splits contiguous parts and each part
// gets its own thread block.  Each block runs the online softmax of
// "Tiling en Online Softmax" over its rows and leaves a normalised partial
// output O_s with its lse_s; the combine kernel applies the same rescaling
// across parts:  L = ln sum_s e^(lse_s),  o = sum_s e^(lse_s - L) O_s.
//
// GB300 mapping: the kernel is HBM-bound (~1 FLOP per byte).  One producer
// lane streams 32-row chunks of K and V (8 KiB each) with cp.async.bulk into
// a 6-stage shared-memory ring under mbarriers; 8 consumer warps each take 4
// rows of every chunk (lane = 4 head-dimension elements), so two blocks per
// SM keep ~190 KiB of loads in flight.
//
// Grouped query heads ("FlashAttention ontleed", "Interactie met de
// KV-cache": several query heads share one key/value head): the g query rows
// of a key/value head read the same cache rows, so one thread block takes up
// to 16 of them at once and each cache byte is read once for all of them.
// Sixteen query rows against a 16-key slice is a 16x16x128 product: small
// for the 5th-generation tensor cores (64 rows at least) but a natural fit
// for warp-level m16n8k16 MMAs with fp32 accumulation, which keep S, P and
// the output in registers.  The kernel stays bound by the cache read.
//
// ALiBi ("03. FlashAttention", "Variantes et extensions": the linear bias
// fused into the kernel): the new token sits at position L - 1, after every
// cached row, so row j of head h gets -slope_h (L - 1 - j) on its score.
#include <cfloat>
#include <mutex>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ int g_status_decode;

constexpr int HD = 128;
constexpr int ROWS = 32;                          // cache rows per stage
constexpr int STAGES = 6;
constexpr int CWARPS = 8;                         // consumer warps
constexpr int ROWS_PER_WARP = ROWS / CWARPS;      // 4
constexpr int NTHREADS = (CWARPS + 1) * 32;       // + one producer warp
constexpr uint32_t CHUNK_BYTES = ROWS * HD * 2;   // 8 KiB of K (or V)

constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + STAGES * CHUNK_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + STAGES * CHUNK_BYTES;   // full[S], empty[S]
constexpr uint32_t OFF_RED = OFF_BAR + 2 * STAGES * 8;       // m[8], l[8], o[8][128]
constexpr uint32_t OFF_FLAG = OFF_RED + (2 * CWARPS + CWARPS * HD) * 4;
constexpr uint32_t SMEM_BYTES = OFF_FLAG + 16 + 128;         // + alignment slack

constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ void bf16x4_to_float(uint2 u, float* f) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
}

__global__ void __launch_bounds__(NTHREADS, 2)
decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                    const __nv_bfloat16* __restrict__ vc, float* __restrict__ part_o,
                    float* __restrict__ part_lse, int L, int S, int chunk, float scale_log2,
                    const float* __restrict__ alibi, int heads) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_FLAG);
  float* red_m = reinterpret_cast<float*>(smem + OFF_RED);
  float* red_l = red_m + CWARPS;
  float* red_o = red_l + CWARPS;

  const int s = blockIdx.x;
  const int bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = s * chunk;
  const int nrows = max(0, min(L, r0 + chunk) - r0);
  const int nchunks = (nrows + ROWS - 1) / ROWS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(sbase + OFF_BAR + 8 * i, 1);
      mbar_init(sbase + OFF_BAR + 8 * (STAGES + i), CWARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == CWARPS) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const size_t base = (static_cast<size_t>(bh) * L + r0) * HD;
      for (int t = 0; t < nchunks; ++t) {
        const int st = t % STAGES;
        if (t >= STAGES && !mbar_wait(sbase + OFF_BAR + 8 * (STAGES + st),
                                      ((t / STAGES) - 1) & 1, abort_flag, &g_status_decode))
          break;
        const int rows = min(ROWS, nrows - t * ROWS);
        const uint32_t bytes = static_cast<uint32_t>(rows) * HD * 2;
        const uint32_t full = sbase + OFF_BAR + 8 * st;
        mbar_arrive_expect_tx(full, 2 * bytes);
        const size_t g = base + static_cast<size_t>(t) * ROWS * HD;
        bulk_load(sbase + OFF_K + st * CHUNK_BYTES, kc + g, bytes, full);
        bulk_load(sbase + OFF_V + st * CHUNK_BYTES, vc + g, bytes, full);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- consumers
    float qf[4];
    {
      const uint2 u = *reinterpret_cast<const uint2*>(q + static_cast<size_t>(bh) * HD + lane * 4);
      bf16x4_to_float(u, qf);
#pragma unroll
      for (int i = 0; i < 4; ++i) qf[i] *= scale_log2;   // scores come out in log2 units
    }
    float m = -INFINITY, l = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const float slope_log2 = alibi != nullptr ? alibi[bh % heads] * 1.4426950408889634f : 0.f;
    for (int t = 0; t < nchunks; ++t) {
      const int st = t % STAGES;
      if (!mbar_wait(sbase + OFF_BAR + 8 * st, (t / STAGES) & 1, abort_flag, &g_status_decode))
        break;
      const int rows = min(ROWS, nrows - t * ROWS);
      const uint8_t* ks = smem + OFF_K + st * CHUNK_BYTES;
      const uint8_t* vs = smem + OFF_V + st * CHUNK_BYTES;
      float sc[ROWS_PER_WARP];
#pragma unroll
      for (int i = 0; i < ROWS_PER_WARP; ++i) {
        const int r = warp * ROWS_PER_WARP + i;
        float part = 0.f;
        if (r < rows) {
          float kf[4];
          bf16x4_to_float(*reinterpret_cast<const uint2*>(ks + r * HD * 2 + lane * 8), kf);
          part = qf[0] * kf[0];
          part = fmaf(qf[1], kf[1], part);
          part = fmaf(qf[2], kf[2], part);
          part = fmaf(qf[3], kf[3], part);
        }
        sc[i] = part;
      }
#pragma unroll
      for (int i = 0; i < ROWS_PER_WARP; ++i) {
        sc[i] = warp_sum(sc[i]);
        const int r = warp * ROWS_PER_WARP + i;
        if (alibi != nullptr)   // ALiBi: -slope (L - 1 - j) in log2 units
          sc[i] = fmaf(-slope_log2, static_cast<float>(L - 1 - (r0 + t * ROWS + r)), sc[i]);
        if (r >= rows) sc[i] = -INFINITY;
      }
      float mx = sc[0];
#pragma unroll
      for (int i = 1; i < ROWS_PER_WARP; ++i) mx = fmaxf(mx, sc[i]);
      const float m_new = fmaxf(m, mx);
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = fast_exp2(m - m_ref);
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] *= corr;
#pragma unroll
      for (int i = 0; i < ROWS_PER_WARP; ++i) {
        const int r = warp * ROWS_PER_WARP + i;
        if (r < rows) {
          const float p = fast_exp2(sc[i] - m_ref);
          psum += p;
          float vf[4];
          bf16x4_to_float(*reinterpret_cast<const uint2*>(vs + r * HD * 2 + lane * 8), vf);
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[c] = fmaf(p, vf[c], acc[c]);
        }
      }
      l = l * corr + psum;
      m = m_new;
      __syncwarp();
      if (lane == 0) mbar_arrive(sbase + OFF_BAR + 8 * (STAGES + st));
    }
    if (lane == 0) {
      red_m[warp] = m;
      red_l[warp] = l;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) red_o[warp * HD + lane * 4 + c] = acc[c];
  }
  __syncthreads();

  // Merge the 8 warps' (m, l, o) with the same rescaling, then store O_s, lse_s.
  if (threadIdx.x < HD) {
    const int c = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < CWARPS; ++w) M = fmaxf(M, red_m[w]);
    const float Mref = (M == -INFINITY) ? 0.f : M;
    float lsum = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < CWARPS; ++w) {
      const float wgt = fast_exp2(red_m[w] - Mref);
      lsum = fmaf(red_l[w], wgt, lsum);
      o = fmaf(red_o[w * HD + c], wgt, o);
    }
    const size_t idx = static_cast<size_t>(bh) * S + s;
    const bool empty = !(lsum > 0.f) || *abort_flag;
    part_o[idx * HD + c] = empty ? 0.f : o / lsum;
    if (c == 0) part_lse[idx] = empty ? -INFINITY : (Mref + log2f(lsum)) * kLn2;
  }
}

__global__ void __launch_bounds__(HD)
decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse_out, int S) {
  const int bh = blockIdx.x;
  const int c = threadIdx.x;
  const float* lse_s = part_lse + static_cast<size_t>(bh) * S;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, lse_s[s]);
  const float Mref = (M == -INFINITY) ? 0.f : M;
  float tot = 0.f, acc = 0.f;
  for (int s = 0; s < S; ++s) {
    const float w = expf(lse_s[s] - Mref);          // empty part: e^-inf = 0
    tot += w;
    acc = fmaf(w, part_o[(static_cast<size_t>(bh) * S + s) * HD + c], acc);
  }
  o[static_cast<size_t>(bh) * HD + c] = __float2bfloat16_rn(tot > 0.f ? acc / tot : 0.f);
  if (lse_out != nullptr && c == 0) lse_out[bh] = Mref + logf(tot);
}

// ------------------------------------------------------------------ GQA split
// One thread block per (split s, key/value head bkv, slice of <= 16 of its g
// query heads).  A producer lane streams 64-row stages of K and V with TMA
// (128-byte swizzle, so every ldmatrix below is free of bank conflicts) into
// a 3-stage ring; warp w of four takes keys [16w, 16w + 16) of each stage:
//   S (16 heads x 16 keys) = Q K^T    8 k-steps x 2 n-tiles of m16n8k16
//   online softmax per head row        (4 lanes share a row: 2 shuffles)
//   O (16 x 128) += P V                1 k-step x 16 n-tiles, P from S regs
// and the four warps merge their (m, l, O) at the end.
constexpr int G_ROWS = 64;                        // cache rows per stage
constexpr int G_STAGES = 3;
constexpr int G_WARPS = 4;                        // consumer warps
constexpr int G_THREADS = (G_WARPS + 1) * 32;
constexpr uint32_t G_BOX = G_ROWS * 128;          // 64 rows x 64 columns bf16 = 8 KiB
constexpr uint32_t G_TILE = 2 * G_BOX;            // 64 rows x 128 columns
constexpr uint32_t G_STAGE = 2 * G_TILE;          // K then V: 32 KiB
constexpr uint32_t G_OFF_BAR = G_STAGES * G_STAGE;
constexpr uint32_t G_OFF_FLAG = G_OFF_BAR + 2 * G_STAGES * 8;
constexpr uint32_t G_SMEM = G_OFF_FLAG + 16 + 1024;          // + alignment slack
// merge area (reuses the stage ring once every stage has been consumed)
constexpr uint32_t G_RED_O = G_WARPS * 16 * HD * 4;           // 32 KiB
static_assert(G_RED_O + 2 * G_WARPS * 16 * 4 <= G_OFF_BAR, "merge area must fit the ring");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Shared address of the 16-byte chunk holding columns [col, col + 8) of row
// `row` in a 64-row x 128-column tile stored as two 64-column swizzled boxes.
__device__ __forceinline__ uint32_t g_chunk_addr(uint32_t tile, int row, int col) {
  return tile + (col >> 6) * G_BOX + sw128_offset(static_cast<uint32_t>(row),
                                                   static_cast<uint32_t>((col & 63) >> 3));
}

__global__ void __launch_bounds__(G_THREADS, 2)
decode_gqa_split_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __nv_bfloat16* __restrict__ q, float* __restrict__ part_o,
                        float* __restrict__ part_lse, int L, int S, int chunk, int group,
                        int nslice, float scale_log2, const float* __restrict__ alibi,
                        int heads) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G_OFF_FLAG);

  const int s = blockIdx.x;
  const int bkv = static_cast<int>(blockIdx.y) / nslice;
  const int slice = static_cast<int>(blockIdx.y) % nslice;
  const int h0 = bkv * group + slice * 16;          // first query head (b*Hq + h) of the slice
  const int nh = min(16, group - slice * 16);       // query heads in the slice
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = s * chunk;
  const int r_end = min(L, r0 + chunk);
  const int nrows = max(0, r_end - r0);
  const int nst = (nrows + G_ROWS - 1) / G_ROWS;
  auto full_bar = [&](int st) { return sbase + G_OFF_BAR + 8u * st; };
  auto empty_bar = [&](int st) { return sbase + G_OFF_BAR + 8u * (G_STAGES + st); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < G_STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), G_WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  float* red_o = reinterpret_cast<float*>(smem);    // [warp][16 rows][128]
  float* red_m = red_o + G_WARPS * 16 * HD;          // [warp][16]
  float* red_l = red_m + G_WARPS * 16;
  const int gid = lane >> 2, tig = lane & 3;
  // consumer state: rows gid and gid + 8 of the slice (m in log2 units; l is
  // this lane's part of the row sum until the end)
  float o[16][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  if (warp == G_WARPS) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      for (int t = 0; t < nst; ++t) {
        const int st = t % G_STAGES;
        if (t >= G_STAGES &&
            !mbar_wait(empty_bar(st), ((t / G_STAGES) - 1) & 1, abort_flag, &g_status_decode))
          break;
        const uint32_t fb = full_bar(st);
        const uint32_t dst = sbase + st * G_STAGE;
        const int row = r0 + t * G_ROWS;              // rows past L read as zero
        mbar_arrive_expect_tx(fb, G_STAGE);
        tma_load_3d(dst, &tmK, fb, 0, row, bkv);
        tma_load_3d(dst + G_BOX, &tmK, fb, 64, row, bkv);
        tma_load_3d(dst + G_TILE, &tmV, fb, 0, row, bkv);
        tma_load_3d(dst + G_TILE + G_BOX, &tmV, fb, 64, row, bkv);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- consumers
    // Q fragments (A operand, rows = query heads of the slice, k = d);
    // rows past the slice are zero.
    uint32_t qa[8][4];
    {
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(q + static_cast<size_t>(h0 + gid) * HD);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(q + static_cast<size_t>(h0 + gid + 8) * HD);
      const bool v0 = gid < nh, v1 = gid + 8 < nh;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        qa[k][0] = v0 ? q0[8 * k + tig] : 0u;
        qa[k][1] = v1 ? q1[8 * k + tig] : 0u;
        qa[k][2] = v0 ? q0[8 * k + 4 + tig] : 0u;
        qa[k][3] = v1 ? q1[8 * k + 4 + tig] : 0u;
      }
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    const int mi = lane >> 3, mr = lane & 7;        // ldmatrix: matrix index, row in it
    // ALiBi slopes of rows gid and gid + 8 (log2 units; 0 without ALiBi)
    const float slope0 = (alibi != nullptr && gid < nh) ? alibi[(h0 + gid) % heads] * 1.4426950408889634f : 0.f;
    const float slope1 = (alibi != nullptr && gid + 8 < nh) ? alibi[(h0 + gid + 8) % heads] * 1.4426950408889634f : 0.f;
    for (int t = 0; t < nst; ++t) {
      const int st = t % G_STAGES;
      if (!mbar_wait(full_bar(st), (t / G_STAGES) & 1, abort_flag, &g_status_decode)) break;
      const uint32_t kt = sbase + st * G_STAGE;
      const uint32_t vt = kt + G_TILE;
      // S = Q K^T over this warp's 16 keys (two n-tiles of 8)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int key = 16 * warp + 8 * (mi >> 1) + mr;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(g_chunk_addr(kt, key, 16 * k + 8 * (mi & 1)), b0, b1, b2, b3);
          mma16816(sc[0], qa[k][0], qa[k][1], qa[k][2], qa[k][3], b0, b1);
          mma16816(sc[1], qa[k][0], qa[k][1], qa[k][2], qa[k][3], b2, b3);
        }
      }
      // keys of this stage past the split (or the cache) are masked; ALiBi
      // adds -slope (L - 1 - j) (rows gid and gid + 8 have their own slopes)
      const int kbase = r0 + t * G_ROWS + 16 * warp + 2 * tig;
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kbase + 8 * n + (e & 1);
          const float bias = -(e < 2 ? slope0 : slope1) * static_cast<float>(L - 1 - key);
          sc[n][e] = key < r_end ? fmaf(sc[n][e], scale_log2, bias) : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float ref0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float ref1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float c0 = fast_exp2(m0 - ref0), c1 = fast_exp2(m1 - ref1);
      m0 = mn0;
      m1 = mn1;
      float p[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        p[n][0] = fast_exp2(sc[n][0] - ref0);
        p[n][1] = fast_exp2(sc[n][1] - ref0);
        p[n][2] = fast_exp2(sc[n][2] - ref1);
        p[n][3] = fast_exp2(sc[n][3] - ref1);
      }
      l0 = l0 * c0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
      l1 = l1 * c1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
      if (__any_sync(0xffffffffu, c0 != 1.f || c1 != 1.f)) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][0] *= c0;
          o[n][1] *= c0;
          o[n][2] *= c1;
          o[n][3] *= c1;
        }
      }
      // O += P V: P (16 x 16 keys) as the A operand straight from registers
      const uint32_t pa0 = pack_bf16x2(p[0][0], p[0][1]);
      const uint32_t pa1 = pack_bf16x2(p[0][2], p[0][3]);
      const uint32_t pa2 = pack_bf16x2(p[1][0], p[1][1]);
      const uint32_t pa3 = pack_bf16x2(p[1][2], p[1][3]);
      {
        const int key = 16 * warp + 8 * (mi & 1) + mr;
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(g_chunk_addr(vt, key, 16 * np + 8 * (mi >> 1)), b0, b1, b2, b3);
          mma16816(o[2 * np], pa0, pa1, pa2, pa3, b0, b1);
          mma16816(o[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st));
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
  // Every stage has been consumed (or the block gave up): the ring is free
  // and serves as the merge area.
  __syncthreads();
  if (warp < G_WARPS) {
    if (tig == 0) {
      red_m[warp * 16 + gid] = m0;
      red_m[warp * 16 + gid + 8] = m1;
      red_l[warp * 16 + gid] = l0;
      red_l[warp * 16 + gid + 8] = l1;
    }
    float* ro = red_o + warp * 16 * HD;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int c = 8 * n + 2 * tig;
      *reinterpret_cast<float2*>(ro + gid * HD + c) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(ro + (gid + 8) * HD + c) = make_float2(o[n][2], o[n][3]);
    }
  }
  __syncthreads();

  // Merge the four warps' (m, l, O) per query head with the online-softmax
  // rescaling, then store the split's normalised O_s and lse_s.
  for (int idx = threadIdx.x; idx < nh * HD; idx += G_THREADS) {
    const int r = idx / HD, c = idx % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < G_WARPS; ++w) M = fmaxf(M, red_m[w * 16 + r]);
    const float Mref = (M == -INFINITY) ? 0.f : M;
    float lsum = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < G_WARPS; ++w) {
      const float wgt = fast_exp2(red_m[w * 16 + r] - Mref);
      lsum = fmaf(red_l[w * 16 + r], wgt, lsum);
      acc = fmaf(red_o[(w * 16 + r) * HD + c], wgt, acc);
    }
    const size_t part = static_cast<size_t>(h0 + r) * S + s;
    const bool empty = !(lsum > 0.f) || *abort_flag;
    part_o[part * HD + c] = empty ? 0.f : acc / lsum;
    if (c == 0) part_lse[part] = empty ? -INFINITY : (Mref + log2f(lsum)) * kLn2;
  }
}

}  // namespace

size_t decode_workspace_bytes(int B, int H, int num_splits) {
  const size_t parts = static_cast<size_t>(B) * H * num_splits;
  return align256(parts * HD * sizeof(float)) + align256(parts * sizeof(float));
}

cudaError_t launch_decode(const void* q, const void* kc, const void* vc, void* o,
                          float* lse_out, int B, int H, int L, int num_splits, float scale,
                          void* ws, cudaStream_t stream, const TimingEvents& ev,
                          const float* alibi) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SMEM_BYTES));
  });
  if (ea != cudaSuccess) return ea;
  const int BH = B * H;
  const size_t parts = static_cast<size_t>(BH) * num_splits;
  float* part_o = static_cast<float*>(ws);
  float* part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                             align256(parts * HD * sizeof(float)));
  const int chunk = (L + num_splits - 1) / num_splits;
  if (ev.before) cudaEventRecord(ev.before, stream);
  decode_split_kernel<<<dim3(num_splits, BH), dim3(NTHREADS), SMEM_BYTES, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(kc),
      static_cast<const __nv_bfloat16*>(vc), part_o, part_lse, L, num_splits, chunk,
      scale * 1.4426950408889634f, alibi, H);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<dim3(BH), dim3(HD), 0, stream>>>(
      part_o, part_lse, static_cast<__nv_bfloat16*>(o), lse_out, num_splits);
  e = cudaGetLastError();
  // the timed span is the whole call: the split pass and its merge
  if (ev.after) cudaEventRecord(ev.after, stream);
  return e;
}

cudaError_t launch_decode_gqa(const CUtensorMap& tmK, const CUtensorMap& tmV, const void* q,
                              void* o, float* lse_out, int B, int Hq, int Hkv, int L,
                              int num_splits, float scale, void* ws, cudaStream_t stream,
                              const TimingEvents& ev, const float* alibi) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(decode_gqa_split_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(G_SMEM));
  });
  if (ea != cudaSuccess) return ea;
  const int group = Hq / Hkv;
  const int nslice = (group + 15) / 16;
  const size_t parts = static_cast<size_t>(B) * Hq * num_splits;
  float* part_o = static_cast<float*>(ws);
  float* part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                             align256(parts * HD * sizeof(float)));
  const int chunk = (L + num_splits - 1) / num_splits;
  if (ev.before) cudaEventRecord(ev.before, stream);
  decode_gqa_split_kernel<<<dim3(num_splits, B * Hkv * nslice), dim3(G_THREADS), G_SMEM,
                            stream>>>(tmK, tmV, static_cast<const __nv_bfloat16*>(q), part_o,
                                      part_lse, L, num_splits, chunk, group, nslice,
                                      scale * 1.4426950408889634f, alibi, Hq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<dim3(B * Hq), dim3(HD), 0, stream>>>(
      part_o, part_lse, static_cast<__nv_bfloat16*>(o), lse_out, num_splits);
  e = cudaGetLastError();
  if (ev.after) cudaEventRecord(ev.after, stream);
  return e;
}

// ---------------------------------------------------------------------------
// Fixed scratch for fa_decode_noalloc.  The split kernel writes every part's
// partial output and lse here (B * H * num_splits parts at most
// kNoAllocMaxParts) before the combine kernel reads them, so nothing in it has
// to start at zero.  Every GPU that loads this library holds the array (about
// 8.5 MB) until the process exits.  All calls share it: calls that overlap on
// the GPU race on its contents.
constexpr size_t kNoAllocFloats = kNoAllocMaxParts * (HD + 1);
static __device__ __align__(256) float g_decode_scratch[kNoAllocFloats];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
}  // namespace

// Device address of the scratch array on the current device.  In host code
// `g_decode_scratch` names a host-side stand-in, so the address a kernel may
// use is looked up once per device (with that device current) and cached.
cudaError_t decode_noalloc_scratch(void** out, size_t* bytes) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  *bytes = sizeof(g_decode_scratch);
  return cudaSuccess;
}

int status_decode(bool clear) {
  int s = 0;
  cudaMemcpyFromSymbol(&s, g_status_decode, sizeof(int));
  if (clear && s != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_status_decode, &zero, sizeof(int));
  }
  return s;
}

}  // namespace fa
