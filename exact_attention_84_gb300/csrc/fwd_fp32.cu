// fwd_fp32.cu -- exact attention forward in true fp32 (FMA, no TF32).
//
// The loop of "FlashAttention ontleed", section "Algoritmische kern in
// pseudocode", in the FlashAttention-2 order (section "FlashAttention-1
// versus FlashAttention-2"): a thread block owns a block of query rows and
// streams K/V tiles through shared memory.  Per tile and row it forms the
// local scores, raises the running maximum, rescales the running sum and
// output by e^(m_old - m_new), adds the new exponentials, and after the last
// tile divides by the running sum and writes O and LSE = m + ln(l) once.
//
// This path serves fp32 callers (tolerance 1e-5 rules out tensor cores);
// the bf16 and fp8 tensor-core paths are in fwd_tc.cu.
#include <cfloat>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ int g_status_fwd_fp32;   // no waits here; kept for a uniform status API

constexpr int kRowsPerBlock = 4;    // 4 warps x 1 query row: 64 blocks on the tiny workload
constexpr int kRowsPerWarp = 1;
constexpr int kKeysPerTile = 32;    // one key per lane

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// DL = d / 32 head-dimension elements per lane.
template <int DL>
__global__ void __launch_bounds__(128) fwd_fp32_kernel(const float* __restrict__ q,
                                                       const float* __restrict__ k,
                                                       const float* __restrict__ v,
                                                       float* __restrict__ o,
                                                       float* __restrict__ lse, int N,
                                                       float scale, int causal) {
  constexpr int D = DL * 32;
  constexpr int D4 = D / 4;                      // float4 per row
  constexpr int V4 = kKeysPerTile * D4 / 128;    // float4 of K (and of V) per thread per tile
  __shared__ __align__(16) float sQ[kRowsPerBlock][D];
  __shared__ float sK[kKeysPerTile][D + 1];   // +1: lane j reads row j conflict-free
  __shared__ __align__(16) float sV[kKeysPerTile][D];

  const int bh = blockIdx.y;
  const int q0 = blockIdx.x * kRowsPerBlock;
  const size_t head = static_cast<size_t>(bh) * N * D;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float4* q4 = reinterpret_cast<const float4*>(q + head);
  const float4* k4 = reinterpret_cast<const float4*>(k + head);
  const float4* v4 = reinterpret_cast<const float4*>(v + head);
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);

  for (int idx = tid; idx < kRowsPerBlock * D4; idx += blockDim.x) {
    const int r = idx / D4, c = idx % D4;
    *reinterpret_cast<float4*>(&sQ[r][4 * c]) =
        (q0 + r < N) ? q4[static_cast<size_t>(q0 + r) * D4 + c] : zero4;
  }
  // A K/V tile is fetched into registers with 16-byte loads, all issued
  // before any is used, one tile ahead of its use, then stored to shared
  // memory: the loads' latency is paid once per tile and hidden behind the
  // previous tile's arithmetic.
  float4 kr[V4], vr[V4];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      const int idx = tid + 128 * i;             // float4 within the 32 x D tile
      const int r = idx / D4, c = idx % D4;
      const bool in = (k0 + r) < N;
      const size_t g = static_cast<size_t>(k0 + r) * D4 + c;
      kr[i] = in ? k4[g] : zero4;
      vr[i] = in ? v4[g] : zero4;
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      const int idx = tid + 128 * i;
      const int r = idx / D4, c = 4 * (idx % D4);
      sK[r][c] = kr[i].x;
      sK[r][c + 1] = kr[i].y;
      sK[r][c + 2] = kr[i].z;
      sK[r][c + 3] = kr[i].w;
      *reinterpret_cast<float4*>(&sV[r][c]) = vr[i];
    }
  };

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DL];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int t = 0; t < DL; ++t) acc[r][t] = 0.f;
  }

  // Keys beyond the last query row of this block are masked for every row.
  const int key_end = causal ? min(N, q0 + kRowsPerBlock) : N;
  if (key_end > 0) fetch(0);
  for (int k0 = 0; k0 < key_end; k0 += kKeysPerTile) {
    __syncthreads();                               // the previous tile has been read
    stash();
    __syncthreads();
    if (k0 + kKeysPerTile < key_end) fetch(k0 + kKeysPerTile);

#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int r = warp * kRowsPerWarp + rr;
      const int qi = q0 + r;
      // 1. local score of key (k0 + lane) for this row (four independent
      // partial sums, so the dot product is not one long dependent chain)
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int c = 0; c < D; c += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) s4[u] = fmaf(sQ[r][c + u], sK[lane][c + u], s4[u]);
      }
      float s = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * scale;
      const int kj = k0 + lane;
      const bool valid = (kj < N) && (!causal || kj <= qi);
      s = valid ? s : -INFINITY;
      // 2. running maximum
      const float m_new = fmaxf(m[rr], warp_max(s));
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      // 3. rescaled exponentials and running sum
      const float p = valid ? expf(s - m_ref) : 0.f;
      const float corr = expf(m[rr] - m_ref);
      l[rr] = l[rr] * corr + warp_sum(p);
      // 4. output rescaled and accumulated: O = diag(corr) O + P V
#pragma unroll
      for (int t = 0; t < DL; ++t) acc[rr][t] *= corr;
#pragma unroll 4
      for (int j = 0; j < kKeysPerTile; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int t = 0; t < DL; ++t) acc[rr][t] = fmaf(pj, sV[j][lane + 32 * t], acc[rr][t]);
      }
      m[rr] = m_new;
    }
  }

  // Final normalisation by the running sum; O and LSE written once.
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int qi = q0 + warp * kRowsPerWarp + rr;
    if (qi >= N) continue;
    const float inv = 1.f / l[rr];
#pragma unroll
    for (int t = 0; t < DL; ++t)
      o[head + static_cast<size_t>(qi) * D + lane + 32 * t] = acc[rr][t] * inv;
    if (lse != nullptr && lane == 0)
      lse[static_cast<size_t>(bh) * N + qi] = m[rr] + logf(l[rr]);
  }
}

}  // namespace

cudaError_t launch_forward_fp32(const float* q, const float* k, const float* v, float* o,
                                float* lse, int B, int H, int N, int d, float scale,
                                int causal, cudaStream_t stream, const TimingEvents& ev) {
  dim3 grid((N + kRowsPerBlock - 1) / kRowsPerBlock, B * H);
  dim3 block(128);
  if (ev.before) cudaEventRecord(ev.before, stream);
  switch (d / 32) {
    case 1: fwd_fp32_kernel<1><<<grid, block, 0, stream>>>(q, k, v, o, lse, N, scale, causal); break;
    case 2: fwd_fp32_kernel<2><<<grid, block, 0, stream>>>(q, k, v, o, lse, N, scale, causal); break;
    case 3: fwd_fp32_kernel<3><<<grid, block, 0, stream>>>(q, k, v, o, lse, N, scale, causal); break;
    case 4: fwd_fp32_kernel<4><<<grid, block, 0, stream>>>(q, k, v, o, lse, N, scale, causal); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (ev.after) cudaEventRecord(ev.after, stream);
  return e;
}

int status_forward_fp32(bool clear) {
  int s = 0;
  cudaMemcpyFromSymbol(&s, g_status_fwd_fp32, sizeof(int));
  if (clear && s != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_status_fwd_fp32, &zero, sizeof(int));
  }
  return s;
}

}  // namespace fa
