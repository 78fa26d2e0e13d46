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
                    float* __restrict__ part_lse, int L, int S, int chunk, float scale_log2) {
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
        if (warp * ROWS_PER_WARP + i >= rows) sc[i] = -INFINITY;
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

}  // namespace

size_t decode_workspace_bytes(int B, int H, int num_splits) {
  const size_t parts = static_cast<size_t>(B) * H * num_splits;
  return align256(parts * HD * sizeof(float)) + align256(parts * sizeof(float));
}

cudaError_t launch_decode(const void* q, const void* kc, const void* vc, void* o,
                          float* lse_out, int B, int H, int L, int num_splits, float scale,
                          void* ws, cudaStream_t stream, const TimingEvents& ev) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
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
      scale * 1.4426950408889634f);
  cudaError_t e = cudaGetLastError();
  if (ev.after) cudaEventRecord(ev.after, stream);
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<dim3(BH), dim3(HD), 0, stream>>>(
      part_o, part_lse, static_cast<__nv_bfloat16*>(o), lse_out, num_splits);
  return cudaGetLastError();
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
