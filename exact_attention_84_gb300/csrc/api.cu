// api.cu -- the extern "C" boundary of libfa.so (declared in include/fa.h).
//
// Every entry point validates its arguments before anything is enqueued,
// builds the TMA tensor maps it needs on the host, obtains workspace
// (caller-owned, or from a library-owned stream-ordered pool), and
// launches the kernels of fwd_fp32.cu, fwd_tc.cu, bwd_bf16.cu and
// decode.cu on the caller's stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"
#include "fa_status.h"

namespace {

thread_local std::string g_last_error;
thread_local fa::TimingEvents g_events;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled is a driver entry point; fetch it through the
// runtime so the library does not link against libcuda directly.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a [BH, N, 128] bf16 tensor; boxes of 64 columns (128 bytes,
// the 128-byte swizzle span) by `box_rows` rows of one head.  Rows past N
// read as zero.
int make_map(CUtensorMap* map, const void* base, int BH, int N, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(N) * 128 * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return FA_OK;
}

// 3-D map over an 8-bit tensor [heads, rows, inner] with rows `stride` bytes
// apart; boxes of 128 bytes (the swizzle span) by `box_rows` rows of one
// head.  Elements past `inner` or `rows` read as zero.
int make_map_u8(CUtensorMap* map, const void* base, int heads, int rows, int inner,
                size_t stride, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride),
                                 static_cast<cuuint64_t>(stride) * rows};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return FA_OK;
}

// Workspace for calls made without one: a stream-ordered pool per device,
// owned by the library, that keeps freed blocks for later calls (the default
// pool returns them to the system at every synchronisation, which makes each
// call pay for a fresh mapping).
cudaError_t workspace_alloc(void** p, size_t bytes, cudaStream_t stream) {
  // Fault injection for tests: FA_DEBUG_FAIL_ALLOC=1 makes every workspace
  // allocation fail as if the device were out of memory.
  const char* inject = std::getenv("FA_DEBUG_FAIL_ALLOC");
  if (inject != nullptr && inject[0] == '1') return cudaErrorMemoryAllocation;
  static std::mutex mu;
  static cudaMemPool_t pools[fa::kMaxDevices] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= fa::kMaxDevices) return cudaErrorInvalidDevice;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (pools[dev] == nullptr) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      e = cudaMemPoolCreate(&pools[dev], &props);
      if (e != cudaSuccess) {
        pools[dev] = nullptr;
        return e;
      }
      uint64_t keep = ~static_cast<uint64_t>(0);
      e = cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
      if (e != cudaSuccess) return e;
    }
    pool = pools[dev];
  }
  return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}

int check_sizes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1)
    return fail(FA_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d H=%d N=%d d=%d)", B, H, N, d);
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1ll << 30) || static_cast<long long>(N) > (1ll << 30))
    return fail(FA_ERR_UNSUPPORTED, "B*H or N too large");
  return FA_OK;
}

int check_scale(float scale) {
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0 (got %g)", double(scale));
  return FA_OK;
}

// Grouped heads and window: Hq = g * Hkv query heads share Hkv key/value
// heads; window 0 means none, window >= 1 needs the causal mask.
int check_heads(const char* fn, int Hq, int Hkv, int causal, int window) {
  if (Hkv < 1 || Hq % Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "%s: Hq (%d) must be a positive multiple of Hkv (%d)", fn, Hq,
                Hkv);
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (window < 0) return fail(FA_ERR_INVALID_ARG, "%s: window must be >= 0 (got %d)", fn, window);
  if (window > 0 && !causal)
    return fail(FA_ERR_UNSUPPORTED, "%s: a sliding window needs causal = 1", fn);
  return FA_OK;
}

// Grid sizes are computed in int: refuse shapes whose thread-block count
// (or element count for the elementwise kernels) would not fit.
int check_grid(const char* fn, long long blocks) {
  if (blocks > 2147483647ll)
    return fail(FA_ERR_UNSUPPORTED, "%s: the problem needs more than 2^31-1 thread blocks", fn);
  return FA_OK;
}

int launch_result(cudaError_t e, const char* what) {
  if (e != cudaSuccess)
    return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

static int forward_impl(const char* fn, const void* q, const void* k, const void* v, void* o,
                        float* lse, int B, int Hq, int Hkv, int N, int d, float scale,
                        int causal, int window, const float* alibi, cudaStream_t stream) {
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (int r = check_sizes(B, Hq, N, d)) return r;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "%s: d must be 128 (got %d)", fn, d);
  if (int r = check_scale(scale)) return r;
  if (int r = check_heads(fn, Hq, Hkv, causal, window)) return r;
  if (int r = check_grid(fn, (N + 255ll) / 256 * B * Hq)) return r;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (alibi && (reinterpret_cast<uintptr_t>(alibi) & 3u)))
    return fail(FA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
  fa::FwdMaps maps;
  if (int r = make_map(&maps.q, q, B * Hq, N, 128)) return r;
  if (int r = make_map(&maps.k, k, B * Hkv, N, 128)) return r;
  if (int r = make_map(&maps.v, v, B * Hkv, N, 128)) return r;
  if (int r = make_map(&maps.o, o, B * Hq, N, 128)) return r;
  return launch_result(fa::launch_forward_bf16(maps, o, lse, B, Hq, Hkv, N, scale, causal,
                                               window >= N ? 0 : window, alibi, stream,
                                               g_events),
                       "forward launch");
}

int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, float scale, int causal, cudaStream_t stream) {
  return forward_impl("fa_forward", q, k, v, o, lse, B, H, H, N, d, scale, causal, 0, nullptr,
                      stream);
}

int fa_forward_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int Hq, int Hkv, int N, int d, float scale, int causal, int window,
                   const float* alibi_slopes, cudaStream_t stream) {
  return forward_impl("fa_forward_gqa", q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, window,
                      alibi_slopes, stream);
}

int fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int Hq, int Hkv, int N, int d, float scale, float q_descale, float k_descale,
                   float v_descale, int causal, int window, const float* alibi_slopes,
                   void* ws, size_t ws_bytes, cudaStream_t stream) {
  const char* fn = "fa_forward_fp8";
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (int r = check_sizes(B, Hq, N, d)) return r;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "%s: d must be 128 (got %d)", fn, d);
  if (int r = check_scale(scale)) return r;
  for (float x : {q_descale, k_descale, v_descale})
    if (!std::isfinite(x) || !(x > 0.f))
      return fail(FA_ERR_INVALID_ARG, "%s: descale factors must be finite and > 0", fn);
  if (int r = check_heads(fn, Hq, Hkv, causal, window)) return r;
  if (int r = check_grid(fn, (N + 255ll) / 256 * B * Hq)) return r;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)))
    return fail(FA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
  if (static_cast<long long>(N) > 65535ll * 64 || static_cast<long long>(B) * Hkv > 65535ll)
    return fail(FA_ERR_UNSUPPORTED, "%s: N or B*Hkv too large", fn);
  const size_t need = fa::forward_fp8_workspace_bytes(B, Hkv, N);
  const bool own = (ws == nullptr);
  if (!own && (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)))
    return fail(FA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned and >= %zu bytes",
                fn, need);
  if (own && workspace_alloc(&ws, need, stream) != cudaSuccess) {
    cudaGetLastError();
    return fail(FA_ERR_NO_MEMORY, "%s: workspace allocation of %zu bytes failed", fn, need);
  }
  fa::FwdMaps maps;
  int r = make_map_u8(&maps.q, q, B * Hq, N, 128, 128, 128);
  if (r == FA_OK) r = make_map_u8(&maps.k, k, B * Hkv, N, 128, 128, 128);
  if (r == FA_OK) r = make_map_u8(&maps.v, ws, B * Hkv, 128, N, fa::fp8_vt_ld(N), 128);
  cudaError_t e = cudaSuccess;
  if (r == FA_OK) {
    e = fa::launch_transpose_v_fp8(v, ws, B, Hkv, N, stream);
    if (e == cudaSuccess)
      e = fa::launch_forward_fp8(maps, o, lse, B, Hq, Hkv, N, scale, q_descale, k_descale,
                                 v_descale, causal, window >= N ? 0 : window, alibi_slopes,
                                 stream, g_events);
  }
  if (own) {
    cudaError_t e2 = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = e2;
  }
  if (r != FA_OK) return r;
  return launch_result(e, "fa_forward_fp8 launch");
}

int fa_forward_fp32(const float* q, const float* k, const float* v, float* o, float* lse,
                    int B, int H, int N, int d, float scale, int causal, cudaStream_t stream) {
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "fa_forward_fp32: null pointer");
  if (int r = check_sizes(B, H, N, d)) return r;
  if (d % 32 != 0 || d > 128)
    return fail(FA_ERR_UNSUPPORTED, "fa_forward_fp32: d must be 32, 64, 96 or 128 (got %d)", d);
  if (int r = check_scale(scale)) return r;
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp32: pointers must be 16-byte aligned");
  if (static_cast<long long>(N) > 65535ll * 16)
    return fail(FA_ERR_UNSUPPORTED, "fa_forward_fp32: N too large");
  if (static_cast<long long>(B) * H > 65535ll)
    return fail(FA_ERR_UNSUPPORTED, "fa_forward_fp32: B*H must be <= 65535");
  return launch_result(
      fa::launch_forward_fp32(q, k, v, o, lse, B, H, N, d, scale, causal, stream, g_events),
      "fa_forward_fp32 launch");
}

static int backward_impl(const char* fn, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dO, void* dq, void* dk,
                         void* dv, int B, int Hq, int Hkv, int N, int d, float scale,
                         int causal, int window, const float* alibi, int deterministic,
                         void* ws, size_t ws_bytes, bool own_ws, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv)
    return fail(FA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (int r = check_sizes(B, Hq, N, d)) return r;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "%s: d must be 128 (got %d)", fn, d);
  if (int r = check_scale(scale)) return r;
  if (int r = check_heads(fn, Hq, Hkv, causal, window)) return r;
  {
    const long long padded = (N + 127ll) / 128 * 128 * B * Hq;        // bwd_pre rows
    if (int r = check_grid(fn, (N + 127ll) / 128 * B * Hkv)) return r;
    if (int r = check_grid(fn, (padded + 15) / 16)) return r;
    if (int r = check_grid(fn, static_cast<long long>(B) * Hq * N / 16 + 1)) return r;  // convert
    if (int r = check_grid(fn, (N + 127ll) / 128 * B * Hq)) return r;   // deterministic dQ
  }
  const void* ptrs[] = {q, k, v, o, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(FA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(alibi) & 3u))
    return fail(FA_ERR_INVALID_ARG, "%s: lse and alibi_slopes must be 4-byte aligned", fn);
  const size_t need = fa::backward_workspace_bytes(B, Hq, N);
  if (!own_ws) {
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
      return fail(FA_ERR_INVALID_ARG,
                  "%s: workspace must be 256-byte aligned and >= %zu bytes", fn, need);
  }
  if (deterministic != 0 && deterministic != 1)
    return fail(FA_ERR_INVALID_ARG, "%s: deterministic must be 0 or 1", fn);
  fa::BwdMaps maps, dq_maps;
  if (int r = make_map(&maps.q, q, B * Hq, N, 64)) return r;     // 64-query blocks
  if (int r = make_map(&maps.dO, dO, B * Hq, N, 64)) return r;
  if (int r = make_map(&maps.k, k, B * Hkv, N, 128)) return r;
  if (int r = make_map(&maps.v, v, B * Hkv, N, 128)) return r;
  if (int r = make_map(&maps.dk, dk, B * Hkv, N, 128)) return r;
  if (int r = make_map(&maps.dv, dv, B * Hkv, N, 128)) return r;
  if (deterministic) {                                            // 128-query and 128-key tiles
    if (int r = make_map(&dq_maps.q, q, B * Hq, N, 128)) return r;
    if (int r = make_map(&dq_maps.dO, dO, B * Hq, N, 128)) return r;
    if (int r = make_map(&dq_maps.k, k, B * Hkv, N, 128)) return r;
    if (int r = make_map(&dq_maps.v, v, B * Hkv, N, 128)) return r;
  }
  if (own_ws) {
    if (workspace_alloc(&ws, need, stream) != cudaSuccess) {
      cudaGetLastError();
      return fail(FA_ERR_NO_MEMORY, "%s: workspace allocation of %zu bytes failed", fn, need);
    }
  }
  cudaError_t e = fa::launch_backward_bf16(maps, q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N,
                                           scale, causal, window >= N ? 0 : window, alibi,
                                           deterministic ? &dq_maps : nullptr, ws, stream,
                                           g_events);
  if (own_ws) {
    cudaError_t e2 = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = e2;
  }
  return launch_result(e, "backward launch");
}

int fa_backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                float scale, int causal, cudaStream_t stream) {
  return backward_impl("fa_backward", q, k, v, o, lse, dO, dq, dk, dv, B, H, H, N, d, scale,
                       causal, 0, nullptr, 0, nullptr, 0, true, stream);
}

int fa_backward_ex(const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const void* dO, void* dq, void* dk, void* dv, int B, int H,
                   int N, int d, float scale, int causal, void* ws, size_t ws_bytes,
                   cudaStream_t stream) {
  return backward_impl("fa_backward_ex", q, k, v, o, lse, dO, dq, dk, dv, B, H, H, N, d, scale,
                       causal, 0, nullptr, 0, ws, ws_bytes, false, stream);
}

int fa_backward_gqa(const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                    int Hq, int Hkv, int N, int d, float scale, int causal, int window,
                    const float* alibi_slopes, int deterministic, void* ws, size_t ws_bytes,
                    cudaStream_t stream) {
  return backward_impl("fa_backward_gqa", q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d,
                       scale, causal, window, alibi_slopes, deterministic, ws, ws_bytes,
                       ws == nullptr, stream);
}

int fa_decode_ex(const void* q, const void* kcache, const void* vcache, void* o,
                 float* lse_out, int B, int H, int Lkv, int d, int num_splits, float scale,
                 void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!q || !kcache || !vcache || !o) return fail(FA_ERR_INVALID_ARG, "fa_decode: null pointer");
  if (int r = check_sizes(B, H, Lkv, d)) return r;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "fa_decode: d must be 128 (got %d)", d);
  if (int r = check_scale(scale)) return r;
  if (num_splits < 1 || num_splits > Lkv || num_splits > 1024)
    return fail(FA_ERR_INVALID_ARG, "fa_decode: num_splits must be in [1, min(Lkv, 1024)] (got %d)",
                num_splits);
  if (static_cast<long long>(B) * H > 65535ll)
    return fail(FA_ERR_UNSUPPORTED, "fa_decode: B*H must be <= 65535");
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
      (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u)))
    return fail(FA_ERR_INVALID_ARG, "fa_decode: pointers must be 16-byte aligned");
  const size_t need = fa::decode_workspace_bytes(B, H, num_splits);
  const bool own = (ws == nullptr);
  if (!own && (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)))
    return fail(FA_ERR_INVALID_ARG,
                "fa_decode_ex: workspace must be 256-byte aligned and >= %zu bytes", need);
  if (own && workspace_alloc(&ws, need, stream) != cudaSuccess) {
    cudaGetLastError();
    return fail(FA_ERR_NO_MEMORY, "fa_decode: workspace allocation of %zu bytes failed", need);
  }
  cudaError_t e = fa::launch_decode(q, kcache, vcache, o, lse_out, B, H, Lkv, num_splits, scale,
                                    ws, stream, g_events);
  if (own) {
    cudaError_t e2 = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = e2;
  }
  return launch_result(e, "fa_decode launch");
}

int fa_decode_splits(int B, int Hq, int Hkv, int Lkv) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lkv < 1 || Hq % Hkv != 0) return 0;
  // Thread blocks per split: one per (b, h) for one query head per cache
  // head, one per (b, cache head, 16 query heads) otherwise; two fit an SM.
  // Aim at about 16 waves of blocks so the last wave is a small part of the
  // work, with at least 512 cache rows per split.
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    cudaGetLastError();
    sms = 148;
  }
  const int g = Hq / Hkv;
  const long long units = g == 1 ? static_cast<long long>(B) * Hq
                                 : static_cast<long long>(B) * Hkv * ((g + 15) / 16);
  const long long want = (16ll * 2 * sms + units - 1) / units;
  long long s = want < 1 ? 1 : want;
  const long long by_len = Lkv / 512 > 1 ? Lkv / 512 : 1;
  if (s > by_len) s = by_len;
  if (s > 1024) s = 1024;
  if (s > Lkv) s = Lkv;
  return static_cast<int>(s);
}

int fa_decode_gqa(const void* q, const void* kcache, const void* vcache, void* o,
                  float* lse_out, int B, int Hq, int Hkv, int Lkv, int d, int num_splits,
                  float scale, const float* alibi_slopes, void* ws, size_t ws_bytes,
                  cudaStream_t stream) {
  const char* fn = "fa_decode_gqa";
  if (!q || !kcache || !vcache || !o) return fail(FA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (int r = check_sizes(B, Hq, Lkv, d)) return r;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "%s: d must be 128 (got %d)", fn, d);
  if (int r = check_scale(scale)) return r;
  if (int r = check_heads(fn, Hq, Hkv, 0, 0)) return r;
  if (num_splits == 0) num_splits = fa_decode_splits(B, Hq, Hkv, Lkv);
  if (num_splits < 1 || num_splits > Lkv || num_splits > 1024)
    return fail(FA_ERR_INVALID_ARG,
                "%s: num_splits must be 0 (automatic) or in [1, min(Lkv, 1024)] (got %d)", fn,
                num_splits);
  const int group = Hq / Hkv;
  if (static_cast<long long>(B) * Hkv * ((group + 15) / 16) > 65535ll ||
      static_cast<long long>(B) * Hq > 65535ll)
    return fail(FA_ERR_UNSUPPORTED, "%s: B*Hq must be <= 65535", fn);
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
      (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u)) ||
      (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)))
    return fail(FA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
  const size_t need = fa::decode_workspace_bytes(B, Hq, num_splits);
  const bool own = (ws == nullptr);
  if (!own && (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)))
    return fail(FA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned and >= %zu bytes",
                fn, need);
  CUtensorMap tk, tv;
  if (group > 1) {
    if (int r = make_map(&tk, kcache, B * Hkv, Lkv, 64)) return r;
    if (int r = make_map(&tv, vcache, B * Hkv, Lkv, 64)) return r;
  }
  if (own && workspace_alloc(&ws, need, stream) != cudaSuccess) {
    cudaGetLastError();
    return fail(FA_ERR_NO_MEMORY, "%s: workspace allocation of %zu bytes failed", fn, need);
  }
  // One query head per key/value head is plain decode (per-row kernel).
  cudaError_t e = group == 1
                      ? fa::launch_decode(q, kcache, vcache, o, lse_out, B, Hq, Lkv, num_splits,
                                          scale, ws, stream, g_events, alibi_slopes)
                      : fa::launch_decode_gqa(tk, tv, q, o, lse_out, B, Hq, Hkv, Lkv,
                                              num_splits, scale, ws, stream, g_events,
                                              alibi_slopes);
  if (own) {
    cudaError_t e2 = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = e2;
  }
  return launch_result(e, "fa_decode_gqa launch");
}

int fa_decode(const void* q, const void* kcache, const void* vcache, void* o, int B, int H,
              int Lkv, int d, int num_splits, cudaStream_t stream) {
  const float scale = d > 0 ? 1.0f / std::sqrt(static_cast<float>(d)) : 1.0f;
  return fa_decode_ex(q, kcache, vcache, o, nullptr, B, H, Lkv, d, num_splits, scale, nullptr,
                      0, stream);
}

int fa_decode_noalloc(const void* q, const void* kcache, const void* vcache, void* o,
                      float* lse_out, int B, int H, int Lkv, int d, int num_splits, float scale,
                      cudaStream_t stream) {
  if (!q || !kcache || !vcache || !o)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_noalloc: null pointer");
  if (int r = check_sizes(B, H, Lkv, d)) return r;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "fa_decode_noalloc: d must be 128 (got %d)", d);
  if (int r = check_scale(scale)) return r;
  if (num_splits < 1 || num_splits > Lkv || num_splits > 1024)
    return fail(FA_ERR_INVALID_ARG,
                "fa_decode_noalloc: num_splits must be in [1, min(Lkv, 1024)] (got %d)", num_splits);
  const long long parts = static_cast<long long>(B) * H * num_splits;
  if (parts > static_cast<long long>(fa::kNoAllocMaxParts))
    return fail(FA_ERR_UNSUPPORTED,
                "fa_decode_noalloc: B*H*num_splits = %lld exceeds the fixed scratch capacity "
                "of %zu parts; use fewer splits or fa_decode_ex",
                parts, fa::kNoAllocMaxParts);
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
      (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u)))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_noalloc: pointers must be 16-byte aligned");
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  cudaError_t e = fa::decode_noalloc_scratch(&scratch, &scratch_bytes);
  if (e != cudaSuccess)
    return fail(FA_ERR_CUDA, "fa_decode_noalloc: scratch address lookup failed: %s",
                cudaGetErrorString(e));
  if (fa::decode_workspace_bytes(B, H, num_splits) > scratch_bytes)
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_noalloc: scratch too small for this call");
  e = fa::launch_decode(q, kcache, vcache, o, lse_out, B, H, Lkv, num_splits, scale, scratch,
                        stream, g_events);
  return launch_result(e, "fa_decode_noalloc launch");
}

size_t fa_workspace_size(int op, int B, int H, int n_or_lkv, int d, int num_splits) {
  if (B < 1 || H < 1 || n_or_lkv < 1 || d != 128) return 0;
  switch (op) {
    case FA_OP_FORWARD: return 0;
    case FA_OP_FORWARD_FP8: return fa::forward_fp8_workspace_bytes(B, H, n_or_lkv);
    case FA_OP_BACKWARD: return fa::backward_workspace_bytes(B, H, n_or_lkv);
    case FA_OP_DECODE:
      if (num_splits < 1 || num_splits > n_or_lkv || num_splits > 1024) return 0;
      return fa::decode_workspace_bytes(B, H, num_splits);
    default: return 0;
  }
}

int fa_get_device_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  int s = 0;
  const int parts[] = {fa::status_forward_fp32(true), fa::status_forward_bf16(true),
                       fa::status_backward_bf16(true), fa::status_decode(true),
                       fa::status_selftest(true)};
  for (int p : parts)
    if (p != 0) s = p;
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (s == fa::kStatusTimeout) return fail(FA_ERR_TIMEOUT, "a kernel wait ran out of time");
  if (s != 0) return fail(FA_ERR_CUDA, "a kernel failed its launch-layout self-check (code %d)", s);
  return ok();
}

int fa_selftest_timeout(unsigned limit_ms, cudaStream_t stream) {
  if (limit_ms < 1 || limit_ms > 10000)
    return fail(FA_ERR_INVALID_ARG, "fa_selftest_timeout: limit_ms must be in [1, 10000]");
  return launch_result(fa::launch_selftest_timeout(static_cast<uint64_t>(limit_ms) * 1000000ull,
                                                   stream),
                       "fa_selftest_timeout launch");
}

int fa_set_timing_events(cudaEvent_t before, cudaEvent_t after) {
  if ((before == nullptr) != (after == nullptr))
    return fail(FA_ERR_INVALID_ARG, "fa_set_timing_events: set both events or neither");
  g_events.before = before;
  g_events.after = after;
  return ok();
}

const char* fa_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
