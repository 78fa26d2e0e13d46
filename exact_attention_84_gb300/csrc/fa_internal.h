// fa_internal.h -- launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Each kernel file owns one device status word
// (a timeout record) and exposes a host function that reads and clears it.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>
#include <cstdint>

namespace fa {

// Optional events recorded around a call's main kernel (nullptr: none).
struct TimingEvents {
  cudaEvent_t before = nullptr;
  cudaEvent_t after = nullptr;
};

// ---- fp32 SIMT forward (fwd_fp32.cu)
cudaError_t launch_forward_fp32(const float* q, const float* k, const float* v, float* o,
                                float* lse, int B, int H, int N, int d, float scale,
                                int causal, cudaStream_t stream, const TimingEvents& ev);
int status_forward_fp32(bool clear);

// ---- bf16 tcgen05 forward (fwd_tc.cu); tensor maps over [B*H, N, 128]
// (Q and the bf16 output O) and [B*Hkv, N, 128] (K, V); window 0 = none.
struct FwdMaps {
  CUtensorMap q, k, v, o;
};
// alibi: device array of H slopes (ALiBi bias -slope_h |i - j|) or nullptr.
cudaError_t launch_forward_bf16(const FwdMaps& maps, void* o, float* lse, int B, int H,
                                int Hkv, int N, float scale, int causal, int window,
                                const float* alibi, cudaStream_t stream,
                                const TimingEvents& ev);
int status_forward_bf16(bool clear);

// ---- fp8 (e4m3) tcgen05 forward (fwd_tc.cu).  maps.q, maps.k over
// [B*H or B*Hkv, N, 128] bytes; maps.v over the transposed copy
// V^T [B*Hkv, 128, ld] (ld = fp8_vt_ld(N)) made by launch_transpose_v_fp8
// in a workspace of forward_fp8_workspace_bytes.
size_t fp8_vt_ld(int N);
size_t forward_fp8_workspace_bytes(int B, int Hkv, int N);
cudaError_t launch_transpose_v_fp8(const void* v, void* vt, int B, int Hkv, int N,
                                   cudaStream_t stream);
cudaError_t launch_forward_fp8(const FwdMaps& maps, void* o, float* lse, int B, int H, int Hkv,
                               int N, float scale, float q_descale, float k_descale,
                               float v_descale, int causal, int window, const float* alibi,
                               cudaStream_t stream, const TimingEvents& ev);

// ---- bf16 backward (bwd_bf16.cu)
struct BwdMaps {
  CUtensorMap q, k, v, dO, dk, dv;
};
size_t backward_workspace_bytes(int B, int H, int N);
// Q, dO, O, LSE, dQ have H query heads; K, V, dK, dV have Hkv (H % Hkv == 0).
// maps: Q, dO with 64-row boxes, K, V, dK, dV with 128-row boxes.  dq_maps: nullptr,
// or (deterministic dQ) Q, dO, K and V with 128-row boxes.
cudaError_t launch_backward_bf16(const BwdMaps& maps, const void* q, const void* k,
                                 const void* v, const void* o, const float* lse,
                                 const void* dO, void* dq, void* dk, void* dv, int B, int H,
                                 int Hkv, int N, float scale, int causal, int window,
                                 const float* alibi, const BwdMaps* dq_maps, void* ws,
                                 cudaStream_t stream, const TimingEvents& ev);
int status_backward_bf16(bool clear);

// ---- split-KV decode (decode.cu)
size_t decode_workspace_bytes(int B, int H, int num_splits);
// alibi: nullptr, or H (query-head) ALiBi slopes: row j of the cache gets
// -slope (L - 1 - j) on its score.
cudaError_t launch_decode(const void* q, const void* kc, const void* vc, void* o,
                          float* lse_out, int B, int H, int L, int num_splits, float scale,
                          void* ws, cudaStream_t stream, const TimingEvents& ev,
                          const float* alibi = nullptr);
int status_decode(bool clear);
// Grouped heads (Hq = g * Hkv): tensor maps over the caches [B*Hkv, L, 128]
// with 64-row boxes; partials and workspace as launch_decode with H = Hq.
cudaError_t launch_decode_gqa(const CUtensorMap& tmK, const CUtensorMap& tmV, const void* q,
                              void* o, float* lse_out, int B, int Hq, int Hkv, int L,
                              int num_splits, float scale, void* ws, cudaStream_t stream,
                              const TimingEvents& ev, const float* alibi = nullptr);

// Fixed device scratch of fa_decode_noalloc (decode.cu): room for
// kNoAllocMaxParts = B * H * num_splits partial results.
constexpr size_t kNoAllocMaxParts = 16384;
constexpr int kMaxDevices = 64;
cudaError_t decode_noalloc_scratch(void** out, size_t* bytes);

// ---- the timeout path of the bounded waits (selftest.cu)
cudaError_t launch_selftest_timeout(uint64_t limit_ns, cudaStream_t stream);
int status_selftest(bool clear);

// Runs `setup` (e.g. the cudaFuncSetAttribute calls of a launcher) once per
// device: function attributes belong to the device they were set on, so a
// process that drives several GPUs needs them on each.  `done` holds one bit
// per device; concurrent first calls may both run `setup`, which is harmless.
template <class Setup>
cudaError_t once_per_device(std::atomic<uint64_t>& done, Setup setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const uint64_t bit = uint64_t{1} << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = setup();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Round a byte count up to 256.
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace fa
