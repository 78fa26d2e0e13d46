/*
 * fa.h -- C ABI of libfa.so: exact scaled-dot-product attention on one
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (sources: the FlashAttention explainer pages
 * "FlashAttention ontleed" (leren.llmnet.nl), "03. FlashAttention"
 * (frontier-llm-systems course notes) and the Lensa ML explainer
 * "FlashAttention" (lensaml.com)):
 *
 *   S = scale * Q K^T            ("03. FlashAttention", "Le probleme", step 1)
 *   S_ij = -inf where j > i      (causal only; the pages name masking but do
 *                                 not define it: square, top-left aligned)
 *   P = row-softmax(S)           (step 2; computed online, tile by tile:
 *                                 "FlashAttention ontleed", "Tiling en
 *                                 Online Softmax" and the pseudocode section)
 *   O = P V                      (step 3; O written to HBM once, after the
 *                                 last K/V tile, divided by the running sum)
 *   LSE_i = m_i + ln(l_i)        (the stored softmax statistics m and l of
 *                                 "Geheugencomplexiteit: van O(N^2) naar
 *                                 O(N)", kept as one fp32 number per row)
 *
 * The N x N score matrix is never written to device memory (Lensa ML step 3:
 * "0 B" of S written).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensors are dense, row-major, contiguous: Q, K, V, O, dO, dQ, dK, dV
 *   are [B, H, N, d]; LSE is [B, H, N] fp32 (natural log); decode q/o are
 *   [B, H, d]; decode caches are [B, H, Lkv, d].
 * - "bf16" tensors hold IEEE bfloat16 values; arithmetic is fp32 inside.
 * - Every pointer is a DEVICE pointer (cudaMalloc'd or equivalent, 16-byte
 *   aligned) unless stated otherwise.  The caller owns every buffer it passes;
 *   the library borrows them for the stream-ordered work only.
 * - Work is enqueued on `stream` and the call returns without synchronising.
 * - Arguments are validated before anything is launched; a failed check
 *   returns FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED and launches nothing.
 *   fa_last_error() then describes the failure.
 * - Kernels bound every wait on the GPU.  A wait that runs out records
 *   FA_ERR_TIMEOUT in a device status word, and the kernel returns early
 *   (outputs are then undefined).  fa_get_device_status() reads that word.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, misalignment */
  FA_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement  */
  FA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed          */
  FA_ERR_TIMEOUT = 4,      /* a bounded wait inside a kernel ran out        */
  FA_ERR_NO_MEMORY = 5     /* a stream-ordered workspace allocation failed  */
} fa_status;

/* Operation codes for fa_workspace_size(). */
enum { FA_OP_FORWARD = 0, FA_OP_BACKWARD = 1, FA_OP_DECODE = 2, FA_OP_FORWARD_FP8 = 3 };

/*
 * fa_forward -- fused tiled forward pass, bf16 in / bf16 out.
 *
 * Follows the loop of "FlashAttention ontleed", section "Algoritmische kern
 * in pseudocode", in the FlashAttention-2 order of its section
 * "FlashAttention-1 versus FlashAttention-2" (Q blocks outer, K/V inner; one
 * Q block per thread block, O written once).
 *
 *   q, k, v  [B,H,N,d] bf16, read only.
 *   o        [B,H,N,d] bf16, written.
 *   lse      [B,H,N] fp32, written (may be NULL when not needed).
 *   B, H, N  >= 1.  d must be 128.
 *   scale    multiplies Q K^T (usually 1/sqrt(d)); must be finite and > 0.
 *   causal   0: no mask; 1: key j hidden from query i when j > i.
 * Returns FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED or FA_ERR_CUDA.
 * Needs no workspace and allocates nothing.
 */
int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int N, int d, float scale, int causal,
               cudaStream_t stream);

/*
 * fa_forward_fp32 -- the same forward pass with fp32 inputs and outputs and
 * true fp32 arithmetic (fused multiply-add; no TF32, no bf16 rounding).
 *
 *   q, k, v, o  [B,H,N,d] fp32;  lse [B,H,N] fp32 (may be NULL).
 *   d must be a multiple of 32 and at most 128.  Other arguments as in
 *   fa_forward.  Allocates nothing.
 */
int fa_forward_fp32(const float* q, const float* k, const float* v, float* o,
                    float* lse, int B, int H, int N, int d, float scale,
                    int causal, cudaStream_t stream);

/*
 * fa_forward_gqa -- fa_forward with grouped query heads and an optional
 * causal sliding window.
 *
 * Grouped-query attention ("FlashAttention ontleed", "Interactie met de
 * KV-cache": several query heads share one key head and one value head):
 * Hq = g * Hkv query heads; query head h reads key/value head h / g.
 * Sliding window ("03. FlashAttention", "Variantes et extensions": the
 * tiling only visits the keys inside the window): with window w >= 1, query
 * i sees keys i-w+1 .. i (the pages give no formula; this causal, w-wide
 * reading is the plainest one).  Key tiles wholly outside the window are
 * skipped, tiles that cut its edge are masked element-wise.
 *
 *   q, o     [B,Hq,N,d] bf16;  k, v [B,Hkv,N,d] bf16;  lse [B,Hq,N] fp32
 *            (may be NULL).
 *   Hkv      >= 1 and Hq % Hkv == 0 (Hkv == Hq is fa_forward).
 *   window   0: none.  >= 1 needs causal == 1 (FA_ERR_UNSUPPORTED
 *            otherwise); a window >= N is the same as none.  < 0:
 *            FA_ERR_INVALID_ARG.
 *   alibi_slopes  NULL, or a DEVICE array of Hq fp32 slopes m_h (4-byte
 *            aligned): ALiBi ("03. FlashAttention", "Variantes et
 *            extensions": the linear bias fused into the kernel) adds
 *            -m_h * |i - j| to the scaled score of query i and key j of
 *            query head h before the softmax (under the causal mask this
 *            is m_h * (j - i)); LSE includes the bias.
 *   Other arguments as in fa_forward.  Allocates nothing.
 */
int fa_forward_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                   int window, const float* alibi_slopes, cudaStream_t stream);

/*
 * fa_forward_fp8 -- the forward pass with 8-bit floating-point inputs
 * ("03. FlashAttention", "FlashAttention v3": hardware FP8 as a lever).
 *
 * q, k, v hold OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; no infinities; 0x7F/0xFF are NaN), one byte per element,
 * in the layouts of fa_forward_gqa.  Their real values are code * descale:
 *   O = softmax(scale * (q_descale Q)(k_descale K)^T [+ mask]) (v_descale V)
 * Products run on the tensor cores with fp32 accumulation; P is rounded to
 * E4M3 (round to nearest even) before the P V product, which adds an error
 * of at most 2^-4 relative to each weight.  o is bf16, lse fp32 (natural
 * log), as in fa_forward.
 *
 *   Hkv, causal, window, alibi_slopes  as in fa_forward_gqa.
 *   descale factors      finite and > 0.
 *   ws                   NULL: a workspace (a transposed copy of V) comes
 *                        from the library pool; otherwise a caller buffer of
 *                        ws_bytes >= fa_workspace_size(FA_OP_FORWARD_FP8,
 *                        B, Hkv, N, d, 0) bytes, 256-byte aligned.
 *   d must be 128.  Returns as fa_forward, or FA_ERR_NO_MEMORY.
 */
int fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int Hq, int Hkv, int N, int d, float scale, float q_descale,
                   float k_descale, float v_descale, int causal, int window,
                   const float* alibi_slopes, void* ws, size_t ws_bytes,
                   cudaStream_t stream);

/*
 * fa_backward -- gradients dQ, dK, dV by recomputation.
 *
 * Only O and the per-row statistic (here LSE) are kept from the forward
 * pass, and P is recomputed tile by tile ("03. FlashAttention", "Backward
 * pass"; "FlashAttention ontleed", "Geheugencomplexiteit").  With
 * P = exp(scale Q K^T - LSE) and D_i = sum_k dO_ik O_ik:
 *   dV = P^T dO,  dS = P * (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q.
 *
 *   q, k, v, o, dO  [B,H,N,d] bf16, read only (o is the forward output).
 *   lse             [B,H,N] fp32 from fa_forward with the same arguments.
 *   dq, dk, dv      [B,H,N,d] bf16, written.
 *   d must be 128.  Other arguments as in fa_forward.
 * Workspace: fa_workspace_size(FA_OP_BACKWARD, ...) bytes (an fp32 dQ
 * accumulator, D and a scaled copy of LSE), taken on `stream` from a
 * stream-ordered memory pool the library keeps per device (freed blocks
 * stay cached for later calls) and released on the same stream.
 * FA_ERR_NO_MEMORY if that allocation fails.  dQ is summed with fp32 atomics: the result is not
 * bitwise reproducible from run to run (the pages accept summation-order
 * differences: "FlashAttention ontleed", "Beperkingen").
 */
int fa_backward(const void* q, const void* k, const void* v, const void* o,
                const float* lse, const void* dO, void* dq, void* dk, void* dv,
                int B, int H, int N, int d, float scale, int causal,
                cudaStream_t stream);

/*
 * fa_backward_ex -- fa_backward with a caller-owned workspace.
 *   ws        device buffer of ws_bytes >= fa_workspace_size(FA_OP_BACKWARD,
 *             B, H, N, d, 0) bytes, 256-byte aligned; contents are
 *             overwritten.  Nothing is allocated.
 */
int fa_backward_ex(const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const void* dO, void* dq, void* dk,
                   void* dv, int B, int H, int N, int d, float scale,
                   int causal, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * fa_backward_gqa -- fa_backward with grouped query heads, an optional
 * causal sliding window and optional ALiBi slopes (same meaning as in
 * fa_forward_gqa; the slopes must match the forward call's), and an
 * optional deterministic dQ.  dK and dV of a
 * key/value head are the sums of the gradients of its g query heads.
 *
 *   q, o, dO, dq  [B,Hq,N,d] bf16;  k, v, dk, dv [B,Hkv,N,d] bf16;
 *   lse           [B,Hq,N] fp32 from fa_forward_gqa with the same arguments.
 *   deterministic 0: dQ is summed over key blocks with fp32 atomics (fast;
 *                 summation order varies from run to run).  1: dK and dV
 *                 come from one kernel and dQ from a second one that walks
 *                 the key blocks of each 128-query block in a fixed order
 *                 and writes dQ once; dQ, dK and dV are then bitwise
 *                 reproducible (about 40% more work: S and dP are computed
 *                 twice).  Other values: FA_ERR_INVALID_ARG.
 *   ws            NULL: the workspace comes from the library pool as in
 *                 fa_backward; otherwise a caller-owned device buffer of
 *                 ws_bytes >= fa_workspace_size(FA_OP_BACKWARD, B, Hq, N, d, 0)
 *                 bytes, 256-byte aligned, and nothing is allocated.
 *   Other arguments as in fa_backward.
 */
int fa_backward_gqa(const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, void* dq, void* dk, void* dv,
                    int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                    int window, const float* alibi_slopes, int deterministic, void* ws,
                    size_t ws_bytes, cudaStream_t stream);

/*
 * fa_decode -- split-KV attention of one new query token per sequence over
 * its KV cache (FlashDecoding: "FlashAttention ontleed", "Interactie met de
 * KV-cache"; "03. FlashAttention", "Variantes et extensions"; Lensa ML FAQ
 * on decoding).  The Lkv cached rows of each (b, h) are cut into
 * num_splits contiguous parts of ceil(Lkv / num_splits) rows (the last one
 * shorter, possibly empty); one thread block per part runs the online
 * softmax over its rows and leaves a partial output O_s and its lse_s; a
 * second kernel merges the parts with the rescaling of "Tiling en Online
 * Softmax" applied across parts:
 *   L = ln sum_s e^(lse_s),  o = sum_s e^(lse_s - L) O_s.
 *
 *   q       [B,H,d] bf16;  kcache, vcache [B,H,Lkv,d] bf16;  o [B,H,d] bf16.
 *   d must be 128; 1 <= num_splits <= min(Lkv, 1024).  scale = 1/sqrt(d)
 *   (no scale argument; use fa_decode_ex for another one).
 * Workspace: fa_workspace_size(FA_OP_DECODE, ...) bytes of fp32 partials,
 * taken on `stream` from the library's per-device stream-ordered pool and
 * released on the same stream.
 */
int fa_decode(const void* q, const void* kcache, const void* vcache, void* o,
              int B, int H, int Lkv, int d, int num_splits,
              cudaStream_t stream);

/*
 * fa_decode_ex -- fa_decode with an explicit scale, an optional fp32 LSE
 * output [B,H] (lse_out may be NULL) and an optional caller-owned workspace
 * (ws may be NULL, then the workspace is allocated as in fa_decode;
 * otherwise ws_bytes >= fa_workspace_size(FA_OP_DECODE, B, H, Lkv, d,
 * num_splits), 256-byte aligned, and nothing is allocated).
 */
int fa_decode_ex(const void* q, const void* kcache, const void* vcache, void* o,
                 float* lse_out, int B, int H, int Lkv, int d, int num_splits,
                 float scale, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * fa_decode_gqa -- fa_decode_ex with grouped query heads: the g = Hq / Hkv
 * query rows that share a key/value head are computed together, so every
 * cache row is read from memory once for all of them ("FlashAttention
 * ontleed", "Interactie met de KV-cache").
 *
 *   q, o      [B,Hq,d] bf16;  kcache, vcache [B,Hkv,Lkv,d] bf16;
 *   lse_out   [B,Hq] fp32 or NULL.
 *   alibi_slopes  NULL, or a DEVICE array of Hq fp32 slopes: the new token
 *             sits at position Lkv - 1, so cache row j of query head h gets
 *             -slope_h * (Lkv - 1 - j) on its score (ALiBi, as in
 *             fa_forward_gqa).
 *   Hkv >= 1, Hq % Hkv == 0, B*Hq <= 65535.  Splits, scale and workspace as
 *   in fa_decode_ex, with the workspace sized by
 *   fa_workspace_size(FA_OP_DECODE, B, Hq, Lkv, d, num_splits); num_splits
 *   0 takes fa_decode_splits(B, Hq, Hkv, Lkv) (size a caller workspace with
 *   that value).
 */
int fa_decode_gqa(const void* q, const void* kcache, const void* vcache, void* o,
                  float* lse_out, int B, int Hq, int Hkv, int Lkv, int d,
                  int num_splits, float scale, const float* alibi_slopes, void* ws,
                  size_t ws_bytes, cudaStream_t stream);

/*
 * fa_decode_splits -- the split count fa_decode_gqa uses for num_splits = 0:
 * enough thread blocks for about 16 waves on the current device, at least
 * 512 cache rows per split, at most min(Lkv, 1024).  Returns 0 for invalid
 * sizes.
 */
int fa_decode_splits(int B, int Hq, int Hkv, int Lkv);

/*
 * fa_decode_noalloc -- fa_decode_ex without any allocation.  The pages have
 * no counterpart: this entry point exists for callers that cannot allocate
 * device memory themselves or let a library do it, e.g. a plugin running
 * inside a host framework that owns every byte of device memory, or a
 * latency-critical loop in which a cudaMalloc could stall the device.  The
 * caller still passes the inputs and outputs, exactly as for fa_decode_ex
 * (lse_out may be NULL); the split partials go to a fixed scratch array
 * that the library holds on every GPU that loads it (about 8.5 MB, until the
 * process exits).
 *
 *   Limit: B * H * num_splits <= 16384 partial results; larger requests are
 *   rejected with FA_ERR_UNSUPPORTED and a message, and nothing is launched.
 *   The first call on a device looks up that device's scratch address
 *   (with the device current); make that first call before any stream
 *   capture.  All calls share the one scratch array and its contents persist
 *   between calls (every partial is written before it is read, so nothing
 *   needs clearing); calls whose work overlaps on the GPU race on it, so
 *   order them on one stream or synchronise between them.
 * Calls no cudaMalloc, cudaFree or other allocating routine.
 */
int fa_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                      void* o, float* lse_out, int B, int H, int Lkv, int d,
                      int num_splits, float scale, cudaStream_t stream);

/*
 * fa_workspace_size -- device workspace bytes needed by an operation.
 *   op           FA_OP_FORWARD (always 0), FA_OP_BACKWARD, FA_OP_DECODE or
 *                FA_OP_FORWARD_FP8.
 *   H            the number of query heads (Hq for the _gqa calls); for
 *                FA_OP_FORWARD_FP8 the number of key/value heads Hkv.
 *   n_or_lkv     N for forward/backward, Lkv for decode.
 *   num_splits   decode only; ignored otherwise.
 * Returns 0 for invalid arguments.
 */
size_t fa_workspace_size(int op, int B, int H, int n_or_lkv, int d,
                         int num_splits);

/*
 * fa_get_device_status -- synchronises `stream`, then returns FA_OK, or
 * FA_ERR_TIMEOUT if any kernel of this library recorded a wait that ran out
 * since the previous call (the record is cleared), or FA_ERR_CUDA if the
 * synchronisation itself failed.
 */
int fa_get_device_status(cudaStream_t stream);

/*
 * fa_selftest_timeout -- diagnostic for the timeout path.  Launches one
 * thread block that waits, with the same bounded wait the kernels use but a
 * limit of limit_ms milliseconds (1 .. 10000), on an mbarrier that nothing
 * completes.  The wait runs out, records FA_ERR_TIMEOUT in the device status
 * word and the block exits normally (no trap or fault; the context stays
 * usable), so the next fa_get_device_status on that stream returns
 * FA_ERR_TIMEOUT and clears it.  Returns FA_OK once launched.
 *
 * Host-side fault injection: with the environment variable
 * FA_DEBUG_FAIL_ALLOC=1 every workspace allocation of the library fails and
 * the calls that need one return FA_ERR_NO_MEMORY without launching.
 */
int fa_selftest_timeout(unsigned limit_ms, cudaStream_t stream);

/*
 * fa_set_timing_events -- measurement hook.  While set (both non-NULL), every
 * later call made on this host thread records `before` on its stream just
 * before launching its main kernel (the fused forward kernel, the backward
 * dK/dV/dQ kernel) and `after` just after it, so cudaEventElapsedTime(before,
 * after) is that kernel's device time.  For the decode calls the span covers
 * both kernels, the split pass and the combine that merges its parts.  The
 * events are created and owned by the caller.  Pass NULL, NULL to stop.
 * Returns FA_OK, or FA_ERR_INVALID_ARG if exactly one event is NULL.
 */
int fa_set_timing_events(cudaEvent_t before, cudaEvent_t after);

/* fa_last_error -- message for the last failure on the calling host thread
 * ("" when none).  The string stays valid until the next call on that
 * thread. */
const char* fa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
