// tl_internal.cuh -- declarations shared by the library's translation units.
#pragma once

#include "tl.h"

#include <cuda_runtime.h>

#include <cstddef>

// Device-side status codes written into the workspace status word.
#define TL_DEVERR_TIMEOUT 1

namespace tl_internal {

#ifdef __CUDACC__
// rint(v / s) for the per-token quantisers, with r = 1/s rounded to nearest:
// v * r is within three units in the last place of the IEEE quotient
// fl(v / s), so it rounds to the same integer unless it lies that close to
// a half-integer (or is not finite); only then is the quotient formed.
// With q = rint(t), t - q is exact (q is within 0.5 of t) and 0.5 - |t - q|
// is t's distance to the nearest half-integer; the fast path asks for more
// than |t| * 2^-20 of it.
__device__ __forceinline__ float quant_round(float v, float s, float r) {
    const float t = __fmul_rn(v, r);
    const float q = rintf(t);
    if (fabsf(__fsub_rn(t, q)) < __fmaf_rn(-fabsf(t), 0x1p-20f, 0.5f)) return q;
    return rintf(__fdiv_rn(v, s));
}
#endif

// Batches from this size up run on the tensor-core prefill kernel.
constexpr int kPrefillMinN = 256;
// Bytes at the start of every workspace reserved for the status word.
constexpr size_t kStatusBytes = 256;

// Workspace layout of every call.  The bytes a call needs zero when it
// starts, and leaves zero when it ends (status word, arrival counters,
// exchange slots), sit at the front; its scratch (partial sums, per-call
// counters cleared at the call's start, converted activations) sits at the
// back, ending at the workspace's end.  A call asks for twice the larger of
// the two (plus alignment), so any calls sharing a workspace of the largest
// size asked for never write into one another's front bytes.
inline size_t round256(size_t b) { return (b + 255) / 256 * 256; }
inline size_t workspace_need(size_t front, size_t back) {
    return 2 * (front > back ? front : back) + 256;
}
// Offset of a call's scratch of `back` bytes in a workspace of `ws_bytes`
// (256-aligned; the workspace itself is 256-aligned).
inline size_t scratch_offset(size_t ws_bytes, size_t back) {
    return (ws_bytes - back) / 256 * 256;
}

// SM count of the current device (its attributes set up on first use).
tl_status device_sms(int *sms);
// Raise the head, fused and block-scale kernels' shared-memory limits on the
// current device.
tl_status head_init_device();
tl_status fused_init_device();
tl_status blockscale_init_device();

// The per-token quantiser (as tl_quantize_act) over bf16 X [N][K]: Q as int8,
// or with bf16_out the same integers held exactly in bf16; launched with the
// programmatic-dependent-launch attribute.
tl_status launch_quant(const void *X_bf16, int N, int K, void *Q, bool bf16_out, float *s,
                       int32_t *z, int symmetric, cudaStream_t stream);

size_t prefill_workspace_bytes(const tl_weight *Ws, int G, int N, int K, int mode, int sms);
bool prefill_supported(int N, int K);
tl_status prefill_init_device();
tl_status launch_prefill(const tl_weight *Ws, int G, const void *X, const float *s,
                         const int32_t *z, void *const *Ys, int N, int mode, int out, void *ws,
                         size_t ws_bytes, unsigned flags, cudaStream_t stream);

// The N <= 8 decode / verify kernel over all N in chunks of 8, with a given
// scratch buffer used by this call alone; `need` is the scratch it requires
// for these shapes and `zeroed` the leading bytes (status word, arrival
// counters and exchange slots) that must be zero when a call starts.
tl_status decode_scratch_bytes(const tl_weight *Ws, int G, size_t *need, size_t *zeroed);
tl_status launch_decode(const tl_weight *Ws, int G, const void *X, const float *s,
                        const int32_t *z, void *const *Ys, int N, int mode, int out, void *ws,
                        size_t ws_bytes, unsigned flags, cudaStream_t stream);

}  // namespace tl_internal
