// tl_internal.cuh -- declarations shared by the library's translation units.
#pragma once

#include "tl.h"

#include <cuda_runtime.h>

#include <cstddef>

// Device-side status codes written into the workspace status word.
#define TL_DEVERR_TIMEOUT 1

namespace tl_internal {

// Batches from this size up run on the tensor-core prefill kernel.
constexpr int kPrefillMinN = 256;
// Bytes at the start of every workspace reserved for the status word.
constexpr size_t kStatusBytes = 256;

size_t prefill_workspace_bytes(const tl_weight *Ws, int G, int N, int K, int mode, int sms);
bool prefill_supported(int N, int K);
tl_status prefill_init_device();
tl_status launch_prefill(const tl_weight *Ws, int G, const void *X, const float *s,
                         const int32_t *z, void *const *Ys, int N, int mode, int out, void *ws,
                         size_t ws_bytes, unsigned flags, cudaStream_t stream);

// The N <= 8 decode / verify kernel over all N in chunks of 8, with a given
// scratch buffer; `need` is the scratch it requires for these shapes and
// `zeroed` the leading bytes (status word and arrival counters) that must
// be zero when a call starts.
tl_status decode_scratch_bytes(const tl_weight *Ws, int G, size_t *need, size_t *zeroed);
tl_status launch_decode(const tl_weight *Ws, int G, const void *X, const float *s,
                        const int32_t *z, void *const *Ys, int N, int mode, int out, void *ws,
                        size_t ws_bytes, unsigned flags, cudaStream_t stream);

}  // namespace tl_internal
