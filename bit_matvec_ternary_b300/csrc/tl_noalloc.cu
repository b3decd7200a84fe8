// tl_noalloc.cu -- tl_linear_noalloc: the decode / speculative-verify linear
// with its scratch memory in a fixed device array instead of a caller
// workspace.
//
// Who needs it: code that may not call cudaMalloc or any allocating routine
// at the point where it runs a linear -- for example a plug-in that runs
// inside another runtime's memory pool, a real-time loop where allocation
// is forbidden after start-up, or a host that only hands out input and
// output buffers.  They still pass inputs and outputs; the split-K partial
// sums and arrival counters live in `g_scratch` below.
//
// The array is a file-scope __device__ variable, so every GPU that loads
// this library holds TL_NOALLOC_SCRATCH_BYTES of it until the process
// exits.  Host code cannot use its name as a device address: every call
// looks the address up with cudaGetSymbolAddress in the current context (a
// __device__ symbol has its own address in each context), with that device
// current.  The first call in a context also loads the module there, so it
// should come before any stream capture.
#include "tl.h"
#include "tl_internal.cuh"

#include <cuda_runtime.h>


namespace {

__device__ __align__(256) unsigned char g_scratch[TL_NOALLOC_SCRATCH_BYTES];

tl_status scratch_address(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return TL_ERR_CUDA;
    *out = p;
    return TL_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

tl_status tl_linear_noalloc(const tl_weight *W, const void *X, const float *s, const int32_t *z,
                            void *Y, int N, int mode, int out_dtype, unsigned flags,
                            void *stream) {
    if (!W || !X || !Y) return TL_ERR_NULL;
    if (!W->packed || !W->scale) return TL_ERR_NULL;
    if (W->layout != TL_LAYOUT_TL2P_V2) return TL_ERR_UNSUPPORTED;
    if (W->M < 1 || W->K < 1 || W->M > TL_MAX_M || W->K > TL_MAX_K || N < 1) return TL_ERR_SHAPE;
    if (mode != TL_MODE_BF16 && mode != TL_MODE_I8) return TL_ERR_MODE;
    if (out_dtype != TL_OUT_F32 && out_dtype != TL_OUT_BF16 && out_dtype != TL_OUT_I32_RAW)
        return TL_ERR_MODE;
    if (out_dtype == TL_OUT_I32_RAW && mode != TL_MODE_I8) return TL_ERR_MODE;
    if (mode == TL_MODE_I8 && (!s || !z || !W->rowsum)) return TL_ERR_NULL;
    if (!aligned(W->packed, 16) || !aligned(W->scale, 4)) return TL_ERR_ALIGN;
    if (mode == TL_MODE_I8 && (!aligned(W->rowsum, 4) || !aligned(s, 4) || !aligned(z, 4)))
        return TL_ERR_ALIGN;
    if (mode == TL_MODE_BF16 && !aligned(X, 2)) return TL_ERR_ALIGN;
    if (!aligned(Y, out_dtype == TL_OUT_BF16 ? 2 : 4)) return TL_ERR_ALIGN;

    size_t need = 0, zeroed = 0;
    tl_status st = tl_internal::decode_scratch_bytes(W, 1, &need, &zeroed);
    if (st != TL_OK) return st;
    if (need > (size_t)TL_NOALLOC_SCRATCH_BYTES) return TL_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != TL_OK) return st;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the last call left; the status word and the
    // arrival counters must start at zero.
    if (cudaMemsetAsync(scratch, 0, zeroed, cs) != cudaSuccess) return TL_ERR_CUDA;
    void *Ys[1] = {Y};
    return tl_internal::launch_decode(W, 1, X, s, z, Ys, N, mode, out_dtype, scratch,
                                      (size_t)TL_NOALLOC_SCRATCH_BYTES, flags, cs);
}

}  // extern "C"
