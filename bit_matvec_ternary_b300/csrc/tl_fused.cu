// tl_fused.cu -- the linears' neighbours, fused with the activation
// quantiser: RMSNorm + quantisation (in front of q/k/v and gate/up) and
// SwiGLU + quantisation (in front of down).
//
// Each decoder layer normalises its input with RMSNorm (eps 1e-6) before
// the q/k/v and gate/up projections, and its feed-forward is SwiGLU
// ("Neutrino-1 8B" model page, "Architecture": Qwen3 geometry).  In mode B
// the next linear reads int8 activations, so the quantiser follows each of
// these directly; fusing them reads the row once and launches once.
//
// One CTA per token (the rows are at most a few tens of KB): the op's bf16
// output row is formed in fp32 and rounded to bf16 into shared memory, its
// minimum and maximum (or largest magnitude) are reduced in a fixed order,
// and the row is quantised exactly as tl_quantize_act quantises a bf16 row,
// so Q, s and z are bit for bit what that call gives on the bf16 output.
//   RMSNorm: y = bf16(x * r * gamma), r = 1 / sqrt(sum x^2 / K + eps), with
//            IEEE division and square root, the sum in a fixed order.
//   SwiGLU:  h = bf16(g / (1 + exp(-g)) * u), exp from the CUDA math library.
#include "tl.h"
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace {

constexpr int kFThreads = 1024;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFMaxRow = 32768;      // bf16 elements of a row staged in shared memory

struct FusedArgs {
    const uint16_t *X;      // rmsnorm: x [N][K]; swiglu: gate [N][K]
    const uint16_t *X2;     // rmsnorm: gamma [K]; swiglu: up [N][K]
    float eps;
    int K;
    uint16_t *Y;            // bf16 out [N][K] or null
    int8_t *Q;              // int8 out [N][K] or null
    float *s;
    int32_t *z;
    int symmetric;
};

__device__ __forceinline__ float bf(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Sum over the CTA in a fixed order (lanes by butterfly, then warps in order).
__device__ __forceinline__ float block_sum(float v, float *red) {
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < kFWarps; ++i) t = __fadd_rn(t, red[i]);
    return t;
}

template <int kOp>   // 0: RMSNorm, 1: SwiGLU
__global__ void __launch_bounds__(kFThreads)
tl_fused_kernel(const __grid_constant__ FusedArgs a) {
    extern __shared__ __align__(16) uint16_t row[];    // the bf16 output row
    __shared__ float red[kFWarps], rlo[kFWarps], rhi[kFWarps];
    __shared__ float s_sh;
    __shared__ int z_sh;
    const int n = blockIdx.x, K = a.K;
    const uint16_t *x = a.X + (long long)n * K;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float r = 0.f;
    if (kOp == 0) {
        float ss = 0.f;
        for (int k = threadIdx.x; k < K; k += kFThreads) {
            const float v = bf(__ldcg(x + k));
            ss = __fadd_rn(ss, __fmul_rn(v, v));
        }
        ss = block_sum(ss, red);
        r = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)K), a.eps)));
    }
    float lo = 0.f, hi = 0.f;
    for (int k = threadIdx.x; k < K; k += kFThreads) {
        float y;
        if (kOp == 0) {
            y = __fmul_rn(__fmul_rn(bf(__ldcg(x + k)), r), bf(__ldg(a.X2 + k)));
        } else {
            const float g = bf(__ldcg(x + k)), u = bf(__ldcg(a.X2 + (long long)n * K + k));
            y = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.f, expf(-g))), u);
        }
        const uint16_t h = __bfloat16_as_ushort(__float2bfloat16_rn(y));
        row[k] = h;
        const float yb = bf(h);
        if (a.symmetric) {
            hi = fmaxf(hi, fabsf(yb));
        } else {
            lo = fminf(lo, yb);
            hi = fmaxf(hi, yb);
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if ((threadIdx.x & 31) == 0) {
        rlo[threadIdx.x >> 5] = lo;
        rhi[threadIdx.x >> 5] = hi;
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (a.Y)
        for (int k = threadIdx.x; k < K; k += kFThreads) a.Y[(long long)n * K + k] = row[k];
    if (!a.Q) return;
    if (threadIdx.x == 0) {
        for (int w = 1; w < kFWarps; ++w) {
            lo = fminf(lo, rlo[w]);
            hi = fmaxf(hi, rhi[w]);
        }
        lo = fminf(lo, rlo[0]);
        hi = fmaxf(hi, rhi[0]);
        float s;
        int z;
        if (a.symmetric) {
            s = hi == 0.f ? 1.f : __fdiv_rn(hi, 127.f);
            z = 0;
        } else if (hi == lo) {
            s = 1.f;
            z = 0;
        } else {
            s = __fdiv_rn(__fsub_rn(hi, lo), 255.f);
            z = -128 - (int)rintf(__fdiv_rn(lo, s));
        }
        s_sh = s;
        z_sh = z;
        a.s[n] = s;
        a.z[n] = z;
    }
    __syncthreads();
    const float s = s_sh, rs = __frcp_rn(s), zf = (float)z_sh;
    const float qlo = a.symmetric ? -127.f : -128.f;
    for (int k = threadIdx.x; k < K; k += kFThreads) {
        const float t = fminf(fmaxf(__fadd_rn(tl_internal::quant_round(bf(row[k]), s, rs), zf), qlo), 127.f);
        a.Q[(long long)n * K + k] = (int8_t)(int)t;
    }
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

tl_status launch_fused(int op, const void *X, const void *X2, float eps, int N, int K, void *Y,
                       int8_t *Q, float *s, int32_t *z, int symmetric, void *stream) {
    if (!X || !X2) return TL_ERR_NULL;
    if (!Y && !Q) return TL_ERR_NULL;
    if (Q && (!s || !z)) return TL_ERR_NULL;
    if (N < 1 || N > 65535 || K < 1 || K > kFMaxRow) return TL_ERR_SHAPE;
    if (!aligned(X, 2) || !aligned(X2, 2) || (Y && !aligned(Y, 2)) || (s && !aligned(s, 4)) ||
        (z && !aligned(z, 4)))
        return TL_ERR_ALIGN;
    if (!(eps >= 0.f)) return TL_ERR_BAD_VALUE;
    int sms = 0;
    const tl_status st = tl_internal::device_sms(&sms);
    if (st != TL_OK) return st;
    FusedArgs a;
    std::memset(&a, 0, sizeof a);
    a.X = static_cast<const uint16_t *>(X);
    a.X2 = static_cast<const uint16_t *>(X2);
    a.eps = eps;
    a.K = K;
    a.Y = static_cast<uint16_t *>(Y);
    a.Q = Q;
    a.s = s;
    a.z = z;
    a.symmetric = symmetric ? 1 : 0;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)N);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = (size_t)K * 2;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = op == 0 ? cudaLaunchKernelEx(&cfg, tl_fused_kernel<0>, a)
                                   : cudaLaunchKernelEx(&cfg, tl_fused_kernel<1>, a);
    return le == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

}  // namespace

namespace tl_internal {
tl_status fused_init_device() {
    if (cudaFuncSetAttribute(tl_fused_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFMaxRow * 2) != cudaSuccess ||
        cudaFuncSetAttribute(tl_fused_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFMaxRow * 2) != cudaSuccess)
        return TL_ERR_CUDA;
    return TL_OK;
}
}  // namespace tl_internal

extern "C" {

tl_status tl_rmsnorm_quant(const void *X, const void *gamma, float eps, int N, int K, void *Y,
                           int8_t *Q, float *s, int32_t *z, int symmetric, void *stream) {
    return launch_fused(0, X, gamma, eps, N, K, Y, Q, s, z, symmetric, stream);
}

tl_status tl_swiglu_quant(const void *G, const void *U, int N, int M, void *H, int8_t *Q, float *s,
                          int32_t *z, int symmetric, void *stream) {
    return launch_fused(1, G, U, 0.f, N, M, H, Q, s, z, symmetric, stream);
}

}  // extern "C"
