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
// A token's row is split over a cluster of CTAs: SwiGLU (exp and a division
// per element) over up to eight CTAs of 256 threads, about 1,024 columns
// each, so that even one token keeps several SMs busy; RMSNorm (a few
// multiplies per element) over one CTA of 1,024 threads per 8,192 columns,
// where two cluster barriers would cost more than they save.  Each CTA
// forms its slice of the op's output in fp32 and rounds it to bf16 into
// shared memory; the RMSNorm sum of squares and the row's minimum and
// maximum (or largest magnitude) are reduced per CTA in a fixed order and
// exchanged through distributed shared memory, each CTA adding its peers'
// values in rank order, so all of them derive the same r, s and z; the row
// is then quantised exactly as tl_quantize_act quantises a bf16 row, so Q, s
// and z are bit for bit what that call gives on the bf16 output.
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

constexpr int kFMaxCluster = 8;      // CTAs per token (portable cluster size)
constexpr int kFMaxRow = 32768;      // bf16 elements of a row
constexpr int kFMaxSlice = 8192;     // columns per CTA, staged in shared memory
// Threads per CTA and columns per CTA, per op (0: RMSNorm, 1: SwiGLU).
__host__ __device__ constexpr int fused_threads(int op) { return op == 0 ? 1024 : 256; }
__host__ __device__ constexpr int fused_cols(int op) { return op == 0 ? 8192 : 1024; }
static_assert(kFMaxRow / fused_cols(0) <= kFMaxCluster && fused_cols(0) <= kFMaxSlice &&
              kFMaxRow / kFMaxCluster <= kFMaxSlice, "row slices");

struct FusedArgs {
    const uint16_t *X;      // rmsnorm: x [N][K]; swiglu: gate [N][K]
    const uint16_t *X2;     // rmsnorm: gamma [K]; swiglu: up [N][K]
    float eps;
    int K;
    int per;                // columns per CTA (a multiple of 8)
    uint16_t *Y;            // bf16 out [N][K] or null
    int8_t *Q;              // int8 out [N][K] or null
    float *s;
    int32_t *z;
    int symmetric;
};

__device__ __forceinline__ float bf(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Sum over the CTA in a fixed order (lanes by butterfly, then warps in order).
template <int kWarps>
__device__ __forceinline__ float block_sum(float v, float *red) {
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < kWarps; ++i) t = __fadd_rn(t, red[i]);
    return t;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster: shared-memory writes before it
// are visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The float at the same shared-memory variable of CTA `rank` of the cluster.
__device__ __forceinline__ float ld_peer(const float *p, uint32_t rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint32_t ra;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// kCl: the token's CTAs form a cluster (more than one); otherwise a plain
// launch, its CTA-local barrier and reads (a cluster launch measured about a
// microsecond slower for one CTA).
template <int kOp, bool kCl>   // 0: RMSNorm, 1: SwiGLU
__global__ void __launch_bounds__(fused_threads(kOp))
tl_fused_kernel(const __grid_constant__ FusedArgs a) {
    constexpr int kFThreads = fused_threads(kOp);
    constexpr int kFWarps = kFThreads / 32;
    auto sync_all = [] {
        if (kCl) cluster_sync();
        else __syncthreads();
    };
    auto peer = [](const float *p, uint32_t rank) { return kCl ? ld_peer(p, rank) : *p; };
    __shared__ uint16_t row[kFMaxSlice];               // this CTA's slice of the bf16 row
    __shared__ float red[kFWarps], rlo[kFWarps], rhi[kFWarps];
    __shared__ float c_ss, c_lo, c_hi;                 // this CTA's partials, read by its peers
    __shared__ float s_sh;
    __shared__ int z_sh;
    const int n = blockIdx.y, K = a.K;
    const uint32_t rank = kCl ? cluster_rank() : 0u;
    const int C = (int)gridDim.x;                      // one cluster per token
    const int k0 = (int)rank * a.per, k1 = min(K, k0 + a.per);
    const uint16_t *x = a.X + (long long)n * K;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float r = 0.f;
    if (kOp == 0) {
        float ss = 0.f;
        for (int k = k0 + threadIdx.x; k < k1; k += kFThreads) {
            const float v = bf(__ldcg(x + k));
            ss = __fadd_rn(ss, __fmul_rn(v, v));
        }
        ss = block_sum<kFWarps>(ss, red);
        if (threadIdx.x == 0) c_ss = ss;
        sync_all();
        float tot = 0.f;
        for (int c = 0; c < C; ++c) tot = __fadd_rn(tot, peer(&c_ss, (uint32_t)c));
        r = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)K), a.eps)));
    }
    float lo = 0.f, hi = 0.f;
    for (int k = k0 + threadIdx.x; k < k1; k += kFThreads) {
        float y;
        if (kOp == 0) {
            y = __fmul_rn(__fmul_rn(bf(__ldcg(x + k)), r), bf(__ldg(a.X2 + k)));
        } else {
            const float g = bf(__ldcg(x + k)), u = bf(__ldcg(a.X2 + (long long)n * K + k));
            y = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.f, expf(-g))), u);
        }
        const uint16_t h = __bfloat16_as_ushort(__float2bfloat16_rn(y));
        row[k - k0] = h;
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
    if (threadIdx.x == 0) {
        for (int w = 0; w < kFWarps; ++w) {
            lo = fminf(lo, rlo[w]);
            hi = fmaxf(hi, rhi[w]);
        }
        c_lo = lo;
        c_hi = hi;
    }
    sync_all();
    if (threadIdx.x == 0) {
        // the row's range (exact whatever the order), then s and z
        for (int c = 0; c < C; ++c) {
            lo = fminf(lo, peer(&c_lo, (uint32_t)c));
            hi = fmaxf(hi, peer(&c_hi, (uint32_t)c));
        }
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
        if (a.Q && rank == 0) {
            a.s[n] = s;
            a.z[n] = z;
        }
    }
    // no CTA goes on (or leaves) while a peer may still read its partials
    sync_all();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (a.Y)
        for (int k = k0 + threadIdx.x; k < k1; k += kFThreads) a.Y[(long long)n * K + k] = row[k - k0];
    if (!a.Q) return;
    const float s = s_sh, rs = __frcp_rn(s), zf = (float)z_sh;
    const float qlo = a.symmetric ? -127.f : -128.f;
    for (int k = k0 + threadIdx.x; k < k1; k += kFThreads) {
        const float t = fminf(fmaxf(__fadd_rn(tl_internal::quant_round(bf(row[k - k0]), s, rs), zf), qlo), 127.f);
        a.Q[(long long)n * K + k] = (int8_t)(int)t;
    }
}

// CTAs per token: about fused_cols(op) columns each, at most a cluster of eight.
int fused_ctas(int op, int K) {
    const int c = (K + fused_cols(op) - 1) / fused_cols(op);
    return c < 1 ? 1 : c > kFMaxCluster ? kFMaxCluster : c;
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
    const int C = fused_ctas(op, K);
    a.per = ((K + C - 1) / C + 7) / 8 * 8;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)C, (unsigned)N);
    cfg.blockDim = dim3((unsigned)fused_threads(op));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C > 1 ? 2 : 1;
    cudaError_t le;
    if (op == 0)
        le = C > 1 ? cudaLaunchKernelEx(&cfg, tl_fused_kernel<0, true>, a)
                   : cudaLaunchKernelEx(&cfg, tl_fused_kernel<0, false>, a);
    else
        le = C > 1 ? cudaLaunchKernelEx(&cfg, tl_fused_kernel<1, true>, a)
                   : cudaLaunchKernelEx(&cfg, tl_fused_kernel<1, false>, a);
    return le == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

}  // namespace

namespace tl_internal {
tl_status fused_init_device() { return TL_OK; }   // static shared memory only
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
