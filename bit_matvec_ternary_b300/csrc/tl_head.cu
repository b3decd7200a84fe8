// tl_head.cu -- the int8 output head with a fused argmax, and the int8
// embedding lookup.
//
// What runs here (Neutrino-1 pages): the projections are ternary, but the
// token embedding and the output head stay int8 with one higher-precision
// scale per row (blog "Neutrino-1: quantization is a training decision",
// "What's actually ternary"); the model page ("Neutrino-1 8B",
// "Architecture") lists them as two untied int8 tensors of vocabulary x
// hidden (151,936 x 4,096, 622 MB each).  Greedy decoding, and the draft /
// verify gate that accepts a drafted token only when it equals the
// verifier's own choice (fermionresearch.com/models, "Neutrino-1 0.6B"),
// read the head's argmax, so the argmax is fused into the head's pass and
// the logits need not be written at all.
//
// Kernel tl_head_kernel (1 <= N <= 8 tokens): HBM-bound, every byte of H is
// read once.  CTA c takes a contiguous range of rows; each warp takes one
// 4 KB row at a time, its lanes streaming the row with 16-byte loads
// (issued all at once, so a row's bytes are in flight together) and
// forming the exact integer dot products with dp4a against the tokens'
// int8 activations staged in shared memory, together with the row's sum.
// The warp reduces them with shuffles, lane n applies the epilogue for
// token n and keeps that token's running best as a 64-bit key (an
// order-preserving image of the fp32 logit above ~index, so the largest key
// is the largest logit at its smallest index).  The CTAs' keys go to the
// workspace; the CTA that arrives last (arrival counter) reduces them and
// writes the tokens and their logits, then clears the counter.
//
// Kernel tl_head_mma_kernel (3 <= N <= 8 tokens, D a multiple of 512 up to
// 4096): at
// eight tokens dp4a and the shared-memory reads of every token's activations
// per 16 bytes of H would bound the dp4a kernel well below the HBM rate, so
// the products go to the tensor cores instead.  A CTA's eight warps work on
// one 16-row group of H at a time, warp w taking columns [w D/8, (w+1) D/8):
// lane (g, t) loads 16 bytes of rows g and g + 8 per 64 columns (all of the
// warp's share in flight at once, in two halves: the next group's half is
// issued as soon as this group's half has been read), turns each int8 pair
// into exact fp16 (a
// byte permute under a 2^10 exponent, then 1152 subtracted), and multiplies
// them by the tokens' activations (staged once per CTA as exact fp16) with
// mma.m16n8k16 into fp32.  Products are integers of at most 2^14 and a warp
// sums at most 512 columns, so every partial sum is an exact fp32 integer;
// the column order inside a 64-column step is permuted identically for both
// operands, which a dot product does not see.  The warps' integer sums and
// dp4a row sums meet in shared memory (two buffers, one barrier a group),
// and warp (group mod 8) adds them in warp order, applies the same epilogue
// and keeps the same keys.
#include "tl.h"
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace {

constexpr int kHWarps = 8;
constexpr int kHThreads = kHWarps * 32;
constexpr int kHCtasPerSm = 2;
constexpr int kHUnroll = 8;            // 16-byte loads in flight per lane (one 4 KB row)
constexpr int kHMaxQBytes = 96 * 1024; // N * D bytes of activations staged per CTA

struct HeadArgs {
    const int8_t *H;
    const float *scale;
    const int8_t *Q;
    const float *s;
    const int32_t *z;
    float *logits;                 // [N][V] or null
    int32_t *token;                // [N]
    float *best;                   // [N]
    unsigned long long *keys;      // [gridDim][N] the CTAs' best keys (scratch)
    unsigned *cnt;                 // CTAs done; zero between calls
    long long V;
    long long rows_per_cta;
    int D, N;
};

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int dp4(uint32_t a, uint32_t b, int c) {
    return __dp4a((int)a, (int)b, c);
}

// Larger key: larger logit; for equal logits, smaller row index.  -0 orders
// as +0, so equal values compare equal.
__device__ __forceinline__ unsigned long long head_key(float y, long long v) {
    uint32_t b = __float_as_uint(y);
    if (b == 0x80000000u) b = 0u;
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)ord << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)v);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
    const uint32_t ord = (uint32_t)(k >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
__device__ __forceinline__ int key_index(unsigned long long k) {
    return (int)(0xFFFFFFFFu - (uint32_t)k);
}

template <int NT>
__global__ void __launch_bounds__(kHThreads, kHCtasPerSm)
tl_head_kernel(const __grid_constant__ HeadArgs a) {
    extern __shared__ __align__(16) uint8_t qs[];      // [N][D] int8 activations
    __shared__ unsigned long long wbest[kHWarps][NT];
    __shared__ int is_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long r0 = (long long)blockIdx.x * a.rows_per_cta;
    const long long r1 = r0 + a.rows_per_cta < a.V ? r0 + a.rows_per_cta : a.V;
    // the rows do not depend on the previous kernel: start the first ones
    // toward L2 before waiting for it
    for (long long v = r0 + threadIdx.x / 16; v < r0 + 2 * kHWarps && v < r1; v += kHThreads / 16)
        for (int b = (threadIdx.x % 16) * 128; b < a.D; b += 16 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.H + v * a.D + b));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int chunks = a.D / 16;                         // 16-byte chunks per row
    for (int i = threadIdx.x; i < a.N * chunks; i += kHThreads)
        reinterpret_cast<uint4 *>(qs)[i] = __ldcg(reinterpret_cast<const uint4 *>(a.Q) + i);
    float s_l = 0.f;
    int z_l = 0;
    if (lane < a.N) {
        s_l = __ldcg(a.s + lane);
        z_l = __ldcg(a.z + lane);
    }
    __syncthreads();

    unsigned long long mybest = 0ull;                    // lane n: token n's best key
    for (long long v = r0 + warp; v < r1; v += kHWarps) {
        const uint4 *hrow = reinterpret_cast<const uint4 *>(a.H + v * a.D);
        int acc[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n] = 0;
        int rs = 0;
        for (int c0 = 0; c0 < chunks; c0 += 32 * kHUnroll) {
            uint4 h[kHUnroll];
#pragma unroll
            for (int u = 0; u < kHUnroll; ++u) {
                const int c = c0 + 32 * u + lane;
                h[u] = c < chunks ? ld_stream(hrow + c) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kHUnroll; ++u) {
                const int c = c0 + 32 * u + lane;
                if (c >= chunks) break;
                rs = dp4(h[u].x, 0x01010101u, rs);
                rs = dp4(h[u].y, 0x01010101u, rs);
                rs = dp4(h[u].z, 0x01010101u, rs);
                rs = dp4(h[u].w, 0x01010101u, rs);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if (n >= a.N) break;
                    const uint4 q = reinterpret_cast<const uint4 *>(qs)[n * chunks + c];
                    acc[n] = dp4(h[u].x, q.x, acc[n]);
                    acc[n] = dp4(h[u].y, q.y, acc[n]);
                    acc[n] = dp4(h[u].z, q.z, acc[n]);
                    acc[n] = dp4(h[u].w, q.w, acc[n]);
                }
            }
        }
        // exact integer sums over the warp (order does not matter)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            rs += __shfl_xor_sync(0xffffffffu, rs, off);
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], off);
        }
        int mine = 0;
#pragma unroll
        for (int n = 0; n < NT; ++n)
            if (n == lane) mine = acc[n];
        if (lane < a.N) {
            const int corrected = mine - z_l * rs;
            const float y = __fmul_rn(__fmul_rn(__int2float_rn(corrected), s_l), __ldg(a.scale + v));
            if (a.logits) a.logits[(long long)lane * a.V + v] = y;
            const unsigned long long k = head_key(y, v);
            if (k > mybest) mybest = k;
        }
    }
    if (lane < NT) wbest[warp][lane] = mybest;
    __syncthreads();
    if (threadIdx.x < a.N) {
        unsigned long long b = 0ull;
        for (int w = 0; w < kHWarps; ++w) b = wbest[w][threadIdx.x] > b ? wbest[w][threadIdx.x] : b;
        __stcg(a.keys + (long long)blockIdx.x * a.N + threadIdx.x, b);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        is_last = atomicAdd(a.cnt, 1u) + 1u == gridDim.x;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // the last CTA: one warp per token over every CTA's key
    for (int n = warp; n < a.N; n += kHWarps) {
        unsigned long long b = 0ull;
        for (int c = lane; c < (int)gridDim.x; c += 32) {
            const unsigned long long k = __ldcg(a.keys + (long long)c * a.N + n);
            b = k > b ? k : b;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, b, off);
            b = o > b ? o : b;
        }
        if (lane == 0) {
            a.token[n] = key_index(b);
            a.best[n] = key_value(b);
        }
    }
    if (threadIdx.x == 0) *a.cnt = 0u;
}

// ---- the tensor-core form for 5..8 tokens
constexpr int kHMmaRows = 16;                  // rows of H per group
constexpr int kHMmaStep = 64;                  // columns per lane step (16 bytes of each row)
constexpr int kHMmaMaxStage = 100 * 1024;      // fp16 activations staged per CTA

__device__ __forceinline__ void mma16816_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Bytes 2h and 2h + 1 of w (signed int8) as an exact fp16 pair: the bytes,
// offset by 128, become the low mantissa bits under exponent 10 (1024 + u),
// and 1152 = 1024 + 128 is subtracted (exact: integers below 2^11).
__device__ __forceinline__ uint32_t i8pair_to_f16x2(uint32_t w, int h) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w ^ 0x80808080u), "r"(0x64646464u),
        "r"(h ? 0x5342u : 0x5140u));
    __half2 v = *reinterpret_cast<const __half2 *>(&r);
    v = __hsub2(v, __halves2half2(__ushort_as_half((unsigned short)0x6480u),
                                  __ushort_as_half((unsigned short)0x6480u)));
    return *reinterpret_cast<const uint32_t *>(&v);
}

__global__ void __launch_bounds__(kHThreads, kHCtasPerSm)
tl_head_mma_kernel(const __grid_constant__ HeadArgs a) {
    extern __shared__ __align__(16) uint8_t xs_raw[];   // fp16 [8][D + 8]
    __shared__ int part[2][kHWarps][32][6];             // 4 dot products, 2 row sums per lane
    __shared__ unsigned long long wbest[kHWarps][8];
    __shared__ int is_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long r0 = (long long)blockIdx.x * a.rows_per_cta;
    const long long r1 = r0 + a.rows_per_cta < a.V ? r0 + a.rows_per_cta : a.V;
    const int stride = a.D + 8;                         // fp16 per staged row (16 bytes of padding)
    const int cols = a.D / kHWarps;                     // this warp's share of a row
    const int c_lo = warp * cols;
    // the rows do not depend on the previous kernel: start the first groups
    // toward L2 before waiting for it
    for (long long v = r0 + threadIdx.x / 16; v < r0 + 2 * kHMmaRows && v < r1; v += kHThreads / 16)
        for (int b = (threadIdx.x % 16) * 128; b < a.D; b += 16 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.H + v * a.D + b));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the tokens' int8 activations as exact fp16; tokens past N are zero
    __half *xs = reinterpret_cast<__half *>(xs_raw);
    for (int i = threadIdx.x; i < 8 * (a.D / 4); i += kHThreads) {
        const int n = i / (a.D / 4), d4 = (i - n * (a.D / 4)) * 4;
        uint32_t w = 0u;
        if (n < a.N) w = __ldcg(reinterpret_cast<const unsigned int *>(a.Q + (long long)n * a.D + d4));
        const uint2 h2 = make_uint2(i8pair_to_f16x2(w, 0), i8pair_to_f16x2(w, 1));
        *reinterpret_cast<uint2 *>(xs + n * stride + d4) = h2;
    }
    // this lane's tokens 2t, 2t + 1
    float s_t[2];
    int z_t[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int n = 2 * t + e;
        s_t[e] = n < a.N ? __ldcg(a.s + n) : 0.f;
        z_t[e] = n < a.N ? __ldcg(a.z + n) : 0;
    }
    __syncthreads();

    unsigned long long best[2] = {0ull, 0ull};          // tokens 2t, 2t + 1 (epilogue groups)
    const __half *xrow = xs + g * stride + 16 * t;      // token g; + column
    // this lane's 16 bytes of rows g and g + 8 of the group at v0, for each of
    // the warp's (at most eight) 64-column steps; zero past the CTA's rows
    uint4 wa[8], wb[8];
    // steps 4h .. 4h + 3 (half h) of the group at v0
    auto load_half = [&](long long v0, int h) {
        const long long ra = v0 + g, rb = v0 + g + 8;
        const int8_t *ha = a.H + ra * a.D + 16 * t;
        const int8_t *hb = a.H + rb * a.D + 16 * t;
#pragma unroll
        for (int u = 4 * h; u < 4 * h + 4; ++u) {
            const int cc = c_lo + u * kHMmaStep;
            const bool in = u * kHMmaStep < cols;
            wa[u] = in && ra < r1 ? ld_stream(reinterpret_cast<const uint4 *>(ha + cc)) : make_uint4(0u, 0u, 0u, 0u);
            wb[u] = in && rb < r1 ? ld_stream(reinterpret_cast<const uint4 *>(hb + cc)) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    if (r0 < r1) {
        load_half(r0, 0);
        load_half(r0, 1);
    }
    int pb = 0;
    for (long long v0 = r0, gi = 0; v0 < r1; v0 += kHMmaRows, ++gi) {
        const long long ra = v0 + g, rb = v0 + g + 8;
        const bool epi = warp == (int)(gi % kHWarps);
        // the epilogue's row scales, early
        const float sca = epi && ra < r1 ? __ldg(a.scale + ra) : 0.f;
        const float scb = epi && rb < r1 ? __ldg(a.scale + rb) : 0.f;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        int rs[2] = {0, 0};
        const bool more = v0 + kHMmaRows < r1;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (u == 4) {
                // the first half's registers are read: the next group's first
                // half goes out now (the empty asm keeps the compiler from
                // hoisting these loads above the MMAs that still read them)
                asm volatile("" ::: "memory");
                if (more) load_half(v0 + kHMmaRows, 0);
            }
            const int cc = c_lo + u * kHMmaStep;
            if (u * kHMmaStep >= cols) continue;
            const uint4 x0 = *reinterpret_cast<const uint4 *>(xrow + cc);
            const uint4 x1 = *reinterpret_cast<const uint4 *>(xrow + cc + 8);
            const uint32_t A[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
            const uint32_t B[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
            const uint32_t X[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int st = 0; st < 4; ++st) {
                // k-step st: columns 4st .. 4st + 3 of this lane's 16
                mma16816_f16(c, i8pair_to_f16x2(A[st], 0), i8pair_to_f16x2(B[st], 0),
                             i8pair_to_f16x2(A[st], 1), i8pair_to_f16x2(B[st], 1), X[2 * st],
                             X[2 * st + 1]);
                rs[0] = dp4(A[st], 0x01010101u, rs[0]);
                rs[1] = dp4(B[st], 0x01010101u, rs[1]);
            }
        }
        // and its second half, before the barrier and the epilogue
        asm volatile("" ::: "memory");
        if (more) load_half(v0 + kHMmaRows, 1);
        // this warp's exact integer sums for the group
        int *mine = part[pb][warp][lane];
#pragma unroll
        for (int i = 0; i < 4; ++i) mine[i] = __float2int_rn(c[i]);
        mine[4] = rs[0];
        mine[5] = rs[1];
        __syncthreads();
        if (epi) {
            int acc[4] = {0, 0, 0, 0}, rsum[2] = {0, 0};
#pragma unroll
            for (int w = 0; w < kHWarps; ++w) {
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] += part[pb][w][lane][i];
                rsum[0] += part[pb][w][lane][4];
                rsum[1] += part[pb][w][lane][5];
            }
            // the row sums over the four lanes of a row
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                rsum[0] += __shfl_xor_sync(0xffffffffu, rsum[0], o);
                rsum[1] += __shfl_xor_sync(0xffffffffu, rsum[1], o);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const long long v = i < 2 ? ra : rb;
                const int e = i & 1, n = 2 * t + e;
                if (v >= r1 || n >= a.N) continue;
                const int corrected = acc[i] - z_t[e] * rsum[i >> 1];
                const float y = __fmul_rn(__fmul_rn(__int2float_rn(corrected), s_t[e]), i < 2 ? sca : scb);
                if (a.logits) a.logits[(long long)n * a.V + v] = y;
                const unsigned long long k = head_key(y, v);
                if (k > best[e]) best[e] = k;
            }
        }
        pb ^= 1;
    }
    // each token's best over this warp's epilogue groups: lanes of equal t
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            const unsigned long long k = __shfl_xor_sync(0xffffffffu, best[e], o);
            best[e] = k > best[e] ? k : best[e];
        }
    if (g == 0) {
        wbest[warp][2 * t] = best[0];
        wbest[warp][2 * t + 1] = best[1];
    }
    __syncthreads();
    if (threadIdx.x < a.N) {
        unsigned long long b = 0ull;
        for (int w = 0; w < kHWarps; ++w) b = wbest[w][threadIdx.x] > b ? wbest[w][threadIdx.x] : b;
        __stcg(a.keys + (long long)blockIdx.x * a.N + threadIdx.x, b);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        is_last = atomicAdd(a.cnt, 1u) + 1u == gridDim.x;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int n = warp; n < a.N; n += kHWarps) {
        unsigned long long b = 0ull;
        for (int c2 = lane; c2 < (int)gridDim.x; c2 += 32) {
            const unsigned long long k = __ldcg(a.keys + (long long)c2 * a.N + n);
            b = k > b ? k : b;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, b, off);
            b = o > b ? o : b;
        }
        if (lane == 0) {
            a.token[n] = key_index(b);
            a.best[n] = key_value(b);
        }
    }
    if (threadIdx.x == 0) *a.cnt = 0u;
}

using HeadFn = void (*)(HeadArgs);
HeadFn head_kernel_for(int nt) {
    switch (nt) {
        case 1: return tl_head_kernel<1>;
        case 2: return tl_head_kernel<2>;
        case 4: return tl_head_kernel<4>;
        default: return tl_head_kernel<8>;
    }
}

// x[n][d] = bf16(E[t][d] * scale[t]) for t = tokens[n]; a token outside
// [0, V) gives a zero row.
__global__ void __launch_bounds__(256)
tl_embed_kernel(const int8_t *__restrict__ E, const float *__restrict__ scale, long long V, int D,
                const int32_t *__restrict__ tokens, __nv_bfloat16 *__restrict__ X) {
    const int n = blockIdx.y;
    const int t = __ldg(tokens + n);
    const bool ok = t >= 0 && (long long)t < V;
    const float sc = ok ? __ldg(scale + t) : 0.f;
    for (int d = blockIdx.x * blockDim.x + threadIdx.x; d < D; d += gridDim.x * blockDim.x) {
        const float y = ok ? __fmul_rn((float)__ldg(E + (long long)t * D + d), sc) : 0.f;
        X[(long long)n * D + d] = __float2bfloat16_rn(y);
    }
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int padded_tokens(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8; }

struct HeadPlan {
    int grid;
    long long rows_per_cta;
    size_t keys_off, bytes;
};

// The tensor-core form: three to eight tokens (measured on the 8B head: 122
// us at three to eight tokens, against 129 and 143.5 us on dp4a at three and
// four, 111 at two), rows split in whole 64-column steps over the eight
// warps, at most eight steps a warp (its loads held in registers; D <= 4096,
// within the exact fp32 range), the fp16 activations within the CTA's
// shared memory.
bool head_mma(int N, int D) {
    return N >= 3 && D % (kHWarps * kHMmaStep) == 0 && D <= kHWarps * 8 * kHMmaStep &&
           (size_t)8 * (D + 8) * 2 <= (size_t)kHMmaMaxStage;
}

HeadPlan head_plan(long long V, int D, int N, int sms) {
    HeadPlan p;
    const long long slots = (long long)sms * kHCtasPerSm;
    p.rows_per_cta = (V + slots - 1) / slots;
    // the tensor-core form takes whole 16-row groups
    if (head_mma(N, D)) p.rows_per_cta = (p.rows_per_cta + kHMmaRows - 1) / kHMmaRows * kHMmaRows;
    p.grid = (int)((V + p.rows_per_cta - 1) / p.rows_per_cta);
    p.keys_off = tl_internal::kStatusBytes + 256;    // status word, then the counter
    p.bytes = p.keys_off + tl_internal::round256((size_t)p.grid * N * 8);
    return p;
}

tl_status check_head_shape(long long V, int D, int N) {
    if (V < 1 || V >= 0x7FFFFFFFll || D < 16 || D % 16 != 0 || D > 32768 || N < 1 || N > 8)
        return TL_ERR_SHAPE;
    if ((long long)N * D > kHMaxQBytes) return TL_ERR_SHAPE;
    return TL_OK;
}

}  // namespace

namespace tl_internal {
tl_status head_init_device() {
    for (int nt = 1; nt <= 8; nt *= 2)
        if (cudaFuncSetAttribute(head_kernel_for(nt), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kHMaxQBytes) != cudaSuccess)
            return TL_ERR_CUDA;
    if (cudaFuncSetAttribute(tl_head_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kHMmaMaxStage) != cudaSuccess)
        return TL_ERR_CUDA;
    return TL_OK;
}
}  // namespace tl_internal

extern "C" {

size_t tl_head_workspace_bytes(int64_t V, int D, int N) {
    if (check_head_shape(V, D, N) != TL_OK) return 0;
    int sms = 148;
    if (tl_internal::device_sms(&sms) != TL_OK) sms = 148;
    return head_plan(V, D, N, sms).bytes;
}

tl_status tl_head_argmax(const int8_t *H, const float *scale, int64_t V, int D, const int8_t *Q,
                         const float *s, const int32_t *z, int N, float *logits, int32_t *token,
                         float *best, void *workspace, size_t workspace_bytes, unsigned flags,
                         void *stream) {
    if (!H || !scale || !Q || !s || !z || !token || !best) return TL_ERR_NULL;
    tl_status st = check_head_shape(V, D, N);
    if (st != TL_OK) return st;
    if (!aligned(H, 16) || !aligned(Q, 16) || !aligned(scale, 4) || !aligned(s, 4) ||
        !aligned(z, 4) || !aligned(token, 4) || !aligned(best, 4) ||
        (logits && !aligned(logits, 4)))
        return TL_ERR_ALIGN;
    if (!workspace) return TL_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return TL_ERR_ALIGN;
    int sms = 0;
    st = tl_internal::device_sms(&sms);
    if (st != TL_OK) return st;
    const HeadPlan p = head_plan(V, D, N, sms);
    if (workspace_bytes < p.bytes) return TL_ERR_WORKSPACE;
    const bool mma = head_mma(N, D);
    HeadArgs a;
    std::memset(&a, 0, sizeof a);
    a.H = H; a.scale = scale; a.Q = Q; a.s = s; a.z = z;
    a.logits = logits; a.token = token; a.best = best;
    char *ws = static_cast<char *>(workspace);
    a.cnt = reinterpret_cast<unsigned *>(ws + tl_internal::kStatusBytes);
    a.keys = reinterpret_cast<unsigned long long *>(ws + p.keys_off);
    a.V = V; a.rows_per_cta = p.rows_per_cta; a.D = D; a.N = N;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kHThreads);
    cfg.dynamicSmemBytes = mma ? (size_t)8 * (D + 8) * 2 : (size_t)N * D;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & TL_FLAG_PDL) ? 1 : 0;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, mma ? tl_head_mma_kernel : head_kernel_for(padded_tokens(N)), a);
    return le == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

tl_status tl_embed(const int8_t *E, const float *scale, int64_t V, int D, const int32_t *tokens,
                   int N, void *X_bf16, void *stream) {
    if (!E || !scale || !tokens || !X_bf16) return TL_ERR_NULL;
    if (V < 1 || D < 1 || N < 1 || N > 65535) return TL_ERR_SHAPE;
    if (!aligned(scale, 4) || !aligned(tokens, 4) || !aligned(X_bf16, 2)) return TL_ERR_ALIGN;
    int sms = 0;
    const tl_status st = tl_internal::device_sms(&sms);
    if (st != TL_OK) return st;
    const dim3 grid((unsigned)((D + 255) / 256 < 64 ? (D + 255) / 256 : 64), (unsigned)N);
    tl_embed_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        E, scale, V, D, tokens, static_cast<__nv_bfloat16 *>(X_bf16));
    return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

}  // extern "C"
