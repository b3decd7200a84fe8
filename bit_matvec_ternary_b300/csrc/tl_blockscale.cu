// tl_blockscale.cu -- the block-wise scale variant of the ternary linear.
//
// The blog ("Neutrino-1: quantization is a training decision", "What's
// actually ternary") describes the weights as blocks, each with its own
// higher-precision scale; the shipped 8B artifact keeps one scale per row
// (model page "Neutrino-1 8B", "Architecture"), which the main kernels use.
// This variant takes a scale per (row, 128-column block):
//     y[n, m] = sum_b scale[m, b] * sum_{k in b} w[m, k] * x[n, k]
// on the same TL2P v2 codes, bf16 activations, fp32 sums.
//
// Kernel: persistent CTAs of kBWarps warps, as many as fit on the SMs, each
// taking the row tiles r = blockIdx.x, blockIdx.x + gridDim.x, ...  A CTA
// first copies its tokens' activation rows into shared memory (zero past K
// up to a whole block; each row padded by 16 bytes, so the eight rows of a
// fragment load fall in different banks) when they fit, else activations
// are read from global memory through L1.  Within a row tile, warp w takes
// the blocks b = w, w + kBWarps, ... of K; lane (g, t) loads its 16 bytes of
// each of its tiles, kBU tiles a group, the next group's loads (of this row
// tile or the next) issued before the current group is multiplied.  Each
// tile's eight k-steps are decoded to bf16 2w (the field 1 - w moved to the
// sign and top exponent bits), multiplied by the tokens' bf16 activations
// on the tensor cores into fresh per-tile accumulators (two chains), and
// folded into the warp's running result with that block's scale (times
// 1/2).  At the end of a row tile the warps' results are added in warp
// order (shared memory, two buffers so one barrier a row tile suffices), so
// the sum is the same on every run and does not depend on the grid size.
#include "tl.h"
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace {

constexpr int kBWarps = 8;        // warps per CTA (the K split of a row tile)
constexpr int kBU = 4;            // tiles per load group
constexpr int kBMaxStage = 100 * 1024;  // shared-memory bytes for staged activations

struct BsArgs {
    const uint4 *packed;
    const float *bscale;          // [M][KB]
    const uint16_t *X;            // bf16 [N][K]
    void *Y;
    int M, K, KB, N, out, R;
    int x4;                       // X rows start on 4-byte boundaries (X aligned, K even)
    int xstride;                  // staged row length in bf16 (KB * 128 + 8)
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The field pair of k-step m of a TL2P v2 word as bf16x2 2w: 00 -> +2,
// 01 -> 0, 10 -> -2.
__device__ __forceinline__ uint32_t dec2w(uint32_t word, int m) {
    return ((word << (14 - 2 * m)) & 0xC000C000u) ^ 0x40004000u;
}

// Two consecutive bf16 activations of token n at column k (k even; zero past
// K or past the batch), from the staged rows or from global memory.
template <bool kStaged>
__device__ __forceinline__ uint32_t xpair(const BsArgs &a, const uint16_t *xsm, int n, int k) {
    if (n >= a.N) return 0u;
    if (kStaged) return *reinterpret_cast<const uint32_t *>(xsm + n * a.xstride + k);
    const uint16_t *x = a.X + (long long)n * a.K;
    // with 4-byte aligned rows the pair is one 32-bit load
    if (a.x4 && k + 1 < a.K) return __ldg(reinterpret_cast<const unsigned int *>(x + k));
    const uint32_t lo = k < a.K ? __ldg(x + k) : 0u;
    const uint32_t hi = k + 1 < a.K ? __ldg(x + k + 1) : 0u;
    return lo | (hi << 16);
}

// This lane's 16 bytes of the tiles of load group grp of row tile r: blocks
// warp + kBWarps * (grp * kBU + u), zero past KB.
__device__ __forceinline__ void load_group(const BsArgs &a, int r, int grp, int warp, int lane,
                                           uint4 (&w)[kBU]) {
    const uint4 *tiles = a.packed + (long long)r * a.KB * 32 + lane;
#pragma unroll
    for (int u = 0; u < kBU; ++u) {
        const int b = warp + kBWarps * (grp * kBU + u);
        w[u] = b < a.KB ? __ldg(tiles + (long long)b * 32) : make_uint4(0u, 0u, 0u, 0u);
    }
}

template <bool kStaged>
__global__ void __launch_bounds__(kBWarps * 32)
tl_blockscale_kernel(const __grid_constant__ BsArgs a) {
    __shared__ float part[2][kBWarps][32][4];
    extern __shared__ __align__(16) uint16_t xsm[];      // [N][xstride] when staged
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    // this warp's blocks of a row tile, in groups of kBU (at least one group,
    // so every warp passes the same row-tile barriers)
    const int nb = warp < a.KB ? (a.KB - warp + kBWarps - 1) / kBWarps : 0;
    const int ng = nb > 0 ? (nb + kBU - 1) / kBU : 1;
    int r = blockIdx.x, grp = 0;
    uint4 w[kBU];
    // the weights do not depend on the previous launch: start them first
    if (r < a.R) load_group(a, r, 0, warp, lane, w);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (kStaged) {
        // 16-byte copies of the N rows (K a multiple of 8, X 16-byte aligned),
        // zero from K to the end of the last block
        const int per_row = a.xstride / 8;
        for (int i = threadIdx.x; i < a.N * per_row; i += kBWarps * 32) {
            const int n = i / per_row, c = i - n * per_row;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (8 * c < a.K) v = __ldg(reinterpret_cast<const uint4 *>(a.X + (long long)n * a.K) + c);
            *reinterpret_cast<uint4 *>(xsm + n * a.xstride + 8 * c) = v;
        }
        __syncthreads();
    }
    float y[4] = {0.f, 0.f, 0.f, 0.f};                   // rows g, g+8 x tokens 2t, 2t+1
    int pb = 0;
    while (r < a.R) {
        // the next group's loads, before this group's arithmetic
        int rn = r, gn = grp + 1;
        if (gn == ng) { gn = 0; rn += gridDim.x; }
        uint4 wn[kBU];
        if (rn < a.R) load_group(a, rn, gn, warp, lane, wn);
        else {
#pragma unroll
            for (int u = 0; u < kBU; ++u) wn[u] = make_uint4(0u, 0u, 0u, 0u);
        }
        const int m0 = r * 16 + g, m1 = m0 + 8;
#pragma unroll
        for (int u = 0; u < kBU; ++u) {
            const int b = warp + kBWarps * (grp * kBU + u);
            if (b >= a.KB) break;
            float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int k = b * 128 + 16 * m + 2 * t;
                const uint32_t b0r = xpair<kStaged>(a, xsm, g, k);
                const uint32_t b1r = xpair<kStaged>(a, xsm, g, k + 8);
                mma16816((m & 1) ? c1 : c0, dec2w(w[u].x, m), dec2w(w[u].y, m), dec2w(w[u].z, m),
                         dec2w(w[u].w, m), b0r, b1r);
            }
            const float s0 = m0 < a.M ? __ldg(a.bscale + (long long)m0 * a.KB + b) : 0.f;
            const float s1 = m1 < a.M ? __ldg(a.bscale + (long long)m1 * a.KB + b) : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float v = __fmul_rn(__fadd_rn(c0[i], c1[i]), 0.5f);
                y[i] = __fmaf_rn(v, i < 2 ? s0 : s1, y[i]);
            }
        }
        if (grp == ng - 1) {
            // the row tile is done in every warp: add the warps' results in order
            if (rn >= a.R) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#pragma unroll
            for (int i = 0; i < 4; ++i) part[pb][warp][lane][i] = y[i];
            __syncthreads();
            if (warp == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = part[pb][0][lane][i];
#pragma unroll
                    for (int w2 = 1; w2 < kBWarps; ++w2) v = __fadd_rn(v, part[pb][w2][lane][i]);
                    const int m = i < 2 ? m0 : m1, n = 2 * t + (i & 1);
                    if (m >= a.M || n >= a.N) continue;
                    const long long o = (long long)n * a.M + m;
                    if (a.out == TL_OUT_F32) static_cast<float *>(a.Y)[o] = v;
                    else static_cast<__nv_bfloat16 *>(a.Y)[o] = __float2bfloat16_rn(v);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) y[i] = 0.f;
            pb ^= 1;
        }
#pragma unroll
        for (int u = 0; u < kBU; ++u) w[u] = wn[u];
        r = rn;
        grp = gn;
    }
}

bool aligned(const void *p, size_t al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; }

}  // namespace

namespace tl_internal {
tl_status blockscale_init_device() {
    return cudaFuncSetAttribute(tl_blockscale_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kBMaxStage) == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}
}  // namespace tl_internal

extern "C" {

tl_status tl_linear_blockscale(const uint32_t *packed, const float *bscale, int M, int K,
                               const void *X, int N, void *Y, int out_dtype, unsigned flags,
                               void *stream) {
    if (!packed || !bscale || !X || !Y) return TL_ERR_NULL;
    if (M < 1 || K < 1 || M > TL_MAX_M || K > TL_MAX_K || N < 1) return TL_ERR_SHAPE;
    if (out_dtype != TL_OUT_F32 && out_dtype != TL_OUT_BF16) return TL_ERR_MODE;
    if (!aligned(packed, 16) || !aligned(bscale, 4) || !aligned(X, 2) ||
        !aligned(Y, out_dtype == TL_OUT_BF16 ? 2 : 4))
        return TL_ERR_ALIGN;
    int sms = 0;
    const tl_status st = tl_internal::device_sms(&sms);
    if (st != TL_OK) return st;
    const int R = (M + 15) / 16;
    const int KB = (K + 127) / 128;
    const int xstride = KB * 128 + 8;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.blockDim = dim3(kBWarps * 32);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & TL_FLAG_PDL) ? 1 : 0;
    const size_t esz = out_dtype == TL_OUT_BF16 ? 2 : 4;
    for (int n0 = 0; n0 < N; n0 += 8) {
        BsArgs a;
        std::memset(&a, 0, sizeof a);
        a.packed = reinterpret_cast<const uint4 *>(packed);
        a.bscale = bscale;
        a.X = static_cast<const uint16_t *>(X) + (size_t)n0 * K;
        a.Y = static_cast<char *>(Y) + (size_t)n0 * M * esz;
        a.M = M; a.K = K; a.KB = KB; a.N = N - n0 < 8 ? N - n0 : 8; a.R = R;
        a.out = out_dtype;
        a.x4 = aligned(a.X, 4) && (K % 2) == 0 ? 1 : 0;
        a.xstride = xstride;
        const size_t stage = (size_t)a.N * xstride * 2;
        const bool staged = aligned(a.X, 16) && (K % 8) == 0 && stage <= (size_t)kBMaxStage;
        const void *fn = staged ? (const void *)tl_blockscale_kernel<true>
                                : (const void *)tl_blockscale_kernel<false>;
        cfg.dynamicSmemBytes = staged ? stage : 0;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBWarps * 32,
                                                          cfg.dynamicSmemBytes) != cudaSuccess ||
            per_sm < 1)
            return TL_ERR_CUDA;
        cfg.gridDim = dim3((unsigned)(R < sms * per_sm ? R : sms * per_sm));
        const cudaError_t e = staged ? cudaLaunchKernelEx(&cfg, tl_blockscale_kernel<true>, a)
                                     : cudaLaunchKernelEx(&cfg, tl_blockscale_kernel<false>, a);
        if (e != cudaSuccess) return TL_ERR_CUDA;
    }
    return TL_OK;
}

}  // extern "C"
