// tl_prefill.cu -- the prefill-sized dense contraction (N >= 256 tokens) on
// the sm_103a tensor cores (tcgen05.mma, accumulator in TMEM).
//
// Same definition as the decode path, y[n,m] = scale[m] * sum_k w[m,k] x[n,k]
// (blog "Neutrino-1: quantization is a training decision", "What's actually
// ternary"), with the weights still packed at rest and decoded on chip
// (model page "Neutrino-1 8B", "Overview"): the packed TL2P tiles are loaded
// into registers, expanded to bf16 +-2.0 / 0 and written into shared memory
// in the 128-byte-swizzled K-major layout the tensor core reads, so no
// bf16 copy of a weight ever reaches global memory.
//
// The work is a list of 128-row x BN-token tiles of Y (of K splits, where a
// group's tiles alone do not cover the SMs), BN = 256 or 128 as the host's
// planner finds faster for the shapes.  The launch is persistent: one CTA per
// SM walks items blockIdx.x, blockIdx.x + gridDim.x, ...:
//   warp 0       TMA producer: activation tiles X[BN tokens][64 k] (bf16)
//   warp 1       TMEM owner and MMA issuer (one elected lane)
//   warps 2..9   weight decoders (one 16-row tile of the item's eight each,
//                two warps per SM sub-partition)
//   warps 10..17 epilogue (TMEM -> registers -> scale -> shared -> TMA store;
//                the two warps of a TMEM lane quarter take half of the tokens)
// A STAGES-deep ring of (A, B) shared-memory stages guarded by mbarriers runs
// on across items, and the accumulator alternates between two TMEM buffers,
// so the epilogue of one item overlaps the MMAs of the next.
// Every wait is bounded: after ~2^31 SM cycles the CTA records
// TL_DEVERR_TIMEOUT in the workspace status word, stops issuing work, waits
// (again bounded) for its own copies in flight, frees TMEM and exits.
//
// Mode B (int8 activations) feeds q as bf16, which is exact, so the fp32
// accumulator holds the exact integer 2 * sum_k w*q (|.| < 2^24).

#include "tl.h"
#include "tl_internal.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

namespace tlp {

constexpr int BM = 128;               // weight rows per CTA (TMEM lanes)
constexpr int BK = 64;                // k per stage (one 128-byte swizzle row)
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int DEC_WARPS = 8;
constexpr int EPI_WARPS = 8;
constexpr int EPI0 = 2 + DEC_WARPS;                 // first epilogue warp
constexpr int THREADS = 32 * (EPI0 + EPI_WARPS);
constexpr int RPW = BM / 16 / DEC_WARPS;            // row tiles decoded per warp
static_assert(RPW * DEC_WARPS * 16 == BM && EPI_WARPS % 4 == 0 && EPI0 % 4 == 2, "warp roles");
constexpr int ACC_BUFS = 2;                         // TMEM accumulators (BN columns each)
constexpr int EST_BYTES = 32 * 32 * 4;              // one epilogue warp's staging of 32 x 32 outputs
// Per token-tile width BN (tokens per item, TMEM columns per accumulator):
// 256 -> four stages of 48 KB, 128 -> six stages of 32 KB; the same shared
// memory either way.
__host__ __device__ constexpr int stages_for(int bn) { return bn == 256 ? 4 : 6; }
__host__ __device__ constexpr int stage_bytes_for(int bn) { return A_BYTES + bn * BK * 2; }
__host__ __device__ constexpr int smem_for(int bn) {
    return stages_for(bn) * stage_bytes_for(bn) + EPI_WARPS * EST_BYTES + 1024 /*align*/ +
           256 /*barriers*/;
}
static_assert(smem_for(256) <= 232448 && smem_for(128) <= 232448, "shared memory per CTA");
static_assert((3 * stages_for(128) + 2 * ACC_BUFS + 2) * 8 <= 256, "barrier area");
constexpr long long WAIT_LIMIT = 1ll << 31;   // SM cycles

struct PrefillArgs {
    const char *packed[TL_MAX_GROUP];
    const float *scale[TL_MAX_GROUP];
    const int32_t *rowsum[TL_MAX_GROUP];
    void *Y[TL_MAX_GROUP];
    int M[TL_MAX_GROUP];
    int mt_off[TL_MAX_GROUP + 1];   // 128-row tiles, prefix over the group
    int G;
    int KB;                          // 128-column TL2P blocks
    int KBS;                         // blocks per K split
    int S;                           // K splits
    int MT, NTT;                     // 128-row tiles, 256-token tiles
    int N;
    int mode, out;
    const float *s;
    const int32_t *z;
    int *status;                     // workspace status word
    unsigned long long *cnt;         // [tiles] splits arrived (S > 1); zero between launches
    float *part;                     // [tiles][S][BN][BM] partial sums (S > 1)
    int ystore;                      // whole tiles leave by TMA stores (ymap below)
};

// Tensor maps of the group's outputs Y_g [N][M_g] (boxes of 32 rows x 32
// tokens) for the TMA-store epilogue.
struct YMaps {
    CUtensorMap m[TL_MAX_GROUP];
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; returns false (and records the timeout) when it gives up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *status) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try(bar, parity)) {
        if (clock64() - t0 > WAIT_LIMIT) {
            atomicExch(status, TL_DEVERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    // K-major operand, 128-byte swizzle: rows of 128 B, 8-row atoms of 1024 B.
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);        // start address
    d |= (uint64_t)(1024u >> 4) << 32;              // stride between 8-row atoms
    d |= (uint64_t)1 << 46;                          // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                          // SWIZZLE_128B
    return d;
}

// kind::f16, A = B = bf16, D = f32, both K-major, M = 128, N = bn.
__host__ __device__ constexpr uint32_t idesc_for(int bn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(bn >> 3) << 17) |
           ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accum));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Write the decoded half hh (columns 64hh .. 64hh+63, k-steps 4hh .. 4hh+3)
// of one 16-row TL2P v2 tile into the A stage as bf16 +-2.0 / 0.  Word j of
// lane (g, t) holds row g + 8(j&1), columns 16s + 8(j>>1) + 2t (+1) in the
// fields at bits 2s (16 + 2s); a field holds 1 - w, so moving it to bits
// 15..14 and flipping bit 14 gives 00 -> 0x4000 (+2), 01 -> 0, 10 -> 0xC000.
// For one k-step the four words are the mma A fragment of a 16 x 16 block,
// i.e. four 8 x 8 matrices (rows +8 for j odd, columns +8 for j >= 2), which
// one stmatrix.x4 writes: lane L gives the address of row L % 8 of matrix
// L / 8.  In the 128-byte swizzle the eight rows of a matrix sit in eight
// different 16-byte bank groups.
__device__ __forceinline__ void store_half(uint32_t a_stage, int rt, int lane, const uint4 &w,
                                           int hh) {
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    const int mi = lane >> 3, r = lane & 7;
    const int row = rt * 16 + r + 8 * (mi & 1);             // row & 7 == r
    const uint32_t row_addr = a_stage + (uint32_t)((row >> 3) * 1024 + r * 128);
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
        const int s = 4 * hh + s4;
        uint32_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = ((wd[j] << (14 - 2 * s)) & 0xC000C000u) ^ 0x40004000u;
        const int chunk = 2 * s4 + (mi >> 1);
        asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(
                         row_addr + (uint32_t)((chunk ^ r) << 4)),
                     "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                     : "memory");
    }
}

// One work item: a 128-row x BN-token tile of one K split.
struct Item {
    int mt_global, nt, split, gi, mt, kb_lo, NKB;
};
__device__ __forceinline__ Item item_of(const PrefillArgs &a, int it) {
    Item t;
    t.mt_global = it % a.MT;
    t.nt = (it / a.MT) % a.NTT;
    t.split = it / (a.MT * a.NTT);
    t.gi = 0;
    while (t.gi + 1 < a.G && a.mt_off[t.gi + 1] <= t.mt_global) ++t.gi;
    t.mt = t.mt_global - a.mt_off[t.gi];
    t.kb_lo = t.split * a.KBS;
    t.NKB = min(a.KB, t.kb_lo + a.KBS) - t.kb_lo;
    return t;
}

// Persistent: CTA c takes items c, c + gridDim.x, ...  Every role walks the
// same items in the same order; the stage ring and its barriers run on
// across items, and the accumulator alternates between two TMEM buffers,
// so the epilogue warps finish one item while the MMAs of the next run.
template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
tl_prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap xmap,
                  const __grid_constant__ YMaps ym) {
    constexpr int STAGES = stages_for(BN);
    constexpr int STAGE_BYTES = stage_bytes_for(BN);
    constexpr int B_BYTES = BN * BK * 2;
    constexpr int EPI_COLS = BN / (EPI_WARPS / 4);      // tokens per epilogue warp
    constexpr uint32_t IDESC = idesc_for(BN);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint8_t *est = smem + STAGES * STAGE_BYTES;                       // epilogue staging
    uint64_t *bars = reinterpret_cast<uint64_t *>(est + EPI_WARPS * EST_BYTES);
    // bars: full_a[S], full_b[S], empty[S], acc_full[2], acc_empty[2]; then the
    // TMEM address and the split epilogue's flag
    const uint32_t bar0 = smem_u32(bars);
    auto full_a = [&](int s) { return bar0 + 8u * s; };
    auto full_b = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto empty = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto acc_full = [&](int b) { return bar0 + 8u * (3 * STAGES + b); };
    auto acc_empty = [&](int b) { return bar0 + 8u * (3 * STAGES + ACC_BUFS + b); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * STAGES + 2 * ACC_BUFS);
    volatile int *last_flag = reinterpret_cast<volatile int *>(bars + 3 * STAGES + 2 * ACC_BUFS + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = a.MT * a.NTT * a.S;
    const int my_items = blockIdx.x < n_items ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_a(s), DEC_WARPS);
            mbar_init(full_b(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), EPI_WARPS);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"((uint32_t)(ACC_BUFS * BN)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ---------------- activation producer
        griddep_wait();
        if (lane == 0) {
            int gs = 0;                                   // stages issued so far
            for (int j = 0; j < my_items && ok; ++j) {
                const Item t = item_of(a, blockIdx.x + j * gridDim.x);
                for (int ks = 0; ks < 2 * t.NKB; ++ks, ++gs) {
                    const int s = gs % STAGES;
                    const uint32_t ph = (uint32_t)(gs / STAGES) & 1u;
                    if (!mbar_wait(empty(s), ph ^ 1u, a.status)) { ok = false; break; }
                    mbar_expect_tx(full_b(s), B_BYTES);
                    tma_load_2d(base + s * STAGE_BYTES + A_BYTES, &xmap, t.kb_lo * 128 + ks * BK,
                                t.nt * BN, full_b(s));
                }
            }
            // drain: every copy this lane issued must land before the CTA exits
            for (int g = (gs > STAGES ? gs - STAGES : 0); g < gs; ++g)
                mbar_wait(full_b(g % STAGES), (uint32_t)(g / STAGES) & 1u, a.status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            int gs = 0;
            int done = 0;                                 // items whose accumulator was committed
            for (int j = 0; j < my_items && ok; ++j) {
                const Item t = item_of(a, blockIdx.x + j * gridDim.x);
                const int b = j & 1;
                // the epilogue of item j - 2 has read this accumulator
                if (j >= ACC_BUFS && !mbar_wait(acc_empty(b), (uint32_t)((j >> 1) - 1) & 1u, a.status)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + (uint32_t)(b * BN);
                for (int ks = 0; ks < 2 * t.NKB; ++ks, ++gs) {
                    const int s = gs % STAGES;
                    const uint32_t ph = (uint32_t)(gs / STAGES) & 1u;
                    if (!mbar_wait(full_a(s), ph, a.status) || !mbar_wait(full_b(s), ph, a.status)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t a_addr = base + s * STAGE_BYTES;
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), IDESC,
                                (ks | kk) != 0);
                    mma_commit(empty(s));
                }
                if (!ok) break;
                mma_commit(acc_full(b));
                done = j + 1;
            }
            // every MMA issued has retired before TMEM is freed
            if (done > 0) mbar_wait(acc_full((done - 1) & 1), (uint32_t)((done - 1) >> 1) & 1u, a.status);
        }
    } else if (warp < EPI0) {
        // ---------------- weight decoders
        const int dw = warp - 2;            // row tiles RPW dw .. RPW dw + RPW - 1 of the item's 8
        int gs = 0;
        for (int j = 0; j < my_items && ok; ++j) {
            const Item t = item_of(a, blockIdx.x + j * gridDim.x);
            const int rt_base = t.mt * 8 + RPW * dw;
            const int rts = (a.M[t.gi] + 15) / 16;
            const char *pk = a.packed[t.gi];
            const int NKB = t.NKB;
            // The weights do not depend on the previous kernel: bring this
            // warp's row tiles' K range into L2 first (their tiles are
            // contiguous along K), so the loads below find them there.
            if (lane < RPW && rt_base + lane < rts && NKB > 0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                 pk + ((long long)(rt_base + lane) * a.KB + t.kb_lo) * 512),
                             "r"((uint32_t)NKB * 512u)
                             : "memory");
            // RPW TL2P tiles (one per row tile) per 128 columns; prefetch ring of 4
            constexpr int RING = 4;
            uint4 ring[RING][RPW];
#pragma unroll
            for (int i = 0; i < RING; ++i)
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    ring[i][r] = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);  // zero weights
                    if (i < NKB && rt_base + r < rts)
                        ring[i][r] = ldg_stream(pk + ((long long)(rt_base + r) * a.KB + t.kb_lo + i) * 512 + lane * 16);
                }
            for (int kb0 = 0; kb0 < NKB && ok; kb0 += RING) {
#pragma unroll
                for (int i = 0; i < RING; ++i) {
                    const int kb = kb0 + i;       // block index within this split
                    if (kb < NKB) {
                        uint4 cur[RPW];
#pragma unroll
                        for (int r = 0; r < RPW; ++r) cur[r] = ring[i][r];
                        const int nb = kb + RING;
#pragma unroll
                        for (int r = 0; r < RPW; ++r)
                            if (nb < NKB && rt_base + r < rts)
                                ring[i][r] = ldg_stream(pk + ((long long)(rt_base + r) * a.KB + t.kb_lo + nb) * 512 + lane * 16);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int g = gs + 2 * kb + h;
                            const int s = g % STAGES;
                            const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
                            // every lane waits; the warp continues only if all of them got through
                            ok = __all_sync(0xffffffffu, ok && mbar_wait(empty(s), ph ^ 1u, a.status));
                            if (ok) {
                                const uint32_t a_stage = base + (uint32_t)(s * STAGE_BYTES);
#pragma unroll
                                for (int r = 0; r < RPW; ++r) store_half(a_stage, RPW * dw + r, lane, cur[r], h);
                                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                                __syncwarp();
                                if (lane == 0) mbar_arrive(full_a(s));
                            }
                        }
                    }
                }
            }
            gs += 2 * NKB;
        }
    } else {
        // ---------------- epilogue: TMEM lanes 32*(warp%4) .. +31 are this warp's rows
        const int ew = warp - EPI0;
        const int q = warp & 3;
        const int c_lo = (ew / 4) * EPI_COLS, c_hi = c_lo + EPI_COLS;   // this warp's tokens
        const int row_local = 32 * q + lane;
        uint8_t *stg = est + ew * EST_BYTES;
        const uint32_t stg_s = smem_u32(stg);
        griddep_wait();                      // outputs may still be read by the previous kernel
        for (int j = 0; j < my_items; ++j) {
            const Item t = item_of(a, blockIdx.x + j * gridDim.x);
            const int b = j & 1;
            const int gi = t.gi, nt = t.nt;
            const bool got = __all_sync(0xffffffffu, ok && mbar_wait(acc_full(b), (uint32_t)(j >> 1) & 1u, a.status));
            ok = got;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t acc_t = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN);
            const int row = t.mt * BM + row_local;
            const int Mg = a.M[gi];
            const bool row_ok = row < Mg;
            const float sc = row_ok ? a.scale[gi][row] : 0.f;
            const int rsum = (row_ok && a.mode == TL_MODE_I8) ? a.rowsum[gi][row] : 0;
            // one finished (row, token) value from the sum of +-2 weights;
            // mode B's step and zero point of token n come from lane n % 32
            auto value = [&](float acc2, float sv, int zv) {
                const float half = acc2 * 0.5f;
                if (a.mode == TL_MODE_BF16) return __fmul_rn(half, sc);
                const int iacc = __float2int_rn(half);
                return __fmul_rn(__fmul_rn((float)(iacc - zv * rsum), sv), sc);
            };
            auto emit = [&](int n, float acc2, float sv, int zv) {
                if (a.mode != TL_MODE_BF16 && a.out == TL_OUT_I32_RAW) {
                    reinterpret_cast<int32_t *>(a.Y[gi])[(long long)n * Mg + row] = __float2int_rn(acc2 * 0.5f);
                    return;
                }
                const float y = value(acc2, sv, zv);
                if (a.out == TL_OUT_F32)
                    reinterpret_cast<float *>(a.Y[gi])[(long long)n * Mg + row] = y;
                else
                    reinterpret_cast<__nv_bfloat16 *>(a.Y[gi])[(long long)n * Mg + row] = __float2bfloat16_rn(y);
            };
            auto release_acc = [&]() {
                // the accumulator is read: the next item's MMAs may use it
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty(b));
            };
            if (!got) {
                release_acc();
            } else if (a.S == 1) {
#pragma unroll 1
                for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(acc_t + (uint32_t)c0, r);
                    if (c0 + 32 >= c_hi) release_acc();
                    const int nl = nt * BN + c0 + lane;
                    const float s_l = a.mode != TL_MODE_BF16 && nl < a.N ? a.s[nl] : 0.f;
                    const int z_l = a.mode != TL_MODE_BF16 && nl < a.N ? a.z[nl] : 0;
                    if (a.ystore) {
                        // 32 tokens x this warp's 32 rows through the warp's staging
                        // buffer and one TMA store (rows past M, tokens past N are
                        // outside the tensor and not written)
                        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                        __syncwarp();
                        const int esz = a.out == TL_OUT_BF16 ? 2 : 4;
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const float sv = __shfl_sync(0xffffffffu, s_l, jj);
                            const int zv = __shfl_sync(0xffffffffu, z_l, jj);
                            uint8_t *dst = stg + (jj * 32 + lane) * esz;
                            const float acc2 = __uint_as_float(r[jj]);
                            if (a.mode != TL_MODE_BF16 && a.out == TL_OUT_I32_RAW)
                                *reinterpret_cast<int32_t *>(dst) = __float2int_rn(acc2 * 0.5f);
                            else if (a.out == TL_OUT_F32)
                                *reinterpret_cast<float *>(dst) = value(acc2, sv, zv);
                            else
                                *reinterpret_cast<__nv_bfloat16 *>(dst) = __float2bfloat16_rn(value(acc2, sv, zv));
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) {
                            asm volatile(
                                "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                                    reinterpret_cast<uint64_t>(&ym.m[gi])),
                                "r"(t.mt * BM + 32 * q), "r"(nt * BN + c0), "r"(stg_s)
                                : "memory");
                            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                        }
                    } else {
                        // element stores (every lane takes part in the shuffles)
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const float sv = __shfl_sync(0xffffffffu, s_l, jj);
                            const int zv = __shfl_sync(0xffffffffu, z_l, jj);
                            const int n = nt * BN + c0 + jj;
                            if (row_ok && n < a.N) emit(n, __uint_as_float(r[jj]), sv, zv);
                        }
                    }
                }
            } else {
                // split K: this split's partial tile goes to the workspace; the
                // item that completes the tile adds the splits in split order
                // and finishes it.  All epilogue warps pass the named barriers
                // below whatever happened before, so none can be left waiting.
                const long long tile = (long long)t.mt_global * a.NTT + nt;
                float *mine = a.part + (tile * a.S + t.split) * BN * BM;
#pragma unroll 1
                for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(acc_t + (uint32_t)c0, r);
                    if (c0 + 32 >= c_hi) release_acc();
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        __stcg(mine + (long long)(c0 + jj) * BM + row_local, __uint_as_float(r[jj]));
                }
            }
            if (a.S > 1) {
                const long long tile = (long long)t.mt_global * a.NTT + nt;
                asm volatile("bar.sync 1, %0;" ::"n"(EPI_WARPS * 32) : "memory");
                if (ew == 0 && lane == 0) {
                    asm volatile("fence.acq_rel.gpu;" ::: "memory");
                    const unsigned long long before = atomicAdd(a.cnt + tile, 1ull);
                    *last_flag = before + 1 == (unsigned long long)a.S ? 1 : 0;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(EPI_WARPS * 32) : "memory");
                const int last = *last_flag;
                // (the flag is read by every warp before it can be written again)
                asm volatile("bar.sync 1, %0;" ::"n"(EPI_WARPS * 32) : "memory");
                if (last) {
                    asm volatile("fence.acq_rel.gpu;" ::: "memory");
                    const float *p0 = a.part + tile * a.S * BN * BM;
                    // 32 tokens at a time: each split's 32 loads are issued together
#pragma unroll 1
                    for (int c0 = c_lo; c0 < c_hi && nt * BN + c0 < a.N; c0 += 32) {
                        const int nl = nt * BN + c0 + lane;
                        const float s_l = a.mode != TL_MODE_BF16 && nl < a.N ? a.s[nl] : 0.f;
                        const int z_l = a.mode != TL_MODE_BF16 && nl < a.N ? a.z[nl] : 0;
                        float acc2[32];
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) acc2[jj] = 0.f;
                        if (row_ok) {
#pragma unroll 1
                            for (int sp = 0; sp < a.S; ++sp) {
                                const float *ps = p0 + ((long long)sp * BN + c0) * BM + row_local;
                                float v[32];
#pragma unroll
                                for (int jj = 0; jj < 32; ++jj) v[jj] = __ldcg(ps + (long long)jj * BM);
#pragma unroll
                                for (int jj = 0; jj < 32; ++jj) acc2[jj] = __fadd_rn(acc2[jj], v[jj]);
                            }
                        }
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const float sv = __shfl_sync(0xffffffffu, s_l, jj);
                            const int zv = __shfl_sync(0xffffffffu, z_l, jj);
                            const int n = nt * BN + c0 + jj;
                            if (row_ok && n < a.N) emit(n, acc2[jj], sv, zv);
                        }
                    }
                    if (ew == 0 && lane == 0) a.cnt[tile] = 0ull;
                }
            }
        }
        // the last TMA stores have left shared memory and reached global memory
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    griddep_launch();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)(ACC_BUFS * BN)));
    }
}

// int8 activations to bf16 (exact), the TMA operand of mode B.  It lets the prefill kernel that follows
// start at once (that kernel decodes weights before it waits), and waits
// itself for the kernel that wrote q.
__global__ void tl_i8_to_bf16_kernel(const int8_t *__restrict__ q, __nv_bfloat16 *__restrict__ out,
                                     long long n) {
    griddep_launch();
    griddep_wait();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long k = i; k < n; k += stride) out[k] = __float2bfloat16_rn((float)q[k]);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    // looked up once; a function-local static is initialised exactly once
    // even when several host threads get here together
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

}  // namespace tlp

// ------------------------------------------------------------------ host side
namespace tl_internal {

namespace {
// Time of one 128-column block of a 128-token item, in blocks of a 256-token
// item, and of each extra K split (its partial tile written, then read back
// by the item that completes the tile), in blocks of a 256-token item; both
// fitted to the 8B groups at 512 tokens on B300: a 256-token block took
// 0.76 us, a 128-token block 0.70 us (the tensor cores do half the work, the
// stage ring and the weight decode do not shrink), and a second split added
// 14.5 us to o, 16.8 us to down.
constexpr double kHalfTileBlock = 0.92;
constexpr double kSplitBlocks = 19.0;

// The plan of one launch: the token-tile width BN, the K splits S (each at
// least 4 blocks of 128 columns) and blocks per split KBS, chosen for the
// fewest block-times on the busiest SM -- rounds of items times blocks per
// split times the block time, plus the splits' cost.  Ties keep BN = 256 and
// fewer splits.
struct PrefillPlan {
    int BN, S, KBS, tiles;
};
PrefillPlan prefill_plan(const tl_weight *Ws, int G, int N, int K, int sms) {
    int mt = 0;
    for (int g = 0; g < G; ++g) mt += (Ws[g].M + tlp::BM - 1) / tlp::BM;
    const int KB = (K + 127) / 128;
    PrefillPlan best{256, 1, KB, 0};
    double best_cost = -1.0;
    for (int bn : {256, 128}) {
        const long long tiles = (long long)mt * ((N + bn - 1) / bn);
        const double blk = bn == 256 ? 1.0 : kHalfTileBlock;
        for (int S = 1; S == 1 || S <= KB / 4; ++S) {
            const int KBS = (KB + S - 1) / S;
            const int Se = (KB + KBS - 1) / KBS;            // no empty split
            if (Se != S) continue;
            const long long waves = (tiles * S + sms - 1) / sms;
            const double c = (double)waves * KBS * blk + kSplitBlocks * blk * (S - 1);
            if (best_cost < 0.0 || c < best_cost) {
                best = PrefillPlan{bn, S, KBS, (int)tiles};
                best_cost = c;
            }
        }
    }
    return best;
}

// Workspace of a prefill call.  At the front, kept zero between calls: the
// status word, then (if K is split) one arrival counter per tile, which the
// item completing a tile sets back to zero.  Its scratch at the back, ending
// at the workspace's end:
//   [bf16 copy of the int8 activations, mode B; the quantised activations as
//    bf16 and their steps and zero points, TL_MODE_I8_FUSED]
//   [fp32 partial tiles, if K is split]
// (offsets below are from the start of that scratch), so prefill and decode
// calls may share one workspace in any order.
struct PrefillLayout {
    size_t front, conv, qs, qz, part, back;
};
PrefillLayout prefill_layout(int N, int K, int mode, int tiles, int S, int BN) {
    using tl_internal::round256;
    PrefillLayout L;
    L.front = kStatusBytes + (S > 1 ? round256((size_t)tiles * 8) : 0);
    L.conv = 0;
    L.qs = L.conv + (mode != TL_MODE_BF16 ? round256((size_t)N * K * 2) : 0);
    L.qz = L.qs + (mode == TL_MODE_I8_FUSED ? round256((size_t)N * 4) : 0);
    L.part = L.qz + (mode == TL_MODE_I8_FUSED ? round256((size_t)N * 4) : 0);
    L.back = L.part + (S > 1 ? (size_t)tiles * S * BN * tlp::BM * 4 : 0);
    return L;
}
}  // namespace

size_t prefill_workspace_bytes(const tl_weight *Ws, int G, int N, int K, int mode, int sms) {
    const PrefillPlan pl = prefill_plan(Ws, G, N, K, sms);
    const PrefillLayout L = prefill_layout(N, K, mode, pl.tiles, pl.S, pl.BN);
    return workspace_need(L.front, L.back);
}

bool prefill_supported(int N, int K) { return N >= kPrefillMinN && (K % 8) == 0; }

tl_status prefill_init_device() {
    if (cudaFuncSetAttribute(tlp::tl_prefill_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tlp::smem_for(256)) != cudaSuccess ||
        cudaFuncSetAttribute(tlp::tl_prefill_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tlp::smem_for(128)) != cudaSuccess)
        return TL_ERR_CUDA;
    return tlp::encode_fn() ? TL_OK : TL_ERR_UNSUPPORTED;
}

tl_status launch_prefill(const tl_weight *Ws, int G, const void *X, const float *s,
                         const int32_t *z, void *const *Ys, int N, int mode, int out, void *ws,
                         size_t ws_bytes, unsigned flags, cudaStream_t stream) {
    const int K = Ws[0].K;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TL_ERR_CUDA;
    if (!ws || ws_bytes < prefill_workspace_bytes(Ws, G, N, K, mode, sms)) return TL_ERR_WORKSPACE;
    tlp::PrefillArgs a;
    std::memset(&a, 0, sizeof a);
    a.G = G;
    a.mt_off[0] = 0;
    for (int g = 0; g < G; ++g) {
        a.packed[g] = reinterpret_cast<const char *>(Ws[g].packed);
        a.scale[g] = Ws[g].scale;
        a.rowsum[g] = Ws[g].rowsum;
        a.Y[g] = Ys[g];
        a.M[g] = Ws[g].M;
        a.mt_off[g + 1] = a.mt_off[g] + (Ws[g].M + tlp::BM - 1) / tlp::BM;
    }
    a.KB = (K + 127) / 128;
    const PrefillPlan pl = prefill_plan(Ws, G, N, K, sms);
    const int BN = pl.BN, tiles = pl.tiles;
    a.S = pl.S;
    a.KBS = pl.KBS;
    a.N = N;
    a.mode = mode == TL_MODE_BF16 ? TL_MODE_BF16 : TL_MODE_I8;   // the kernel's arithmetic
    a.out = out;
    a.s = s;
    a.z = z;
    a.status = static_cast<int *>(ws);

    const PrefillLayout L = prefill_layout(N, K, mode, tiles, a.S, BN);
    char *wsc = static_cast<char *>(ws) + scratch_offset(ws_bytes, L.back);
    const void *xb = X;
    __nv_bfloat16 *conv = reinterpret_cast<__nv_bfloat16 *>(wsc + L.conv);
    const long long n = (long long)N * K;
    // the arrival counters sit in the front bytes, zero between calls
    a.cnt = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kStatusBytes);
    a.part = reinterpret_cast<float *>(wsc + L.part);
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    if (mode == TL_MODE_I8_FUSED) {
        // quantise X per token straight into the bf16 operand, with its steps
        // and zero points in the workspace
        float *qs = reinterpret_cast<float *>(wsc + L.qs);
        int32_t *qz = reinterpret_cast<int32_t *>(wsc + L.qz);
        const tl_status qst = launch_quant(X, N, K, conv, true, qs, qz,
                                           (flags & TL_FLAG_SYMMETRIC) ? 1 : 0, stream);
        if (qst != TL_OK) return qst;
        a.s = qs;
        a.z = qz;
        xb = conv;
    } else if (mode == TL_MODE_I8) {
        cudaLaunchConfig_t cc;
        std::memset(&cc, 0, sizeof cc);
        cc.gridDim = dim3(592);
        cc.blockDim = dim3(256);
        cc.stream = stream;
        cc.attrs = pdl;
        cc.numAttrs = (flags & TL_FLAG_PDL) ? 1 : 0;
        if (cudaLaunchKernelEx(&cc, tlp::tl_i8_to_bf16_kernel, static_cast<const int8_t *>(X), conv,
                               n) != cudaSuccess)
            return TL_ERR_CUDA;
        xb = conv;
    }
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)tlp::BK, (cuuint32_t)BN};
    const cuuint32_t estr[2] = {1, 1};
    auto fn = tlp::encode_fn();
    if (!fn) return TL_ERR_UNSUPPORTED;
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(xb), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return TL_ERR_ALIGN;

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    a.MT = a.mt_off[G];
    a.NTT = (N + BN - 1) / BN;
    // persistent: one CTA per SM (shared memory allows one), each taking
    // every gridDim-th item
    cfg.gridDim = dim3((unsigned)std::min(a.MT * a.NTT * a.S, sms));
    cfg.blockDim = dim3(tlp::THREADS);
    cfg.dynamicSmemBytes = tlp::smem_for(BN);
    cfg.stream = stream;
    // (mode B: the conversion or quantiser kernel above, PDL-aware, is the one
    // it follows)
    cfg.attrs = pdl;
    cfg.numAttrs = (flags & TL_FLAG_PDL) ? 1 : 0;
    // Outputs that TMA can write whole tiles of (16-byte aligned, rows of a
    // multiple of 16 bytes) leave by TMA stores; otherwise by element stores.
    tlp::YMaps ym;
    std::memset(&ym, 0, sizeof ym);
    a.ystore = a.S == 1 ? 1 : 0;
    const size_t esz = out == TL_OUT_BF16 ? 2 : 4;
    const CUtensorMapDataType ydt = out == TL_OUT_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : out == TL_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                        : CU_TENSOR_MAP_DATA_TYPE_INT32;
    for (int g = 0; g < G && a.ystore; ++g) {
        if (reinterpret_cast<uintptr_t>(Ys[g]) % 16 != 0 || ((size_t)Ws[g].M * esz) % 16 != 0) {
            a.ystore = 0;
            break;
        }
        const cuuint64_t ydims[2] = {(cuuint64_t)Ws[g].M, (cuuint64_t)N};
        const cuuint64_t ystr[1] = {(cuuint64_t)Ws[g].M * esz};
        const cuuint32_t ybox[2] = {32, 32};
        if (fn(&ym.m[g], ydt, 2, Ys[g], ydims, ystr, ybox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            a.ystore = 0;
    }
    if (cudaLaunchKernelEx(&cfg, BN == 256 ? tlp::tl_prefill_kernel<256> : tlp::tl_prefill_kernel<128>,
                           a, map, ym) != cudaSuccess)
        return TL_ERR_CUDA;
    return TL_OK;
}

}  // namespace tl_internal

extern "C" {

tl_status tl_prefill_plan(const tl_weight *Ws, int G, int N, int sms, int32_t *plan) {
    if (!Ws || !plan) return TL_ERR_NULL;
    if (G < 1 || G > TL_MAX_GROUP || N < 1 || sms < 1) return TL_ERR_SHAPE;
    for (int g = 0; g < G; ++g)
        if (Ws[g].M < 1 || Ws[g].K < 1 || Ws[g].M > TL_MAX_M || Ws[g].K > TL_MAX_K ||
            Ws[g].K != Ws[0].K)
            return TL_ERR_SHAPE;
    const tl_internal::PrefillPlan p = tl_internal::prefill_plan(Ws, G, N, Ws[0].K, sms);
    const long long items = (long long)p.tiles * p.S;
    const int32_t v[TL_PREFILL_PLAN_FIELDS] = {p.BN, p.S, p.KBS, p.tiles,
                                               (int32_t)(items < sms ? items : sms)};
    for (int i = 0; i < TL_PREFILL_PLAN_FIELDS; ++i) plan[i] = v[i];
    return TL_OK;
}

}  // extern "C"
