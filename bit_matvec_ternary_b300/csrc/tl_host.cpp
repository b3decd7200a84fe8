// tl_host.cpp -- host side of the C ABI: the TL2P v2 packer, the validator,
// status strings.  No CUDA here.
//
// Packing is the offline step next to the per-row metadata the model page
// describes ("Neutrino-1 8B", "Architecture": per-row "scales, and row
// sums"); the bit layout is the library's own TL2P v2 (see include/tl.h).
// The packer walks the packed image word by word and gathers each word's
// sixteen codes, so every word is written exactly once.

#include "tl.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// 2-bit field of one weight: 1 - w (00 = +1, 01 = 0, 10 = -1).
inline uint32_t code_of(int8_t w) { return (uint32_t)(1 - w); }
constexpr uint32_t kZeroCode = 1u;   // padding

struct Shape {
    int64_t M, K, Mp, Kp, RT, KB;
};

Shape shape_of(int64_t M, int64_t K) {
    Shape s;
    s.M = M; s.K = K;
    s.Mp = round_up(M, 16); s.Kp = round_up(K, 128);
    s.RT = s.Mp / 16; s.KB = s.Kp / 128;
    return s;
}

// Builds the 128 words of tile (r, b).  Word j of lane (g, t) holds row
// g + 8*(j & 1), columns 16s + 8*(j >> 1) + 2t (+1) at bits 2s (16 + 2s).
void pack_tile(const int8_t *W, const Shape &sh, int64_t r, int64_t b, uint32_t *out) {
    for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3;
        for (int j = 0; j < 4; ++j) {
            const int64_t row = r * 16 + g + 8 * (j & 1);
            uint32_t word = 0;
            for (int s = 0; s < 8; ++s) {
                const int64_t col = b * 128 + 16 * s + 8 * (j >> 1) + 2 * t;
                uint32_t lo = kZeroCode, hi = kZeroCode;
                if (row < sh.M) {
                    if (col < sh.K) lo = code_of(W[row * sh.K + col]);
                    if (col + 1 < sh.K) hi = code_of(W[row * sh.K + col + 1]);
                }
                word |= lo << (2 * s);
                word |= hi << (16 + 2 * s);
            }
            out[lane * 4 + j] = word;
        }
    }
}

void pack_rows(const int8_t *W, const Shape &sh, int64_t r0, int64_t r1, uint32_t *packed,
               int32_t *rowsum) {
    for (int64_t r = r0; r < r1; ++r) {
        for (int64_t b = 0; b < sh.KB; ++b)
            pack_tile(W, sh, r, b, packed + (r * sh.KB + b) * 128);
        for (int64_t m = r * 16; m < std::min<int64_t>(sh.M, r * 16 + 16); ++m) {
            int64_t acc = 0;
            const int8_t *row = W + m * sh.K;
            for (int64_t k = 0; k < sh.K; ++k) acc += row[k];
            rowsum[m] = (int32_t)acc;
        }
    }
}

template <class F>
void parallel_rows(int64_t n, int64_t work_per_item, F fn) {
    unsigned hw = std::thread::hardware_concurrency();
    int64_t threads = std::max<int64_t>(1, std::min<int64_t>(hw ? hw : 1, 64));
    if (n * work_per_item < (int64_t)1 << 22) threads = 1;
    threads = std::min(threads, n);
    if (threads <= 1) { fn(0, n); return; }
    std::vector<std::thread> pool;
    for (int64_t i = 0; i < threads; ++i)
        pool.emplace_back(fn, n * i / threads, n * (i + 1) / threads);
    for (auto &th : pool) th.join();
}

}  // namespace

extern "C" {

size_t tl_packed_bytes(int64_t M, int64_t K) {
    if (M < 1 || K < 1) return 0;
    return (size_t)(round_up(M, 16) * round_up(K, 128) / 4);
}

tl_status tl_pack(const int8_t *W, int64_t M, int64_t K, const float *scale_in,
                  uint32_t *packed, float *scale_out, int32_t *rowsum) {
    if (!W || !packed || !rowsum) return TL_ERR_NULL;
    if (M < 1 || K < 1 || M > TL_MAX_M || K > TL_MAX_K) return TL_ERR_SHAPE;
    if ((scale_in == nullptr) != (scale_out == nullptr)) return TL_ERR_NULL;
    const Shape sh = shape_of(M, K);
    std::atomic<int64_t> bad{0};
    parallel_rows(M, K, [&](int64_t m0, int64_t m1) {
        int64_t local = 0;
        for (int64_t i = m0 * K; i < m1 * K; ++i)
            if (W[i] < -1 || W[i] > 1) ++local;
        bad += local;
    });
    if (bad.load()) return TL_ERR_BAD_VALUE;
    parallel_rows(sh.RT, 16 * sh.Kp, [&](int64_t r0, int64_t r1) {
        pack_rows(W, sh, r0, r1, packed, rowsum);
    });
    if (scale_in && scale_out && scale_in != scale_out)
        std::memcpy(scale_out, scale_in, (size_t)M * sizeof(float));
    return TL_OK;
}

tl_status tl_validate_packed(const uint32_t *packed, int64_t M, int64_t K, int64_t *bad_codes) {
    if (!packed) return TL_ERR_NULL;
    if (M < 1 || K < 1 || M > TL_MAX_M || K > TL_MAX_K) return TL_ERR_SHAPE;
    const Shape sh = shape_of(M, K);
    int64_t bad = 0;
    for (int64_t r = 0; r < sh.RT; ++r)
        for (int64_t b = 0; b < sh.KB; ++b) {
            const uint32_t *tile = packed + (r * sh.KB + b) * 128;
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, t = lane & 3;
                for (int j = 0; j < 4; ++j) {
                    const uint32_t word = tile[lane * 4 + j];
                    const int64_t row = r * 16 + g + 8 * (j & 1);
                    for (int s = 0; s < 8; ++s) {
                        const int64_t col = b * 128 + 16 * s + 8 * (j >> 1) + 2 * t;
                        for (int e = 0; e < 2; ++e) {
                            const uint32_t c = (word >> (2 * s + 16 * e)) & 3u;
                            if (c == 3u) ++bad;                                   // invalid field
                            else if (c != kZeroCode && (row >= M || col + e >= K)) ++bad;  // padding
                        }
                    }
                }
            }
        }
    if (bad_codes) *bad_codes = bad;
    return bad ? TL_ERR_BAD_VALUE : TL_OK;
}

// Block-wise scales (blog "Neutrino-1: quantization is a training
// decision", "What's actually ternary"): each block of a row has its own
// scale, the block's mean absolute weight, and its codes are
// round(clamp(w / scale, -1, 1)).  The mean is taken in double over the
// block's real columns, in column order, and stored as fp32; the ratio uses
// that fp32 scale, in double, rounded half to even.
tl_status tl_ternarize_absmean(const float *W, int64_t M, int64_t K, int8_t *T, float *bscale) {
    if (!W || !T || !bscale) return TL_ERR_NULL;
    if (M < 1 || K < 1 || M > TL_MAX_M || K > TL_MAX_K) return TL_ERR_SHAPE;
    std::atomic<int64_t> bad{0};
    parallel_rows(M, K, [&](int64_t m0, int64_t m1) {
        int64_t local = 0;
        for (int64_t i = m0 * K; i < m1 * K; ++i)
            if (!std::isfinite(W[i])) ++local;
        bad += local;
    });
    if (bad.load()) return TL_ERR_BAD_VALUE;
    const int64_t KB = (K + TL_SCALE_BLOCK - 1) / TL_SCALE_BLOCK;
    parallel_rows(M, K, [&](int64_t m0, int64_t m1) {
        for (int64_t m = m0; m < m1; ++m) {
            const float *row = W + m * K;
            for (int64_t b = 0; b < KB; ++b) {
                const int64_t k0 = b * TL_SCALE_BLOCK, k1 = std::min(K, k0 + TL_SCALE_BLOCK);
                double acc = 0.0;
                for (int64_t k = k0; k < k1; ++k) acc += std::fabs((double)row[k]);
                const float sc = (float)(acc / (double)(k1 - k0));
                bscale[m * KB + b] = sc;
                for (int64_t k = k0; k < k1; ++k) {
                    const double q = sc > 0.0f ? (double)row[k] / (double)sc : 0.0;
                    const double c = q > 1.0 ? 1.0 : (q < -1.0 ? -1.0 : q);
                    T[m * K + k] = (int8_t)std::nearbyint(c);
                }
            }
        }
    });
    return TL_OK;
}

const char *tl_status_string(tl_status s) {
    switch (s) {
        case TL_OK: return "ok";
        case TL_ERR_NULL: return "a required pointer is NULL";
        case TL_ERR_SHAPE: return "shape out of range";
        case TL_ERR_ALIGN: return "pointer misaligned";
        case TL_ERR_BAD_VALUE: return "weight or code outside the ternary set";
        case TL_ERR_MODE: return "unknown or unsupported mode / output type";
        case TL_ERR_UNSUPPORTED: return "unsupported layout or device";
        case TL_ERR_CUDA: return "CUDA runtime error";
        case TL_ERR_TIMEOUT: return "bounded device wait timed out";
        case TL_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

int tl_version(void) { return 100; }

}  // extern "C"
