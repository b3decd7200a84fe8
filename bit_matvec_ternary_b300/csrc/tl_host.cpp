// tl_host.cpp -- host side of the C ABI: the TL2P v1 packer, the validator,
// status strings.  No CUDA here.
//
// Packing is the offline step next to the per-row metadata the model page
// describes ("Neutrino-1 8B", "Architecture": per-row "scales, and row
// sums"); the bit layout is the library's own TL2P v1 (see include/tl.h).
// The packer walks the packed image word by word and gathers each word's
// sixteen codes, so every word is written exactly once.

#include "tl.h"

#include <algorithm>
#include <atomic>
#include <cstring>
#include <thread>
#include <vector>

namespace {

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// 2-bit code of one weight: bit 1 = sign, bit 0 = non-zero.
inline uint32_t code_of(int8_t w) { return w == 0 ? 0u : (w > 0 ? 1u : 3u); }

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

// Builds the 128 words of tile (r, b).
void pack_tile(const int8_t *W, const Shape &sh, int64_t r, int64_t b, uint32_t *out) {
    for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3;
        for (int j = 0; j < 4; ++j) {
            uint32_t word = 0;
            for (int q = 0; q < 8; ++q) {
                const int step = 2 * j + q / 4;      // 16-column step inside the tile
                const int f = q & 3;                 // mma A-fragment register
                const int hi_cols = f >> 1, hi_row = f & 1;
                const int64_t row = r * 16 + g + 8 * hi_row;
                const int64_t col = b * 128 + 16 * step + 8 * hi_cols + 2 * t;
                uint32_t lo = 0, hi = 0;
                if (row < sh.M) {
                    if (col < sh.K) lo = code_of(W[row * sh.K + col]);
                    if (col + 1 < sh.K) hi = code_of(W[row * sh.K + col + 1]);
                }
                word |= lo << (14 - 2 * q);
                word |= hi << (30 - 2 * q);
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
                    for (int q = 0; q < 8; ++q) {
                        const int step = 2 * j + q / 4, f = q & 3;
                        const int64_t row = r * 16 + g + 8 * (f & 1);
                        const int64_t col = b * 128 + 16 * step + 8 * (f >> 1) + 2 * t;
                        for (int e = 0; e < 2; ++e) {
                            const uint32_t c = (word >> ((e ? 30 : 14) - 2 * q)) & 3u;
                            if (c == 2u) ++bad;                       // sign without non-zero
                            else if (c != 0u && (row >= M || col + e >= K)) ++bad;  // padding
                        }
                    }
                }
            }
        }
    if (bad_codes) *bad_codes = bad;
    return bad ? TL_ERR_BAD_VALUE : TL_OK;
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
