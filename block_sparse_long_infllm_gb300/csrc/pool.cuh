// pool.cuh -- exact mean of c bf16 rows rounded once to bf16 (semantic-kernel pooling, "MiniCPM4:
// 如何在手机电脑上高效运行大语言模型", section 1.1), in integer arithmetic: per column the lanes
// agree on the largest bf16 exponent, every value becomes an integer multiple of 2^-40 of that
// magnitude (exact for every value within 2^40 of the largest -- the condition under which an
// fp64 sum of bf16 values is exact as well), the integers are added, and the quotient by c, with
// its remainder as a sticky bit, is rounded once, nearest with ties to even.  (This GPU's fp64
// rate is a few operations per clock per SM, so no fp64 is used.)
#pragma once

#include "common.cuh"

namespace infllmv2 {

constexpr int kMeanLanes = 16;                    // lanes per (kernel, 8-element slice)
constexpr int kMeanRows = 128 / kMeanLanes;       // rows per lane: kernel_size <= block_size <= 128

// bf16 bits of (A / c) * 2^E0 (negated when neg), rounded once, nearest with ties to even; A < 2^62.
__device__ __forceinline__ uint32_t bf16_of_ratio(unsigned long long A, int c, int E0, bool neg) {
    if (A == 0ull) return 0u;  // +0, as an fp64 sum that starts from +0 gives
    const uint32_t sign = neg ? 0x8000u : 0u;
    const int t = __clzll(static_cast<long long>(A)) - 2;   // N = A << t in [2^61, 2^62)
    const unsigned long long N = A << t;
    unsigned long long Q;
    bool sticky;
    if ((c & (c - 1)) == 0) {  // a power of two (the pages' 32): a shift
        const int lc = __ffs(c) - 1;
        Q = N >> lc;
        sticky = (N & static_cast<unsigned long long>(c - 1)) != 0ull;
    } else {
        Q = N / static_cast<unsigned long long>(c);
        sticky = N - Q * static_cast<unsigned long long>(c) != 0ull;
    }
    const int nb = 64 - __clzll(static_cast<long long>(Q));  // >= 55: Q >= 2^61 / 128
    int X = nb - 1 + E0 - t;                                // exponent of the leading bit
    const int sh = X >= -126 ? nb - 8 : nb - 8 + (-126 - X); // bits below the kept ones (subnormal: fewer kept)
    if (sh >= 63) return sign;                              // below half the smallest subnormal
    unsigned long long top = Q >> sh;
    const unsigned long long rem = Q & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (sticky || (top & 1ull)))) ++top;
    if (X < -126) return sign | static_cast<uint32_t>(top);  // subnormal (128: the smallest normal)
    if (top == 256ull) {
        top = 128ull;
        ++X;
    }
    const int ef = X + 127;
    if (ef >= 255) return sign | 0x7F80u;
    return sign | (static_cast<uint32_t>(ef) << 7) | static_cast<uint32_t>(top & 127ull);
}

// Exact mean of the c rows of one 8-element slice; lane ln (of the 16 aligned lanes sharing the
// slice) loads rows ln, ln + 16, ...; row `sub_row` is taken from `sub_val` instead of memory.
// Every lane of the group returns the 8 bf16 results, packed.
__device__ __forceinline__ uint4 exact_mean_slice(const uint4* src, size_t row_stride, int c, int ln, int sub_row,
                                                  uint4 sub_val) {
    uint32_t w[kMeanRows][4];
    const int n_u = (c + kMeanLanes - 1) / kMeanLanes;  // row rounds any lane of the group has
#pragma unroll
    for (int u = 0; u < kMeanRows; ++u) {
        const int i = ln + kMeanLanes * u;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (u < n_u && i < c) x = i == sub_row ? sub_val : ldg_v4(src + static_cast<size_t>(i) * row_stride);
        w[u][0] = x.x;
        w[u][1] = x.y;
        w[u][2] = x.z;
        w[u][3] = x.w;
    }
    int emax[8];  // largest biased exponent per column (1 for zeros and subnormals)
#pragma unroll
    for (int e = 0; e < 8; ++e) emax[e] = 1;
#pragma unroll
    for (int u = 0; u < kMeanRows; ++u) {
        if (u >= n_u) break;
#pragma unroll
        for (int e = 0; e < 8; ++e) emax[e] = max(emax[e], static_cast<int>((w[u][e >> 1] >> (16 * (e & 1) + 7)) & 0xFFu));
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int off = 1; off < kMeanLanes; off <<= 1) emax[e] = max(emax[e], __shfl_xor_sync(0xffffffffu, emax[e], off));
    long long S[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) S[e] = 0;
#pragma unroll
    for (int u = 0; u < kMeanRows; ++u) {
        if (u >= n_u) break;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t h = (w[u][e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
            const int ef = static_cast<int>((h >> 7) & 0xFFu);
            const long long mant = ef != 0 ? static_cast<long long>(128u | (h & 127u)) : static_cast<long long>(h & 127u);
            const int sh = max(ef, 1) - (emax[e] - 40);  // value = mant * 2^(max(ef,1) - 134)
            const long long v = sh >= 0 ? (mant << sh) : (mant >> min(-sh, 62));
            S[e] += (h & 0x8000u) ? -v : v;
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int off = 1; off < kMeanLanes; off <<= 1) S[e] += __shfl_xor_sync(0xffffffffu, S[e], off);
    // lane ln rounds column ln % 8 of the group's sums; the 8 results are then gathered
    const int em = ln & 7;
    long long Sm = S[0];
    int xm = emax[0];
#pragma unroll
    for (int e = 1; e < 8; ++e)
        if (e == em) {
            Sm = S[e];
            xm = emax[e];
        }
    const uint32_t bits =
        bf16_of_ratio(static_cast<unsigned long long>(Sm < 0 ? -Sm : Sm), c, xm - 40 - 134, Sm < 0);
    const int g0 = (threadIdx.x & 31) & ~(kMeanLanes - 1);  // first lane of this group in the warp
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        out[e] = __shfl_sync(0xffffffffu, bits, g0 + 2 * e) | (__shfl_sync(0xffffffffu, bits, g0 + 2 * e + 1) << 16);
    return make_uint4(out[0], out[1], out[2], out[3]);
}

}  // namespace infllmv2
