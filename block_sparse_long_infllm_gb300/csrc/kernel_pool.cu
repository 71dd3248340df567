// kernel_pool.cu -- semantic-kernel pooling ("MiniCPM4: 如何在手机电脑上高效运行大语言模型",
// section 1.1 "InfLLM v2": overlapping semantic kernels of 32 tokens with stride 16).
//
// kernel[j] = bf16_rne(mean of K rows [j*s, j*s + c)).  Four lanes own one kernel and one
// 8-element slice of the head dimension and read its c rows with 128-bit loads (a warp covers
// two kernels' slices of 64 bytes per row, coalesced into 32-byte sectors).  The sum is carried in
// fp64: the sum of up to 2^20 bf16 values whose magnitudes span less than 2^40 is exact in
// a 53-bit significand, so the result is the exact mean rounded once (the same value any
// summation order gives).  The work is negligible next to scoring (one read of each new
// token), so no tensor cores or staging are used.
#include "common.cuh"
#include "internal.h"

namespace infllmv2 {

// Round a double to bf16, nearest with ties to even, from the binary64 layout: keep the sign,
// re-bias the exponent (1023 -> 127) and round the 52-bit fraction to 7 bits.
__device__ __forceinline__ uint16_t f64_to_bf16_rne(double x) {
    unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
    const unsigned long long sign = u >> 63;
    unsigned long long mag = u & 0x7FFFFFFFFFFFFFFFull;
    if (mag == 0) return static_cast<uint16_t>(sign << 15);
    const int e_in = static_cast<int>(mag >> 52) - 1023;
    if (e_in < -126) {
        // bf16 subnormal range: the spacing is 2^-133, so round x * 2^133 to an integer.
        const double two_133 = __longlong_as_double(static_cast<long long>(1023 + 133) << 52);
        const double scaled = fabs(x) * two_133;
        const unsigned long long m = static_cast<unsigned long long>(__double2ll_rn(scaled));
        return static_cast<uint16_t>((sign << 15) | m);  // m == 128 carries into the exponent
    }
    const unsigned long long lsb = (mag >> 45) & 1ull;
    mag += 0xFFFFFFFFFFFull + lsb;  // 2^44 - 1 + lsb: round half to even at bit 45
    const int e = static_cast<int>(mag >> 52) - 1023 + 127;
    if (e >= 255) return static_cast<uint16_t>((sign << 15) | 0x7F80u);  // overflow -> inf
    const unsigned m7 = static_cast<unsigned>((mag >> 45) & 0x7Full);
    return static_cast<uint16_t>((sign << 15) | (static_cast<unsigned>(e) << 7) | m7);
}

// Four adjacent lanes share one (kernel, 8-element slice): lane q sums rows q, q+4, q+8, ... of
// the kernel's c rows with independent 128-bit loads, and the four exact fp64 partial sums are
// added with shuffles (exact, so the order does not matter).
template <int D>
__global__ void __launch_bounds__(256) kernel_pool_kernel(const __nv_bfloat16* __restrict__ k,
                                                          __nv_bfloat16* __restrict__ kern,
                                                          int L_max, int M_max, int j_first,
                                                          int n_new, int c, int s) {
    constexpr int kChunks = D / 8;
    const int bg = blockIdx.y;
    const int gid = blockIdx.x * blockDim.x + threadIdx.x;
    const int q4 = gid & 3;
    const int item = gid >> 2;
    const bool live = item < n_new * kChunks;
    const int j = j_first + (live ? item / kChunks : 0);
    const int ch = item % kChunks;
    const uint4* src =
        reinterpret_cast<const uint4*>(k + (static_cast<size_t>(bg) * L_max + static_cast<size_t>(j) * s) * D) + ch;
    double acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0;
    if (live) {
#pragma unroll 8
        for (int i = q4; i < c; i += 4) {
            const uint4 v = ldg_v4(src + static_cast<size_t>(i) * kChunks);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += static_cast<double>(bf16_lo(w[e]));
                acc[2 * e + 1] += static_cast<double>(bf16_hi(w[e]));
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 1);
        acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 2);
    }
    if (!live || q4 != 0) return;
    const double cd = static_cast<double>(c);
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t lo = f64_to_bf16_rne(acc[2 * e] / cd);
        const uint32_t hi = f64_to_bf16_rne(acc[2 * e + 1] / cd);
        out[e] = lo | (hi << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(kern + (static_cast<size_t>(bg) * M_max + j) * D) + ch;
    *dst = make_uint4(out[0], out[1], out[2], out[3]);
}

cudaError_t launch_kernel_pool(const void* k_cache, void* kernel_cache, int B, int Hkv, int L_max,
                               int M_max, int d, int j_first, int n_new, int c, int s,
                               cudaStream_t stream) {
    if (n_new <= 0) return cudaSuccess;
    const int threads = 256;
    const int per_bg = 4 * n_new * (d / 8);
    dim3 grid((per_bg + threads - 1) / threads, B * Hkv);
    const auto* kp = static_cast<const __nv_bfloat16*>(k_cache);
    auto* op = static_cast<__nv_bfloat16*>(kernel_cache);
    if (d == 128)
        kernel_pool_kernel<128><<<grid, threads, 0, stream>>>(kp, op, L_max, M_max, j_first, n_new, c, s);
    else
        kernel_pool_kernel<64><<<grid, threads, 0, stream>>>(kp, op, L_max, M_max, j_first, n_new, c, s);
    return cudaGetLastError();
}

}  // namespace infllmv2
