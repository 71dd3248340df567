// kernel_pool.cu -- semantic-kernel pooling ("MiniCPM4: 如何在手机电脑上高效运行大语言模型",
// section 1.1 "InfLLM v2": overlapping semantic kernels of 32 tokens with stride 16).
//
// kernel[j] = bf16_rne(mean of K rows [j*s, j*s + c)), the exact mean rounded once (pool.cuh).
// Sixteen lanes own one kernel and one 8-element slice of the head dimension; each holds at most
// 8 of the c <= 128 rows (16-byte loads, all in flight at once).
#include "internal.h"
#include "pool.cuh"

namespace infllmv2 {

template <int D>
__global__ void __launch_bounds__(256) kernel_pool_kernel(const __nv_bfloat16* __restrict__ k,
                                                          __nv_bfloat16* __restrict__ kern,
                                                          int L_max, int M_max, int j_first,
                                                          int n_new, int c, int s) {
    constexpr int kChunks = D / 8;
    const int bg = blockIdx.y;
    const int gid = blockIdx.x * blockDim.x + threadIdx.x;
    const int ln = gid % kMeanLanes;
    const int item = gid / kMeanLanes;
    const bool live = item < n_new * kChunks;
    const int j = j_first + (live ? item / kChunks : 0);
    const int ch = item % kChunks;
    const uint4* src =
        reinterpret_cast<const uint4*>(k + (static_cast<size_t>(bg) * L_max + static_cast<size_t>(j) * s) * D) + ch;
    const uint4 r = exact_mean_slice(src, kChunks, live ? c : 0, ln, -1, make_uint4(0u, 0u, 0u, 0u));
    if (!live || ln != 0) return;
    reinterpret_cast<uint4*>(kern + (static_cast<size_t>(bg) * M_max + j) * D)[ch] = r;
}

// Kernels completed by each sequence's chunk when many sequences with different chunk lengths are
// prefilled at once (SeqMap): for row (b, g), every kernel whose last token lies in the chunk, the
// last len(b) tokens of its cache.  As kernel_pool_kernel, one 16-lane group per (kernel, slice).
template <int D>
__global__ void __launch_bounds__(256) kernel_pool_seq_kernel(const __nv_bfloat16* __restrict__ k,
                                                              __nv_bfloat16* __restrict__ kern,
                                                              const int* __restrict__ kv_len, SeqMap sm, int Hkv,
                                                              int L_max, int M_max, int c, int s,
                                                              int* __restrict__ err) {
    constexpr int kChunks = D / 8;
    const int bg = blockIdx.y, b = bg / Hkv;
    const int gid = blockIdx.x * blockDim.x + threadIdx.x;
    const int ln = gid % kMeanLanes, item = gid / kMeanLanes, ch = item % kChunks;
    const int L = kv_len[b], n_tok = sm.len(b);
    int j_first = 0, n_new = 0;
    if (n_tok < 0 || n_tok > sm.Tq || L < n_tok || L > L_max) {
        if (gid == 0) raise_error(err, kDevErrIndex);
    } else if (n_tok > 0) {
        const int num = L - n_tok - c + 1;  // kernels ending at or after the chunk's first token
        j_first = num <= 0 ? 0 : (num + s - 1) / s;
        const int j_last = L >= c ? (L - c) / s : -1;
        n_new = j_last - j_first + 1;
        if (j_last >= M_max) {
            if (gid == 0) raise_error(err, kDevErrIndex);
            n_new = 0;
        }
    }
    const bool live = item < n_new * kChunks;
    const int j = j_first + (live ? item / kChunks : 0);
    const uint4* src =
        reinterpret_cast<const uint4*>(k + (static_cast<size_t>(bg) * L_max + static_cast<size_t>(j) * s) * D) + ch;
    const uint4 r = exact_mean_slice(src, kChunks, live ? c : 0, ln, -1, make_uint4(0u, 0u, 0u, 0u));
    if (live && ln == 0) reinterpret_cast<uint4*>(kern + (static_cast<size_t>(bg) * M_max + j) * D)[ch] = r;
}

cudaError_t launch_kernel_pool_seq(const void* k_cache, void* kernel_cache, const int* kv_len, const SeqMap& sm,
                                   int B, int Hkv, int L_max, int M_max, int d, int c, int s, int* err,
                                   cudaStream_t stream) {
    const int n_max = sm.Tq / s + 2;  // kernels a chunk of at most Tq tokens can complete
    const int per_bg = kMeanLanes * n_max * (d / 8);
    dim3 grid((per_bg + 255) / 256, B * Hkv);
    const auto* kp = static_cast<const __nv_bfloat16*>(k_cache);
    auto* op = static_cast<__nv_bfloat16*>(kernel_cache);
    if (d == 128)
        kernel_pool_seq_kernel<128><<<grid, 256, 0, stream>>>(kp, op, kv_len, sm, Hkv, L_max, M_max, c, s, err);
    else
        kernel_pool_seq_kernel<64><<<grid, 256, 0, stream>>>(kp, op, kv_len, sm, Hkv, L_max, M_max, c, s, err);
    return cudaGetLastError();
}

// Decode-step append: K and V of each (sequence, KV head)'s new token into row kv_len - 1 of the
// caches ("CPM.cu：端侧大模型推理的 CUDA 加速引擎", section 4: static caches written in place), and,
// when that token completes semantic kernel j = (kv_len - c) / s, the kernel exactly as
// kernel_pool_kernel computes it, the new row read from the input rather than from the cache row
// this CTA writes.  One CTA of 2*D threads per row: 16 lanes per 8-element slice.
template <int D>
__global__ void __launch_bounds__(2 * D) append_kernel(const __nv_bfloat16* __restrict__ k_new,
                                                       const __nv_bfloat16* __restrict__ v_new,
                                                       __nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ v,
                                                       __nv_bfloat16* __restrict__ kern,
                                                       const int* __restrict__ kv_len, int Hkv, int L_max,
                                                       int M_max, int c, int s, int* __restrict__ err) {
    constexpr int kChunks = D / 8;
    const int bg = blockIdx.x;
    const int tid = threadIdx.x, ch = tid / kMeanLanes, ln = tid % kMeanLanes;
    const int L = kv_len[bg / Hkv];
    if (L < 1 || L > L_max) {
        if (tid == 0) raise_error(err, kDevErrIndex);
        return;
    }
    const int p = L - 1;
    const uint4 kn = ldg_v4(reinterpret_cast<const uint4*>(k_new + static_cast<size_t>(bg) * D) + ch);
    if (ln == 0) {
        const uint4 vn = ldg_v4(reinterpret_cast<const uint4*>(v_new + static_cast<size_t>(bg) * D) + ch);
        const size_t row = (static_cast<size_t>(bg) * L_max + p) * D;
        reinterpret_cast<uint4*>(k + row)[ch] = kn;
        reinterpret_cast<uint4*>(v + row)[ch] = vn;
    }
    if (L < c || (L - c) % s != 0) return;  // no kernel ends at the new token
    const int j = (L - c) / s;
    if (j >= M_max) {
        if (tid == 0) raise_error(err, kDevErrIndex);
        return;
    }
    const int r0 = j * s;
    const uint4* src = reinterpret_cast<const uint4*>(k + (static_cast<size_t>(bg) * L_max + r0) * D) + ch;
    const uint4 r = exact_mean_slice(src, kChunks, c, ln, p - r0, kn);
    if (ln == 0) reinterpret_cast<uint4*>(kern + (static_cast<size_t>(bg) * M_max + j) * D)[ch] = r;
}

cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, void* kernel_cache,
                          const int* kv_len, int B, int Hkv, int L_max, int M_max, int d, int c, int s, int* err,
                          cudaStream_t stream) {
    const auto* kn = static_cast<const __nv_bfloat16*>(k_new);
    const auto* vn = static_cast<const __nv_bfloat16*>(v_new);
    auto* kc = static_cast<__nv_bfloat16*>(k_cache);
    auto* vc = static_cast<__nv_bfloat16*>(v_cache);
    auto* kp = static_cast<__nv_bfloat16*>(kernel_cache);
    if (d == 128)
        append_kernel<128><<<B * Hkv, 256, 0, stream>>>(kn, vn, kc, vc, kp, kv_len, Hkv, L_max, M_max, c, s, err);
    else
        append_kernel<64><<<B * Hkv, 128, 0, stream>>>(kn, vn, kc, vc, kp, kv_len, Hkv, L_max, M_max, c, s, err);
    return cudaGetLastError();
}

cudaError_t launch_kernel_pool(const void* k_cache, void* kernel_cache, int B, int Hkv, int L_max,
                               int M_max, int d, int j_first, int n_new, int c, int s,
                               cudaStream_t stream) {
    if (n_new <= 0) return cudaSuccess;
    const int threads = 256;
    const int per_bg = kMeanLanes * n_new * (d / 8);
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
