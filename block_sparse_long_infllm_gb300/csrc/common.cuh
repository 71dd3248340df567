// common.cuh -- device helpers shared by the InfLLM v2 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace infllmv2 {

// Method parameters as the kernels see them (mirrors infllmv2_params).
struct Params {
    int block_size;
    int kernel_size;
    int kernel_stride;
    int topk;
    int n_init;
    int n_local;
    int dense_len;
    float scale;  // softmax scale, already resolved (never 0)
};

// Bits of the device error word.
enum : int { kDevErrTimeout = 1, kDevErrIndex = 2 };

__device__ __forceinline__ void raise_error(int* err, int code) {
    if (err) atomicOr(err, code);
}

// Floor division for a possibly negative numerator and a positive divisor.
__host__ __device__ __forceinline__ int floor_div(int a, int b) {
    return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// Query layout of a prefill call ("CPM.cu：端侧大模型推理的 CUDA 加速引擎", section 4: chunked
// prefill, here for many sequences in one launch).  Fixed chunks (cu == nullptr): sequence b's Tq
// queries are token rows b*Tq .. b*Tq + Tq - 1.  Packed variable-length chunks: sequence b's queries
// are token rows cu[b] .. cu[b+1] - 1 of `total`.  q and o are [token row, head]; selection-shaped
// arrays (idx, counts, scores) are [B, Hkv, Tq] fixed or [Hkv, total] packed; lse is [B, Hq, Tq]
// fixed or [Hq, total] packed.  A sequence's queries are the last len(b) tokens of its cache.
struct SeqMap {
    const int* cu;  // [B + 1] device offsets, or nullptr
    int Tq;         // fixed chunk length, or the longest packed chunk
    int total;      // token rows: B*Tq, or cu[B]
    __device__ __forceinline__ int tok0(int b) const { return cu != nullptr ? cu[b] : b * Tq; }
    __device__ __forceinline__ int len(int b) const { return cu != nullptr ? cu[b + 1] - cu[b] : Tq; }
    __device__ __forceinline__ size_t sel(int b, int g, int Hkv, int t) const {
        return cu != nullptr ? static_cast<size_t>(g) * total + cu[b] + t
                             : (static_cast<size_t>(b) * Hkv + g) * Tq + t;
    }
    __device__ __forceinline__ size_t lse(int b, int h, int Hq, int t) const {
        return cu != nullptr ? static_cast<size_t>(h) * total + cu[b] + t
                             : (static_cast<size_t>(b) * Hq + h) * Tq + t;
    }
    // inverse of sel(): selection row r -> (b, g, t)
    __device__ __forceinline__ void row_of(long long r, int B, int Hkv, int* b, int* g, int* t) const {
        if (cu == nullptr) {
            *t = static_cast<int>(r % Tq);
            *g = static_cast<int>((r / Tq) % Hkv);
            *b = static_cast<int>(r / (static_cast<long long>(Tq) * Hkv));
            return;
        }
        *g = static_cast<int>(r / total);
        const int tok = static_cast<int>(r % total);
        int lo = 0, hi = B;  // the last b with cu[b] <= tok
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu[mid] <= tok) lo = mid; else hi = mid;
        }
        *b = lo;
        *t = tok - cu[lo];
    }
};

// Number of complete semantic kernels among the first L tokens.
__host__ __device__ __forceinline__ int kernels_in(int L, int c, int s) {
    return L < c ? 0 : (L - c) / s + 1;
}

// Kernels sharing at least one token with block blk: j*s < (blk+1)*bs and j*s + c > blk*bs.
__host__ __device__ __forceinline__ int first_kernel_of_block(int blk, int bs, int c, int s) {
    int j = floor_div(blk * bs - c, s) + 1;
    return j < 0 ? 0 : j;
}
__host__ __device__ __forceinline__ int last_kernel_of_block(int blk, int bs, int s) {
    return ((blk + 1) * bs - 1) / s;
}

// 128-bit read-only global load.
__device__ __forceinline__ uint4 ldg_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 128-bit streaming load: read once, do not keep in L1.
__device__ __forceinline__ uint4 ldg_v4_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate (legacy warp MMA).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x on the special-function unit (PTX ex2.approx; inputs of -inf give +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Select the 16-bit element `e` (0 = low) of word pair (w0, w1) as two halves of one word:
// result = { lo: element e of w0, hi: element e of w1 }.
__device__ __forceinline__ uint32_t pair_halves(uint32_t w0, uint32_t w1, int e) {
    return e == 0 ? __byte_perm(w0, w1, 0x5410) : __byte_perm(w0, w1, 0x7632);
}

// Programmatic dependent launch: a kernel launched with the programmatic-serialisation
// attribute may start before its predecessor on the stream has finished; pdl_wait() blocks
// until the predecessor grid has completed and its memory is visible (it returns at once for a
// normally launched kernel).  pdl_trigger() lets the successor start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kern` on `stream`; with `pdl` the launch may overlap the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Monotone map from fp32 to uint32 (larger float -> larger key); -0 is folded into +0
// so that equal scores always compare equal.
__device__ __forceinline__ uint32_t ordered_key(float s) {
    uint32_t u = __float_as_uint(s + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace infllmv2
