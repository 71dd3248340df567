// score_tc.cu -- block scores for a prefill chunk on the 5th-generation tensor cores
// ("MiniCPM4: 如何在手机电脑上高效运行大语言模型", section 1.1 "InfLLM v2": query-kernel relevance
// at kernel granularity, max over the kernels of a block and over a group's heads).
//
// The scoring is a GEMM per KV head: every (query token, head) row against every visible
// semantic kernel.  One CTA owns 16 query tokens x the 16 heads of one KV head (256 Q rows,
// the MMA's N) and walks the kernel cache in chunks of 128 kernels (the MMA's M), so each
// accumulator lane holds one kernel against all 256 rows: the max over a token's 16 heads and
// the visibility test (the kernel ends at or before the token's position) are thread-local.
// The per-(token, kernel) maxima go to shared memory, where the block max over the kernels a
// block overlaps is taken and written to S[b, g, t, block].  Chunks cover whole blocks (31
// blocks of 64 tokens or 15 of 128), so no block straddles two chunks.
//   * producer warp (warp 8, one lane): TMA of the Q tile once and of each chunk's kernel rows
//     into two shared stages; one tcgen05 MMA group per chunk into one of two TMEM buffers;
//   * epilogue warps (warps 0-7, two per TMEM lane quarter, one half of the 16 tokens each):
//     TMEM -> registers (all four loads of a thread in flight before one wait) -> maxima ->
//     shared -> S.
// Waits are bounded (device error word + abort flag), TMEM is freed before exit.
#include <algorithm>

#include "internal.h"
#include "umma.cuh"

namespace infllmv2 {

constexpr int kScTokens = 16;            // query tokens per CTA: N = 16 x 16 heads = 256
constexpr int kScN = kScTokens * 16;
constexpr int kScM = 128;                // kernels per chunk
constexpr int kScThreads = 288;  // 8 epilogue warps + the producer warp
constexpr int kScEpi = 256;      // epilogue threads
constexpr int kScSpan = 16;      // kernels a block may overlap on the division-free block-max pass

template <int D>
struct ScSmem {
    static constexpr int kQ = kScN * D * 2;       // Q tile (B operand)
    static constexpr int kK = kScM * D * 2;       // one chunk of kernel rows (A operand)
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQ;              // 2 stages
    static constexpr int kMaxOff = kQ + 2 * kK;   // [kScTokens][kScM] floats
    static constexpr int kBarOff = kMaxOff + kScTokens * kScM * 4;
    static constexpr int kBytes = kBarOff + 128 + 1024;
};

// AND of `v` over the 256 epilogue threads (named barrier 1; also synchronises them).
__device__ __forceinline__ bool epilogue_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n"
        " .reg .pred p, q;\n"
        " setp.ne.u32 q, %1, 0;\n"
        " bar.red.and.pred p, 1, 256, q;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v))
        : "memory");
    return r != 0;
}

template <int D>
__global__ void __launch_bounds__(kScThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kern,
                const int* __restrict__ kv_len, SeqMap sm, int tree, int Hq, int Hkv, int L_max, int M_max, int nblk_max,
                Params p,
                int blocks_per_chunk, float* __restrict__ S, int* __restrict__ err) {
    using SM = ScSmem<D>;
    constexpr int G = 16;
    constexpr uint32_t kIdesc = idesc_bf16_f32(kScM, kScN, 0, 0);
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    float* kmax = reinterpret_cast<float*>(base + SM::kMaxOff);  // [token][kernel row]
    uint64_t* bar_q = reinterpret_cast<uint64_t*>(base + SM::kBarOff);
    uint64_t* bar_k = bar_q + 1;     // [2] kernel chunk landed
    uint64_t* bar_acc = bar_q + 3;   // [2] MMA of a chunk done
    uint64_t* bar_free = bar_q + 5;  // [2] epilogue done with a TMEM buffer (256 arrivals)
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_q + 8);
    volatile int* s_abort = reinterpret_cast<volatile int*>(bar_q + 9);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bg = blockIdx.y;
    const int b = bg / Hkv, g = bg % Hkv;
    const int t0 = blockIdx.x * kScTokens;
    const int bs = p.block_size, c = p.kernel_size, s = p.kernel_stride;
    const int Lb = kv_len[b];
    const int Tq = sm.len(b), tok = sm.tok0(b);  // this sequence's chunk: token rows tok .. tok + Tq - 1
    // query t sits at Lb - Tq + t (a chunk) or, for tree drafts, all at the last cached position Lb - 1
    const int pos0 = tree ? Lb - 1 : Lb - Tq;  // position of query t is pos0 + (tree ? 0 : t)
    if (Tq < 0 || Tq > sm.Tq ||
        (Tq > 0 && (Lb < (tree ? 1 : Tq) || Lb > L_max || kernels_in(Lb, c, s) > M_max))) {
        if (tid == 0 && blockIdx.x == 0) raise_error(err, kDevErrIndex);
        return;
    }
    if (t0 >= Tq) return;  // packed chunks shorter than the longest
    if (Lb < p.dense_len) return;  // dense sequence: every block is selected, no scores needed
    const int n_tok = min(kScTokens, Tq - t0);
    const int pos_last = tree ? pos0 : pos0 + t0 + n_tok - 1;
    const int bt_max = pos_last / bs;
    // chunks split, split + n_split, ... of the blocks are this CTA's (blockIdx.z = split)
    const int split = blockIdx.z, n_split = gridDim.z;
    const int n_chunks_all = bt_max / blocks_per_chunk + 1;
    const int n_chunks = n_chunks_all > split ? (n_chunks_all - split + n_split - 1) / n_split : 0;
    if (n_chunks == 0) return;

    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_k[i], 1);
            mbar_init(&bar_acc[i], 1);
            mbar_init(&bar_free[i], kScEpi);
        }
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == 8) {
        // ======================= producer
        if (lane == 0) {
            const uint32_t sQ = smem_u32(base + SM::kQOff);
            int k_issued[2] = {0, 0}, mma_issued = 0;
            // local chunk k is chunk split + n_split * k of the tile
            auto chunk_row = [&](int k) { return first_kernel_of_block((split + n_split * k) * blocks_per_chunk, bs, c, s); };
            auto load = [&](int ch) {
                const int st = ch & 1;
                mbar_arrive_expect_tx(&bar_k[st], SM::kK);
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_2d(base + SM::kKOff + st * SM::kK + sub * (kScM * 128), &tm_kern, 64 * sub,
                                bg * M_max + chunk_row(ch), &bar_k[st]);
                ++k_issued[st];
            };
            auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
                if (*s_abort) return false;
                if (mbar_wait(bar, parity)) return true;
                raise_error(err, kDevErrTimeout);
                *s_abort = 1;
                return false;
            };
            // Q tile: 16 tokens x 16 heads, one 16-row box per token and 64-column half
            mbar_arrive_expect_tx(bar_q, SM::kQ);
            for (int tk = 0; tk < kScTokens; ++tk) {
                const int t = min(t0 + tk, Tq - 1);
                const int qrow = (tok + t) * Hq + g * G;
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_2d(base + SM::kQOff + sub * (kScN * 128) + tk * (G * 128), &tm_q, 64 * sub, qrow, bar_q);
            }
            load(0);
            if (n_chunks > 1) load(1);
            bool ok = wait(bar_q, 0);
            for (int ch = 0; ok && ch < n_chunks; ++ch) {
                const int st = ch & 1;
                if (!(ok = wait(&bar_k[st], (ch >> 1) & 1))) break;
                if (ch >= 2 && !(ok = wait(&bar_free[st], ((ch - 2) >> 1) & 1))) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(base + SM::kKOff + st * SM::kK);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ao = (kk / 4) * (kScM * 128) + (kk % 4) * 32;
                    const uint32_t bo = (kk / 4) * (kScN * 128) + (kk % 4) * 32;
                    mma_ss(tmem + st * kScN, sw128_desc(ka + ao, 16, 1024), sw128_desc(sQ + bo, 16, 1024), kIdesc,
                           kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar_acc[st]);
                ++mma_issued;
                if (ch + 2 < n_chunks) {  // the stage is free once this chunk's MMA is done
                    if (!(ok = wait(&bar_acc[st], (ch >> 1) & 1))) break;
                    load(ch + 2);
                }
            }
            const long long drain = kWaitBudgetCycles / 8;
            for (int st = 0; st < 2; ++st)
                if (k_issued[st] > 0) mbar_wait(&bar_k[st], (k_issued[st] - 1) & 1, drain);
            if (mma_issued > 0) mbar_wait(&bar_acc[(mma_issued - 1) & 1], ((mma_issued - 1) >> 1) & 1, drain);
        }
    } else {
        // ======================= epilogue: thread r = 32*(warp%4) + lane owns kernel row r of each
        // chunk; warps w and w+4 take tokens 0-7 and 8-15 (TMEM columns 128*(w/4) ...)
        const int r = 32 * (warp % 4) + lane;
        const int th = warp / 4;
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
        // the block-max pass without divisions: block size a power of two and a multiple of the
        // stride, a block overlapping at most kScSpan kernels, at most 32 blocks per chunk
        const int kr = bs / s, kcs = (c + s - 1) / s, bs_shift = __ffs(bs) - 1;
        const int nb_log = blocks_per_chunk <= 16 ? 4 : 5;
        const bool kr_fast = bs % s == 0 && (bs & (bs - 1)) == 0 && kr + kcs - 1 <= kScSpan && blocks_per_chunk <= 32;
        for (int ch = 0; ch < n_chunks; ++ch) {
            const int st = ch & 1;
            const bool waited = !*s_abort && mbar_wait(&bar_acc[st], (ch >> 1) & 1);
            // all eight epilogue warps leave together: they meet at the named barrier below
            if (!epilogue_all(waited)) {
                if (tid == 0 && !*s_abort) raise_error(err, kDevErrTimeout);
                *s_abort = 1;
                break;
            }
            tc_fence_after();
            const int b0 = (split + n_split * ch) * blocks_per_chunk;
            const int j0 = first_kernel_of_block(b0, bs, c, s);
            const int j = j0 + r;
            const int jend = j * s + c - 1;  // last token of kernel j
            {
                uint32_t ra[32], rb[32], rc[32], rd[32];
                const uint32_t ta = tmem + st * kScN + lane_off + th * 128;
                tmem_ld32(ta, ra);
                tmem_ld32(ta + 32, rb);
                tmem_ld32(ta + 64, rc);
                tmem_ld32(ta + 96, rd);
                tmem_ld_wait(ra);
                reg_fence(rb);
                reg_fence(rc);
                reg_fence(rd);
                auto head_max = [&](const uint32_t (&v)[32], int u) {
                    float m = __uint_as_float(v[16 * u]);
#pragma unroll
                    for (int h = 1; h < G; ++h) m = fmaxf(m, __uint_as_float(v[16 * u + h]));
                    return m;
                };
                float mx[8];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    mx[u] = head_max(ra, u);
                    mx[2 + u] = head_max(rb, u);
                    mx[4 + u] = head_max(rc, u);
                    mx[6 + u] = head_max(rd, u);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int tk = th * 8 + u;
                    const int pos = tree ? pos0 : pos0 + t0 + tk;
                    kmax[tk * kScM + r] = (tk < n_tok && jend <= pos) ? mx[u] : -INFINITY;
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_free[st]);  // this thread is done with the TMEM buffer
            asm volatile("bar.sync 1, 256;" ::: "memory");
            // block max over the kernels each block overlaps, for every token of the tile
            const int nb = min(blocks_per_chunk, bt_max + 1 - b0);
            if (kr_fast) {
                // block size a multiple of the stride (r kernels per block): block blk overlaps
                // kernels max(0, blk*r - ceil(c/s) + 1) .. (blk+1)*r - 1, at most kScSpan of them;
                // item e = (token e >> nb_log, block e & (2^nb_log - 1)), no divisions, the span's
                // loads all in flight before the maximum
                for (int e = tid; e < (kScTokens << nb_log); e += kScEpi) {
                const int tk = e >> nb_log, i = e & ((1 << nb_log) - 1);
                const int blk = b0 + i;
                const int pos = tree ? pos0 : pos0 + t0 + tk;
                if (tk < n_tok && i < nb && blk <= (pos >> bs_shift)) {
                    const int ja = max(0, blk * kr - kcs + 1) - j0;
                    const int jz = min((blk + 1) * kr - 1 - j0, kScM - 1);
                    float v[kScSpan];
#pragma unroll
                    for (int u = 0; u < kScSpan; ++u) v[u] = ja + u <= jz ? kmax[tk * kScM + ja + u] : -INFINITY;
#pragma unroll
                    for (int w2 = kScSpan / 2; w2 > 0; w2 >>= 1)
#pragma unroll
                        for (int u = 0; u < w2; ++u) v[u] = fmaxf(v[u], v[u + w2]);
                    S[sm.sel(b, g, Hkv, t0 + tk) * nblk_max + blk] = v[0];
                }
                }
            } else {
                for (int e = tid; e < n_tok * nb; e += kScEpi) {
                    const int tk = e / nb, blk = b0 + e % nb;
                    const int pos = tree ? pos0 : pos0 + t0 + tk;
                    if (blk > pos / bs) continue;
                    const int ja = first_kernel_of_block(blk, bs, c, s) - j0;
                    const int jz = min(last_kernel_of_block(blk, bs, s) - j0, kScM - 1);
                    float m = -INFINITY;
                    for (int jj = ja; jj <= jz; ++jj) m = fmaxf(m, kmax[tk * kScM + jj]);
                    S[sm.sel(b, g, Hkv, t0 + tk) * nblk_max + blk] = m;
                }
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");  // kmax is rewritten by the next chunk
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Blocks per 128-kernel chunk such that a chunk's blocks overlap at most 128 kernels.
int score_tc_blocks_per_chunk(const Params& p) {
    for (int nb = 256; nb >= 1; --nb)
        if (last_kernel_of_block(nb - 1, p.block_size, p.kernel_stride) -
                first_kernel_of_block(0, p.block_size, p.kernel_size, p.kernel_stride) + 1 <= kScM &&
            (nb * p.block_size + p.kernel_size) / p.kernel_stride + 1 <= kScM)
            return nb;
    return 0;
}

bool score_tc_supported(const SelectArgs& a) {
    return a.Hq / a.Hkv == 16 && (a.d == 64 || a.d == 128) && a.M_max > 0 &&
           score_tc_blocks_per_chunk(a.p) > 0;
}

cudaError_t launch_score_tc(const SelectArgs& a, float* S) {
    const int nb = score_tc_blocks_per_chunk(a.p);
    const int nblk_max = (a.L_max + a.p.block_size - 1) / a.p.block_size;
    CUtensorMap tq, tk;
    const SeqMap sm = a.seqmap();
    const uint64_t q_rows = static_cast<uint64_t>(sm.total) * a.Hq;
    const uint64_t k_rows = static_cast<uint64_t>(a.B) * a.Hkv * a.M_max;
    if (!make_tmap_bf16_2d(&tq, a.q, a.d, q_rows, 64, 16) || !make_tmap_bf16_2d(&tk, a.kernel_cache, a.d, k_rows, 64, kScM))
        return cudaErrorInvalidValue;
    // few query tiles (a draft tree, a short chunk): split each tile's chunks of blocks over CTAs
    const int tiles = ((a.Tq + kScTokens - 1) / kScTokens) * a.B * a.Hkv;
    const int chunks_max = (nblk_max - 1) / nb + 1;
    const int n_split = std::max(1, std::min(chunks_max, 300 / std::max(tiles, 1)));
    dim3 grid((a.Tq + kScTokens - 1) / kScTokens, a.B * a.Hkv, n_split);
    if (a.d == 128) {
        auto kfn = score_tc_kernel<128>;
        constexpr int smem = ScSmem<128>::kBytes;
        if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); e != cudaSuccess)
            return e;
        return launch_kernel(kfn, grid, dim3(kScThreads), smem, a.stream, false, tq, tk, a.kv_len, sm, a.tree, a.Hq, a.Hkv,
                             a.L_max, a.M_max, nblk_max, a.p, nb, S, a.err);
    }
    auto kfn = score_tc_kernel<64>;
    constexpr int smem = ScSmem<64>::kBytes;
    if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); e != cudaSuccess)
        return e;
    return launch_kernel(kfn, grid, dim3(kScThreads), smem, a.stream, false, tq, tk, a.kv_len, sm, a.tree, a.Hq, a.Hkv,
                         a.L_max, a.M_max, nblk_max, a.p, nb, S, a.err);
}

}  // namespace infllmv2
