// decode_cluster.cu -- single-token decode of one row per thread-block cluster: block scores,
// top-k selection, attention over the selected blocks and the merge of the partial results
// ("MiniCPM4: 如何在手机电脑上高效运行大语言模型", section 1.1 "InfLLM v2": semantic-kernel
// block scores, top-k with forced initial and local blocks, attention on the selected blocks;
// "CPM.cu：端侧大模型推理的 CUDA 加速引擎": sparse attention inside the decode step).
//
// A decode row is (sequence b, KV head g): the G query heads that share one selection.  At
// 128K tokens a row reads ~2 MB of semantic kernels and ~2 MB of selected K/V, a fraction of a
// microsecond of HBM time per SM, so the cost is the chain of dependent steps.  A cluster of CL
// CTAs (one per SM) takes the whole row and keeps every intermediate in shared memory:
//   1. CTA r scores the blocks [r*CB, (r+1)*CB): TMA copies of their kernel rows (issued before
//      the cache length is read, for the longest cache), warp MMAs q.k for the G heads, max over
//      the heads, then over the kernels overlapping each block -> its scores in shared memory.
//   2. Cluster barrier.  Every CTA reads all of the row's scores from its peers' shared memory
//      and computes the same selection: forced initial and local blocks, and the top-k of the
//      others by their scores' order-preserving keys (k-th largest key found two bits per round
//      from block-wide counts; ties go to the lower block), or every block below dense_len.
//   3. CTA r attends to the selected blocks r, r+CL, ...: TMA copies of their K and V, the
//      warp-MMA online softmax of attn_warp.cuh (32 keys per warp), a merge of the 8 warps into
//      an fp32 partial (m, l, o) in shared memory.
//   4. Cluster barrier.  CTA r merges the CL partials of heads r, r+CL, ... from its peers'
//      shared memory into o (bf16) and lse, and a last barrier keeps every CTA's shared memory
//      alive until its peers have read it.
// No global memory is written but the outputs, and nothing is carried between launches.
#include <algorithm>

#include "attn_warp.cuh"
#include "internal.h"
#include "pool.cuh"
#include "umma.cuh"

namespace infllmv2 {

constexpr int kDcThreads = 256;   // 8 warps
constexpr int kDcKRows = 768;     // kernel rows of one scoring pass (6 TMA boxes of 128 rows)
constexpr int kDcMaxSel = 4096;   // selection capacity covered (the list lives in shared memory)
constexpr int kDcMaxPer = 16;     // keys per thread in the selection: rows of up to 4096 blocks
constexpr int kDcCand = 384;      // candidates ranked exactly after the pre-threshold
constexpr int kDcFastPer = 8;     // strided keys per thread on the fast selection path (<= 2048 blocks)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ float dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// All threads of all CTAs of the cluster: earlier shared-memory writes (local or remote) are
// visible to every CTA after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

struct ClusterShape {
    int nblk_max;  // blocks of an L_max cache
    int CB;        // blocks scored per CTA
    int SC;        // blocks per scoring pass (kernel rows <= kDcKRows - 8)
    int S_cap;     // selection capacity (entries of the list)
};

template <int D, int BS>
struct ClusterSmem {
    static constexpr int kTile = BS * D * 2;                  // one K (or V) block
    static constexpr int kX = (D / 64) * kDcKRows * 128;      // scoring tiles / K,V tiles / merge scratch
    static constexpr int kPB = kX / (2 * kTile) < 8 ? kX / (2 * kTile) : 8;  // blocks per attention pass
    static constexpr int kMerge = (8 * 16 * 2 + 8 * 16 * (D + 4)) * 4;
    static constexpr int kPartial = (32 + 16 * D) * 4;         // m[16], l[16], o[16][D]
    static_assert(kMerge <= kX, "merge scratch fits the tile memory");
    // offsets from the 1024-aligned base: tiles | partial (the Q tile while scoring) | keys[nblk_max]
    // | ks | sel[S_cap] | barriers
    static_assert(kPartial >= (D / 64) * 16 * 128, "the Q tile fits the partial");
    __host__ __device__ static int off_p() { return kX; }
    __host__ __device__ static int off_keys() { return kX + ((kPartial + 15) & ~15); }
    __host__ __device__ static int off_ks(int nblk_max) { return off_keys() + ((4 * nblk_max + 15) & ~15); }
    __host__ __device__ static int off_sel(int nblk_max) { return off_ks(nblk_max) + 4 * kDcKRows; }
    __host__ __device__ static int off_bar(int nblk_max, int S_cap) { return (off_sel(nblk_max) + 4 * S_cap + 15) & ~15; }
    static int bytes(int nblk_max, int S_cap) { return off_bar(nblk_max, S_cap) + 8 * (1 + kPB) + 1024; }
};

template <int D, int BS, bool kAppend>
__global__ void __launch_bounds__(kDcThreads, 1)
decode_cluster_kernel(const __grid_constant__ CUtensorMap tm_kern, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q,
                      const __nv_bfloat16* __restrict__ q,
                      const int* __restrict__ kv_len, int Hq, int Hkv, int G, int L_max, int M_max, Params p,
                      ClusterShape sh, int* __restrict__ idx_out, int idx_stride, int* __restrict__ counts_out,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse, float scale_log2,
                      int* __restrict__ err, const __nv_bfloat16* __restrict__ k_new,
                      const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* k_w, __nv_bfloat16* v_w,
                      __nv_bfloat16* kern_w) {
    using SM = ClusterSmem<D, BS>;
    constexpr int PB = SM::kPB;
    constexpr int kTile = SM::kTile;
    constexpr int kTilesPerBlock = BS / 32;
    constexpr int kRowPad = D + 4;
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint32_t* keys = reinterpret_cast<uint32_t*>(base + SM::off_keys());           // [nblk_max], filled by all CTAs
    float* ks = reinterpret_cast<float*>(base + SM::off_ks(sh.nblk_max));           // [kDcKRows]
    float* part = reinterpret_cast<float*>(base + SM::off_p());                     // m, l, o
    int* sel = reinterpret_cast<int*>(base + SM::off_sel(sh.nblk_max));             // [S_cap]
    uint64_t* bar_a = reinterpret_cast<uint64_t*>(base + SM::off_bar(sh.nblk_max, sh.S_cap));
    uint64_t* bar_b = bar_a + 1;  // [PB]
    __shared__ int s_wsum[2][kDcThreads / 32];
    __shared__ int s_cnt[3][4];
    __shared__ float s_w[32];
    __shared__ float s_f[8][16];  // merge weights of the 8 warps per row
    __shared__ unsigned long long s_cv[kDcCand];          // candidates >= tau: key << 32 | ~block
    __shared__ int s_rk[kDcCand];                          // their ranks
    __shared__ uint32_t s_bits[kDcFastPer * kDcThreads / 32];  // chosen blocks (fast path), one bit each
    __shared__ int s_wpre[kDcFastPer * kDcThreads / 32];       // chosen blocks below each bitmap word
    __shared__ uint64_t s_bar_piece[kDcKRows / 128];       // scoring: kernel rows of piece p landed
    __shared__ uint64_t s_bar_mma[2], s_bar_free[2];       // scoring accumulator buffers: written / read
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const uint32_t rank = cluster_ctarank();
    const int ncta = static_cast<int>(cluster_nctarank());
    const int row = blockIdx.x / ncta;
    const int b = row / Hkv, g = row % Hkv;
    const int c = p.kernel_size, s = p.kernel_stride;

    if (tid == 0) {
        prefetch_tmap(&tm_kern);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
        mbar_init(bar_a, 1);
        for (int k = 0; k < PB; ++k) mbar_init(&bar_b[k], 1);
        for (int k = 0; k < kDcKRows / 128; ++k) mbar_init(&s_bar_piece[k], 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s_bar_mma[k], 1);
            mbar_init(&s_bar_free[k], 128);
        }
        fence_mbar_init();
    }
    if (warp == 0) {  // scoring accumulators: 2 x 16 TMEM columns (kernel row x head, fp32)
        tmem_alloc(&s_tmem, 32);
        tmem_relinquish();
    }
    if (tid < 12) (&s_cnt[0][0])[tid] = 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // Launched with programmatic stream serialisation: the set-up above may overlap the previous
    // kernel's tail; nothing the previous kernel may write is read before this wait.
    pdl_trigger();
    pdl_wait();

    // ================= 1. scores of this CTA's blocks, pushed as keys to every CTA
    // Thread 128 (warp 4) issues the TMA copies (Q once, then 128-row pieces of kernel rows) and,
    // per piece, the tcgen05 MMAs S[kernel row][head] = K_kernel Q^T (M=128, N=16, K=d) into one of
    // two TMEM buffers; warps 0-3 read each piece back (one kernel row per thread) and keep the
    // maximum over the G heads.  A piece is scored as soon as it lands.
    constexpr int kPieces = kDcKRows / 128;
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, 16, 0, 0);
    const int blkA0 = static_cast<int>(rank) * sh.CB;
    const int blkA1 = min(blkA0 + sh.CB, sh.nblk_max);
    const bool issuer = tid == 128;
    const uint32_t sQ = smem_u32(part);
    uint32_t piece_uses = 0;  // issuer: bit p = phase parity of s_bar_piece[p]
    int gi = 0;               // scoring MMA groups so far (issuer and readers count alike)
    auto pass_rows = [&](int sub0, int& jlo, int& jend) {
        const int sub1 = min(sub0 + sh.SC, blkA1);
        jlo = first_kernel_of_block(sub0, BS, c, s);
        jend = min(last_kernel_of_block(sub1 - 1, BS, s), M_max - 1);
        return jend - jlo + 1;
    };
    auto issue_pass = [&](int sub0) {  // kernel rows of blocks [sub0, sub0 + SC) for the longest cache
        int jlo, jend;
        const int nrows = pass_rows(sub0, jlo, jend);
        for (int pc = 0; pc * 128 < nrows; ++pc) {
            mbar_arrive_expect_tx(&s_bar_piece[pc], (D / 64) * 128 * 128);
            for (int half = 0; half < D / 64; ++half)
                tma_load_2d(base + half * (kDcKRows * 128) + pc * (128 * 128), &tm_kern, 64 * half,
                            row * M_max + jlo + pc * 128, &s_bar_piece[pc]);
        }
    };
    if (issuer) {
        mbar_arrive_expect_tx(bar_a, (D / 64) * 16 * 128);
        for (int half = 0; half < D / 64; ++half)
            tma_load_2d(part + half * (16 * 128 / 4), &tm_q, 64 * half, b * Hq + g * G, bar_a);
        if (blkA0 < blkA1) issue_pass(blkA0);
    }
    // Q fragments: rows = heads (rows >= G read as zero), for the attention
    QFrag<D> Q;
    load_q(Q, q + (static_cast<size_t>(b) * Hq + static_cast<size_t>(g) * G) * D, D, G);
    const int L = kv_len[b];
    const bool len_ok = L >= 1 && L <= L_max && kernels_in(L, c, s) <= M_max;
    const int bt = len_ok ? (L - 1) / BS : -1;
    const bool dense = L < p.dense_len;
    auto forced = [&](int blk) { return blk < p.n_init || blk > bt - p.n_local; };
    // Decode-step append (the kAppend instance): CTA 0 writes this row's new K and V into cache row L-1
    // (the attention below reads them after the first cluster barrier), and warp 5 of every CTA
    // pools its share of the 8-element slices of the kernel the new token completes, for the steps
    // to come.  This step's scores never need that kernel: it overlaps only the query's own block
    // and the one before, both local (forced) blocks under the condition the host checks.
    if constexpr (kAppend) {
      if (len_ok) {
        const int pn = L - 1;
        const uint4* kn = reinterpret_cast<const uint4*>(k_new + static_cast<size_t>(row) * D);
        if (rank == 0 && warp == 6 && lane < D / 8) {
            const size_t wr = (static_cast<size_t>(row) * L_max + pn) * D;
            reinterpret_cast<uint4*>(k_w + wr)[lane] = ldg_v4(kn + lane);
            reinterpret_cast<uint4*>(v_w + wr)[lane] =
                ldg_v4(reinterpret_cast<const uint4*>(v_new + static_cast<size_t>(row) * D) + lane);
        }
        if (warp == 5 && L >= c && (L - c) % s == 0) {
            const int jn = (L - c) / s, r0 = jn * s;  // jn < M_max: len_ok
            const uint4* kr = reinterpret_cast<const uint4*>(k_w + (static_cast<size_t>(row) * L_max + r0) * D);
            for (int sl0 = 2 * static_cast<int>(rank); sl0 < D / 8; sl0 += 2 * ncta) {
                const int sl = sl0 + (lane >> 4);
                const bool live = sl < D / 8;
                const uint4 sub = live ? ldg_v4(kn + sl) : make_uint4(0u, 0u, 0u, 0u);
                const uint4 mean = exact_mean_slice(kr + (live ? sl : 0), D / 8, live ? c : 0, lane & 15, pn - r0, sub);
                if (live && (lane & 15) == 0)
                    reinterpret_cast<uint4*>(kern_w + (static_cast<size_t>(row) * M_max + jn) * D)[sl] = mean;
            }
        }
      }
    }
    const uint32_t keys_base = smem_u32(keys);
    bool q_landed = false;
    for (int sub0 = blkA0; sub0 < blkA1; sub0 += sh.SC) {
        int jlo, jend;
        const int nrows = pass_rows(sub0, jlo, jend);
        const int sub1 = min(sub0 + sh.SC, blkA1);
        const bool work = len_ok && !dense && sub0 <= bt && nrows > 0;
        const int bz = min(sub1, bt + 1);  // blocks [sub0, bz) are scored
        const int jhi = work ? min(min(last_kernel_of_block(bz - 1, BS, s), kernels_in(L, c, s) - 1), jend) : -1;
        const int nj = work ? jhi - jlo + 1 : 0;  // visible kernel rows of the pass
        const int n_issued = nrows > 0 ? (nrows + 127) / 128 : 0;
        const int n_mma = nj > 0 ? (nj + 127) / 128 : 0;
        if (issuer) {
            bool ok = true;
            if (n_mma > 0 && !q_landed) {
                ok = mbar_wait(bar_a, 0);
                q_landed = true;
            }
            for (int pc = 0; pc < n_issued; ++pc) {
                // every issued piece must land before its tiles are reused, scored or not
                const bool landed = mbar_wait(&s_bar_piece[pc], (piece_uses >> pc) & 1u);
                ok = ok && landed;
                piece_uses ^= 1u << pc;
                if (pc >= n_mma) continue;
                const int buf = (gi + pc) & 1;
                if (gi + pc >= 2) ok = ok && mbar_wait(&s_bar_free[buf], ((gi + pc - 2) >> 1) & 1);
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ko = (kk / 4) * (kDcKRows * 128) + (kk % 4) * 32;
                        const uint32_t qo = (kk / 4) * (16 * 128) + (kk % 4) * 32;
                        mma_ss(tmem + 16 * buf, sw128_desc(smem_u32(base) + pc * (128 * 128) + ko, 16, 1024),
                               sw128_desc(sQ + qo, 16, 1024), kIdesc, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit(&s_bar_mma[buf]);  // also when not issued: the readers' waits stay in step
            }
            if (!ok) raise_error(err, kDevErrTimeout);
        } else if (warp < 4) {
            for (int pc = 0; pc < n_mma; ++pc) {
                const int buf = (gi + pc) & 1;
                const bool got = mbar_wait(&s_bar_mma[buf], ((gi + pc) >> 1) & 1);
                tc_fence_after();
                uint32_t v[16];
                tmem_ld16(tmem + 16 * buf + (static_cast<uint32_t>(32 * warp) << 16), v);
                tmem_ld_wait16(v);
                tc_fence_before();
                mbar_arrive(&s_bar_free[buf]);
                const int r = pc * 128 + 32 * warp + lane;  // kernel row jlo + r
                if (got && r < nj) {
                    float m = -INFINITY;
#pragma unroll
                    for (int h = 0; h < 16; ++h)
                        if (h < G) m = fmaxf(m, __uint_as_float(v[h]));
                    ks[r] = m;
                } else if (!got && lane == 0) {
                    raise_error(err, kDevErrTimeout);
                }
            }
        }
        gi += n_mma;
        __syncthreads();
        if (work) {
            // block score = max over its visible kernels; its selection key goes to every CTA
            for (int blk = sub0 + tid; blk < bz; blk += kDcThreads) {
                const int ja = max(first_kernel_of_block(blk, BS, c, s), jlo);
                const int jz = min(last_kernel_of_block(blk, BS, s), jhi);
                float m = -INFINITY;
                for (int jj = ja; jj <= jz; ++jj) m = fmaxf(m, ks[jj - jlo]);
                const uint32_t key = forced(blk) ? 0u : ordered_key(m);  // 0: not a candidate
                const uint32_t a = keys_base + 4u * blk;
                for (int j = 0; j < ncta; ++j) dsmem_st_u32(dsmem_addr(a, j), key);
            }
        }
        __syncthreads();  // tiles and ks free for the next pass
        if (issuer && sub0 + sh.SC < blkA1) issue_pass(sub0 + sh.SC);
    }
    if (issuer && !q_landed) mbar_wait(bar_a, 0);  // the Q copy has landed before its tile is reused
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
    cluster_sync();

    // ================= 2. the row's selection, computed by every CTA from all the keys
    int count = 0;
    {
        const int n = bt + 1;
        const int a_init = min(p.n_init, max(n, 0));
        const int lo_local = max(bt - p.n_local + 1, 0);
        const int n_forced = len_ok ? a_init + (n - max(lo_local, a_init)) : 0;
        const int nc = n - n_forced;
        const bool take_all = len_ok && (dense || nc <= p.topk);
        const bool select = len_ok && !take_all && p.topk > 0;
        const int nn = max(n, 0);
        const int lo_f = max(lo_local, a_init);  // first local block not already an initial one
        int total = 0;
        bool done = false;
        if (select && nn <= kDcFastPer * kDcThreads && p.topk <= kDcThreads) {
            // Fast path.  tau = the k-th largest of the threads' maxima over the strided keys
            // t, t + 256, ... (neighbouring blocks have correlated scores: a stride spreads each
            // thread over the row), found bit by bit from block-wide predicate counts.  At least
            // k keys are >= tau and, unless the scores are heavily tied, only a few more; those
            // candidates are ranked exactly (key descending, block ascending, one 64-bit
            // compare), and the list is the initial blocks, the k best candidates in block order
            // and the local blocks.
            const int k = p.topk;
            uint32_t kv[kDcFastPer];
            uint32_t mx = 0u;
#pragma unroll
            for (int u = 0; u < kDcFastPer; ++u) {
                const int i = tid + u * kDcThreads;
                kv[u] = i < nn ? keys[i] : 0u;
                mx = max(mx, kv[u]);
            }
            const int nz = __syncthreads_count(mx != 0u);
            uint32_t k_and = __reduce_and_sync(0xffffffffu, mx != 0u ? mx : ~0u);
            uint32_t k_or = __reduce_or_sync(0xffffffffu, mx);
            if (lane == 0) {
                s_wsum[0][warp] = static_cast<int>(k_and);
                s_wsum[1][warp] = static_cast<int>(k_or);
            }
            __syncthreads();
            k_and = ~0u;
            k_or = 0u;
#pragma unroll
            for (int w = 0; w < kDcThreads / 32; ++w) {
                k_and &= static_cast<uint32_t>(s_wsum[0][w]);
                k_or |= static_cast<uint32_t>(s_wsum[1][w]);
            }
            if (nz >= k) {
                const uint32_t diff = k_and ^ k_or;
                int bit = diff == 0u ? -1 : 31 - __clz(diff);
                uint32_t tau = bit >= 31 ? 0u : (k_and & (~0u << (bit + 1)));
                for (; bit >= 0; --bit) {
                    const uint32_t trial = tau | (1u << bit);
                    const int cnt = __syncthreads_count(mx >= trial);
                    if (cnt >= k) tau = trial;
                    if (cnt == k) break;
                }
                int nc_t = 0;
#pragma unroll
                for (int u = 0; u < kDcFastPer; ++u) nc_t += (kv[u] != 0u && kv[u] >= tau) ? 1 : 0;
                int incl = nc_t;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int x = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += x;
                }
                __syncthreads();  // s_wsum reuse
                if (lane == 31) s_wsum[0][warp] = incl;
                __syncthreads();
                int c_before = incl - nc_t, c_total = 0;
#pragma unroll
                for (int w = 0; w < kDcThreads / 32; ++w) {
                    if (w < warp) c_before += s_wsum[0][w];
                    c_total += s_wsum[0][w];
                }
                if (c_total <= kDcCand) {
                    // candidate value: key in the high word, complemented block in the low word,
                    // so that a larger value is a better block
#pragma unroll
                    for (int u = 0; u < kDcFastPer; ++u)
                        if (kv[u] != 0u && kv[u] >= tau)
                            s_cv[c_before++] = (static_cast<unsigned long long>(kv[u]) << 32) |
                                               static_cast<uint32_t>(~(tid + u * kDcThreads));
                    for (int i = tid; i < c_total; i += kDcThreads) s_rk[i] = 0;
                    for (int i = tid; i < kDcFastPer * kDcThreads / 32; i += kDcThreads) s_bits[i] = 0u;
                    __syncthreads();
                    // rank of candidate i = number of better candidates; `sp` threads share each
                    // candidate, each comparing it with one slice of the others
                    const int sp = max(1, kDcThreads / c_total);
                    const int seg = (c_total + sp - 1) / sp;
                    {
                        const int i = tid / sp, part = tid % sp;
                        if (i < c_total) {
                            const unsigned long long vi = s_cv[i];
                            const int j1 = min(c_total, (part + 1) * seg);
                            int r0 = 0, r1 = 0, r2 = 0, r3 = 0;  // four independent chains of loads
                            int j = part * seg;
                            for (; j + 4 <= j1; j += 4) {
                                r0 += s_cv[j] > vi ? 1 : 0;
                                r1 += s_cv[j + 1] > vi ? 1 : 0;
                                r2 += s_cv[j + 2] > vi ? 1 : 0;
                                r3 += s_cv[j + 3] > vi ? 1 : 0;
                            }
                            for (; j < j1; ++j) r0 += s_cv[j] > vi ? 1 : 0;
                            const int rnk = r0 + r1 + r2 + r3;
                            if (rnk) atomicAdd(&s_rk[i], rnk);
                        }
                        for (int i2 = kDcThreads / sp + tid; i2 < c_total; i2 += kDcThreads) {  // c_total > 256
                            const unsigned long long vi = s_cv[i2];
                            int rnk = 0;
                            for (int j = 0; j < c_total; ++j) rnk += s_cv[j] > vi ? 1 : 0;
                            atomicAdd(&s_rk[i2], rnk);
                        }
                    }
                    __syncthreads();
                    // position of a chosen candidate = chosen blocks below it: bitmap of the chosen
                    // blocks, word prefix popcounts (one warp), then one popcount per candidate
                    for (int i = tid; i < c_total; i += kDcThreads)
                        if (s_rk[i] < k) {
                            const uint32_t blk = ~static_cast<uint32_t>(s_cv[i]);
                            atomicOr(&s_bits[blk >> 5], 1u << (blk & 31));
                        }
                    __syncthreads();
                    if (warp == 0) {
                        const int c0 = __popc(s_bits[2 * lane]), c1 = __popc(s_bits[2 * lane + 1]);
                        int incl = c0 + c1;
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1) {
                            const int x = __shfl_up_sync(0xffffffffu, incl, off);
                            if (lane >= off) incl += x;
                        }
                        s_wpre[2 * lane] = incl - c0 - c1;
                        s_wpre[2 * lane + 1] = incl - c1;
                    }
                    __syncthreads();
                    for (int i = tid; i < c_total; i += kDcThreads)
                        if (s_rk[i] < k) {
                            const uint32_t blk = ~static_cast<uint32_t>(s_cv[i]);
                            sel[a_init + s_wpre[blk >> 5] + __popc(s_bits[blk >> 5] & ((1u << (blk & 31)) - 1u))] =
                                static_cast<int>(blk);
                        }
                    for (int i = tid; i < a_init; i += kDcThreads) sel[i] = i;
                    for (int i = tid; i < nn - lo_f; i += kDcThreads) sel[a_init + k + i] = lo_f + i;
                    total = a_init + k + (nn - lo_f);
                    done = true;
                }
            }
            __syncthreads();
        }
        if (!done) {
            // General path: thread t holds the keys of blocks [t*per, t*per + per); the k-th
            // largest key T is decided two bits per round from block-wide counts; the list is
            // compacted in block order.
            const int per = (nn + kDcThreads - 1) / kDcThreads;
            const int i0 = min(tid * per, nn), i1 = min(i0 + per, nn);
            uint32_t kr[kDcMaxPer];
#pragma unroll
            for (int u = 0; u < kDcMaxPer; ++u) kr[u] = select && i0 + u < i1 ? keys[i0 + u] : 0u;
            uint32_t T = 0;
            int krem = 0;
            if (select) {
                uint32_t k_and = ~0u, k_or = 0u;
#pragma unroll
                for (int u = 0; u < kDcMaxPer; ++u)
                    if (kr[u] != 0u) {
                        k_and &= kr[u];
                        k_or |= kr[u];
                    }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    k_and &= __shfl_xor_sync(0xffffffffu, k_and, off);
                    k_or |= __shfl_xor_sync(0xffffffffu, k_or, off);
                }
                if (lane == 0) {
                    s_wsum[0][warp] = static_cast<int>(k_and);
                    s_wsum[1][warp] = static_cast<int>(k_or);
                }
                __syncthreads();
                k_and = ~0u;
                k_or = 0u;
#pragma unroll
                for (int w = 0; w < kDcThreads / 32; ++w) {
                    k_and &= static_cast<uint32_t>(s_wsum[0][w]);
                    k_or |= static_cast<uint32_t>(s_wsum[1][w]);
                }
                // bits above the highest one where candidate keys differ are common to all; below
                // it the k-th largest key is decided two bits per round from the counts of keys >=
                // three trial values (warp reductions, shared atomics, one barrier; the counters of
                // round r+1, last read in round r-2, are cleared in round r)
                const uint32_t diff = k_and ^ k_or;
                int bit = diff == 0u ? -1 : 31 - __clz(diff);
                T = bit >= 31 ? 0u : (k_and & (~0u << (bit + 1)));
                const int k = p.topk;
                int buf = 0;
                while (bit >= 0) {
                    const int nb = bit >= 1 ? 2 : 1;
                    const int lo = bit - nb + 1;
                    uint32_t tr[3];
                    int cn[3] = {0, 0, 0};
#pragma unroll
                    for (int u = 0; u < 3; ++u) tr[u] = T | (static_cast<uint32_t>(u + 1) << lo);
#pragma unroll
                    for (int u = 0; u < kDcMaxPer; ++u)
#pragma unroll
                        for (int v = 0; v < 3; ++v) cn[v] += kr[u] >= tr[v] ? 1 : 0;
#pragma unroll
                    for (int v = 0; v < 3; ++v) cn[v] = __reduce_add_sync(0xffffffffu, cn[v]);
                    if (lane == 0)
#pragma unroll
                        for (int v = 0; v < 3; ++v) atomicAdd(&s_cnt[buf][v], cn[v]);
                    if (tid < 3) s_cnt[(buf + 1) % 3][tid] = 0;
                    __syncthreads();
                    int pick = -1;
                    for (int v = (nb == 2 ? 2 : 0); v >= 0; --v)
                        if (s_cnt[buf][v] >= k) {
                            pick = v;
                            break;
                        }
                    const bool exact = pick >= 0 && s_cnt[buf][pick] == k;
                    if (pick >= 0) T = tr[pick];
                    bit -= nb;
                    buf = (buf + 1) % 3;
                    if (exact) break;  // exactly k keys clear T: no ties to break
                }
                // keys above T are taken, and of the keys equal to T the lowest blocks
                int above = 0;
#pragma unroll
                for (int u = 0; u < kDcMaxPer; ++u) above += kr[u] > T ? 1 : 0;
                above = __reduce_add_sync(0xffffffffu, above);
                if (lane == 0) atomicAdd(&s_cnt[buf][3], above);  // slot 3: zero since the start
                __syncthreads();
                krem = k - s_cnt[buf][3];
            }
            // ---- ascending compaction: forced, keys above T, the first krem keys equal to T
            int n_sel = 0, n_tie = 0;
            if (len_ok) {
                if (!select) {
                    for (int i = i0; i < i1; ++i) n_sel += (take_all || forced(i)) ? 1 : 0;
                } else {
#pragma unroll
                    for (int u = 0; u < kDcMaxPer; ++u) {
                        if (i0 + u >= i1) break;
                        if (forced(i0 + u)) {
                            ++n_sel;
                        } else {
                            n_sel += kr[u] > T;
                            n_tie += kr[u] == T;
                        }
                    }
                }
            }
            int sel_incl = n_sel, tie_incl = n_tie;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, sel_incl, off);
                const int y = __shfl_up_sync(0xffffffffu, tie_incl, off);
                if (lane >= off) {
                    sel_incl += x;
                    tie_incl += y;
                }
            }
            __syncthreads();  // s_wsum reuse
            if (lane == 31) {
                s_wsum[0][warp] = sel_incl;
                s_wsum[1][warp] = tie_incl;
            }
            __syncthreads();
            int sel_before = sel_incl - n_sel, tie_before = tie_incl - n_tie, sel_total = 0, tie_total = 0;
#pragma unroll
            for (int w = 0; w < kDcThreads / 32; ++w) {
                if (w < warp) {
                    sel_before += s_wsum[0][w];
                    tie_before += s_wsum[1][w];
                }
                sel_total += s_wsum[0][w];
                tie_total += s_wsum[1][w];
            }
            int pos = sel_before + min(tie_before, krem);
            int tie_rank = tie_before;
            if (len_ok) {
                if (!select) {
                    for (int i = i0; i < i1; ++i)
                        if (take_all || forced(i)) {
                            if (pos < sh.S_cap) sel[pos] = i;
                            ++pos;
                        }
                } else {
#pragma unroll
                    for (int u = 0; u < kDcMaxPer; ++u) {
                        if (i0 + u >= i1) break;
                        bool pick = forced(i0 + u) || kr[u] > T;
                        if (!pick && kr[u] == T) {
                            pick = tie_rank < krem;
                            ++tie_rank;
                        }
                        if (pick) {
                            if (pos < sh.S_cap) sel[pos] = i0 + u;
                            ++pos;
                        }
                    }
                }
            }
            total = sel_total + min(tie_total, krem);
        }
        count = min(total, sh.S_cap);
        __syncthreads();  // sel complete
        if (rank == 0) {
            if (tid == 0 && (total > sh.S_cap || !len_ok)) raise_error(err, kDevErrIndex);
            if (idx_out != nullptr) {
                int* out = idx_out + static_cast<size_t>(row) * idx_stride;
                for (int i = tid; i < idx_stride; i += kDcThreads) out[i] = i < count ? sel[i] : -1;
                if (tid == 0) counts_out[row] = count;
            }
        }
    }

    // ================= 3. attention over the selected blocks rank, rank + CL, ...
    WarpAcc<D> A;
    acc_init(A);
    // an appended K/V row (generic stores of CTA 0, released and acquired by the cluster barrier)
    // is read below by this thread's bulk copies
    if constexpr (kAppend)
        if (tid == 0) fence_proxy_async_global();
    {
        const int mine = count > static_cast<int>(rank) ? (count - static_cast<int>(rank) + ncta - 1) / ncta : 0;
        uint32_t ph_b = 0;
        for (int t0 = 0; t0 < mine; t0 += PB) {
            if (tid == 0) {
#pragma unroll
                for (int k = 0; k < PB; ++k) {
                    const int t = t0 + k;
                    const int blk = t < mine ? sel[static_cast<int>(rank) + ncta * t] : -1;
                    if (blk >= 0) {
                        const int krow = row * L_max + blk * BS;
                        mbar_arrive_expect_tx(&bar_b[k], 2 * kTile);
#pragma unroll
                        for (int sub = 0; sub < D / 64; ++sub) {
                            tma_load_2d(base + (2 * k) * kTile + sub * BS * 128, &tm_k, 64 * sub, krow, &bar_b[k]);
                            tma_load_2d(base + (2 * k + 1) * kTile + sub * BS * 128, &tm_v, 64 * sub, krow, &bar_b[k]);
                        }
                    } else {
                        mbar_arrive(&bar_b[k]);  // keep every slot's phase in step
                    }
                }
            }
            __syncthreads();
            for (int tile = warp; tile < PB * kTilesPerBlock; tile += kDcThreads / 32) {
                const int k = tile / kTilesPerBlock;
                const int t = t0 + k;
                if (t >= mine) continue;
                const int blk = sel[static_cast<int>(rank) + ncta * t];
                const int r0 = (tile % kTilesPerBlock) * 32;
                const int n_ok = L - (blk * BS + r0);
                if (n_ok <= 0) continue;
                const uint32_t valid = n_ok >= 32 ? 0xffffffffu : ((1u << n_ok) - 1u);
                if (mbar_wait(&bar_b[k], ph_b)) {
                    attend32_smem<D>(A, Q, smem_u32(base + (2 * k) * kTile), smem_u32(base + (2 * k + 1) * kTile), BS,
                                     r0, valid, scale_log2);
                } else if (lane == 0) {
                    raise_error(err, kDevErrTimeout);
                }
            }
            // every copy of this pass has landed and been read before the tiles are refilled
            if (tid == 0) {
#pragma unroll
                for (int k = 0; k < PB; ++k)
                    if (!mbar_wait(&bar_b[k], ph_b)) raise_error(err, kDevErrTimeout);
            }
            ph_b ^= 1u;
            __syncthreads();
        }
    }
    acc_finish_rowsum(A);
    {
        // merge the 8 warps (scratch in the tile memory) into this CTA's partial
        float* sm_m = reinterpret_cast<float*>(base);
        float* sm_l = sm_m + 8 * 16;
        float* sm_o = sm_l + 8 * 16;  // [8][16][kRowPad]
        if (cq == 0) {
            sm_m[warp * 16 + gq] = A.m[0];
            sm_m[warp * 16 + gq + 8] = A.m[1];
            sm_l[warp * 16 + gq] = A.l[0];
            sm_l[warp * 16 + gq + 8] = A.l[1];
        }
        // column c of a row is stored at c + c/32: the four lanes of a quad write different banks
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = o_col(D, cq, nt, e);
                sm_o[(warp * 16 + gq + 8 * (e >> 1)) * kRowPad + col + (col >> 5)] = A.o[nt][e];
            }
        __syncthreads();
        if (tid < 16) {  // per row: the warps' weights, the CTA's max and sum
            const int r = tid;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 8; ++w) M = fmaxf(M, sm_m[w * 16 + r]);
            const float ref = M == -INFINITY ? 0.f : M;
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const float f = fast_exp2(sm_m[w * 16 + r] - ref);
                s_f[w][r] = f;
                l += sm_l[w * 16 + r] * f;
            }
            part[r] = M;
            part[16 + r] = l;
        }
        __syncthreads();
        for (int e = tid; e < 16 * D; e += kDcThreads) {
            const int r = e / D, col = e % D;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) acc += sm_o[(w * 16 + r) * kRowPad + col + (col >> 5)] * s_f[w][r];
            part[32 + e] = acc;
        }
    }
    cluster_sync();

    // ================= 4. merge of the CTAs' partials: heads rank, rank + CL, ...
    const uint32_t p_base = smem_u32(part);
    for (int h = static_cast<int>(rank); h < G; h += ncta) {
        if (warp == 0) {
            // weights of the CTAs for head h
            float m = -INFINITY, l = 0.f;
            if (lane < ncta) {
                m = dsmem_f32(dsmem_addr(p_base + 4u * h, lane));
                l = dsmem_f32(dsmem_addr(p_base + 4u * (16 + h), lane));
            }
            float M = m;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            const float ref = M == -INFINITY ? 0.f : M;
            const float f = lane < ncta ? fast_exp2(m - ref) : 0.f;
            float Ls = l * f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
            s_w[lane] = f;
            if (lane == 0) {
                s_wsum[0][0] = __float_as_int(M);
                s_wsum[0][1] = __float_as_int(Ls);
            }
        }
        __syncthreads();
        const float M = __int_as_float(s_wsum[0][0]), Ls = __int_as_float(s_wsum[0][1]);
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        for (int d = tid; d < D; d += kDcThreads) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = j < ncta ? dsmem_f32(dsmem_addr(p_base + 4u * (32 + h * D + d), j)) : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) acc += v[j] * s_w[j];
            o[(static_cast<size_t>(b) * Hq + g * G + h) * D + d] = __float2bfloat16_rn(acc * inv);
        }
        if (lse != nullptr && tid == 0)
            lse[static_cast<size_t>(b) * Hq + g * G + h] = Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994530942f : -INFINITY;
        __syncthreads();
    }
    cluster_sync();  // peers have finished reading this CTA's shared memory
}

template <int D, int BS>
static cudaError_t launch_cluster_t(const DecodeArgs& a, const void* kernel_cache, int M_max, int* idx_out,
                                    int idx_stride, int* counts_out) {
    using SM = ClusterSmem<D, BS>;
    ClusterShape sh{};
    const int c = a.p.kernel_size, s = a.p.kernel_stride;
    sh.nblk_max = (a.L_max + BS - 1) / BS;
    if (sh.nblk_max > kDcMaxPer * kDcThreads) return cudaErrorNotSupported;
    // SC blocks span at most (SC*BS + c)/s + 2 kernel rows; keep 8 rows of slack for the last
    // n-tile of 8 rows
    sh.SC = std::max(1, ((kDcKRows - 10) * s - c) / BS);
    sh.S_cap = selection_capacity(a.p, a.L_max);
    if (sh.S_cap > kDcMaxSel) return cudaErrorNotSupported;
    const int smem = SM::bytes(sh.nblk_max, sh.S_cap);
    auto kfn = a.k_new != nullptr ? decode_cluster_kernel<D, BS, true> : decode_cluster_kernel<D, BS, false>;
    cudaFuncAttributes fa{};
    if (cudaError_t e = cudaFuncGetAttributes(&fa, kfn); e != cudaSuccess) return e;
    if (smem + static_cast<int>(fa.sharedSizeBytes) > 227 * 1024) return cudaErrorNotSupported;
    if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); e != cudaSuccess)
        return e;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        (void)cudaGetLastError();  // then only the portable sizes (<= 8) are offered below
    const int rows = a.B * a.Hkv;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kDcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // (cluster size search without the serialisation attribute)
    // cluster size: the largest whose clusters all fit on the device at once (one wave of rows);
    // if none does, the one that keeps the most SMs busy
    int CL = 0, best_sms = 0, fallback = 0;
    for (int cand : {16, 12, 8, 4, 2}) {
        attr[0].val.clusterDim.x = cand;
        cfg.gridDim = dim3(cand * rows);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kfn, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            continue;
        }
        if (n >= rows) {
            CL = cand;
            break;
        }
        if (n * cand > best_sms) {
            best_sms = n * cand;
            fallback = cand;
        }
    }
    if (CL == 0) CL = fallback;
    if (CL == 0) return cudaErrorNotSupported;
    sh.CB = (sh.nblk_max + CL - 1) / CL;
    attr[0].val.clusterDim.x = CL;
    cfg.gridDim = dim3(rows * CL);
    cfg.numAttrs = 2;  // + programmatic stream serialisation: set-up overlaps the previous kernel
    CUtensorMap tkern, tk, tv, tq;
    const uint64_t krows = static_cast<uint64_t>(a.B) * a.Hkv * M_max;
    const uint64_t cache_rows = static_cast<uint64_t>(a.B) * a.Hkv * a.L_max;
    if (!make_tmap_bf16_2d(&tkern, kernel_cache, D, krows, 64, 128) ||
        !make_tmap_bf16_2d(&tk, a.k_cache, D, cache_rows, 64, BS) ||
        !make_tmap_bf16_2d(&tv, a.v_cache, D, cache_rows, 64, BS) ||
        !make_tmap_bf16_2d(&tq, a.q, D, static_cast<uint64_t>(a.B) * a.Hq, 64, 16))
        return cudaErrorNotSupported;
    const int G = a.Hq / a.Hkv;
    const float scale_log2 = a.p.scale * 1.4426950408889634f;
    return cudaLaunchKernelEx(&cfg, kfn, tkern, tk, tv, tq, static_cast<const __nv_bfloat16*>(a.q), a.kv_len, a.Hq, a.Hkv,
                              G, a.L_max, M_max, a.p, sh, idx_out, idx_stride, counts_out,
                              static_cast<__nv_bfloat16*>(a.o), a.lse, scale_log2, a.err,
                              static_cast<const __nv_bfloat16*>(a.k_new), static_cast<const __nv_bfloat16*>(a.v_new),
                              static_cast<__nv_bfloat16*>(a.k_w), static_cast<__nv_bfloat16*>(a.v_w),
                              static_cast<__nv_bfloat16*>(a.kern_w));
}

bool decode_cluster_supported(const DecodeArgs& a, int M_max) {
    const int G = a.Hkv > 0 ? a.Hq / a.Hkv : 0;
    const int bs = a.p.block_size;
    if (a.tree_mask != nullptr || a.n_draft != 1) return false;
    if (G < 1 || G > 16 || (a.d != 64 && a.d != 128) || (bs != 64 && bs != 128)) return false;
    // the tensor maps' boxes must fit the tensors
    if (static_cast<long long>(a.B) * a.Hkv * M_max < 128 || static_cast<long long>(a.B) * a.Hkv * a.L_max < bs ||
        static_cast<long long>(a.B) * a.Hq < 16)
        return false;
    return true;
}

bool decode_cluster_can_append(const Params& p) {
    // a kernel of c tokens ending at the query spans at most ceil((c-1)/bs) + 1 blocks back from it
    const int span = (p.kernel_size - 1 + p.block_size - 1) / p.block_size + 1;
    return p.n_local >= span;
}

cudaError_t launch_decode_cluster(const DecodeArgs& a, const void* kernel_cache, int M_max, int* idx_out,
                                  int idx_stride, int* counts_out) {
    const int bs = a.p.block_size;
    if (a.d == 128)
        return bs == 64 ? launch_cluster_t<128, 64>(a, kernel_cache, M_max, idx_out, idx_stride, counts_out)
                        : launch_cluster_t<128, 128>(a, kernel_cache, M_max, idx_out, idx_stride, counts_out);
    return bs == 64 ? launch_cluster_t<64, 64>(a, kernel_cache, M_max, idx_out, idx_stride, counts_out)
                    : launch_cluster_t<64, 128>(a, kernel_cache, M_max, idx_out, idx_stride, counts_out);
}

}  // namespace infllmv2
