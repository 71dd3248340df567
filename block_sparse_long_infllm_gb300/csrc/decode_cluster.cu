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
//      the heads, then over the kernels overlapping each block -> its order-preserving keys.
//      Keys and lists travel by bulk copies into the peers' shared memory (counted on the
//      receiving CTA's barrier).
//   2. Every CTA computes the same selection: forced initial and local blocks, and the top-k of
//      the others (ties go to the lower block), or every block below dense_len.  Each CTA sorts
//      its blocks' keys and sends its best 16 to every peer; every candidate of those lists finds
//      its exact rank in the row by binary searches in the other lists.  That decides the top-k
//      unless some CTA holds 16 or more of it; then (and for rows the lists do not cover) the
//      CTAs exchange all their keys and a threshold from block-wide counts plus an exact ranking
//      of the few keys above it decides.  The forced blocks' K and V are brought towards L2 at the start, the few
//      candidates' while they are ranked (bulk prefetches), and before the programmatic wait the
//      CTA prefetches its q and kernel rows: a prefetch reads no value.
//   3. CTA r attends to the selected blocks r, r+CL, ...: TMA copies of their K and V, the
//      warp-MMA online softmax of attn_warp.cuh (32 keys per warp), a merge of the 8 warps into
//      an fp32 partial (m, l, o) per head.
//   4. CTA r merges heads r, r+CL, ...: every CTA copies its partial of a head into the owner's
//      shared memory (bulk copies, counted on the owner's barrier), and the owner writes o (bf16)
//      and lse.  Two halves of the cluster barrier order the copies after the peers' set-up and
//      after their selection (whose memory the partials reuse); there is no barrier at the end.
// No global memory is written but the outputs, and nothing is carried between launches.
#include <algorithm>
#include <mutex>
#include <vector>

#include "attn_warp.cuh"
#include "internal.h"
#include "pool.cuh"

namespace infllmv2 {

constexpr int kDcThreads = 256;   // 8 warps
constexpr int kDcKRows = 768;     // kernel rows of one scoring pass (6 TMA boxes of 128 rows)
constexpr int kDcMaxSel = 4096;   // selection capacity covered (the list lives in shared memory)
constexpr int kDcMaxPer = 16;     // keys per thread in the selection: rows of up to 4096 blocks
constexpr int kDcCand = 384;      // candidates ranked exactly after the pre-threshold
constexpr int kDcFastPer = 8;     // strided keys per thread on the fast selection path (<= 2048 blocks)
constexpr int kDcLT = 16;         // best candidates of each CTA sent to every peer (the list path)

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
// The cluster barrier in two halves, executed by every thread of every CTA (arrive, then wait, in
// turn).  The arrive is relaxed: it orders no memory access by itself (a release arrive also waited
// for this CTA's bulk copies in flight, microseconds here); the barrier initialisations it follows
// are published by their own fence, and it is only ever used to say that shared memory has been
// read (values already consumed) or that barriers exist.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Bring the 128-byte line holding p, or `bytes` from p (16-byte aligned, a multiple of 16) by the
// bulk-copy unit, into L2.  Hints: no value is read, so they may run ahead of the programmatic
// wait (L2 stays coherent with the previous kernel's writes).
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}
// Sort one 64-bit value per lane of the warp, largest first (a bitonic network over shuffles).
__device__ __forceinline__ unsigned long long warp_sort_desc64(unsigned long long v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool keep_max = ((lane & k) == 0) == ((lane & j) == 0);
            v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
        }
    return v;
}
__device__ __forceinline__ unsigned long long lds_u64(uint32_t addr) {
    unsigned long long v;
    asm("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(addr));
    return v;
}
// Number of entries greater than x in the lists l < n_lists, l != skip, of 16 values each (sorted
// largest first, 128 bytes apart from shared address `base`; all NL lists lie in shared memory):
// binary searches advanced in lockstep, every load unconditional and every step a select, so the
// NL searches are independent chains without branches (lanes of a warp differ in `skip`).
template <int NL>
__device__ __forceinline__ int count_greater_lists(uint32_t base, int n_lists, int skip, unsigned long long x) {
    int pos[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) pos[l] = 0;
#pragma unroll
    for (int step = 8; step >= 1; step >>= 1)
#pragma unroll
        for (int l = 0; l < NL; ++l) pos[l] += lds_u64(base + 128u * l + 8u * (pos[l] + step - 1)) > x ? step : 0;
    int total = 0;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
        const bool last_greater = lds_u64(base + 128u * l + 120u) > x;
        const int c = pos[l] + ((pos[l] == 15) & last_greater ? 1 : 0);
        total += (l < n_lists && l != skip) ? c : 0;
    }
    return total;
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from this CTA's shared
// memory to a cluster address (a peer's shared memory); completion is counted in bytes on the
// barrier at cluster address `bar`, in the destination CTA.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
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
    static constexpr int kMergeRow = D + D / 8;                // 8-warp merge scratch row: 4 floats of pad per 32
    static constexpr int kMerge = (8 * 16 * 2 + 8 * 16 * kMergeRow) * 4;
    static constexpr int kPRow = D + 4;                        // a head's partial: m, l, 2 unused, o[D]
    static constexpr int kPartial = 16 * kPRow * 4;            // this CTA's partials, after the merge scratch
    static constexpr int kSlots = 24 * kPRow * 4;              // partials merged here: CL x heads owned <= 24
    static_assert(kMerge % 16 == 0 && kMerge + kPartial <= kX, "merge scratch and partials fit the tile memory");
    // offsets from the 1024-aligned base: tiles | keys[nblk_max + 64] and ks[kDcKRows] (while selecting),
    // then the slots of the partials this CTA merges | sel[S_cap] | barriers
    __host__ __device__ static int off_keys() { return kX; }
    __host__ __device__ static int off_ks(int nblk_max) { return kX + ((4 * (nblk_max + 64) + 15) & ~15); }
    __host__ __device__ static int off_sel(int nblk_max) {
        const int a = off_ks(nblk_max) + 4 * kDcKRows, b = kX + kSlots;
        return a > b ? a : b;
    }
    __host__ __device__ static int off_bar(int nblk_max, int S_cap) { return (off_sel(nblk_max) + 4 * S_cap + 15) & ~15; }
    static int bytes(int nblk_max, int S_cap) { return off_bar(nblk_max, S_cap) + 8 * (kPB + 2) + 1024; }
};

template <int D, int BS, bool kAppend>
__global__ void __launch_bounds__(kDcThreads, 1)
decode_cluster_kernel(const __grid_constant__ CUtensorMap tm_kern, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* kern_rows, const __nv_bfloat16* kc,
                      const __nv_bfloat16* vc, const int* __restrict__ kv_len, int Hq, int Hkv, int G, int L_max, int M_max, Params p,
                      ClusterShape sh, int* __restrict__ idx_out, int idx_stride, int* __restrict__ counts_out,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse, float scale_log2,
                      int* __restrict__ err, const __nv_bfloat16* __restrict__ k_new,
                      const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* k_w, __nv_bfloat16* v_w,
                      __nv_bfloat16* kern_w) {
    using SM = ClusterSmem<D, BS>;
    constexpr int PB = SM::kPB;
    constexpr int kTile = SM::kTile;
    constexpr int kTilesPerBlock = BS / 32;
    constexpr int kMergeRow = SM::kMergeRow;
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint32_t* keys = reinterpret_cast<uint32_t*>(base + SM::off_keys());           // [nblk_max], filled by all CTAs
    float* ks = reinterpret_cast<float*>(base + SM::off_ks(sh.nblk_max));           // [kDcKRows]
    float* part = reinterpret_cast<float*>(base + SM::kMerge);                       // [16][kPRow], after attention
    int* sel = reinterpret_cast<int*>(base + SM::off_sel(sh.nblk_max));             // [S_cap]
    uint64_t* bar_b = reinterpret_cast<uint64_t*>(base + SM::off_bar(sh.nblk_max, sh.S_cap));  // [PB]
    uint64_t* bar_keys = bar_b + PB;      // the peers' keys have landed
    uint64_t* bar_part = bar_b + PB + 1;  // the partials of the heads merged here have landed
    constexpr int kPRow = SM::kPRow;
    __shared__ int s_wsum[2][kDcThreads / 32];
    __shared__ int s_cnt[3][4];
    __shared__ unsigned long long s_cv[kDcCand];          // candidates >= tau: key << 32 | ~block
    __shared__ int s_rk[kDcCand];                          // their ranks
    __shared__ uint32_t s_bits[kDcFastPer * kDcThreads / 32];  // chosen blocks (fast path), one bit each
    __shared__ int s_wpre[kDcFastPer * kDcThreads / 32];       // chosen blocks below each bitmap word
    __shared__ uint32_t s_mx[kDcThreads];                  // the threads' maxima of their strided keys
    __shared__ int s_byrank[kDcThreads];                   // chosen candidates' blocks by rank
    __shared__ uint32_t s_tau[2];                          // threshold, and whether k maxima are nonzero
    __shared__ int s_nc;                                   // candidates compacted so far
    __shared__ uint64_t s_bar_piece[kDcKRows / 128];       // scoring: kernel rows of piece p landed
    __shared__ __align__(16) unsigned long long s_wtop[kDcThreads / 32][kDcLT];  // each warp's best, sorted
    __shared__ __align__(16) unsigned long long s_gcand[16][kDcLT];  // CTA r's best, sorted (filled by CTA r)
    __shared__ int s_grk[16 * kDcLT];                      // their ranks in the row
    __shared__ uint64_t s_bar_cand;                        // the peers' lists have landed
    __shared__ int s_lt_fail;                              // some CTA may hold more of the top-k than it sent

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const uint32_t rank = cluster_ctarank();
    const int ncta = static_cast<int>(cluster_nctarank());
    const int row = blockIdx.x / ncta;
    const int b = row / Hkv, g = row % Hkv;
    const int c = p.kernel_size, s = p.kernel_stride;
    const int nh = static_cast<int>(rank) < G ? (G - 1 - static_cast<int>(rank)) / ncta + 1 : 0;  // heads merged here
    auto key_bytes = [&](int j) {  // keys CTA j sends: its blocks, rounded up to 16 bytes
        const int n = max(0, min(sh.nblk_max - j * sh.CB, sh.CB));
        return static_cast<uint32_t>(((n + 3) & ~3) * 4);
    };

    if (tid == 0) {
        prefetch_tmap(&tm_kern);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        for (int k = 0; k < PB; ++k) mbar_init(&bar_b[k], 1);
        for (int k = 0; k < kDcKRows / 128; ++k) mbar_init(&s_bar_piece[k], 1);
        mbar_init(bar_keys, 1);
        mbar_init(bar_part, 1);
        mbar_init(&s_bar_cand, 1);
        fence_mbar_init();
        uint32_t in_keys = 0;
        for (int j = 0; j < ncta; ++j)
            if (j != static_cast<int>(rank)) in_keys += key_bytes(j);
        mbar_arrive_expect_tx(bar_keys, in_keys);
        mbar_arrive_expect_tx(&s_bar_cand, static_cast<uint32_t>((ncta - 1) * kDcLT * 8));
        s_lt_fail = 0;
        mbar_arrive_expect_tx(bar_part, static_cast<uint32_t>(nh * ncta * kPRow * 4));
    }
    if (tid < 12) (&s_cnt[0][0])[tid] = 0;
    __syncthreads();
    // Launched with programmatic stream serialisation: the set-up above may overlap the previous
    // kernel's tail; nothing the previous kernel may write is read before this wait.
    pdl_trigger();
    {   // While the previous kernel finishes: this CTA's lines of q and of the cache length, and its
        // kernel rows of the first scoring pass for the longest cache (bulk prefetches of up to 128
        // rows, lane p of warp 1 rows 128p ...), towards L2 and into the address translations.
        const char* qb = reinterpret_cast<const char*>(q + (static_cast<size_t>(b) * Hq + static_cast<size_t>(g) * G) * D);
        if (tid < (G * D * 2 + 127) / 128) prefetch_l2_line(qb + 128 * tid);
        if (tid == kDcThreads - 1) prefetch_l2_line(kv_len + b);
        const int pa0 = static_cast<int>(rank) * sh.CB, pa1 = min(pa0 + sh.CB, sh.nblk_max);
        if (warp == 1 && pa0 < pa1) {
            const int j0 = first_kernel_of_block(pa0, BS, c, s);
            const int j1 = min(last_kernel_of_block(min(pa0 + sh.SC, pa1) - 1, BS, s), M_max - 1);
            const int r0 = j0 + 128 * lane;
            if (r0 <= j1)
                bulk_prefetch_l2(kern_rows + (static_cast<size_t>(row) * M_max + r0) * D,
                                 static_cast<uint32_t>(min(128, j1 - r0 + 1) * D * 2));
        }
    }
    pdl_wait();

    // ================= 1. scores of this CTA's blocks, pushed as keys to every CTA
    // Lane 0 of warp p issues the TMA copy of piece p (128 kernel rows) of a pass; warp w scores the
    // 32-row tiles w, w + 8, ... of the pass as their pieces land: S[head][kernel row] = Q K^T by
    // warp MMAs (the Q fragments of the attention below), then the maximum over the G heads.  (With
    // N = 16 heads a tcgen05 MMA does too little work per issue: one thread issuing the 8 MMAs of a
    // 128-row piece took longer than the piece took to land.)
    const int blkA0 = static_cast<int>(rank) * sh.CB;
    const int blkA1 = min(blkA0 + sh.CB, sh.nblk_max);
    uint32_t piece_uses = 0;  // bit p = phase parity of s_bar_piece[p] (the same in every thread)
    auto pass_rows = [&](int sub0, int& jlo, int& jend) {
        const int sub1 = min(sub0 + sh.SC, blkA1);
        jlo = first_kernel_of_block(sub0, BS, c, s);
        jend = min(last_kernel_of_block(sub1 - 1, BS, s), M_max - 1);
        return jend - jlo + 1;
    };
    // kernel rows of blocks [sub0, sub0 + SC) for the longest cache: piece p is issued by lane 0 of
    // warp p (a copy issue holds its thread; one thread issuing all of them delayed the last)
    static_assert(kDcKRows / 128 <= kDcThreads / 32, "a warp per piece");
    auto issue_pass = [&](int sub0) {
        int jlo, jend;
        const int nrows = pass_rows(sub0, jlo, jend);
        const int pc = warp;
        if (lane == 0 && pc * 128 < nrows) {
            mbar_arrive_expect_tx(&s_bar_piece[pc], (D / 64) * 128 * 128);
            for (int half = 0; half < D / 64; ++half)
                tma_load_2d(base + half * (kDcKRows * 128) + pc * (128 * 128), &tm_kern, 64 * half,
                            row * M_max + jlo + pc * 128, &s_bar_piece[pc]);
        }
    };
    if (blkA0 < blkA1) issue_pass(blkA0);
    // Q fragments: rows = heads (rows >= G read as zero), for the attention
    QFrag<D> Q;
    load_q(Q, q + (static_cast<size_t>(b) * Hq + static_cast<size_t>(g) * G) * D, D, G);
    const int L = kv_len[b];
    const bool len_ok = L >= 1 && L <= L_max && kernels_in(L, c, s) <= M_max;
    const int bt = len_ok ? (L - 1) / BS : -1;
    const bool dense = L < p.dense_len;
    auto forced = [&](int blk) { return blk < p.n_init || blk > bt - p.n_local; };
    // K and V of block blk, brought into L2 ahead of the attention's copies: lines t0, t0 + nt, ...
    // of its visible rows (K lines first, then V)
    constexpr int kLines = BS * D * 2 / 128;  // 128-byte lines of one block of K (or V)
    auto prefetch_block = [&](int blk, int t0, int nt) {
        const int n_lines = min(BS, L - blk * BS) * (D * 2 / 128);
        const size_t off = (static_cast<size_t>(row) * L_max + static_cast<size_t>(blk) * BS) * D;
        const char* kb = reinterpret_cast<const char*>(kc + off);
        const char* vb = reinterpret_cast<const char*>(vc + off);
        for (int w = t0; w < 2 * kLines; w += nt) {
            const int wl = w < kLines ? w : w - kLines;
            if (wl < n_lines) prefetch_l2_line((w < kLines ? kb : vb) + 128 * wl);
        }
    };
    if (len_ok && warp == kDcThreads / 32 - 1)  // the forced blocks are attended whatever the scores
        for (int i = 0; i < p.n_init + p.n_local; ++i) {
            const int blk = i < p.n_init ? i : bt - (i - p.n_init);
            if (blk >= 0 && blk <= bt && blk % ncta == static_cast<int>(rank)) prefetch_block(blk, lane, 32);
        }
    // Decode-step append (the kAppend instance): warp 6 holds this row's new K and V, which the CTA
    // that attends the last selected block (the query's own) writes into cache row L-1 before its
    // copies; warp 5 of every CTA pools its share of the 8-element slices of the kernel the new
    // token completes, for the steps to come.  This step's scores never need that kernel: it
    // overlaps only the query's own block and the one before, both local (forced) blocks under the
    // condition the host checks.
    uint4 k_row = make_uint4(0u, 0u, 0u, 0u), v_row = k_row;
    if constexpr (kAppend) {
      if (len_ok) {
        const int pn = L - 1;
        const uint4* kn = reinterpret_cast<const uint4*>(k_new + static_cast<size_t>(row) * D);
        if (warp == 6 && lane < D / 8) {
            k_row = ldg_v4(kn + lane);
            v_row = ldg_v4(reinterpret_cast<const uint4*>(v_new + static_cast<size_t>(row) * D) + lane);
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
    // first half of the cluster barrier: this CTA's barriers are initialised; the peers wait for it
    // before their first copy into this CTA
    cluster_arrive_relaxed();
    const uint32_t keys_base = smem_u32(keys);
    const uint32_t sK = smem_u32(base);
    for (int sub0 = blkA0; sub0 < blkA1; sub0 += sh.SC) {
        int jlo, jend;
        const int nrows = pass_rows(sub0, jlo, jend);
        const int sub1 = min(sub0 + sh.SC, blkA1);
        const bool work = len_ok && !dense && sub0 <= bt && nrows > 0;
        const int bz = min(sub1, bt + 1);  // blocks [sub0, bz) are scored
        const int jhi = work ? min(min(last_kernel_of_block(bz - 1, BS, s), kernels_in(L, c, s) - 1), jend) : -1;
        const int nj = work ? jhi - jlo + 1 : 0;  // visible kernel rows of the pass
        const int n_issued = nrows > 0 ? (nrows + 127) / 128 : 0;
        for (int t = warp; 32 * t < nj; t += kDcThreads / 32) {
            const int pc = t >> 2;  // the 128-row piece holding the tile
            if (!__all_sync(0xffffffffu, mbar_wait(&s_bar_piece[pc], (piece_uses >> pc) & 1u))) {
                if (lane == 0) raise_error(err, kDevErrTimeout);
                continue;
            }
            uint4 kw[4][D / 32];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int r = 32 * t + 8 * nt + key_perm<D>(gq);  // (the key order of attn_warp.cuh)
#pragma unroll
                for (int i = 0; i < D / 32; ++i) {
                    const int col = 32 * i + 8 * cq;
                    kw[nt][i] = lds_v4(sK + (col / 64) * (kDcKRows * 128) + swz128(r, (col % 64) / 8));
                }
            }
            float sc[4][4];
            qk_tiles<D>(sc, Q, kw);
            // column 2cq + j of n-tile nt is kernel row 32t + 8nt + key_perm<D>(2cq + j); rows gq and gq + 8
            // are heads
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float m = fmaxf(gq < G ? sc[nt][j] : -INFINITY, gq + 8 < G ? sc[nt][2 + j] : -INFINITY);
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                    const int r = 32 * t + 8 * nt + key_perm<D>(2 * cq + j);
                    if (gq == 0 && r < nj) ks[r] = m;
                }
        }
        // every issued piece has landed before its tiles are reused, scored or not
        if (tid == 0)
            for (int pc = 0; pc < n_issued; ++pc)
                if (!mbar_wait(&s_bar_piece[pc], (piece_uses >> pc) & 1u)) raise_error(err, kDevErrTimeout);
        piece_uses ^= (1u << n_issued) - 1u;
        __syncthreads();
        if (work) {
            // block score = max over its visible kernels; its selection key goes to every CTA
            for (int blk = sub0 + tid; blk < bz; blk += kDcThreads) {
                const int ja = max(first_kernel_of_block(blk, BS, c, s), jlo);
                const int jz = min(last_kernel_of_block(blk, BS, s), jhi);
                float m = -INFINITY;
                for (int jj = ja; jj <= jz; ++jj) m = fmaxf(m, ks[jj - jlo]);
                keys[blk] = forced(blk) ? 0u : ordered_key(m);  // 0: not a candidate
            }
        }
        __syncthreads();  // tiles and ks free for the next pass
        if (sub0 + sh.SC < blkA1) issue_pass(sub0 + sh.SC);
    }
    // The row's selection parameters (the same in every CTA of the cluster)
    const int n = bt + 1;
    const int a_init = min(p.n_init, max(n, 0));
    const int lo_local = max(bt - p.n_local + 1, 0);
    const int n_forced = len_ok ? a_init + (n - max(lo_local, a_init)) : 0;
    const int nc = n - n_forced;
    const bool take_all = len_ok && (dense || nc <= p.topk);
    const bool select = len_ok && !take_all && p.topk > 0;
    const int nn = max(n, 0);
    const int lo_f = max(lo_local, a_init);  // first local block not already an initial one
    // the list path (below) decides from the CTAs' lists alone; the keys travel only without it
    const bool list_path = select && sh.CB <= kDcThreads && p.topk < ncta * kDcLT &&
                           nn <= kDcFastPer * kDcThreads;  // (s_bits: 2048 blocks)
    // This CTA's best candidates: the kDcLT largest of its blocks' 64-bit values key << 32 | ~block
    // (0: not a candidate; larger = better, ties to the lower block), sorted: each warp sorts 32 of
    // them, then each of the warps' kDcLT best finds its rank among the warps' lists by binary
    // searches.  The lists of all CTAs decide the row's top-k exactly unless some CTA holds more of
    // it than it sent (checked below).
    unsigned long long* my_cand = &s_gcand[rank][0];
    if (tid < kDcLT) my_cand[tid] = 0ull;
    if (list_path) {  // (one block per thread: CB <= 256)
        const int blk = blkA0 + tid;
        unsigned long long v = 0ull;
        if (len_ok && !dense && blk < blkA1 && blk <= bt && !forced(blk)) {
            const uint32_t kk = keys[blk];
            if (kk != 0u) v = (static_cast<unsigned long long>(kk) << 32) | static_cast<uint32_t>(~blk);
        }
        v = warp_sort_desc64(v);
        if (lane < kDcLT) s_wtop[warp][lane] = v;
    }
    __syncthreads();
    if (list_path && tid < (kDcThreads / 32) * kDcLT) {
        const int w0 = tid / kDcLT;
        const unsigned long long x = s_wtop[w0][tid % kDcLT];
        const int r = tid % kDcLT + count_greater_lists<kDcThreads / 32>(smem_u32(&s_wtop[0][0]), kDcThreads / 32, w0, x);
        if (x != 0ull && r < kDcLT) my_cand[r] = x;
    }
    // this CTA's list (and, without the list path, its keys) -> every peer: bulk copies into the
    // same offsets of the peers' shared memory, counted on their barriers
    fence_proxy_async_shared();
    __syncthreads();
    cluster_wait();
    auto send_keys = [&]() {  // by warp 0: lane j copies to peer j
        const uint32_t nb = key_bytes(static_cast<int>(rank));
        if (nb > 0 && lane < ncta && lane != static_cast<int>(rank))
            bulk_copy_to_peer(dsmem_addr(keys_base + 4u * blkA0, lane), keys_base + 4u * blkA0, nb,
                              dsmem_addr(smem_u32(bar_keys), lane));
    };
    if (warp == 0) {
        if (lane < ncta && lane != static_cast<int>(rank))
            bulk_copy_to_peer(dsmem_addr(smem_u32(my_cand), lane), smem_u32(my_cand), kDcLT * 8,
                              dsmem_addr(smem_u32(&s_bar_cand), lane));
        if (!list_path) send_keys();
        bulk_commit();
    }
    bool keys_sent = !list_path, keys_in = false, cand_in = false;  // (uniform over the cluster)
    auto wait_keys = [&]() {
        if (keys_sent && !keys_in && !mbar_wait(bar_keys, 0) && tid == 0) raise_error(err, kDevErrTimeout);
        keys_in = true;
    };
    auto wait_cand = [&]() {
        if (!cand_in && !mbar_wait(&s_bar_cand, 0) && tid == 0) raise_error(err, kDevErrTimeout);
        cand_in = true;
    };

    // ================= 2. the row's selection, computed by every CTA from all the keys
    int count = 0;
    // fast path: the attention's list is init blocks [0, r_ainit) | s_byrank[0, r_k) | local blocks
    // from r_lof; otherwise sel[] in block order
    bool by_rank = false;
    int r_ainit = 0, r_lof = 0, r_k = 0, r_nc = 0, r_nn = 0;
    const unsigned long long* r_cv = s_cv;  // the ranked candidates (value, rank) of the fast paths
    const int* r_rk = s_rk;
    auto list_blk = [&](int e) {
        if (!by_rank) return sel[e];
        if (e < r_ainit) return e;
        if (e < r_ainit + r_k) return s_byrank[e - r_ainit];
        return r_lof + (e - r_ainit - r_k);
    };
    {
        int total = 0;
        bool done = false;
        if (list_path) {
            // List path.  While the lists travel, this CTA's likely share of the chosen blocks (its
            // best ceil(k * blocks here / blocks) candidates) goes towards L2 ahead of the attention's
            // copies.  Then every candidate of the lists finds its rank in the row by binary
            // searches in the other lists; ranks below k are the chosen ones.  A CTA that sent a full
            // list whose last entry is chosen may hold more chosen blocks than it sent: then the
            // threshold path below decides from all the keys instead (sent now, by every CTA).
            const int k = p.topk;
            const int mine = max(0, min(blkA1, nn) - blkA0);
            const int n_pf = min(kDcLT, (k * mine + nn - 1) / max(nn, 1));
            if (tid >= 32 && tid < 32 + 2 * n_pf) {
                const unsigned long long x = my_cand[(tid - 32) >> 1];
                if (x != 0ull) {
                    const int blk = static_cast<int>(~static_cast<uint32_t>(x));
                    const size_t off = (static_cast<size_t>(row) * L_max + static_cast<size_t>(blk) * BS) * D;
                    bulk_prefetch_l2((tid & 1) ? vc + off : kc + off, static_cast<uint32_t>(min(BS, L - blk * BS) * D * 2));
                }
            }
            wait_cand();
            const int n_all = ncta * kDcLT;
            if (tid < n_all) {
                const int r0 = tid / kDcLT, p0 = tid % kDcLT;
                const unsigned long long x = s_gcand[r0][p0];
                int rk = 0x7fffffff;
                if (x != 0ull) {
                    rk = p0 + count_greater_lists<16>(smem_u32(&s_gcand[0][0]), ncta, r0, x);
                    if (rk < k) {
                        s_byrank[rk] = static_cast<int>(~static_cast<uint32_t>(x));
                        if (p0 == kDcLT - 1) s_lt_fail = 1;
                    }
                }
                s_grk[tid] = rk;
            }
            for (int i3 = tid; i3 < kDcFastPer * kDcThreads / 32; i3 += kDcThreads) s_bits[i3] = 0u;
            __syncthreads();
            if (s_lt_fail == 0) {
                total = a_init + k + (nn - lo_f);
                done = true;
                by_rank = true;
                r_ainit = a_init;
                r_lof = lo_f;
                r_k = k;
                r_nc = n_all;
                r_cv = &s_gcand[0][0];
                r_rk = s_grk;
                r_nn = nn;
            } else {
                if (warp == 0) {
                    send_keys();
                    bulk_commit();
                }
                keys_sent = true;
            }
        }
        if (!done && select && nn <= kDcFastPer * kDcThreads && p.topk <= kDcThreads) {
            wait_keys();
            // Fast path.  tau = the k-th largest of the threads' maxima over the strided keys
            // t, t + 256, ... (neighbouring blocks have correlated scores: a stride spreads each
            // thread over the row), found bit by bit by one warp.  At least k keys are >= tau and,
            // unless the scores are heavily tied, only a few more; those candidates are ranked
            // exactly (key descending, block ascending, one 64-bit compare).  The attention takes
            // the list init blocks | chosen candidates by rank | local blocks; the block-order
            // list is built only when the caller asks for it.
            const int k = p.topk;
            uint32_t kv[kDcFastPer];
            uint32_t mx = 0u;
#pragma unroll
            for (int u = 0; u < kDcFastPer; ++u) {
                const int i = tid + u * kDcThreads;
                kv[u] = i < nn ? keys[i] : 0u;
                mx = max(mx, kv[u]);
            }
            s_mx[tid] = mx;
            if (tid == 0) s_nc = 0;
            __syncthreads();
            if (warp == 0) {
                uint32_t m8[kDcThreads / 32];
                uint32_t nz = 0u, k_and = ~0u, k_or = 0u;
#pragma unroll
                for (int j = 0; j < kDcThreads / 32; ++j) {
                    m8[j] = s_mx[lane + 32 * j];
                    if (m8[j] != 0u) {
                        ++nz;
                        k_and &= m8[j];
                    }
                    k_or |= m8[j];
                }
                nz = __reduce_add_sync(0xffffffffu, nz);
                k_and = __reduce_and_sync(0xffffffffu, k_and);
                k_or = __reduce_or_sync(0xffffffffu, k_or);
                uint32_t tau = 0u;
                if (nz >= static_cast<uint32_t>(k)) {
                    const uint32_t diff = k_and ^ k_or;
                    int bit = diff == 0u ? -1 : 31 - __clz(diff);
                    tau = bit >= 31 ? 0u : (k_and & (~0u << (bit + 1)));
                    for (; bit >= 0; --bit) {
                        const uint32_t trial = tau | (1u << bit);
                        uint32_t cnt = 0u;
#pragma unroll
                        for (int j = 0; j < kDcThreads / 32; ++j) cnt += m8[j] >= trial ? 1u : 0u;
                        cnt = __reduce_add_sync(0xffffffffu, cnt);
                        if (cnt >= static_cast<uint32_t>(k)) tau = trial;
                        if (cnt == static_cast<uint32_t>(k)) break;
                    }
                }
                if (lane == 0) {
                    s_tau[0] = tau;
                    s_tau[1] = nz >= static_cast<uint32_t>(k) ? 1u : 0u;
                }
            }
            __syncthreads();
            const uint32_t tau = s_tau[0];
            if (s_tau[1] != 0u) {
                // candidates -> s_cv, compacted by one shared counter (warp-aggregated); their order
                // is arbitrary, their ranks are not
                int nc_t = 0;
#pragma unroll
                for (int u = 0; u < kDcFastPer; ++u) nc_t += (kv[u] != 0u && kv[u] >= tau) ? 1 : 0;
                int incl = nc_t;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int x = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += x;
                }
                int wbase = 0;
                if (lane == 31 && incl > 0) wbase = atomicAdd(&s_nc, incl);
                int pos = __shfl_sync(0xffffffffu, wbase, 31) + incl - nc_t;
#pragma unroll
                for (int u = 0; u < kDcFastPer; ++u)
                    if (kv[u] != 0u && kv[u] >= tau) {
                        if (pos < kDcCand)
                            s_cv[pos] = (static_cast<unsigned long long>(kv[u]) << 32) |
                                        static_cast<uint32_t>(~(tid + u * kDcThreads));
                        ++pos;
                    }
                __syncthreads();
                const int c_total = s_nc;
                if (c_total <= k + k / 2 && tid < 2 * ((c_total - static_cast<int>(rank) + ncta - 1) / ncta)) {
                    // few candidates beyond the k to be chosen: K (even threads) and V of candidates
                    // rank, rank + CL, ... go towards L2 while they are ranked
                    const int blk = static_cast<int>(~static_cast<uint32_t>(s_cv[static_cast<int>(rank) + ncta * (tid >> 1)]));
                    const size_t off = (static_cast<size_t>(row) * L_max + static_cast<size_t>(blk) * BS) * D;
                    bulk_prefetch_l2((tid & 1) ? vc + off : kc + off, static_cast<uint32_t>(min(BS, L - blk * BS) * D * 2));
                }
                if (c_total <= kDcCand) {
                    // rank of candidate i = number of better candidates; sp (a power of two) threads
                    // of one warp share each candidate and add their counts by shuffles
                    const int sp = c_total <= kDcThreads / 4 ? 4 : c_total <= kDcThreads / 2 ? 2 : 1;
                    const int seg = (c_total + sp - 1) / sp;
                    const int i = tid / sp, part = tid % sp;
                    int rnk = 0;
                    unsigned long long vi = 0ull;
                    if (i < c_total) {
                        vi = s_cv[i];
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
                        rnk = r0 + r1 + r2 + r3;
                    }
                    for (int off = 1; off < sp; off <<= 1) rnk += __shfl_xor_sync(0xffffffffu, rnk, off);
                    if (part == 0 && i < c_total) {
                        s_rk[i] = rnk;
                        if (rnk < k) s_byrank[rnk] = static_cast<int>(~static_cast<uint32_t>(vi));
                    }
                    for (int i2 = kDcThreads + tid; i2 < c_total; i2 += kDcThreads) {  // c_total > 256
                        const unsigned long long v2 = s_cv[i2];
                        int r2 = 0;
                        for (int j = 0; j < c_total; ++j) r2 += s_cv[j] > v2 ? 1 : 0;
                        s_rk[i2] = r2;
                        if (r2 < k) s_byrank[r2] = static_cast<int>(~static_cast<uint32_t>(v2));
                    }
                    for (int i3 = tid; i3 < kDcFastPer * kDcThreads / 32; i3 += kDcThreads) s_bits[i3] = 0u;
                    __syncthreads();
                    total = a_init + k + (nn - lo_f);
                    done = true;
                    by_rank = true;
                    r_ainit = a_init;
                    r_lof = lo_f;
                    r_k = k;
                    r_nc = c_total;
                    r_nn = nn;
                }
            }
            __syncthreads();
        }
        if (!done) {
            wait_keys();
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
        if constexpr (kAppend) {
            // the new K/V row, by the CTA that attends the last selected block, ahead of its copies
            if (len_ok && count > 0 && static_cast<int>(rank) == (count - 1) % ncta && warp == 6 && lane < D / 8) {
                const size_t wr = (static_cast<size_t>(row) * L_max + (L - 1)) * D;
                reinterpret_cast<uint4*>(k_w + wr)[lane] = k_row;
                reinterpret_cast<uint4*>(v_w + wr)[lane] = v_row;
                fence_proxy_async_global();
            }
        }
        __syncthreads();  // sel complete
        if (rank == 0) {
            if (tid == 0 && (total > sh.S_cap || !len_ok)) raise_error(err, kDevErrIndex);
            if (idx_out != nullptr && !by_rank) {  // (fast path: written by the last CTA behind its copies)
                int* out = idx_out + static_cast<size_t>(row) * idx_stride;
                for (int i = tid; i < idx_stride; i += kDcThreads) out[i] = i < count ? sel[i] : -1;
                if (tid == 0) counts_out[row] = count;
            }
        }
    }
    // The block lists of the fast path, by the last CTA (which attends the fewest blocks) while its
    // attention copies are in flight: the chosen candidates in block order by a bitmap, word prefix
    // popcounts (one warp) and one popcount per candidate, framed by the initial and local blocks.
    bool lists_pending = by_rank && static_cast<int>(rank) == ncta - 1 && idx_out != nullptr;
    auto write_lists = [&]() {
        for (int i = tid; i < r_nc; i += kDcThreads)
            if (r_rk[i] < r_k) {
                const uint32_t blk = ~static_cast<uint32_t>(r_cv[i]);
                atomicOr(&s_bits[blk >> 5], 1u << (blk & 31));
            }
        __syncthreads();
        if (warp == 0) {
            const int c0 = __popc(s_bits[2 * lane]), c1 = __popc(s_bits[2 * lane + 1]);
            int wi = c0 + c1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += x;
            }
            s_wpre[2 * lane] = wi - c0 - c1;
            s_wpre[2 * lane + 1] = wi - c1;
        }
        __syncthreads();
        int* out = idx_out + static_cast<size_t>(row) * idx_stride;
        for (int i = tid; i < r_nc; i += kDcThreads)
            if (r_rk[i] < r_k) {
                const uint32_t blk = ~static_cast<uint32_t>(r_cv[i]);
                const int at = r_ainit + s_wpre[blk >> 5] + __popc(s_bits[blk >> 5] & ((1u << (blk & 31)) - 1u));
                if (at < count) out[at] = static_cast<int>(blk);
            }
        for (int i = tid; i < idx_stride; i += kDcThreads) {
            if (i >= count) out[i] = -1;
            else if (i < r_ainit) out[i] = i;
            else if (i >= r_ainit + r_k) out[i] = r_lof + (i - r_ainit - r_k);
        }
        if (tid == 0) counts_out[row] = count;
        lists_pending = false;
    };
    // second half-barrier: this CTA no longer reads its keys or scores (and its copies of its keys
    // have been read), whose memory takes the peers' partials after the attention
    // (and every peer's copies into this CTA's keys and lists have landed)
    wait_keys();
    wait_cand();
    if (warp == 0) bulk_wait_read_all();
    cluster_arrive_relaxed();

    // ================= 3. attention over the selected blocks rank, rank + CL, ...
    WarpAcc<D> A;
    acc_init(A);
    {
        const int mine = count > static_cast<int>(rank) ? (count - static_cast<int>(rank) + ncta - 1) / ncta : 0;
        auto blk_at = [&](int t) { return list_blk(static_cast<int>(rank) + ncta * t); };
        uint32_t ph_b = 0;
        for (int t0 = 0; t0 < mine; t0 += PB) {
            if (lane == 0 && warp < PB) {  // slot k by warp k
                const int k = warp;
                const int t = t0 + k;
                const int blk = t < mine ? blk_at(t) : -1;
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
            __syncthreads();
            if (lists_pending) write_lists();
            for (int tile = warp; tile < PB * kTilesPerBlock; tile += kDcThreads / 32) {
                const int k = tile / kTilesPerBlock;
                const int t = t0 + k;
                if (t >= mine) continue;
                const int blk = blk_at(t);
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
    if (lists_pending) write_lists();  // (a CTA without blocks to attend)
    acc_finish_rowsum(A);
    {
        // merge the 8 warps (scratch in the tile memory) into this CTA's partial
        float* sm_m = reinterpret_cast<float*>(base);
        float* sm_l = sm_m + 8 * 16;
        float* sm_o = sm_l + 8 * 16;  // [8][16][kMergeRow]
        if (cq == 0) {
            sm_m[warp * 16 + gq] = A.m[0];
            sm_m[warp * 16 + gq + 8] = A.m[1];
            sm_l[warp * 16 + gq] = A.l[0];
            sm_l[warp * 16 + gq + 8] = A.l[1];
        }
        // column c of a row is stored at c + 4 (c / 32).  A lane's n-tiles nt .. nt + 3 of one
        // accumulator slot are 4 consecutive columns (the layout of attn_warp.cuh), stored as one
        // 16-byte word; the 4 lanes of a quad land in different 16-byte bank groups.
        auto mpad = [](int col) { return col + 4 * (col >> 5); };
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int nt = 0; nt < D / 8; nt += 4) {
                const int col = o_col(D, cq, nt, e);
                *reinterpret_cast<float4*>(&sm_o[(warp * 16 + gq + 8 * (e >> 1)) * kMergeRow + mpad(col)]) =
                    make_float4(A.o[nt][e], A.o[nt + 1][e], A.o[nt + 2][e], A.o[nt + 3][e]);
            }
        __syncthreads();
        // thread t: row t / 16 (a head), columns 8 (t % 16) .. +7 per pass; each thread forms the
        // row's warp weights itself
        constexpr int kCols = 8, kTpr = D / kCols;  // threads per row
        for (int e0 = tid * kCols; e0 < 16 * D; e0 += kDcThreads * kCols) {
            const int r = e0 / D, col0 = e0 % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 8; ++w) M = fmaxf(M, sm_m[w * 16 + r]);
            const float ref = M == -INFINITY ? 0.f : M;
            float f[8], l = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                f[w] = fast_exp2(sm_m[w * 16 + r] - ref);
                l += sm_l[w * 16 + r] * f[w];
            }
            if ((tid % kTpr) == 0) {
                part[r * kPRow] = M;
                part[r * kPRow + 1] = l;
            }
            float acc[kCols];
#pragma unroll
            for (int i = 0; i < kCols; ++i) acc[i] = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w)
#pragma unroll
                for (int i = 0; i < kCols; i += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(&sm_o[(w * 16 + r) * kMergeRow + mpad(col0 + i)]);
                    acc[i] += x.x * f[w];
                    acc[i + 1] += x.y * f[w];
                    acc[i + 2] += x.z * f[w];
                    acc[i + 3] += x.w * f[w];
                }
#pragma unroll
            for (int i = 0; i < kCols; i += 4)
                *reinterpret_cast<float4*>(&part[r * kPRow + 4 + col0 + i]) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
        }
    }
    // ================= 4. merge of the CTAs' partials: CTA r merges heads r, r + CL, ...
    // Every CTA copies its partial of head h into slot (h / CL, its rank) of CTA h % CL, once the
    // peers are past their selection (their key memory holds the slots).
    const uint32_t slots = keys_base;  // [nh][CL][kPRow] fp32
    fence_proxy_async_shared();
    __syncthreads();
    cluster_wait();
    if (warp == 0) {  // lane h copies head h
        const int h = lane;
        if (h < G) {
            const int owner = h % ncta, hl = h / ncta;
            const uint32_t dst = slots + 4u * static_cast<uint32_t>((hl * ncta + static_cast<int>(rank)) * kPRow);
            bulk_copy_to_peer(dsmem_addr(dst, owner), smem_u32(part + h * kPRow), kPRow * 4,
                              dsmem_addr(smem_u32(bar_part), owner));
        }
        bulk_commit();
    }
    if (!mbar_wait(bar_part, 0) && tid == 0) raise_error(err, kDevErrTimeout);
    const float* sl = reinterpret_cast<const float*>(keys);
    for (int e = tid; e < nh * D; e += kDcThreads) {
        const int hl = e / D, d = e % D, h = static_cast<int>(rank) + ncta * hl;
        const float* ph = sl + hl * ncta * kPRow;
        float m[16], l[16], v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            m[j] = j < ncta ? ph[j * kPRow] : -INFINITY;
            l[j] = j < ncta ? ph[j * kPRow + 1] : 0.f;
            v[j] = j < ncta ? ph[j * kPRow + 4 + d] : 0.f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int j = 0; j < 16; ++j) M = fmaxf(M, m[j]);
        const float ref = M == -INFINITY ? 0.f : M;
        float Ls = 0.f, acc = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float f = j < ncta ? fast_exp2(m[j] - ref) : 0.f;
            Ls += l[j] * f;
            acc += v[j] * f;
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        o[(static_cast<size_t>(b) * Hq + g * G + h) * D + d] = __float2bfloat16_rn(acc * inv);
        if (lse != nullptr && d == 0)
            lse[static_cast<size_t>(b) * Hq + g * G + h] = Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994530942f : -INFINITY;
    }
    // this CTA's copies have read its partials before it exits
    if (warp == 0) bulk_wait_read_all();
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
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    // The kernel's attributes and the cluster size for (kernel, device, rows, shared memory) are
    // settled once (the function-attribute and occupancy queries cost host time on every call);
    // the dynamic shared-memory limit only ever grows, so earlier choices stay launchable.
    struct Choice {
        const void* fn;
        int dev, rows, smem, CL;
    };
    static std::mutex mtx;
    static std::vector<Choice> choices;
    static std::vector<Choice> smem_set;  // per (kernel, device): the largest limit set (in .smem)
    CUtensorMap tkern, tk, tv;
    const uint64_t krows = static_cast<uint64_t>(a.B) * a.Hkv * M_max;
    const uint64_t cache_rows = static_cast<uint64_t>(a.B) * a.Hkv * a.L_max;
    if (!make_tmap_bf16_2d(&tkern, kernel_cache, D, krows, 64, 128) ||
        !make_tmap_bf16_2d(&tk, a.k_cache, D, cache_rows, 64, BS) ||
        !make_tmap_bf16_2d(&tv, a.v_cache, D, cache_rows, 64, BS))
        return cudaErrorNotSupported;
    const int G = a.Hq / a.Hkv;
    const float scale_log2 = a.p.scale * 1.4426950408889634f;
    const void* fn = reinterpret_cast<const void*>(kfn);
    // a launch from a remembered choice that fails (the device was reset and the attributes with
    // it) settles the choice afresh and launches once more
    for (int attempt = 0; attempt < 2; ++attempt) {
        int CL = 0;
        bool remembered = false;
        {
            std::lock_guard<std::mutex> lock(mtx);
            if (attempt > 0) {
                auto drop = [&](std::vector<Choice>& v) {
                    v.erase(std::remove_if(v.begin(), v.end(),
                                           [&](const Choice& ch) { return ch.fn == fn && ch.dev == dev; }),
                            v.end());
                };
                drop(choices);
                drop(smem_set);
            }
            for (const Choice& ch : choices)
                if (ch.fn == fn && ch.dev == dev && ch.rows == rows && ch.smem == smem) CL = ch.CL;
            remembered = CL != 0;
            if (CL == 0) {
                cudaFuncAttributes fa{};
                if (cudaError_t e = cudaFuncGetAttributes(&fa, kfn); e != cudaSuccess) return e;
                if (smem + static_cast<int>(fa.sharedSizeBytes) > 227 * 1024) return cudaErrorNotSupported;
                Choice* lim = nullptr;
                for (Choice& ch : smem_set)
                    if (ch.fn == fn && ch.dev == dev) lim = &ch;
                if (lim == nullptr || lim->smem < smem) {
                    if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                        e != cudaSuccess)
                        return e;
                    if (lim == nullptr)
                        smem_set.push_back(Choice{fn, dev, 0, smem, 0});
                    else
                        lim->smem = smem;
                }
                if (cudaFuncSetAttribute(kfn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
                    (void)cudaGetLastError();  // then only the portable sizes (<= 8) are offered below
                // cluster size: the largest whose clusters all fit on the device at once (one wave
                // of rows); if none does, the one that keeps the most SMs busy.  Every size from 16
                // down is tried whose partial slots fit (the heads a CTA merges x CL <= 24): the
                // clusters must fit in the GPU's processing clusters, so which sizes fit depends on
                // the row count (8 rows: 12; 16 rows: 9 on a GB300).
                cfg.numAttrs = 1;  // (the search without the serialisation attribute)
                int best_sms = 0, fallback = 0;
                for (int cand = 16; cand >= 2; --cand) {
                    if (((16 + cand - 1) / cand) * cand * SM::kPRow * 4 > SM::kSlots) continue;
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
                if (CL > 0) choices.push_back(Choice{fn, dev, rows, smem, CL});
            }
        }
        if (CL == 0 || ((16 + CL - 1) / CL) * CL * SM::kPRow * 4 > SM::kSlots) return cudaErrorNotSupported;
        sh.CB = ((sh.nblk_max + CL - 1) / CL + 3) & ~3;  // a multiple of 4: each CTA's keys are 16-byte copies
        attr[0].val.clusterDim.x = CL;
        cfg.gridDim = dim3(rows * CL);
        cfg.numAttrs = 2;  // + programmatic stream serialisation: set-up overlaps the previous kernel
        const cudaError_t e = cudaLaunchKernelEx(
            &cfg, kfn, tkern, tk, tv, static_cast<const __nv_bfloat16*>(a.q),
            static_cast<const __nv_bfloat16*>(kernel_cache), static_cast<const __nv_bfloat16*>(a.k_cache),
            static_cast<const __nv_bfloat16*>(a.v_cache), a.kv_len, a.Hq, a.Hkv, G, a.L_max, M_max, a.p, sh, idx_out,
            idx_stride, counts_out, static_cast<__nv_bfloat16*>(a.o), a.lse, scale_log2, a.err,
            static_cast<const __nv_bfloat16*>(a.k_new), static_cast<const __nv_bfloat16*>(a.v_new),
            static_cast<__nv_bfloat16*>(a.k_w), static_cast<__nv_bfloat16*>(a.v_w), static_cast<__nv_bfloat16*>(a.kern_w));
        if (e == cudaSuccess || !remembered) return e;
        (void)cudaGetLastError();
    }
    return cudaErrorNotSupported;
}

bool decode_cluster_supported(const DecodeArgs& a, int M_max) {
    const int G = a.Hkv > 0 ? a.Hq / a.Hkv : 0;
    const int bs = a.p.block_size;
    if (a.tree_mask != nullptr || a.n_draft != 1) return false;
    if (G < 1 || G > 16 || (a.d != 64 && a.d != 128) || (bs != 64 && bs != 128)) return false;
    // the tensor maps' boxes must fit the tensors
    if (static_cast<long long>(a.B) * a.Hkv * M_max < 128 || static_cast<long long>(a.B) * a.Hkv * a.L_max < bs)
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
