// select.cu -- block scoring and top-k block selection
// ("MiniCPM4: 如何在手机电脑上高效运行大语言模型", section 1.1 "InfLLM v2": dynamic selection of
// the top-K relevant blocks through semantic kernels, with the opening and sliding-window
// tokens always kept; "MiniCPM40极速狂飙端侧模型的比赛结束了", section "InfLLM v2：重新定义
// 注意力机制": dense attention below 8192 tokens).
//
// score_kernel: S[b,g,t,blk] = max over the heads of group g and over the kernels that share
//   a token with blk and end at or before the query's position, of q.kernel (unscaled: the
//   scale does not change the ranking).  The dot products run on the tensor cores as warp
//   MMAs (m16n8k16, bf16 in, fp32 accumulate): one MMA row per (token, head), 16 rows =
//   16/G tokens x G heads, so the head max is a shuffle across the rows of a token.  The
//   head dimension is permuted identically for Q and the kernels (a dot product does not
//   depend on the order of its terms), which lets every lane fetch its operands with one
//   128-bit load per 32 elements straight from global memory, fully coalesced.
// score_decode_kernel: the same scores for few queries (decode, trees): one token per CTA,
//   the chunk's semantic kernels arrive in shared memory by one TMA tensor copy.
// topk_kernel: one CTA per (b, g, t).  A radix select over the order-preserving 32-bit image
//   of the fp32 scores finds the k-th largest score; blocks tied with it are taken in
//   ascending id order, so "score descending, lower id first" holds exactly.  The chosen and
//   forced blocks are compacted in ascending id order with warp ballots.
#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace infllmv2 {

template <int D, int WARPS, int MT>
__global__ void __launch_bounds__(WARPS * 32)
score_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kern,
             const int* __restrict__ kv_len, SeqMap sm, int Hq, int Hkv, int G, int L_max,
             int M_max, int nblk_max, int tree, Params p, int blocks_per_cta, int kmax,
             float* __restrict__ S, int* __restrict__ err) {
    constexpr int NKS = WARPS / MT;  // warps sharing one m-tile split its kernels
    extern __shared__ float ks[];    // [tokens_per_cta][kmax] max over heads, per kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int bg = blockIdx.z;
    const int b = bg / Hkv, g = bg % Hkv;
    const int tpm = 16 / G;             // tokens per m-tile
    const int tpc = MT * tpm;           // tokens per CTA
    const int t0 = blockIdx.y * tpc;
    const int bs = p.block_size, c = p.kernel_size, s = p.kernel_stride;

    const int L = kv_len[b];
    const int Tq = sm.len(b), tok = sm.tok0(b);  // this sequence's queries: token rows tok .. tok + Tq - 1
    const bool bad_len = Tq < 0 || Tq > sm.Tq || (Tq > 0 && (tree ? (L < 1 || L > L_max) : (L < Tq || L > L_max)));
    if (bad_len || (Tq > 0 && kernels_in(L, c, s) > M_max)) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(err, kDevErrIndex);
        return;
    }
    if (t0 >= Tq) return;
    if (L < p.dense_len) return;  // dense sequence: every block is selected, no scores needed
    const int t_last = min(t0 + tpc, Tq) - 1;
    const int pos_max = tree ? L - 1 : L - Tq + t_last;
    const int bt_max = pos_max / bs;
    const int blk0 = blockIdx.x * blocks_per_cta;
    if (blk0 > bt_max) return;
    const int blk1 = min(blk0 + blocks_per_cta, bt_max + 1);
    const int jlo = first_kernel_of_block(blk0, bs, c, s);
    const int jhi = min(last_kernel_of_block(blk1 - 1, bs, s), kernels_in(pos_max + 1, c, s) - 1);
    const int nj = jhi - jlo + 1;

    // ---- Q fragments of this warp's m-tile (rows: token r/G, head r%G)
    const int mt = warp % MT;
    const int kslice = warp / MT;
    uint32_t a[D / 16][4];
    int tok_r[2], pos_r[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = gq + 8 * half;
        const int tl = mt * tpm + r / G;
        const int t = t0 + tl;
        tok_r[half] = tl;
        pos_r[half] = tree ? L - 1 : L - Tq + t;
        const bool ok = t < Tq;
        const __nv_bfloat16* qrow = q + ((static_cast<size_t>(tok) + (ok ? t : 0)) * Hq + g * G + r % G) * D;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            uint4 w = ok ? ldg_v4(qrow + 32 * i + 8 * cq) : make_uint4(0, 0, 0, 0);
            a[2 * i][half] = w.x;
            a[2 * i][2 + half] = w.y;
            a[2 * i + 1][half] = w.z;
            a[2 * i + 1][2 + half] = w.w;
        }
    }

    // ---- kernels in n-tiles of 8; this warp takes every NKS-th n-tile
    const __nv_bfloat16* kbase = kern + static_cast<size_t>(bg) * M_max * D;
    const int n_tiles = nj > 0 ? (nj + 7) / 8 : 0;
    for (int nt = kslice; nt < n_tiles; nt += NKS) {
        const int jb = jlo + nt * 8;
        const int jrow = min(jb + gq, jhi);
        const __nv_bfloat16* krow = kbase + static_cast<size_t>(jrow) * D + 8 * cq;
        uint4 w[D / 32];
#pragma unroll
        for (int i = 0; i < D / 32; ++i) w[i] = ldg_v4(krow + 32 * i);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            mma_16816(acc, a[2 * i], w[i].x, w[i].y);
            mma_16816(acc, a[2 * i + 1], w[i].z, w[i].w);
        }
        // visibility: kernel jj counts for a query at pos iff it ends at or before pos
        const int j0 = jb + 2 * cq;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int jj = j0 + (e & 1);
            const int pr = pos_r[e >> 1];
            if (jj > jhi || jj * s + c - 1 > pr) acc[e] = -INFINITY;
        }
        // max over the heads of each token
        if (G == 16) {
            float v0 = fmaxf(acc[0], acc[2]), v1 = fmaxf(acc[1], acc[3]);
#pragma unroll
            for (int m = 4; m < 32; m <<= 1) {
                v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, m));
                v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, m));
            }
            if (gq == 0) {
                float* dst = ks + tok_r[0] * kmax + (j0 - jlo);
                if (j0 <= jhi) dst[0] = v0;
                if (j0 + 1 <= jhi) dst[1] = v1;
            }
        } else {
            for (int m = 4; m < 4 * G; m <<= 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = fmaxf(acc[e], __shfl_xor_sync(0xffffffffu, acc[e], m));
            }
            if (gq % G == 0) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float* dst = ks + tok_r[half] * kmax + (j0 - jlo);
                    if (j0 <= jhi) dst[0] = acc[2 * half];
                    if (j0 + 1 <= jhi) dst[1] = acc[2 * half + 1];
                }
            }
        }
    }
    __syncthreads();

    // ---- block max over overlapping kernels
    const int nb = blk1 - blk0;
    for (int e = threadIdx.x; e < tpc * nb; e += WARPS * 32) {
        const int tl = e / nb;
        const int blk = blk0 + e % nb;
        const int t = t0 + tl;
        if (t >= Tq) continue;
        const int pos = tree ? L - 1 : L - Tq + t;
        if (blk > pos / bs) continue;
        const int ja = max(first_kernel_of_block(blk, bs, c, s), jlo);
        const int jz = min(last_kernel_of_block(blk, bs, s), jhi);
        float m = -INFINITY;
        for (int jj = ja; jj <= jz; ++jj) m = fmaxf(m, ks[tl * kmax + (jj - jlo)]);
        S[sm.sel(b, g, Hkv, t) * nblk_max + blk] = m;
    }
}



// Rows of the kernel-cache box a decode scoring CTA loads (>= kernels of one chunk).
constexpr int kScoreBoxRows = 136;

// Decode-shaped scoring: one query token (G <= 16 heads, one MMA m-tile) per CTA and a chunk of
// blocks.  Thread 0 issues one TMA tensor copy per 64 head-dim columns of the chunk's kernel
// rows (<= 136 x 256 B) into 128-byte-swizzled shared memory, so every CTA's whole chunk is in
// flight at once; warps then read their B fragments from shared memory without bank conflicts.
template <int D>
__global__ void __launch_bounds__(128)
score_decode_kernel(const __grid_constant__ CUtensorMap tm_kern, const __nv_bfloat16* __restrict__ q,
                    const int* __restrict__ kv_len, SeqMap sm, int Hq, int Hkv, int G, int L_max, int M_max,
                    int nblk_max, int tree, Params p, int blocks_per_cta, float* __restrict__ S,
                    int* __restrict__ err) {
    constexpr int kBox = kScoreBoxRows * 128;  // bytes of one 64-column box
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    float* ks = reinterpret_cast<float*>(base + (D / 64) * kBox);  // [kScoreBoxRows] head max per kernel
    uint64_t* bar = reinterpret_cast<uint64_t*>(ks + kScoreBoxRows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int t = blockIdx.y;
    const int bg = blockIdx.z;
    const int b = bg / Hkv, g = bg % Hkv;
    const int bs = p.block_size, c = p.kernel_size, s = p.kernel_stride;
    pdl_trigger();
    const int L = kv_len[b];
    const int Tq = sm.len(b), tok = sm.tok0(b);
    const bool bad_len = Tq < 0 || Tq > sm.Tq || (Tq > 0 && (tree ? (L < 1 || L > L_max) : (L < Tq || L > L_max)));
    if (bad_len || (Tq > 0 && kernels_in(L, c, s) > M_max)) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && t == 0) raise_error(err, kDevErrIndex);
        return;
    }
    if (t >= Tq) return;
    if (L < p.dense_len) return;
    const int pos = tree ? L - 1 : L - Tq + t;
    const int bt = pos / bs;
    const int blk0 = blockIdx.x * blocks_per_cta;
    if (blk0 > bt) return;
    const int blk1 = min(blk0 + blocks_per_cta, bt + 1);
    const int jlo = first_kernel_of_block(blk0, bs, c, s);
    const int jhi = min(last_kernel_of_block(blk1 - 1, bs, s), kernels_in(pos + 1, c, s) - 1);
    const int nj = jhi - jlo + 1;
    const int n_tiles = nj > 0 ? (nj + 7) / 8 : 0;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        if (n_tiles > 0) {
            mbar_arrive_expect_tx(bar, (D / 64) * kBox);
#pragma unroll
            for (int sub = 0; sub < D / 64; ++sub)
                tma_load_2d(base + sub * kBox, &tm_kern, 64 * sub, bg * M_max + jlo, bar);
        }
    }
    // ---- Q fragments (rows = heads; rows >= G are zero)
    uint32_t a[D / 16][4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = gq + 8 * half;
        const bool ok = r < G;
        const __nv_bfloat16* qrow = q + ((static_cast<size_t>(tok) + t) * Hq + g * G + (ok ? r : 0)) * D;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            const uint4 v = ok ? ldg_v4(qrow + 32 * i + 8 * cq) : make_uint4(0, 0, 0, 0);
            a[2 * i][half] = v.x;
            a[2 * i][2 + half] = v.y;
            a[2 * i + 1][half] = v.z;
            a[2 * i + 1][2 + half] = v.w;
        }
    }
    __syncthreads();  // barrier initialised before anyone waits on it
    bool ok = n_tiles == 0 || mbar_wait(bar, 0);
    if (!ok && lane == 0) raise_error(err, kDevErrTimeout);
    const uint32_t kb = smem_u32(base);
    for (int nt = warp; ok && nt < n_tiles; nt += 4) {
        const int row = nt * 8 + gq;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            const int col = 32 * i + 8 * cq;
            const uint4 w = lds_v4(kb + (col / 64) * kBox + swz128(row, (col % 64) / 8));
            mma_16816(acc, a[2 * i], w.x, w.y);
            mma_16816(acc, a[2 * i + 1], w.z, w.w);
        }
        const int j0 = jlo + nt * 8 + 2 * cq;
        // rows past G are padding: keep them out of the head max
        if (gq >= G) acc[0] = acc[1] = -INFINITY;
        if (gq + 8 >= G) acc[2] = acc[3] = -INFINITY;
        float v0 = fmaxf(acc[0], acc[2]), v1 = fmaxf(acc[1], acc[3]);
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) {
            v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, m));
            v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, m));
        }
        if (gq == 0) {
            // every kernel up to jhi ends at or before pos, so all are visible
            if (j0 <= jhi) ks[j0 - jlo] = v0;
            if (j0 + 1 <= jhi) ks[j0 + 1 - jlo] = v1;
        }
    }
    __syncthreads();
    if (!ok) {
        if (threadIdx.x == 0) mbar_wait(bar, 0);  // let a late copy land before the CTA exits
        return;
    }
    for (int blk = blk0 + threadIdx.x; blk < blk1; blk += 128) {
        const int ja = max(first_kernel_of_block(blk, bs, c, s), jlo);
        const int jz = min(last_kernel_of_block(blk, bs, s), jhi);
        float m = -INFINITY;
        for (int jj = ja; jj <= jz; ++jj) m = fmaxf(m, ks[jj - jlo]);
        S[sm.sel(b, g, Hkv, t) * nblk_max + blk] = m;
    }
}

__device__ __forceinline__ bool is_forced(int blk, int bt, const Params& p) {
    return blk < p.n_init || blk > bt - p.n_local;
}

// Top-k selection, one CTA per (b, g, t) row.  Thread t owns the contiguous blocks
// [t*PER, t*PER + PER) and keeps their candidate keys (the order-preserving 32-bit image of each
// non-forced block's score) in registers.  The k-th largest key T is found below the bits all
// candidate keys share: for long rows by a radix select, 8 bits per round from a shared histogram
// of the next digit (three barriers a round); for short rows bit by bit (one count, one warp
// reduction and one barrier per bit, stopping once exactly k keys clear).  Keys above T are taken, and of the keys equal to T (exact ties) the
// `rem` with the lowest block ids.  One block-wide scan of (chosen, tied) counts then places
// every chosen block in ascending order.
template <int NT, int PER>
__global__ void __launch_bounds__(NT)
topk_kernel(const float* __restrict__ S, const int* __restrict__ kv_len, SeqMap sm, int B, int Hkv, int nblk_max,
            int L_max, int tree, Params p, int* __restrict__ idx, int* __restrict__ counts, int S_max,
            int* __restrict__ err) {
    constexpr int NW = NT / 32;
    __shared__ uint32_t s_and[NW], s_or[NW];
    __shared__ int s_hist[256];
    __shared__ int s_cnt[2][NW];
    __shared__ int s_sel[3];  // this round's digit, keys with a larger one, whether its bin is exactly the rest
    __shared__ int s_wsel[NW], s_wtie[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    int b, g_unused, t;
    sm.row_of(row, B, Hkv, &b, &g_unused, &t);
    pdl_wait();
    pdl_trigger();
    // the row's scores, loaded before (and independently of) the cache length that bounds them
    const float* srow = S + static_cast<size_t>(row) * nblk_max;
    float sv[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) sv[u] = tid * PER + u < nblk_max ? __ldcg(srow + tid * PER + u) : 0.f;
    const int L = kv_len[b];
    const int Tq = sm.len(b);
    int* out = idx + static_cast<size_t>(row) * S_max;
    const bool bad_len = Tq < 1 || Tq > sm.Tq || (tree ? (L < 1 || L > L_max) : (L < Tq || L > L_max));
    if (bad_len) {
        for (int i = tid; i < S_max; i += NT) out[i] = -1;
        if (tid == 0) {
            counts[row] = 0;
            raise_error(err, kDevErrIndex);
        }
        return;
    }
    const int pos = tree ? L - 1 : L - Tq + t;
    const int bt = pos / p.block_size;
    const int n = bt + 1;
    const int a_init = min(p.n_init, n);
    const int lo_local = max(bt - p.n_local + 1, 0);
    const int n_forced = a_init + (n - max(lo_local, a_init));
    const int nc = n - n_forced;
    const bool take_all = L < p.dense_len || nc <= p.topk;
    const bool take_none = !take_all && p.topk == 0;  // only the forced blocks
    const bool select = !take_all && !take_none;
    const int blk_base = tid * PER;

    uint32_t key[PER];
    bool cand[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int blk = blk_base + u;
        cand[u] = select && blk < n && !is_forced(blk, bt, p);
        key[u] = cand[u] ? ordered_key(sv[u]) : 0u;
    }

    // threshold: keys >= T are taken (all of them when tie_limit is not hit)
    uint32_t T = 0;
    int rem = 1 << 30;  // how many keys equal to T to take (the rest of T's ties are left out)
    if (select) {
        uint32_t k_and = ~0u, k_or = 0u;
#pragma unroll
        for (int u = 0; u < PER; ++u)
            if (cand[u]) {
                k_and &= key[u];
                k_or |= key[u];
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            k_and &= __shfl_xor_sync(0xffffffffu, k_and, off);
            k_or |= __shfl_xor_sync(0xffffffffu, k_or, off);
        }
        if (lane == 0) {
            s_and[warp] = k_and;
            s_or[warp] = k_or;
        }
        __syncthreads();
        k_and = ~0u;
        k_or = 0u;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            k_and &= s_and[w];
            k_or |= s_or[w];
        }
        const uint32_t diff = k_and ^ k_or;
        const int k = p.topk;
        const int top = diff == 0 ? -1 : 31 - __clz(diff);
        T = top >= 31 ? 0u : (k_and & (~0u << (top + 1)));  // bits above `top` are common to all
        // Radix select of the k-th largest key below the common bits, 8 bits per round: a histogram
        // of the next digit over the keys that match T on the bits decided so far (shared atomics,
        // one per distinct digit of a warp), then warp 0 walks the bins from the largest digit down
        // to the one where the count reaches the rank still sought.  At the end T is the k-th
        // largest key and `kr` of the keys equal to T are taken (the lowest blocks).
        int kr = k;
        bool bin_exact = false;  // a round's bin held exactly the keys still sought: all of them are taken
        // Long rows (few CTAs, each on its own SM: tree drafts, decode rows) take the radix select;
        // short rows (prefill chunks: many CTAs per SM hide each other's barriers) decide one bit
        // per round, which costs fewer instructions there.
        const bool radix = n > 512;
        for (int lo = radix ? top + 1 : 0; lo > 0;) {
            const int nb = lo < 8 ? lo : 8;
            const int shift = lo - nb;
            const uint32_t hi_mask = lo >= 32 ? 0u : (~0u << lo);
            for (int x = tid; x < 256; x += NT) s_hist[x] = 0;
            __syncthreads();
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const bool in = cand[u] && ((key[u] ^ T) & hi_mask) == 0u;
                const uint32_t dg = in ? (key[u] >> shift) & ((1u << nb) - 1u) : 0xffffffffu;
                const unsigned grp = __match_any_sync(0xffffffffu, dg);
                if (in && (__ffs(grp) - 1) == lane) atomicAdd(&s_hist[dg], __popc(grp));
            }
            __syncthreads();
            if (warp == 0) {
                int c[8], sum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = s_hist[255 - 8 * lane - j];
                    sum += c[j];
                }
                int incl = sum;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int x = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += x;
                }
                int acc = incl - sum;  // keys with a larger digit than this lane's bins
                if (acc < kr && kr <= incl) {
                    int jf = 0, above = 0;
                    bool found = false;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (!found && acc + c[j] >= kr) {
                            found = true;
                            jf = j;
                            above = acc;
                        }
                        acc += c[j];
                    }
                    s_sel[0] = 255 - 8 * lane - jf;
                    s_sel[1] = above;
                    s_sel[2] = above + c[jf] == kr;
                }
            }
            __syncthreads();
            T |= static_cast<uint32_t>(s_sel[0]) << shift;
            kr -= s_sel[1];
            lo = shift;
            if (s_sel[2]) {  // every key with T's bits so far is taken: the lower digits need no rounds
                bin_exact = true;
                break;
            }
        }
        if (radix) {
            rem = bin_exact ? (1 << 30) : kr;  // keys equal to T: all of the bin, or the kr lowest blocks
        } else {
            // bit by bit: for each bit, the number of keys >= (T | bit) by one count, one warp
            // reduction and one barrier; stop as soon as exactly k keys clear the trial value
            bool exact = false;
            int buf = 0;
            for (int bit = top; bit >= 0; --bit, buf ^= 1) {
                const uint32_t trial = T | (1u << bit);
                int c = 0;
#pragma unroll
                for (int u = 0; u < PER; ++u) c += (cand[u] && key[u] >= trial) ? 1 : 0;
                c = __reduce_add_sync(0xffffffffu, c);
                if (lane == 0) s_cnt[buf][warp] = c;
                __syncthreads();
                int total = 0;
#pragma unroll
                for (int w = 0; w < NW; ++w) total += s_cnt[buf][w];
                if (total >= k) T = trial;  // the k-th largest key has this bit set
                if (total == k) {          // exactly k keys clear `trial`: no ties to break
                    exact = true;
                    break;
                }
            }
            if (!exact) {
                // T is the k-th largest key itself; take the keys above it and enough of its ties
                int c = 0;
#pragma unroll
                for (int u = 0; u < PER; ++u) c += (cand[u] && key[u] > T) ? 1 : 0;
                c = __reduce_add_sync(0xffffffffu, c);
                if (lane == 0) s_cnt[buf][warp] = c;
                __syncthreads();
                int above = 0;
#pragma unroll
                for (int w = 0; w < NW; ++w) above += s_cnt[buf][w];
                rem = k - above;
            }
        }
    }
    const uint32_t mask = ~0u;

    // ---- chosen = forced, or key above T, or one of the first `rem` keys equal to T
    int n_sel = 0, n_tie = 0;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int blk = blk_base + u;
        if (blk >= n) continue;
        if (take_all || is_forced(blk, bt, p)) {
            ++n_sel;
        } else if (cand[u]) {
            const uint32_t km = key[u] & mask;
            n_sel += km > T;
            n_tie += km == T;
        }
    }
    // block-wide exclusive scans of the two counts
    int sel_incl = n_sel, tie_incl = n_tie;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, sel_incl, off);
        const int c = __shfl_up_sync(0xffffffffu, tie_incl, off);
        if (lane >= off) {
            sel_incl += a;
            tie_incl += c;
        }
    }
    if (lane == 31) {
        s_wsel[warp] = sel_incl;
        s_wtie[warp] = tie_incl;
    }
    __syncthreads();
    int sel_before = sel_incl - n_sel, tie_before = tie_incl - n_tie, sel_total = 0, tie_total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) {
            sel_before += s_wsel[w];
            tie_before += s_wtie[w];
        }
        sel_total += s_wsel[w];
        tie_total += s_wtie[w];
    }
    const int ties_taken = min(tie_total, rem);
    // ties taken before this thread shift every later position
    int pos_out = sel_before + min(tie_before, rem);
    int tie_rank = tie_before;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int blk = blk_base + u;
        if (blk >= n) continue;
        bool sel = take_all || is_forced(blk, bt, p);
        if (!sel && cand[u]) {
            const uint32_t km = key[u] & mask;
            if (km > T) {
                sel = true;
            } else if (km == T) {
                sel = tie_rank < rem;
                ++tie_rank;
            }
        }
        if (sel) {
            if (pos_out < S_max) out[pos_out] = blk;
            ++pos_out;
        }
    }
    const int total = sel_total + ties_taken;
    for (int i = total + tid; i < S_max; i += NT) out[i] = -1;
    if (tid == 0) {
        counts[row] = min(total, S_max);
        if (total > S_max) raise_error(err, kDevErrIndex);
    }
}

// Selection capacity for a cache of L_max tokens (see infllmv2_selection_capacity).
int selection_capacity(const Params& p, int L_max) {
    const int nblk = (L_max + p.block_size - 1) / p.block_size;
    int cap = p.topk + p.n_init + p.n_local;
    if (p.dense_len > 1) {
        const int dense_blocks = (min(p.dense_len - 1, L_max) + p.block_size - 1) / p.block_size;
        cap = max(cap, dense_blocks);
    }
    return min(cap, nblk);
}

size_t select_workspace_bytes(int B, int Tq, int Hkv, int L_max, const Params& p) {
    const size_t nblk = (L_max + p.block_size - 1) / p.block_size;
    return static_cast<size_t>(B) * Hkv * Tq * nblk * sizeof(float);
}

static int score_kmax(int bpc, const Params& p) { return (bpc * p.block_size + p.kernel_size) / p.kernel_stride + 2; }

template <int D, int WARPS, int MT>
static cudaError_t launch_score_t(const SelectArgs& a, float* S) {
    const int G = a.Hq / a.Hkv;
    const int tpc = MT * (16 / G);
    const Params& p = a.p;
    const int nblk_max = (a.L_max + p.block_size - 1) / p.block_size;
    const int bpc = a.blocks_per_cta;
    const int kmax = score_kmax(bpc, p);
    const size_t smem = static_cast<size_t>(tpc) * kmax * sizeof(float);
    dim3 grid((nblk_max + bpc - 1) / bpc, (a.Tq + tpc - 1) / tpc, a.B * a.Hkv);
    auto kfn = score_kernel<D, WARPS, MT>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kfn<<<grid, WARPS * 32, smem, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.kernel_cache), a.kv_len,
        a.seqmap(), a.Hq, a.Hkv, G, a.L_max, a.M_max, nblk_max, a.tree, p, bpc, kmax, S, a.err);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_score_decode_t(const SelectArgs& a, float* S, int bpc) {
    const int G = a.Hq / a.Hkv;
    const Params& p = a.p;
    const int nblk_max = (a.L_max + p.block_size - 1) / p.block_size;
    CUtensorMap tm;
    const uint64_t rows = static_cast<uint64_t>(a.B) * a.Hkv * a.M_max;
    if (!make_tmap_bf16_2d(&tm, a.kernel_cache, D, rows, 64, kScoreBoxRows)) return cudaErrorInvalidValue;
    const int smem = (D / 64) * kScoreBoxRows * 128 + kScoreBoxRows * 4 + 8 + 1024;
    auto kfn = score_decode_kernel<D>;
    if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); e != cudaSuccess)
        return e;
    dim3 grid((nblk_max + bpc - 1) / bpc, a.Tq, a.B * a.Hkv);
    return launch_kernel(kfn, grid, dim3(128), smem, a.stream, false, tm, static_cast<const __nv_bfloat16*>(a.q),
                         a.kv_len, a.seqmap(), a.Hq, a.Hkv, G, a.L_max, a.M_max, nblk_max, a.tree, p, bpc, S, a.err);
}

cudaError_t launch_block_select(const SelectArgs& a, float* S) {
    const Params& p = a.p;
    const int G = a.Hq / a.Hkv;
    const int nblk_max = (a.L_max + p.block_size - 1) / p.block_size;
    cudaError_t e = cudaSuccess;
    const bool many = static_cast<long long>(a.Tq) * G >= 64;
    bool decode_shaped = false;
    if (!many && a.M_max > 0) {
        // one token per CTA; the chunk's kernels must fit the TMA box
        int bpc = a.blocks_per_cta;
        while (bpc > 1 && score_kmax(bpc, p) > kScoreBoxRows) bpc /= 2;
        if (score_kmax(bpc, p) <= kScoreBoxRows) {
            decode_shaped = true;
            e = a.d == 128 ? launch_score_decode_t<128>(a, S, bpc) : launch_score_decode_t<64>(a, S, bpc);
        }
    }
    if (!decode_shaped && many && score_tc_supported(a)) {
        // many queries, 16 heads per KV head: the tensor-core GEMM scorer
        e = launch_score_tc(a, S);
        if (e == cudaSuccess) decode_shaped = false;
    } else if (!decode_shaped) {
        // many queries: each warp owns one m-tile and the CTA's warps share the kernels through L1
        if (a.d == 128) e = many ? launch_score_t<128, 4, 4>(a, S) : launch_score_t<128, 4, 1>(a, S);
        else e = many ? launch_score_t<64, 4, 4>(a, S) : launch_score_t<64, 4, 1>(a, S);
    }
    if (e != cudaSuccess) return e;
    prof_mark(a.stream, "score");
    const SeqMap sm = a.seqmap();
    const int rows = a.Hkv * sm.total;
    if (nblk_max <= 128 * 4)
        e = launch_kernel(topk_kernel<128, 4>, dim3(rows), dim3(128), 0, a.stream, true, S, a.kv_len, sm,
                          a.B, a.Hkv, nblk_max, a.L_max, a.tree, p, a.idx, a.counts, a.S_max, a.err);
    else if (nblk_max <= 512 * 2)
        e = launch_kernel(topk_kernel<512, 2>, dim3(rows), dim3(512), 0, a.stream, true, S, a.kv_len, sm,
                          a.B, a.Hkv, nblk_max, a.L_max, a.tree, p, a.idx, a.counts, a.S_max, a.err);
    else if (nblk_max <= 256 * 8)
        e = launch_kernel(topk_kernel<256, 8>, dim3(rows), dim3(256), 0, a.stream, true, S, a.kv_len, sm,
                          a.B, a.Hkv, nblk_max, a.L_max, a.tree, p, a.idx, a.counts, a.S_max, a.err);
    else if (nblk_max <= 512 * 16)
        e = launch_kernel(topk_kernel<512, 16>, dim3(rows), dim3(512), 0, a.stream, true, S, a.kv_len, sm,
                          a.B, a.Hkv, nblk_max, a.L_max, a.tree, p, a.idx, a.counts, a.S_max, a.err);
    else
        e = launch_kernel(topk_kernel<1024, 32>, dim3(rows), dim3(1024), 0, a.stream, true, S, a.kv_len,
                          sm, a.B, a.Hkv, nblk_max, a.L_max, a.tree, p, a.idx, a.counts, a.S_max, a.err);
    prof_mark(a.stream, "topk");
    return e;
}

}  // namespace infllmv2
