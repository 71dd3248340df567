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
// topk_kernel: one CTA per (b, g, t).  Candidate keys are (ordered score << 32 | ~block id),
//   unique, so "score descending, lower id first on ties" is plain key order.  A radix
//   select over 8-bit digits finds the k-th largest key (usually in 2-3 passes), then the
//   chosen and forced blocks are compacted in ascending id order with warp ballots.
#include "common.cuh"
#include "internal.h"

namespace infllmv2 {

template <int D, int WARPS, int MT>
__global__ void __launch_bounds__(WARPS * 32)
score_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kern,
             const int* __restrict__ kv_len, int Tq, int Hq, int Hkv, int G, int L_max,
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
    const bool bad_len = tree ? (L < 1 || L > L_max) : (L < Tq || L > L_max);
    if (bad_len || kernels_in(L, c, s) > M_max) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(err, kDevErrIndex);
        return;
    }
    if (L < p.dense_len) return;  // dense sequence: every block is selected, no scores needed
    if (t0 >= Tq) return;
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
        const __nv_bfloat16* qrow = q + ((static_cast<size_t>(b) * Tq + (ok ? t : 0)) * Hq + g * G + r % G) * D;
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
        S[(static_cast<size_t>(bg) * Tq + t) * nblk_max + blk] = m;
    }
}

__device__ __forceinline__ bool is_forced(int blk, int bt, const Params& p) {
    return blk < p.n_init || blk > bt - p.n_local;
}

__device__ __forceinline__ uint64_t cand_key(float s, int blk) {
    return (static_cast<uint64_t>(ordered_key(s)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(blk));
}

template <int NT>
__global__ void __launch_bounds__(NT)
topk_kernel(const float* __restrict__ S, const int* __restrict__ kv_len, int Tq, int Hkv,
            int nblk_max, int L_max, int tree, Params p, int* __restrict__ idx,
            int* __restrict__ counts, int S_max, int* __restrict__ err) {
    constexpr int NW = NT / 32;
    __shared__ unsigned hist[256];
    __shared__ int s_digit, s_above, s_cnt;
    __shared__ int s_warp[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    const int t = row % Tq;
    const int b = row / (Tq * Hkv);
    const int L = kv_len[b];
    int* out = idx + static_cast<size_t>(row) * S_max;
    const bool bad_len = tree ? (L < 1 || L > L_max) : (L < Tq || L > L_max);
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
    const float* srow = S + static_cast<size_t>(row) * nblk_max;
    const int a_init = min(p.n_init, n);
    const int lo_local = max(bt - p.n_local + 1, 0);
    const int n_forced = a_init + (n - max(lo_local, a_init));
    const int nc = n - n_forced;
    const bool take_all = L < p.dense_len || nc <= p.topk;

    uint64_t prefix = 0, mask = 0;
    if (!take_all) {
        int rem = p.topk;
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += NT) hist[i] = 0;
            __syncthreads();
            for (int blk = tid; blk < n; blk += NT) {
                if (is_forced(blk, bt, p)) continue;
                const uint64_t key = cand_key(srow[blk], blk);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l holds bins 255-8l .. 248-8l, highest first
                unsigned cnt[8], tot = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    cnt[e] = hist[255 - (lane * 8 + e)];
                    tot += cnt[e];
                }
                unsigned incl = tot;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const unsigned v = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += v;
                }
                unsigned above = incl - tot;
                if (above < static_cast<unsigned>(rem) && static_cast<unsigned>(rem) <= incl) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (above + cnt[e] >= static_cast<unsigned>(rem)) {
                            s_digit = 255 - (lane * 8 + e);
                            s_above = static_cast<int>(above);
                            s_cnt = static_cast<int>(cnt[e]);
                            break;
                        }
                        above += cnt[e];
                    }
                }
            }
            __syncthreads();
            const int digit = s_digit;
            rem -= s_above;
            prefix |= static_cast<uint64_t>(digit) << shift;
            mask |= 0xFFull << shift;
            if (s_cnt == rem) break;  // every key of this digit is needed: threshold found
        }
    }

    // ---- compaction in ascending block order
    int total = 0;
    for (int base = 0; base < n; base += NT) {
        const int blk = base + tid;
        bool sel = false;
        if (blk < n) {
            sel = take_all || is_forced(blk, bt, p) || ((cand_key(srow[blk], blk) & mask) >= prefix);
        }
        const unsigned ballot = __ballot_sync(0xffffffffu, sel);
        __syncthreads();  // s_warp of the previous round fully consumed
        if (lane == 0) s_warp[warp] = __popc(ballot);
        __syncthreads();
        int before = total, round_total = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int v = s_warp[w];
            if (w < warp) before += v;
            round_total += v;
        }
        if (sel) {
            const int pos_out = before + __popc(ballot & ((1u << lane) - 1u));
            if (pos_out < S_max) out[pos_out] = blk;
        }
        total += round_total;
    }
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

template <int D, int WARPS, int MT>
static cudaError_t launch_score_t(const SelectArgs& a, float* S) {
    const int G = a.Hq / a.Hkv;
    const int tpc = MT * (16 / G);
    const Params& p = a.p;
    const int nblk_max = (a.L_max + p.block_size - 1) / p.block_size;
    const int bpc = a.blocks_per_cta;
    const int kmax = (bpc * p.block_size + p.kernel_size) / p.kernel_stride + 2;
    const size_t smem = static_cast<size_t>(tpc) * kmax * sizeof(float);
    dim3 grid((nblk_max + bpc - 1) / bpc, (a.Tq + tpc - 1) / tpc, a.B * a.Hkv);
    auto kfn = score_kernel<D, WARPS, MT>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kfn<<<grid, WARPS * 32, smem, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.kernel_cache), a.kv_len,
        a.Tq, a.Hq, a.Hkv, G, a.L_max, a.M_max, nblk_max, a.tree, p, bpc, kmax, S, a.err);
    return cudaGetLastError();
}

cudaError_t launch_block_select(const SelectArgs& a, float* S) {
    const Params& p = a.p;
    const int G = a.Hq / a.Hkv;
    const int nblk_max = (a.L_max + p.block_size - 1) / p.block_size;
    cudaError_t e;
    // few queries: all warps of a CTA split one token-tile's kernels; many queries: each warp
    // owns one m-tile and the CTA's warps share the kernels through L1.
    const bool many = static_cast<long long>(a.Tq) * G >= 64;
    if (a.d == 128) e = many ? launch_score_t<128, 4, 4>(a, S) : launch_score_t<128, 4, 1>(a, S);
    else e = many ? launch_score_t<64, 4, 4>(a, S) : launch_score_t<64, 4, 1>(a, S);
    if (e != cudaSuccess) return e;
    prof_mark(a.stream, "score");
    const int rows = a.B * a.Hkv * a.Tq;
    if (nblk_max <= 512)
        topk_kernel<128><<<rows, 128, 0, a.stream>>>(S, a.kv_len, a.Tq, a.Hkv, nblk_max, a.L_max, a.tree, p,
                                                     a.idx, a.counts, a.S_max, a.err);
    else
        topk_kernel<512><<<rows, 512, 0, a.stream>>>(S, a.kv_len, a.Tq, a.Hkv, nblk_max, a.L_max, a.tree, p,
                                                     a.idx, a.counts, a.S_max, a.err);
    prof_mark(a.stream, "topk");
    return cudaGetLastError();
}

}  // namespace infllmv2
