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


// Decode-shaped scoring: one query token (G <= 16 heads, one MMA m-tile) per CTA and a chunk of
// blocks; each warp issues the loads of all its kernel n-tiles before its first MMA, so the
// whole chunk (about 33 KB) is in flight at once and the scan runs at memory speed.
template <int D, int NPW>
__global__ void __launch_bounds__(128)
score_decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kern,
                    const int* __restrict__ kv_len, int Tq, int Hq, int Hkv, int G, int L_max, int M_max,
                    int nblk_max, int tree, Params p, int blocks_per_cta, int kmax,
                    float* __restrict__ S, int* __restrict__ err) {
    extern __shared__ float ks[];  // [kmax] max over heads per kernel of the chunk
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int t = blockIdx.y;
    const int bg = blockIdx.z;
    const int b = bg / Hkv, g = bg % Hkv;
    const int bs = p.block_size, c = p.kernel_size, s = p.kernel_stride;
    pdl_trigger();
    const int L = kv_len[b];
    const bool bad_len = tree ? (L < 1 || L > L_max) : (L < Tq || L > L_max);
    if (bad_len || kernels_in(L, c, s) > M_max) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && t == 0) raise_error(err, kDevErrIndex);
        return;
    }
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

    // ---- kernel rows: all of this warp's n-tiles, issued up front
    const __nv_bfloat16* kbase = kern + static_cast<size_t>(bg) * M_max * D + 8 * cq;
    uint4 w[NPW][D / 32];
#pragma unroll
    for (int u = 0; u < NPW; ++u) {
        const int nt = warp * NPW + u;
        const int jrow = min(jlo + nt * 8 + gq, jhi);
        const bool live = nt < n_tiles;
        const __nv_bfloat16* krow = kbase + static_cast<size_t>(live ? jrow : jlo) * D;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) w[u][i] = live ? ldg_v4_stream(krow + 32 * i) : make_uint4(0, 0, 0, 0);
    }
    // ---- Q fragments (rows = heads; rows >= G are zero)
    uint32_t a[D / 16][4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = gq + 8 * half;
        const bool ok = r < G;
        const __nv_bfloat16* qrow = q + ((static_cast<size_t>(b) * Tq + t) * Hq + g * G + (ok ? r : 0)) * D;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            const uint4 v = ok ? ldg_v4(qrow + 32 * i + 8 * cq) : make_uint4(0, 0, 0, 0);
            a[2 * i][half] = v.x;
            a[2 * i][2 + half] = v.y;
            a[2 * i + 1][half] = v.z;
            a[2 * i + 1][2 + half] = v.w;
        }
    }
#pragma unroll
    for (int u = 0; u < NPW; ++u) {
        const int nt = warp * NPW + u;
        if (nt >= n_tiles) break;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            mma_16816(acc, a[2 * i], w[u][i].x, w[u][i].y);
            mma_16816(acc, a[2 * i + 1], w[u][i].z, w[u][i].w);
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
    for (int blk = blk0 + threadIdx.x; blk < blk1; blk += 128) {
        const int ja = max(first_kernel_of_block(blk, bs, c, s), jlo);
        const int jz = min(last_kernel_of_block(blk, bs, s), jhi);
        float m = -INFINITY;
        for (int jj = ja; jj <= jz; ++jj) m = fmaxf(m, ks[jj - jlo]);
        S[(static_cast<size_t>(bg) * Tq + t) * nblk_max + blk] = m;
    }
}

__device__ __forceinline__ bool is_forced(int blk, int bt, const Params& p) {
    return blk < p.n_init || blk > bt - p.n_local;
}

__device__ __forceinline__ uint64_t cand_key(float s, int blk) {
    return (static_cast<uint64_t>(ordered_key(s)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(blk));
}

// Top-k selection, one CTA per (b, g, t) row.  Each thread keeps up to PER candidate keys in
// registers (blocks tid, tid+NT, ...); rows longer than NT*PER re-read the scores each pass.
// The radix select starts at the first bit where the candidates' keys differ (found with an
// AND/OR reduction), uses 8-bit digits, and counts digits with warp-aggregated shared atomics
// (lanes holding the same digit add once), so scores crowded into a few exponents cost no
// atomic contention.
template <int NT, int PER>
__global__ void __launch_bounds__(NT)
topk_kernel(const float* __restrict__ S, const int* __restrict__ kv_len, int Tq, int Hkv,
            int nblk_max, int L_max, int tree, Params p, int* __restrict__ idx,
            int* __restrict__ counts, int S_max, int* __restrict__ err) {
    constexpr int NW = NT / 32;
    __shared__ unsigned hist[256];
    __shared__ unsigned long long s_and[NW], s_or[NW];
    __shared__ int s_digit, s_above, s_cnt;
    __shared__ int s_warp[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    const int t = row % Tq;
    const int b = row / (Tq * Hkv);
    pdl_wait();
    pdl_trigger();
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
    const bool take_none = !take_all && p.topk == 0;  // only the forced blocks
    const bool in_regs = n <= NT * PER;

    uint64_t key[PER];
    bool live[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int blk = tid + u * NT;
        live[u] = !take_all && !take_none && in_regs && blk < n && !is_forced(blk, bt, p);
        key[u] = live[u] ? cand_key(__ldcg(srow + blk), blk) : 0ull;
    }
    auto get_key = [&](int blk, bool& ok) -> uint64_t {
        ok = blk < n && !is_forced(blk, bt, p);
        return ok ? cand_key(__ldcg(srow + blk), blk) : 0ull;
    };

    uint64_t prefix = 0, mask = 0;
    if (!take_all && !take_none) {
        // common leading bits of all candidate keys
        uint64_t k_and = ~0ull, k_or = 0ull;
        if (in_regs) {
#pragma unroll
            for (int u = 0; u < PER; ++u)
                if (live[u]) { k_and &= key[u]; k_or |= key[u]; }
        } else {
            for (int blk = tid; blk < n; blk += NT) {
                bool ok;
                const uint64_t kk = get_key(blk, ok);
                if (ok) { k_and &= kk; k_or |= kk; }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            k_and &= __shfl_xor_sync(0xffffffffu, k_and, off);
            k_or |= __shfl_xor_sync(0xffffffffu, k_or, off);
        }
        if (lane == 0) { s_and[warp] = k_and; s_or[warp] = k_or; }
        __syncthreads();
        k_and = ~0ull;
        k_or = 0ull;
#pragma unroll
        for (int w = 0; w < NW; ++w) { k_and &= s_and[w]; k_or |= s_or[w]; }
        const uint64_t diff = k_and ^ k_or;  // non-zero: keys are unique and nc > topk >= 1
        const int top = 63 - __clzll(diff);  // highest bit where candidates differ
        mask = top >= 63 ? 0ull : (~0ull << (top + 1));
        prefix = k_and & mask;
        int rem = p.topk;
        for (int shift = max(top - 7, 0);; shift = max(shift - 8, 0)) {
            const int width = min(8, top + 1 - shift);  // first pass may be narrower than 8 bits
            for (int i = tid; i < 256; i += NT) hist[i] = 0;
            __syncthreads();
            auto count = [&](uint64_t kk, bool ok) {
                const unsigned dig = static_cast<unsigned>((kk >> shift) & 255u);
                const bool hit = ok && (kk & mask) == prefix;
                const unsigned peers = __match_any_sync(0xffffffffu, hit ? dig : 256u + lane);
                if (hit && lane == __ffs(peers) - 1) atomicAdd(&hist[dig], static_cast<unsigned>(__popc(peers)));
            };
            if (in_regs) {
#pragma unroll
                for (int u = 0; u < PER; ++u) count(key[u], live[u]);
            } else {
                for (int base = 0; base < n; base += NT) {
                    bool ok;
                    const uint64_t kk = get_key(base + tid, ok);
                    count(kk, ok);
                }
            }
            __syncthreads();
            if (warp == 0) {
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
            const uint64_t dmask = ((1ull << width) - 1ull) << shift;
            rem -= s_above;
            prefix |= static_cast<uint64_t>(s_digit) << shift;
            mask |= dmask;
            if (s_cnt == rem || shift == 0) break;  // every key of this digit is needed
            __syncthreads();
        }
    }

    // ---- compaction in ascending block order
    int total = 0;
    for (int base = 0; base < n; base += NT) {
        const int blk = base + tid;
        bool sel = false;
        if (blk < n) {
            if (take_all || is_forced(blk, bt, p)) sel = true;
            else if (!take_none) sel = (cand_key(__ldcg(srow + blk), blk) & mask) >= prefix;
        }
        const unsigned ballot = __ballot_sync(0xffffffffu, sel);
        __syncthreads();
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
        a.Tq, a.Hq, a.Hkv, G, a.L_max, a.M_max, nblk_max, a.tree, p, bpc, kmax, S, a.err);
    return cudaGetLastError();
}

// Kernel n-tiles per warp of score_decode_kernel for a chunk of bpc blocks.
constexpr int kDecodeNPW = 5;

template <int D>
static cudaError_t launch_score_decode_t(const SelectArgs& a, float* S, int bpc) {
    const int G = a.Hq / a.Hkv;
    const Params& p = a.p;
    const int nblk_max = (a.L_max + p.block_size - 1) / p.block_size;
    const int kmax = score_kmax(bpc, p);
    dim3 grid((nblk_max + bpc - 1) / bpc, a.Tq, a.B * a.Hkv);
    return launch_kernel(score_decode_kernel<D, kDecodeNPW>, grid, dim3(128), static_cast<size_t>(kmax) * sizeof(float),
                         a.stream, false, static_cast<const __nv_bfloat16*>(a.q),
                         static_cast<const __nv_bfloat16*>(a.kernel_cache), a.kv_len, a.Tq, a.Hq, a.Hkv, G, a.L_max,
                         a.M_max, nblk_max, a.tree, p, bpc, kmax, S, a.err);
}

cudaError_t launch_block_select(const SelectArgs& a, float* S) {
    const Params& p = a.p;
    const int G = a.Hq / a.Hkv;
    const int nblk_max = (a.L_max + p.block_size - 1) / p.block_size;
    cudaError_t e;
    const bool many = static_cast<long long>(a.Tq) * G >= 64;
    bool decode_shaped = false;
    if (!many) {
        // one token per CTA; the chunk must fit 4 warps x kDecodeNPW n-tiles of 8 kernels
        int bpc = a.blocks_per_cta;
        while (bpc > 1 && score_kmax(bpc, p) > 4 * kDecodeNPW * 8) bpc /= 2;
        if (score_kmax(bpc, p) <= 4 * kDecodeNPW * 8) {
            decode_shaped = true;
            e = a.d == 128 ? launch_score_decode_t<128>(a, S, bpc) : launch_score_decode_t<64>(a, S, bpc);
        }
    }
    if (!decode_shaped) {
        // many queries: each warp owns one m-tile and the CTA's warps share the kernels through L1
        if (a.d == 128) e = many ? launch_score_t<128, 4, 4>(a, S) : launch_score_t<128, 4, 1>(a, S);
        else e = many ? launch_score_t<64, 4, 4>(a, S) : launch_score_t<64, 4, 1>(a, S);
    }
    if (e != cudaSuccess) return e;
    prof_mark(a.stream, "score");
    const int rows = a.B * a.Hkv * a.Tq;
    const bool pdl = decode_shaped;
    if (nblk_max <= 256)
        e = launch_kernel(topk_kernel<128, 2>, dim3(rows), dim3(128), 0, a.stream, pdl, S, a.kv_len, a.Tq, a.Hkv,
                          nblk_max, a.L_max, a.tree, p, a.idx, a.counts, a.S_max, a.err);
    else
        e = launch_kernel(topk_kernel<256, 8>, dim3(rows), dim3(256), 0, a.stream, pdl, S, a.kv_len, a.Tq, a.Hkv,
                          nblk_max, a.L_max, a.tree, p, a.idx, a.counts, a.S_max, a.err);
    prof_mark(a.stream, "topk");
    return e;
}

}  // namespace infllmv2
