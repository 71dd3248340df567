// decode.cu -- split-KV sparse attention for single-token decode and tree-speculative
// verification, and the merge of the splits ("MiniCPM4: 如何在手机电脑上高效运行大语言模型",
// section 1.1 "InfLLM v2": attention on the selected blocks only, uint64-packed mask for
// tree-speculative decoding; "CPM.cu：端侧大模型推理的 CUDA 加速引擎": tree verification inside
// flash attention).
//
// One decode row is (sequence b, draft i, KV head g): G query heads sharing one selection.
// Decode is bound by HBM reads of the selected K/V blocks, and a row has only ~4K keys, so
// the selected-block list is cut into splits of `BPS` blocks (128 keys), one CTA each.  A
// CTA's first thread issues TMA tensor copies of each selected block's K and V (16 KB each at
// 64 x 128) into 128-byte-swizzled shared tiles, one mbarrier per block, so the whole split is
// in flight at once; each of the four warps then feeds one 32-key tile through the warp-MMA
// flash-attention state of attn_warp.cuh, the warps merge in shared memory and the CTA writes
// one fp32 partial (m, l, o) per row.  In tree mode one extra split per row attends to the
// draft tokens whose bits are set in the row's uint64 mask.  decode_combine_kernel merges a
// row's partials into bf16 o and fp32 lse.  All four kernels of a decode call chain with
// programmatic dependent launch.
#include "attn_warp.cuh"
#include "internal.h"

namespace infllmv2 {

template <int D, int BS, int BPS>
struct SplitSmem {
    static constexpr int kTile = BS * D * 2;                         // one block of K (or V)
    static constexpr int kBytes = 2 * BPS * kTile + 8 * BPS + 1024;  // tiles, barriers, alignment slack
};

template <int D, int BS, int BPS>
__global__ void __launch_bounds__(128)
decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ dk,
                    const __nv_bfloat16* __restrict__ dv, const uint64_t* __restrict__ tree_mask,
                    const int* __restrict__ kv_len, const int* __restrict__ idx, const int* __restrict__ counts,
                    int idx_stride, int n_draft, int Hq, int Hkv, int G, int L_max, int n_split_cache, int n_split,
                    float scale_log2, float* __restrict__ part, int* __restrict__ err) {
    constexpr int kTile = SplitSmem<D, BS, BPS>::kTile;
    constexpr int kTilesPerBlock = BS / 32;
    constexpr int kRowPad = D + 4;
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + 2 * BPS * kTile);
    __shared__ int s_blk[BPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, c4 = lane & 3;
    const int row_id = blockIdx.y;
    const int g = row_id % Hkv;
    const int i = (row_id / Hkv) % n_draft;
    const int b = row_id / (Hkv * n_draft);
    const int sp = blockIdx.x;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
#pragma unroll
        for (int k = 0; k < BPS; ++k) mbar_init(&bars[k], 1);
        fence_mbar_init();
    }
    // q and the caches were written before this call: load Q while the selection finishes
    QFrag<D> Q;
    load_q(Q, q + ((static_cast<size_t>(b) * n_draft + i) * Hq + static_cast<size_t>(g) * G) * D, D, G);
    pdl_wait();
    pdl_trigger();
    const int L = kv_len[b];
    const bool len_ok = L >= 1 && L <= L_max;
    const int sel_row = (b * Hkv + g) * n_draft + i;
    const int cnt = counts[sel_row];
    // splits past the row's selected blocks hold nothing; the merge never reads them
    if (sp < n_split_cache && sp * BPS >= cnt) return;
    const bool cache_split = sp < n_split_cache && len_ok;
    __syncthreads();  // barrier initialisation visible to every thread

    WarpAcc<D> A;
    acc_init(A);
    if (cache_split) {
        // this CTA takes chunks sp, sp + n_split_cache, ... of BPS selected blocks (more than one
        // only for rows below dense_len, whose selection can exceed the sparse capacity)
        const int* list = idx + static_cast<size_t>(sel_row) * idx_stride;
        const int bt = (L - 1) / BS;
        uint32_t phase = 0;
        for (int ch = sp; ch * BPS < cnt; ch += n_split_cache, phase ^= 1u) {
            if (threadIdx.x == 0) {
#pragma unroll
                for (int k = 0; k < BPS; ++k) {
                    const int at = ch * BPS + k;
                    int blk = at < cnt ? list[at] : -1;
                    if (at < cnt && (blk < 0 || blk > bt)) {
                        raise_error(err, kDevErrIndex);
                        blk = -1;
                    }
                    s_blk[k] = blk;
                    if (blk >= 0) {
                        const int row = (b * Hkv + g) * L_max + blk * BS;
                        mbar_arrive_expect_tx(&bars[k], 2 * kTile);
#pragma unroll
                        for (int sub = 0; sub < D / 64; ++sub) {
                            tma_load_2d(base + (2 * k) * kTile + sub * BS * 128, &tm_k, 64 * sub, row, &bars[k]);
                            tma_load_2d(base + (2 * k + 1) * kTile + sub * BS * 128, &tm_v, 64 * sub, row, &bars[k]);
                        }
                    } else {
                        mbar_arrive(&bars[k]);  // keep every slot's phase in step
                    }
                }
            }
            __syncthreads();
            for (int tile = warp; tile < BPS * kTilesPerBlock; tile += 4) {
                const int k = tile / kTilesPerBlock;
                const int blk = s_blk[k];
                if (blk < 0) continue;
                const int r0 = (tile % kTilesPerBlock) * 32;
                const int n_ok = L - (blk * BS + r0);
                if (n_ok <= 0) continue;
                const uint32_t valid = n_ok >= 32 ? 0xffffffffu : ((1u << n_ok) - 1u);
                if (!mbar_wait(&bars[k], phase)) {
                    if (lane == 0) raise_error(err, kDevErrTimeout);
                    continue;
                }
                attend32_smem<D>(A, Q, smem_u32(base + (2 * k) * kTile), smem_u32(base + (2 * k + 1) * kTile), BS,
                                 r0, valid, scale_log2);
            }
            // every copy of this chunk has landed and been read before the tiles are refilled
            if (threadIdx.x == 0) {
#pragma unroll
                for (int k = 0; k < BPS; ++k)
                    if (!mbar_wait(&bars[k], phase)) raise_error(err, kDevErrTimeout);
            }
            __syncthreads();
        }
    } else if (sp >= n_split_cache && tree_mask != nullptr && len_ok) {
        const int j0 = warp * 32;
        if (j0 < n_draft) {
            const uint64_t bits = tree_mask[static_cast<size_t>(b) * n_draft + i] >> j0;
            const int n_rows = n_draft - j0;
            uint32_t valid = static_cast<uint32_t>(bits);
            if (n_rows < 32) valid &= (1u << n_rows) - 1u;
            const size_t off = ((static_cast<size_t>(b) * Hkv + g) * n_draft + j0) * D;
            attend32(A, Q, dk + off, dv + off, valid, scale_log2);
        }
    } else if (!len_ok && sp == 0 && threadIdx.x == 0) {
        raise_error(err, kDevErrIndex);
    }
    acc_finish_rowsum(A);
    __syncthreads();  // the tiles are reused for the merge

    // ---- merge the four warps (reusing the tile memory)
    float* sm_m = reinterpret_cast<float*>(base);
    float* sm_l = sm_m + 4 * 16;
    float* sm_o = sm_l + 4 * 16;  // [4][16][kRowPad]
    if (c4 == 0) {
        sm_m[warp * 16 + g8] = A.m[0];
        sm_m[warp * 16 + g8 + 8] = A.m[1];
        sm_l[warp * 16 + g8] = A.l[0];
        sm_l[warp * 16 + g8 + 8] = A.l[1];
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sm_o[(warp * 16 + g8 + 8 * (e >> 1)) * kRowPad + o_col(D, c4, nt, e)] = A.o[nt][e];
    __syncthreads();
    float* dst = part + (static_cast<size_t>(row_id) * n_split + sp) * PartialLayout<D>::kFloats;
    for (int e = threadIdx.x; e < 16 * D; e += 128) {
        const int r = e / D, col = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w * 16 + r]);
        const float ref = M == -INFINITY ? 0.f : M;
        float acc = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float f = fast_exp2(sm_m[w * 16 + r] - ref);
            acc += sm_o[(w * 16 + r) * kRowPad + col] * f;
            l += sm_l[w * 16 + r] * f;
        }
        dst[32 + e] = acc;
        if (col == 0) {
            dst[r] = M;
            dst[16 + r] = l;
        }
    }
}

// Merge of one (row, head)'s split partials: warp 0 turns the splits' maxima into weights
// (shared memory), then each of the D threads sums its output element over the splits.
template <int D>
__global__ void __launch_bounds__(D)
decode_combine_kernel(const float* __restrict__ part, const int* __restrict__ counts, int blocks_per_split,
                      int n_split_cache, int n_split, int n_draft, int Hq, int Hkv, int G,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
    extern __shared__ float s_f[];  // [n_split] weights
    __shared__ float s_M, s_L;
    __shared__ int s_nread, s_used;
    const int row_id = blockIdx.x;
    const int r = blockIdx.y;
    const int g = row_id % Hkv;
    const int i = (row_id / Hkv) % n_draft;
    const int b = row_id / (Hkv * n_draft);
    pdl_wait();
    const float* src = part + static_cast<size_t>(row_id) * n_split * PartialLayout<D>::kFloats;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        // the cache splits that hold selected blocks, then the draft split (tree mode)
        const int cnt = counts[(b * Hkv + g) * n_draft + i];
        const int used = min((cnt + blocks_per_split - 1) / blocks_per_split, n_split_cache);
        const int n_read = used + (n_split - n_split_cache);
        float M = -INFINITY;
        for (int k = lane; k < n_read; k += 32) {
            const int s = k < used ? k : n_split_cache + (k - used);
            M = fmaxf(M, __ldcg(src + s * PartialLayout<D>::kFloats + r));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float ref = M == -INFINITY ? 0.f : M;
        float l = 0.f;
        for (int k = lane; k < n_read; k += 32) {
            const int s = k < used ? k : n_split_cache + (k - used);
            const float* ps = src + s * PartialLayout<D>::kFloats;
            const float f = fast_exp2(__ldcg(ps + r) - ref);
            s_f[k] = f;
            l += __ldcg(ps + 16 + r) * f;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) {
            s_M = M;
            s_L = l;
            s_nread = n_read;
            s_used = used;
        }
    }
    __syncthreads();
    const int n_read = s_nread, used = s_used;
    const int d = threadIdx.x;
    float acc = 0.f;
#pragma unroll 8
    for (int k = 0; k < n_read; ++k) {
        const int s = k < used ? k : n_split_cache + (k - used);
        acc += __ldcg(src + s * PartialLayout<D>::kFloats + 32 + r * D + d) * s_f[k];
    }
    const float l = s_L;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int h = g * G + r;
    o[((static_cast<size_t>(b) * n_draft + i) * Hq + h) * D + d] = __float2bfloat16_rn(acc * inv);
    if (lse != nullptr && d == 0)
        lse[(static_cast<size_t>(b) * Hq + h) * n_draft + i] =
            l > 0.f ? (s_M + log2f(l)) * 0.69314718055994530942f : -INFINITY;
}

size_t decode_partial_bytes(int B, int n_draft, int Hkv, int d, int n_split) {
    const size_t per = d == 128 ? PartialLayout<128>::kFloats : PartialLayout<64>::kFloats;
    return static_cast<size_t>(B) * n_draft * Hkv * n_split * per * sizeof(float);
}

void decode_split_shape(const Params& p, int L_max, bool tree, long long rows, int* blocks_per_split,
                        int* n_split_cache, int* n_split) {
    // 128 keys per chunk (one 32-key tile per warp): two 64-token blocks or one 128-token block;
    // one CTA per chunk of a sparse row's selection (top-k + forced); longer (dense) selections
    // loop over several chunks per CTA.  A tree has a row per draft: with many rows, fewer CTAs per
    // row (each looping over more chunks) keep the grid near kTreeCtas and cut the partials that
    // the merge reads back.
    constexpr long long kTreeCtas = 600;
    const int bps = p.block_size >= 128 ? 1 : 128 / p.block_size;
    const int nblk = (L_max + p.block_size - 1) / p.block_size;
    const int sparse_cap = max(1, min(p.topk + p.n_init + p.n_local, nblk));
    int nsc = (sparse_cap + bps - 1) / bps;
    if (tree && rows > 0) nsc = static_cast<int>(max(1ll, min(static_cast<long long>(nsc), kTreeCtas / rows)));
    *blocks_per_split = bps;
    *n_split_cache = nsc;
    *n_split = nsc + (tree ? 1 : 0);
}

template <int D, int BS, int BPS>
static cudaError_t launch_split_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, const int* idx,
                                  const int* counts, int idx_stride, int nsc, int ns, float* part) {
    const int G = a.Hq / a.Hkv;
    const int rows = a.B * a.n_draft * a.Hkv;
    const float scale_log2 = a.p.scale * 1.4426950408889634f;
    constexpr int smem = SplitSmem<D, BS, BPS>::kBytes;
    auto kfn = decode_split_kernel<D, BS, BPS>;
    if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); e != cudaSuccess)
        return e;
    return launch_kernel(kfn, dim3(ns, rows), dim3(128), smem, a.stream, true, tk, tv,
                         static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.draft_k),
                         static_cast<const __nv_bfloat16*>(a.draft_v), a.tree_mask, a.kv_len, idx, counts, idx_stride,
                         a.n_draft, a.Hq, a.Hkv, G, a.L_max, nsc, ns, scale_log2, part, a.err);
}

cudaError_t launch_decode_attention(const DecodeArgs& a, const int* idx, const int* counts, int idx_stride,
                                    float* part) {
    int bps, nsc, ns;
    decode_split_shape(a.p, a.L_max, a.tree_mask != nullptr, static_cast<long long>(a.B) * a.n_draft * a.Hkv, &bps,
                       &nsc, &ns);
    const int G = a.Hq / a.Hkv;
    const int rows = a.B * a.n_draft * a.Hkv;
    const int bs = a.p.block_size;
    CUtensorMap tk, tv;
    const uint64_t cache_rows = static_cast<uint64_t>(a.B) * a.Hkv * a.L_max;
    if (!make_tmap_bf16_2d(&tk, a.k_cache, a.d, cache_rows, 64, bs) ||
        !make_tmap_bf16_2d(&tv, a.v_cache, a.d, cache_rows, 64, bs))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (a.d == 128)
        e = bs == 64 ? launch_split_t<128, 64, 2>(a, tk, tv, idx, counts, idx_stride, nsc, ns, part)
                     : launch_split_t<128, 128, 1>(a, tk, tv, idx, counts, idx_stride, nsc, ns, part);
    else
        e = bs == 64 ? launch_split_t<64, 64, 2>(a, tk, tv, idx, counts, idx_stride, nsc, ns, part)
                     : launch_split_t<64, 128, 1>(a, tk, tv, idx, counts, idx_stride, nsc, ns, part);
    if (e != cudaSuccess) return e;
    prof_mark(a.stream, "attend");
    const size_t csmem = static_cast<size_t>(ns) * sizeof(float);
    auto* op = static_cast<__nv_bfloat16*>(a.o);
    if (a.d == 128)
        e = launch_kernel(decode_combine_kernel<128>, dim3(rows, G), dim3(128), csmem, a.stream, true, part, counts,
                          bps, nsc, ns, a.n_draft, a.Hq, a.Hkv, G, op, a.lse);
    else
        e = launch_kernel(decode_combine_kernel<64>, dim3(rows, G), dim3(64), csmem, a.stream, true, part, counts, bps,
                          nsc, ns, a.n_draft, a.Hq, a.Hkv, G, op, a.lse);
    prof_mark(a.stream, "combine");
    return e;
}

}  // namespace infllmv2
