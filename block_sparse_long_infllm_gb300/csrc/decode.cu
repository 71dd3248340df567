// decode.cu -- split-KV sparse attention for single-token decode and tree-speculative
// verification, and the merge of the splits ("MiniCPM4: 如何在手机电脑上高效运行大语言模型",
// section 1.1 "InfLLM v2": attention on the selected blocks only, uint64-packed mask for
// tree-speculative decoding; "CPM.cu：端侧大模型推理的 CUDA 加速引擎": tree verification inside
// flash attention).
//
// One decode row is (sequence b, draft i, KV head g): G query heads sharing one selection.
// Decode is bound by HBM reads of the selected K/V blocks, and a row has only ~4K keys, so
// the selected-block list is cut into splits of `blocks_per_split` blocks, one CTA each, to
// put enough bytes in flight on all SMs.  Each of a CTA's four warps streams 32-key tiles
// (16-byte loads that skip L1) through the warp MMA flash-attention state of attn_warp.cuh;
// the warps merge in shared memory and the CTA writes one fp32 partial (m, l, o) per row.
// In tree mode one extra split per row attends to the draft tokens whose bits are set in
// the row's uint64 mask.  decode_combine_kernel merges a row's partials into bf16 o and lse.
#include "attn_warp.cuh"
#include "internal.h"

namespace infllmv2 {

template <int D>
struct PartialLayout {
    static constexpr int kFloats = 16 + 16 + 16 * D;  // m[16], l[16], o[16][D]
};

template <int D>
__global__ void __launch_bounds__(128)
decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                    const __nv_bfloat16* __restrict__ vc, const __nv_bfloat16* __restrict__ dk,
                    const __nv_bfloat16* __restrict__ dv, const uint64_t* __restrict__ tree_mask,
                    const int* __restrict__ kv_len, const int* __restrict__ idx,
                    const int* __restrict__ counts, int idx_stride, int n_draft, int Hq, int Hkv, int G,
                    int L_max, int bs, int blocks_per_split, int n_split_cache, int n_split,
                    float scale_log2, float* __restrict__ part, int* __restrict__ err) {
    constexpr int kRowPad = D + 4;
    __shared__ float sm_m[4][16], sm_l[4][16];
    __shared__ float sm_o[4][16][kRowPad];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, c4 = lane & 3;
    const int row_id = blockIdx.y;
    const int g = row_id % Hkv;
    const int i = (row_id / Hkv) % n_draft;
    const int b = row_id / (Hkv * n_draft);
    const int sp = blockIdx.x;
    // q and the caches were written before this call: load Q while the selection finishes
    QFrag<D> Q;
    load_q(Q, q + ((static_cast<size_t>(b) * n_draft + i) * Hq + static_cast<size_t>(g) * G) * D, D, G);
    pdl_wait();
    pdl_trigger();
    const int L = kv_len[b];
    const bool len_ok = L >= 1 && L <= L_max;
    // splits past the row's selected blocks hold nothing; the merge never reads them
    if (sp < n_split_cache && sp * blocks_per_split >= counts[(b * Hkv + g) * n_draft + i]) return;

    WarpAcc<D> A;
    acc_init(A);
    if (len_ok) {
        if (sp < n_split_cache) {
            const int sel_row = (b * Hkv + g) * n_draft + i;
            const int cnt = counts[sel_row];
            const int* list = idx + static_cast<size_t>(sel_row) * idx_stride;
            const int first = sp * blocks_per_split;
            const int last = min(first + blocks_per_split, cnt);
            const int tiles_per_block = bs / 32;
            const int n_tiles = (last - first) * tiles_per_block;
            const int bt = (L - 1) / bs;
            const size_t head_base = (static_cast<size_t>(b) * Hkv + g) * L_max;
            for (int tile = warp; tile < n_tiles; tile += 4) {
                const int blk = list[first + tile / tiles_per_block];
                if (blk < 0 || blk > bt) {
                    if (lane == 0) raise_error(err, kDevErrIndex);
                    continue;
                }
                const int x0 = blk * bs + (tile % tiles_per_block) * 32;
                const int n_ok = L - x0;
                if (n_ok <= 0) continue;
                const uint32_t valid = n_ok >= 32 ? 0xffffffffu : ((1u << n_ok) - 1u);
                attend32(A, Q, kc + (head_base + x0) * D, vc + (head_base + x0) * D, valid, scale_log2);
            }
        } else if (tree_mask != nullptr) {
            const int j0 = warp * 32;
            if (j0 < n_draft) {
                const uint64_t bits = tree_mask[static_cast<size_t>(b) * n_draft + i] >> j0;
                const int n_rows = n_draft - j0;
                uint32_t valid = static_cast<uint32_t>(bits);
                if (n_rows < 32) valid &= (1u << n_rows) - 1u;
                const size_t base = ((static_cast<size_t>(b) * Hkv + g) * n_draft + j0) * D;
                attend32(A, Q, dk + base, dv + base, valid, scale_log2);
            }
        }
    } else if (sp == 0 && threadIdx.x == 0) {
        raise_error(err, kDevErrIndex);
    }
    acc_finish_rowsum(A);

    // ---- merge the four warps
    if (c4 == 0) {
        sm_m[warp][g8] = A.m[0];
        sm_m[warp][g8 + 8] = A.m[1];
        sm_l[warp][g8] = A.l[0];
        sm_l[warp][g8 + 8] = A.l[1];
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sm_o[warp][g8 + 8 * (e >> 1)][o_col(D, c4, nt, e)] = A.o[nt][e];
    __syncthreads();
    float* dst = part + (static_cast<size_t>(row_id) * n_split + sp) * PartialLayout<D>::kFloats;
    for (int e = threadIdx.x; e < 16 * D; e += 128) {
        const int r = e / D, col = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w][r]);
        const float ref = M == -INFINITY ? 0.f : M;
        float acc = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float f = fast_exp2(sm_m[w][r] - ref);
            acc += sm_o[w][r][col] * f;
            l += sm_l[w][r] * f;
        }
        dst[32 + e] = acc;
        if (col == 0) {
            dst[r] = M;
            dst[16 + r] = l;
        }
    }
}

// Merge of a row's split partials: D/4 threads per query head (four output elements each),
// 512/D heads per CTA, so a batch of rows spreads over many SMs and every thread's split
// loop issues independent loads.
template <int D>
__global__ void __launch_bounds__(128)
decode_combine_kernel(const float* __restrict__ part, const int* __restrict__ counts, int blocks_per_split,
                      int n_split_cache, int n_split, int n_draft, int Hq, int Hkv, int G,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
    constexpr int TPH = D / 4;        // threads per head row
    constexpr int HPC = 128 / TPH;    // head rows per CTA
    const int row_id = blockIdx.x;
    const int r = blockIdx.y * HPC + threadIdx.x / TPH;
    const int dq = (threadIdx.x % TPH) * 4;
    const int g = row_id % Hkv;
    const int i = (row_id / Hkv) % n_draft;
    const int b = row_id / (Hkv * n_draft);
    pdl_wait();
    if (r >= G) return;
    const float* src = part + static_cast<size_t>(row_id) * n_split * PartialLayout<D>::kFloats;
    // the cache splits that hold selected blocks, then the draft split (tree mode)
    const int cnt = counts[(b * Hkv + g) * n_draft + i];
    const int used = min((cnt + blocks_per_split - 1) / blocks_per_split, n_split_cache);
    const int n_read = used + (n_split - n_split_cache);
    float M = -INFINITY;
    for (int k = 0; k < n_read; ++k) {
        const int s = k < used ? k : n_split_cache + (k - used);
        M = fmaxf(M, __ldcg(src + s * PartialLayout<D>::kFloats + r));
    }
    const float ref = M == -INFINITY ? 0.f : M;
    float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < n_read; ++k) {
        const int s = k < used ? k : n_split_cache + (k - used);
        const float* ps = src + s * PartialLayout<D>::kFloats;
        const float f = fast_exp2(__ldcg(ps + r) - ref);
        l += __ldcg(ps + 16 + r) * f;
        const float4 ov = __ldcg(reinterpret_cast<const float4*>(ps + 32 + r * D + dq));
        acc[0] += ov.x * f;
        acc[1] += ov.y * f;
        acc[2] += ov.z * f;
        acc[3] += ov.w * f;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int h = g * G + r;
    uint2 packed;
    packed.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    packed.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(o + ((static_cast<size_t>(b) * n_draft + i) * Hq + h) * D + dq) = packed;
    if (lse != nullptr && dq == 0)
        lse[(static_cast<size_t>(b) * Hq + h) * n_draft + i] =
            l > 0.f ? (M + log2f(l)) * 0.69314718055994530942f : -INFINITY;
}

size_t decode_partial_bytes(int B, int n_draft, int Hkv, int d, int n_split) {
    const size_t per = d == 128 ? PartialLayout<128>::kFloats : PartialLayout<64>::kFloats;
    return static_cast<size_t>(B) * n_draft * Hkv * n_split * per * sizeof(float);
}

void decode_split_shape(int S_cap, int bs, bool tree, int* blocks_per_split, int* n_split_cache, int* n_split) {
    // 128 keys per split (one 32-key tile per warp) for 64-token blocks, one block for 128.
    const int bps = bs >= 128 ? 1 : 128 / bs;
    *blocks_per_split = bps;
    *n_split_cache = (S_cap + bps - 1) / bps;
    *n_split = *n_split_cache + (tree ? 1 : 0);
}

cudaError_t launch_decode_attention(const DecodeArgs& a, const int* idx, const int* counts, int idx_stride,
                                    int S_cap, float* part) {
    int bps, nsc, ns;
    decode_split_shape(S_cap, a.p.block_size, a.tree_mask != nullptr, &bps, &nsc, &ns);
    const int G = a.Hq / a.Hkv;
    const int rows = a.B * a.n_draft * a.Hkv;
    const float scale_log2 = a.p.scale * 1.4426950408889634f;
    const auto* qp = static_cast<const __nv_bfloat16*>(a.q);
    const auto* kp = static_cast<const __nv_bfloat16*>(a.k_cache);
    const auto* vp = static_cast<const __nv_bfloat16*>(a.v_cache);
    const auto* dkp = static_cast<const __nv_bfloat16*>(a.draft_k);
    const auto* dvp = static_cast<const __nv_bfloat16*>(a.draft_v);
    auto* op = static_cast<__nv_bfloat16*>(a.o);
    cudaError_t e;
    if (a.d == 128) {
        e = launch_kernel(decode_split_kernel<128>, dim3(ns, rows), dim3(128), 0, a.stream, true, qp, kp, vp, dkp, dvp,
                          a.tree_mask, a.kv_len, idx, counts, idx_stride, a.n_draft, a.Hq, a.Hkv, G, a.L_max,
                          a.p.block_size, bps, nsc, ns, scale_log2, part, a.err);
        if (e != cudaSuccess) return e;
        prof_mark(a.stream, "attend");
        e = launch_kernel(decode_combine_kernel<128>, dim3(rows, (G + 3) / 4), dim3(128), 0, a.stream, true, part,
                          counts, bps, nsc, ns, a.n_draft, a.Hq, a.Hkv, G, op, a.lse);
    } else {
        e = launch_kernel(decode_split_kernel<64>, dim3(ns, rows), dim3(128), 0, a.stream, true, qp, kp, vp, dkp, dvp,
                          a.tree_mask, a.kv_len, idx, counts, idx_stride, a.n_draft, a.Hq, a.Hkv, G, a.L_max,
                          a.p.block_size, bps, nsc, ns, scale_log2, part, a.err);
        if (e != cudaSuccess) return e;
        prof_mark(a.stream, "attend");
        e = launch_kernel(decode_combine_kernel<64>, dim3(rows, (G + 7) / 8), dim3(128), 0, a.stream, true, part,
                          counts, bps, nsc, ns, a.n_draft, a.Hq, a.Hkv, G, op, a.lse);
    }
    prof_mark(a.stream, "combine");
    return e;
}

}  // namespace infllmv2
