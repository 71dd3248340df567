// prefill.cu -- block-sparse causal attention for a prefill chunk, one warp per query token
// ("MiniCPM4: 如何在手机电脑上高效运行大语言模型", section 1.1 "InfLLM v2": attention on the
// selected blocks only; "CPM.cu：端侧大模型推理的 CUDA 加速引擎", section 4: chunked prefill).
//
// Each token's G heads share one selection, so a warp owns the 16 MMA rows of one token and
// walks that token's own blocks -- no work is spent on blocks another token chose.  Keys past
// the query's position or past kv_len are masked.  This is the warp-MMA path; it serves every
// supported shape.
#include "attn_warp.cuh"
#include "internal.h"

namespace infllmv2 {

template <int D>
__global__ void __launch_bounds__(128)
prefill_warp_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                    const __nv_bfloat16* __restrict__ vc, const int* __restrict__ idx,
                    const int* __restrict__ counts, int S_max, const int* __restrict__ kv_len, SeqMap sm,
                    int Hq, int Hkv, int G, int L_max, int bs, float scale_log2,
                    __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int* __restrict__ err) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, c4 = lane & 3;
    const int t = blockIdx.x * 4 + warp;
    const int b = blockIdx.y / Hkv, g = blockIdx.y % Hkv;
    const int Tq = sm.len(b), tok = sm.tok0(b);
    const int L = kv_len[b];
    if (Tq < 0 || Tq > sm.Tq || (t < Tq && (L < Tq || L > L_max))) {
        if (lane == 0) raise_error(err, kDevErrIndex);
        return;
    }
    if (t >= Tq) return;
    const int pos = L - Tq + t;
    const int bt = pos / bs;
    QFrag<D> Q;
    const size_t q_off = ((static_cast<size_t>(tok) + t) * Hq + static_cast<size_t>(g) * G) * D;
    load_q(Q, q + q_off, D, G);
    WarpAcc<D> A;
    acc_init(A);
    const size_t sel_row = sm.sel(b, g, Hkv, t);
    int nsel = idx != nullptr ? counts[sel_row] : bt + 1;
    if (idx != nullptr && (nsel < 0 || nsel > S_max)) {  // a caller-written count outside its idx row
        if (lane == 0) raise_error(err, kDevErrIndex);
        nsel = nsel < 0 ? 0 : S_max;
    }
    const int* list = idx != nullptr ? idx + static_cast<size_t>(sel_row) * S_max : nullptr;
    const size_t head_base = (static_cast<size_t>(b) * Hkv + g) * L_max;
    const int limit = pos + 1;  // keys x < limit (pos < L always)
    for (int r = 0; r < nsel; ++r) {
        const int blk = list != nullptr ? list[r] : r;
        if (blk < 0 || blk > bt) {
            if (lane == 0) raise_error(err, kDevErrIndex);
            continue;
        }
        for (int x0 = blk * bs; x0 < (blk + 1) * bs; x0 += 32) {
            const int n_ok = limit - x0;
            if (n_ok <= 0) break;
            const uint32_t valid = n_ok >= 32 ? 0xffffffffu : ((1u << n_ok) - 1u);
            attend32(A, Q, kc + (head_base + x0) * D, vc + (head_base + x0) * D, valid, scale_log2);
        }
    }
    acc_finish_rowsum(A);
    // ---- normalise and store: this lane owns D/4 consecutive elements of rows g8 and g8+8
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = g8 + 8 * half;
        if (r >= G) continue;
        const float inv = A.l[half] > 0.f ? 1.f / A.l[half] : 0.f;
        __nv_bfloat16* dst = o + q_off + static_cast<size_t>(r) * D + (D / 4) * c4;
        uint32_t w[D / 8];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2)
#pragma unroll
            for (int nt = 0; nt < D / 8; nt += 2)
                w[(e2 * (D / 8) + nt) / 2] =
                    pack_bf16x2(A.o[nt][2 * half + e2] * inv, A.o[nt + 1][2 * half + e2] * inv);
#pragma unroll
        for (int u = 0; u < D / 32; ++u)
            reinterpret_cast<uint4*>(dst)[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        if (lse != nullptr && c4 == 0)
            lse[sm.lse(b, g * G + r, Hq, t)] =
                A.l[half] > 0.f ? (A.m[half] + log2f(A.l[half])) * 0.69314718055994530942f : -INFINITY;
    }
}

cudaError_t launch_prefill_attention(const PrefillArgs& a) {
    if (tc_prefill_supported(a)) {
        // tensor-core path; shapes it cannot hold in shared memory fall through to the warp path
        const cudaError_t e = launch_prefill_tc(a);
        if (e != cudaErrorInvalidValue) return e;
        (void)cudaGetLastError();
    }
    const int G = a.Hq / a.Hkv;
    const float scale_log2 = a.p.scale * 1.4426950408889634f;
    const SeqMap sm = a.seqmap();
    dim3 grid((a.Tq + 3) / 4, a.B * a.Hkv);
    const auto* qp = static_cast<const __nv_bfloat16*>(a.q);
    const auto* kp = static_cast<const __nv_bfloat16*>(a.k_cache);
    const auto* vp = static_cast<const __nv_bfloat16*>(a.v_cache);
    auto* op = static_cast<__nv_bfloat16*>(a.o);
    if (a.d == 128)
        prefill_warp_kernel<128><<<grid, 128, 0, a.stream>>>(qp, kp, vp, a.idx, a.counts, a.S_max, a.kv_len, sm,
                                                             a.Hq, a.Hkv, G, a.L_max, a.p.block_size, scale_log2,
                                                             op, a.lse, a.err);
    else
        prefill_warp_kernel<64><<<grid, 128, 0, a.stream>>>(qp, kp, vp, a.idx, a.counts, a.S_max, a.kv_len, sm,
                                                            a.Hq, a.Hkv, G, a.L_max, a.p.block_size, scale_log2,
                                                            op, a.lse, a.err);
    return cudaGetLastError();
}

}  // namespace infllmv2
