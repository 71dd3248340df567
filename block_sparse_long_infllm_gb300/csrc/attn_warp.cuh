// attn_warp.cuh -- one warp's flash-attention state for 16 query rows, fed 32 keys at a time
// (the online-softmax form of "attention on the selected blocks only", "MiniCPM4: 如何在手机
// 电脑上高效运行大语言模型", section 1.1 "InfLLM v2").
//
// Rows are the G heads of one query token (padded to 16).  QK^T and PV run as m16n8k16 warp
// MMAs with fp32 accumulators; the softmax runs in fp32 in the log2 domain.  Operands come
// from global memory with 128-bit loads, or from TMA-filled 128-byte-swizzled shared tiles:
//   * QK^T: the head dimension is permuted the same way for Q and K (the sum over d does
//     not depend on the order of its terms) so each lane's 16 bytes of a K row feed two
//     k-steps of its B fragment;
//   * PV: output column n of n-tile nt is head-dim element (D/8)*n + nt, so each lane
//     reads D/8 consecutive elements of its four V rows and, in the end, owns D/4
//     consecutive output elements of each of its two rows.
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace infllmv2 {

// Key order inside an n-tile of 8 keys: MMA column j holds key key_perm<D>(j) of the tile's 8.
// The B fragments of QK^T give lane (g, c) column g; those of PV give it columns 2c, 2c + 1 (+8).
// In a 128-byte-swizzled shared tile (16-byte chunk x of row y stored at chunk x ^ (y & 7)) the
// eight lanes of one shared-memory wavefront must read eight different chunk positions:
//   * K rows: a lane pair (columns 2q, 2q + 1) reads the same four chunks of two rows, so the two
//     rows must differ in bit 2;
//   * V rows (lanes read head-dim chunks 2 apart for d = 128, 1 apart for d = 64, over the four
//     rows of the even or of the odd columns): the even columns map to rows {0, 1, 4, 5} for
//     d = 128 and {0, 2, 4, 6} for d = 64, the odd ones to the rest.
// In the identity order the K reads (and for d = 128 the V reads) were 2-way bank conflicts.  The
// order of the keys does not change the result: every place that maps a column to a key (loads,
// the valid mask, the scoring's kernel rows) uses this one table.
template <int D>
__device__ __forceinline__ int key_perm(int j) {
    constexpr uint32_t kTable = D == 128 ? 0x35247160u : 0x36147250u;  // [0,6,1,7,4,2,5,3], [0,5,2,7,4,1,6,3]
    return static_cast<int>((kTable >> (4 * j)) & 7u);
}

// One split's fp32 partial of a decode row: running maxima m[16] (log2 domain), row sums l[16]
// and unnormalised outputs o[16][D] for the (up to 16) heads of the row.
template <int D>
struct PartialLayout {
    static constexpr int kFloats = 16 + 16 + 16 * D;
};

template <int D>
struct QFrag {
    uint32_t a[D / 16][4];
};

template <int D>
struct WarpAcc {
    float o[D / 8][4];  // o[nt][0..1]: row g, o[nt][2..3]: row g+8
    float m[2];         // running max of the scaled log2 logits, rows g and g+8
    float l[2];         // this lane's share of the row sums
};

// Load the A fragments of 16 rows; row r's data starts at rows + r*row_stride, rows r >= n_rows
// read as zero.
template <int D>
__device__ __forceinline__ void load_q(QFrag<D>& Q, const __nv_bfloat16* rows, int row_stride, int n_rows) {
    const int g = (threadIdx.x & 31) >> 2, c = threadIdx.x & 3;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = g + 8 * half;
        const bool ok = r < n_rows;
        const __nv_bfloat16* src = rows + static_cast<size_t>(ok ? r : 0) * row_stride + 8 * c;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            const uint4 w = ok ? ldg_v4(src + 32 * i) : make_uint4(0, 0, 0, 0);
            Q.a[2 * i][half] = w.x;
            Q.a[2 * i][2 + half] = w.y;
            Q.a[2 * i + 1][half] = w.z;
            Q.a[2 * i + 1][2 + half] = w.w;
        }
    }
}

template <int D>
__device__ __forceinline__ void acc_init(WarpAcc<D>& A) {
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) A.o[nt][e] = 0.f;
    A.m[0] = A.m[1] = -INFINITY;
    A.l[0] = A.l[1] = 0.f;
}

// Online-softmax update with the scores s (this lane's values of 4 n-tiles x 16 rows x 8 keys,
// unscaled, keys masked by `valid`) and the V fragments vw of the same 32 keys, then O += P V.
template <int D>
__device__ __forceinline__ void softmax_pv(WarpAcc<D>& A, float (&s)[4][4], const uint32_t (&vw)[2][4][D / 16],
                                           uint32_t valid, float scale_log2) {
    const int c = threadIdx.x & 3;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int key = nt * 8 + key_perm<D>(2 * c + (e & 1));
            s[nt][e] = ((valid >> key) & 1u) ? s[nt][e] * scale_log2 : -INFINITY;
            mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
        }
    }
    float ref[2], corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float m_new = fmaxf(A.m[h], mx[h]);
        ref[h] = m_new == -INFINITY ? 0.f : m_new;
        corr[h] = fast_exp2(A.m[h] - ref[h]);
        A.m[h] = m_new;
        A.l[h] *= corr[h];
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        A.o[nt][0] *= corr[0];
        A.o[nt][1] *= corr[0];
        A.o[nt][2] *= corr[1];
        A.o[nt][3] *= corr[1];
    }
    uint32_t pa[2][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            pv[e] = fast_exp2(s[nt][e] - ref[e >> 1]);
            A.l[e >> 1] += pv[e];
        }
        const int kk = nt >> 1, hi = nt & 1;
        pa[kk][2 * hi + 0] = pack_bf16x2(pv[0], pv[1]);
        pa[kk][2 * hi + 1] = pack_bf16x2(pv[2], pv[3]);
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
            const uint32_t b0 = pair_halves(vw[kk][0][nt >> 1], vw[kk][1][nt >> 1], nt & 1);
            const uint32_t b1 = pair_halves(vw[kk][2][nt >> 1], vw[kk][3][nt >> 1], nt & 1);
            mma_16816(A.o[nt], pa[kk], b0, b1);
        }
    }
}

// S = Q K^T for 4 n-tiles of 8 keys from per-lane 16-byte K slices kw[nt][i] (head-dim
// elements 32i + 8c .. +7 of key nt*8 + g).
template <int D>
__device__ __forceinline__ void qk_tiles(float (&s)[4][4], const QFrag<D>& Q, const uint4 (&kw)[4][D / 32]) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            mma_16816(s[nt], Q.a[2 * i], kw[nt][i].x, kw[nt][i].y);
            mma_16816(s[nt], Q.a[2 * i + 1], kw[nt][i].z, kw[nt][i].w);
        }
    }
}

// Feed 32 keys whose rows are k_rows[kk*D], v_rows[kk*D] (kk = 0..31) in global memory; bit kk
// of `valid` says key kk takes part.  Rows of keys that do not take part are never read.
template <int D>
__device__ __forceinline__ void attend32(WarpAcc<D>& A, const QFrag<D>& Q, const __nv_bfloat16* k_rows,
                                         const __nv_bfloat16* v_rows, uint32_t valid, float scale_log2) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    constexpr int VW = D / 16;  // 32-bit words per lane per V row
    uint32_t vw[2][4][VW];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int key = 16 * kk + 8 * (r >> 1) + key_perm<D>(2 * c + (r & 1));
            const bool ok = (valid >> key) & 1u;
            const uint4* src = reinterpret_cast<const uint4*>(v_rows + static_cast<size_t>(key) * D + (D / 8) * g);
#pragma unroll
            for (int u = 0; u < VW / 4; ++u) {
                const uint4 w = ok ? ldg_v4_stream(src + u) : make_uint4(0, 0, 0, 0);
                vw[kk][r][4 * u + 0] = w.x;
                vw[kk][r][4 * u + 1] = w.y;
                vw[kk][r][4 * u + 2] = w.z;
                vw[kk][r][4 * u + 3] = w.w;
            }
        }
    }
    uint4 kw[4][D / 32];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int key = nt * 8 + key_perm<D>(g);
        const bool ok = (valid >> key) & 1u;
        const __nv_bfloat16* src = k_rows + static_cast<size_t>(key) * D + 8 * c;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) kw[nt][i] = ok ? ldg_v4_stream(src + 32 * i) : make_uint4(0, 0, 0, 0);
    }
    float s[4][4];
    qk_tiles<D>(s, Q, kw);
    softmax_pv<D>(A, s, vw, valid, scale_log2);
}

// Same for 32 keys starting at row `row0` of K and V tiles in shared memory, each stored as
// D/64 boxes of `rows` x 128 bytes with the 128-byte swizzle (tma.cuh), 1024-byte aligned.
// V rows of keys that do not take part read as zero (the cache past kv_len is arbitrary).
template <int D>
__device__ __forceinline__ void attend32_smem(WarpAcc<D>& A, const QFrag<D>& Q, uint32_t k_tile, uint32_t v_tile,
                                              int rows, int row0, uint32_t valid, float scale_log2) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const uint32_t box = static_cast<uint32_t>(rows) * 128u;
    constexpr int VW = D / 16;
    uint32_t vw[2][4][VW];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int key = 16 * kk + 8 * (r >> 1) + key_perm<D>(2 * c + (r & 1));
            const bool ok = (valid >> key) & 1u;
            const int row = row0 + key;
#pragma unroll
            for (int u = 0; u < VW / 4; ++u) {
                // elements (D/8)g + 8u .. +7 of the row: box col/64, chunk (col % 64)/8
                const int col = (D / 8) * g + 8 * u;
                const uint32_t addr = v_tile + (col / 64) * box + swz128(row, (col % 64) / 8);
                const uint4 w = ok ? lds_v4(addr) : make_uint4(0, 0, 0, 0);
                vw[kk][r][4 * u + 0] = w.x;
                vw[kk][r][4 * u + 1] = w.y;
                vw[kk][r][4 * u + 2] = w.z;
                vw[kk][r][4 * u + 3] = w.w;
            }
        }
    }
    uint4 kw[4][D / 32];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int row = row0 + nt * 8 + key_perm<D>(g);
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            const int col = 32 * i + 8 * c;
            kw[nt][i] = lds_v4(k_tile + (col / 64) * box + swz128(row, (col % 64) / 8));
        }
    }
    float s[4][4];
    qk_tiles<D>(s, Q, kw);
    softmax_pv<D>(A, s, vw, valid, scale_log2);
}

// Sum the lanes' shares of the row sums (after the last tile).
template <int D>
__device__ __forceinline__ void acc_finish_rowsum(WarpAcc<D>& A) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        A.l[h] += __shfl_xor_sync(0xffffffffu, A.l[h], 1);
        A.l[h] += __shfl_xor_sync(0xffffffffu, A.l[h], 2);
    }
}

// Head-dim element held in o[nt][e]: row half e>>1, column (D/8)*(2c + (e&1)) + nt.
__device__ __forceinline__ int o_col(int D, int c, int nt, int e) { return (D / 8) * (2 * c + (e & 1)) + nt; }

}  // namespace infllmv2
