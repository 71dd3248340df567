// bwd.cu -- gradients of block-sparse attention over a fixed selection (InfLLM v2 is trainable
// sparse attention: "MiniCPM4：如何在手机电脑上高效运行大语言模型", section 1.1; the selection is a
// discrete choice, so the gradient flows through the attention over the selected keys).
//
// For a row (token t, head h) with softmax weights p over its keys and D = dO . O:
//   dS = P o (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// Steps, all on the caller's stream:
//   1. bwd_rowdot_kernel: D for every (token, head) from the forward's bf16 O and dO (and, beside
//      it, lse * log2 e in the same row order for the tensor-core kernel).
//   2. bwd_count / scan / fill kernels: the inverse of the selection, per (sequence, KV head,
//      block) the chunk tokens that chose it (so dK, dV are summed per key block without
//      per-element atomics); bwd_units_kernel cuts the lists into work units of at most
//      kBwdUnitTok tokens.
// With head dim 128, block size 128 and 16 query heads per KV head the gradients come from the
// tensor-core kernel of bwd_tc.cu; otherwise from two warp-MMA kernels:
//   3. bwd_dq_kernel: one warp per (token, KV head) = the G query heads of a selection (16 MMA
//      rows): S = Q K^T and dP = dO V^T recomputed per 32-key tile with m16n8k16 MMAs, P from the
//      forward's lse, dQ += dS K.
//   4. bwd_dkdv_kernel: one CTA per (key block, slice of its token list), one warp per 16 keys:
//      per attending token, S^T = K Q^T and dP^T = V dO^T, then dV += P^T dO and dK += dS^T Q with
//      the token's Q and dO staged in padded shared memory and read transposed by ldmatrix; the
//      slices of a block add their sums into fp32 dK, dV (zeroed first).
// P and dS enter the MMAs as bf16 (the usual flash-attention backward precision); every sum is
// fp32.
#include "attn_warp.cuh"
#include "internal.h"

namespace infllmv2 {

constexpr int kBwdSplit = 128;  // tokens of a block's list per dK/dV CTA

// ---- 1. D = dO . O per (token, head); with `ld`, also (lse * log2 e, D) per row.  d / 8 threads
// per row, 16 bytes of O and of dO each.
__global__ void bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                  const float* __restrict__ lse, int rows, int Tq, int Hq, int d, float* __restrict__ D,
                                  float2* __restrict__ ld) {
    const int tpr = d / 8;  // 8 or 16: a power of two dividing the warp
    const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
    const int row = gtid / tpr, part = gtid % tpr;
    const bool live = row < rows;
    float acc = 0.f;
    if (live) {
        const uint4 a = ldg_v4(o + static_cast<size_t>(row) * d + 8 * part);
        const uint4 b = ldg_v4(dout + static_cast<size_t>(row) * d + 8 * part);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) acc += bf16_lo(aw[e]) * bf16_lo(bw[e]) + bf16_hi(aw[e]) * bf16_hi(bw[e]);
    }
    for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && part == 0) {
        D[row] = acc;
        if (ld != nullptr) {
            const int h = row % Hq, bt = row / Hq;  // row (b*Tq + t)*Hq + h; lse is [B][Hq][Tq]
            const int bb = bt / Tq, t = bt % Tq;
            ld[row] = make_float2(lse[(static_cast<size_t>(bb) * Hq + h) * Tq + t] * 1.4426950408889634f, acc);
        }
    }
}

// ---- 2. inverse selection: count, scan, fill
// Entry (row, r) of the selection: row = (b*Hkv + g)*Tq + t; block idx[row][r] (r < counts[row]),
// or every block 0..bt when idx is null.
__device__ __forceinline__ int bwd_entry(const int* idx, const int* counts, int S_max, int row, int r, int bt,
                                         int nblk, int* err) {
    if (idx == nullptr) return r <= bt ? r : -1;
    const int cnt = counts[row];
    if (cnt < 0 || cnt > S_max || cnt > nblk) {  // (more entries than blocks: duplicates)
        if (r == 0) raise_error(err, kDevErrIndex);
        return -1;
    }
    if (r >= cnt) return -1;
    const int blk = idx[static_cast<size_t>(row) * S_max + r];
    if (blk < 0 || blk > bt) {
        raise_error(err, kDevErrIndex);
        return -1;
    }
    return blk;
}

// Entry e = r * n_rows + row (rows fastest): a warp sees 32 consecutive tokens at the same
// selection slot, which mostly name the same few blocks (the selection lists are ascending), so the
// per-block counters are bumped once per distinct block of the warp.
__device__ __forceinline__ int bwd_entry_at(const int* idx, const int* counts, int S_max, const int* kv_len, int B,
                                            int Tq, int Hkv, int L_max, int bs, int per_row, int nblk, long long e,
                                            int* err, int* row_out) {
    const int n_rows = B * Hkv * Tq;
    const int row = static_cast<int>(e % n_rows), r = static_cast<int>(e / n_rows);
    *row_out = row;
    if (r >= per_row) return -1;
    const int b = row / (Hkv * Tq);
    const int L = kv_len[b];
    if (L < Tq || L > L_max) {
        if (r == 0 && row % (Hkv * Tq) == 0) raise_error(err, kDevErrIndex);
        return -1;
    }
    const int t = row % Tq;
    const int bt = (L - Tq + t) / bs;
    return bwd_entry(idx, counts, S_max, row, r, bt, nblk, err);
}

__global__ void bwd_count_kernel(const int* __restrict__ idx, const int* __restrict__ counts, int S_max,
                                 const int* __restrict__ kv_len, int B, int Tq, int Hkv, int L_max, int bs, int per_row,
                                 int nblk, int* __restrict__ bcnt, int* __restrict__ err) {
    const long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long n = static_cast<long long>(B) * Hkv * Tq * per_row;
    int row = 0;
    const int blk = e < n ? bwd_entry_at(idx, counts, S_max, kv_len, B, Tq, Hkv, L_max, bs, per_row, nblk, e, err, &row)
                          : -1;
    const int key = blk >= 0 ? (row / Tq) * nblk + blk : -1;
    const unsigned same = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&bcnt[key], __popc(same));
}

// Exclusive scans of one (b, g)'s block counts -> token offsets boff [nblk + 1], and of the units
// per block (ceil(count / kBwdUnitTok)) -> unit offsets uoff [nblk + 1].
__global__ void __launch_bounds__(1024) bwd_scan_kernel(const int* __restrict__ bcnt, int nblk, int* __restrict__ boff,
                                                        int* __restrict__ uoff) {
    __shared__ int s_warp[2][32];
    __shared__ int s_carry[2];
    const int bg = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int* c = bcnt + static_cast<size_t>(bg) * nblk;
    int* out = boff + static_cast<size_t>(bg) * (nblk + 1);
    int* uout = uoff + static_cast<size_t>(bg) * (nblk + 1);
    if (tid < 2) s_carry[tid] = 0;
    __syncthreads();
    for (int base = 0; base < nblk; base += 1024) {
        const int i = base + tid;
        const int v0 = i < nblk ? c[i] : 0;
        const int v1 = (v0 + kBwdUnitTok - 1) / kBwdUnitTok;
        int a0 = v0, a1 = v1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int x0 = __shfl_up_sync(0xffffffffu, a0, off);
            const int x1 = __shfl_up_sync(0xffffffffu, a1, off);
            if (lane >= off) {
                a0 += x0;
                a1 += x1;
            }
        }
        if (lane == 31) {
            s_warp[0][warp] = a0;
            s_warp[1][warp] = a1;
        }
        __syncthreads();
        if (warp == 0) {
            int w0 = s_warp[0][lane], w1 = s_warp[1][lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int x0 = __shfl_up_sync(0xffffffffu, w0, off);
                const int x1 = __shfl_up_sync(0xffffffffu, w1, off);
                if (lane >= off) {
                    w0 += x0;
                    w1 += x1;
                }
            }
            s_warp[0][lane] = w0;  // inclusive over warps
            s_warp[1][lane] = w1;
        }
        __syncthreads();
        const int before0 = s_carry[0] + (warp > 0 ? s_warp[0][warp - 1] : 0) + a0 - v0;
        const int before1 = s_carry[1] + (warp > 0 ? s_warp[1][warp - 1] : 0) + a1 - v1;
        if (i < nblk) {
            out[i] = before0;
            uout[i] = before1;
        }
        __syncthreads();
        if (tid == 1023) {
            s_carry[0] = before0 + v0;
            s_carry[1] = before1 + v1;
        }
        __syncthreads();
    }
    if (tid == 0) {
        out[nblk] = s_carry[0];
        uout[nblk] = s_carry[1];
    }
}

__global__ void bwd_fill_kernel(const int* __restrict__ idx, const int* __restrict__ counts, int S_max,
                                const int* __restrict__ kv_len, int B, int Tq, int Hkv, int L_max, int bs, int per_row,
                                int nblk, const int* __restrict__ boff, int* __restrict__ cursor,
                                int* __restrict__ list, long long list_stride, int* __restrict__ err) {
    const long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long n = static_cast<long long>(B) * Hkv * Tq * per_row;
    int row = 0;
    const int blk = e < n ? bwd_entry_at(idx, counts, S_max, kv_len, B, Tq, Hkv, L_max, bs, per_row, nblk, e, nullptr,
                                         &row)
                          : -1;
    const int bg = row / Tq;
    const int key = blk >= 0 ? bg * nblk + blk : -1;
    const unsigned same = __match_any_sync(0xffffffffu, key);
    const int lane = threadIdx.x & 31, leader = __ffs(same) - 1;
    int at = 0;
    if (key >= 0 && lane == leader) at = atomicAdd(&cursor[key], __popc(same));
    at = __shfl_sync(same, at, leader) + __popc(same & ((1u << lane) - 1u));
    if (key >= 0) list[bg * list_stride + boff[static_cast<size_t>(bg) * (nblk + 1) + blk] + at] = row % Tq;
}

// Work units {b*Hkv + g, block, first, end}: each block's token list cut into slices of at most
// kBwdUnitTok tokens, ordered by (b, g), then block.
__global__ void bwd_units_kernel(const int* __restrict__ boff, const int* __restrict__ uoff, int rows, int nblk,
                                 int4* __restrict__ units) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= rows * nblk) return;
    const int bg = e / nblk, blk = e % nblk;
    int ubase = 0;
    for (int r = 0; r < bg; ++r) ubase += uoff[static_cast<size_t>(r) * (nblk + 1) + nblk];
    const int* bo = boff + static_cast<size_t>(bg) * (nblk + 1);
    const int first = bo[blk], end = bo[blk + 1];
    int u = ubase + uoff[static_cast<size_t>(bg) * (nblk + 1) + blk];
    for (int s = first; s < end; s += kBwdUnitTok, ++u) units[u] = make_int4(bg, blk, s, min(s + kBwdUnitTok, end));
}

// ---- 3. dQ: one warp per (b, t, g)
template <int D>
__global__ void __launch_bounds__(128)
bwd_dq_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cache,
              const __nv_bfloat16* __restrict__ v_cache, const __nv_bfloat16* __restrict__ dout,
              const float* __restrict__ lse, const float* __restrict__ Drow, const int* __restrict__ idx,
              const int* __restrict__ counts, int S_max, const int* __restrict__ kv_len, int B, int Tq, int Hq,
              int Hkv, int L_max, int bs, float scale, float* __restrict__ dq, int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (wid >= B * Tq * Hkv) return;
    const int g = wid % Hkv, t = (wid / Hkv) % Tq, b = wid / (Hkv * Tq);
    const int G = Hq / Hkv;
    const int gq = lane >> 2, cq = lane & 3;
    const int L = kv_len[b];
    if (L < Tq || L > L_max) return;  // reported by the count kernel
    const int pos = L - Tq + t;
    const int bt = pos / bs;
    const float scale_log2 = scale * 1.4426950408889634f;
    const size_t qrow = (static_cast<size_t>(b) * Tq + t) * Hq + static_cast<size_t>(g) * G;
    QFrag<D> Q, dO;
    load_q(Q, q + qrow * D, D, G);
    load_q(dO, dout + qrow * D, D, G);
    float lse2[2], Dr[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int h = gq + 8 * half;
        lse2[half] = h < G ? lse[(static_cast<size_t>(b) * Hq + g * G + h) * Tq + t] * 1.4426950408889634f : INFINITY;
        Dr[half] = h < G ? Drow[qrow + h] : 0.f;
    }
    float acc[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    const int row = (b * Hkv + g) * Tq + t;
    const int nsel = idx != nullptr ? min(min(max(counts[row], 0), S_max), (L_max + bs - 1) / bs) : bt + 1;
    const size_t cache0 = static_cast<size_t>(b * Hkv + g) * L_max;
    constexpr int VW = D / 16;
    for (int r = 0; r < nsel; ++r) {
        const int blk = idx != nullptr ? idx[static_cast<size_t>(row) * S_max + r] : r;
        if (blk < 0 || blk > bt) continue;  // reported by the count kernel
        for (int r0 = 0; r0 < bs; r0 += 32) {
            const int x0 = blk * bs + r0;
            const int n_ok = min(pos, L - 1) - x0 + 1;
            if (n_ok <= 0) break;
            const uint32_t valid = n_ok >= 32 ? 0xffffffffu : ((1u << n_ok) - 1u);
            const __nv_bfloat16* krow = k_cache + (cache0 + x0) * D;
            const __nv_bfloat16* vrow = v_cache + (cache0 + x0) * D;
            // K and V rows in the QK^T layout (16 bytes of key nt*8 + gq at 32i + 8cq)
            uint4 kw[4][D / 32], vq[4][D / 32];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int key = nt * 8 + gq;
                const bool ok = (valid >> key) & 1u;
#pragma unroll
                for (int i = 0; i < D / 32; ++i) {
                    kw[nt][i] = ok ? ldg_v4(krow + static_cast<size_t>(key) * D + 32 * i + 8 * cq) : make_uint4(0, 0, 0, 0);
                    vq[nt][i] = ok ? ldg_v4(vrow + static_cast<size_t>(key) * D + 32 * i + 8 * cq) : make_uint4(0, 0, 0, 0);
                }
            }
            float s[4][4], dp[4][4];
            qk_tiles<D>(s, Q, kw);
            qk_tiles<D>(dp, dO, vq);
            // dS = P (dP - D) as the A operand of dQ += dS K
            uint32_t da[2][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = nt * 8 + 2 * cq + (e & 1);
                    const float p = ((valid >> key) & 1u) ? fast_exp2(s[nt][e] * scale_log2 - lse2[e >> 1]) : 0.f;
                    v[e] = p * (dp[nt][e] - Dr[e >> 1]);
                }
                const int kk = nt >> 1, hi = nt & 1;
                da[kk][2 * hi + 0] = pack_bf16x2(v[0], v[1]);
                da[kk][2 * hi + 1] = pack_bf16x2(v[2], v[3]);
            }
            // K rows in the PV layout: lane reads D/8 consecutive elements of its four rows
            uint32_t kp[2][4][VW];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int key = 16 * kk + 2 * cq + (rr & 1) + 8 * (rr >> 1);
                    const bool ok = (valid >> key) & 1u;
                    const uint4* src = reinterpret_cast<const uint4*>(krow + static_cast<size_t>(key) * D + (D / 8) * gq);
#pragma unroll
                    for (int u = 0; u < VW / 4; ++u) {
                        const uint4 w = ok ? ldg_v4(src + u) : make_uint4(0, 0, 0, 0);
                        kp[kk][rr][4 * u + 0] = w.x;
                        kp[kk][rr][4 * u + 1] = w.y;
                        kp[kk][rr][4 * u + 2] = w.z;
                        kp[kk][rr][4 * u + 3] = w.w;
                    }
                }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    const uint32_t b0 = pair_halves(kp[kk][0][nt >> 1], kp[kk][1][nt >> 1], nt & 1);
                    const uint32_t b1 = pair_halves(kp[kk][2][nt >> 1], kp[kk][3][nt >> 1], nt & 1);
                    mma_16816(acc[nt], da[kk], b0, b1);
                }
        }
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int h = gq + 8 * (e >> 1);
            if (h < G) dq[(qrow + h) * D + o_col(D, cq, nt, e)] = acc[nt][e] * scale;
        }
}

// ---- 4. dK, dV: one CTA per (key block, slice of its token list), one warp per 16 keys
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <int D, int BS>
__global__ void __launch_bounds__(BS * 2)
bwd_dkdv_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cache,
                const __nv_bfloat16* __restrict__ v_cache, const __nv_bfloat16* __restrict__ dout,
                const float* __restrict__ lse, const float* __restrict__ Drow, const int* __restrict__ kv_len,
                int Tq, int Hq, int Hkv, int L_max, int nblk, int max_splits, const int* __restrict__ boff,
                const int* __restrict__ list, long long list_stride, float scale, float* __restrict__ dk,
                float* __restrict__ dv) {
    constexpr int kPad = D + 8;  // bf16 per staged row: 16-byte rows, conflict-free ldmatrix
    __shared__ __align__(16) __nv_bfloat16 s_q[16][kPad];
    __shared__ __align__(16) __nv_bfloat16 s_do[16][kPad];
    __shared__ float s_lse2[16], s_D[16];
    const int bg = blockIdx.y;
    const int blk = blockIdx.x / max_splits, split = blockIdx.x % max_splits;
    const int b = bg / Hkv, g = bg % Hkv;
    const int G = Hq / Hkv;
    const int L = kv_len[b];
    if (L < Tq || L > L_max) return;
    const int* off = boff + static_cast<size_t>(bg) * (nblk + 1);
    const int lo = off[blk] + split * kBwdSplit, hi = min(off[blk + 1], lo + kBwdSplit);
    if (lo >= hi) return;
    const int* toks = list + bg * list_stride;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int key0 = blk * BS + 16 * warp;  // this warp's 16 keys
    const size_t cache0 = static_cast<size_t>(bg) * L_max;
    const float scale_log2 = scale * 1.4426950408889634f;
    // K and V of the warp's keys as A fragments (rows = keys; past the cache: zero, masked below)
    QFrag<D> KA, VA;
    {
        const int nk = max(0, min(16, L - key0));  // rows past the cache read as zero (not loaded)
        load_q(KA, k_cache + (cache0 + key0) * D, D, nk);
        load_q(VA, v_cache + (cache0 + key0) * D, D, nk);
    }
    float akv[D / 8][4], akk[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) akv[nt][e] = akk[nt][e] = 0.f;
    const uint32_t sq_base = smem_u32(&s_q[0][0]), sdo_base = smem_u32(&s_do[0][0]);
    for (int it = lo; it < hi; ++it) {
        const int t = toks[it];
        const int pos = L - Tq + t;
        const size_t qrow = (static_cast<size_t>(b) * Tq + t) * Hq + static_cast<size_t>(g) * G;
        __syncthreads();  // the previous token's rows are no longer read
        for (int e = tid; e < 16 * (D / 8); e += BS * 2) {
            const int h = e / (D / 8), c8 = (e % (D / 8)) * 8;
            uint4 wq = make_uint4(0, 0, 0, 0), wd = make_uint4(0, 0, 0, 0);
            if (h < G) {
                wq = ldg_v4(q + (qrow + h) * D + c8);
                wd = ldg_v4(dout + (qrow + h) * D + c8);
            }
            *reinterpret_cast<uint4*>(&s_q[h][c8]) = wq;
            *reinterpret_cast<uint4*>(&s_do[h][c8]) = wd;
        }
        if (tid < 16) {
            const int h = tid;
            s_lse2[h] = h < G ? lse[(static_cast<size_t>(b) * Hq + g * G + h) * Tq + t] * 1.4426950408889634f : INFINITY;
            s_D[h] = h < G ? Drow[qrow + h] : 0.f;
        }
        __syncthreads();
        // S^T = K Q^T, dP^T = V dO^T: rows = keys, columns = heads (two n-tiles of 8)
        float st[2][4], dpt[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) st[nt][e] = dpt[nt][e] = 0.f;
            const int h = nt * 8 + gq;
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
                const uint4 wq = lds_v4(sq_base + (h * kPad + 32 * i + 8 * cq) * 2);
                const uint4 wd = lds_v4(sdo_base + (h * kPad + 32 * i + 8 * cq) * 2);
                mma_16816(st[nt], KA.a[2 * i], wq.x, wq.y);
                mma_16816(st[nt], KA.a[2 * i + 1], wq.z, wq.w);
                mma_16816(dpt[nt], VA.a[2 * i], wd.x, wd.y);
                mma_16816(dpt[nt], VA.a[2 * i + 1], wd.z, wd.w);
            }
        }
        // P^T and dS^T (keys past the token or the cache, and padding heads, are zero)
        uint32_t pa[4], da[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float pv[4], dv4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + gq + 8 * (e >> 1);
                const int h = nt * 8 + 2 * cq + (e & 1);
                const bool ok = key <= pos && key < L && h < G;
                const float p = ok ? fast_exp2(st[nt][e] * scale_log2 - s_lse2[h]) : 0.f;
                pv[e] = p;
                dv4[e] = p * (dpt[nt][e] - s_D[h]);
            }
            pa[2 * nt + 0] = pack_bf16x2(pv[0], pv[1]);
            pa[2 * nt + 1] = pack_bf16x2(pv[2], pv[3]);
            da[2 * nt + 0] = pack_bf16x2(dv4[0], dv4[1]);
            da[2 * nt + 1] = pack_bf16x2(dv4[2], dv4[3]);
        }
        // dV += P^T dO, dK += dS^T Q: B = the staged rows read transposed (k = head, n = column)
        const int mrow = lane & 15, mcol = (lane >> 4) * 8;  // ldmatrix row of lanes 0-15 / 16-31
#pragma unroll
        for (int nt = 0; nt < D / 8; nt += 2) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(sdo_base + (mrow * kPad + nt * 8 + mcol) * 2, b0, b1, b2, b3);
            mma_16816(akv[nt], pa, b0, b1);
            mma_16816(akv[nt + 1], pa, b2, b3);
            ldmatrix_x4_trans(sq_base + (mrow * kPad + nt * 8 + mcol) * 2, b0, b1, b2, b3);
            mma_16816(akk[nt], da, b0, b1);
            mma_16816(akk[nt + 1], da, b2, b3);
        }
    }
    // sums of this slice into dK, dV (fp32, zeroed before the launch)
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int key = key0 + gq + 8 * (e >> 1);
            if (key >= L) continue;
            const int col = nt * 8 + 2 * cq + (e & 1);
            atomicAdd(&dv[(cache0 + key) * D + col], akv[nt][e]);
            atomicAdd(&dk[(cache0 + key) * D + col], akk[nt][e] * scale);
        }
}

// Workspace: D [B*Tq*Hq] | (lse log2e, D) [B*Tq*Hq] | block counts | cursors | work counter |
// token offsets | unit offsets | token lists | units; every part 256-byte aligned.
struct BwdWs {
    size_t D, ld, bcnt, cursor, counter, boff, uoff, list, units, total;
    int nblk;
    long long list_stride;
};

static BwdWs bwd_ws(int B, int Tq, int Hq, int Hkv, int L_max, int bs) {
    auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    BwdWs w{};
    w.nblk = (L_max + bs - 1) / bs;
    const size_t rows = static_cast<size_t>(B) * Hkv, nblk = static_cast<size_t>(w.nblk);
    const size_t qrows = static_cast<size_t>(B) * Tq * Hq;
    w.list_stride = static_cast<long long>(Tq) * w.nblk;
    const size_t max_units = rows * (static_cast<size_t>(Tq) * nblk / kBwdUnitTok + nblk + 1);
    size_t o = 0;
    w.D = o;       o += al(qrows * 4);
    w.ld = o;      o += al(qrows * 8);
    w.bcnt = o;    o += al(rows * nblk * 4);
    w.cursor = o;  o += al(rows * nblk * 4);
    w.counter = o; o += 256;
    w.boff = o;    o += al(rows * (nblk + 1) * 4);
    w.uoff = o;    o += al(rows * (nblk + 1) * 4);
    w.list = o;    o += al(rows * static_cast<size_t>(Tq) * nblk * 4);
    w.units = o;   o += al(max_units * 16);
    w.total = o;
    return w;
}

size_t bwd_workspace_bytes(int B, int Tq, int Hq, int Hkv, int L_max, int bs) {
    return bwd_ws(B, Tq, Hq, Hkv, L_max, bs).total;
}

template <int D, int BS>
static cudaError_t launch_bwd_t(const BwdArgs& a) {
    const BwdWs w = bwd_ws(a.B, a.Tq, a.Hq, a.Hkv, a.L_max, BS);
    const int nblk = w.nblk;
    const size_t rows = static_cast<size_t>(a.B) * a.Hkv;
    char* ws = static_cast<char*>(a.workspace);
    float* Dr = reinterpret_cast<float*>(ws + w.D);
    float2* ld = reinterpret_cast<float2*>(ws + w.ld);
    int* bcnt = reinterpret_cast<int*>(ws + w.bcnt);
    int* cursor = reinterpret_cast<int*>(ws + w.cursor);
    int* counter = reinterpret_cast<int*>(ws + w.counter);
    int* boff = reinterpret_cast<int*>(ws + w.boff);
    int* uoff = reinterpret_cast<int*>(ws + w.uoff);
    int* list = reinterpret_cast<int*>(ws + w.list);
    int4* units = reinterpret_cast<int4*>(ws + w.units);
    const long long list_stride = w.list_stride;
    const bool tc = bwd_tc_supported(a);
    const float scale = a.p.scale;
    cudaStream_t st = a.stream;
    cudaError_t e;
    if ((e = cudaMemsetAsync(ws + w.bcnt, 0, w.boff - w.bcnt, st)) != cudaSuccess) return e;  // counts, cursors, counter
    const size_t cache = rows * a.L_max * D * sizeof(float);
    if ((e = cudaMemsetAsync(a.dk, 0, cache, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.dv, 0, cache, st)) != cudaSuccess) return e;
    const int qrows = a.B * a.Tq * a.Hq;
    if (tc && (e = cudaMemsetAsync(a.dq, 0, static_cast<size_t>(qrows) * D * sizeof(float), st)) != cudaSuccess)
        return e;
    bwd_rowdot_kernel<<<static_cast<unsigned>((static_cast<long long>(qrows) * (D / 8) + 255) / 256), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(a.o),
                                                              static_cast<const __nv_bfloat16*>(a.dout), a.lse, qrows,
                                                              a.Tq, a.Hq, D, Dr, tc ? ld : nullptr);
    const int per_row = a.idx != nullptr ? a.S_max : nblk;
    const long long entries = static_cast<long long>(rows) * a.Tq * per_row;
    const unsigned eb = static_cast<unsigned>((entries + 255) / 256);
    bwd_count_kernel<<<eb, 256, 0, st>>>(a.idx, a.counts, a.S_max, a.kv_len, a.B, a.Tq, a.Hkv, a.L_max, BS, per_row,
                                         nblk, bcnt, a.err);
    bwd_scan_kernel<<<static_cast<unsigned>(rows), 1024, 0, st>>>(bcnt, nblk, boff, uoff);
    bwd_fill_kernel<<<eb, 256, 0, st>>>(a.idx, a.counts, a.S_max, a.kv_len, a.B, a.Tq, a.Hkv, a.L_max, BS, per_row,
                                        nblk, boff, cursor, list, list_stride, a.err);
    if (tc) {
        const int pairs = static_cast<int>(rows) * nblk;
        bwd_units_kernel<<<(pairs + 255) / 256, 256, 0, st>>>(boff, uoff, static_cast<int>(rows), nblk, units);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        prof_mark(st, "bwd_prep");
        e = launch_bwd_tc(a, BwdTcWork{ld, units, uoff, list, list_stride, nblk, counter});
        prof_mark(st, "bwd_grad");
        return e;
    }
    prof_mark(st, "bwd_prep");
    const int warps = a.B * a.Tq * a.Hkv;
    bwd_dq_kernel<D><<<(warps + 3) / 4, 128, 0, st>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_cache),
        static_cast<const __nv_bfloat16*>(a.v_cache), static_cast<const __nv_bfloat16*>(a.dout), a.lse, Dr, a.idx,
        a.counts, a.S_max, a.kv_len, a.B, a.Tq, a.Hq, a.Hkv, a.L_max, BS, scale, a.dq, a.err);
    const int max_splits = (a.Tq + kBwdSplit - 1) / kBwdSplit;
    bwd_dkdv_kernel<D, BS><<<dim3(nblk * max_splits, static_cast<unsigned>(rows)), BS * 2, 0, st>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_cache),
        static_cast<const __nv_bfloat16*>(a.v_cache), static_cast<const __nv_bfloat16*>(a.dout), a.lse, Dr, a.kv_len,
        a.Tq, a.Hq, a.Hkv, a.L_max, nblk, max_splits, boff, list, list_stride, scale, a.dk, a.dv);
    e = cudaGetLastError();
    prof_mark(st, "bwd_grad");
    return e;
}

cudaError_t launch_attention_bwd(const BwdArgs& a) {
    const int bs = a.p.block_size;
    if (a.d == 128) return bs == 64 ? launch_bwd_t<128, 64>(a) : launch_bwd_t<128, 128>(a);
    return bs == 64 ? launch_bwd_t<64, 64>(a) : launch_bwd_t<64, 128>(a);
}

}  // namespace infllmv2
