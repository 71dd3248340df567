// bwd_tc.cu -- gradients of the block-sparse attention on the 5th-generation tensor cores, for head
// dim 128, block size 128 and 16 query heads per KV head (InfLLM v2 trains through its sparse
// attention: "MiniCPM4: 如何在手机电脑上高效运行大语言模型", section 1.1; the selection is a discrete
// choice held fixed, the gradient flows through the attention over the selected keys).
//
// Work unit: one key block of one (sequence, KV head) and a slice of at most kBwdUnitTok of the
// chunk tokens that selected it (the inverse of the selection, built beforehand).  The unit's K and
// V stay in shared memory while its tokens stream through in tiles of 4 tokens x 16 heads = 64
// query rows.  Per tile, with the block's 128 keys as the MMA rows:
//   S^T  = K Q^T                     TMEM, 64 columns, two buffers
//   dP^T = V dO^T                    TMEM, 64 columns
//   P^T  = exp2(S^T scale log2e - lse log2e)   bf16, written back over its S^T columns (A operand)
//   dS^T = P^T o (dP^T - D)          bf16 into shared memory (K-major A of dK, MN-major B of dQ^T)
//   dV  += P^T dO,  dK += dS^T Q     TMEM accumulators over the unit (128 columns each)
//   dQ^T = K^T dS^T                  TMEM, 64 columns, head dim on the lanes; added into dq from
//                                    registers by fp32 reductions at L2 (a warp covers 32
//                                    consecutive head-dim elements of a row: one 128-byte request)
// At the end of a unit dV and dK (times the softmax scale) are staged as 128-byte-swizzled fp32
// boxes and added into dk and dv by tiled bulk reductions: the slices of one block may run on
// different CTAs, and dq collects the partial sums of every block a token selected.
//
// Roles: warps 0-7 epilogue (warp w owns TMEM lanes 32*(w%4)..+31 -- keys for S, dP, dV, dK and
// head-dim rows for dQ^T -- and query-row half w/4 of the tile), warp 8 issues the MMAs (one lane),
// warp 9 loads (TMA).  The grid is persistent: each CTA takes units from a global counter.  Every
// wait is bounded; one that runs out raises the device error word and an abort flag that ends every
// loop, the MMA and load threads drain what they issued and the TMEM is freed before exit.
#include "internal.h"
#include "umma.cuh"

namespace infllmv2 {

constexpr int kBtTok = 4;              // tokens per tile
constexpr int kBtRows = 16 * kBtTok;   // query rows per tile (4 tokens x 16 heads)
constexpr int kBtStages = 3;           // Q / dO tiles in flight
constexpr int kBtThreads = 320;        // 8 epilogue warps, MMA warp, load warp

template <int D, int BS>
struct BtSmem {
    static constexpr int kKV = BS * D * 2;                       // K or V block
    static constexpr int kTile = kBtRows * D * 2;                // Q or dO tile
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKV;
    static constexpr int kRingOff = 2 * kKV;                     // [stage] {Q, dO}
    static constexpr int kDsOff = kRingOff + kBtStages * 2 * kTile;  // dS^T: BS rows x 64 bf16
    static constexpr int kFlushOff = kRingOff;                   // dV, dK staging over ring and dS
    static constexpr int kLdOff = kFlushOff + 2 * BS * D * 4;    // [stage][64] (lse log2e, D)
    static constexpr int kTokOff = kLdOff + kBtStages * kBtRows * 8;  // the unit's tokens
    static constexpr int kMiscOff = kTokOff + kBwdUnitTok * 4;   // unit {bg, blk, count}, tmem base, abort
    static constexpr int kBarOff = kMiscOff + 64;
    static constexpr int kBytes = kBarOff + 32 * 8 + 1024;       // + alignment slack
    static_assert(kDsOff + BS * kBtRows * 2 <= kLdOff, "ring and dS^T lie inside the dV, dK staging");
};

template <int D, int BS>
__global__ void __launch_bounds__(kBtThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
              const float2* __restrict__ ld, const int4* __restrict__ units, const int* __restrict__ uoff, int nblk,
              int rows, const int* __restrict__ list, long long list_stride, const int* __restrict__ kv_len, int Tq,
              int Hq, int Hkv, int L_max, float scale, int* __restrict__ counter, float* __restrict__ dq,
              int* __restrict__ err) {
    using SM = BtSmem<D, BS>;
    constexpr int G = 16;
    static_assert(D == 128 && BS == 128, "one TMEM lane per key and per head-dim row");
    constexpr uint32_t kIdescS = idesc_bf16_f32(BS, kBtRows, 0, 0);  // S^T, dP^T: M = keys, N = query rows
    constexpr uint32_t kIdescKV = idesc_bf16_f32(BS, D, 0, 1);       // dV, dK: B = dO / Q, MN-major
    constexpr uint32_t kIdescQ = idesc_bf16_f32(D, kBtRows, 1, 1);   // dQ^T: A = K^T, B = dS^T, MN-major
    constexpr uint32_t kColS = 0, kColDP = 2 * kBtRows, kColDQ = 3 * kBtRows, kColDV = 4 * kBtRows,
                       kColDK = kColDV + D;
    static_assert(kColDK + D <= 512, "TMEM columns");
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + SM::kBarOff);
    uint64_t* bar_kv = bars + 0;         // K, V of the unit landed (or: no unit left)
    uint64_t* bar_full = bars + 1;       // [3] Q, dO, (lse, D) of a tile landed
    uint64_t* bar_free = bars + 4;       // [3] every MMA reading a ring stage has completed
    uint64_t* bar_s = bars + 7;          // [2] S^T(j) done
    uint64_t* bar_dp = bars + 9;         // [2] dP^T(j) done
    uint64_t* bar_p = bars + 11;         // [2] P^T(j) in TMEM (256 epilogue threads)
    uint64_t* bar_ds = bars + 13;        // [2] dS^T(j) in shared memory (256)
    uint64_t* bar_dqf = bars + 15;       // dQ^T(j) done
    uint64_t* bar_dqe = bars + 16;       // dQ^T buffer read out (256)
    uint64_t* bar_unit = bars + 17;      // every MMA of the unit done
    uint64_t* bar_ufree = bars + 18;     // the unit's staging has been read: next unit may load
    uint64_t* bar_stg_free = bars + 19;  // fp32 staging may be rewritten
    uint64_t* bar_stg_full = bars + 20;  // fp32 staging written (256)
    uint64_t* bar_fin = bars + 21;       // every MMA issued has completed
    int* s_unit = reinterpret_cast<int*>(base + SM::kMiscOff);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(base + SM::kMiscOff + 16);
    volatile int* s_abort = reinterpret_cast<volatile int*>(base + SM::kMiscOff + 20);
    int* s_tok = reinterpret_cast<int*>(base + SM::kTokOff);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        mbar_init(bar_kv, 1);
        for (int i = 0; i < kBtStages; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_free[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_s[i], 1);
            mbar_init(&bar_dp[i], 1);
            mbar_init(&bar_p[i], 256);
            mbar_init(&bar_ds[i], 256);
        }
        mbar_init(bar_dqf, 1);
        mbar_init(bar_dqe, 256);
        mbar_init(bar_unit, 1);
        mbar_init(bar_ufree, 1);
        mbar_init(bar_stg_free, 1);
        mbar_init(bar_stg_full, 256);
        mbar_init(bar_fin, 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == 9) {
        // ======================= loader: unit K / V, then the tiles' Q, dO and (lse, D) rows
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        int total = 0;
        for (int r = lane; r < rows; r += 32) total += uoff[static_cast<size_t>(r) * (nblk + 1) + nblk];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
        int j = 0, kv_loads = 0;
        int fills[kBtStages] = {0, 0, 0};
        bool ok = true, sentinel = false;
        for (int u = 0; ok; ++u) {
            bool w = true;
            if (u > 0 && lane == 0) w = tc_wait(bar_ufree, (u - 1) & 1, s_abort, err);
            if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
            int uid = 0;
            if (lane == 0) uid = atomicAdd(counter, 1);
            uid = __shfl_sync(0xffffffffu, uid, 0);
            if (uid >= total) {
                if (lane == 0) {
                    s_unit[1] = -1;
                    mbar_arrive(bar_kv);
                }
                sentinel = true;
                break;
            }
            const int4 un = units[uid];
            const int bg = un.x, blk = un.y, cnt = un.w - un.z;
            const int* toks = list + bg * list_stride + un.z;
            for (int i = lane; i < cnt; i += 32) s_tok[i] = toks[i];
            __syncwarp();
            const int b = bg / Hkv, g = bg % Hkv;
            if (lane == 0) {
                s_unit[0] = bg;
                s_unit[1] = blk;
                s_unit[2] = cnt;
                mbar_arrive_expect_tx(bar_kv, 2 * SM::kKV);
                const int kv_row = bg * L_max + blk * BS;
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub) {
                    tma_load_2d(base + SM::kKOff + sub * (BS * 128), &tm_k, 64 * sub, kv_row, bar_kv);
                    tma_load_2d(base + SM::kVOff + sub * (BS * 128), &tm_v, 64 * sub, kv_row, bar_kv);
                }
                ++kv_loads;
            }
            const int ntiles = (cnt + kBtTok - 1) / kBtTok;
            for (int i = 0; i < ntiles; ++i, ++j) {
                const int st = j % kBtStages;
                // stage st held tile j-3: free once its dV, dK, dQ^T MMAs completed
                if (j >= kBtStages && lane == 0) w = tc_wait(&bar_free[st], ((j / kBtStages) - 1) & 1, s_abort, err);
                if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
                if (lane == 0) {
                    unsigned char* qt = base + SM::kRingOff + st * 2 * SM::kTile;
                    float2* lt = reinterpret_cast<float2*>(base + SM::kLdOff) + st * kBtRows;
                    mbar_arrive_expect_tx(&bar_full[st], 2 * SM::kTile + kBtRows * 8);
                    for (int k = 0; k < kBtTok; ++k) {
                        // a tile past the slice's end repeats its last token (masked, never written)
                        const int t = s_tok[min(kBtTok * i + k, cnt - 1)];
                        const int row = (b * Tq + t) * Hq + g * G;
#pragma unroll
                        for (int sub = 0; sub < D / 64; ++sub) {
                            tma_load_2d(qt + sub * (kBtRows * 128) + k * (G * 128), &tm_q, 64 * sub, row, &bar_full[st]);
                            tma_load_2d(qt + SM::kTile + sub * (kBtRows * 128) + k * (G * 128), &tm_do, 64 * sub, row,
                                        &bar_full[st]);
                        }
                        bulk_load(lt + k * G, ld + row, G * 8, &bar_full[st]);
                    }
                    ++fills[st];
                }
            }
        }
        // drain: every copy issued has landed before shared memory goes away
        if (lane == 0) {
            const long long drain = kWaitBudgetCycles / 8;
            for (int st = 0; st < kBtStages; ++st)
                if (fills[st] > 0) mbar_wait(&bar_full[st], (fills[st] - 1) & 1, drain);
            if (kv_loads > 0 && !sentinel) mbar_wait(bar_kv, (kv_loads - 1) & 1, drain);
        }
    } else if (warp == 8) {
        // ======================= MMA issuer (one lane)
        if (lane == 0) {
            const uint32_t kb = smem_u32(base + SM::kKOff), vb = smem_u32(base + SM::kVOff);
            const uint32_t ring = smem_u32(base + SM::kRingOff), dsb = smem_u32(base + SM::kDsOff);
            // dst = A B^T with A a block (K or V, BS rows) and B a tile (Q or dO, 64 rows), both K-major
            auto qk = [&](uint32_t dst, uint32_t a0, uint32_t b0) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ao = (kk / 4) * (BS * 128) + (kk % 4) * 32;
                    const uint32_t bo = (kk / 4) * (kBtRows * 128) + (kk % 4) * 32;
                    mma_ss(dst, sw128_desc(a0 + ao, 16, 1024), sw128_desc(b0 + bo, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
            };
            int j = 0;
            bool ok = true, issued = false;
            for (int u = 0; ok; ++u) {
                if (!(ok = tc_wait(bar_kv, u & 1, s_abort, err))) break;
                if (s_unit[1] < 0) break;
                const int ntiles = (s_unit[2] + kBtTok - 1) / kBtTok;
                tc_fence_after();
                for (int i = 0; i < ntiles; ++i, ++j) {
                    const int st = j % kBtStages;
                    const uint32_t qb = ring + st * 2 * SM::kTile, dob = qb + SM::kTile;
                    if (i == 0) {
                        // (the dP^T buffer was read out before dK of the previous tile was issued)
                        if (!(ok = tc_wait(&bar_full[st], (j / kBtStages) & 1, s_abort, err))) break;
                        tc_fence_after();
                        qk(tmem + kColS + (j & 1) * kBtRows, kb, qb);
                        mma_commit(&bar_s[j & 1]);
                        qk(tmem + kColDP, vb, dob);
                        mma_commit(&bar_dp[j & 1]);
                        issued = true;
                    }
                    if (i + 1 < ntiles) {
                        // S^T(j+1) into the other buffer, whose P^T(j-1) dV(j-1) has read: the commit
                        // after dQ^T(j-1) covers it (already complete by now: dP(j) followed it)
                        const int st1 = (j + 1) % kBtStages;
                        if (j > 0 && !(ok = tc_wait(&bar_free[(j - 1) % kBtStages], ((j - 1) / kBtStages) & 1,
                                                    s_abort, err)))
                            break;
                        if (!(ok = tc_wait(&bar_full[st1], ((j + 1) / kBtStages) & 1, s_abort, err))) break;
                        tc_fence_after();
                        qk(tmem + kColS + ((j + 1) & 1) * kBtRows, kb, ring + st1 * 2 * SM::kTile);
                        mma_commit(&bar_s[(j + 1) & 1]);
                    }
                    // dV += P^T dO: P^T rows 32h..32h+31 of the tile are packed at column 32h of its buffer
                    if (!(ok = tc_wait(&bar_p[j & 1], (j >> 1) & 1, s_abort, err))) break;
                    tc_fence_after();
                    const uint32_t tP = tmem + kColS + (j & 1) * kBtRows;
#pragma unroll
                    for (int kk = 0; kk < kBtRows / 16; ++kk)
                        mma_ts(tmem + kColDV, tP + (kk / 2) * 32 + (kk % 2) * 8,
                               sw128_desc(dob + kk * 16 * 128, kBtRows * 128, 1024), kIdescKV, (i > 0 || kk > 0) ? 1u : 0u);
                    // dK += dS^T Q
                    if (!(ok = tc_wait(&bar_ds[j & 1], (j >> 1) & 1, s_abort, err))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBtRows / 16; ++kk)
                        mma_ss(tmem + kColDK, sw128_desc(dsb + kk * 32, 16, 1024),
                               sw128_desc(qb + kk * 16 * 128, kBtRows * 128, 1024), kIdescKV, (i > 0 || kk > 0) ? 1u : 0u);
                    // dQ^T = K^T dS^T once dQ^T(j-1) has been read out
                    if (j > 0 && !(ok = tc_wait(bar_dqe, (j - 1) & 1, s_abort, err))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BS / 16; ++kk)
                        mma_ss(tmem + kColDQ, sw128_desc(kb + kk * 16 * 128, BS * 128, 1024),
                               sw128_desc(dsb + kk * 16 * 128, kBtRows * 128, 1024), kIdescQ, kk > 0 ? 1u : 0u);
                    mma_commit(bar_dqf);
                    mma_commit(&bar_free[st]);
                    if (i + 1 < ntiles) {
                        qk(tmem + kColDP, vb, ring + ((j + 1) % kBtStages) * 2 * SM::kTile + SM::kTile);
                        mma_commit(&bar_dp[(j + 1) & 1]);
                    }
                }
                if (!ok) break;
                mma_commit(bar_unit);
            }
            if (issued) {
                mma_commit(bar_fin);
                mbar_wait(bar_fin, 0, kWaitBudgetCycles / 8);
            }
        }
    } else {
        // ======================= epilogue: 8 warps, TMEM lane quarter q4, query-row half h
        const int q4 = warp & 3, h = warp >> 2;
        const int r = 32 * q4 + lane;  // key of the block (S, dP, dV, dK) / head-dim row (dQ^T)
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const float scale_log2 = scale * 1.4426950408889634f;
        int j = 0, nstg = 0;
        bool ok = true;
        // One use of the fp32 staging area: the bulk unit has read its previous contents ...
        auto stage_begin = [&]() -> bool {
            if (tid == 0) {
                bulk_wait_read_all();
                mbar_arrive(bar_stg_free);
            }
            return tc_wait(bar_stg_free, nstg & 1, s_abort, err);
        };
        // ... and every epilogue thread's writes are visible to it (thread 0 then issues).
        auto stage_end = [&]() -> bool {
            fence_proxy_async_shared();
            mbar_arrive(bar_stg_full);
            return tid == 0 ? tc_wait(bar_stg_full, nstg & 1, s_abort, err) : true;
        };
        // dQ^T(jj) (tile ii of the unit) -> dq: element (head-dim row r, query row 32h + c)
        auto drain_dq = [&](int jj, int ii, int b, int g, int cnt) -> bool {
            if (!tc_wait(bar_dqf, jj & 1, s_abort, err)) return false;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tmem + kColDQ + 32 * h + lane_off, v);
            tmem_ld_wait(v);
            tc_fence_before();
            mbar_arrive(bar_dqe);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int k = kBtTok * ii + 2 * h + e;
                if (k >= cnt) break;
                float* dst = dq + (static_cast<size_t>(b * Tq + s_tok[k]) * Hq + g * G) * D + r;
#pragma unroll
                for (int c = 0; c < 16; ++c) atomicAdd(dst + c * D, __uint_as_float(v[16 * e + c]) * scale);
            }
            return true;
        };
        for (int u = 0; ok; ++u) {
            if (!(ok = tc_wait(bar_kv, u & 1, s_abort, err))) break;
            const int bg = s_unit[0], blk = s_unit[1], cnt = s_unit[2];
            if (blk < 0) break;
            const int b = bg / Hkv, g = bg % Hkv;
            const int Lb = kv_len[b];
            const int key = blk * BS + r;
            const int ntiles = (cnt + kBtTok - 1) / kBtTok;
            for (int i = 0; i < ntiles; ++i, ++j) {
                const int st = j % kBtStages;
                if (!(ok = tc_wait(&bar_full[st], (j / kBtStages) & 1, s_abort, err))) break;
                int pos[2];  // positions of this half's two tokens (-1: past the slice)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = kBtTok * i + 2 * h + e;
                    pos[e] = k < cnt ? Lb - Tq + s_tok[k] : -1;
                }
                // (lse log2e, D) of this half's 32 query rows, two rows per 16-byte broadcast load
                const float4* lv = reinterpret_cast<const float4*>(base + SM::kLdOff) + (st * kBtRows + 32 * h) / 2;
                if (!(ok = tc_wait(&bar_s[j & 1], (j >> 1) & 1, s_abort, err))) break;
                tc_fence_after();
                const uint32_t tS = tmem + kColS + (j & 1) * kBtRows + 32 * h + lane_off;
                uint32_t sv[32];
                tmem_ld32(tS, sv);
                tmem_ld_wait(sv);
                float p[32], dr[32];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float4 l2 = lv[e];
                    const bool live = key <= pos[e >> 3];
                    p[2 * e] = live ? fast_exp2(fmaf(__uint_as_float(sv[2 * e]), scale_log2, -l2.x)) : 0.f;
                    p[2 * e + 1] = live ? fast_exp2(fmaf(__uint_as_float(sv[2 * e + 1]), scale_log2, -l2.z)) : 0.f;
                    dr[2 * e] = l2.y;
                    dr[2 * e + 1] = l2.w;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(p[2 * e], p[2 * e + 1]);
                tmem_st16(tS, pk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar_p[j & 1]);
                if (!(ok = tc_wait(&bar_dp[j & 1], (j >> 1) & 1, s_abort, err))) break;
                tc_fence_after();
                uint32_t dv[32];
                tmem_ld32(tmem + kColDP + 32 * h + lane_off, dv);
                tmem_ld_wait(dv);
                uint32_t dsw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    dsw[e] = pack_bf16x2(p[2 * e] * (__uint_as_float(dv[2 * e]) - dr[2 * e]),
                                         p[2 * e + 1] * (__uint_as_float(dv[2 * e + 1]) - dr[2 * e + 1]));
                // row r of the dS^T tile: 64 bf16 = 8 chunks of 16 bytes, this half's are 4h..4h+3
                unsigned char* row = base + SM::kDsOff + r * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(row + (((4 * h + c) ^ (r & 7)) << 4)) =
                        make_uint4(dsw[4 * c], dsw[4 * c + 1], dsw[4 * c + 2], dsw[4 * c + 3]);
                tc_fence_before();
                fence_proxy_async_shared();
                mbar_arrive(&bar_ds[j & 1]);
                if (i > 0 && !(ok = drain_dq(j - 1, i - 1, b, g, cnt))) break;
            }
            if (!ok) break;
            if (!(ok = tc_wait(bar_unit, u & 1, s_abort, err))) break;
            tc_fence_after();
            if (!(ok = drain_dq(j - 1, ntiles - 1, b, g, cnt))) break;
            // dV, dK -> fp32 boxes of 32 columns (box n of tensor x at kFlushOff + (4x + n) * BS * 128)
            if (!(ok = stage_begin())) break;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
#pragma unroll
                for (int y = 0; y < 2; ++y) {
                    uint32_t v[32];
                    tmem_ld32(tmem + (x ? kColDK : kColDV) + 64 * h + 32 * y + lane_off, v);
                    tmem_ld_wait(v);
                    const float f = x ? scale : 1.f;
                    unsigned char* box = base + SM::kFlushOff + (x * (D / 32) + 2 * h + y) * (BS * 128) + r * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<float4*>(box + ((c ^ (r & 7)) << 4)) =
                            make_float4(__uint_as_float(v[4 * c]) * f, __uint_as_float(v[4 * c + 1]) * f,
                                        __uint_as_float(v[4 * c + 2]) * f, __uint_as_float(v[4 * c + 3]) * f);
                }
            }
            tc_fence_before();
            const bool fine = stage_end();
            if (tid == 0 && fine) {
                const int y0 = bg * L_max + blk * BS;
#pragma unroll
                for (int n = 0; n < D / 32; ++n) {
                    tma_reduce_add_2d(&tm_dv, base + SM::kFlushOff + n * (BS * 128), 32 * n, y0);
                    tma_reduce_add_2d(&tm_dk, base + SM::kFlushOff + (D / 32 + n) * (BS * 128), 32 * n, y0);
                }
                bulk_commit();
                bulk_wait_read_all();
                mbar_arrive(bar_ufree);
            }
            ++nstg;
            ok = fine;
            if (!ok) break;
        }
        if (tid == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

bool bwd_tc_supported(const BwdArgs& a) { return a.d == 128 && a.p.block_size == 128 && a.Hq == 16 * a.Hkv; }

cudaError_t launch_bwd_tc(const BwdArgs& a, const BwdTcWork& w) {
    constexpr int D = 128, BS = 128;
    using SM = BtSmem<D, BS>;
    CUtensorMap tq, tdo, tk, tv, tdk, tdv;
    const uint64_t q_rows = static_cast<uint64_t>(a.B) * a.Tq * a.Hq;
    const uint64_t kv_rows = static_cast<uint64_t>(a.B) * a.Hkv * a.L_max;
    if (!make_tmap_bf16_2d(&tq, a.q, D, q_rows, 64, 16) || !make_tmap_bf16_2d(&tdo, a.dout, D, q_rows, 64, 16) ||
        !make_tmap_bf16_2d(&tk, a.k_cache, D, kv_rows, 64, BS) || !make_tmap_bf16_2d(&tv, a.v_cache, D, kv_rows, 64, BS) ||
        !make_tmap_f32_2d(&tdk, a.dk, D, kv_rows, 32, BS) || !make_tmap_f32_2d(&tdv, a.dv, D, kv_rows, 32, BS))
        return cudaErrorInvalidValue;
    auto kfn = bwd_tc_kernel<D, BS>;
    if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
        e != cudaSuccess)
        return e;
    int dev = 0, n_sm = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    if (cudaError_t e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev); e != cudaSuccess) return e;
    return launch_kernel(kfn, dim3(n_sm), dim3(kBtThreads), SM::kBytes, a.stream, false, tq, tdo, tk, tv, tdk, tdv,
                         w.ld, w.units, w.uoff, w.nblk, a.B * a.Hkv, w.list, w.list_stride, a.kv_len, a.Tq, a.Hq,
                         a.Hkv, a.L_max, a.p.scale, w.counter, a.dq, a.err);
}

}  // namespace infllmv2
