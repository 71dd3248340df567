// prefill_tc.cu -- block-sparse causal attention for a prefill chunk on the 5th-generation tensor
// cores ("MiniCPM4: 如何在手机电脑上高效运行大语言模型", section 1.1 "InfLLM v2": attention on the
// selected blocks only; "CPM.cu：端侧大模型推理的 CUDA 加速引擎", section 4: chunked prefill).
//
// One CTA owns a tile of 8 query tokens x the 16 query heads of one KV head: 128 rows, one
// TMEM lane each.  The tile walks the union of its tokens' selected blocks (a token's heads
// share one selection); a row whose token did not select a block masks it out.
//   * Load warp (warp 9, one lane): TMA loads of Q (once) and of each block's K and V into
//     three-stage (K) and two-stage (V) rings of 128-byte-swizzled shared tiles; a stage is
//     reloaded once the MMA that read it has completed.
//   * Two MMA warps (one lane each) issue the tcgen05 MMAs: warp 8 S = Q K^T into one of three
//     TMEM buffers (M=128, N=block_size, K=d), warp 10 O += P V with P read from TMEM (A operand)
//     and V from shared memory (MN-major B).  An MMA issue holds the issuing thread for about
//     the MMA's own duration; with two issuers, one thread's barrier waits overlap the other's
//     MMAs and the tensor core is not left idle while a wait resolves.
//   * Softmax warps (warps 0-7; two warps per row, each with half of the key columns): S from
//     TMEM; causal mask on the query's own block; online max/sum in fp32 (the pair combines its
//     row maxima through shared memory); the running max is raised only when it grows by more
//     than 2^8, and only then is O rescaled in TMEM; P goes back to TMEM as bf16 over S.
//     Rows of tokens that did not choose a block get zero P rows; a warp none of whose rows
//     chose the block only stores those zeros, so the union tile costs softmax work only where
//     a token really attends.
// With three S buffers, S of blocks j+1 and j+2 can be computed (and PV of block j-1 finish)
// while the softmax of block j runs, so the softmax warps find the next S ready.  Every wait is a
// bounded mbarrier wait: one that runs out sets the device error word and an abort flag that
// ends every loop; the load and MMA warps drain what they issued and the TMEM is freed before
// exit.
#include <algorithm>

#include "internal.h"
#include "tc_extra.cuh"
#include "umma.cuh"

namespace infllmv2 {

constexpr int kTcTokens = 8;   // tokens per tile: 8 x 16 heads = 128 rows
constexpr int kTcRows = 128;
constexpr int kTcKStages = 3;  // K tiles in flight; stage j % 3 also names the TMEM S buffer of block j
constexpr int kTcThreads = 352;  // 8 softmax warps (two per TMEM lane quarter), S-MMA, load, PV-MMA warps

template <int D, int BS>
struct TcSmem {
    static constexpr int kQ = D * kTcRows * 2;     // Q tile
    static constexpr int kKV = D * BS * 2;         // one K (or V) block
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQ;                    // kTcKStages stages
    static constexpr int kVOff = kQ + kTcKStages * kKV;  // 2 stages
    static constexpr int kBarOff = kVOff + 2 * kKV;      // q, k[3], v[2], s[3], o[3], p[3], fin[2]  (17 x 8 B)
    static constexpr int kMiscOff = kBarOff + 256; // tmem base, abort flag, union size
    static constexpr int kPairOff = kBarOff + 256 + 64;  // [2][128] partial maxima, [2][128] partial sums
    static constexpr int kUnionOff2 = kPairOff + 4 * 128 * 4;
    static int bytes(int max_union, int nwords) { return kUnionOff2 + 8 * max_union + 8 * nwords + 1024; }
};

// AND of `v` over the 64 threads of named barrier `id` (also synchronises them).
__device__ __forceinline__ bool pair_all(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n"
        " .reg .pred p, q;\n"
        " setp.ne.u32 q, %1, 0;\n"
        " bar.red.and.pred p, %2, 64, q;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id)
        : "memory");
    return r != 0;
}

// Three-input maximum and paired fp32 arithmetic (one instruction for two lanes of data).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(__float_as_uint(lo)), "r"(__float_as_uint(hi)));
    return d;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
    uint32_t a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(v));
    lo = __uint_as_float(a);
    hi = __uint_as_float(b);
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

template <int D, int BS>
__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const int* __restrict__ idx,
                  const int* __restrict__ counts, int S_max, const int* __restrict__ kv_len, SeqMap sm, int Hq, int Hkv,
                  int L_max, int max_union, float scale_log2, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                  int* __restrict__ err) {
    using SM = TcSmem<D, BS>;
    constexpr int G = 16;
    constexpr uint32_t kIdescS = idesc_bf16_f32(kTcRows, BS, 0, 0);
    constexpr uint32_t kIdescO = idesc_bf16_f32(kTcRows, D, 0, 1);
    constexpr uint32_t kTmemCols = (3 * BS + D) <= 256 ? 256u : 512u;
    static_assert(3 * BS + D <= 512, "three S buffers and O must fit the 512 TMEM columns");
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* bar_q = reinterpret_cast<uint64_t*>(base + SM::kBarOff);
    uint64_t* bar_k = bar_q + 1;  // [3] K block landed
    uint64_t* bar_v = bar_q + 4;  // [2] V block landed
    // Rings indexed by block j: K, S, O and P on j % 3 (completed phase parity (j / 3) & 1), V on
    // j & 1.  Each next completion of a barrier needs a step that its waiter has not yet allowed,
    // so no parity wait below can fall two phases behind.
    uint64_t* bar_s = bar_q + 6;    // [3] S(j) = Q K^T done
    uint64_t* bar_o = bar_q + 9;    // [3] O += P(j) V(j) done
    uint64_t* bar_p = bar_q + 12;   // [3] P(j) written by all 256 softmax threads
    uint64_t* bar_fin = bar_q + 15; // [2] every MMA of the S / PV issuer has completed
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(base + SM::kMiscOff);
    volatile int* s_abort = reinterpret_cast<volatile int*>(base + SM::kMiscOff + 4);
    int* s_U = reinterpret_cast<int*>(base + SM::kMiscOff + 8);
    int* ublk = reinterpret_cast<int*>(base + SM::kUnionOff2);          // [max_union] union blocks, ascending
    uint32_t* umask = reinterpret_cast<uint32_t*>(ublk + max_union);   // [max_union] tokens that chose each

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y / Hkv, g = blockIdx.y % Hkv;
    const int t0 = blockIdx.x * kTcTokens;
    const int Lb = kv_len[b];
    const int Tq = sm.len(b), tok = sm.tok0(b);  // this sequence's chunk: token rows tok .. tok + Tq - 1
    if (Tq < 0 || Tq > sm.Tq || (t0 < Tq && (Lb < Tq || Lb > L_max))) {
        if (tid == 0) raise_error(err, kDevErrIndex);
        return;
    }
    if (t0 >= Tq) return;  // packed chunks shorter than the longest
    const int n_tok = min(kTcTokens, Tq - t0);
    const int bt_max = (Lb - Tq + t0 + n_tok - 1) / BS;
    const int nwords = bt_max / 32 + 1;
    uint32_t* bitmap = umask + max_union;                           // [nwords]
    int* wpre = reinterpret_cast<int*>(bitmap + nwords);            // [nwords] exclusive popcount prefix

    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int i = 0; i < kTcKStages; ++i) {
            mbar_init(&bar_k[i], 1);
            mbar_init(&bar_s[i], 1);
            mbar_init(&bar_o[i], 1);
            mbar_init(&bar_p[i], 256);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_v[i], 1);
            mbar_init(&bar_fin[i], 1);
        }
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }

    // ---- union of the tile's selections: bitmap over blocks, then ranks by prefix popcounts
    for (int w = tid; w < nwords; w += kTcThreads) bitmap[w] = 0;
    for (int u = tid; u < max_union; u += kTcThreads) umask[u] = 0;
    __syncthreads();
    const int* cnt_row = counts != nullptr ? counts + sm.sel(b, g, Hkv, t0) : nullptr;
    const int* idx_row = idx != nullptr ? idx + sm.sel(b, g, Hkv, t0) * S_max : nullptr;
    const int per_tok = idx != nullptr ? S_max : bt_max + 1;
    auto entry = [&](int e, int& tk) -> int {  // block id of entry e (token tk), or -1
        tk = e / per_tok;
        const int r = e % per_tok;
        const int bt = (Lb - Tq + t0 + tk) / BS;
        if (idx == nullptr) return r <= bt ? r : -1;
        const int cnt = min(max(cnt_row[tk], 0), S_max);
        if (r >= cnt) return -1;
        const int blk = idx_row[static_cast<size_t>(tk) * S_max + r];
        return (blk < 0 || blk > bt) ? -2 : blk;
    };
    for (int e = tid; e < n_tok * per_tok; e += kTcThreads) {
        int tk;
        const int blk = entry(e, tk);
        if (blk == -2) raise_error(err, kDevErrIndex);
        if (blk >= 0) atomicOr(&bitmap[blk >> 5], 1u << (blk & 31));
    }
    if (idx != nullptr && tid < n_tok) {
        const int cnt = cnt_row[tid];
        if (cnt < 0 || cnt > S_max) raise_error(err, kDevErrIndex);
    }
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int w0 = 0; w0 < nwords; w0 += 32) {
            const int w = w0 + lane;
            const int c = w < nwords ? __popc(bitmap[w]) : 0;
            int incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            if (w < nwords) wpre[w] = run + incl - c;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) *s_U = run;
    }
    __syncthreads();
    for (int e = tid; e < n_tok * per_tok; e += kTcThreads) {
        int tk;
        const int blk = entry(e, tk);
        if (blk < 0) continue;
        const int rank = wpre[blk >> 5] + __popc(bitmap[blk >> 5] & ((1u << (blk & 31)) - 1u));
        if (rank < max_union) {
            ublk[rank] = blk;
            atomicOr(&umask[rank], 1u << tk);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int U = min(*s_U, max_union);
    const uint32_t tmem = *s_tmem;
    const uint32_t tO = tmem + 3 * BS;  // S buffers at tmem + i * BS, i = 0, 1, 2

    if (warp == 9) {
        // ======================= load warp: TMA (one lane)
        if (lane == 0 && U > 0) {
            const int kv_row0 = (b * Hkv + g) * L_max;
            int k_issued[kTcKStages] = {}, v_issued[2] = {0, 0};  // loads issued per stage
            auto load = [&](int j, bool is_v) {
                const int st = is_v ? (j & 1) : (j % kTcKStages);
                uint64_t* bar = is_v ? &bar_v[st] : &bar_k[st];
                unsigned char* dst = base + (is_v ? SM::kVOff : SM::kKOff) + st * SM::kKV;
                mbar_arrive_expect_tx(bar, SM::kKV);
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_2d(dst + sub * BS * 128, is_v ? &tm_v : &tm_k, 64 * sub, kv_row0 + ublk[j] * BS, bar);
                (is_v ? v_issued : k_issued)[st] += 1;
            };
            // Q: one 16-row box per token (its 16 heads) and 64-column half
            mbar_arrive_expect_tx(bar_q, SM::kQ);
            for (int tk = 0; tk < kTcTokens; ++tk) {
                const int t = min(t0 + tk, Tq - 1);
                const int qrow = (tok + t) * Hq + g * G;
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_2d(base + SM::kQOff + sub * (kTcRows * 128) + tk * (G * 128), &tm_q, 64 * sub, qrow, bar_q);
            }
            for (int j = 0; j < kTcKStages && j < U; ++j) load(j, false);
            for (int i = 0; i < U; ++i) {
                // V stage i & 1 held V(i-2): free once PV(i-2) is done
                if (i >= 2 && !tc_wait(&bar_o[(i - 2) % kTcKStages], ((i - 2) / kTcKStages) & 1, s_abort, err)) break;
                load(i, true);
                // K stage i % 3 held K(i): free once S(i) is done
                if (i + kTcKStages < U) {
                    if (!tc_wait(&bar_s[i % kTcKStages], (i / kTcKStages) & 1, s_abort, err)) break;
                    load(i + kTcKStages, false);
                }
            }
            // drain: every copy issued has landed before shared memory goes away (only the last
            // load of a stage can be pending: each earlier one was consumed by a completed MMA)
            const long long drain = kWaitBudgetCycles / 8;
            for (int st = 0; st < kTcKStages; ++st)
                if (k_issued[st] > 0) mbar_wait(&bar_k[st], (k_issued[st] - 1) & 1, drain);
            for (int st = 0; st < 2; ++st)
                if (v_issued[st] > 0) mbar_wait(&bar_v[st], (v_issued[st] - 1) & 1, drain);
        }
    } else if (warp == 8) {
        // ======================= S issuer (one lane): S(j) into TMEM buffer j % 3 from K stage j % 3
        if (lane == 0 && U > 0) {
            const uint32_t sQ = smem_u32(base + SM::kQOff);
            bool issued = false;
            bool ok = tc_wait(bar_q, 0, s_abort, err);
            for (int j = 0; ok && j < U; ++j) {
                const int st = j % kTcKStages;
                // buffer j % 3 held P(j-3): free once PV(j-3) is done
                if (j >= kTcKStages && !(ok = tc_wait(&bar_o[st], ((j - kTcKStages) / kTcKStages) & 1, s_abort, err)))
                    break;
                if (!(ok = tc_wait(&bar_k[st], (j / kTcKStages) & 1, s_abort, err))) break;
                tc_fence_after();
                const uint32_t kb = smem_u32(base + SM::kKOff + st * SM::kKV);
                const uint32_t dS = tmem + st * BS;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = (kk / 4) * (kTcRows * 128) + (kk % 4) * 32;
                    const uint32_t ko = (kk / 4) * (BS * 128) + (kk % 4) * 32;
                    mma_ss(dS, sw128_desc(sQ + qo, 16, 1024), sw128_desc(kb + ko, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar_s[st]);
                issued = true;
            }
            if (issued) {  // one commit covers every MMA this thread issued
                mma_commit(&bar_fin[0]);
                mbar_wait(&bar_fin[0], 0, kWaitBudgetCycles / 8);
            }
        }
    } else if (warp == 10) {
        // ======================= PV issuer (one lane): O += P(j) V(j), P in TMEM buffer j % 3
        if (lane == 0 && U > 0) {
            bool issued = false;
            bool ok = true;
            for (int j = 0; ok && j < U; ++j) {
                const int st = j % kTcKStages;
                if (!(ok = tc_wait(&bar_p[st], (j / kTcKStages) & 1, s_abort, err))) break;
                if (!(ok = tc_wait(&bar_v[j & 1], (j >> 1) & 1, s_abort, err))) break;
                tc_fence_after();
                const uint32_t vb = smem_u32(base + SM::kVOff + (j & 1) * SM::kKV);
                const uint32_t aP = tmem + st * BS;
#pragma unroll
                for (int kk = 0; kk < BS / 16; ++kk) {
                    // B = V (keys x d, d contiguous): 16 keys per step = 2 groups of 8 rows; the
                    // 64-column halves of d are BS*128 bytes apart
                    const uint64_t bdesc = sw128_desc(vb + kk * 16 * 128, BS * 128, 1024);
                    mma_ts(tO, aP + kk * 8, bdesc, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bar_o[st]);
                issued = true;
            }
            if (issued) {
                mma_commit(&bar_fin[1]);
                mbar_wait(&bar_fin[1], 0, kWaitBudgetCycles / 8);
            }
        }
    } else {
        // ======================= softmax warps: warp w owns TMEM lanes 32*(w%4) .. +31 (rows r =
        // (token r/16, head r%16)) and half h = w/4 of the key columns and of the output columns;
        // the two warps of a lane quarter exchange partial row maxima through shared memory.
        constexpr int HB = BS / 2;  // key columns per half
        constexpr int HD = D / 2;   // output columns per half
        float* pmax = reinterpret_cast<float*>(base + SM::kPairOff);  // [2][128]
        float* psum = pmax + 2 * 128;                                  // [2][128]
        const int h = warp / 4;
        const int r = 32 * (warp % 4) + lane;
        const int pair_bar = 1 + (warp % 4);  // named barrier of warps w and w+4 (64 threads)
        const int tk = r / G;
        const bool live = tk < n_tok;
        const int pos = Lb - Tq + t0 + tk;
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
        float m_run = -INFINITY;  // running max of the raw scores q.k (unscaled), same in both halves
        float l_run = 0.f;        // this half's share of the row sum
        bool ok = true;
        int sb = 0;               // S buffer of block j: j % 3, completed phase parity (j / 3) & 1
        uint32_t sph = 0;
        // S(j) is loaded from TMEM one step ahead: the load of block j+1 is issued before this
        // warp waits for its P(j) stores, so the two latencies overlap.  Both warps of a pair
        // see the same tokens, so they take the same branches and meet at the same barriers.
        uint32_t ra[32], rb[32];
        float ma = -INFINITY, mb = -INFINITY;  // the loaded columns' maxima (load-reduce)
        auto chooses = [&](int jj) -> bool {  // warp-uniform: does any row of this warp attend block jj?
            return __any_sync(0xffffffffu, live && ((umask[jj] >> tk) & 1u));
        };
        auto load_s = [&](int sbuf) {
            const uint32_t tS = tmem + sbuf * BS + lane_off + h * HB;
            tmem_ld32_max(tS, ra, ma);
            if constexpr (HB == 64) tmem_ld32_max(tS + 32, rb, mb);
        };
        if (U > 0) {
            const bool waited = !*s_abort && mbar_wait(&bar_s[0], 0);
            if (!pair_all(pair_bar, waited)) {
                if (!*s_abort && lane == 0) raise_error(err, kDevErrTimeout);
                *s_abort = 1;
                ok = false;
            } else if (chooses(0)) {
                tc_fence_after();
                load_s(0);
            }
        }
        for (int j = 0; ok && j < U; ++j) {
            const bool chose = live && ((umask[j] >> tk) & 1u);
            const uint32_t tS = tmem + sb * BS + lane_off;
            const int sb1 = sb + 1 == kTcKStages ? 0 : sb + 1;
            const uint32_t sph1 = sb1 == 0 ? sph ^ 1u : sph;
            if (__any_sync(0xffffffffu, chose)) {
                // S(j) of this half, in place in the load registers (column c in ra / rb)
                tmem_ld_wait_max32(ra, ma);
                if constexpr (HB == 64) {
                    reg_fence(rb);
                    asm volatile("" : "+f"(mb));
                }
                auto sv = [&](int c) -> float { return __uint_as_float(c < 32 ? ra[c] : rb[c - 32]); };
                // valid keys of a row that chose the block: x = blk*BS + c <= pos (only the
                // query's own block is partial); rows that did not choose it get p = 0 below
                const int n_valid = min(BS, pos - ublk[j] * BS + 1) - h * HB;
                // row maximum of this half: from the load-reduces, except in the query's own
                // (partial) block, whose keys past the query are masked first
                float mh = HB == 64 ? fmaxf(ma, mb) : ma;
                if (__any_sync(0xffffffffu, chose && n_valid < HB)) {
#pragma unroll
                    for (int c = 0; c < HB; ++c) {
                        uint32_t& x = c < 32 ? ra[c] : rb[c - 32];
                        x = c < n_valid ? x : __float_as_uint(-INFINITY);
                    }
                    // eight independent chains of three-input maxima
                    float mc[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) mc[k] = sv(k);
#pragma unroll
                    for (int c = 8; c + 16 <= HB; c += 16)
#pragma unroll
                        for (int k = 0; k < 8; ++k) mc[k] = fmax3f(mc[k], sv(c + k), sv(c + 8 + k));
#pragma unroll
                    for (int k = 0; k < 8; ++k) mc[k] = fmaxf(mc[k], sv(HB - 8 + k));
                    mh = fmax3f(fmax3f(mc[0], mc[1], mc[2]), fmax3f(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
                }
                pmax[h * 128 + r] = mh;
                asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
                const float mb = fmaxf(mh, pmax[(1 - h) * 128 + r]);
                // raise the running max only when it grows by more than 8 in the log2 domain
                bool rescale = false;
                float factor = 1.f;
                if (chose && (mb - m_run) * scale_log2 > 8.f) {
                    if (m_run != -INFINITY) {
                        rescale = true;
                        factor = fast_exp2((m_run - mb) * scale_log2);
                        l_run *= factor;
                    }
                    m_run = mb;
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // O must hold PV(j-1) before it is rescaled (PV(j-1) done implies PV(j-2) done:
                    // one issuer, one accumulator)
                    if (j >= 1 && !mbar_wait(&bar_o[(j - 1) % kTcKStages], ((j - 1) / kTcKStages) & 1)) {
                        raise_error(err, kDevErrTimeout);
                        *s_abort = 1;
                    }
                    __syncwarp();
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < HD; c0 += 32) {
                        uint32_t rr[32];
                        tmem_ld32(tO + lane_off + h * HD + c0, rr);
                        tmem_ld_wait(rr);
#pragma unroll
                        for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * factor);
                        tmem_st32(tO + lane_off + h * HD + c0, rr);
                    }
                    tmem_st_wait();
                }
                // p = 2^((s - m) * scale_log2): one paired FFMA per two columns, one EX2 each
                // (-inf offset for rows that did not choose the block: p = 0); the row sum runs
                // in four paired accumulators (eight independent chains)
                const float neg = !chose ? -INFINITY : (m_run == -INFINITY ? 0.f : -m_run * scale_log2);
                const uint64_t sc2 = f32x2(scale_log2, scale_log2), ng2 = f32x2(neg, neg);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c0 = 0; c0 < HB; c0 += 32) {  // 32 columns -> 16 packed P words per store
                    uint32_t pw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float x0, x1;
                        f32x2_split(ffma2(f32x2(sv(c0 + 2 * e), sv(c0 + 2 * e + 1)), sc2, ng2), x0, x1);
                        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                        acc[e & 3] = fadd2(acc[e & 3], f32x2(p0, p1));
                        pw[e] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tS + (h * HB + c0) / 2, pw);
                }
                if (chose) {
                    float a0, a1, b0, b1;
                    f32x2_split(fadd2(acc[0], acc[1]), a0, a1);
                    f32x2_split(fadd2(acc[2], acc[3]), b0, b1);
                    l_run += (a0 + b0) + (a1 + b1);
                }
            } else {
                // no row of this warp chose the block: its P columns are zero (nothing else to do)
                uint32_t z[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
                for (int c0 = 0; c0 < HB; c0 += 32) tmem_st16(tS + (h * HB + c0) / 2, z);
            }
            // S(j+1): if it is already complete, start its load before the wait for the P stores
            const bool more = j + 1 < U;
            const bool next = more && chooses(j + 1);
            const bool ready = more && mbar_test_wait(&bar_s[sb1], sph1);
            if (ready && next) {
                tc_fence_after();
                load_s(sb1);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar_p[sb]);
            if (more) {
                const bool waited = ready || (!*s_abort && mbar_wait(&bar_s[sb1], sph1));
                if (!pair_all(pair_bar, waited)) {
                    if (!*s_abort && lane == 0) raise_error(err, kDevErrTimeout);
                    *s_abort = 1;
                    ok = false;
                    break;
                }
                if (!ready && next) {
                    tc_fence_after();
                    load_s(sb1);
                }
            }
            sb = sb1;
            sph = sph1;
        }
        // ---- epilogue: O / l -> bf16, lse
        psum[h * 128 + r] = l_run;
        asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
        const float l_row = l_run + psum[(1 - h) * 128 + r];
        const bool go = __all_sync(0xffffffffu, ok && U > 0 && !*s_abort);
        const int hq = g * G + (r % G);
        if (U == 0 && live) {  // nothing selected: zero output
            __nv_bfloat16* dst = o + ((static_cast<size_t>(tok) + t0 + tk) * Hq + hq) * D + h * HD;
            for (int c = 0; c < HD; c += 8) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
            if (lse != nullptr && h == 0) lse[sm.lse(b, hq, Hq, t0 + tk)] = -INFINITY;
        }
        if (go) {
            // PV(U-1) done implies every earlier PV done; S(U-1) was issued after PV(U-4)
            // completed, so the barrier of PV(U-1) is at most one phase behind.
            const bool done = mbar_wait(&bar_o[(U - 1) % kTcKStages], ((U - 1) / kTcKStages) & 1);
            if (!__all_sync(0xffffffffu, done)) {
                if (lane == 0) raise_error(err, kDevErrTimeout);
                *s_abort = 1;
            } else {
                tc_fence_after();
                const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
                const int t = t0 + tk;
                __nv_bfloat16* dst = o + ((static_cast<size_t>(tok) + (live ? t : 0)) * Hq + hq) * D + h * HD;
#pragma unroll
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t rr[32];
                    tmem_ld32(tO + lane_off + h * HD + c0, rr);
                    tmem_ld_wait(rr);
                    if (live) {
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * inv, __uint_as_float(rr[2 * e + 1]) * inv);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            reinterpret_cast<uint4*>(dst + c0)[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                }
                if (live && lse != nullptr && h == 0)
                    lse[sm.lse(b, hq, Hq, t)] =
                        l_row > 0.f ? (m_run * scale_log2 + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

bool tc_prefill_supported(const PrefillArgs& a) {
    const int G = a.Hq / a.Hkv;
    return G == 16 && (a.d == 64 || a.d == 128) && (a.p.block_size == 64 || a.p.block_size == 128);
}

template <int D, int BS>
static cudaError_t launch_tc_t(const PrefillArgs& a) {
    using SM = TcSmem<D, BS>;
    const int nblk = (a.L_max + BS - 1) / BS;
    const int per_tok = a.idx != nullptr ? a.S_max : nblk;
    const int max_union = std::min(kTcTokens * per_tok, nblk);
    const int nwords = nblk / 32 + 1;
    const int smem = SM::bytes(max_union, nwords);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv;
    const SeqMap sm = a.seqmap();
    const uint64_t q_rows = static_cast<uint64_t>(sm.total) * a.Hq;
    const uint64_t kv_rows = static_cast<uint64_t>(a.B) * a.Hkv * a.L_max;
    if (!make_tmap_bf16_2d(&tq, a.q, D, q_rows, 64, 16) || !make_tmap_bf16_2d(&tk, a.k_cache, D, kv_rows, 64, BS) ||
        !make_tmap_bf16_2d(&tv, a.v_cache, D, kv_rows, 64, BS))
        return cudaErrorInvalidValue;
    auto kfn = prefill_tc_kernel<D, BS>;
    if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); e != cudaSuccess)
        return e;
    dim3 grid((a.Tq + kTcTokens - 1) / kTcTokens, a.B * a.Hkv);
    const float scale_log2 = a.p.scale * 1.4426950408889634f;
    return launch_kernel(kfn, grid, dim3(kTcThreads), smem, a.stream, false, tq, tk, tv, a.idx, a.counts, a.S_max,
                         a.kv_len, sm, a.Hq, a.Hkv, a.L_max, max_union, scale_log2,
                         static_cast<__nv_bfloat16*>(a.o), a.lse, a.err);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a) {
    if (a.d == 128) return a.p.block_size == 128 ? launch_tc_t<128, 128>(a) : launch_tc_t<128, 64>(a);
    return a.p.block_size == 128 ? launch_tc_t<64, 128>(a) : launch_tc_t<64, 64>(a);
}

}  // namespace infllmv2
