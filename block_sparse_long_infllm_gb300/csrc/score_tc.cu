// score_tc.cu -- block scores for a prefill chunk on the 5th-generation tensor cores
// ("MiniCPM4: 如何在手机电脑上高效运行大语言模型", section 1.1 "InfLLM v2": query-kernel relevance
// at kernel granularity, max over the kernels of a block and over a group's heads).
//
// The scoring is a GEMM per KV head: every (query token, head) row against every visible
// semantic kernel.  A work unit is a tile of 16 query tokens x the 16 heads of one KV head (256 Q
// rows, the MMA's N) against one chunk of 128 kernels (the MMA's M), so each accumulator lane
// holds one kernel against all 256 rows: the max over a token's 16 heads and the visibility test
// (the kernel ends at or before the token's position) are thread-local.  Chunks cover whole
// blocks (31 blocks of 64 tokens or 15 of 128), so no block straddles two chunks.  When the block
// size is a power-of-two multiple r >= 4 of the stride, a chunk starts ceil(c/s) - 1 kernels
// before its first block (a negative kernel index reads the TMA fill value and is masked), so
// block i of the chunk overlaps kernel rows r*i .. r*i + r + ceil(c/s) - 2: each lane folds in the
// rows after it, then warp shuffles take the max over the r aligned lanes while handing tokens
// between lanes (the rows past a warp's last come from the next warp through a small shared
// array, one barrier per chunk among the four warps of the same tokens).  Otherwise the
// per-(token, kernel) maxima go to shared memory, where each block's max over its kernels is
// taken.  The result goes to S[b, g, t, block].
//
// The kernel is persistent: one CTA per SM walks a contiguous share of the (tile x chunk) space,
// so a tile's chunks may be split between two CTAs (packed sequences of uneven lengths take one
// CTA per tile instead).  Per CTA:
//   * loader warp: TMA of each chunk's kernel rows into a ring of four shared stages (a stage is
//     refilled once the MMA group reading it is done), four lanes issuing the boxes; at a new
//     tile, its Q rows started towards L2;
//   * MMA warp (one lane): at a new tile, its Q (two 3-D boxes) once the previous tile's MMAs are
//     done with the buffer; one tcgen05 MMA group per chunk into one of two TMEM buffers;
//   * epilogue warps (warps 0-15, four per TMEM lane quarter, 4 of the 16 tokens each): TMEM
//     load-reduces (each token's 16 columns and their maximum in one load) -> block maxima -> S.
// Waits are bounded (device error word + abort flag), TMEM is freed before exit.
#include <algorithm>
#include <climits>

#include "internal.h"
#include "tc_extra.cuh"
#include "umma.cuh"

namespace infllmv2 {

constexpr int kScTokens = 16;            // query tokens per CTA: N = 16 x 16 heads = 256
constexpr int kScN = kScTokens * 16;
constexpr int kScM = 128;                // kernels per chunk
constexpr int kScEpiWarps = 16;  // epilogue warps: four per TMEM lane quarter
constexpr int kScEpi = 32 * kScEpiWarps;          // epilogue threads
constexpr int kScThreads = kScEpi + 64;           // + the MMA warp and the loader warp
constexpr int kScTpt = kScTokens * 4 / kScEpiWarps;  // tokens per epilogue thread
constexpr int kScStages = 4;     // kernel-row chunks in flight
constexpr int kScTail = 3;       // most kernels a block overlaps past its stride-aligned group (shuffle pass)

template <int D>
struct ScSmem {
    static constexpr int kQ = kScN * D * 2;       // Q tile (B operand)
    static constexpr int kK = kScM * D * 2;       // one chunk of kernel rows (A operand)
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQ;              // kScStages stages
    static constexpr int kMaxOff = kQ + kScStages * kK;  // [kScTokens][kScM] floats (general pass)
    // [2][4][kScTokens] floats: the tail maxima each lane quarter publishes, per chunk parity
    // (the area has room for kScTail rows of them)
    static constexpr int kXOff = kMaxOff + kScTokens * kScM * 4;
    static constexpr int kBarOff = kXOff + 2 * 4 * kScTail * kScTokens * 4;
    static constexpr int kBytes = kBarOff + 192 + 1024;
};

// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// AND of `v` over the epilogue threads (named barrier 1; also synchronises them).
__device__ __forceinline__ bool epilogue_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n"
        " .reg .pred p, q;\n"
        " setp.ne.u32 q, %1, 0;\n"
        " bar.red.and.pred p, 1, %2, q;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(kScEpi)
        : "memory");
    return r != 0;
}

// AND of `v` over the four epilogue warps that take tokens 4 th .. 4 th + 3, one per TMEM lane
// quarter (named barrier 2 + th; also synchronises them).
__device__ __forceinline__ bool token_group_all(bool v, int th) {
    uint32_t r;
    asm volatile(
        "{\n"
        " .reg .pred p, q;\n"
        " setp.ne.u32 q, %1, 0;\n"
        " bar.red.and.pred p, %2, %3, q;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(2 + th), "n"(128)
        : "memory");
    return r != 0;
}

// A query tile: 16 tokens of one sequence against the kernels of one KV head.
struct ScTile {
    int b, g;      // sequence, KV head
    int t0;        // first token (within the sequence's chunk)
    int n_tok;     // tokens in the tile
    int tok;       // the sequence's first token row
    int pos0;      // position of the sequence's query 0 (every draft's, for a tree)
    int n_chunks;  // chunks of blocks to score (0: nothing, e.g. a dense sequence)
};

struct ScArgs {
    const int* kv_len;
    SeqMap sm;
    int tree, Hkv, L_max, M_max;
    Params p;
    int blocks_per_chunk;
    int tiles_x;   // tiles per (sequence, KV head): ceil(longest chunk / 16)
    int c_max;     // chunks of the longest cache
    int n_virt;    // tiles x c_max: the work space the CTAs split into contiguous ranges
};

// Tile `tile` (KV-head-major: consecutive tiles read the same kernel rows).  A sequence outside the
// entry point's limits has no chunks and, with `report`, raises kDevErrIndex.
__device__ __forceinline__ ScTile sc_tile(const ScArgs& a, int tile, bool report, int* err) {
    ScTile t;
    const int x = tile % a.tiles_x, bg = tile / a.tiles_x;
    t.b = bg / a.Hkv;
    t.g = bg % a.Hkv;
    t.t0 = x * kScTokens;
    t.n_tok = 0;
    t.n_chunks = 0;
    const int Lb = a.kv_len[t.b], Tq = a.sm.len(t.b);
    t.tok = a.sm.tok0(t.b);
    // query t sits at Lb - Tq + t (a chunk) or, for tree drafts, all at the last cached position
    t.pos0 = a.tree ? Lb - 1 : Lb - Tq;
    if (Tq < 0 || Tq > a.sm.Tq ||
        (Tq > 0 && (Lb < (a.tree ? 1 : Tq) || Lb > a.L_max ||
                    kernels_in(Lb, a.p.kernel_size, a.p.kernel_stride) > a.M_max))) {
        if (report && x == 0) raise_error(err, kDevErrIndex);
        return t;
    }
    // packed chunks shorter than the longest; dense sequences (every block selected) need no scores
    if (t.t0 >= Tq || Lb < a.p.dense_len) return t;
    t.n_tok = min(kScTokens, Tq - t.t0);
    const int pos_last = a.tree ? t.pos0 : t.pos0 + t.t0 + t.n_tok - 1;
    t.n_chunks = pos_last / a.p.block_size / a.blocks_per_chunk + 1;
    return t;
}

// Walks a CTA's range of the work space (tile x c_max + chunk): next() moves to the next chunk that
// exists (a tile's chunks past its last block are skipped), `first` tells a tile's first chunk in
// the range.  Every role of the CTA walks the same sequence.
struct ScCursor {
    int v, v_end;  // next work-space index, end of the range
    int tile, kk;  // its tile and chunk
    int k = 0;     // the chunk next() returned
    bool first = false, fresh = false, loaded = false;
    ScTile t;
    __device__ __forceinline__ ScCursor(int v0, int v1, int c_max)
        : v(v0), v_end(v1), tile(v0 / c_max), kk(v0 - (v0 / c_max) * c_max) {}
    __device__ __forceinline__ bool next(const ScArgs& a, bool report, int* err) {
        while (v < v_end) {
            if (!loaded) {
                t = sc_tile(a, tile, report, err);
                loaded = fresh = true;
            }
            if (kk < t.n_chunks) {  // (a tile's chunks are 0 .. n_chunks - 1)
                k = kk;
                first = fresh;
                fresh = false;
                ++v;
                if (++kk == a.c_max) {
                    ++tile;
                    kk = 0;
                    loaded = false;
                }
                return true;
            }
            v += a.c_max - kk;  // the rest of this tile has no chunks
            ++tile;
            kk = 0;
            loaded = false;
        }
        return false;
    }
};

template <int D>
__global__ void __launch_bounds__(kScThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kern, ScArgs a,
                int Hq, int nblk_max, float* __restrict__ S, int* __restrict__ err) {
    using SM = ScSmem<D>;
    constexpr int G = 16;
    constexpr uint32_t kIdesc = idesc_bf16_f32(kScM, kScN, 0, 0);
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    float* kmax = reinterpret_cast<float*>(base + SM::kMaxOff);  // [token][kernel row]
    float* xrow = reinterpret_cast<float*>(base + SM::kXOff);    // [chunk parity][quarter][token]
    uint64_t* bar_q = reinterpret_cast<uint64_t*>(base + SM::kBarOff);  // the tile's Q landed (a phase per tile)
    uint64_t* bar_k = bar_q + 1;                 // [kScStages] kernel chunk landed
    uint64_t* bar_acc = bar_k + kScStages;       // [2] MMA of a chunk done
    uint64_t* bar_free = bar_acc + 2;            // [2] epilogue done with a TMEM buffer (kScEpi arrivals)
    uint64_t* bar_kfree = bar_free + 2;          // [kScStages] the MMA group reading a stage is done
    uint64_t* bar_qfree = bar_kfree + kScStages; // the MMAs of a tile are done with Q
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_qfree + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(bar_qfree + 2);
    static_assert((2 + 2 * kScStages + 4) * 8 + 16 <= 192, "barrier area");

    // the top-k kernel after this one may start launching now: it waits (griddepcontrol.wait) for
    // this whole grid to complete before it reads the scores
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Params& p = a.p;
    const int bs = p.block_size, c = p.kernel_size, s = p.kernel_stride;
    const int bpc = a.blocks_per_chunk;
    // this CTA's contiguous range of the work space: the tiles' chunks are split over the grid
    // evenly (a tile may be shared by two CTAs), whatever the number of tiles
    const int v0 = static_cast<int>(static_cast<long long>(a.n_virt) * blockIdx.x / gridDim.x);
    const int v1 = static_cast<int>(static_cast<long long>(a.n_virt) * (blockIdx.x + 1) / gridDim.x);
    {
        // a range without a chunk to score (e.g. one tile past a packed sequence's end) ends here,
        // before any setup; an invalid sequence is reported by the CTA holding its first tile
        ScCursor probe(v0, v1, a.c_max);
        if (!probe.next(a, tid == 0, err)) return;
    }
    // the shuffle pass: block size a power-of-two multiple kr of the stride (4 <= kr <= 32), at
    // most kScTail kernels past a block's group, and a chunk's blocks within its 128 kernel rows
    const int kr = bs / s, kcs = (c + s - 1) / s;
    const bool kr_fast = bs % s == 0 && kr >= 4 && kr <= 32 && (kr & (kr - 1)) == 0 && kcs - 1 <= kScTail &&
                         kcs - 1 <= kr && bpc * kr + kcs - 1 <= kScM;
    // first kernel row of chunk k of a tile; may be negative
    auto chunk_row = [&](int k) {
        const int b0 = k * bpc;
        return kr_fast ? b0 * kr - (kcs - 1) : first_kernel_of_block(b0, bs, c, s);
    };

    if (tid == 0) {
        mbar_init(bar_q, 1);
        mbar_init(bar_qfree, 1);
        for (int i = 0; i < kScStages; ++i) {
            mbar_init(&bar_k[i], 1);
            mbar_init(&bar_kfree[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_acc[i], 1);
            mbar_init(&bar_free[i], kScEpi);
        }
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

    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (*s_abort) return false;
        if (mbar_wait(bar, parity)) return true;
        raise_error(err, kDevErrTimeout);
        *s_abort = 1;
        return false;
    };
    // A tile's Q is one 3-D box {64 columns, 16 heads, 16 tokens} per 64-column half, rows (token,
    // head) in the MMA's layout.  A ragged tile's last box rows hold the next sequence's queries or
    // the fill value: their scores are never stored.
    if (warp == kScEpiWarps + 1) {
        // ======================= loader warp: the kernel-row copies, issued apart from the MMA
        // issuer (a thread that issues an MMA group is held for about its duration, so copies
        // issued by the same warp waited behind it); the boxes of a copy go out from different lanes
        ScCursor cur(v0, v1, a.c_max);
        int n_loaded = 0;  // chunks are loaded in order: stage st holds loads st, st + kScStages, ...
        while (cur.next(a, false, err)) {
            const ScTile& t = cur.t;
            // a new tile: start its Q rows towards L2, for the MMA warp's copy when the previous
            // tile's MMAs are done (this warp runs up to kScStages chunks ahead of them)
            if (cur.first && n_loaded > 0 && lane < D / 64) tma_prefetch_3d(&tm_q, 64 * lane, t.g * G, t.tok + t.t0);
            // chunk n_loaded into stage n_loaded % kScStages once the MMA group of the chunk before
            // it in that stage is done: lane 2 sub + rh issues rows 64 rh .. 64 rh + 63 of column half sub
            const int st = n_loaded % kScStages;
            bool ok = true;
            if (lane == 0 && n_loaded >= kScStages) ok = wait(&bar_kfree[st], (n_loaded / kScStages - 1) & 1);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            if (lane == 0) mbar_arrive_expect_tx(&bar_k[st], SM::kK);
            __syncwarp();
            if (lane < 2 * (D / 64)) {
                const int sub = lane >> 1, rh = lane & 1;
                tma_load_2d(base + SM::kKOff + st * SM::kK + sub * (kScM * 128) + rh * (64 * 128), &tm_kern, 64 * sub,
                            (t.b * a.Hkv + t.g) * a.M_max + chunk_row(cur.k) + 64 * rh, &bar_k[st]);
            }
            ++n_loaded;
        }
        // every copy has landed before shared memory goes away
        if (lane == 0) {
            const long long drain = kWaitBudgetCycles / 8;
            for (int st = 0; st < kScStages && st < n_loaded; ++st) {
                const int uses = (n_loaded - st + kScStages - 1) / kScStages;  // loads into stage st
                mbar_wait(&bar_k[st], (uses - 1) & 1, drain);
            }
        }
    } else if (warp == kScEpiWarps) {
        // ======================= MMA warp (one lane): one tcgen05 group per chunk into TMEM buffer
        // ch & 1; a commit frees the chunk's stage for the loader, another hands the buffer to the
        // epilogue.  At a tile's first chunk it copies the tile's Q once the previous tile's MMAs
        // are done with the one buffer.
        if (lane == 0) {
            const uint32_t sQ = smem_u32(base + SM::kQOff);
            ScCursor cur(v0, v1, a.c_max);
            int ch = 0, n_q = 0;  // chunks issued, Q tiles copied
            bool ok = true;
            while (ok && cur.next(a, false, err)) {
                if (cur.first) {
                    if (n_q > 0) {
                        mma_commit(bar_qfree);
                        if (!(ok = wait(bar_qfree, (n_q - 1) & 1))) break;
                    }
                    mbar_arrive_expect_tx(bar_q, SM::kQ);
#pragma unroll
                    for (int sub = 0; sub < D / 64; ++sub)
                        tma_load_3d(base + SM::kQOff + sub * (kScN * 128), &tm_q, 64 * sub, cur.t.g * G,
                                    cur.t.tok + cur.t.t0, bar_q);
                    ++n_q;
                    if (!(ok = wait(bar_q, (n_q - 1) & 1))) break;
                }
                const int st = ch % kScStages, tb = ch & 1;
                if (!(ok = wait(&bar_k[st], (ch / kScStages) & 1))) break;
                if (ch >= 2 && !(ok = wait(&bar_free[tb], ((ch - 2) >> 1) & 1))) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(base + SM::kKOff + st * SM::kK);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ao = (kk / 4) * (kScM * 128) + (kk % 4) * 32;
                    const uint32_t bo = (kk / 4) * (kScN * 128) + (kk % 4) * 32;
                    mma_ss(tmem + tb * kScN, sw128_desc(ka + ao, 16, 1024), sw128_desc(sQ + bo, 16, 1024), kIdesc,
                           kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar_acc[tb]);
                mma_commit(&bar_kfree[st]);
                ++ch;
            }
            const long long drain = kWaitBudgetCycles / 8;
            if (n_q > 0) mbar_wait(bar_q, (n_q - 1) & 1, drain);  // the last Q copy has landed
            if (ch > 0) mbar_wait(&bar_acc[(ch - 1) & 1], ((ch - 1) >> 1) & 1, drain);
        }
    } else {
        // ======================= epilogue: thread r = 32*(warp%4) + lane owns kernel row r of each
        // chunk; warps w, w+4, w+8, w+12 take tokens 0-3, 4-7, 8-11, 12-15 (TMEM columns 64*(w/4) ...)
        const int q4 = warp % 4;
        const int r = 32 * q4 + lane;
        const int th = warp / 4;
        const int tk0 = th * kScTpt;  // this thread's first token
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        // this thread's kernel row r of a chunk: maxima over the 16 heads of tokens tk0 .. tk0 + 3,
        // one load-reduce of 16 columns per token
        auto row_maxima = [&](int tb, float (&mx)[kScTpt]) {
            static_assert(kScTpt == 4, "four 16-column load-reduces");
            uint32_t r0[16], r1[16], r2[16], r3[16];  // the columns (unused), written by the loads
            const uint32_t ta = tmem + tb * kScN + lane_off + tk0 * G;
            tmem_ld16_max(ta, r0, mx[0]);
            tmem_ld16_max(ta + G, r1, mx[1]);
            tmem_ld16_max(ta + 2 * G, r2, mx[2]);
            tmem_ld16_max(ta + 3 * G, r3, mx[3]);
            tmem_ld_wait_max2(r0, r1, mx[0], mx[1]);
            tmem_ld_wait_max2(r2, r3, mx[2], mx[3]);
        };
        ScCursor cur(v0, v1, a.c_max);
        const bool report = tid == 0;
        int ch = 0;  // chunks taken (TMEM buffer ch & 1)
        if (kr_fast) {
            // After the block maxima below, lane l of a group of kr holds token tau(l) = 2 (l & 1) +
            // ((l >> 1) & 1) of this thread's four (lanes l and l + 4, l + 8 ... hold the same one).
            const int tau = 2 * (lane & 1) + ((lane >> 1) & 1);
            const int kr_log = __ffs(kr) - 1;
            const int T = kcs - 1;  // kernels of a block past its aligned group of kr
            // the group that ends this lane quarter takes its T tail rows from the next quarter
            const bool takes_tail = T > 0 && q4 < 3 && lane >= 32 - kr && (lane & (kr - 1)) < 4;
            int my_bt = -1, my_row = 0, jv_first = -1;
            while (cur.next(a, report, err)) {
                const ScTile& t = cur.t;
                if (cur.first) {
                    // token tau's last block and row of S; the tile's first query's last visible
                    // kernel (no row of a chunk that ends at or before it needs the mask: that query
                    // has the tile's smallest position)
                    my_bt = -1;
                    if (tk0 + tau < t.n_tok) {
                        const int pos = a.tree ? t.pos0 : t.pos0 + t.t0 + tk0 + tau;
                        my_bt = pos / bs;
                        my_row = static_cast<int>(a.sm.sel(t.b, t.g, a.Hkv, t.t0 + tk0 + tau));
                    }
                    const int pos_first = a.tree ? t.pos0 : t.pos0 + t.t0;
                    jv_first = pos_first + 1 >= c ? (pos_first + 1 - c) / s : -1;
                }
                const int tb = ch & 1;
                const bool waited = !*s_abort && mbar_wait(&bar_acc[tb], (ch >> 1) & 1);
                tc_fence_after();
                const int b0 = cur.k * bpc;
                const int jlo = b0 * kr - T;  // kernel of row 0 (negative: before the cache)
                float mx[kScTpt];
                row_maxima(tb, mx);
                tc_fence_before();
                mbar_arrive(&bar_free[tb]);  // this thread is done with the TMEM buffer
                if (jlo < 0 || jlo + kScM - 1 > jv_first) {  // (uniform) a row before the cache or past a query
                    const int j = jlo + r;
#pragma unroll
                    for (int u = 0; u < kScTpt; ++u) {
                        // the token's last visible kernel (-1: no such token)
                        const int tk = tk0 + u;
                        const int pos = a.tree ? t.pos0 : t.pos0 + t.t0 + tk;
                        const int jv = tk < t.n_tok && pos + 1 >= c ? (pos + 1 - c) / s : -1;
                        if (j < 0 || j > jv) mx[u] = -INFINITY;
                    }
                }
                // Block i of the chunk is rows kr i .. kr i + kr - 1 + T.  Each lane takes the maxima
                // of the T rows after it: a group's lanes then cover its block, except that the rows
                // past lane 31 come from the next quarter's lanes 0 .. T - 1, published here (rows of
                // the other lanes of a group are in the block already, so the fold needs no mask).
                float f[kScTpt];
#pragma unroll
                for (int u = 0; u < kScTpt; ++u) f[u] = mx[u];
                for (int tt = 1; tt <= T; ++tt) {
                    if (tt == T && lane == 0)
                        *reinterpret_cast<float4*>(xrow + (tb * 4 + q4) * kScTokens + tk0) =
                            make_float4(f[0], f[1], f[2], f[3]);
#pragma unroll
                    for (int u = 0; u < kScTpt; ++u) f[u] = fmaxf(f[u], __shfl_down_sync(0xffffffffu, mx[u], tt));
                }
                // maxima over each group of kr lanes (kr >= 4), exchanging tokens on the way: after
                // the xor-1 step a lane keeps two tokens, after the xor-2 step one (tau)
                const bool o1 = lane & 1, o2 = lane & 2;
                float k0 = o1 ? f[2] : f[0], k1 = o1 ? f[3] : f[1];
                k0 = fmaxf(k0, __shfl_xor_sync(0xffffffffu, o1 ? f[0] : f[2], 1));
                k1 = fmaxf(k1, __shfl_xor_sync(0xffffffffu, o1 ? f[1] : f[3], 1));
                float m = fmaxf(o2 ? k1 : k0, __shfl_xor_sync(0xffffffffu, o2 ? k0 : k1, 2));
                for (int off = 4; off < kr; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                // the four warps of these tokens meet here (the tails are published; a failed wait ends
                // all of them, the other groups see the abort flag at their next wait)
                if (!token_group_all(waited, th)) {
                    if (tid == 0 && !*s_abort) raise_error(err, kDevErrTimeout);
                    *s_abort = 1;
                    break;
                }
                if (takes_tail) m = fmaxf(m, xrow[(tb * 4 + q4 + 1) * kScTokens + tk0 + tau]);
                const int i = r >> kr_log;  // this lane's block in the chunk
                const int blk = b0 + i;
                if ((lane & (kr - 1)) < 4 && i < bpc && blk <= my_bt)
                    S[static_cast<size_t>(my_row) * nblk_max + blk] = m;
                ++ch;
            }
        } else {
            while (cur.next(a, report, err)) {
                const ScTile& t = cur.t;
                const int tb = ch & 1;
                const bool waited = !*s_abort && mbar_wait(&bar_acc[tb], (ch >> 1) & 1);
                // all epilogue warps leave together: they meet at the named barrier below
                if (!epilogue_all(waited)) {
                    if (tid == 0 && !*s_abort) raise_error(err, kDevErrTimeout);
                    *s_abort = 1;
                    break;
                }
                tc_fence_after();
                const int b0 = cur.k * bpc;
                const int j0 = first_kernel_of_block(b0, bs, c, s);
                const int j = j0 + r;
                const int jend = j * s + c - 1;  // last token of kernel j
                float mx[kScTpt];
                row_maxima(tb, mx);
#pragma unroll
                for (int u = 0; u < kScTpt; ++u) {
                    const int tk = tk0 + u;
                    const int pos = a.tree ? t.pos0 : t.pos0 + t.t0 + tk;
                    kmax[tk * kScM + r] = (tk < t.n_tok && jend <= pos) ? mx[u] : -INFINITY;
                }
                tc_fence_before();
                mbar_arrive(&bar_free[tb]);  // this thread is done with the TMEM buffer
                asm volatile("bar.sync 1, %0;" ::"n"(kScEpi) : "memory");
                // block max over the kernels each block overlaps, for every token of the tile
                const int pos_last = a.tree ? t.pos0 : t.pos0 + t.t0 + t.n_tok - 1;
                const int nb = min(bpc, pos_last / bs + 1 - b0);
                for (int e2 = tid; e2 < t.n_tok * nb; e2 += kScEpi) {
                    const int tk = e2 / nb, blk = b0 + e2 % nb;
                    const int pos = a.tree ? t.pos0 : t.pos0 + t.t0 + tk;
                    if (blk > pos / bs) continue;
                    const int ja = first_kernel_of_block(blk, bs, c, s) - j0;
                    const int jz = min(last_kernel_of_block(blk, bs, s) - j0, kScM - 1);
                    float mm = -INFINITY;
                    for (int jj = ja; jj <= jz; ++jj) mm = fmaxf(mm, kmax[tk * kScM + jj]);
                    S[a.sm.sel(t.b, t.g, a.Hkv, t.t0 + tk) * nblk_max + blk] = mm;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kScEpi) : "memory");  // kmax is rewritten by the next chunk
                ++ch;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Blocks per 128-kernel chunk such that a chunk's blocks overlap at most 128 kernels.
int score_tc_blocks_per_chunk(const Params& p) {
    for (int nb = 256; nb >= 1; --nb)
        if (last_kernel_of_block(nb - 1, p.block_size, p.kernel_stride) -
                first_kernel_of_block(0, p.block_size, p.kernel_size, p.kernel_stride) + 1 <= kScM &&
            (nb * p.block_size + p.kernel_size) / p.kernel_stride + 1 <= kScM)
            return nb;
    return 0;
}

// The work space of a launch: tiles x chunks of the longest cache (0 when there is nothing to
// score; -1 when it does not fit the kernel's int indexing).
static long long score_tc_work(const SelectArgs& a, int blocks_per_chunk) {
    const int nblk_max = (a.L_max + a.p.block_size - 1) / a.p.block_size;
    if (nblk_max <= 0 || a.Tq <= 0) return 0;
    const long long n = static_cast<long long>((a.Tq + kScTokens - 1) / kScTokens) * a.B * a.Hkv *
                        ((nblk_max - 1) / blocks_per_chunk + 1);
    return n <= INT_MAX / 2 ? n : -1;
}

bool score_tc_supported(const SelectArgs& a) {
    return a.Hq / a.Hkv == 16 && (a.d == 64 || a.d == 128) && a.M_max > 0 &&
           score_tc_blocks_per_chunk(a.p) > 0 && score_tc_work(a, score_tc_blocks_per_chunk(a.p)) >= 0;
}

cudaError_t launch_score_tc(const SelectArgs& a, float* S) {
    const int nb = score_tc_blocks_per_chunk(a.p);
    const int nblk_max = (a.L_max + a.p.block_size - 1) / a.p.block_size;
    const long long n_virt = score_tc_work(a, nb);
    if (n_virt < 0) return cudaErrorInvalidValue;
    if (n_virt == 0) return cudaSuccess;
    CUtensorMap tq, tk;
    const SeqMap sm = a.seqmap();
    const uint64_t k_rows = static_cast<uint64_t>(a.B) * a.Hkv * a.M_max;
    if (!make_tmap_bf16_3d(&tq, a.q, a.d, a.Hq, sm.total, 64, 16, kScTokens) ||
        !make_tmap_bf16_2d(&tk, a.kernel_cache, a.d, k_rows, 64, kScM / 2))
        return cudaErrorInvalidValue;
    ScArgs sa;
    sa.kv_len = a.kv_len;
    sa.sm = sm;
    sa.tree = a.tree;
    sa.Hkv = a.Hkv;
    sa.L_max = a.L_max;
    sa.M_max = a.M_max;
    sa.p = a.p;
    sa.blocks_per_chunk = nb;
    sa.tiles_x = (a.Tq + kScTokens - 1) / kScTokens;
    sa.c_max = (nblk_max - 1) / nb + 1;
    sa.n_virt = static_cast<int>(n_virt);
    // Equal-length sequences: one CTA per SM (shared memory and TMEM allow no second), each a
    // contiguous share of the work.  Packed sequences of different lengths leave most of the work
    // space empty and unevenly so: one CTA per tile there, balanced by the hardware's scheduling.
    int dev = 0, n_sm = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    if (cudaError_t e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev); e != cudaSuccess) return e;
    const long long n_tiles = n_virt / sa.c_max;
    const dim3 grid(static_cast<unsigned>(sm.cu != nullptr ? n_tiles : std::min<long long>(std::max(n_sm, 1), n_virt)));
    if (a.d == 128) {
        auto kfn = score_tc_kernel<128>;
        constexpr int smem = ScSmem<128>::kBytes;
        if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); e != cudaSuccess)
            return e;
        return launch_kernel(kfn, grid, dim3(kScThreads), smem, a.stream, false, tq, tk, sa, a.Hq, nblk_max, S, a.err);
    }
    auto kfn = score_tc_kernel<64>;
    constexpr int smem = ScSmem<64>::kBytes;
    if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); e != cudaSuccess)
        return e;
    return launch_kernel(kfn, grid, dim3(kScThreads), smem, a.stream, false, tq, tk, sa, a.Hq, nblk_max, S, a.err);
}

}  // namespace infllmv2
