// tree_attn.cu -- the attention of tree-speculative verification: every draft attends to its own
// selected blocks of the cache and to the drafts its uint64 mask bit set names, under one softmax
// ("MiniCPM4: 如何在手机电脑上高效运行大语言模型", section 1.1 "InfLLM v2": attention on the
// selected blocks only, uint64-compressed attention mask for tree-speculative decoding;
// "CPM.cu：端侧大模型推理的 CUDA 加速引擎": tree verification inside flash attention).
//
// One row is (sequence b, KV head g, draft i): the G query heads of draft i that share its
// selection (the selection kernel's row order).  A thread-block cluster of CL CTAs takes a row:
//   * CTA r attends the row's list entries r, r + CL, ...: their K and V blocks stream through a
//     ring of shared-memory slots by TMA (full / empty mbarriers per slot) and eight warps each
//     feed 32-key tiles through the warp-MMA online softmax of attn_warp.cuh.  A copy issue holds
//     its thread for a while, so the issues are spread over the warps: warp k fills slot k at the
//     start, and the warp that reads a block's first tile refills its slot with the block NS
//     later once every tile of the slot has been read (a per-slot generation count tells the
//     readers which block a slot's current phase holds).  The last CTA (which has the fewest
//     entries) also attends the draft keys whose mask bits are set.
//   * The eight warps merge into one fp32 (m, l, o) partial per head; CTA r copies its partial of
//     head h into a slot of CTA h mod CL (bulk copies into the peer's shared memory, counted on
//     its barrier), which merges the CL partials of its heads and writes o (bf16) and lse.
// Nothing goes through global memory between the CTAs, so there is no merge kernel; with more
// rows than clusters fit at once, CL = 1 and each CTA takes a whole row.
#include <algorithm>
#include <mutex>
#include <vector>

#include "attn_warp.cuh"
#include "internal.h"

namespace infllmv2 {

constexpr int kTaWarps = 8;                          // warps attending 32-key tiles
constexpr int kTaThreads = kTaWarps * 32;
constexpr int kTaRingBytes = 6 * 32768;              // K/V slots
constexpr int kTaList = 512;                         // entries of a CTA's list staged in shared memory

template <int D, int BS>
struct TreeSmem {
    static constexpr int kTile = BS * D * 2;  // one block of K (or V)
    static constexpr int kFit = kTaRingBytes / (2 * kTile);
    static constexpr int kSlots = kFit < 8 ? kFit : 8;
    static constexpr int kPRow = D + 4;        // a head's partial: m, l, 2 unused, o[D]
    static constexpr int kMergeRow = D + D / 8;  // the 8-warp merge scratch: 4 floats of pad per 32 columns
    static constexpr int kMerge = (8 * 16 * 2 + 8 * 16 * kMergeRow) * 4;
    static_assert(kMerge + 16 * kPRow * 4 <= kTaRingBytes, "merge scratch and partial fit the ring");
    static constexpr int kPart = kMerge;                       // this CTA's partial [16][kPRow]
    static constexpr int kInSlots = kTaRingBytes;              // partials merged here [24][kPRow]
    static constexpr int kBars = kInSlots + 24 * kPRow * 4;    // full[kSlots], empty[kSlots], part
    static constexpr int kBytes = kBars + 8 * (2 * kSlots + 1) + 1024;
};

__device__ __forceinline__ uint32_t ta_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t ta_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t ta_mapa(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
// The cluster barrier in two halves (relaxed arrive, acquire wait), executed once each by every
// thread of every CTA: here it only says that every CTA's barriers have been initialised.
__device__ __forceinline__ void ta_cluster_arrive() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void ta_cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void ta_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

template <int D, int BS>
__global__ void __launch_bounds__(kTaThreads, 1)
tree_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ dk,
                 const __nv_bfloat16* __restrict__ dv, const uint64_t* __restrict__ tree_mask,
                 const int* __restrict__ kv_len, const int* __restrict__ idx, const int* __restrict__ counts,
                 int idx_stride, int n_draft, int Hq, int Hkv, int G, int L_max, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ lse, float scale_log2, int* __restrict__ err) {
    using SM = TreeSmem<D, BS>;
    constexpr int NS = SM::kSlots;
    constexpr int kTile = SM::kTile;
    constexpr int TPB = BS / 32;  // 32-key tiles per block
    constexpr int kPRow = SM::kPRow;
    constexpr int kMergeRow = SM::kMergeRow;
    extern __shared__ unsigned char smem_dyn[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    float* part = reinterpret_cast<float*>(base + SM::kPart);
    float* in_slots = reinterpret_cast<float*>(base + SM::kInSlots);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + SM::kBars);
    uint64_t* empty = full + NS;
    uint64_t* bar_part = full + 2 * NS;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int rank = static_cast<int>(ta_ctarank());
    const int ncta = static_cast<int>(ta_nctarank());
    const int row = blockIdx.x / ncta;  // (b * Hkv + g) * n_draft + i
    const int i = row % n_draft;
    const int g = (row / n_draft) % Hkv;
    const int b = row / (n_draft * Hkv);
    const int nh = rank < G ? (G - 1 - rank) / ncta + 1 : 0;  // heads merged here
    __shared__ int s_list[kTaList];  // this CTA's blocks (-1: out of range), read once
    __shared__ int s_gen[8];         // per slot: blocks issued into it so far

    if (tid < 8) s_gen[tid] = 0;
    if (tid == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        for (int k = 0; k < NS; ++k) {
            mbar_init(&full[k], 1);
            mbar_init(&empty[k], TPB);
        }
        mbar_init(bar_part, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_part, static_cast<uint32_t>(nh * ncta * kPRow * 4));
    }
    __syncthreads();
    if (ncta > 1) ta_cluster_arrive();  // this CTA's barriers exist; peers wait for it before copying in

    // Q of the draft's G heads (an input of the call, not written by the selection kernels)
    QFrag<D> Q;
    load_q(Q, q + ((static_cast<size_t>(b) * n_draft + i) * Hq + static_cast<size_t>(g) * G) * D, D, G);
    pdl_wait();
    pdl_trigger();
    const int L = kv_len[b];
    const bool len_ok = L >= 1 && L <= L_max;
    const int bt = len_ok ? (L - 1) / BS : -1;
    const int cnt = len_ok ? counts[row] : 0;
    const int* list = idx + static_cast<size_t>(row) * idx_stride;
    const int mine = cnt > rank ? (cnt - rank + ncta - 1) / ncta : 0;
    if (!len_ok && rank == 0 && tid == 0) raise_error(err, kDevErrIndex);
    auto entry_g = [&](int t) {  // the block of this CTA's t-th entry, -1 if it is out of range
        const int blk = list[rank + ncta * t];  // (written by the selection kernel before this one)
        return (blk >= 0 && blk <= bt) ? blk : -1;
    };
    // every thread loads a share of the list once (independent loads), so that neither the
    // producer's issue loop nor the consumers wait on a global load per block
    for (int t = tid; t < min(mine, kTaList); t += kTaThreads) s_list[t] = entry_g(t);
    __syncthreads();
    auto entry = [&](int t) { return t < kTaList ? s_list[t] : entry_g(t); };

    WarpAcc<D> A;
    acc_init(A);
    // block t (its entry already checked) into slot t % NS, counted on full[t % NS]
    auto issue = [&](int t) {
        const int s = t % NS;
        const int blk = entry(t);
        if (blk >= 0) {
            const int krow = (b * Hkv + g) * L_max + blk * BS;
            mbar_arrive_expect_tx(&full[s], 2 * kTile);
#pragma unroll
            for (int sub = 0; sub < D / 64; ++sub) {
                tma_load_2d(base + (2 * s) * kTile + sub * BS * 128, &tm_k, 64 * sub, krow, &full[s]);
                tma_load_2d(base + (2 * s + 1) * kTile + sub * BS * 128, &tm_v, 64 * sub, krow, &full[s]);
            }
        } else {
            raise_error(err, kDevErrIndex);
            mbar_arrive(&full[s]);  // nothing to load: the tiles skip the block
        }
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&s_gen[s]) = t / NS + 1;  // block t is the slot's next phase
    };
    if (lane == 0 && warp < NS && warp < mine) issue(warp);
    // The last CTA of the row also attends the drafts the mask bits name (warp w: draft keys
    // 32w .. 32w + 31), ahead of its block tiles.
    if (rank == ncta - 1 && len_ok && 32 * warp < n_draft) {
        const uint64_t bits = tree_mask[static_cast<size_t>(b) * n_draft + i] >> (32 * warp);
        const int n_rows = n_draft - 32 * warp;
        uint32_t valid = static_cast<uint32_t>(bits);
        if (n_rows < 32) valid &= (1u << n_rows) - 1u;
        const size_t off = ((static_cast<size_t>(b) * Hkv + g) * n_draft + 32 * warp) * D;
        attend32(A, Q, dk + off, dv + off, valid, scale_log2);
    }
    // block tiles: tile tau = t * TPB + h of block t; warp w takes tau = w, w + 8, ...  A warp may
    // reach block t before the block NS earlier in its slot has been read by other warps; it first
    // waits for the slot's generation to show block t issued, so that the parity wait below is on
    // the slot's current phase, never one ahead (which the parity test would take for the last
    // completed one).
    for (int tau = warp; tau < mine * TPB; tau += kTaWarps) {
        const int t = tau / TPB, h = tau % TPB, s = t % NS;
        const uint32_t ph = (t / NS) & 1u;
        const int blk = entry(t);
        bool issued = true;
        if (lane == 0) {
            const volatile int* gen = &s_gen[s];
            if (*gen <= t / NS) {
                const long long t0 = clock64();
                while (*gen <= t / NS)
                    if (clock64() - t0 > kWaitBudgetCycles) {
                        issued = false;
                        break;
                    }
            }
        }
        issued = __shfl_sync(0xffffffffu, issued, 0);
        if (issued && mbar_wait(&full[s], ph)) {
            const int r0 = h * 32;
            const int n_ok = blk >= 0 ? L - (blk * BS + r0) : 0;
            if (n_ok > 0) {
                const uint32_t valid = n_ok >= 32 ? 0xffffffffu : ((1u << n_ok) - 1u);
                attend32_smem<D>(A, Q, smem_u32(base + (2 * s) * kTile), smem_u32(base + (2 * s + 1) * kTile), BS,
                                 r0, valid, scale_log2);
            }
        } else if (lane == 0) {
            raise_error(err, kDevErrTimeout);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[s]);  // this tile of slot s has been read
            if (h == 0 && t + NS < mine) {  // refill once every tile of the slot has been read
                if (!mbar_wait(&empty[s], ph)) raise_error(err, kDevErrTimeout);
                issue(t + NS);
            }
        }
        __syncwarp();
    }
    acc_finish_rowsum(A);
    // every slot has landed and been read: every block's tiles waited for it
    __syncthreads();

    // ---- merge the eight warps into this CTA's partial (scratch in the ring)
    {
        float* sm_m = reinterpret_cast<float*>(base);
        float* sm_l = sm_m + 8 * 16;
        float* sm_o = sm_l + 8 * 16;  // [8][16][kMergeRow]
        auto mpad = [](int col) { return col + 4 * (col >> 5); };
        {
            if (cq == 0) {
                sm_m[warp * 16 + gq] = A.m[0];
                sm_m[warp * 16 + gq + 8] = A.m[1];
                sm_l[warp * 16 + gq] = A.l[0];
                sm_l[warp * 16 + gq + 8] = A.l[1];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int nt = 0; nt < D / 8; nt += 4) {
                    const int col = o_col(D, cq, nt, e);
                    *reinterpret_cast<float4*>(&sm_o[(warp * 16 + gq + 8 * (e >> 1)) * kMergeRow + mpad(col)]) =
                        make_float4(A.o[nt][e], A.o[nt + 1][e], A.o[nt + 2][e], A.o[nt + 3][e]);
                }
        }
        __syncthreads();
        constexpr int kCols = 8, kTpr = D / kCols;
        for (int e0 = tid * kCols; e0 < 16 * D; e0 += kTaThreads * kCols) {
            const int r = e0 / D, col0 = e0 % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 8; ++w) M = fmaxf(M, sm_m[w * 16 + r]);
            const float ref = M == -INFINITY ? 0.f : M;
            float f[8], l = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                f[w] = fast_exp2(sm_m[w * 16 + r] - ref);
                l += sm_l[w * 16 + r] * f[w];
            }
            if ((tid % kTpr) == 0) {
                part[r * kPRow] = M;
                part[r * kPRow + 1] = l;
            }
            float acc[kCols];
#pragma unroll
            for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w)
#pragma unroll
                for (int c = 0; c < kCols; c += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(&sm_o[(w * 16 + r) * kMergeRow + mpad(col0 + c)]);
                    acc[c] += x.x * f[w];
                    acc[c + 1] += x.y * f[w];
                    acc[c + 2] += x.z * f[w];
                    acc[c + 3] += x.w * f[w];
                }
#pragma unroll
            for (int c = 0; c < kCols; c += 4)
                *reinterpret_cast<float4*>(&part[r * kPRow + 4 + col0 + c]) =
                    make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
        }
    }

    // ---- the row's output: head h from the CL partials of head h (CTA h mod CL merges it)
    const float* src;
    int n_src, src_stride, heads_here;
    if (ncta == 1) {
        __syncthreads();
        src = part;
        n_src = 1;
        src_stride = 0;
        heads_here = G;
    } else {
        fence_proxy_async_shared();
        __syncthreads();
        ta_cluster_wait();
        if (warp == 0) {  // lane h copies head h
            const int h = lane;
            if (h < G) {
                const int owner = h % ncta, hl = h / ncta;
                const uint32_t dst = smem_u32(in_slots) + 4u * static_cast<uint32_t>((hl * ncta + rank) * kPRow);
                ta_copy_to_peer(ta_mapa(dst, owner), smem_u32(part + h * kPRow), kPRow * 4,
                                ta_mapa(smem_u32(bar_part), owner));
            }
            bulk_commit();
        }
        if (!mbar_wait(bar_part, 0) && tid == 0) raise_error(err, kDevErrTimeout);
        src = in_slots;
        n_src = ncta;
        src_stride = kPRow;
        heads_here = nh;
    }
    // heads_here heads: local head hl is head rank + ncta * hl (ncta == 1: hl itself); its partials
    // sit at src + (hl * n_src + j) * kPRow (ncta == 1: part + hl * kPRow)
    for (int e = tid; e < heads_here * D; e += kTaThreads) {
        const int hl = e / D, d = e % D;
        const int h = ncta == 1 ? hl : rank + ncta * hl;
        const float* ph = ncta == 1 ? part + hl * kPRow : src + hl * n_src * src_stride;
        float M = -INFINITY;
        for (int j = 0; j < n_src; ++j) M = fmaxf(M, ph[j * kPRow]);
        const float ref = M == -INFINITY ? 0.f : M;
        float Ls = 0.f, acc = 0.f;
        for (int j = 0; j < n_src; ++j) {
            const float f = fast_exp2(ph[j * kPRow] - ref);
            Ls += ph[j * kPRow + 1] * f;
            acc += ph[j * kPRow + 4 + d] * f;
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const int hq = g * G + h;
        o[((static_cast<size_t>(b) * n_draft + i) * Hq + hq) * D + d] = __float2bfloat16_rn(acc * inv);
        if (lse != nullptr && d == 0)
            lse[(static_cast<size_t>(b) * Hq + hq) * n_draft + i] =
                Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994530942f : -INFINITY;
    }
    // this CTA's copies have read its partials before it exits
    if (ncta > 1 && warp == 0) bulk_wait_read_all();
}

bool tree_attention_supported(const DecodeArgs& a) {
    const int G = a.Hkv > 0 ? a.Hq / a.Hkv : 0;
    if (a.tree_mask == nullptr || a.n_draft < 1 || a.n_draft > 64) return false;
    if (G < 1 || G > 16 || (a.d != 64 && a.d != 128)) return false;
    const int bs = a.p.block_size;
    if (bs != 64 && bs != 128) return false;
    return static_cast<long long>(a.B) * a.Hkv * a.L_max >= bs;  // the tensor maps' boxes fit
}

template <int D, int BS>
static cudaError_t launch_tree_t(const DecodeArgs& a, const int* idx, const int* counts, int idx_stride) {
    using SM = TreeSmem<D, BS>;
    constexpr int smem = SM::kBytes;
    auto kfn = tree_attn_kernel<D, BS>;
    const int rows = a.B * a.Hkv * a.n_draft;
    const int G = a.Hq / a.Hkv;
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    // attributes and the cluster size, settled once per (kernel, device, rows)
    struct Choice {
        const void* fn;
        int dev, rows, CL;
    };
    static std::mutex mtx;
    static std::vector<Choice> choices;
    const void* fn = reinterpret_cast<const void*>(kfn);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kTaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    int CL = 0;
    {
        std::lock_guard<std::mutex> lock(mtx);
        for (const Choice& ch : choices)
            if (ch.fn == fn && ch.dev == dev && ch.rows == rows) CL = ch.CL;
        if (CL == 0) {
            if (cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                e != cudaSuccess)
                return e;
            // the largest cluster whose clusters (one per row) all fit the device at once; else one
            // CTA per row
            cfg.numAttrs = 1;
            CL = 1;
            for (int cand : {8, 4, 2}) {
                attr[0].val.clusterDim.x = cand;
                cfg.gridDim = dim3(cand * rows);
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, kfn, &cfg) != cudaSuccess) {
                    (void)cudaGetLastError();
                    continue;
                }
                if (n >= rows) {
                    CL = cand;
                    break;
                }
            }
            choices.push_back(Choice{fn, dev, rows, CL});
        }
    }
    CUtensorMap tk, tv;
    const uint64_t cache_rows = static_cast<uint64_t>(a.B) * a.Hkv * a.L_max;
    if (!make_tmap_bf16_2d(&tk, a.k_cache, D, cache_rows, 64, BS) ||
        !make_tmap_bf16_2d(&tv, a.v_cache, D, cache_rows, 64, BS))
        return cudaErrorInvalidValue;
    attr[0].val.clusterDim.x = CL;
    cfg.gridDim = dim3(rows * CL);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kfn, tk, tv, static_cast<const __nv_bfloat16*>(a.q),
                              static_cast<const __nv_bfloat16*>(a.draft_k), static_cast<const __nv_bfloat16*>(a.draft_v),
                              a.tree_mask, a.kv_len, idx, counts, idx_stride, a.n_draft, a.Hq, a.Hkv, G, a.L_max,
                              static_cast<__nv_bfloat16*>(a.o), a.lse, a.p.scale * 1.4426950408889634f, a.err);
}

cudaError_t launch_tree_attention(const DecodeArgs& a, const int* idx, const int* counts, int idx_stride) {
    const int bs = a.p.block_size;
    cudaError_t e;
    if (a.d == 128)
        e = bs == 64 ? launch_tree_t<128, 64>(a, idx, counts, idx_stride) : launch_tree_t<128, 128>(a, idx, counts, idx_stride);
    else
        e = bs == 64 ? launch_tree_t<64, 64>(a, idx, counts, idx_stride) : launch_tree_t<64, 128>(a, idx, counts, idx_stride);
    if (e == cudaSuccess) prof_mark(a.stream, "attend");
    return e;
}

}  // namespace infllmv2
