// internal.h -- launch interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace infllmv2 {

struct SelectArgs {
    const void* q;
    const void* kernel_cache;
    const int* kv_len;
    int B, Tq, Hq, Hkv, d, L_max, M_max;
    int tree;  // queries are tree drafts after the cache (all at the last cached position)
    int* idx;
    int* counts;
    int S_max;
    int blocks_per_cta;
    Params p;
    int* err;
    cudaStream_t stream;
    const int* cu_q = nullptr;  // packed variable-length chunks (SeqMap); Tq is then the longest
    int total_q = 0;            // token rows when packed
    SeqMap seqmap() const { return SeqMap{cu_q, Tq, cu_q != nullptr ? total_q : B * Tq}; }
};

struct PrefillArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int* idx;
    const int* counts;
    int S_max;
    const int* kv_len;
    int B, Tq, Hq, Hkv, d, L_max;
    void* o;
    float* lse;
    Params p;
    int* err;
    cudaStream_t stream;
    const int* cu_q = nullptr;  // packed variable-length chunks (SeqMap); Tq is then the longest
    int total_q = 0;            // token rows when packed
    SeqMap seqmap() const { return SeqMap{cu_q, Tq, cu_q != nullptr ? total_q : B * Tq}; }
};

struct DecodeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int* kv_len;
    const void* draft_k;
    const void* draft_v;
    const uint64_t* tree_mask;
    int B, n_draft, Hq, Hkv, d, L_max;
    void* o;
    float* lse;
    Params p;
    int* err;
    cudaStream_t stream;
    // decode-step append (cluster path): the new token's K and V per (sequence, KV head), written
    // with the kernel it completes into the caches below; null = plain decode
    const void* k_new = nullptr;
    const void* v_new = nullptr;
    void* k_w = nullptr;
    void* v_w = nullptr;
    void* kern_w = nullptr;
};

struct BwdArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const void* o;
    const void* dout;
    const float* lse;
    const int* idx;
    const int* counts;
    int S_max;
    const int* kv_len;
    int B, Tq, Hq, Hkv, d, L_max;
    float* dq;
    float* dk;
    float* dv;
    void* workspace;
    Params p;
    int* err;
    cudaStream_t stream;
};

// 2-D bf16 tensor map over `rows` rows of `inner` elements (row stride inner*2 bytes) with
// box [box_rows][box_inner] and the 128-byte swizzle; false if the driver refuses.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                       uint32_t box_rows);
// The same over fp32 elements (row stride inner*4 bytes; box_inner*4 must be at most 128).
bool make_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows);
// 3-D bf16 tensor map over [d2][d1][d0] packed elements (strides d0*2 and d0*d1*2 bytes) with
// box [box2][box1][box0] and the 128-byte swizzle (box0*2 at most 128); false if the driver refuses.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                       uint32_t box1, uint32_t box2);

// Stage timing (infllmv2_profile_*): no-ops unless profiling is enabled.
void prof_begin(cudaStream_t stream);
void prof_mark(cudaStream_t stream, const char* stage);

cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, void* kernel_cache,
                          const int* kv_len, int B, int Hkv, int L_max, int M_max, int d, int c, int s, int* err,
                          cudaStream_t stream);
cudaError_t launch_kernel_pool_seq(const void* k_cache, void* kernel_cache, const int* kv_len, const SeqMap& sm,
                                   int B, int Hkv, int L_max, int M_max, int d, int c, int s, int* err,
                                   cudaStream_t stream);
cudaError_t launch_kernel_pool(const void* k_cache, void* kernel_cache, int B, int Hkv, int L_max,
                               int M_max, int d, int j_first, int n_new, int c, int s,
                               cudaStream_t stream);

int selection_capacity(const Params& p, int L_max);
size_t select_workspace_bytes(int B, int Tq, int Hkv, int L_max, const Params& p);
cudaError_t launch_block_select(const SelectArgs& a, float* S);
bool score_tc_supported(const SelectArgs& a);
cudaError_t launch_score_tc(const SelectArgs& a, float* S);

cudaError_t launch_prefill_attention(const PrefillArgs& a);
bool tc_prefill_supported(const PrefillArgs& a);
cudaError_t launch_prefill_tc(const PrefillArgs& a);

void decode_split_shape(const Params& p, int L_max, bool tree, long long rows, int* blocks_per_split,
                        int* n_split_cache, int* n_split);
size_t decode_partial_bytes(int B, int n_draft, int Hkv, int d, int n_split);
size_t bwd_workspace_bytes(int B, int Tq, int Hq, int Hkv, int L_max, int bs);
cudaError_t launch_attention_bwd(const BwdArgs& a);
// Tensor-core backward (d = 128, block size 128, 16 query heads per KV head) over the work list
// that launch_attention_bwd builds; see bwd_tc.cu.
constexpr int kBwdUnitTok = 128;  // tokens of a block's list per backward work unit
struct BwdTcWork {
    const float2* ld;     // [B*Tq*Hq] (lse * log2 e, dO . O) per query row
    const int4* units;    // work units {b*Hkv + g, block, first, end} into the token lists
    const int* uoff;      // [B*Hkv][nblk + 1] unit offsets per (b, g); [.][nblk] = units of (b, g)
    const int* list;      // token lists per (b, g, block)
    long long list_stride;
    int nblk;
    int* counter;         // zeroed work counter
};
bool bwd_tc_supported(const BwdArgs& a);
cudaError_t launch_bwd_tc(const BwdArgs& a, const BwdTcWork& w);

cudaError_t launch_decode_attention(const DecodeArgs& a, const int* idx, const int* counts, int idx_stride,
                                    float* part);
// Tree verification's attention (draft tree, uint64 masks) with one thread-block cluster per
// (sequence, KV head, draft) row merging in shared memory: o and lse written directly.
bool tree_attention_supported(const DecodeArgs& a);
cudaError_t launch_tree_attention(const DecodeArgs& a, const int* idx, const int* counts, int idx_stride);

// Single-token decode (no draft tree) with one thread-block cluster per row: scores, selection,
// attention and merge, every intermediate in shared memory.  cudaErrorNotSupported when the
// shape or the device is outside what it covers (the caller then runs the separate selection
// and attention kernels).  idx_out / counts_out may be null.
bool decode_cluster_supported(const DecodeArgs& a, int M_max);
// Whether the cluster kernel may append in the same launch: the kernel a new token completes must
// overlap only blocks that are always local (forced), so that this step's scores never need it.
bool decode_cluster_can_append(const Params& p);
cudaError_t launch_decode_cluster(const DecodeArgs& a, const void* kernel_cache, int M_max, int* idx_out,
                                  int idx_stride, int* counts_out);

}  // namespace infllmv2
