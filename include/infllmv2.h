/*
 * infllmv2.h -- C ABI of libinfllmv2.so: InfLLM v2 trainable block-sparse
 * attention (semantic-kernel pooling, block scoring, top-k block selection,
 * block-sparse flash attention) for NVIDIA GB300 (sm_103a).
 *
 * The method, as the pages describe it:
 *   [MiniCPM4-1.1]  "MiniCPM4: 如何在手机电脑上高效运行大语言模型"
 *                   (xugj520.cn), section 1.1 "InfLLM v2" -- context split into
 *                   blocks; overlapping semantic kernels of 32 tokens, stride
 *                   16; each query keeps its top-K most relevant blocks; the
 *                   opening tokens and the sliding window are always kept;
 *                   attention runs on the kept blocks only; kernel-level
 *                   relevance avoids token-level work; a uint64-packed mask
 *                   supports tree-speculative decoding.
 *   [MiniCPM4.0-sparse] "MiniCPM40极速狂飙端侧模型的比赛结束了"
 *                   (shadowrocket9.top), section "InfLLM v2：重新定义注意力
 *                   机制" -- 64-token blocks, top-64 blocks, dense attention
 *                   below 8192 tokens; its deployment guide sets
 *                   sparse_config = {topk, block_size, dense_len}.
 *   [CPM.cu]        "CPM.cu：端侧大模型推理的 CUDA 加速引擎" (pomoai.com),
 *                   section 4 -- static memory (preallocated KV cache),
 *                   CUDA graphs, chunked prefill.
 * The pages disagree on block size (64 vs 128) and top-k (64 vs 6), so every
 * method parameter is a runtime argument (infllmv2_params).
 *
 * Conventions for every entry point
 *   - Tensors are plain device pointers, row-major, densely packed, 16-byte
 *     aligned (infllmv2_decode_host also takes host buffers, as its comment
 *     says).  bf16 tensors are passed as void*.  Index/length arrays are
 *     device int32.  The caller owns every buffer and the stream; the library
 *     never allocates device memory (the static-memory design of [CPM.cu]).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All work is enqueued on it; calls return before the GPU finishes.
 *   - Argument errors are found on the host and returned before anything is
 *     enqueued.  Errors only the device can see (a kv_len out of range, a
 *     selected block past the query's own block, a wait that ran out) set a
 *     device error word; infllmv2_sync_status() reports and clears it.
 *   - Supported: bf16 Q/K/V; head_dim d in {64, 128}; query heads per KV head
 *     G = Hq/Hkv in {1, 2, 4, 8, 16}; block_size in {64, 128}; kernel_size and
 *     kernel_stride positive with kernel_size <= block_size; n_local_blocks >= 1;
 *     at most 64 draft tokens (one uint64 mask word each).
 *
 * Layouts (B = batch, Tq = queries per sequence, Hq/Hkv = query/KV heads)
 *   q            [B, Tq, Hq, d]        bf16; heads g*G .. g*G+G-1 share KV head g
 *   k_cache      [B, Hkv, L_max, d]    bf16; token x of a sequence is row x
 *   v_cache      [B, Hkv, L_max, d]    bf16
 *   kernel_cache [B, Hkv, M_max, d]    bf16; kernel j = mean of tokens
 *                                      [j*stride, j*stride + kernel_size)
 *   kv_len       [B]                   int32; tokens in the cache, including
 *                                      the tokens of this call
 *   o            [B, Tq, Hq, d]        bf16
 *   lse          [B, Hq, Tq]           fp32, natural-log sum of exp(scale*q.k)
 *   idx          [B, Hkv, Tq, S_max]   int32 selected block ids, ascending,
 *                                      padded with -1
 *   counts       [B, Hkv, Tq]          int32 number of valid entries in idx
 */
#ifndef INFLLMV2_H_
#define INFLLMV2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Method parameters ([MiniCPM4-1.1]; sparse_config of [MiniCPM4.0-sparse]). */
typedef struct infllmv2_params {
    int32_t block_size;      /* tokens per KV block: 64 or 128                        */
    int32_t kernel_size;     /* tokens per semantic kernel (the pages: 32)            */
    int32_t kernel_stride;   /* token stride between kernels (the pages: 16)          */
    int32_t topk;            /* blocks chosen by score, on top of the forced ones     */
    int32_t n_init_blocks;   /* leading blocks always kept ("opening tokens")         */
    int32_t n_local_blocks;  /* blocks ending at the query's own block, always kept   */
    int32_t dense_len;       /* sequences with kv_len < dense_len attend densely      */
    float softmax_scale;     /* 0 selects 1/sqrt(d)                                   */
} infllmv2_params;

typedef enum infllmv2_status {
    INFLLMV2_OK = 0,
    INFLLMV2_ERR_INVALID_ARG = -1,     /* null/misaligned pointer, bad size or range   */
    INFLLMV2_ERR_UNSUPPORTED = -2,     /* d, G, block size ... outside the set above   */
    INFLLMV2_ERR_WORKSPACE = -3,       /* workspace missing or smaller than required   */
    INFLLMV2_ERR_CUDA = -4,            /* a CUDA runtime call failed (launch, ...)     */
    INFLLMV2_ERR_DEVICE_TIMEOUT = -5,  /* a bounded device-side wait ran out           */
    INFLLMV2_ERR_DEVICE_INDEX = -6,    /* device saw kv_len or a block id out of range */
    INFLLMV2_ERR_NOT_IMPLEMENTED = -7
} infllmv2_status;

/* Entry ids for infllmv2_workspace_size. */
enum {
    INFLLMV2_ENTRY_BLOCK_SELECT = 1,
    INFLLMV2_ENTRY_SPARSE_ATTN_FWD = 2,
    INFLLMV2_ENTRY_DECODE = 3,
    INFLLMV2_ENTRY_SPARSE_ATTN_BWD = 4
};

/* Human-readable text of a status code (static storage, never NULL). */
const char* infllmv2_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int infllmv2_version(void);

/*
 * Synchronise `stream`, then report and clear the device error word of the
 * current device.  Returns INFLLMV2_OK, INFLLMV2_ERR_DEVICE_TIMEOUT,
 * INFLLMV2_ERR_DEVICE_INDEX or INFLLMV2_ERR_CUDA.
 */
int infllmv2_sync_status(void* stream);

/*
 * Most selected blocks any query can get for these parameters and an L_max-token
 * cache: topk + n_init + n_local, or every causal block while kv_len < dense_len
 * (whichever is larger, capped at ceil(L_max/block_size)).  idx buffers need at
 * least this many columns (S_max).  Returns -1 on invalid parameters.
 */
int infllmv2_selection_capacity(const infllmv2_params* params, int L_max);

/*
 * Bytes of device workspace an entry point needs (entry = INFLLMV2_ENTRY_*).
 * Tq is the number of queries per sequence (n_draft for decode).  Returns 0
 * for invalid arguments (and for entries that need none).
 */
size_t infllmv2_workspace_size(int entry, int B, int Tq, int Hq, int Hkv, int d, int L_max,
                               const infllmv2_params* params);

/*
 * Step 1, semantic kernels ([MiniCPM4-1.1], semantic-kernel item):
 *   kernel_cache[b,g,j,:] = bf16_rne( (1/kernel_size) * sum of k_cache[b,g,x,:]
 *                           over x in [j*stride, j*stride + kernel_size) )
 * for every kernel j whose last token lies in [tok_begin, tok_end) -- that is,
 * the kernels that become complete once tokens [tok_begin, tok_end) are in the
 * cache.  Call it after appending tokens (a prefill chunk, or each decode token;
 * a new kernel completes every `stride` tokens).  Sums are exact -- integer
 * fixed-point sums of the bf16 inputs under a shared per-column exponent -- and
 * the mean is rounded to bf16 once, nearest-even.
 * Requires 0 <= tok_begin <= tok_end <= L_max and
 * M_max >= (tok_end - kernel_size)/kernel_stride + 1.  Other kernels are untouched.
 */
int infllmv2_kernel_pool(const void* k_cache, void* kernel_cache, int B, int Hkv, int L_max,
                         int M_max, int d, int tok_begin, int tok_end,
                         const infllmv2_params* params, void* stream);

/*
 * Variable-length batched prefill ([CPM.cu] section 4 chunked prefill, many
 * sequences with different chunk lengths in one launch).  Sequence b's chunk is
 * len_b = cu_q[b+1] - cu_q[b] queries: the last len_b tokens of its cache, so
 * query t sits at position kv_len[b] - len_b + t.  Packed layouts (total_q =
 * cu_q[B] query rows; cu_q is device int32 [B+1], ascending, cu_q[0] = 0):
 *   q, o     [total_q, Hq, d]       row cu_q[b] + t
 *   idx      [Hkv, total_q, S_max]  counts [Hkv, total_q]
 *   lse      [Hq, total_q]
 * Tq_max (host) bounds every len_b; total_q (host) is cu_q[B].  A len_b outside
 * [0, Tq_max] or a kv_len[b] < len_b sets the device error word and skips that
 * sequence.  Each varlen call computes exactly what its fixed-chunk counterpart
 * computes for every sequence on its own.
 *
 * infllmv2_kernel_pool_varlen: the kernels completed by each sequence's chunk
 * (step 1, as infllmv2_kernel_pool per sequence).
 */
int infllmv2_kernel_pool_varlen(const void* k_cache, void* kernel_cache, const int32_t* kv_len,
                                const int32_t* cu_q, int B, int Hkv, int L_max, int M_max, int d,
                                int Tq_max, const infllmv2_params* params, void* stream);

/* Steps 2-3 for packed chunks (as infllmv2_block_select per sequence).  Requires
 * ws_bytes >= infllmv2_workspace_size(INFLLMV2_ENTRY_BLOCK_SELECT, 1, total_q, ...). */
int infllmv2_block_select_varlen(const void* q, const void* kernel_cache, const int32_t* kv_len,
                                 const int32_t* cu_q, int B, int Tq_max, int total_q, int Hq,
                                 int Hkv, int d, int L_max, int M_max, int32_t* idx,
                                 int32_t* counts, int S_max, void* workspace, size_t ws_bytes,
                                 const infllmv2_params* params, void* stream);

/* Step 4 for packed chunks (as infllmv2_sparse_attn_fwd per sequence); idx NULL:
 * dense causal attention. */
int infllmv2_sparse_attn_fwd_varlen(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* idx, const int32_t* counts, int S_max,
                                    const int32_t* kv_len, const int32_t* cu_q, int B, int Tq_max,
                                    int total_q, int Hq, int Hkv, int d, int L_max, void* o,
                                    float* lse, const infllmv2_params* params, void* stream);

/*
 * Decode-step append (the per-token cache update of [CPM.cu] section 4, static
 * preallocated caches, together with step 1's pooling; one launch, so a CUDA
 * graph of infllmv2_append + infllmv2_decode is one whole decode step).
 * For every sequence b and KV head g, with p = kv_len[b] - 1 (kv_len counts the
 * new token):
 *   k_cache[b,g,p,:] = k_new[b,g,:];  v_cache[b,g,p,:] = v_new[b,g,:]
 * and, if the new token is the last token of semantic kernel
 *   j = (kv_len[b] - kernel_size) / kernel_stride   (kv_len[b] >= kernel_size and
 *   kv_len[b] - kernel_size divisible by kernel_stride),
 * kernel_cache[b,g,j,:] is computed exactly as infllmv2_kernel_pool does.
 *   k_new, v_new  [B, Hkv, d] bf16, read only.
 *   kv_len        [B] device int32, per sequence (read on the device).
 * kernel_cache may be NULL only when M_max == 0.  Device errors (kv_len[b] < 1 or
 * > L_max, a kernel index >= M_max) set the error word; that row is skipped.
 * Cache rows other than p and kernels other than j are untouched.
 */
int infllmv2_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                    void* kernel_cache, const int32_t* kv_len, int B, int Hkv, int d,
                    int L_max, int M_max, const infllmv2_params* params, void* stream);

/*
 * Steps 2-3, block scores and top-k selection for a causal chunk
 * ([MiniCPM4-1.1] dynamic block selection and local retention;
 * [MiniCPM4.0-sparse] dense switch).  Query t of sequence b sits at position
 * p = kv_len[b] - Tq + t (the chunk is the last Tq tokens of the cache; Tq = 1
 * is single-token decode).  With bt = p / block_size:
 *   S[t,g,blk] = max over heads h of group g and over kernels j that share a
 *                token with blk and end at or before p, of q[t,h] . kernel[j]
 *   forced     = blocks [0, n_init) and [bt - n_local + 1, bt], within [0, bt]
 *   selected   = forced + the topk other blocks <= bt by (S desc, id asc);
 *                every block <= bt when kv_len[b] < dense_len.
 * Writes idx [B,Hkv,Tq,S_max] (ascending, -1 padded) and counts [B,Hkv,Tq].
 * Needs S_max >= infllmv2_selection_capacity(params, L_max), kernels pooled up
 * to kv_len[b], kv_len[b] in [Tq, L_max], and
 * ws_bytes >= infllmv2_workspace_size(INFLLMV2_ENTRY_BLOCK_SELECT, ...).
 * Once the call's work is done, the workspace starts with the scores S as float
 * [B, Hkv, Tq, ceil(L_max / block_size)]: entries of blocks 0..bt of each query
 * of a sequence with kv_len[b] >= dense_len are written, the others are
 * unspecified; they stay there until the workspace is used again.
 */
int infllmv2_block_select(const void* q, const void* kernel_cache, const int32_t* kv_len, int B,
                          int Tq, int Hq, int Hkv, int d, int L_max, int M_max, int32_t* idx,
                          int32_t* counts, int S_max, void* workspace, size_t ws_bytes,
                          const infllmv2_params* params, void* stream);

/*
 * Step 4, block-sparse attention for a causal chunk ([MiniCPM4-1.1], attention
 * on the selected blocks only; chunked prefill of [CPM.cu]).  For query t of
 * sequence b at p = kv_len[b] - Tq + t and head h of group g:
 *   keys = tokens x <= p of the blocks idx[b,g,t,0..counts-1]
 *   o    = softmax_x(scale * q.k_x) v_x    (fp32 online softmax, bf16 output)
 * idx == NULL (and counts == NULL) means dense causal attention (every block).
 * lse may be NULL.  Selected ids must lie in [0, bt] (checked on the device).
 * Requires ws_bytes >= infllmv2_workspace_size(INFLLMV2_ENTRY_SPARSE_ATTN_FWD, ...).
 */
int infllmv2_sparse_attn_fwd(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* idx, const int32_t* counts, int S_max,
                             const int32_t* kv_len, int B, int Tq, int Hq, int Hkv, int d,
                             int L_max, void* o, float* lse, void* workspace, size_t ws_bytes,
                             const infllmv2_params* params, void* stream);

/*
 * Gradients of step 4 for a causal chunk with the selection held fixed (InfLLM
 * v2 is trainable sparse attention, [MiniCPM4-1.1]; the block choice is
 * discrete, so the gradient flows through the attention over the selected
 * keys).  Inputs as for infllmv2_sparse_attn_fwd, plus that call's output o
 * and lse (required here) and dout [B, Tq, Hq, d] bf16.  With P the weights of
 * a row and D = dout . o:
 *   dS = P o (dout v^T - D);  dq = scale dS k;  dk = scale dS^T q;  dv = P^T dout
 * dq [B, Tq, Hq, d] and dk, dv [B, Hkv, L_max, d] are fp32 and overwritten (dk,
 * dv are summed over the heads of a group and over the chunk's rows; cache rows
 * no row attends to get 0).  idx == NULL: dense causal, as in the forward.
 * Requires ws_bytes >= infllmv2_workspace_size(INFLLMV2_ENTRY_SPARSE_ATTN_BWD, ...).
 */
int infllmv2_sparse_attn_bwd(const void* q, const void* k_cache, const void* v_cache, const void* o,
                             const float* lse, const void* dout, const int32_t* idx,
                             const int32_t* counts, int S_max, const int32_t* kv_len, int B, int Tq,
                             int Hq, int Hkv, int d, int L_max, float* dq, float* dk, float* dv,
                             void* workspace, size_t ws_bytes, const infllmv2_params* params,
                             void* stream);

/*
 * Steps 2-4 for decoding: selection from the cached kernels, split-KV
 * attention over the selected blocks, and the merge of the splits.
 *   tree_mask == NULL: single-token decode (n_draft must be 1); the query is
 *     the newest cached token, p = kv_len[b] - 1.
 *   tree_mask != NULL: tree-speculative verification ([MiniCPM4-1.1] uint64
 *     mask; [CPM.cu] tree verification inside flash attention).  n_draft <= 64
 *     draft tokens come after kv_len[b] committed tokens; bit j of
 *     tree_mask[b,i] says draft i attends to draft j (the mask holds the
 *     draft's own bit and its ancestors').  Each draft selects its own blocks
 *     from all cached kernels (bt = the last cached block) and attends to
 *     every cached token of them plus the masked drafts, whose keys and values
 *     come from draft_k/draft_v [B, Hkv, n_draft, d] (not pooled, not cached).
 * q [B, n_draft, Hq, d]; o [B, n_draft, Hq, d]; lse [B, Hq, n_draft] or NULL;
 * idx_out [B, Hkv, n_draft, S_max] / counts_out [B, Hkv, n_draft] receive the
 * selection when not NULL (S_max is ignored when idx_out is NULL).
 * Requires ws_bytes >= infllmv2_workspace_size(INFLLMV2_ENTRY_DECODE, ...).
 * Single-token decode runs as one kernel (one thread-block cluster per
 * (sequence, KV head) row, every intermediate on chip) when the shape allows
 * (G <= 16, d in {64, 128}, block 64/128, at most 4096 blocks); trees and
 * other shapes run separate scoring, top-k, split and merge kernels that use
 * the workspace.  Results are the same either way.
 */
int infllmv2_decode(const void* q, const void* k_cache, const void* v_cache,
                    const void* kernel_cache, const int32_t* kv_len, const void* draft_k,
                    const void* draft_v, const uint64_t* tree_mask, int B, int n_draft, int Hq,
                    int Hkv, int d, int L_max, int M_max, void* o, float* lse, int32_t* idx_out,
                    int32_t* counts_out, int S_max, void* workspace, size_t ws_bytes,
                    const infllmv2_params* params, void* stream);

/*
 * infllmv2_decode of one single-token step whose query, cache lengths and
 * output live in host memory: q_host [B, Hq, d] bf16 and kv_len_host [B] in,
 * o_host [B, Hq, d] bf16 (and lse_host [B, Hq] fp32, when not NULL) out; on
 * return the host output is complete.  Two ways, chosen per call:
 *   - zero-copy: when every host buffer is 16-byte aligned and usable by the
 *     device -- any host memory on a device that reads pageable memory through
 *     the host's page tables (cudaDevAttrPageableMemoryAccess and
 *     ...UsesHostPageTables, as a GPU attached to a Grace CPU), else memory
 *     page-locked and mapped into the device's address space (cudaHostAlloc /
 *     cudaMallocHost, or registered with mapping) -- and the single-kernel
 *     decode covers the shape, that kernel reads q and the lengths and writes
 *     o and lse straight through host memory (on a Grace host, over
 *     NVLink-C2C); the buffers must then be valid host memory of the stated
 *     sizes (the device reads and writes them as they are); device errors go
 *     to a page-locked error word of the calling host thread (allocated on its
 *     first such call, kept until the process exits); one launch and one wait.
 *     The staging buffers are not touched.
 *   - staged: otherwise q and kv_len are copied to the caller's device staging
 *     buffers q_dev, kv_len_dev on `stream` (cudaMemcpyAsync, one per buffer),
 *     infllmv2_decode runs on them into o_dev (and lse_dev), o and lse are
 *     copied back, the device error word is read in the same round trip and
 *     the stream is waited for.
 * q_dev, kv_len_dev, o_dev, lse_dev are the caller's device staging buffers
 * (16-byte aligned; lse_dev is required when lse_host is given; the library
 * allocates no device memory); the other arguments are those of
 * infllmv2_decode (n_draft = 1, no selection output).  Arguments are checked
 * before anything is enqueued.  Returns the first of: an argument error,
 * infllmv2_decode's status, INFLLMV2_ERR_CUDA for a failed copy or wait, and
 * the call's device error (INFLLMV2_ERR_DEVICE_INDEX or _TIMEOUT; the staged
 * way reads and clears the device error word as infllmv2_sync_status does).
 */
int infllmv2_decode_host(const void* q_host, const int32_t* kv_len_host, void* o_host, float* lse_host,
                         void* q_dev, int32_t* kv_len_dev, void* o_dev, float* lse_dev,
                         const void* k_cache, const void* v_cache, const void* kernel_cache, int B,
                         int Hq, int Hkv, int d, int L_max, int M_max, void* workspace,
                         size_t ws_bytes, const infllmv2_params* params, void* stream);

/*
 * Whether infllmv2_decode_host's zero-copy way takes pageable host buffers on
 * the current device: *direct = 1 when the device reads and writes pageable
 * memory coherently through the host's page tables (a GPU attached to a Grace
 * CPU over NVLink-C2C), else 0 (then only page-locked, mapped buffers avoid the
 * staged copies; also 0 when no device can be queried).  Returns INFLLMV2_OK,
 * or INFLLMV2_ERR_INVALID_ARG when direct is NULL.
 */
int infllmv2_host_memory_direct(int* direct);

/*
 * One whole single-token decode step: infllmv2_append (the new token's K and V
 * into row kv_len[b]-1 of the caches, and the semantic kernel it completes),
 * then infllmv2_decode of q over the updated caches ([CPM.cu] section 4: the
 * per-token cache update and attention of a CUDA-graph decode step).  kv_len
 * counts the new token.  Arguments as for those two calls (k_new, v_new
 * [B, Hkv, d] bf16; caches writable; M_max >= 1).  When the kernel the new
 * token completes can only overlap the query's forced local blocks
 * (n_local_blocks >= ceil((kernel_size-1)/block_size) + 1) and the
 * single-kernel decode covers the shape, both happen in that one launch: this
 * step's scores never use the new kernel, so it is pooled alongside.  Otherwise
 * the append kernel runs first.  Results are the same either way.
 */
int infllmv2_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                         void* v_cache, void* kernel_cache, const int32_t* kv_len, int B, int Hq,
                         int Hkv, int d, int L_max, int M_max, void* o, float* lse,
                         int32_t* idx_out, int32_t* counts_out, int S_max, void* workspace,
                         size_t ws_bytes, const infllmv2_params* params, void* stream);

/*
 * Allocation-free decode.  The paper has no counterpart: this entry point is
 * for callers of this library that cannot provide a workspace -- a process whose
 * device memory is reserved up front by its own pool, a plugin that receives
 * only input and output pointers, or a loop that must not allocate after
 * start-up.  It behaves exactly like infllmv2_decode (same arguments without
 * workspace/ws_bytes, same results) but takes its scratch from one fixed array
 * of INFLLMV2_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.
 *   - Problems whose decode workspace (infllmv2_workspace_size with
 *     INFLLMV2_ENTRY_DECODE) exceeds that size are rejected with
 *     INFLLMV2_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on each device looks up the array's device address with
 *     cudaGetSymbolAddress (the device must be current); make that first call
 *     before any stream capture.
 *   - All calls share the array and it keeps the last call's contents (nothing
 *     in it needs to start at zero).  Calls that overlap on the GPU -- other
 *     streams, other host threads -- race on it; serialise them.
 *   - It never calls cudaMalloc, cudaFree or any allocating routine.
 */
#define INFLLMV2_NOALLOC_SCRATCH_BYTES (16u << 20)
int infllmv2_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                            const void* kernel_cache, const int32_t* kv_len, const void* draft_k,
                            const void* draft_v, const uint64_t* tree_mask, int B, int n_draft,
                            int Hq, int Hkv, int d, int L_max, int M_max, void* o, float* lse,
                            int32_t* idx_out, int32_t* counts_out, int S_max,
                            const infllmv2_params* params, void* stream);

/*
 * Stage timing (the pages' CPM.cu lists a performance-analysis module next to
 * the inference entry; this is the library's counterpart).  While enabled,
 * every entry point records a CUDA event on its stream before its first kernel
 * and after each kernel it launches; infllmv2_profile_read then waits for
 * those events and writes the elapsed milliseconds of each stage of the most
 * recent call into ms[0 .. *n_stages-1] (at most max_stages), and
 * infllmv2_profile_stage_name(i) names stage i ("pool", "score", "topk",
 * "attend", "combine").  Events live in the library, per device, created on
 * first use; enabling costs one event record per kernel.  Not thread-safe.
 * Returns INFLLMV2_OK or INFLLMV2_ERR_CUDA.
 */
int infllmv2_profile_enable(int on);
int infllmv2_profile_read(float* ms, int max_stages, int* n_stages);
const char* infllmv2_profile_stage_name(int i);

#ifdef __cplusplus
}
#endif

#endif /* INFLLMV2_H_ */
