// api.cu -- the C ABI of libinfllmv2.so (declared in include/infllmv2.h): argument checks,
// workspace carving and kernel launches.  Nothing here allocates device memory: the caller
// owns every buffer, as in the static-memory design of "CPM.cu：端侧大模型推理的 CUDA 加速引擎"
// (section 4, preallocated KV cache).
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "infllmv2.h"
#include "internal.h"

using infllmv2::Params;

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxDevices = 64;
constexpr int kMaxLen = 1 << 28;
constexpr int kMaxBlocks = 1024 * 32;  // blocks per sequence the top-k kernel holds in registers

// Device error word: bits of infllmv2::kDevErr*, set by kernels, read and cleared by
// infllmv2_sync_status.
__device__ int g_device_error;

std::mutex g_err_mutex;
int* g_err_ptr[kMaxDevices] = {};

int* device_error_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (g_err_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    return g_err_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The device-side address of a host buffer that is page-locked and mapped into the device's
// address space (cudaHostAlloc / cudaMallocHost / cudaHostRegister with mapping), else nullptr.
void* mapped_host(const void* p) {
    if (p == nullptr) return nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// Whether the current device reads and writes pageable host memory coherently through the host's
// page tables (address translation services, as between Grace and the GPU over NVLink-C2C): then
// every host buffer is usable by a kernel at its own address, page-locked or not.  Asked once per
// device.
bool host_memory_direct() {
    static std::once_flag once[kMaxDevices];
    static bool direct[kMaxDevices] = {};
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cur < 0 || cur >= kMaxDevices) return false;
    std::call_once(once[cur], [cur] {
        int pageable = 0, host_tables = 0;
        if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, cur) != cudaSuccess ||
            cudaDeviceGetAttribute(&host_tables, cudaDevAttrPageableMemoryAccessUsesHostPageTables, cur) != cudaSuccess) {
            (void)cudaGetLastError();
            return;
        }
        direct[cur] = pageable != 0 && host_tables != 0;
    });
    return direct[cur];
}

// This host thread's page-locked, mapped error word (allocated on first use, kept until the process
// exits): the zero-copy host-buffer decode gives it to its kernel and reads it back after the wait.
// *dev receives its address on the current device.
volatile int* host_error_word(int** dev) {
    thread_local int* word = nullptr;
    thread_local int* word_dev[kMaxDevices] = {};
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cur < 0 || cur >= kMaxDevices) return nullptr;
    if (word == nullptr) {
        void* h = nullptr;
        if (cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        word = static_cast<int*>(h);
    }
    if (word_dev[cur] == nullptr) {
        void* d = nullptr;
        if (cudaHostGetDevicePointer(&d, word, 0) != cudaSuccess || d == nullptr) {
            (void)cudaGetLastError();
            return nullptr;
        }
        word_dev[cur] = static_cast<int*>(d);
    }
    *dev = word_dev[cur];
    return word;
}

bool supported_group(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16; }

// Checks the parameter struct; fills the kernel-side copy (with the scale resolved for d).
int check_params(const infllmv2_params* in, int d, Params* out) {
    if (in == nullptr) return INFLLMV2_ERR_INVALID_ARG;
    const infllmv2_params& p = *in;
    if (p.kernel_size <= 0 || p.kernel_stride <= 0 || p.topk < 0 || p.n_init_blocks < 0 ||
        p.n_local_blocks < 1 || p.dense_len < 0 || !(p.softmax_scale >= 0.f) || !isfinite(p.softmax_scale))
        return INFLLMV2_ERR_INVALID_ARG;
    if (p.block_size != 64 && p.block_size != 128) return INFLLMV2_ERR_UNSUPPORTED;
    if (p.kernel_size > p.block_size || p.kernel_stride > p.block_size) return INFLLMV2_ERR_UNSUPPORTED;
    out->block_size = p.block_size;
    out->kernel_size = p.kernel_size;
    out->kernel_stride = p.kernel_stride;
    out->topk = p.topk;
    out->n_init = p.n_init_blocks;
    out->n_local = p.n_local_blocks;
    out->dense_len = p.dense_len;
    out->scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf(static_cast<float>(d > 0 ? d : 1));
    return INFLLMV2_OK;
}

int check_heads(int Hq, int Hkv, int d) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return INFLLMV2_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return INFLLMV2_ERR_UNSUPPORTED;
    if (!supported_group(Hq / Hkv)) return INFLLMV2_ERR_UNSUPPORTED;
    return INFLLMV2_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? INFLLMV2_OK : INFLLMV2_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int n_blocks(int L_max, int bs) { return (L_max + bs - 1) / bs; }

// Decode workspace: scores | idx | counts | split partials, each 256-byte aligned.
struct DecodeWs {
    size_t scores, idx, counts, part, total;
};

// Sized for the larger of the tree and the single-token split shapes, whether or not a mask is
// passed.
DecodeWs decode_ws(int B, int n_draft, int Hkv, int d, int L_max, const Params& p) {
    DecodeWs w{};
    const int S_cap = infllmv2::selection_capacity(p, L_max);
    const size_t rows = static_cast<size_t>(B) * Hkv * n_draft;
    int bps, nsc, ns_tree, ns_single;
    infllmv2::decode_split_shape(p, L_max, true, static_cast<long long>(rows), &bps, &nsc, &ns_tree);
    infllmv2::decode_split_shape(p, L_max, false, static_cast<long long>(rows), &bps, &nsc, &ns_single);
    const int ns = ns_tree > ns_single ? ns_tree : ns_single;
    w.scores = 0;
    w.idx = align256(w.scores + rows * n_blocks(L_max, p.block_size) * sizeof(float));
    w.counts = align256(w.idx + rows * S_cap * sizeof(int));
    w.part = align256(w.counts + rows * sizeof(int));
    w.total = align256(w.part + infllmv2::decode_partial_bytes(B, n_draft, Hkv, d, ns));
    return w;
}

int blocks_per_score_cta(const Params& p) { return 2048 / p.block_size; }

// ---- stage timing
constexpr int kMaxStages = 8;
struct ProfState {
    cudaEvent_t ev[kMaxStages + 1] = {};
    const char* name[kMaxStages] = {};
    int n = -1;  // marks recorded after the begin event of the last call
    bool ready = false;
};
bool g_prof_on = false;
ProfState g_prof[kMaxDevices];

ProfState* prof_state() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    ProfState& st = g_prof[dev];
    if (!st.ready) {
        for (auto& e : st.ev)
            if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        st.ready = true;
    }
    return &st;
}

}  // namespace

namespace infllmv2 {

void prof_begin(cudaStream_t stream) {
    if (!g_prof_on) return;
    ProfState* st = prof_state();
    if (st == nullptr) return;
    st->n = 0;
    cudaEventRecord(st->ev[0], stream);
}

void prof_mark(cudaStream_t stream, const char* stage) {
    if (!g_prof_on) return;
    ProfState* st = prof_state();
    if (st == nullptr || st->n < 0 || st->n >= kMaxStages) return;
    st->name[st->n] = stage;
    st->n += 1;
    cudaEventRecord(st->ev[st->n], stream);
}

}  // namespace infllmv2

namespace {
using infllmv2::prof_begin;
using infllmv2::prof_mark;
}  // namespace

extern "C" {

const char* infllmv2_status_string(int status) {
    switch (status) {
        case INFLLMV2_OK: return "ok";
        case INFLLMV2_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or range)";
        case INFLLMV2_ERR_UNSUPPORTED: return "unsupported configuration (head dim, group size, block size)";
        case INFLLMV2_ERR_WORKSPACE: return "workspace missing or too small";
        case INFLLMV2_ERR_CUDA: return "CUDA runtime error";
        case INFLLMV2_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
        case INFLLMV2_ERR_DEVICE_INDEX: return "device saw kv_len or a selected block id out of range";
        case INFLLMV2_ERR_NOT_IMPLEMENTED: return "not implemented";
        default: return "unknown status";
    }
}

int infllmv2_version(void) { return kVersion; }

int infllmv2_profile_enable(int on) {
    g_prof_on = on != 0;
    if (g_prof_on && prof_state() == nullptr) return INFLLMV2_ERR_CUDA;
    return INFLLMV2_OK;
}

int infllmv2_profile_read(float* ms, int max_stages, int* n_stages) {
    ProfState* st = prof_state();
    if (st == nullptr) return INFLLMV2_ERR_CUDA;
    const int n = st->n < 0 ? 0 : st->n;
    if (n_stages != nullptr) *n_stages = n;
    for (int i = 0; i < n && i < max_stages; ++i) {
        if (cudaEventSynchronize(st->ev[i + 1]) != cudaSuccess) return INFLLMV2_ERR_CUDA;
        if (cudaEventElapsedTime(&ms[i], st->ev[i], st->ev[i + 1]) != cudaSuccess) return INFLLMV2_ERR_CUDA;
    }
    return INFLLMV2_OK;
}

const char* infllmv2_profile_stage_name(int i) {
    ProfState* st = prof_state();
    if (st == nullptr || i < 0 || i >= st->n || st->name[i] == nullptr) return "";
    return st->name[i];
}

int infllmv2_sync_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return INFLLMV2_ERR_CUDA;
    int* ep = device_error_ptr();
    if (ep == nullptr) return INFLLMV2_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, ep, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return INFLLMV2_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(ep, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return INFLLMV2_ERR_CUDA;
    }
    if (word & infllmv2::kDevErrTimeout) return INFLLMV2_ERR_DEVICE_TIMEOUT;
    if (word & infllmv2::kDevErrIndex) return INFLLMV2_ERR_DEVICE_INDEX;
    return INFLLMV2_OK;
}

int infllmv2_selection_capacity(const infllmv2_params* params, int L_max) {
    Params p;
    if (L_max <= 0 || L_max > kMaxLen || check_params(params, 128, &p) != INFLLMV2_OK) return -1;
    return infllmv2::selection_capacity(p, L_max);
}

size_t infllmv2_workspace_size(int entry, int B, int Tq, int Hq, int Hkv, int d, int L_max,
                               const infllmv2_params* params) {
    Params p;
    if (B < 0 || Tq < 0 || L_max <= 0 || L_max > kMaxLen) return 0;
    if (check_params(params, d, &p) != INFLLMV2_OK || check_heads(Hq, Hkv, d) != INFLLMV2_OK) return 0;
    switch (entry) {
        case INFLLMV2_ENTRY_BLOCK_SELECT: return align256(infllmv2::select_workspace_bytes(B, Tq, Hkv, L_max, p));
        case INFLLMV2_ENTRY_SPARSE_ATTN_FWD: return 0;
        case INFLLMV2_ENTRY_DECODE: return decode_ws(B, Tq, Hkv, d, L_max, p).total;
        case INFLLMV2_ENTRY_SPARSE_ATTN_BWD:
            return align256(infllmv2::bwd_workspace_bytes(B, Tq, Hq, Hkv, L_max, p.block_size));
        default: return 0;
    }
}

int infllmv2_kernel_pool(const void* k_cache, void* kernel_cache, int B, int Hkv, int L_max, int M_max,
                         int d, int tok_begin, int tok_end, const infllmv2_params* params, void* stream) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (d != 64 && d != 128) return INFLLMV2_ERR_UNSUPPORTED;
    if (B < 0 || Hkv <= 0 || L_max <= 0 || L_max > kMaxLen || M_max < 0) return INFLLMV2_ERR_INVALID_ARG;
    if (tok_begin < 0 || tok_begin > tok_end || tok_end > L_max) return INFLLMV2_ERR_INVALID_ARG;
    const int c = p.kernel_size, s = p.kernel_stride;
    const int num = tok_begin - c + 1;
    const int j_first = num <= 0 ? 0 : (num + s - 1) / s;
    const int j_last = tok_end >= c ? (tok_end - c) / s : -1;
    const int n_new = j_last - j_first + 1;
    if (B == 0 || n_new <= 0) return INFLLMV2_OK;
    if (j_last >= M_max) return INFLLMV2_ERR_INVALID_ARG;
    if (!k_cache || !kernel_cache || !aligned16(k_cache) || !aligned16(kernel_cache)) return INFLLMV2_ERR_INVALID_ARG;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    prof_begin(st);
    const cudaError_t e = infllmv2::launch_kernel_pool(k_cache, kernel_cache, B, Hkv, L_max, M_max, d, j_first,
                                                       n_new, c, s, st);
    prof_mark(st, "pool");
    return cuda_status(e);
}

int infllmv2_kernel_pool_varlen(const void* k_cache, void* kernel_cache, const int32_t* kv_len, const int32_t* cu_q,
                                int B, int Hkv, int L_max, int M_max, int d, int Tq_max,
                                const infllmv2_params* params, void* stream) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (d != 64 && d != 128) return INFLLMV2_ERR_UNSUPPORTED;
    if (B < 0 || Hkv <= 0 || L_max <= 0 || L_max > kMaxLen || M_max < 0 || Tq_max < 0 || Tq_max > L_max)
        return INFLLMV2_ERR_INVALID_ARG;
    if (B == 0 || Tq_max == 0 || M_max == 0) return INFLLMV2_OK;
    if (!k_cache || !kernel_cache || !kv_len || !cu_q || !aligned16(k_cache) || !aligned16(kernel_cache) ||
        !aligned16(kv_len))
        return INFLLMV2_ERR_INVALID_ARG;
    int* err = device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    prof_begin(st);
    const cudaError_t e = infllmv2::launch_kernel_pool_seq(k_cache, kernel_cache, kv_len,
                                                           infllmv2::SeqMap{cu_q, Tq_max, 0}, B, Hkv, L_max, M_max, d,
                                                           p.kernel_size, p.kernel_stride, err, st);
    prof_mark(st, "pool");
    return cuda_status(e);
}

int infllmv2_block_select_varlen(const void* q, const void* kernel_cache, const int32_t* kv_len, const int32_t* cu_q,
                                 int B, int Tq_max, int total_q, int Hq, int Hkv, int d, int L_max, int M_max,
                                 int32_t* idx, int32_t* counts, int S_max, void* workspace, size_t ws_bytes,
                                 const infllmv2_params* params, void* stream) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (int rc = check_heads(Hq, Hkv, d)) return rc;
    if (B < 0 || Tq_max < 0 || total_q < 0 || L_max <= 0 || L_max > kMaxLen || M_max < 0) return INFLLMV2_ERR_INVALID_ARG;
    if (B == 0 || Tq_max == 0 || total_q == 0) return INFLLMV2_OK;
    if (Tq_max > L_max || Tq_max > total_q) return INFLLMV2_ERR_INVALID_ARG;
    if (S_max < infllmv2::selection_capacity(p, L_max)) return INFLLMV2_ERR_INVALID_ARG;
    if (n_blocks(L_max, p.block_size) > kMaxBlocks) return INFLLMV2_ERR_UNSUPPORTED;
    if (!q || !kernel_cache || !kv_len || !cu_q || !idx || !counts) return INFLLMV2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kernel_cache) || !aligned16(kv_len) || !aligned16(idx) || !aligned16(counts))
        return INFLLMV2_ERR_INVALID_ARG;
    const size_t need = align256(infllmv2::select_workspace_bytes(1, total_q, Hkv, L_max, p));
    if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return INFLLMV2_ERR_WORKSPACE;
    int* err = device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    infllmv2::SelectArgs a{q, kernel_cache, kv_len, B, Tq_max, Hq, Hkv, d, L_max, M_max, 0, idx, counts, S_max,
                           blocks_per_score_cta(p), p, err, static_cast<cudaStream_t>(stream)};
    a.cu_q = cu_q;
    a.total_q = total_q;
    prof_begin(a.stream);
    return cuda_status(infllmv2::launch_block_select(a, static_cast<float*>(workspace)));
}

int infllmv2_sparse_attn_fwd_varlen(const void* q, const void* k_cache, const void* v_cache, const int32_t* idx,
                                    const int32_t* counts, int S_max, const int32_t* kv_len, const int32_t* cu_q,
                                    int B, int Tq_max, int total_q, int Hq, int Hkv, int d, int L_max, void* o,
                                    float* lse, const infllmv2_params* params, void* stream) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (int rc = check_heads(Hq, Hkv, d)) return rc;
    if (B < 0 || Tq_max < 0 || total_q < 0 || L_max <= 0 || L_max > kMaxLen) return INFLLMV2_ERR_INVALID_ARG;
    if (B == 0 || Tq_max == 0 || total_q == 0) return INFLLMV2_OK;
    if (Tq_max > L_max || Tq_max > total_q) return INFLLMV2_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !kv_len || !cu_q || !o) return INFLLMV2_ERR_INVALID_ARG;
    if ((idx == nullptr) != (counts == nullptr)) return INFLLMV2_ERR_INVALID_ARG;
    if (idx != nullptr && (S_max <= 0 || !aligned16(idx) || !aligned16(counts))) return INFLLMV2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(kv_len))
        return INFLLMV2_ERR_INVALID_ARG;
    if (lse != nullptr && !aligned16(lse)) return INFLLMV2_ERR_INVALID_ARG;
    int* err = device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    infllmv2::PrefillArgs a{q, k_cache, v_cache, idx, counts, S_max, kv_len, B, Tq_max, Hq, Hkv, d, L_max,
                            o, lse, p, err, static_cast<cudaStream_t>(stream)};
    a.cu_q = cu_q;
    a.total_q = total_q;
    prof_begin(a.stream);
    const cudaError_t e = infllmv2::launch_prefill_attention(a);
    prof_mark(a.stream, "attend");
    return cuda_status(e);
}

int infllmv2_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, void* kernel_cache,
                    const int32_t* kv_len, int B, int Hkv, int d, int L_max, int M_max, const infllmv2_params* params,
                    void* stream) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (d != 64 && d != 128) return INFLLMV2_ERR_UNSUPPORTED;
    if (B < 0 || Hkv <= 0 || L_max <= 0 || L_max > kMaxLen || M_max < 0) return INFLLMV2_ERR_INVALID_ARG;
    if (B == 0) return INFLLMV2_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !kv_len || (M_max > 0 && !kernel_cache)) return INFLLMV2_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(kv_len) ||
        (kernel_cache && !aligned16(kernel_cache)))
        return INFLLMV2_ERR_INVALID_ARG;
    int* err = device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    prof_begin(st);
    const cudaError_t e = infllmv2::launch_append(k_new, v_new, k_cache, v_cache, kernel_cache, kv_len, B, Hkv, L_max,
                                                  M_max, d, p.kernel_size, p.kernel_stride, err, st);
    prof_mark(st, "append");
    return cuda_status(e);
}

int infllmv2_block_select(const void* q, const void* kernel_cache, const int32_t* kv_len, int B, int Tq, int Hq,
                          int Hkv, int d, int L_max, int M_max, int32_t* idx, int32_t* counts, int S_max,
                          void* workspace, size_t ws_bytes, const infllmv2_params* params, void* stream) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (int rc = check_heads(Hq, Hkv, d)) return rc;
    if (B < 0 || Tq < 0 || L_max <= 0 || L_max > kMaxLen || M_max < 0) return INFLLMV2_ERR_INVALID_ARG;
    if (B == 0 || Tq == 0) return INFLLMV2_OK;
    if (Tq > L_max) return INFLLMV2_ERR_INVALID_ARG;
    if (S_max < infllmv2::selection_capacity(p, L_max)) return INFLLMV2_ERR_INVALID_ARG;
    if (n_blocks(L_max, p.block_size) > kMaxBlocks) return INFLLMV2_ERR_UNSUPPORTED;
    if (!q || !kernel_cache || !kv_len || !idx || !counts) return INFLLMV2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kernel_cache) || !aligned16(kv_len) || !aligned16(idx) || !aligned16(counts))
        return INFLLMV2_ERR_INVALID_ARG;
    const size_t need = align256(infllmv2::select_workspace_bytes(B, Tq, Hkv, L_max, p));
    if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return INFLLMV2_ERR_WORKSPACE;
    int* err = device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    infllmv2::SelectArgs a{q, kernel_cache, kv_len, B, Tq, Hq, Hkv, d, L_max, M_max, 0, idx, counts, S_max,
                           blocks_per_score_cta(p), p, err, static_cast<cudaStream_t>(stream)};
    prof_begin(a.stream);
    return cuda_status(infllmv2::launch_block_select(a, static_cast<float*>(workspace)));
}

int infllmv2_sparse_attn_fwd(const void* q, const void* k_cache, const void* v_cache, const int32_t* idx,
                             const int32_t* counts, int S_max, const int32_t* kv_len, int B, int Tq, int Hq,
                             int Hkv, int d, int L_max, void* o, float* lse, void* workspace, size_t ws_bytes,
                             const infllmv2_params* params, void* stream) {
    (void)workspace;
    (void)ws_bytes;
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (int rc = check_heads(Hq, Hkv, d)) return rc;
    if (B < 0 || Tq < 0 || L_max <= 0 || L_max > kMaxLen) return INFLLMV2_ERR_INVALID_ARG;
    if (B == 0 || Tq == 0) return INFLLMV2_OK;
    if (Tq > L_max) return INFLLMV2_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !kv_len || !o) return INFLLMV2_ERR_INVALID_ARG;
    if ((idx == nullptr) != (counts == nullptr)) return INFLLMV2_ERR_INVALID_ARG;
    if (idx != nullptr && (S_max <= 0 || !aligned16(idx) || !aligned16(counts))) return INFLLMV2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(kv_len))
        return INFLLMV2_ERR_INVALID_ARG;
    if (lse != nullptr && !aligned16(lse)) return INFLLMV2_ERR_INVALID_ARG;
    int* err = device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    infllmv2::PrefillArgs a{q, k_cache, v_cache, idx, counts, S_max, kv_len, B, Tq, Hq, Hkv, d, L_max,
                            o, lse, p, err, static_cast<cudaStream_t>(stream)};
    prof_begin(a.stream);
    const cudaError_t e = infllmv2::launch_prefill_attention(a);
    prof_mark(a.stream, "attend");
    return cuda_status(e);
}

int infllmv2_sparse_attn_bwd(const void* q, const void* k_cache, const void* v_cache, const void* o,
                             const float* lse, const void* dout, const int32_t* idx, const int32_t* counts,
                             int S_max, const int32_t* kv_len, int B, int Tq, int Hq, int Hkv, int d, int L_max,
                             float* dq, float* dk, float* dv, void* workspace, size_t ws_bytes,
                             const infllmv2_params* params, void* stream) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (int rc = check_heads(Hq, Hkv, d)) return rc;
    if (B < 0 || Tq < 0 || L_max <= 0 || L_max > kMaxLen) return INFLLMV2_ERR_INVALID_ARG;
    if (B == 0 || Tq == 0) return INFLLMV2_OK;
    if (Tq > L_max) return INFLLMV2_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !o || !lse || !dout || !kv_len || !dq || !dk || !dv)
        return INFLLMV2_ERR_INVALID_ARG;
    if ((idx == nullptr) != (counts == nullptr)) return INFLLMV2_ERR_INVALID_ARG;
    if (idx != nullptr && (S_max <= 0 || !aligned16(idx) || !aligned16(counts))) return INFLLMV2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(dout) || !aligned16(kv_len) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return INFLLMV2_ERR_INVALID_ARG;
    const size_t need = align256(infllmv2::bwd_workspace_bytes(B, Tq, Hq, Hkv, L_max, p.block_size));
    if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return INFLLMV2_ERR_WORKSPACE;
    int* err = device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    infllmv2::BwdArgs a{q, k_cache, v_cache, o, dout, lse, idx, counts, S_max, kv_len, B, Tq, Hq, Hkv, d, L_max,
                        dq, dk, dv, workspace, p, err, static_cast<cudaStream_t>(stream)};
    prof_begin(a.stream);  // stages "bwd_prep" (inverse of the selection) and "bwd_grad" (the gradients)
    return cuda_status(infllmv2::launch_attention_bwd(a));
}

static int decode_impl(bool launch, const void* q, const void* k_cache, const void* v_cache, const void* kernel_cache,
                       const int32_t* kv_len, const void* draft_k, const void* draft_v, const uint64_t* tree_mask,
                       int B, int n_draft, int Hq, int Hkv, int d, int L_max, int M_max, void* o, float* lse,
                       int32_t* idx_out, int32_t* counts_out, int S_max, void* workspace, size_t ws_bytes,
                       const infllmv2_params* params, void* stream, int* err_word = nullptr,
                       bool cluster_only = false);

int infllmv2_decode(const void* q, const void* k_cache, const void* v_cache, const void* kernel_cache,
                    const int32_t* kv_len, const void* draft_k, const void* draft_v, const uint64_t* tree_mask,
                    int B, int n_draft, int Hq, int Hkv, int d, int L_max, int M_max, void* o, float* lse,
                    int32_t* idx_out, int32_t* counts_out, int S_max, void* workspace, size_t ws_bytes,
                    const infllmv2_params* params, void* stream) {
    return decode_impl(true, q, k_cache, v_cache, kernel_cache, kv_len, draft_k, draft_v, tree_mask, B, n_draft, Hq, Hkv,
                       d, L_max, M_max, o, lse, idx_out, counts_out, S_max, workspace, ws_bytes, params, stream);
}

int infllmv2_host_memory_direct(int* direct) {
    if (direct == nullptr) return INFLLMV2_ERR_INVALID_ARG;
    *direct = host_memory_direct() ? 1 : 0;
    return INFLLMV2_OK;
}

int infllmv2_decode_host(const void* q_host, const int32_t* kv_len_host, void* o_host, float* lse_host, void* q_dev,
                         int32_t* kv_len_dev, void* o_dev, float* lse_dev, const void* k_cache, const void* v_cache,
                         const void* kernel_cache, int B, int Hq, int Hkv, int d, int L_max, int M_max, void* workspace,
                         size_t ws_bytes, const infllmv2_params* params, void* stream) {
    if (lse_host != nullptr && lse_dev == nullptr) return INFLLMV2_ERR_INVALID_ARG;
    if (int rc = decode_impl(false, q_dev, k_cache, v_cache, kernel_cache, kv_len_dev, nullptr, nullptr, nullptr, B, 1,
                             Hq, Hkv, d, L_max, M_max, o_dev, lse_dev, nullptr, nullptr, 0, workspace, ws_bytes, params,
                             stream))
        return rc;
    if (B == 0) return INFLLMV2_OK;
    if (q_host == nullptr || kv_len_host == nullptr || o_host == nullptr) return INFLLMV2_ERR_INVALID_ARG;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Zero-copy: when every host buffer is page-locked and mapped (and 16-byte aligned), the
    // single-kernel decode reads q and the lengths and writes o and lse straight through host
    // memory (NVLink-C2C between Grace and the GPU), its errors go to this thread's page-locked
    // error word, and the call is one launch and one wait.
    {
        const bool direct = host_memory_direct();
        auto dev_view = [direct](const void* h) { return direct ? const_cast<void*>(h) : mapped_host(h); };
        void* qm = dev_view(q_host);
        void* km = qm != nullptr ? dev_view(kv_len_host) : nullptr;
        void* om = km != nullptr ? dev_view(o_host) : nullptr;
        void* lm = (om != nullptr && lse_host != nullptr) ? dev_view(lse_host) : nullptr;
        int* wd = nullptr;
        volatile int* wh = (om != nullptr && (lse_host == nullptr || lm != nullptr)) ? host_error_word(&wd) : nullptr;
        if (wh != nullptr && aligned16(qm) && aligned16(km) && aligned16(om) && (lm == nullptr || aligned16(lm))) {
            *wh = 0;
            const int rc = decode_impl(true, qm, k_cache, v_cache, kernel_cache, static_cast<const int32_t*>(km), nullptr,
                                       nullptr, nullptr, B, 1, Hq, Hkv, d, L_max, M_max, om, static_cast<float*>(lm),
                                       nullptr, nullptr, 0, workspace, ws_bytes, params, stream, wd, true);
            if (rc != INFLLMV2_ERR_UNSUPPORTED) {
                if (rc != INFLLMV2_OK) return rc;
                if (cudaStreamSynchronize(st) != cudaSuccess) return INFLLMV2_ERR_CUDA;
                const int word = *wh;
                if (word != 0)
                    return (word & infllmv2::kDevErrTimeout) ? INFLLMV2_ERR_DEVICE_TIMEOUT : INFLLMV2_ERR_DEVICE_INDEX;
                return INFLLMV2_OK;
            }
        }
    }
    // Otherwise: the caller's device staging buffers, one copy per buffer each way.
    int* ep = device_error_ptr();
    if (ep == nullptr) return INFLLMV2_ERR_CUDA;
    const size_t nq = static_cast<size_t>(B) * Hq * d * 2, nl = static_cast<size_t>(B) * Hq * sizeof(float);
    int rc = INFLLMV2_OK;
    if (cudaMemcpyAsync(q_dev, q_host, nq, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(kv_len_dev, kv_len_host, static_cast<size_t>(B) * sizeof(int32_t), cudaMemcpyHostToDevice,
                        st) != cudaSuccess)
        rc = INFLLMV2_ERR_CUDA;
    if (rc == INFLLMV2_OK)
        rc = decode_impl(true, q_dev, k_cache, v_cache, kernel_cache, kv_len_dev, nullptr, nullptr, nullptr, B, 1, Hq, Hkv,
                         d, L_max, M_max, o_dev, lse_dev, nullptr, nullptr, 0, workspace, ws_bytes, params, stream);
    if (rc == INFLLMV2_OK &&
        (cudaMemcpyAsync(o_host, o_dev, nq, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
         (lse_host != nullptr && cudaMemcpyAsync(lse_host, lse_dev, nl, cudaMemcpyDeviceToHost, st) != cudaSuccess)))
        rc = INFLLMV2_ERR_CUDA;
    // the device error word, in the same round trip (a copy to pageable memory returns when done)
    int word = 0;
    if (cudaMemcpyAsync(&word, ep, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess && rc == INFLLMV2_OK)
        rc = INFLLMV2_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess && rc == INFLLMV2_OK) rc = INFLLMV2_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(ep, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess && rc == INFLLMV2_OK)
            rc = INFLLMV2_ERR_CUDA;
        if (rc == INFLLMV2_OK)
            rc = (word & infllmv2::kDevErrTimeout) ? INFLLMV2_ERR_DEVICE_TIMEOUT : INFLLMV2_ERR_DEVICE_INDEX;
    }
    return rc;
}

int infllmv2_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         void* kernel_cache, const int32_t* kv_len, int B, int Hq, int Hkv, int d, int L_max, int M_max,
                         void* o, float* lse, int32_t* idx_out, int32_t* counts_out, int S_max, void* workspace,
                         size_t ws_bytes, const infllmv2_params* params, void* stream) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (int rc = check_heads(Hq, Hkv, d)) return rc;
    if (B < 0 || L_max <= 0 || L_max > kMaxLen || M_max < 0) return INFLLMV2_ERR_INVALID_ARG;
    if (B == 0) return INFLLMV2_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !kernel_cache || !kv_len || !o) return INFLLMV2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(kernel_cache) || !aligned16(kv_len) || !aligned16(o) || (lse != nullptr && !aligned16(lse)))
        return INFLLMV2_ERR_INVALID_ARG;
    if (n_blocks(L_max, p.block_size) > kMaxBlocks) return INFLLMV2_ERR_UNSUPPORTED;
    const int S_cap = infllmv2::selection_capacity(p, L_max);
    if ((idx_out == nullptr) != (counts_out == nullptr)) return INFLLMV2_ERR_INVALID_ARG;
    if (idx_out != nullptr && (S_max < S_cap || !aligned16(idx_out) || !aligned16(counts_out)))
        return INFLLMV2_ERR_INVALID_ARG;
    const DecodeWs w = decode_ws(B, 1, Hkv, d, L_max, p);
    if (workspace == nullptr || ws_bytes < w.total || !aligned16(workspace)) return INFLLMV2_ERR_WORKSPACE;
    int* err = device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    infllmv2::DecodeArgs da{q, k_cache, v_cache, kv_len, nullptr, nullptr, nullptr, B, 1, Hq, Hkv, d, L_max,
                            o, lse, p, err, st};
    if (M_max > 0 && infllmv2::decode_cluster_can_append(p) && infllmv2::decode_cluster_supported(da, M_max)) {
        da.k_new = k_new;
        da.v_new = v_new;
        da.k_w = k_cache;
        da.v_w = v_cache;
        da.kern_w = kernel_cache;
        prof_begin(st);
        const cudaError_t e = infllmv2::launch_decode_cluster(da, kernel_cache, M_max, idx_out, S_max, counts_out);
        if (e != cudaErrorNotSupported) {
            prof_mark(st, "fused");
            return cuda_status(e);
        }
        (void)cudaGetLastError();  // not launched: append, then decode
    }
    if (int rc = cuda_status(infllmv2::launch_append(k_new, v_new, k_cache, v_cache, kernel_cache, kv_len, B, Hkv, L_max,
                                                     M_max, d, p.kernel_size, p.kernel_stride, err, st)))
        return rc;
    return infllmv2_decode(q, k_cache, v_cache, kernel_cache, kv_len, nullptr, nullptr, nullptr, B, 1, Hq, Hkv, d, L_max,
                           M_max, o, lse, idx_out, counts_out, S_max, workspace, ws_bytes, params, stream);
}

// infllmv2_decode's body; with launch == false it only checks the arguments (no CUDA call).
// err_word: the error word the kernels set (default: the library's device word).  cluster_only:
// return INFLLMV2_ERR_UNSUPPORTED (having launched nothing) unless the single-kernel decode covers
// the call -- the zero-copy host path uses it, because that kernel reads q and the lengths and
// writes o and lse with plain loads and stores only.
static int decode_impl(bool launch, const void* q, const void* k_cache, const void* v_cache, const void* kernel_cache,
                       const int32_t* kv_len, const void* draft_k, const void* draft_v, const uint64_t* tree_mask,
                       int B, int n_draft, int Hq, int Hkv, int d, int L_max, int M_max, void* o, float* lse,
                       int32_t* idx_out, int32_t* counts_out, int S_max, void* workspace, size_t ws_bytes,
                       const infllmv2_params* params, void* stream, int* err_word, bool cluster_only) {
    Params p;
    if (int rc = check_params(params, d, &p)) return rc;
    if (int rc = check_heads(Hq, Hkv, d)) return rc;
    if (B < 0 || n_draft < 0 || L_max <= 0 || L_max > kMaxLen || M_max < 0) return INFLLMV2_ERR_INVALID_ARG;
    const bool tree = tree_mask != nullptr;
    if (!tree && n_draft > 1) return INFLLMV2_ERR_INVALID_ARG;
    if (tree && n_draft > 64) return INFLLMV2_ERR_UNSUPPORTED;
    if (B == 0 || n_draft == 0) return INFLLMV2_OK;
    if (!q || !k_cache || !v_cache || !kernel_cache || !kv_len || !o) return INFLLMV2_ERR_INVALID_ARG;
    if (tree && (!draft_k || !draft_v || !aligned16(draft_k) || !aligned16(draft_v) ||
                 (reinterpret_cast<uintptr_t>(tree_mask) & 7u) != 0))
        return INFLLMV2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(kernel_cache) ||
        !aligned16(kv_len) || !aligned16(o))
        return INFLLMV2_ERR_INVALID_ARG;
    if (lse != nullptr && !aligned16(lse)) return INFLLMV2_ERR_INVALID_ARG;
    if (n_blocks(L_max, p.block_size) > kMaxBlocks) return INFLLMV2_ERR_UNSUPPORTED;
    const int S_cap = infllmv2::selection_capacity(p, L_max);
    if ((idx_out == nullptr) != (counts_out == nullptr)) return INFLLMV2_ERR_INVALID_ARG;
    if (idx_out != nullptr && (S_max < S_cap || !aligned16(idx_out) || !aligned16(counts_out)))
        return INFLLMV2_ERR_INVALID_ARG;
    const DecodeWs w = decode_ws(B, n_draft, Hkv, d, L_max, p);
    if (workspace == nullptr || ws_bytes < w.total || !aligned16(workspace)) return INFLLMV2_ERR_WORKSPACE;
    if (!launch) return INFLLMV2_OK;
    int* err = err_word != nullptr ? err_word : device_error_ptr();
    if (err == nullptr) return INFLLMV2_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    int* idx = idx_out != nullptr ? idx_out : reinterpret_cast<int*>(ws + w.idx);
    int* counts = counts_out != nullptr ? counts_out : reinterpret_cast<int*>(ws + w.counts);
    const int stride = idx_out != nullptr ? S_max : S_cap;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    infllmv2::DecodeArgs da{q, k_cache, v_cache, kv_len, draft_k, draft_v, tree_mask, B, n_draft, Hq, Hkv, d, L_max,
                            o, lse, p, err, st};
    if (cluster_only && !infllmv2::decode_cluster_supported(da, M_max)) return INFLLMV2_ERR_UNSUPPORTED;
    prof_begin(st);
    if (infllmv2::decode_cluster_supported(da, M_max)) {
        const cudaError_t e = infllmv2::launch_decode_cluster(da, kernel_cache, M_max, idx_out, S_max, counts_out);
        if (e != cudaErrorNotSupported) {
            prof_mark(st, "fused");
            return cuda_status(e);
        }
        (void)cudaGetLastError();  // not launched: take the separate kernels
        if (cluster_only) return INFLLMV2_ERR_UNSUPPORTED;
    }
    infllmv2::SelectArgs sa{q, kernel_cache, kv_len, B, n_draft, Hq, Hkv, d, L_max, M_max, tree ? 1 : 0, idx, counts,
                            stride, blocks_per_score_cta(p), p, err, st};
    if (int rc = cuda_status(infllmv2::launch_block_select(sa, reinterpret_cast<float*>(ws + w.scores)))) return rc;
    if (tree && infllmv2::tree_attention_supported(da))
        return cuda_status(infllmv2::launch_tree_attention(da, idx, counts, stride));
    return cuda_status(
        infllmv2::launch_decode_attention(da, idx, counts, stride, reinterpret_cast<float*>(ws + w.part)));
}

}  // extern "C"
