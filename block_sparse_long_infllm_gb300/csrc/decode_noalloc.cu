// decode_noalloc.cu -- infllmv2_decode_noalloc: single-token decode and tree verification for
// callers that cannot hand the library a workspace buffer.
//
// Who needs it: some programs cannot (or may not) obtain device memory at the point where
// they decode.  A process whose whole device memory is reserved up front by its own pool
// has nothing left for a raw cudaMalloc; a plugin inside a host application often receives
// only its input and output pointers and no way to ask for scratch; a latency-critical loop
// may forbid allocation after start-up because cudaMalloc can synchronise the device and
// take unbounded time.  infllmv2_decode needs scratch (block scores, the selection, the
// split-KV partials), so this variant takes it from one fixed array that lives in the
// library itself instead.
//
// The array is a file-scope __device__ object of INFLLMV2_NOALLOC_SCRATCH_BYTES: every GPU
// that loads the library holds it until the process exits.  Host code may not use the
// array's name as a device address (in host code it names a host-side shadow), so the
// first call on each device looks up the real address with cudaGetSymbolAddress while that
// device is current, and later calls on the device reuse it.  That first call should
// therefore come before any stream capture.
//
// All calls share the one array and it keeps the previous call's contents.  Nothing in it
// has to start at zero: every region the decode kernels read (scores, selection, partials)
// is written earlier in the same call.  Calls whose work overlaps on the GPU (different
// streams, or different host threads) race on the array and must be serialised by the
// caller.  No cudaMalloc, cudaFree or allocating library routine is called.
#include <cuda_runtime.h>

#include <mutex>

#include "infllmv2.h"

namespace {

constexpr size_t kScratchBytes = INFLLMV2_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once per device).
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int infllmv2_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const void* kernel_cache, const int32_t* kv_len, const void* draft_k,
                                       const void* draft_v, const uint64_t* tree_mask, int B, int n_draft,
                                       int Hq, int Hkv, int d, int L_max, int M_max, void* o, float* lse,
                                       int32_t* idx_out, int32_t* counts_out, int S_max,
                                       const infllmv2_params* params, void* stream) {
    if (B > 0 && n_draft > 0) {
        const size_t need =
            infllmv2_workspace_size(INFLLMV2_ENTRY_DECODE, B, n_draft, Hq, Hkv, d, L_max, params);
        if (need > kScratchBytes) return INFLLMV2_ERR_WORKSPACE;  // the problem exceeds the fixed scratch
    }
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return INFLLMV2_ERR_CUDA;
    return infllmv2_decode(q, k_cache, v_cache, kernel_cache, kv_len, draft_k, draft_v, tree_mask, B, n_draft,
                           Hq, Hkv, d, L_max, M_max, o, lse, idx_out, counts_out, S_max, scratch, kScratchBytes,
                           params, stream);
}
