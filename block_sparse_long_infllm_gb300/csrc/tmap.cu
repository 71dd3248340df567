// tmap.cu -- host-side construction of TMA tensor maps (driver entry point resolved through the
// runtime, so the library links no libcuda).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace infllmv2 {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

// The last few maps this thread encoded, by their arguments: a map is a pure function of them (the
// driver only checks and packs them), so a repeated call copies the earlier result instead of
// paying the encode again on every launch.
struct TmapKey {
    int type;
    const void* base;
    uint64_t inner, rows;
    uint32_t box_inner, box_rows;
    bool operator==(const TmapKey& o) const {
        return type == o.type && base == o.base && inner == o.inner && rows == o.rows && box_inner == o.box_inner &&
               box_rows == o.box_rows;
    }
};
constexpr int kTmapCache = 64;

static bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType type, uint64_t elem_bytes, const void* base,
                         uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
    thread_local TmapKey keys[kTmapCache];
    thread_local CUtensorMap maps[kTmapCache];
    thread_local int n_cached = 0, next = 0;
    const TmapKey key{static_cast<int>(type), base, inner, rows, box_inner, box_rows};
    for (int i = 0; i < n_cached; ++i)
        if (keys[i] == key) {
            *map = maps[i];
            return true;
        }
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    keys[next] = key;
    maps[next] = *map;
    next = (next + 1) % kTmapCache;
    if (n_cached < kTmapCache) ++n_cached;
    return true;
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                       uint32_t box_rows) {
    return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, rows, box_inner, box_rows);
}

bool make_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows) {
    return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, inner, rows, box_inner, box_rows);
}

}  // namespace infllmv2
