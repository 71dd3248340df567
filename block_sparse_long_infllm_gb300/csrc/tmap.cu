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
    uint64_t dim[3];
    uint32_t box[3];
    bool operator==(const TmapKey& o) const {
        return type == o.type && base == o.base && dim[0] == o.dim[0] && dim[1] == o.dim[1] && dim[2] == o.dim[2] &&
               box[0] == o.box[0] && box[1] == o.box[1] && box[2] == o.box[2];
    }
};
constexpr int kTmapCache = 64;

// A tensor of up to three dimensions (dim[2] == 0: two), packed innermost first, 128-byte swizzle.
static bool make_tmap(CUtensorMap* map, CUtensorMapDataType type, uint64_t elem_bytes, const void* base,
                      const uint64_t (&dim)[3], const uint32_t (&box)[3]) {
    thread_local TmapKey keys[kTmapCache];
    thread_local CUtensorMap maps[kTmapCache];
    thread_local int n_cached = 0, next = 0;
    const TmapKey key{static_cast<int>(type), base, {dim[0], dim[1], dim[2]}, {box[0], box[1], box[2]}};
    for (int i = 0; i < n_cached; ++i)
        if (keys[i] == key) {
            *map = maps[i];
            return true;
        }
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint32_t rank = dim[2] != 0 ? 3 : 2;
    const cuuint64_t dims[3] = {dim[0], dim[1], dim[2]};
    const cuuint64_t strides[2] = {dim[0] * elem_bytes, dim[0] * dim[1] * elem_bytes};
    const cuuint32_t boxes[3] = {box[0], box[1], box[2]};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = fn(map, type, rank, const_cast<void*>(base), dims, strides, boxes, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    keys[next] = key;
    maps[next] = *map;
    next = (next + 1) % kTmapCache;
    if (n_cached < kTmapCache) ++n_cached;
    return true;
}

static bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType type, uint64_t elem_bytes, const void* base,
                         uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
    const uint64_t dim[3] = {inner, rows, 0};
    const uint32_t box[3] = {box_inner, box_rows, 0};
    return make_tmap(map, type, elem_bytes, base, dim, box);
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                       uint32_t box_rows) {
    return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, rows, box_inner, box_rows);
}

bool make_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows) {
    return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, inner, rows, box_inner, box_rows);
}

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                       uint32_t box1, uint32_t box2) {
    if (d2 == 0) return false;
    const uint64_t dim[3] = {d0, d1, d2};
    const uint32_t box[3] = {box0, box1, box2};
    return make_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dim, box);
}

}  // namespace infllmv2
