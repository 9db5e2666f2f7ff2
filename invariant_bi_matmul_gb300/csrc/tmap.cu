// tmap.cu -- host-side TMA tensor-map encoding (cuTensorMapEncodeTiled, reached through
// the runtime's driver entry-point query so no -lcuda is needed) with a small cache keyed
// by pointer, shape, stride, box and swizzle.
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "tmap.h"

namespace bi {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

struct MapKey {
    uintptr_t ptr;
    uint64_t inner, outer, stride;
    uint32_t box_inner, box_outer, swizzle;
    uint32_t box_blocks;  // 0: rank-2 map; >0: rank-3 K-blocked map with this many blocks
    bool f16;             // element type: IEEE binary16 instead of bf16
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && inner == o.inner && outer == o.outer && stride == o.stride &&
               box_inner == o.box_inner && box_outer == o.box_outer && swizzle == o.swizzle &&
               box_blocks == o.box_blocks && f16 == o.f16;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
        h ^= k.inner + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= k.outer + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= k.stride + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= (uint64_t(k.box_inner) << 32 | k.box_outer) + (h << 6) + (h >> 2);
        return size_t(h ^ k.swizzle ^ (uint64_t(k.box_blocks) << 40) ^ (uint64_t(k.f16) << 63));
    }
};

std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

bool tmap_bf16_impl(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer, uint64_t stride,
                uint32_t box_inner, uint32_t box_outer, int swizzle_bytes, uint32_t box_blocks,
                bool f16) {
    const MapKey key{reinterpret_cast<uintptr_t>(ptr), inner, outer, stride, box_inner, box_outer,
                     uint32_t(swizzle_bytes), box_blocks, f16};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return true;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    CUtensorMap m;
    const CUtensorMapDataType dt =
        f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult r;
    if (box_blocks == 0) {
        const cuuint64_t dims[2] = {inner, outer};
        const cuuint64_t strides[1] = {stride * 2};
        const cuuint32_t box[2] = {box_inner, box_outer};
        const cuuint32_t estr[2] = {1, 1};
        r = fn(&m, dt, 2, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // [outer][inner] viewed as (box_inner-wide column, row, column block): element
        // (c, r, b) = base[r*stride + b*box_inner + c]; inner must be a multiple of box_inner
        const cuuint64_t dims[3] = {box_inner, outer, inner / box_inner};
        const cuuint64_t strides[2] = {stride * 2, uint64_t(box_inner) * 2};
        const cuuint32_t box[3] = {box_inner, box_outer, box_blocks};
        const cuuint32_t estr[3] = {1, 1, 1};
        r = fn(&m, dt, 3, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() > 4096) g_maps.clear();
    g_maps.emplace(key, m);
    *out = m;
    return true;
}

}  // namespace

namespace {

// (encoded on every call: one driver call, no cache)
bool tmap_2d_plain(CUtensorMap* out, CUtensorMapDataType type, const void* ptr, uint64_t inner,
                   uint64_t outer, uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(out, type, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

bool tmap_2d_u8(CUtensorMap* out, const void* ptr, uint64_t inner_bytes, uint64_t outer,
                uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    return tmap_2d_plain(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, inner_bytes, outer,
                         stride_bytes, box_inner, box_outer);
}

bool tmap_3d_bf16(CUtensorMap* out, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1,
                  uint32_t box2) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1 * 2, stride2 * 2};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool tmap_2d_u16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                 uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    return tmap_2d_plain(out, CU_TENSOR_MAP_DATA_TYPE_UINT16, ptr, inner, outer, stride_bytes,
                         box_inner, box_outer);
}

bool tmap_2d_bf16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                  uint64_t stride, uint32_t box_inner, uint32_t box_outer, int swizzle_bytes,
                  bool f16) {
    return tmap_bf16_impl(out, ptr, inner, outer, stride, box_inner, box_outer, swizzle_bytes, 0,
                          f16);
}

bool tmap_kblocked_bf16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                        uint64_t stride, uint32_t box_inner, uint32_t box_outer,
                        uint32_t box_blocks, int swizzle_bytes, bool f16) {
    if (box_blocks == 0 || inner % box_inner != 0) return false;
    return tmap_bf16_impl(out, ptr, inner, outer, stride, box_inner, box_outer, swizzle_bytes,
                          box_blocks, f16);
}

}  // namespace bi
