// Cached TMA tensor maps (CUtensorMap) for the kernels' tiled bulk copies.
// The driver's encoder is reached through the runtime's entry-point query, so
// the library links only against the CUDA runtime.
#include <cuda.h>

#include <mutex>
#include <unordered_map>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(f);
    });
    return fn;
}

struct MapKey {
    const void* base;
    int dtype;
    int64_t dims[3], strides[2];
    int box[3];
    bool operator==(const MapKey& o) const {
        for (int i = 0; i < 3; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
        return base == o.base && dtype == o.dtype && strides[0] == o.strides[0] &&
               strides[1] == o.strides[1];
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        size_t h = std::hash<const void*>()(k.base) ^ (size_t)k.dtype * 0x9e3779b97f4a7c15ull;
        for (int i = 0; i < 3; ++i) h = h * 31 + std::hash<int64_t>()(k.dims[i]) + (size_t)k.box[i];
        return h * 31 + std::hash<int64_t>()(k.strides[0] ^ (k.strides[1] << 20));
    }
};

}  // namespace

int tiled_map_3d(const void* base, CUtensorMapDataType dtype, const int64_t dims[3],
                 const int64_t strides[2], const int box[3], CUtensorMap* out) {
    static std::mutex mu;
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    MapKey key{base, (int)dtype, {dims[0], dims[1], dims[2]}, {strides[0], strides[1]},
               {box[0], box[1], box[2]}};
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return PKV_OK;
    }
    EncodeFn enc = encode_fn();
    if (!enc) return PKV_ERR_CUDA;
    CUtensorMap m;
    const cuuint64_t d[3] = {(cuuint64_t)dims[0], (cuuint64_t)dims[1], (cuuint64_t)dims[2]};
    const cuuint64_t st[2] = {(cuuint64_t)strides[0], (cuuint64_t)strides[1]};
    const cuuint32_t bx[3] = {(cuuint32_t)box[0], (cuuint32_t)box[1], (cuuint32_t)box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&m, dtype, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    if (cache.size() > 4096) cache.clear();
    cache.emplace(key, m);
    *out = m;
    return PKV_OK;
}

}  // namespace pkv
