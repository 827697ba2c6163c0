#include "tensor_map.h"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace tp {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_tiled = nullptr;
PFN_cuTensorMapEncodeIm2col_v12000 g_im2col = nullptr;
std::once_flag g_once;
bool g_found = false;

void resolve()
{
    std::call_once(g_once, [] {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound;
        cudaDriverEntryPointQueryResult q2 = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000, cudaEnableDefault, &q1) ==
                cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f2, 12000, cudaEnableDefault, &q2) ==
                cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess) {
            g_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f1);
            g_im2col = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(f2);
            g_found = true;
        }
    });
}

// The encode functions are driver calls and need a current context. A host
// thread that has not touched the CUDA runtime yet has none (reading the
// current device does not create it), so make the device's primary context
// current first, as every runtime call does implicitly.
void bind_primary_context()
{
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaSetDevice(dev);
}

uint32_t elem_bytes(CUtensorMapDataType t)
{
    switch (t) {
    case CU_TENSOR_MAP_DATA_TYPE_UINT8: return 1;
    case CU_TENSOR_MAP_DATA_TYPE_UINT16:
    case CU_TENSOR_MAP_DATA_TYPE_FLOAT16:
    case CU_TENSOR_MAP_DATA_TYPE_BFLOAT16: return 2;
    case CU_TENSOR_MAP_DATA_TYPE_FLOAT64:
    case CU_TENSOR_MAP_DATA_TYPE_UINT64:
    case CU_TENSOR_MAP_DATA_TYPE_INT64: return 8;
    default: return 4;
    }
}

// A small cache of encoded maps (host memory only): a map depends only on its
// descriptor fields, so repeated calls on the same buffers and shapes reuse it
// instead of asking the driver again. Round-robin replacement.
constexpr int kCacheSize = 64;

bool same(const TiledDesc& a, const TiledDesc& b)
{
    if (a.dtype != b.dtype || a.rank != b.rank || a.base != b.base || a.swizzle != b.swizzle) return false;
    for (uint32_t i = 0; i < a.rank; ++i)
        if (a.dims[i] != b.dims[i] || a.box[i] != b.box[i]) return false;
    for (uint32_t i = 0; i + 1 < a.rank; ++i)
        if (a.strides_bytes[i] != b.strides_bytes[i]) return false;
    return true;
}

bool same(const Im2colDesc& a, const Im2colDesc& b)
{
    if (a.dtype != b.dtype || a.base != b.base || a.swizzle != b.swizzle || a.channels != b.channels ||
        a.pixels != b.pixels)
        return false;
    for (int i = 0; i < 4; ++i)
        if (a.dims[i] != b.dims[i] || a.elem_strides[i] != b.elem_strides[i]) return false;
    for (int i = 0; i < 3; ++i)
        if (a.strides_bytes[i] != b.strides_bytes[i]) return false;
    for (int i = 0; i < 2; ++i)
        if (a.lower[i] != b.lower[i] || a.upper[i] != b.upper[i]) return false;
    return true;
}

template <typename Desc>
struct MapCache {
    struct Entry {
        Desc key;
        CUtensorMap map;
        bool valid;
    };
    Entry e[kCacheSize] = {};
    int next = 0;
    std::mutex mu;

    bool find(const Desc& d, CUtensorMap* out)
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < kCacheSize; ++i)
            if (e[i].valid && same(e[i].key, d)) {
                *out = e[i].map;
                return true;
            }
        return false;
    }

    void put(const Desc& d, const CUtensorMap& m)
    {
        std::lock_guard<std::mutex> lock(mu);
        e[next].key = d;
        e[next].map = m;
        e[next].valid = true;
        next = (next + 1) % kCacheSize;
    }
};

MapCache<TiledDesc> g_tiled_cache;
MapCache<Im2colDesc> g_im2col_cache;

}  // namespace

bool tiled_ok(const TiledDesc& d)
{
    if (d.rank < 1 || d.rank > 5) return false;
    if ((reinterpret_cast<uintptr_t>(d.base) & 15u) != 0) return false;
    const uint32_t eb = elem_bytes(d.dtype);
    for (uint32_t i = 0; i < d.rank; ++i) {
        if (d.dims[i] == 0 || d.dims[i] > (1ull << 32)) return false;
        if (d.box[i] == 0 || d.box[i] > 256) return false;
    }
    for (uint32_t i = 0; i + 1 < d.rank; ++i) {
        if (d.strides_bytes[i] % 16 != 0 || d.strides_bytes[i] >= (1ull << 40)) return false;
    }
    if ((d.box[0] * eb) % 16 != 0) return false;
    if (d.swizzle == CU_TENSOR_MAP_SWIZZLE_128B && d.box[0] * eb > 128) return false;
    return true;
}

int encode_tiled(CUtensorMap* out, const TiledDesc& d)
{
    if (g_tiled_cache.find(d, out)) return ST_OK;
    resolve();
    if (!g_found) return ST_CUDA;
    if (!tiled_ok(d)) return ST_INVALID_ARG;
    bind_primary_context();
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_tiled(out, d.dtype, d.rank, d.base, reinterpret_cast<const cuuint64_t*>(d.dims),
                         reinterpret_cast<const cuuint64_t*>(d.strides_bytes),
                         reinterpret_cast<const cuuint32_t*>(d.box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         d.swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return ST_DRIVER_ENCODE;
    g_tiled_cache.put(d, *out);
    return ST_OK;
}

int encode_im2col(CUtensorMap* out, const Im2colDesc& d)
{
    if (g_im2col_cache.find(d, out)) return ST_OK;
    resolve();
    if (!g_found) return ST_CUDA;
    if ((reinterpret_cast<uintptr_t>(d.base) & 15u) != 0) return ST_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
        if (d.strides_bytes[i] % 16 != 0) return ST_INVALID_ARG;
    bind_primary_context();
    CUresult r = g_im2col(out, d.dtype, 4, d.base, reinterpret_cast<const cuuint64_t*>(d.dims),
                          reinterpret_cast<const cuuint64_t*>(d.strides_bytes), d.lower, d.upper, d.channels,
                          d.pixels, reinterpret_cast<const cuuint32_t*>(d.elem_strides),
                          CU_TENSOR_MAP_INTERLEAVE_NONE, d.swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return ST_DRIVER_ENCODE;
    g_im2col_cache.put(d, *out);
    return ST_OK;
}

}  // namespace tp
