// Host builder for TMA tensor maps over cuTensorMapEncodeTiled /
// cuTensorMapEncodeIm2col, resolved through the runtime's driver entry point.
//
// Descriptor rules ("CUDA 13 TMA Descriptor Notes", breaking changes 1-3, and
// the cuda.h documentation of the two encoders): global strides are given in
// BYTES for every dimension above the first (tensorRank - 1 entries), each a
// multiple of 16; the base address is 16-byte aligned; bf16 tensors use
// CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; out-of-bounds elements of a load are
// zero-filled, out-of-bounds elements of a store are dropped.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace tp {

// Everything a tiled encode needs, kept as plain data so the host logic can be
// checked without a GPU (see tp_gemm_plan).
struct TiledDesc {
    CUtensorMapDataType dtype;
    uint32_t rank;
    void* base;
    uint64_t dims[5];
    uint64_t strides_bytes[4];  // rank - 1 entries
    uint32_t box[5];
    CUtensorMapSwizzle swizzle;
};

struct Im2colDesc {
    CUtensorMapDataType dtype;
    void* base;
    uint64_t dims[4];           // {C, W, H, N}
    uint64_t strides_bytes[3];  // {W, H, N} strides in bytes
    int lower[2];               // pixel box lower corner {W, H}
    int upper[2];               // pixel box upper corner {W, H}
    uint32_t channels;          // channels per pixel (one 128-byte row)
    uint32_t pixels;            // pixels per column (rows of the A tile)
    uint32_t elem_strides[4];   // traversal strides {1, stride, stride, 1}
    CUtensorMapSwizzle swizzle;
};

// Returns 0 on success, else a tp status code (ST_DRIVER_ENCODE when the
// driver rejects the descriptor, ST_CUDA when the encoder cannot be found).
int encode_tiled(CUtensorMap* out, const TiledDesc& d);
int encode_im2col(CUtensorMap* out, const Im2colDesc& d);

// Static checks the encoders would also make: alignment of the base, byte
// strides multiple of 16, box limits. True when TMA can describe the tensor.
bool tiled_ok(const TiledDesc& d);

}  // namespace tp
