// tensor_map.h -- the driver's tensor-map encoder (cuTensorMapEncodeTiled),
// looked up once through the runtime so the library does not link libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace pgqa {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The encoder, or nullptr when the driver does not provide it.
EncodeTiledFn tensor_map_encoder();

} // namespace pgqa
