// tmap.cuh -- host helpers for tensor-map (TMA) copies, shared by the kernels that use them.
#pragma once

#include <cuda.h>  // CUtensorMap and its encoding enums (the encoder itself is fetched at run time)
#include <cuda_runtime.h>

#include <mutex>

namespace kvq8 {

// cuTensorMapEncodeTiled from the driver, looked up once per process.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Device address of the library's timeout flag (the one kvq8_device_error reads) on the
// current device.
unsigned int* device_error_flag();

}  // namespace kvq8
