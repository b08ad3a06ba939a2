// tmap.h -- host-side TMA tensor-map encoding shared by the launchers.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "plan.h"

namespace attn {

// The driver's cuTensorMapEncodeTiled, looked up once (a function-local
// static: initialised once even when host threads race for it).
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// A 16-bit [B][H][S][D] view (element strides) as a 4-D map (d, s, h, b) with
// boxes of 64 elements x `rows` rows and the 128-byte swizzle.
inline bool tmap_view16(CUtensorMap *m, const View &v, int dtype, int64_t d, int64_t s, int64_t h, int64_t b,
                        uint32_t rows)
{
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(s), cuuint64_t(h), cuuint64_t(b)};
    const int64_t sb = b > 1 ? v.sb : s * v.ss;  // unused extent-1 dim: any legal stride
    cuuint64_t strides[3] = {cuuint64_t(v.ss * 2), cuuint64_t(v.sh * 2), cuuint64_t((sb > 0 ? sb : 8) * 2)};
    cuuint32_t box[4] = {64, rows, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, dtype == ATTN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     v.ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace attn
