// tmap.cu -- TMA tensor maps for the tcgen05 kernels (host side).
//
// cuTensorMapEncodeTiled is a driver entry point; it is looked up through the runtime so the
// library does not link libcuda directly.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc_attn.cuh"

namespace acache {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
        else
            (void)cudaGetLastError();
    }
    return fn;
}
}  // namespace

bool make_map_box(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint32_t* box) {
    auto enc = encode_fn();
    if (!enc || rank < 1 || rank > 5) return false;
    cuuint64_t gdim[5], gstride[4];
    cuuint32_t bx[5], estr[5];
    uint64_t stride = 2;
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i] ? dims[i] : 1;
        if (i > 0) gstride[i - 1] = stride;
        stride *= gdim[i];
        bx[i] = box[i];
        estr[i] = 1;
    }
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), gdim, gstride, bx,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, int row_dim,
              uint32_t box_rows) {
    uint32_t box[5] = {64, 1, 1, 1, 1};
    box[row_dim] = box_rows;
    return make_map_box(m, ptr, rank, dims, box);
}

}  // namespace acache
