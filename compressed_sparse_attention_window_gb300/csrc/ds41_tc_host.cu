// ds41_tc_host.cu - host side of the tensor-core building blocks: the
// driver's tensor-map encoder, looked up once per process, and the 2-D bf16
// tensor maps the TMA copies use.
#include <mutex>

#include "ds41_tc.cuh"

namespace ds41 {
namespace tc {

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::mutex g_encode_mu;

int get_encode(PFN_cuTensorMapEncodeTiled_v12000* out) {
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult qr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &qr);
        if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn)
            return fail(DS41_E_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return DS41_OK;
}

int make_map_bf16(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* ptr,
                  int64_t rows, int64_t cols, int box_cols, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DS41_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DS41_OK;
}

int make_map_u8_sw64(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* ptr,
                     int64_t rows, int64_t cols, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DS41_E_CUDA, "cuTensorMapEncodeTiled (u8) failed (%d)", (int)r);
    return DS41_OK;
}

}  // namespace tc
}  // namespace ds41
