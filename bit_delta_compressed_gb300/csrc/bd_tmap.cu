// bd_tmap.cu -- host helpers of the tensor-core kernels: TMA descriptors
// (cuTensorMapEncodeTiled, fetched once from the driver) and the dynamic
// shared-memory attribute, set once per device and kernel slot.
#include <mutex>

#include "bd_tc_common.cuh"

namespace bd {
namespace {
std::mutex g_tc_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_smem_set[64][4] = {};

bool encoder() {
    std::lock_guard<std::mutex> lock(g_tc_mutex);
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return true;
}
}  // namespace

bool make_tmap_bf16_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows) {
    if (!encoder()) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_u8_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols_bytes,
                        uint32_t box_rows) {
    if (!encoder()) return false;
    cuuint64_t dims[2] = {cols_bytes, rows};
    cuuint64_t strides[1] = {cols_bytes};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bits(CUtensorMap* map, const void* base, uint64_t rows, uint64_t words, uint32_t box_rows) {
    if (!encoder()) return false;
    cuuint64_t dims[2] = {words, rows};
    cuuint64_t strides[1] = {words * 4};
    cuuint32_t box[2] = {4, box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool set_smem_attr(const void* kernel, int bytes, int slot) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(g_tc_mutex);
    if (g_smem_set[dev][slot] >= bytes) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    g_smem_set[dev][slot] = bytes;
    return true;
}

}  // namespace bd
