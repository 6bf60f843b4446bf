// tc_host.cu -- host helpers of the tcgen05 GEMMs: TMA tensor-map encoding
// through the CUDA runtime's driver entry point (no link against libcuda).
#include "qz_tc.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace qz {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void load_encode() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
} // namespace

// A 2-D byte tensor of `outer` rows x `inner` bytes (row pitch `row_bytes`),
// read in boxes of box_outer rows x box_inner bytes with the 128-byte swizzle.
bool encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    std::call_once(g_once, load_encode);
    if (!g_encode) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A 2-D tensor of `outer` rows x `inner` elements of `elem_bytes` (1, 2 or 4
// bytes; row pitch `row_bytes`), read in boxes of box_outer x box_inner
// elements, with the 128-byte swizzle or none. Out-of-range box elements read
// as zero.
bool encode_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
    std::call_once(g_once, load_encode);
    if (!g_encode) return false;
    const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT32;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// As encode_tmap_2d, with the 32-, 64- or 128-byte swizzle (swizzle_bytes):
// 16-byte chunk c of a row sits at chunk c ^ ((address >> 7) & (swizzle_bytes / 16 - 1))
// within its block, i.e. for 32-byte rows c ^ ((r >> 2) & 1), for 64-byte rows
// c ^ ((r >> 1) & 3), for 128-byte rows c ^ (r & 7).
bool encode_tmap_2d_swz(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle_bytes) {
    std::call_once(g_once, load_encode);
    if (!g_encode) return false;
    const CUtensorMapSwizzle sw = swizzle_bytes == 32    ? CU_TENSOR_MAP_SWIZZLE_32B
                                  : swizzle_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                         : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT32;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

} // namespace qz
