// Host side of the scoring kernel: TMA tensor maps and the launch of one
// (dtype, H, D) instantiation.  Included by the per-dtype translation units.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "score_impl.cuh"

namespace idx {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// 2D map over a row-major [outer, inner] array of `elem` bytes per element,
// box = [box_outer, box_inner], swizzled at box_inner * elem bytes (64 or 128).
inline CUresult make_map_2d(CUtensorMap* m, const void* base, int elem, uint64_t inner,
                            uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_SUPPORTED;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * (uint64_t)elem};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const uint32_t row_b = box_inner * (uint32_t)elem;
    return enc(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               row_b == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// 3D strided view of k [keys, D] as [nsamp, S, D]: coordinate (d, phase, i)
// addresses key phase + S * i, so one box of 128 i-rows is the stride-S
// sample of one phase (page 1, section 2: a strided tensor map loads the
// single-key sample in one TMA).
inline CUresult make_map_strided(CUtensorMap* m, const void* base, int elem, uint64_t D,
                                 uint64_t S, uint64_t nsamp, uint32_t box_inner) {
    auto enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_SUPPORTED;
    const cuuint64_t dims[3] = {D, S, nsamp > 0 ? nsamp : 1};
    const cuuint64_t strides[2] = {D * (uint64_t)elem, S * D * (uint64_t)elem};
    const cuuint32_t box[3] = {box_inner, 1, 128};
    const cuuint32_t estr[3] = {1, 1, 1};
    const uint32_t row_b = box_inner * (uint32_t)elem;
    return enc(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               row_b == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int DT, int H, int RB>
cudaError_t launch_score_t(const ScoreLaunch& L, cudaStream_t s) {
    using C = ScoreCfg<DT, H, RB>;
    const ScoreArgs& a = L.a;
    if (a.rows == 0) return cudaSuccess;
    CUtensorMap tq, tk, tks;
    const int elem = C::ELEM;
    if (make_map_2d(&tq, L.q, elem, (uint64_t)L.D, (uint64_t)a.rows * H, C::CHUNK_ELEMS, 256) !=
            CUDA_SUCCESS ||
        make_map_2d(&tk, L.k, elem, (uint64_t)L.D, (uint64_t)a.keys, C::CHUNK_ELEMS, 128) !=
            CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // the strided sample view for the launches that score the sample
    if (a.mode == SM_SAMPLE) {
        if (make_map_strided(&tks, L.k, elem, (uint64_t)L.D, (uint64_t)a.S, (uint64_t)a.nsamp,
                             C::CHUNK_ELEMS) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        tks = tk;
    }
    const bool split = a.ksplit > 1 || a.nruns != kRuns;
    auto kern = split ? score_kernel<DT, H, RB, true> : score_kernel<DT, H, RB, false>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(score_kernel<DT, H, RB, false>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(score_kernel<DT, H, RB, true>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            C::SMEM_ALLOC);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int nblk = (a.rows + C::R - 1) / C::R;
    long long gx;
    if (a.mode == SM_RESCAN) {
        gx = a.grid_x > 0 && a.grid_x < nblk ? a.grid_x : nblk;
    } else {
        if (a.ksplit < 1 || a.nwhole < 0 || a.nwhole > nblk || (a.ksplit == 1 && a.nwhole != nblk))
            return cudaErrorInvalidValue;
        // persistent: at most one CTA per SM, each taking units in turn
        const long long units = a.nwhole + (long long)(nblk - a.nwhole) * a.ksplit;
        if (units > 0x7fffffffll) return cudaErrorInvalidValue;
        gx = a.grid_x > 0 && a.grid_x < units ? a.grid_x : units;
    }
    if (gx > 0x7fffffffll) return cudaErrorInvalidValue;
    return launch_k(kern, dim3((unsigned)gx), dim3(C::THREADS), C::SMEM_ALLOC, s, L.pdl != 0, tq,
                    tk, tks, a);
}

}  // namespace idx
