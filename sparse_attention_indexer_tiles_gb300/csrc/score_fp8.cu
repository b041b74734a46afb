// e4m3 instantiations of the scoring kernel (kind::f8f6f4 MMA).
#include "score_launch.cuh"

namespace idx {

cudaError_t launch_score_fp8(const ScoreLaunch& L, cudaStream_t s) {
    const int RB = L.D;
    switch (L.H * 1000 + RB) {
        case 8064: return launch_score_t<IDX_FP8_E4M3, 8, 64>(L, s);
        case 16064: return launch_score_t<IDX_FP8_E4M3, 16, 64>(L, s);
        case 32064: return launch_score_t<IDX_FP8_E4M3, 32, 64>(L, s);
        case 64064: return launch_score_t<IDX_FP8_E4M3, 64, 64>(L, s);
        case 8128: return launch_score_t<IDX_FP8_E4M3, 8, 128>(L, s);
        case 16128: return launch_score_t<IDX_FP8_E4M3, 16, 128>(L, s);
        case 32128: return launch_score_t<IDX_FP8_E4M3, 32, 128>(L, s);
        case 64128: return launch_score_t<IDX_FP8_E4M3, 64, 128>(L, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace idx
