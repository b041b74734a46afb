// bf16 instantiations of the scoring kernel (kind::f16 MMA).
#include "score_launch.cuh"

namespace idx {

cudaError_t launch_score_bf16(const ScoreLaunch& L, cudaStream_t s) {
    const int RB = L.D * 2;
    switch (L.H * 1000 + RB) {
        case 8128: return launch_score_t<IDX_BF16, 8, 128>(L, s);
        case 16128: return launch_score_t<IDX_BF16, 16, 128>(L, s);
        case 32128: return launch_score_t<IDX_BF16, 32, 128>(L, s);
        case 64128: return launch_score_t<IDX_BF16, 64, 128>(L, s);
        case 8256: return launch_score_t<IDX_BF16, 8, 256>(L, s);
        case 16256: return launch_score_t<IDX_BF16, 16, 256>(L, s);
        case 32256: return launch_score_t<IDX_BF16, 32, 256>(L, s);
        case 64256: return launch_score_t<IDX_BF16, 64, 256>(L, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace idx
