// Argument block and launcher of the MXFP4 -> e4m3 expansion.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace idx {

struct Mxfp4Args {
    const uint8_t* x;   // [n, D/2] packed e2m1 (element 2i in the low nibble)
    const uint8_t* sf;  // [n, D/32] e8m0 block scales
    long long n;
    int D;
    uint8_t* out;       // [n, D] e4m3
    int* d_status;
};

cudaError_t launch_mxfp4_to_e4m3(const Mxfp4Args& a, int sm_count, cudaStream_t s);

}  // namespace idx
