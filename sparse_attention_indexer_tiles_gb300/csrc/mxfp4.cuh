// Argument block and launcher of the MXFP4 -> e4m3 expansion.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace idx {

// One launch expands up to two arrays (an MXFP4 call's q and k): segment 1 is
// skipped when its n is 0.
struct Mxfp4Segment {
    const uint8_t* x;   // [n, D/2] packed e2m1 (element 2i in the low nibble)
    const uint8_t* sf;  // [n, D/32] e8m0 block scales
    long long n;
    uint8_t* out;       // [n, D] e4m3
};

struct Mxfp4Args {
    Mxfp4Segment seg[2];
    int D;
    int* d_status;
};

cudaError_t launch_mxfp4_to_e4m3(const Mxfp4Args& a, cudaStream_t s);

}  // namespace idx
