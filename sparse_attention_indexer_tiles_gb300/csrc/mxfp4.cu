// MXFP4 -> e4m3, exactly (page "[sglang] logits를 쓰지 않는 top-k", section 1
// names an fp4 indexer over 64-byte keys; the element format is OCP MX:
// e2m1 elements, one e8m0 scale per block of 32 along D).
//
// An e2m1 element is ±(1 + f/2)·2^E0 with one fraction bit f (E0 in 0..2) or
// ±0.5 (the subnormal) or ±0; times the block scale 2^e it is ±(1 + f/2)·2^E,
// E = E0 + e.  e4m3 holds that exactly as a normal number for -6 <= E <= 8
// (exponent field E + 7, fraction bits f00) and as a subnormal m·2^-9 with
// m = (2 + f)·2^(E+8) an integer in 1..7 for E >= -8, or E = -9 with f = 0.
// Outside that the element is saturated (±448) or flushed (±0) and the launch
// raises IDX_DEV_RANGE.  One thread converts one block: 16 bytes in, 32 out.
#include "common.cuh"
#include "mxfp4.cuh"

namespace idx {

namespace {

// e4m3 code of e2m1 code c (4 bits) times 2^e; `bad` when not exact
IDX_DEVI uint32_t e2m1_scaled_to_e4m3(uint32_t c, int e, bool& bad) {
    const uint32_t sign = (c & 8u) << 4;
    const uint32_t ex = (c >> 1) & 3u, m = c & 1u;
    if (ex == 0u && m == 0u) return sign;                  // ±0
    const int E = (ex == 0u ? -1 : (int)ex - 1) + e;      // 0.5 = 1.0·2^-1
    const uint32_t f = ex == 0u ? 0u : m;                 // the fraction bit
    if (E >= -6) {
        if (E > 8) {
            bad = true;
            return sign | 0x7Eu;                          // 448
        }
        return sign | ((uint32_t)(E + 7) << 3) | (f << 2);
    }
    if (E >= -8) return sign | ((2u + f) << (E + 8));    // m·2^-9, m = (2 + f)·2^(E+8)
    if (E == -9 && f == 0u) return sign | 1u;             // 2^-9
    bad = true;
    return sign;
}

__global__ void __launch_bounds__(256) mxfp4_to_e4m3_kernel(Mxfp4Args a) {
    const long long blocks = a.n * (long long)(a.D / 32);
    const long long stride = (long long)gridDim.x * blockDim.x;
    bool bad = false;
    for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < blocks;
         b += stride) {
        const uint4 in = __ldg(reinterpret_cast<const uint4*>(a.x) + b);
        const uint32_t code = __ldg(a.sf + b);
        if (code == 255u) bad = true;                     // the e8m0 NaN
        const int e = (int)code - 127;
        const uint32_t w[4] = {in.x, in.y, in.z, in.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // output word i = elements 4i .. 4i + 3 = the nibbles of input bytes 2i, 2i + 1
            const uint32_t two = (w[i >> 1] >> (16 * (i & 1))) & 0xffffu;
            uint32_t v = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v |= e2m1_scaled_to_e4m3((two >> (4 * j)) & 15u, e, bad) << (8 * j);
            o[i] = v;
        }
        uint4* dst = reinterpret_cast<uint4*>(a.out) + 2 * b;
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    if (bad) raise_status(a.d_status, IDX_DEV_RANGE);
}

}  // namespace

cudaError_t launch_mxfp4_to_e4m3(const Mxfp4Args& a, int sm_count, cudaStream_t s) {
    const long long blocks = a.n * (long long)(a.D / 32);
    if (blocks == 0) return cudaSuccess;
    const long long want = (blocks + 255) / 256;
    const long long cap = 8ll * sm_count;
    const int grid = (int)(want < cap ? want : cap);
    mxfp4_to_e4m3_kernel<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace idx
