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
// raises IDX_DEV_RANGE.
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

// Over block scales 2^-8 .. 2^6 every e2m1 element is exact in e4m3 (the
// tightest ends: 0.5 and 1.5 at 2^-8 are 2^-9 and 3·2^-9; 6 at 2^6 is 384), so
// there a block is a byte lookup: the e4m3 codes of the 8 magnitudes at that
// scale sit in one 8-byte word, a byte permute picks four of them by the
// nibbles' low 3 bits, and the nibbles' sign bits are spread to bit 7 of each
// byte.  Any other scale takes the element-by-element path above.
constexpr uint32_t kFastLo = 127u - 8u, kFastN = 15u;

// One 32-element block: 16 bytes of codes and its scale code in, 32 e4m3 bytes out.
IDX_DEVI void convert_block(const uint2 (&mag)[16], uint4 in, uint32_t code, uint4* dst,
                            bool& bad) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[8];
    if (code - kFastLo < kFastN) {
        const uint2 t = mag[code - kFastLo];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // input word i holds elements 8i .. 8i + 7, element 8i + j in nibble j;
            // output words 2i, 2i + 1 hold them one per byte
            const uint32_t m = w[i] & 0x77777777u, sg = w[i] & 0x88888888u;
            const uint32_t q0 = __byte_perm(sg, 0u, 0x1100), q1 = __byte_perm(sg, 0u, 0x3322);
            // even bytes want bit 3 of the duplicated source byte, odd ones bit 7
            const uint32_t s0 = (((q0 << 4) & 0x00ff00ffu) | (q0 & 0xff00ff00u)) & 0x80808080u;
            const uint32_t s1 = (((q1 << 4) & 0x00ff00ffu) | (q1 & 0xff00ff00u)) & 0x80808080u;
            o[2 * i] = __byte_perm(t.x, t.y, m & 0xffffu) | s0;
            o[2 * i + 1] = __byte_perm(t.x, t.y, m >> 16) | s1;
        }
    } else {
        if (code == 255u) bad = true;                     // the e8m0 NaN
        const int e = (int)code - 127;
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
    }
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Blocks of both segments form one index range, one block per thread; the
// grid covers the range (the loop only matters past the grid-size limit).
__global__ void __launch_bounds__(256) mxfp4_to_e4m3_kernel(Mxfp4Args a) {
    __shared__ uint2 mag[16];  // row s: byte k = magnitude code k at scale 2^(s - 8)
    if (threadIdx.x < 16 * 8) {
        const uint32_t s = threadIdx.x >> 3, k = threadIdx.x & 7u;
        bool unused = false;
        reinterpret_cast<uint8_t*>(mag)[threadIdx.x] =
            (uint8_t)(s < kFastN ? e2m1_scaled_to_e4m3(k, (int)s - 8, unused) : 0u);
    }
    __syncthreads();
    const long long per = a.D / 32;
    const long long b0 = a.seg[0].n * per, blocks = b0 + a.seg[1].n * per;
    const long long stride = (long long)gridDim.x * blockDim.x;
    bool bad = false;
    for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < blocks;
         b += stride) {
        const bool first = b < b0;  // field by field: no indexed copy of the parameters
        const long long j = first ? b : b - b0;
        const uint4 in = __ldg(reinterpret_cast<const uint4*>(first ? a.seg[0].x : a.seg[1].x) + j);
        const uint32_t code = __ldg((first ? a.seg[0].sf : a.seg[1].sf) + j);
        convert_block(mag, in, code,
                      reinterpret_cast<uint4*>(first ? a.seg[0].out : a.seg[1].out) + 2 * j, bad);
    }
    if (bad) raise_status(a.d_status, IDX_DEV_RANGE);
}

}  // namespace

cudaError_t launch_mxfp4_to_e4m3(const Mxfp4Args& a, cudaStream_t s) {
    const long long blocks = (a.seg[0].n + a.seg[1].n) * (long long)(a.D / 32);
    if (blocks == 0) return cudaSuccess;
    const long long want = (blocks + 255) / 256;
    const int grid = (int)(want < 0x7fffffffll ? want : 0x7fffffffll);
    mxfp4_to_e4m3_kernel<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace idx
