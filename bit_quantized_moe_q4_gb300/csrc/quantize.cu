// moe_q4_quantize: float weights -> Q4_0-family blocks on the GPU.
//
// Page "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU",
// Methodology 2 "Quantization": group-wise symmetric 4-bit weights of the
// Q4_0 family.  The page names the family but prints no encoder; the rule
// here is that family's usual one (the reading the CPU oracle follows): per
// block of 32 consecutive weights of a row,
//   m = the element of largest magnitude (the first one on a tie), sign kept
//   d = fp16(m / -8)                       (round to nearest even)
//   q = min(15, max(0, floor(x / d + 8.5)))  against the stored d;  d = 0 -> q = 8
// so that w = d (q - 8) decodes it.  d may be negative.
//
// Exactness: m / -8 is exact in fp32, so the fp16 rounding of d is that of
// the real quotient.  The code decision is taken exactly: an fp32 estimate
// of x / d + 8.5 (off by less than 2^-19, so its floor by at most one) is
// corrected with exact comparisons x >= (n - 8.5) d (d > 0; <= for d < 0),
// whose right-hand side has at most 5 + 11 significant bits and is therefore
// an exact fp32 product.  The result equals the rounding of the exact
// rational, bit for bit, for every finite input with |m / 8| <= 65504.
//
// One warp per block: lane i holds element i; the block maximum and its
// first position come from a warp reduction on the magnitudes' bit
// patterns (non-negative floats order like their bits).
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int kQuantWarps = 8;

// Exact test of floor(x / d + 8.5) >= n for d != 0.
__device__ __forceinline__ bool code_at_least(float x, float d, int n) {
    const float t = ((float)n - 8.5f) * d;  // exact: <= 16 significant bits
    return d > 0.0f ? x >= t : x <= t;
}

template <bool BF16, bool BLOCK18>
__global__ void __launch_bounds__(kQuantWarps * 32) q4_quantize_kernel(
    const void* __restrict__ src, long long nblocks, uint8_t* __restrict__ dst,
    uint16_t* __restrict__ dst_scales) {
    const int lane = threadIdx.x % 32;
    const long long blk = (long long)blockIdx.x * kQuantWarps + threadIdx.x / 32;
    if (blk >= nblocks) return;  // whole warp
    const size_t i = (size_t)blk * kGroup + lane;
    const float x = BF16 ? bf16_bits_to_float(static_cast<const uint16_t*>(src)[i])
                         : static_cast<const float*>(src)[i];
    // largest magnitude, first position on a tie
    const uint32_t mag = __float_as_uint(x) & 0x7fffffffu;
    const uint32_t top = __reduce_max_sync(0xffffffffu, mag);
    const int first = __ffs(__ballot_sync(0xffffffffu, mag == top)) - 1;
    const float m = __shfl_sync(0xffffffffu, x, first);
    const uint16_t db = __half_as_ushort(__float2half_rn(m * -0.125f));
    const float d = half_bits_to_float(db);
    int q = 8;
    if (d != 0.0f) {
        const float est = floorf(__fdiv_rn(x, d) + 8.5f);
        q = (int)fminf(fmaxf(est, 0.0f), 15.0f);
        if (q < 15 && code_at_least(x, d, q + 1)) ++q;
        if (q > 0 && !code_at_least(x, d, q)) --q;
    }
    if (BLOCK18) {
        // fp16 scale little-endian, then byte j = element j | element j+16 << 4
        const int hi = __shfl_down_sync(0xffffffffu, q, 16);
        uint8_t* b = dst + (size_t)blk * 18;
        if (lane < 16) b[2 + lane] = (uint8_t)(q | (hi << 4));
        if (lane == 0) {
            b[0] = (uint8_t)(db & 0xffu);
            b[1] = (uint8_t)(db >> 8);
        }
    } else {
        dst[i] = (uint8_t)q;
        if (lane == 0) dst_scales[blk] = db;
    }
}

}  // namespace

cudaError_t launch_quantize(int src_type, const void* src, long long rows, int K, int fmt,
                            void* dst, void* dst_scales, cudaStream_t s) {
    const long long nblocks = rows * (K / kGroup);
    if (nblocks == 0) return cudaSuccess;
    const long long grid = (nblocks + kQuantWarps - 1) / kQuantWarps;
    if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
    const dim3 g((unsigned)grid), b(kQuantWarps * 32);
    uint8_t* d8 = static_cast<uint8_t*>(dst);
    uint16_t* ds = static_cast<uint16_t*>(dst_scales);
    const bool bf = src_type == MOE_SRC_BF16, b18 = fmt == MOE_Q4_BLOCK18;
    if (bf && b18) q4_quantize_kernel<true, true><<<g, b, 0, s>>>(src, nblocks, d8, ds);
    else if (bf) q4_quantize_kernel<true, false><<<g, b, 0, s>>>(src, nblocks, d8, ds);
    else if (b18) q4_quantize_kernel<false, true><<<g, b, 0, s>>>(src, nblocks, d8, ds);
    else q4_quantize_kernel<false, false><<<g, b, 0, s>>>(src, nblocks, d8, ds);
    return cudaGetLastError();
}

}  // namespace moeq4
