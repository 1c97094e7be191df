// Weighted combine with residual for the prefill layer (the decode layer
// combines inside its down-projection kernel):
//   out[t] = x[t] + sum_j w[t, j] * y(t, j), j = 0..k-1 in order.
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

// Eight consecutive y values as floats: fp16 (prefill) or fp32 (decode).
__device__ __forceinline__ void load8(const uint16_t* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// out[t, :] = x[t, :] + sum_{j=0..k-1} y[slot_pos[t, j], :], accumulated in
// fp32 in j order.  y rows already carry the routing weight.  One thread per
// 8 columns.
template <bool OUT_FP32, typename Y>
__global__ void combine_kernel(const uint16_t* __restrict__ x, const Y* __restrict__ y,
                               const int32_t* __restrict__ slot_pos, int T, int H, int k,
                               void* __restrict__ out) {
    pdl_wait();  // the down GEMM's rows
    pdl_trigger();
    const int cols8 = H / 8;
    const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (i >= (size_t)T * cols8) return;
    const int t = (int)(i / cols8), c = (int)(i % cols8) * 8;
    float acc[8];
    {
        const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)t * H + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            acc[2 * p] = __uint_as_float(w[p] << 16);
            acc[2 * p + 1] = __uint_as_float(w[p] & 0xffff0000u);
        }
    }
    for (int j = 0; j < k; ++j) {
        const int pos = slot_pos[(size_t)t * k + j];
        float v[8];
        load8(y + (size_t)pos * H + c, v);
#pragma unroll
        for (int p = 0; p < 8; ++p) acc[p] += v[p];
    }
    if (OUT_FP32) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + (size_t)t * H + c);
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            w[p] = (uint32_t)float_to_bf16_bits(acc[2 * p]) |
                   ((uint32_t)float_to_bf16_bits(acc[2 * p + 1]) << 16);
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + (size_t)t * H + c) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One warp per token: the sum of squares in fp32 (each lane over its columns
// in order, then a butterfly), r = 1 / sqrt(mean + eps) (correctly rounded
// divide and square root), xn = bf16_rn(x * r).
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* __restrict__ x, int T, int H,
                                                      float eps, uint16_t* __restrict__ xn) {
    pdl_wait();  // x (the preceding work on the stream)
    pdl_trigger();
    const int t = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x % 32;
    if (t >= T) return;  // whole warp
    const uint16_t* row = x + (size_t)t * H;
    float ss = 0.f;
    for (int c = lane * 8; c < H; c += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float a = __uint_as_float(w[p] << 16), b = __uint_as_float(w[p] & 0xffff0000u);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
        }
    }
    ss = warp_sum(ss);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, (float)H) + eps));
    uint16_t* orow = xn + (size_t)t * H;
    for (int c = lane * 8; c < H; c += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float a = __uint_as_float(w[p] << 16) * r, b = __uint_as_float(w[p] & 0xffff0000u) * r;
            o[p] = (uint32_t)float_to_bf16_bits(a) | ((uint32_t)float_to_bf16_bits(b) << 16);
        }
        *reinterpret_cast<uint4*>(orow + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps, uint16_t* xn,
                           cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(rmsnorm_kernel, dim3((T + 7) / 8), dim3(256), 0, s, x, T, H, eps, xn);
}

cudaError_t launch_combine(const uint16_t* x, const void* y, bool y_fp32, const int32_t* slot_pos,
                           int T, int H, int k, bool out_fp32, void* out, cudaStream_t s) {
    const size_t n = (size_t)T * (H / 8);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    const float* yf = static_cast<const float*>(y);
    const uint16_t* yh = static_cast<const uint16_t*>(y);
    const dim3 g(blocks), b(threads);
    if (out_fp32 && y_fp32)
        return launch_pdl(combine_kernel<true, float>, g, b, 0, s, x, yf, slot_pos, T, H, k, out);
    if (out_fp32)
        return launch_pdl(combine_kernel<true, uint16_t>, g, b, 0, s, x, yh, slot_pos, T, H, k, out);
    if (y_fp32)
        return launch_pdl(combine_kernel<false, float>, g, b, 0, s, x, yf, slot_pos, T, H, k, out);
    return launch_pdl(combine_kernel<false, uint16_t>, g, b, 0, s, x, yh, slot_pos, T, H, k, out);
}

}  // namespace moeq4
