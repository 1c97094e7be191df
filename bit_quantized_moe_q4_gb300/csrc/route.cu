// Router: logits = x W_r^T in fp32, then top-k with warp shuffles and a
// softmax over the k chosen logits.
//
// The page "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU"
// (Methodology 1, prefill "grouped 4-bit GEMM for the MoE routing") routes
// every token to a few experts before the grouped GEMM.  Selection rule used
// here: top-k by logit; equal logits go to the lower expert index, decided by
// integer comparison of the indices; the weights are a softmax over the k
// chosen logits (equal to a full softmax renormalised over the k).
//
// Two shapes:
//   fused  16 tokens x all experts per CTA; logits stay in shared memory and
//          the CTA's warps pick the top-k.  Used for many tokens, and whenever
//          no logits buffer is available.  Optionally writes an fp16 copy of x
//          (the prefill GEMM operand) while it reads x anyway.
//   small  one warp per expert over all tokens (decode, T <= 32), spreading
//          the router matrix over many SMs; a second kernel picks the top-k.
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int RT = 16;   // tokens per fused CTA
constexpr int RK = 32;   // k-chunk of the fused CTA
constexpr int EMAX = kMaxExperts;

__global__ void __launch_bounds__(256) route_fused_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ wr, int T,
                                                          int H, int E, int k,
                                                          float* __restrict__ logits,
                                                          int32_t* __restrict__ idx,
                                                          float* __restrict__ w,
                                                          uint16_t* __restrict__ x16) {
    // Padded to 33 columns so both the row-wise fills and the column reads of
    // the inner loop are free of bank conflicts.
    __shared__ float xs[RT][RK + 1];
    __shared__ float ws[EMAX][RK + 1];
    const int t0 = blockIdx.x * RT;
    // thread (tx, ty): tokens 2ty, 2ty+1 and experts tx, tx+32, ..., tx+224
    const int tid = threadIdx.x, tx = tid % 32, ty = tid / 32;
    float acc[2][8];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < H; k0 += RK) {
        for (int i = tid; i < RT * RK; i += 256) {
            const int t = i / RK, kk = i % RK;
            const int tg = t0 + t, kg = k0 + kk;
            const bool in = tg < T && kg < H;
            const float v = in ? bf16_bits_to_float(x[(size_t)tg * H + kg]) : 0.f;
            xs[t][kk] = v;
            if (x16 && in) x16[(size_t)tg * H + kg] = float_to_half_bits_sat(v);
        }
        for (int i = tid; i < E * RK; i += 256) {
            const int e = i / RK, kk = i % RK;
            const int kg = k0 + kk;
            ws[e][kk] = (kg < H) ? wr[(size_t)e * H + kg] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < RK; ++kk) {
            const float xa[2] = {xs[ty * 2][kk], xs[ty * 2 + 1][kk]};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (tx + 32 * j < E) {  // experts beyond E are never read
                    const float wv = ws[tx + 32 * j][kk];
                    acc[0][j] = fmaf(xa[0], wv, acc[0][j]);
                    acc[1][j] = fmaf(xa[1], wv, acc[1][j]);
                }
            }
        }
        __syncthreads();
    }
    // logits of the CTA's tokens -> shared memory (reusing ws as [RT][EMAX])
    float* lg = &ws[0][0];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) lg[(ty * 2 + i) * EMAX + tx + 32 * j] = acc[i][j];
    __syncthreads();
    if (logits) {
        for (int i = tid; i < RT * E; i += 256) {
            const int t = i / E, e = i % E;
            if (t0 + t < T) logits[(size_t)(t0 + t) * E + e] = lg[t * EMAX + e];
        }
    }
    const int warp = tid / 32, lane = tid % 32;
    for (int t = warp; t < RT; t += 8) {
        const int tg = t0 + t;
        if (tg >= T) break;
        int si;
        float sw;
        warp_topk(lg + t * EMAX, E, k, si, sw);
        if (lane < k) {
            idx[(size_t)tg * k + lane] = si;
            w[(size_t)tg * k + lane] = sw;
        }
    }
}

// One warp per expert over all T (<= TMAX) tokens; needs H % 128 == 0.
template <int TMAX>
__global__ void __launch_bounds__(128) logits_small_kernel(const uint16_t* __restrict__ x,
                                                           const float* __restrict__ wr, int T,
                                                           int H, int E,
                                                           float* __restrict__ logits) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int e = blockIdx.x * 4 + warp;
    if (e >= E) return;
    float acc[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
    const float* wrow = wr + (size_t)e * H;
    for (int c = lane * 4; c < H; c += 128) {
        const float4 wv = *reinterpret_cast<const float4*>(wrow + c);
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
            if (t < T) {
                const uint2 xv = *reinterpret_cast<const uint2*>(x + (size_t)t * H + c);
                acc[t] = fmaf(__uint_as_float(xv.x << 16), wv.x, acc[t]);
                acc[t] = fmaf(__uint_as_float(xv.x & 0xffff0000u), wv.y, acc[t]);
                acc[t] = fmaf(__uint_as_float(xv.y << 16), wv.z, acc[t]);
                acc[t] = fmaf(__uint_as_float(xv.y & 0xffff0000u), wv.w, acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
            const float v = warp_sum(acc[t]);
            if (lane == 0) logits[(size_t)t * E + e] = v;
        }
    }
}

__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                   int k, int32_t* __restrict__ idx,
                                                   float* __restrict__ w) {
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
    if (t >= T) return;
    int si;
    float sw;
    warp_topk(logits + (size_t)t * E, E, k, si, sw);
    if (lane < k) {
        idx[(size_t)t * k + lane] = si;
        w[(size_t)t * k + lane] = sw;
    }
}

}  // namespace

// `logits` may be null; the split path is taken only when it is not.
cudaError_t launch_route(const uint16_t* x, const float* wr, int T, int H, int E, int k,
                         float* logits, int32_t* idx, float* w, uint16_t* x16, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (logits && !x16 && T <= 32 && (H % 128) == 0) {
        const dim3 grid((E + 3) / 4);
        if (T <= 4)
            logits_small_kernel<4><<<grid, 128, 0, s>>>(x, wr, T, H, E, logits);
        else if (T <= 16)
            logits_small_kernel<16><<<grid, 128, 0, s>>>(x, wr, T, H, E, logits);
        else
            logits_small_kernel<32><<<grid, 128, 0, s>>>(x, wr, T, H, E, logits);
        topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, k, idx, w);
    } else {
        route_fused_kernel<<<(T + RT - 1) / RT, 256, 0, s>>>(x, wr, T, H, E, k, logits, idx, w, x16);
    }
    return cudaGetLastError();
}

}  // namespace moeq4
