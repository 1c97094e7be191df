// W4A8 decode path: exact int32 group dot products of 4-bit weight codes with
// int8 activations, scaled per group in fp32.
//
// Page "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU",
// Methodology 1 "Decode (CPU)" and Key Contributions 2: a W4A8 integer
// multiply-add kernel (there SSSE3 pmaddubsw on the host).  Here each group
// dot G = sum_{i in block} (q_i - 8) * a_i is formed with dp4a on the GPU:
// sum q*a (codes unsigned, activations signed) minus 8 * sum a, both exact in
// int32 (|G| <= 32 * 8 * 127).  A row is sum_g d_w[g] * d_a[g] * G[g] in fp32.
//
// Kernels (one CTA per (non-empty expert, row block); tokens of the expert's
// bucket are all handled by the CTA, so each weight byte is read once):
//   gate/up: 32 features x (gate, up) rows, K = H; then h = silu(g) * u and
//            its int8 quantisation per 32 features (one group per CTA).
//   down:    64 rows of W_d, K = I; y = routing weight * row sum (fp32).
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int TMAX = MOE_DECODE_MAX_T;

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Rearranges 8 int8 activations (x0..x7, one 8-column chunk) so that the two
// words line up with the packed code nibbles: the low nibbles of a code word
// (mask 0x0F0F0F0F) are columns 0,4,1,5 and the high nibbles 2,6,3,7.
__device__ __forceinline__ uint2 permute_chunk(uint32_t a, uint32_t b) {
    // a = x0 x1 x2 x3 (byte 0 first), b = x4 x5 x6 x7
    const uint32_t lo = __byte_perm(a, b, 0x5140);  // x0 x4 x1 x5
    const uint32_t hi = __byte_perm(a, b, 0x7362);  // x2 x6 x3 x7
    return make_uint2(lo, hi);
}

// Loads the int8 activations of `c` bucket rows into shared memory in the
// permuted order, plus per-group scales (as float) and per-group sums.
__device__ void stage_activations(const int8_t* __restrict__ q, const uint16_t* __restrict__ d,
                                  const int32_t* rows, int c, int K, uint32_t* s_q, float* s_d,
                                  int* s_sum) {
    const int chunks = K / 8;
    for (int i = threadIdx.x; i < c * chunks; i += blockDim.x) {
        const int n = i / chunks, ch = i % chunks;
        const uint2 v = *reinterpret_cast<const uint2*>(q + (size_t)rows[n] * K + ch * 8);
        const uint2 p = permute_chunk(v.x, v.y);
        s_q[(size_t)n * (K / 4) + ch * 2] = p.x;
        s_q[(size_t)n * (K / 4) + ch * 2 + 1] = p.y;
    }
    const int G = K / kGroup;
    for (int i = threadIdx.x; i < c * G; i += blockDim.x) {
        const int n = i / G, g = i % G;
        s_d[i] = half_bits_to_float(d[(size_t)rows[n] * G + g]);
        const int8_t* src = q + (size_t)rows[n] * K + g * kGroup;
        int s = 0;
        for (int j = 0; j < kGroup; ++j) s += src[j];
        s_sum[i] = s;
    }
}

// Group dot of one packed 32-code group (4 words) with one staged activation
// group (8 permuted words).
__device__ __forceinline__ int group_dot(const uint4 w, const uint32_t* a, int asum) {
    const uint4 a0 = *reinterpret_cast<const uint4*>(a);
    const uint4 a1 = *reinterpret_cast<const uint4*>(a + 4);
    int acc = 0;
    acc = dp4a_us(w.x & 0x0F0F0F0Fu, a0.x, acc);
    acc = dp4a_us((w.x >> 4) & 0x0F0F0F0Fu, a0.y, acc);
    acc = dp4a_us(w.y & 0x0F0F0F0Fu, a0.z, acc);
    acc = dp4a_us((w.y >> 4) & 0x0F0F0F0Fu, a0.w, acc);
    acc = dp4a_us(w.z & 0x0F0F0F0Fu, a1.x, acc);
    acc = dp4a_us((w.z >> 4) & 0x0F0F0F0Fu, a1.y, acc);
    acc = dp4a_us(w.w & 0x0F0F0F0Fu, a1.z, acc);
    acc = dp4a_us((w.w >> 4) & 0x0F0F0F0Fu, a1.w, acc);
    return acc - 8 * asum;
}

// Each warp: 8 rows; lane = (K-block parity, row, group-in-block).  Returns
// the lane's partial row sums for every token, reduced over the four lanes of
// its row (valid in lanes with parity 0 and group 0).
__device__ __forceinline__ void rows_w4a8(const uint8_t* __restrict__ wpk, int rb_per_e, int e,
                                          int row, int K, const uint32_t* s_q, const float* s_d,
                                          const int* s_sum, int c, float (&acc)[TMAX],
                                          int32_t* dots, size_t dots_row_stride,
                                          size_t dots_tok_stride) {
    const int lane = threadIdx.x % 32;
    const int half = lane / 16, gsel = lane % 2;
    const int KB = K / kTileK, G = K / kGroup;
    const int rb = row / kTileRows, r = row % kTileRows;
    const uint8_t* base = wpk + ((size_t)e * rb_per_e + rb) * KB * kTileBytes;
#pragma unroll
    for (int n = 0; n < TMAX; ++n) acc[n] = 0.f;
#pragma unroll 4
    for (int kb = half; kb < KB; kb += 2) {
        const uint8_t* tile = base + (size_t)kb * kTileBytes;
        const uint4 w = *reinterpret_cast<const uint4*>(tile + r * 32 + gsel * 16);
        const float dw =
            half_bits_to_float(*reinterpret_cast<const uint16_t*>(tile + kTileCodeBytes + r * 4 + gsel * 2));
        const int g = kb * 2 + gsel;
#pragma unroll
        for (int n = 0; n < TMAX; ++n) {
            if (n < c) {
                const int dot = group_dot(w, s_q + (size_t)n * (K / 4) + g * 8, s_sum[n * G + g]);
                acc[n] = fmaf((float)dot, dw * s_d[n * G + g], acc[n]);
                if (dots) dots[(size_t)n * dots_tok_stride + (size_t)row * dots_row_stride + g] = dot;
            }
        }
    }
#pragma unroll
    for (int n = 0; n < TMAX; ++n) {
        acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], 1);
        acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], 16);
    }
}

__global__ void __launch_bounds__(256) decode_gateup_kernel(
    const uint8_t* __restrict__ wgu, const int8_t* __restrict__ q_x,
    const uint16_t* __restrict__ d_x, const int32_t* __restrict__ counters,
    const int32_t* __restrict__ touched, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ bucket_token, int H, int I, int8_t* __restrict__ q_h,
    uint16_t* __restrict__ d_h, int32_t* __restrict__ dots_dbg) {
    extern __shared__ __align__(16) uint8_t smem[];
    if ((int)blockIdx.x >= counters[kCntTouched]) return;
    const int e = touched[blockIdx.x];
    const int off = offsets[e], c = offsets[e + 1] - off;
    const int fb = blockIdx.y;  // 32 features
    __shared__ int rows[TMAX];
    __shared__ float s_acc[64][TMAX + 1];
    const int G = H / kGroup;
    uint32_t* s_q = reinterpret_cast<uint32_t*>(smem);
    float* s_d = reinterpret_cast<float*>(smem + (size_t)TMAX * H);
    int* s_sum = reinterpret_cast<int*>(s_d + TMAX * G);
    if (threadIdx.x < c) rows[threadIdx.x] = bucket_token[off + threadIdx.x];
    __syncthreads();
    stage_activations(q_x, d_x, rows, c, H, s_q, s_d, s_sum);
    __syncthreads();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int m = warp / 4;                     // 0 gate, 1 up
    const int rl = (lane % 16) / 2;
    const int f = fb * 32 + (warp % 4) * 8 + rl;  // feature
    const int row = m * I + f;                    // row of the [2I, H] gate/up tensor
    float acc[TMAX];
    int32_t* dots = dots_dbg ? dots_dbg + (size_t)off * (2 * I) * G : nullptr;
    rows_w4a8(wgu, (2 * I) / kTileRows, e, row, H, s_q, s_d, s_sum, c, acc, dots, G,
              (size_t)(2 * I) * G);
    if ((lane & 17) == 0) {
#pragma unroll
        for (int n = 0; n < TMAX; ++n)
            if (n < c) s_acc[m * 32 + (warp % 4) * 8 + rl][n] = acc[n];
    }
    __syncthreads();
    // SwiGLU and the int8 quantisation of h: one group of 32 features per CTA
    for (int n = warp; n < c; n += 8) {
        const float g = s_acc[lane][n], u = s_acc[32 + lane][n];
        const float h = g / (1.0f + __expf(-g)) * u;
        const float amax = warp_max(fabsf(h));
        const uint16_t db = act_scale_bits(amax);
        const size_t slot = (size_t)off + n;
        q_h[slot * I + fb * 32 + lane] = (int8_t)act_code(h, half_bits_to_float(db));
        if (lane == 0) d_h[slot * (I / kGroup) + fb] = db;
    }
}

__global__ void __launch_bounds__(256) decode_down_kernel(
    const uint8_t* __restrict__ wd, const int8_t* __restrict__ q_h,
    const uint16_t* __restrict__ d_h, const int32_t* __restrict__ counters,
    const int32_t* __restrict__ touched, const int32_t* __restrict__ offsets,
    const float* __restrict__ slot_w, int H, int I, float* __restrict__ y,
    int32_t* __restrict__ dots_dbg) {
    extern __shared__ __align__(16) uint8_t smem[];
    if ((int)blockIdx.x >= counters[kCntTouched]) return;
    const int e = touched[blockIdx.x];
    const int off = offsets[e], c = offsets[e + 1] - off;
    __shared__ int rows[TMAX];
    const int G = I / kGroup;
    uint32_t* s_q = reinterpret_cast<uint32_t*>(smem);
    float* s_d = reinterpret_cast<float*>(smem + (size_t)TMAX * I);
    int* s_sum = reinterpret_cast<int*>(s_d + TMAX * G);
    if (threadIdx.x < c) rows[threadIdx.x] = off + threadIdx.x;  // h rows are bucket rows
    __syncthreads();
    stage_activations(q_h, d_h, rows, c, I, s_q, s_d, s_sum);
    __syncthreads();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rl = (lane % 16) / 2;
    const int row = blockIdx.y * 64 + warp * 8 + rl;
    float acc[TMAX];
    int32_t* dots = dots_dbg ? dots_dbg + (size_t)off * H * G : nullptr;
    rows_w4a8(wd, H / kTileRows, e, row, I, s_q, s_d, s_sum, c, acc, dots, G, (size_t)H * G);
    if ((lane & 17) == 0) {
#pragma unroll
        for (int n = 0; n < TMAX; ++n)
            if (n < c) y[((size_t)off + n) * H + row] = acc[n] * slot_w[off + n];
    }
}

size_t decode_smem(int K) { return (size_t)TMAX * K + (size_t)TMAX * (K / kGroup) * 8; }

}  // namespace

cudaError_t launch_decode_gateup(const void* wgu, const Workspace& ws, int T, int H, int I,
                                 int E, int k, int32_t* dots_dbg, cudaStream_t s) {
    const int max_touched = min(E, T * k);
    if (max_touched == 0) return cudaSuccess;
    const size_t smem = decode_smem(H);
    cudaFuncSetAttribute(decode_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(max_touched, I / 32);
    decode_gateup_kernel<<<grid, 256, smem, s>>>(
        static_cast<const uint8_t*>(wgu), ws.q_x, ws.d_x, ws.counters, ws.touched, ws.offsets,
        ws.bucket_token, H, I, ws.q_h, ws.d_h, dots_dbg);
    return cudaGetLastError();
}

cudaError_t launch_decode_down(const void* wd, const Workspace& ws, int T, int H, int I, int E,
                               int k, int32_t* dots_dbg, cudaStream_t s) {
    const int max_touched = min(E, T * k);
    if (max_touched == 0) return cudaSuccess;
    const size_t smem = decode_smem(I);
    cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(max_touched, H / 64);
    decode_down_kernel<<<grid, 256, smem, s>>>(static_cast<const uint8_t*>(wd), ws.q_h, ws.d_h,
                                               ws.counters, ws.touched, ws.offsets, ws.slot_w, H,
                                               I, static_cast<float*>(ws.y), dots_dbg);
    return cudaGetLastError();
}

}  // namespace moeq4
