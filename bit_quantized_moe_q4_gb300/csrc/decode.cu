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
// One decode layer is three kernels, chained with programmatic dependent
// launch so each next grid is resident before its predecessor ends:
//   route    a thread-block cluster reads the router matrix spread over its
//            CTAs (one warp per expert), writes every logit into the leader
//            CTA's shared memory (distributed shared memory), quantises x to
//            int8 per 32, and after a cluster barrier the leader picks the
//            top-k, the softmax weights and the expert buckets;
//   gate/up  one CTA per (non-empty expert, 32 features): 32 gate + 32 up rows
//            over K = H, every weight load issued before the first use; then
//            h = silu(g) * u and its int8 quantisation (one 32-group per CTA);
//   down     one CTA per (non-empty expert, 64 rows of W_d) over K = I; y =
//            routing weight * row (fp32); the last CTA to finish a 64-row
//            block (ticket counter) adds the residual and the k expert rows of
//            every token in slot order, writing the output.
// Every weight byte of a touched expert is read once, by one CTA.
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int kRouteThreads = 256;  // 8 warps per cluster CTA
constexpr int kGuThreads = 256;
constexpr int kDnThreads = 256;
constexpr int kGpl = 16;            // weight groups per lane per pass (16 B each)

struct DecodeArgs {
    const uint16_t* x;
    const float* wr;
    const uint8_t* wgu;
    const uint8_t* wd;
    int T, H, I, E, k;
    float* logits;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* offsets;
    int32_t* touched;
    int32_t* counters;
    int32_t* tickets;  // [H / kDecodeDownRows] combine tickets of the down kernel
    int32_t* bucket_token;
    int32_t* bucket_slot;
    float* slot_w;
    int32_t* slot_pos;
    int8_t* q_x;
    uint16_t* d_x;
    int8_t* q_h;
    uint16_t* d_h;
    float* y;
    void* out;
    int out_fp32;
    int32_t* dots_gu;  // optional debug outputs
    int32_t* dots_d;
};

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 16-byte streaming load of read-once weights (not kept in L1).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Rearranges 8 int8 activations (x0..x7, one 8-column chunk) so that the two
// words line up with the packed code nibbles: the low nibbles of a code word
// (mask 0x0F0F0F0F) are columns 0,4,1,5 and the high nibbles 2,6,3,7.
__device__ __forceinline__ uint2 permute_chunk(uint32_t a, uint32_t b) {
    return make_uint2(__byte_perm(a, b, 0x5140), __byte_perm(a, b, 0x7362));
}

// Loads `c` int8 rows of length K into shared memory in the permuted order,
// with each 32-group's scale (as float) and code sum.
__device__ void stage_activations(const int8_t* __restrict__ q, const uint16_t* __restrict__ d,
                                  const int* rows, int c, int K, uint32_t* s_q, float* s_d,
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
        const int4* src = reinterpret_cast<const int4*>(q + (size_t)rows[n] * K + g * kGroup);
        int s = 0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int4 v = src[hh];
            const int w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) s = __dp4a(w[j], 0x01010101, s);  // signed byte sum
        }
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

// One thread's share of a packed row r (within its 128-row tiles starting at
// tbase): groups g = p, p + 4, ... (p = lane % 4), kGpl at a time, every load
// of a pass issued before its first use.  The activations of the `c` bucket
// rows are staged into shared memory while the first loads are in flight.
// The weights stay in registers while the tokens go by kTc at a time; each
// row's fp32 sums (fixed order: per lane over its groups, then over the 4
// lanes of the row) land in row_sum[0..c-1] (shared memory, written by the
// p == 0 lane).  Optionally writes the int32 group dots.
constexpr int kTc = 4;
__device__ __forceinline__ void row_w4a8(const uint8_t* __restrict__ tbase, int r, int K, int p,
                                         int c, const int* s_rows, const int8_t* q_src,
                                         const uint16_t* d_src, uint32_t* s_q, float* s_d,
                                         int* s_sum, float* row_sum, int32_t* dots,
                                         size_t dots_tok_stride) {
    const int G = K / kGroup;
    for (int g0 = 0; g0 < G; g0 += 4 * kGpl) {
        uint4 w[kGpl];
        uint32_t dwb[kGpl];
#pragma unroll
        for (int i = 0; i < kGpl; ++i) {
            const int g = g0 + p + 4 * i;
            if (g < G) {
                const uint8_t* t = tbase + (size_t)(g >> 1) * kTileBytes;
                w[i] = ldg_stream(t + r * 32 + (g & 1) * 16);
                dwb[i] = *reinterpret_cast<const uint16_t*>(t + kTileCodeBytes + r * 4 + (g & 1) * 2);
            }
        }
        if (g0 == 0) {
            stage_activations(q_src, d_src, s_rows, c, K, s_q, s_d, s_sum);
            __syncthreads();
        }
        for (int n0 = 0; n0 < c; n0 += kTc) {
            float acc[kTc];
#pragma unroll
            for (int j = 0; j < kTc; ++j) acc[j] = 0.f;
#pragma unroll
            for (int i = 0; i < kGpl; ++i) {
                const int g = g0 + p + 4 * i;
                if (g < G) {
                    const float dw = half_bits_to_float((uint16_t)dwb[i]);
#pragma unroll
                    for (int j = 0; j < kTc; ++j) {
                        const int n = n0 + j;
                        if (n < c) {
                            const int dot = group_dot(w[i], s_q + (size_t)n * (K / 4) + g * 8,
                                                      s_sum[n * G + g]);
                            acc[j] = fmaf((float)dot, dw * s_d[n * G + g], acc[j]);
                            if (dots) dots[(size_t)n * dots_tok_stride + g] = dot;
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kTc; ++j) {
                acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 1);
                acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 2);
            }
            if (p == 0) {
#pragma unroll
                for (int j = 0; j < kTc; ++j)
                    if (n0 + j < c) row_sum[n0 + j] = (g0 == 0 ? 0.f : row_sum[n0 + j]) + acc[j];
            }
        }
    }
}

// ---------------------------------------------------------------- route
template <int TM>
__global__ void __launch_bounds__(kRouteThreads) decode_route_kernel(const DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t dsm[];  // x as bf16 [T][H]
    __shared__ float s_logits[MOE_DECODE_MAX_T][kMaxExperts];
    __shared__ int s_idx[MOE_DECODE_MAX_T][MOE_MAX_TOPK];
    __shared__ float s_w[MOE_DECODE_MAX_T][MOE_MAX_TOPK];
    __shared__ uint32_t s_bits[kMaxExperts];
    __shared__ int s_off[kMaxExperts];
    const int T = a.T, H = a.H, E = a.E, k = a.k;
    const uint32_t rank = cluster_ctarank(), ncta = cluster_nctarank();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    pdl_trigger();  // the gate/up grid may be scheduled now; it waits for our end
    const int W = (int)ncta * (kRouteThreads / 32);
    const int gw = (int)rank * (kRouteThreads / 32) + warp;
    // The first 2048 columns of this warp's first router row are requested
    // before x is staged, so both loads overlap.
    constexpr int kWl = 16;  // float4 per lane per pass (2048 columns)
    float4 wpre[kWl];
    if (gw < E) {
        const float* row = a.wr + (size_t)gw * H;
#pragma unroll
        for (int i = 0; i < kWl; ++i) {
            const int c = lane * 4 + 128 * i;
            if (c < H) wpre[i] = __ldg(reinterpret_cast<const float4*>(row + c));
        }
    }
    uint16_t* sx = reinterpret_cast<uint16_t*>(dsm);
    for (int i = threadIdx.x; i < T * H / 8; i += blockDim.x)
        reinterpret_cast<uint4*>(sx)[i] = reinterpret_cast<const uint4*>(a.x)[i];
    __syncthreads();

    const uint32_t leader_logits = mapa_shared(smem_u32(&s_logits[0][0]), 0);
    for (int e = gw; e < E; e += W) {
        float acc[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) acc[t] = 0.f;
        const float* row = a.wr + (size_t)e * H;
        for (int c0 = 0; c0 < H; c0 += 128 * kWl) {
            if (!(e == gw && c0 == 0)) {
#pragma unroll
                for (int i = 0; i < kWl; ++i) {
                    const int c = c0 + lane * 4 + 128 * i;
                    if (c < H) wpre[i] = __ldg(reinterpret_cast<const float4*>(row + c));
                }
            }
#pragma unroll
            for (int i = 0; i < kWl; ++i) {
                const int c = c0 + lane * 4 + 128 * i;
                if (c < H) {
                    const float4 wv = wpre[i];
#pragma unroll
                    for (int t = 0; t < TM; ++t) {
                        if (t < T) {
                            const uint2 xv = *reinterpret_cast<const uint2*>(sx + t * H + c);
                            acc[t] = fmaf(__uint_as_float(xv.x << 16), wv.x, acc[t]);
                            acc[t] = fmaf(__uint_as_float(xv.x & 0xffff0000u), wv.y, acc[t]);
                            acc[t] = fmaf(__uint_as_float(xv.y << 16), wv.z, acc[t]);
                            acc[t] = fmaf(__uint_as_float(xv.y & 0xffff0000u), wv.w, acc[t]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            if (t < T) {
                const float v = warp_sum(acc[t]);
                if (lane == 0)
                    st_cluster_f32(leader_logits + (uint32_t)(t * kMaxExperts + e) * 4u, v);
            }
        }
    }
    // int8 quantisation of x, spread over the cluster's warps
    const int G = H / kGroup;
    for (int q = gw; q < T * G; q += W) {
        const int t = q / G, g = q % G;
        const float v = bf16_bits_to_float(sx[t * H + g * kGroup + lane]);
        const float amax = warp_max(fabsf(v));
        const uint16_t db = act_scale_bits(amax);
        a.q_x[(size_t)t * H + g * kGroup + lane] = (int8_t)act_code(v, half_bits_to_float(db));
        if (lane == 0) a.d_x[(size_t)t * G + g] = db;
    }
    cluster_sync_all();
    if (rank != 0) return;

    // ---- leader CTA: top-k, weights, buckets ----
    for (int t = warp; t < T; t += kRouteThreads / 32) {
        int si;
        float sw;
        warp_topk(&s_logits[t][0], E, k, si, sw);
        if (lane < k) {
            s_idx[t][lane] = si;
            s_w[t][lane] = sw;
            a.topk_idx[t * k + lane] = si;
            a.topk_w[t * k + lane] = sw;
        }
    }
    for (int i = threadIdx.x; i < T * E; i += blockDim.x) a.logits[i] = s_logits[i / E][i % E];
    for (int i = threadIdx.x; i < H / kDecodeDownRows; i += blockDim.x) a.tickets[i] = 0;
    for (int e = threadIdx.x; e < kMaxExperts; e += blockDim.x) s_bits[e] = 0u;
    __syncthreads();
    if (warp != 0) return;
    // token t is lane t (T <= 32): per-expert bitmask of the tokens that chose it
    if (lane < T)
        for (int j = 0; j < k; ++j) atomicOr(&s_bits[s_idx[lane][j]], 1u << lane);
    __syncwarp();
    constexpr int EPL = kMaxExperts / 32;  // experts per lane in the scans
    int cnt[EPL];
    int tot = 0, nt = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane * EPL + i;
        cnt[i] = e < E ? __popc(s_bits[e]) : 0;
        tot += cnt[i];
        nt += cnt[i] > 0;
    }
    int inc = tot, incn = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        const int vn = __shfl_up_sync(0xffffffffu, incn, o);
        if (lane >= o) {
            inc += v;
            incn += vn;
        }
    }
    int base = inc - tot, nbase = incn - nt;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane * EPL + i;
        if (e < E) {
            s_off[e] = base;
            a.offsets[e] = base;
            if (cnt[i] > 0) a.touched[nbase++] = e;
            base += cnt[i];
        }
    }
    const int total = __shfl_sync(0xffffffffu, inc, 31);
    const int ntouched = __shfl_sync(0xffffffffu, incn, 31);
    if (lane == 0) {
        a.offsets[E] = total;
        a.counters[kCntTouched] = ntouched;
    }
    __syncwarp();
    if (lane < T) {
        const uint32_t below = (1u << lane) - 1u;
        for (int j = 0; j < k; ++j) {
            const int e = s_idx[lane][j];
            const int pos = s_off[e] + __popc(s_bits[e] & below);
            a.bucket_token[pos] = lane;
            a.bucket_slot[pos] = j;
            a.slot_w[pos] = s_w[lane][j];
            a.slot_pos[lane * k + j] = pos;
        }
    }
}

// -------------------------------------------------------------- gate/up
__global__ void __launch_bounds__(kGuThreads, 2) decode_gateup_kernel(const DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ float s_acc[64][MOE_DECODE_MAX_T + 1];
    __shared__ int s_rows[MOE_DECODE_MAX_T];
    pdl_wait();     // routing, buckets and q_x of this call
    pdl_trigger();  // the down grid may be scheduled now
    if ((int)blockIdx.x >= a.counters[kCntTouched]) return;
    const int H = a.H, I = a.I, G = H / kGroup;
    const int e = a.touched[blockIdx.x];
    const int off = a.offsets[e], c = a.offsets[e + 1] - off;
    const int fb = blockIdx.y;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rloc = warp * 8 + lane / 4;  // 0..31 gate, 32..63 up
    const int m = rloc / 32;
    const int f = fb * 32 + (rloc % 32);
    const int prow = m * I + f;            // row of the [2I, H] gate/up tensor
    const int p = lane % 4;
    uint32_t* s_q = reinterpret_cast<uint32_t*>(dsm);
    float* s_d = reinterpret_cast<float*>(dsm + (size_t)c * H);
    int* s_sum = reinterpret_cast<int*>(s_d + c * G);
    if (threadIdx.x < c) s_rows[threadIdx.x] = a.bucket_token[off + threadIdx.x];
    __syncthreads();
    const uint8_t* tbase =
        a.wgu + ((size_t)e * (2 * I / kTileRows) + prow / kTileRows) * (H / kTileK) * kTileBytes;
    int32_t* dots = a.dots_gu ? a.dots_gu + ((size_t)off * 2 * I + prow) * G : nullptr;
    row_w4a8(tbase, prow % kTileRows, H, p, c, s_rows, a.q_x, a.d_x, s_q, s_d, s_sum,
             &s_acc[rloc][0], dots, (size_t)2 * I * G);
    __syncthreads();
    // SwiGLU and the int8 quantisation of h: one 32-feature group per CTA
    for (int n = warp; n < c; n += kGuThreads / 32) {
        const float g = s_acc[lane][n], u = s_acc[32 + lane][n];
        const float h = g / (1.0f + __expf(-g)) * u;
        const float amax = warp_max(fabsf(h));
        const uint16_t db = act_scale_bits(amax);
        const size_t slot = (size_t)off + n;
        a.q_h[slot * I + fb * 32 + lane] = (int8_t)act_code(h, half_bits_to_float(db));
        if (lane == 0) a.d_h[slot * (I / kGroup) + fb] = db;
    }
}

// ------------------------------------------------------- down + combine
__global__ void __launch_bounds__(kDnThreads, 2) decode_down_kernel(const DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ float s_acc[kDecodeDownRows][MOE_DECODE_MAX_T + 1];
    __shared__ int s_rows[MOE_DECODE_MAX_T];
    __shared__ int s_last;
    pdl_wait();  // h codes of this call (and, transitively, the routing)
    const int ntouched = a.counters[kCntTouched];
    if ((int)blockIdx.x >= ntouched) return;
    const int H = a.H, I = a.I, G = I / kGroup;
    const int e = a.touched[blockIdx.x];
    const int off = a.offsets[e], c = a.offsets[e + 1] - off;
    const int rb = blockIdx.y;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rloc = warp * 8 + lane / 4;
    const int row = rb * kDecodeDownRows + rloc;
    const int p = lane % 4;
    uint32_t* s_q = reinterpret_cast<uint32_t*>(dsm);
    float* s_d = reinterpret_cast<float*>(dsm + (size_t)c * I);
    int* s_sum = reinterpret_cast<int*>(s_d + c * G);
    if (threadIdx.x < c) s_rows[threadIdx.x] = off + threadIdx.x;  // h rows are bucket rows
    __syncthreads();
    const uint8_t* tbase =
        a.wd + ((size_t)e * (H / kTileRows) + row / kTileRows) * (I / kTileK) * kTileBytes;
    int32_t* dots = a.dots_d ? a.dots_d + ((size_t)off * H + row) * G : nullptr;
    row_w4a8(tbase, row % kTileRows, I, p, c, s_rows, a.q_h, a.d_h, s_q, s_d, s_sum,
             &s_acc[rloc][0], dots, (size_t)H * G);
    if (p == 0)
        for (int n = 0; n < c; ++n) a.y[((size_t)off + n) * H + row] = s_acc[rloc][n] * a.slot_w[off + n];
    // The last CTA to finish this 64-row block combines it for every token.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&a.tickets[rb], 1) == ntouched - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int T = a.T, k = a.k;
    for (int i = threadIdx.x; i < T * kDecodeDownRows; i += blockDim.x) {
        const int t = i / kDecodeDownRows, col = rb * kDecodeDownRows + i % kDecodeDownRows;
        float v = bf16_bits_to_float(a.x[(size_t)t * H + col]);
        for (int j = 0; j < k; ++j) v += __ldcg(a.y + (size_t)a.slot_pos[t * k + j] * H + col);
        if (a.out_fp32)
            static_cast<float*>(a.out)[(size_t)t * H + col] = v;
        else
            static_cast<uint16_t*>(a.out)[(size_t)t * H + col] = float_to_bf16_bits(v);
    }
}

size_t act_smem(int TM, int K) { return (size_t)TM * K + (size_t)TM * (K / kGroup) * 8; }

int g_cluster_size[64] = {};

// Cluster size of the route kernel: 16 CTAs where the device can place such a
// cluster, else the portable 8.  Chosen once per device.
template <int TM>
int route_cluster_size(size_t smem) {
    int dev = 0;
    cudaGetDevice(&dev);
    int& cs = g_cluster_size[dev & 63];
    if (cs != 0) return cs;
    cudaFuncSetAttribute(decode_route_kernel<TM>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t q{};
    cudaLaunchAttribute qa[1];
    q.gridDim = dim3(16);
    q.blockDim = dim3(kRouteThreads);
    q.dynamicSmemBytes = smem;
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = 16;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    q.attrs = qa;
    q.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, decode_route_kernel<TM>, &q) == cudaSuccess &&
        nclusters > 0)
        cs = 16;
    else
        cs = 8;
    cudaGetLastError();  // a refused query leaves no error behind
    return cs;
}

template <int TM>
cudaError_t launch_all(const DecodeArgs& a, void** ev, bool capturing, cudaStream_t s) {
    cudaError_t err;
    auto mark = [&](int i) -> cudaError_t {
        return (ev && ev[i]) ? record_stage(ev[i], s, capturing) : cudaSuccess;
    };
    const size_t rsm = (size_t)a.T * a.H * 2;
    err = cudaFuncSetAttribute(decode_route_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)rsm);
    if (err != cudaSuccess) return err;
    const int cs = route_cluster_size<TM>(rsm);
    if (cs > 8) {
        err = cudaFuncSetAttribute(decode_route_kernel<TM>,
                                   cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess) return err;
    }
    {
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute at[1];
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = rsm;
        cfg.stream = s;
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = cs;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, decode_route_kernel<TM>, a);
        if (err != cudaSuccess) return err;
    }
    for (int i = 1; i <= 3; ++i)
        if ((err = mark(i)) != cudaSuccess) return err;
    const int max_touched = min(a.E, a.T * a.k);
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    {
        const size_t smem = act_smem(a.T, a.H);
        err = cudaFuncSetAttribute(decode_gateup_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(max_touched, a.I / 32);
        cfg.blockDim = dim3(kGuThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, decode_gateup_kernel, a);
        if (err != cudaSuccess) return err;
    }
    if ((err = mark(4)) != cudaSuccess) return err;
    {
        const size_t smem = act_smem(a.T, a.I);
        err = cudaFuncSetAttribute(decode_down_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(max_touched, a.H / kDecodeDownRows);
        cfg.blockDim = dim3(kDnThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, decode_down_kernel, a);
        if (err != cudaSuccess) return err;
    }
    if ((err = mark(5)) != cudaSuccess || (err = mark(6)) != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const uint16_t* x, const float* wr, const void* wgu, const void* wd,
                          int T, int H, int I, int E, int k, bool out_fp32, void* out,
                          const Workspace& ws, int32_t* dots_gu, int32_t* dots_d,
                          void** events, bool capturing, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    DecodeArgs a{};
    a.x = x;
    a.wr = wr;
    a.wgu = static_cast<const uint8_t*>(wgu);
    a.wd = static_cast<const uint8_t*>(wd);
    a.T = T;
    a.H = H;
    a.I = I;
    a.E = E;
    a.k = k;
    a.logits = ws.logits;
    a.topk_idx = ws.topk_idx;
    a.topk_w = ws.topk_w;
    a.offsets = ws.offsets;
    a.touched = ws.touched;
    a.counters = ws.counters;
    a.tickets = ws.tickets;
    a.bucket_token = ws.bucket_token;
    a.bucket_slot = ws.bucket_slot;
    a.slot_w = ws.slot_w;
    a.slot_pos = ws.slot_pos;
    a.q_x = ws.q_x;
    a.d_x = ws.d_x;
    a.q_h = ws.q_h;
    a.d_h = ws.d_h;
    a.y = static_cast<float*>(ws.y);
    a.out = out;
    a.out_fp32 = out_fp32 ? 1 : 0;
    a.dots_gu = dots_gu;
    a.dots_d = dots_d;
    if (T <= 1) return launch_all<1>(a, events, capturing, s);
    if (T <= 2) return launch_all<2>(a, events, capturing, s);
    if (T <= 4) return launch_all<4>(a, events, capturing, s);
    if (T <= 8) return launch_all<8>(a, events, capturing, s);
    if (T <= 16) return launch_all<16>(a, events, capturing, s);
    return launch_all<32>(a, events, capturing, s);
}

}  // namespace moeq4
