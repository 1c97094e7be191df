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
// Three shapes:
//   gemm   (many tokens, a buffer for K parts available) a register-blocked
//          fp32 GEMM: each CTA forms 64 tokens x 128 experts over one slice
//          of the hidden dimension (the slices keep every SM busy); a second
//          kernel adds the slices in order and picks the top-k, one warp per
//          token.  The GEMM CTAs also write the fp16 copy of x that the
//          prefill tensor-core GEMM reads, each for its own tokens and slice.
//   fused  16 tokens x all experts per CTA; logits stay in shared memory and
//          the CTA's warps pick the top-k (no buffer needed).
//   small  one warp per expert over all tokens (T <= 32), spreading the
//          router matrix over many SMs; a second kernel picks the top-k.
//   tensor (prefill, T >= 128) the same K-sliced product on the tensor cores:
//          W_r is first split exactly into three bf16 matrices
//          (W_r = hi + mid + lo, each part the bf16 rounding of what the
//          earlier parts leave), so every product of a bf16 x with a part is
//          exact in the fp32 accumulator and the sum over the three parts is
//          x W_r^T with fp32 accumulation, as in the fp32 kernels.  One CTA
//          forms 128 experts x 128 tokens over one slice of the hidden
//          dimension with tcgen05.mma (TMA-loaded 128-byte-swizzled tiles,
//          accumulator in tensor memory); the top-k kernel of the gemm shape
//          adds the slices in order.
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

// ---- register-blocked fp32 router GEMM ------------------------------------
constexpr int GT = 64;    // tokens per CTA
constexpr int GE = 128;   // experts per CTA
constexpr int GK = 16;    // hidden columns per shared-memory stage
constexpr int G_THREADS = 256;

// parts[s][t][e] = sum over h in slice s of x[t, h] * W[e, h] (fp32).
// Warp w owns tokens 8w..8w+7, lane l experts 4l..4l+3: per column 32 FMAs
// for two broadcast 16-byte loads of x and one 16-byte load of W.
__global__ void __launch_bounds__(G_THREADS) router_gemm_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ wr, int T, int H, int E, int ksplit,
    float* __restrict__ parts, uint16_t* __restrict__ x16) {
    __shared__ __align__(16) float xs[2][GK][GT];
    __shared__ __align__(16) float ws[2][GK][GE];
    pdl_wait();  // x (the preceding work on the stream)
    pdl_trigger();
    const int t0 = blockIdx.x * GT, e0 = blockIdx.y * GE, split = blockIdx.z;
    const int kspan = H / ksplit, kbeg = split * kspan;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    // loader roles: W: rows e = e0 + (tid % 64) + 64 r (r = 0, 1), column quad
    // q = tid / 64 (4 columns); x: token tid / 2, half tid % 2 (8 columns)
    const int we = tid % 64, wq = tid / 64;
    const int xt = tid / 2, xh = tid % 2;
    const bool x_loader = tid < 2 * GT;
    const bool write_x16 = x16 != nullptr && blockIdx.y == 0;
    float4 wreg[2];
    uint4 xreg;
    auto load = [&](int k0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int e = e0 + we + 64 * r;
            wreg[r] = (e < E) ? __ldg(reinterpret_cast<const float4*>(wr + (size_t)e * H + k0 + wq * 4))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (x_loader) {
            const int t = t0 + xt;
            xreg = (t < T) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + k0 + xh * 8))
                           : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    auto store = [&](int buf, int k0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            ws[buf][wq * 4 + 0][we + 64 * r] = wreg[r].x;
            ws[buf][wq * 4 + 1][we + 64 * r] = wreg[r].y;
            ws[buf][wq * 4 + 2][we + 64 * r] = wreg[r].z;
            ws[buf][wq * 4 + 3][we + 64 * r] = wreg[r].w;
        }
        if (x_loader) {
            const uint32_t w4[4] = {xreg.x, xreg.y, xreg.z, xreg.w};
            uint32_t h4[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float lo = __uint_as_float(w4[c] << 16), hi = __uint_as_float(w4[c] & 0xffff0000u);
                xs[buf][xh * 8 + 2 * c][xt] = lo;
                xs[buf][xh * 8 + 2 * c + 1][xt] = hi;
                h4[c] = (uint32_t)float_to_half_bits_sat(lo) | ((uint32_t)float_to_half_bits_sat(hi) << 16);
            }
            const int t = t0 + xt;
            if (write_x16 && t < T)
                *reinterpret_cast<uint4*>(x16 + (size_t)t * H + k0 + xh * 8) =
                    make_uint4(h4[0], h4[1], h4[2], h4[3]);
        }
    };
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const int nstage = kspan / GK;
    load(kbeg);
    store(0, kbeg);
    __syncthreads();
    for (int st = 0; st < nstage; ++st) {
        const int buf = st & 1;
        if (st + 1 < nstage) load(kbeg + (st + 1) * GK);  // next stage in flight
#pragma unroll
        for (int kk = 0; kk < GK; ++kk) {
            const float4 xa = *reinterpret_cast<const float4*>(&xs[buf][kk][warp * 8]);
            const float4 xb = *reinterpret_cast<const float4*>(&xs[buf][kk][warp * 8 + 4]);
            const float4 wv = *reinterpret_cast<const float4*>(&ws[buf][kk][lane * 4]);
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
            const float wvv[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wvv[j], acc[i][j]);
        }
        if (st + 1 < nstage) {
            store(buf ^ 1, kbeg + (st + 1) * GK);
            __syncthreads();
        }
    }
    float* out = parts + (size_t)split * T * E;
    const int e = e0 + lane * 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = t0 + warp * 8 + i;
        if (t >= T) break;
        if (e + 3 < E && (E % 4) == 0) {  // 16-byte aligned only when E % 4 == 0
            *reinterpret_cast<float4*>(out + (size_t)t * E + e) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (e + j < E) out[(size_t)t * E + e + j] = acc[i][j];
        }
    }
}

// One warp per token: logits = the K-slice parts added in slice order, then
// the top-k.  `logits` (optional, may equal parts when there is one slice)
// receives the sums.
__global__ void __launch_bounds__(256) topk_from_parts_kernel(const float* __restrict__ parts,
                                                              int ksplit, int T, int E, int k,
                                                              float* logits, int32_t* idx, float* w) {
    __shared__ float row[8][EMAX];
    pdl_wait();  // the K-slice parts
    pdl_trigger();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;  // whole warp
    constexpr int PER = EMAX / 32;
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) v[i] = 0.f;
    for (int s0 = 0; s0 < ksplit; s0 += 4) {
        float pv[4][PER];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int e = lane + 32 * i;
                pv[u][i] = (s0 + u < ksplit && e < E)
                               ? __ldcg(parts + ((size_t)(s0 + u) * T + t) * E + e) : 0.f;
            }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < PER; ++i) v[i] += pv[u][i];  // slices in order (adding 0 is exact)
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            row[warp][e] = v[i];
            if (logits) logits[(size_t)t * E + e] = v[i];
        }
    }
    __syncwarp();
    int si;
    float sw;
    warp_topk(row[warp], E, k, si, sw);
    if (lane < k) {
        idx[(size_t)t * k + lane] = si;
        w[(size_t)t * k + lane] = sw;
    }
}


// One CTA per 32-token chunk, one warp per token: the token's logits (the
// K-slice parts added in slice order), its top-k, and then the chunk's
// bucketing counts: a per-expert bitmask of the chunk's tokens that chose it
// gives each expert's count in the chunk and each (token, slot) pair's rank
// among the chunk's tokens of its expert (the first pass of the bucketing).
__global__ void __launch_bounds__(1024, 1) topk_chunk_kernel(
    const float* __restrict__ parts, int ksplit, int T, int E, int k, float* logits, int32_t* idx,
    float* w, int32_t* __restrict__ chunk_count, int32_t* __restrict__ entry_rank) {
    __shared__ __align__(16) float row[32][EMAX];
    __shared__ uint32_t bits[EMAX];
    pdl_wait();  // the K-slice parts
    pdl_trigger();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int chunk = blockIdx.x, t = chunk * 32 + warp;
    for (int e = threadIdx.x; e < EMAX; e += blockDim.x) bits[e] = 0u;
    __syncthreads();
    int si = 0;
    if (t < T) {  // whole warp
        if ((E % 4) == 0 && E <= 128 && ksplit <= 8) {
            // lane: experts 4 lane .. 4 lane + 3, one 16-byte load per slice,
            // every slice in flight at once
            const int e = 4 * lane;
            float4 pv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                pv[u] = (u < ksplit && e < E)
                            ? __ldcg(reinterpret_cast<const float4*>(parts + ((size_t)u * T + t) * E + e))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 8; ++u) {  // slices in order (adding 0 is exact)
                v.x += pv[u].x;
                v.y += pv[u].y;
                v.z += pv[u].z;
                v.w += pv[u].w;
            }
            if (e < E) {
                *reinterpret_cast<float4*>(&row[warp][e]) = v;
                if (logits) {
                    float* lr = logits + (size_t)t * E + e;
                    if ((reinterpret_cast<uintptr_t>(lr) & 15u) == 0) {
                        *reinterpret_cast<float4*>(lr) = v;
                    } else {
                        lr[0] = v.x;
                        lr[1] = v.y;
                        lr[2] = v.z;
                        lr[3] = v.w;
                    }
                }
            }
        } else {
            constexpr int PER = EMAX / 32;
            float v[PER];
#pragma unroll
            for (int i = 0; i < PER; ++i) v[i] = 0.f;
            for (int s0 = 0; s0 < ksplit; s0 += 2) {
                float pv[2][PER];
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < PER; ++i) {
                        const int e = lane + 32 * i;
                        pv[u][i] = (s0 + u < ksplit && e < E)
                                       ? __ldcg(parts + ((size_t)(s0 + u) * T + t) * E + e) : 0.f;
                    }
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < PER; ++i) v[i] += pv[u][i];  // slices in order
            }
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int e = lane + 32 * i;
                if (e < E) {
                    row[warp][e] = v[i];
                    if (logits) logits[(size_t)t * E + e] = v[i];
                }
            }
        }
        __syncwarp();
        float sw;
        warp_topk(row[warp], E, k, si, sw);
        if (lane < k) {
            idx[(size_t)t * k + lane] = si;
            w[(size_t)t * k + lane] = sw;
            atomicOr(&bits[si], 1u << warp);
        }
    }
    __syncthreads();
    if (t < T && lane < k) entry_rank[(size_t)t * k + lane] = __popc(bits[si] & ((1u << warp) - 1u));
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_count[(size_t)chunk * E + e] = __popc(bits[e]);
}

// ---- tensor-core router (prefill) -----------------------------------------
constexpr int TC_M = 128;                          // experts per CTA (MMA M)
constexpr int TC_N = 128;                          // tokens per CTA (MMA N)
constexpr int TC_STAGES = 3;
constexpr int TC_TILE_BYTES = 128 * 128;           // 128 rows x 64 bf16, swizzled
constexpr int TC_STAGE_BYTES = 4 * TC_TILE_BYTES;  // three W_r parts + x
constexpr int TC_OFF_BAR = TC_STAGES * TC_STAGE_BYTES;
constexpr int TC_SMEM = TC_OFF_BAR + 128 + 1024;   // barriers, TMEM slot, alignment slack
constexpr int TC_THREADS = 192;  // warp 0: TMA; warp 1: MMA; warps 2..5: x16 copy + epilogue
constexpr int TC_SMS = 148;      // SM count the slice choice plans for
constexpr int TC_MIN_T = 128;

// planes[p][e][h], p = 0, 1, 2: w = planes[0] + planes[1] + planes[2] exactly
// (bf16 keeps fp32's exponent range; each part takes the next 8 significant
// bits of what is left).
__global__ void __launch_bounds__(256) split_wr_kernel(const float* __restrict__ wr, int n4,
                                                       uint16_t* __restrict__ planes) {
    // The parts live in the caller's workspace, which the preceding work on
    // the stream may still be using (a decode call on the same workspace
    // lets its successor start early): write them only after the wait.
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(wr) + i);
        const float f[4] = {v.x, v.y, v.z, v.w};
        uint16_t q[3][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float r = f[j];
#pragma unroll
            for (int p = 0; p < 3; ++p) {
                q[p][j] = float_to_bf16_bits(r);
                r -= bf16_bits_to_float(q[p][j]);  // exact: the rounding error of the part
            }
        }
#pragma unroll
        for (int p = 0; p < 3; ++p)
            reinterpret_cast<uint2*>(planes + (size_t)p * n4 * 4)[i] =
                make_uint2(q[p][0] | ((uint32_t)q[p][1] << 16), q[p][2] | ((uint32_t)q[p][3] << 16));
    }
}

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major) and an
// fp32 accumulator of M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// parts[split][t][e] for experts e0..e0+127 and tokens t0..t0+127 over the
// hidden slice of this CTA.  tm_w maps the three parts as one [max(3E, 128),
// H] bf16 tensor (the rows past 3E are padding), tm_x maps x as [T, H] (T >=
// 128); rows past the end read as zero.  A box row past the CTA's part (the
// next part, or padding) only feeds an accumulator row of an expert >= E,
// which is not stored.  CTAs of the first expert block also write the fp16 copy of
// their x slice.
__global__ void __launch_bounds__(TC_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                     int T, int H, int E, int ksplit, float* __restrict__ parts,
                     uint16_t* __restrict__ x16, int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw_base);
    const int t0 = blockIdx.x * TC_N, e0 = blockIdx.y * TC_M, split = blockIdx.z;
    const int nkb = H / (kTileK * ksplit), kb0 = split * nkb;
    const bool conv = x16 != nullptr && blockIdx.y == 0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr int S = TC_STAGES;
    const uint32_t bar0 = base + TC_OFF_BAR;
    auto full = [&](int st) { return bar0 + 8u * st; };
    auto empty = [&](int st) { return bar0 + 8u * (S + st); };
    const uint32_t acc_full = bar0 + 8u * (2 * S);
    const uint32_t mma_done = acc_full + 8u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + TC_OFF_BAR + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + TC_OFF_BAR + 68);

    if (threadIdx.x == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(full(st), 1);
            mbar_init(empty(st), 1 + (conv ? 4 : 0));
        }
        mbar_init(acc_full, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(base + TC_OFF_BAR + 64, TC_N);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&]() {
        record_status(status, kStatusTimeout);
        *abort_flag = 1;
    };
    pdl_wait();  // the W_r parts (preceding kernel) and x
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int i = 0;
            for (; i < nkb; ++i) {
                const int st = i % S;
                if (*abort_flag || !mbar_wait(empty(st), ((i / S) & 1) ^ 1)) {
                    fail();
                    break;
                }
                const uint32_t dst = base + st * TC_STAGE_BYTES;
                const int kx = (kb0 + i) * kTileK;
                mbar_arrive_expect_tx(full(st), TC_STAGE_BYTES);
#pragma unroll
                for (int p = 0; p < 3; ++p)
                    tma_load_2d(dst + p * TC_TILE_BYTES, &tm_w, kx, p * E + e0, full(st));
                tma_load_2d(dst + 3 * TC_TILE_BYTES, &tm_x, kx, t0, full(st));
            }
            // the copies already issued land before the CTA can go away
            for (int j = (i > S ? i - S : 0); j < i; ++j) mbar_wait(full(j % S), (j / S) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        const uint32_t idesc = idesc_bf16_f32(TC_M, TC_N);
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            const int st = i % S;
            if (*abort_flag || !mbar_wait(full(st), (i / S) & 1)) {
                fail();
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t sb = base + st * TC_STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bdesc = sw128_kmajor_desc(sb + 3 * TC_TILE_BYTES + kk * 32);
#pragma unroll
                    for (int p = 0; p < 3; ++p)
                        mma_f16(tmem, sw128_kmajor_desc(sb + p * TC_TILE_BYTES + kk * 32), bdesc,
                                idesc, (i | kk | p) != 0);
                }
                mma_commit(empty(st));
            }
            __syncwarp();
        }
        if (ok && lane == 0) mma_commit(acc_full);
        // every MMA issued here completes before tensor memory is released
        if (lane == 0) {
            mma_commit(mma_done);
            mbar_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // --------------------------------------------- x16 copy, epilogue
        const int quad = warp % 4;
        bool ok = true;
        if (conv) {
            const int ct = (warp - 2) * 32 + lane;  // 0..127
            for (int i = 0; i < nkb && ok; ++i) {
                const int st = i % S;
                if (*abort_flag || !mbar_wait(full(st), (i / S) & 1)) {
                    fail();
                    ok = false;
                    break;
                }
                const uint8_t* xs = sbase + st * TC_STAGE_BYTES + 3 * TC_TILE_BYTES;
                const int kx = (kb0 + i) * kTileK;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int q = ct + 128 * u, r = q / 8, c = q % 8;
                    const uint4 v = *reinterpret_cast<const uint4*>(xs + r * 128 + ((c ^ (r & 7)) * 16));
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                    uint32_t h4[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        h4[j] = (uint32_t)float_to_half_bits_sat(__uint_as_float(w4[j] << 16)) |
                                ((uint32_t)float_to_half_bits_sat(__uint_as_float(w4[j] & 0xffff0000u)) << 16);
                    if (t0 + r < T)
                        *reinterpret_cast<uint4*>(x16 + (size_t)(t0 + r) * H + kx + c * 8) =
                            make_uint4(h4[0], h4[1], h4[2], h4[3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(st));
            }
        }
        const bool bad = !ok || *abort_flag || !mbar_wait(acc_full, 0);
        if (__any_sync(0xffffffffu, bad)) {  // tcgen05.ld below needs the whole warp
            fail();
        } else {
            tc_fence_after();
            const int e = e0 + quad * 32 + lane;
            float* out = parts + (size_t)split * T * E;
            for (int c0 = 0; c0 < TC_N && t0 + c0 < T; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (t0 + c0 + j < T && e < E) out[(size_t)(t0 + c0 + j) * E + e] = __uint_as_float(v[j]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TC_N);
}

bool use_tc_router(int T) { return T >= TC_MIN_T; }

// Slices of the hidden dimension: fewest waves x K-blocks per CTA, fewer
// slices on a tie.
int tc_ksplit(int T, int H, int E) {
    const int tiles = ((T + TC_N - 1) / TC_N) * ((E + TC_M - 1) / TC_M);
    int best = 1;
    long best_cost = -1;
    for (int ks = 1; ks <= 8; ks *= 2) {
        if (H % (kTileK * ks)) break;
        const long waves = (tiles * ks + TC_SMS - 1) / TC_SMS;
        const long cost = waves * (H / (kTileK * ks));
        if (best_cost < 0 || cost < best_cost) {
            best = ks;
            best_cost = cost;
        }
    }
    return best;
}
}  // namespace

int route_ksplit(int T, int H, int E) {
    if (use_tc_router(T)) return tc_ksplit(T, H, E);
    const int ctas = ((T + GT - 1) / GT) * ((E + GE - 1) / GE);
    int s = 1;
    while (s < 8 && ctas * s * 2 <= 2 * 152 && H % (GK * s * 2) == 0) s *= 2;
    return s;
}

size_t route_parts_floats(int T, int H, int E) { return (size_t)route_ksplit(T, H, E) * T * E; }

int tc_plane_rows(int E) { return 3 * E > TC_M ? 3 * E : TC_M; }

size_t route_planes_bytes(int T, int H, int E) {
    return use_tc_router(T) ? (size_t)tc_plane_rows(E) * H * 2 : 0;
}

cudaError_t launch_route_gemm(const uint16_t* x, const float* wr, int T, int H, int E, int k,
                              float* parts, float* logits, int32_t* idx, float* w, uint16_t* x16,
                              uint16_t* planes, int* status, int32_t* chunk_count,
                              int32_t* entry_rank, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    // the top-k over the K-slice parts; with chunk buffers it also counts
    // the bucketing's 32-token chunks
    auto topk = [&](int ks) {
        float* lg = parts == logits ? nullptr : logits;
        if (chunk_count && entry_rank)
            return launch_pdl(topk_chunk_kernel, dim3((T + 31) / 32), dim3(1024), 0, s,
                              (const float*)parts, ks, T, E, k, lg, idx, w, chunk_count,
                              entry_rank);
        return launch_pdl(topk_from_parts_kernel, dim3((T + 7) / 8), dim3(256), 0, s,
                          (const float*)parts, ks, T, E, k, lg, idx, w);
    };
    if (planes != nullptr && parts != logits && use_tc_router(T)) {
        const int ks = tc_ksplit(T, H, E);
        const int n4 = E * H / 4;
        cudaError_t err = launch_pdl(split_wr_kernel, dim3((n4 + 255) / 256), dim3(256), 0, s, wr,
                                     n4, planes);
        if (err != cudaSuccess) return err;
        CUtensorMap tm_w, tm_x;
        if (!encode_tmap_2d_f16(&tm_w, planes, (uint64_t)tc_plane_rows(E), H, kTileK, TC_M, true) ||
            !encode_tmap_2d_f16(&tm_x, x, T, H, kTileK, TC_N, true))
            return cudaErrorInvalidValue;
        err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   TC_SMEM);
        if (err != cudaSuccess) return err;
        const dim3 grid((T + TC_N - 1) / TC_N, (E + TC_M - 1) / TC_M, ks);
        err = launch_pdl(router_tc_kernel, grid, dim3(TC_THREADS), TC_SMEM, s, tm_w, tm_x, T, H, E,
                         ks, parts, x16, status);
        if (err != cudaSuccess) return err;
        return topk(ks);
    }
    // with the logits buffer as the only part, the sums are already in place
    const int ks = (parts == logits) ? 1 : route_ksplit(T, H, E);
    const dim3 grid((T + GT - 1) / GT, (E + GE - 1) / GE, ks);
    cudaError_t err = launch_pdl(router_gemm_kernel, grid, dim3(G_THREADS), 0, s, x, wr, T, H, E,
                                 ks, parts, x16);
    if (err != cudaSuccess) return err;
    return topk(ks);
}

// `logits` may be null; the split path is taken only when it is not.
cudaError_t launch_route(const uint16_t* x, const float* wr, int T, int H, int E, int k,
                         float* logits, int32_t* idx, float* w, uint16_t* x16, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (logits && !x16 && T > 32 && (H % GK) == 0)
        return launch_route_gemm(x, wr, T, H, E, k, logits, logits, idx, w, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, s);
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
