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
// One decode layer is two kernels chained with programmatic dependent launch
// (each is scheduled while its predecessor drains and waits for it with
// griddepcontrol.wait before touching its results):
//
//   prep     one CTA per router row.  Before the wait it stages its row of
//            W_r (one bulk copy; W_r does not depend on the preceding work).
//            After it: clears this call's synchronisation counters and, one
//            warp per token, forms the optional pre-norm of x (RMSNorm, the
//            same arithmetic and order as the prefill path), the row's logit
//            (fixed order: per lane over its columns, then a butterfly), and
//            - one CTA per token - the token's int8 codes of x per 32
//            columns with their scales.
//
//   layer    one CTA per SM, launched cooperatively (all CTAs resident: they
//            wait on one another's results).  Every CTA reads all T x E
//            logits and takes the same decisions itself: top-k and softmax
//            weights (one warp per token), the expert buckets (a token
//            bitmask per expert, a scan over experts).  CTA 0 stores the
//            routing results.  The packed weights of the touched experts are
//            cut into tasks of whole 4608-byte tiles - one 128-row block
//            times a range of 64-column blocks (the K range is split in
//            `nsg` / `nsd` parts so that there are enough tasks for every
//            SM) - and each CTA takes an equal contiguous share of the
//            gate/up tasks, then of the down tasks.  Two groups of eight
//            consumer warps take the tasks alternately (warp w of a group:
//            rows 16w..16w+15 of the block; a lane: one row and one 32-column
//            half of each tile).  Each group has its own ring of tile slots
//            and its own producer warp, which streams the group's tiles in
//            the order the group consumes them, one 1-D bulk copy (TMA) per
//            tile, up to a ring's worth of lanes at a time; at one token every
//            tile of the CTA's share is requested at once.  (One ring per
//            consumer sequence keeps the mbarrier phase protocol sound: every
//            waiter meets a slot's phases in order, the previous one already
//            seen.)  The consumers keep per-token fp32 row sums over the
//            task's K range:
//              gate/up  each task stores its K part of the row sums; the
//                       task that completes a 128-feature block of h (its
//                       gate and up blocks, every K part: a counter tells
//                       the last one) adds the parts in K order, forms
//                       h = silu(g) * u and its int8 codes per 32 features,
//                       stores them and counts the block done for the expert;
//              down     a task waits until every h block of its expert is
//                       done, loads h, and stores its K part of the
//                       weighted rows, routing weight * (W_d h); the task
//                       that completes a 128-column block of the output
//                       (every touched expert, every K part) adds, per
//                       token, the residual and the k slots' parts in slot
//                       and K order and writes the output columns.
//
// All sums run in a fixed order, so repeated calls give the same bits.  Every
// weight byte of a touched expert is read once, by one CTA.  Every wait is
// bounded; on expiry the kernel records MOE_ERR_TIMEOUT and stops issuing.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int kGroupWarps = 8;                          // 8 warps x 16 rows = one 128-row block
constexpr int kGroups = 2;                              // consumer groups, alternating tasks
constexpr int kConsumerWarps = kGroups * kGroupWarps;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kLayerThreads = kConsumerThreads + kGroups * 32;  // + a producer warp per group
constexpr int kWarpProducer0 = kConsumerWarps;          // group g's producer: warp kWarpProducer0 + g
constexpr int kSlotTiles = 4;                           // packed tiles per ring slot (one bulk copy),
                                                        // fewer when shared memory is short
constexpr int kMaxSlots = 32;                           // slots of both groups' rings
constexpr int kRingStride = kMaxSlots / 2;              // barrier and slot stride of a group's ring
constexpr int kRedBytes = kGroupWarps * 32 * 32;        // per group: 8 warps x 32 lanes x 8 floats
// Dynamic shared memory of the layer kernel: leaves room on the SM (228 KB)
// for its static part (13.1 KB) and a prep CTA of the next call (its router
// row, 8 KB at H = 2048) next to it.
constexpr int kLayerSmemBudget = 200 * 1024;
constexpr int kPrepThreads = 128;
constexpr int kMaxTk = MOE_DECODE_MAX_T * MOE_MAX_TOPK;
// Bucket rows of a unit of the clustered kernel, at most: a larger bucket is
// cut into slices (of 1, 2 or 4 rows at most, by T and the weight bits), so
// that the work split can spread one expert's tokens over several clusters.
constexpr int kSliceRows = 4;
constexpr int kMaxSlices = 16 * MOE_MAX_TOPK;  // slices of a launch (T <= 16)
// Tasks the K split aims for (gate/up and down alike): the split depends only
// on the number of touched experts and the shape, so results are
// reproducible.  A task keeps at least two tiles.
constexpr int kTargetTasks = 152 * 16;
constexpr int kMaxSplit = 16;
// Bytes of K-part sums the split may use (gate/up, down); beyond them the
// split is capped.
constexpr size_t kPartBudgetGU = 4u << 20;
constexpr size_t kPartBudgetD = 2u << 20;
// Cost of a tile in the work split, in units of one bucket row's group dot
// products: streaming it weighs as much as this many rows.
constexpr int kTileCost = 3;
// Routing ranks the logits with every thread when a token's E logits times
// its T x E elements need at most this many comparisons a thread.
constexpr int kRankCompares = 128;

struct PrepArgs {
    const uint16_t* x;
    const float* wr;
    int T, H, E, prenorm;
    float* logits;     // [T, E]
    uint8_t* xq;       // [T, H] int8 codes, dp4a order (below)
    int2* xs;          // [T, H/32] {fp32 bits of the scale, -8 * sum of the codes}
    int8_t* q_x;       // [T, H] the codes in column order (stage output)
    uint16_t* d_x;     // [T, H/32] fp16 scales (stage output)
    int* sync;         // counters of the layer kernel, cleared here
    int nsync;
    int* status;
};

struct LayerArgs {
    const uint16_t* x_res;  // the layer input (residual)
    const uint8_t* wgu;
    const uint8_t* wd;
    int T, H, I, E, k;
    const float* logits;
    const uint8_t* xq;
    const int2* xs;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* offsets;
    int32_t* touched;
    int32_t* counters;
    int32_t* bucket_token;
    int32_t* bucket_slot;
    float* gu_part;     // [nsg, T*k, 2I] K parts of the gate (0..I-1) and up (I..2I-1) sums
    int8_t* q_h;        // [T*k, I] stage output (column order), when write_qh
    uint16_t* d_h;      // [T*k, I/32]
    float* y_part;      // [nsd, T*k, H] K parts of the weighted expert outputs
    int* cnt_h;         // [nslot, I/128] stored gate/up K parts per h block
    int* cnt_y;         // [H/128] finished down tasks per output column block
    int cap_g, cap_d;   // upper bounds of the K splits (size of the part buffers)
    int ndiv_g, ndiv_d; // divisors of H/64 (resp. I/64) up to the cap, ascending
    int div_g[16], div_d[16];
    void* out;
    int out_fp32;
    int32_t* dots_gu;   // optional stage outputs
    int32_t* dots_d;
    int write_qh;
    int* status;
    // shared-memory plan (bytes from the dynamic base)
    int ns;             // slots of each group's ring
    int st;             // packed tiles per slot (kSlotTiles, or fewer for large T)
    int off_bar, off_ax, off_ah, ah_bytes, off_red;
    // clustered layer kernel: bytes of the rings and the K-part exchange
    // buffers (laid out in the kernel once the largest bucket is known),
    // and the groups' h buffers
    int ring_bytes, off_h, h_bytes;
};

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// dp4a order of an 8-column chunk of int8 activations (x0..x7 as bytes of
// a, b): the first word holds x0, x4, x1, x5 and the second x2, x6, x3, x7,
// matching the bytes that the masks 0x0F0F0F0F and (w >> 4) & 0x0F0F0F0F
// pick out of a packed code word (even columns in nibbles 0..3, odd columns
// in nibbles 4..7).
__device__ __forceinline__ uint2 permute_chunk(uint32_t a, uint32_t b) {
    return make_uint2(__byte_perm(a, b, 0x5140), __byte_perm(a, b, 0x7362));
}

// Group dot of one 32-code group (its words split into low and high nibbles)
// with one activation group in dp4a order; `init` is -8 * sum of the codes.
__device__ __forceinline__ int group_dot(const uint32_t (&wl)[4], const uint32_t (&wh)[4],
                                         const uint8_t* act, int init) {
    const uint4 a0 = *reinterpret_cast<const uint4*>(act);
    const uint4 a1 = *reinterpret_cast<const uint4*>(act + 16);
    int p = init, q = 0;  // two independent chains (exact integer sums in any order)
    p = dp4a_us(wl[0], a0.x, p);
    q = dp4a_us(wh[0], a0.y, q);
    p = dp4a_us(wl[1], a0.z, p);
    q = dp4a_us(wh[1], a0.w, q);
    p = dp4a_us(wl[2], a1.x, p);
    q = dp4a_us(wh[2], a1.y, q);
    p = dp4a_us(wl[3], a1.z, p);
    q = dp4a_us(wh[3], a1.w, q);
    return p + q;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// A lane's 32 codes of a tile row as words that pair with the activation
// words of group_dot: WB = 4, the low and the high nibbles of its four code
// words; WB = 8, the first and the second word of each of its four 8-code
// chunks (stored in the activations' order).
template <int WB>
__device__ __forceinline__ void unpack_codes(const uint8_t* p, uint32_t (&wl)[4], uint32_t (&wh)[4]) {
    if constexpr (WB == 8) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(p);
        const uint4 v1 = *reinterpret_cast<const uint4*>(p + 16);
        wl[0] = v0.x; wh[0] = v0.y; wl[1] = v0.z; wh[1] = v0.w;
        wl[2] = v1.x; wh[2] = v1.y; wl[3] = v1.z; wh[3] = v1.w;
    } else {
        const uint4 wv = *reinterpret_cast<const uint4*>(p);
        wl[0] = wv.x & 0x0F0F0F0Fu; wl[1] = wv.y & 0x0F0F0F0Fu;
        wl[2] = wv.z & 0x0F0F0F0Fu; wl[3] = wv.w & 0x0F0F0F0Fu;
        wh[0] = (wv.x >> 4) & 0x0F0F0F0Fu; wh[1] = (wv.y >> 4) & 0x0F0F0F0Fu;
        wh[2] = (wv.z >> 4) & 0x0F0F0F0Fu; wh[3] = (wv.w >> 4) & 0x0F0F0F0Fu;
    }
}

// Group dot of WB-bit codes with one activation group: WB = 4 as group_dot
// (codes 0..15, `init` = -8 * sum of the activations); WB = 8, signed codes
// times signed activations from 0.
template <int WB>
__device__ __forceinline__ int group_dot_w(const uint32_t (&wl)[4], const uint32_t (&wh)[4],
                                           const uint8_t* act, int init) {
    if constexpr (WB == 8) {
        const uint4 a0 = *reinterpret_cast<const uint4*>(act);
        const uint4 a1 = *reinterpret_cast<const uint4*>(act + 16);
        int p = 0, q = 0;
        p = dp4a_ss(wl[0], a0.x, p);
        q = dp4a_ss(wh[0], a0.y, q);
        p = dp4a_ss(wl[1], a0.z, p);
        q = dp4a_ss(wh[1], a0.w, q);
        p = dp4a_ss(wl[2], a1.x, p);
        q = dp4a_ss(wh[2], a1.y, q);
        p = dp4a_ss(wl[3], a1.z, p);
        q = dp4a_ss(wh[3], a1.w, q);
        return p + q;
    } else {
        return group_dot(wl, wh, act, init);
    }
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int N>
struct IntC {
    static constexpr int value = N;
};
template <bool B>
struct BoolC {
    static constexpr bool value = B;
};

}  // namespace

// Smallest divisor d of KB (d <= cap, d <= KB / 2 unless KB = 1) with
// units * d >= target; if there is none, the largest such divisor.
// Non-increasing in `units`.
__host__ __device__ inline int decode_split_for(int units, int KB, int target, int cap) {
    int best = 1;
    const int dmax = KB > 1 ? KB / 2 : 1;
    for (int d = 1; d <= dmax && d <= cap; ++d) {
        if (KB % d) continue;
        best = d;
        if ((long long)units * d >= target) return d;
    }
    return best;
}

namespace {

// ------------------------------------------------------------------ prep
// Each token has tpt = 128 >> ceil(log2 T) threads (4 <= tpt <= 128); thread
// `sub` of token t holds the 8-column units sub, sub + tpt, ... of its row,
// eight at a time.  Its partial sums (one per unit slot mod 8, in column
// order within a unit) are added in slot order, then across the token's
// threads by a butterfly (and across its warps in warp order, through
// shared memory, when tpt > 32).  mode 1: the norm, then router row e's
// logits; mode 2: the norm, then the int8 codes of block cb of the token
// groups (a quad of threads a 32-column group).  At most 80 registers a
// thread: next to a layer kernel of the previous call
// (576 threads x 96) the SM has 128 x 80 left, so the next layer's prep can
// stage its router row while that kernel runs.
constexpr int kPrepBatch = 8;  // units a thread loads at once

__device__ __forceinline__ void unpack8(const uint4 v, float (&xf)[8]) {
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        xf[2 * p] = __uint_as_float(wv[p] << 16);
        xf[2 * p + 1] = __uint_as_float(wv[p] & 0xffff0000u);
    }
}

constexpr int kPrepBarId = 4;  // named barrier of the row's 128 threads
constexpr int kRouteBarId = 5; // named barrier of the four warps routing one token
constexpr int kCombineBarId = 6;  // named barrier of the eight combine warps
enum { kRouteGeneral = 0, kRouteOneTokenFast = 1, kRouteOneTokenOnly = 2 };

// The prep work of one CTA on threads 0..127, for every token of x: the
// optional RMSNorm factor, then by `mode`
//   0: router row e's logit (row staged in shared memory at w) and the int8
//      codes of the 32-column groups g of token t with (t * H/32 + g) % nrow
//      == e (nrow: the number of router rows);
//   1: router row e's logit only;
//   2: the int8 codes of the groups cb*32 .. cb*32 + 31 in (token, group)
//      order, one quad of threads each (a CTA beside the logit CTAs).
// s_red: 4 floats, s_r: MOE_DECODE_MAX_T floats of shared memory.
__device__ __forceinline__ void prep_row(const PrepArgs& a, const uint16_t* x, int e, const float* w,
                                         float* s_red, float* s_r, int mode, int cb = 0) {
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int H = a.H, T = a.T;
    const int H8 = H / 8, G32 = H / kGroup;
    int tpt = kPrepThreads;
    while (tpt > 4 && kPrepThreads / tpt < T) tpt >>= 1;  // T <= 32
    const int t = tid / tpt, sub = tid % tpt;
    const bool act = t < T;
    const int nm = (H8 + tpt - 1) / tpt;  // unit slots of a thread (the last ones may be past the row)
    const uint16_t* xr = x + (size_t)(act ? t : 0) * H;
    uint4 v[kPrepBatch];
    auto load = [&](int m0) {
#pragma unroll
        for (int z = 0; z < kPrepBatch; ++z) {
            const int u = sub + tpt * (m0 + z);
            v[z] = act && m0 + z < nm && u < H8 ? __ldcg(reinterpret_cast<const uint4*>(xr) + u)
                                                : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // the sum over the token's threads: butterfly within the warp, then the
    // token's warps in order
    auto token_sum = [&](float x) -> float {
        for (int o = 1; o < 32 && o < tpt; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (tpt > 32) {
            named_sync(kPrepBarId, kPrepThreads);  // s_red is free
            if (lane == 0) s_red[warp] = x;
            named_sync(kPrepBarId, kPrepThreads);
            const int w0 = (t * tpt) / 32;
            x = 0.f;
            for (int q = 0; q < tpt / 32; ++q) x += s_red[w0 + q];
        }
        return x;
    };
    float r = 1.0f;
    const bool one_batch = nm <= kPrepBatch;
    if (a.prenorm) {
        // RMSNorm of the token, in fp32
        float ssu[kPrepBatch];
#pragma unroll
        for (int z = 0; z < kPrepBatch; ++z) ssu[z] = 0.f;
        for (int m0 = 0; m0 < nm; m0 += kPrepBatch) {
            load(m0);
#pragma unroll
            for (int z = 0; z < kPrepBatch; ++z) {
                if (m0 + z < nm) {  // (uniform)
                    float xf[8];
                    unpack8(v[z], xf);
#pragma unroll
                    for (int q = 0; q < 8; ++q) ssu[z] = fmaf(xf[q], xf[q], ssu[z]);
                }
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int z = 0; z < kPrepBatch; ++z) ss += ssu[z];
        ss = token_sum(ss);
        r = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, (float)H) + 1e-6f));
        if (act && sub == 0) s_r[t] = r;  // for the coding pass
    }
    if (mode != 2) {
    float accu[kPrepBatch];  // the logit's partial sums, one per unit slot
#pragma unroll
    for (int z = 0; z < kPrepBatch; ++z) accu[z] = 0.f;
    for (int m0 = 0; m0 < nm; m0 += kPrepBatch) {
        if (!(a.prenorm && one_batch)) load(m0);  // one batch: still held from the norm
#pragma unroll
        for (int z = 0; z < kPrepBatch; ++z) {
            if (m0 + z < nm) {  // (uniform)
                const int u = sub + tpt * (m0 + z);
                const bool valid = act && u < H8;
                float xf[8];
                unpack8(v[z], xf);
                if (a.prenorm) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) xf[q] = bf16_bits_to_float(float_to_bf16_bits(xf[q] * r));
                }
                if (valid) {
                    const float4 w0 = *reinterpret_cast<const float4*>(w + u * 8);
                    const float4 w1 = *reinterpret_cast<const float4*>(w + u * 8 + 4);
                    float acc = accu[z];
                    acc = fmaf(xf[0], w0.x, acc);
                    acc = fmaf(xf[1], w0.y, acc);
                    acc = fmaf(xf[2], w0.z, acc);
                    acc = fmaf(xf[3], w0.w, acc);
                    acc = fmaf(xf[4], w1.x, acc);
                    acc = fmaf(xf[5], w1.y, acc);
                    acc = fmaf(xf[6], w1.z, acc);
                    acc = fmaf(xf[7], w1.w, acc);
                    accu[z] = acc;
                }
            }
        }
    }
    float acc = 0.f;
#pragma unroll
    for (int z = 0; z < kPrepBatch; ++z) acc += accu[z];
    acc = token_sum(acc);
    if (act && sub == 0) a.logits[(size_t)t * a.E + e] = acc;
    }
    if (mode == 1) return;
    // mode 2: the int8 codes of block cb of the T * H/32 groups (32 groups,
    // one quad of threads each), from x and the token's norm factor again
    if (a.prenorm) named_sync(kPrepBarId, kPrepThreads);  // s_r is stored
    const int quad = tid / 4, ql = tid % 4;
    const unsigned qmask = 0xFu << (lane & ~3);
    const int fi = cb * (kPrepThreads / 4) + quad, t2 = fi / G32, g = fi - t2 * G32;
    if (t2 < T) {  // (uniform in the quad)
        const int u = g * 4 + ql;  // this lane's 8 columns
        float xf[8];
        unpack8(__ldcg(reinterpret_cast<const uint4*>(x + (size_t)t2 * H) + u), xf);
        if (a.prenorm) {
            const float r2 = s_r[t2];
#pragma unroll
            for (int q = 0; q < 8; ++q) xf[q] = bf16_bits_to_float(float_to_bf16_bits(xf[q] * r2));
        }
        float amax = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(xf[q]));
        amax = fmaxf(amax, __shfl_xor_sync(qmask, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(qmask, amax, 2));
        const uint16_t db = act_scale_bits(amax);
        const float d = half_bits_to_float(db);
        uint32_t lo = 0u, hi = 0u;
        int gsum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int qc = act_code(xf[q], d);
            gsum += qc;
            if (q < 4) lo |= ((uint32_t)qc & 0xffu) << (8 * q);
            else hi |= ((uint32_t)qc & 0xffu) << (8 * (q - 4));
        }
        gsum += __shfl_xor_sync(qmask, gsum, 1);
        gsum += __shfl_xor_sync(qmask, gsum, 2);
        *reinterpret_cast<uint2*>(a.xq + (size_t)t2 * H + u * 8) = permute_chunk(lo, hi);
        *reinterpret_cast<uint2*>(a.q_x + (size_t)t2 * H + u * 8) = make_uint2(lo, hi);
        if (ql == 0) {
            a.xs[t2 * G32 + g] = make_int2(__float_as_int(d), -8 * gsum);
            a.d_x[t2 * G32 + g] = db;
        }
    }
}

// CTAs 0..E-1: router row e (its logits); CTAs E..: blocks of 32 int8-coded
// groups of x.
__global__ void __maxnreg__(80) decode_prep_kernel(const PrepArgs a) {
    extern __shared__ __align__(128) uint8_t psm[];  // this CTA's router row [H] fp32
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ float s_red[kPrepThreads / 32];
    __shared__ float s_r[MOE_DECODE_MAX_T];
    const int tid = threadIdx.x, e = blockIdx.x, H = a.H;
    const bool coder = e >= a.E;
    const uint32_t bar = smem_u32(&s_bar);
    if (tid == 0 && !coder) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, (uint32_t)(H * 4));
        bulk_g2s(smem_u32(psm), a.wr + (size_t)e * H, (uint32_t)(H * 4), bar);
    }
    __syncthreads();
    pdl_wait();     // x and the workspace belong to this call from here on
    pdl_trigger();  // the layer kernel may be scheduled; it waits for our end
    for (int i = e * kPrepThreads + tid; i < a.nsync; i += gridDim.x * kPrepThreads) a.sync[i] = 0;
    if (coder) {
        prep_row(a, a.x, 0, nullptr, s_red, s_r, 2, e - a.E);
        return;
    }
    if (!mbar_wait(bar, 0)) record_status(a.status, kStatusTimeout);
    prep_row(a, a.x, e, reinterpret_cast<const float*>(psm), s_red, s_r, 1);
}

// ----------------------------------------------------------------- layer
// The first task of worker v of V when every touched slot has the same
// bucket size and there are no more runs (nruns, P consecutive tasks each)
// than workers: run r is shared by workers ceil(rV/nruns) ..
// ceil((r+1)V/nruns) - 1 (at least one), each taking an equal part of its
// tasks, so no worker's share crosses a run.
__device__ __forceinline__ int run_bound(int v, int V, int nruns, int P) {
    if (v >= V) return nruns * P;
    const int r = (int)((long long)v * nruns / V);
    const int w0 = (int)(((long long)r * V + nruns - 1) / nruns);
    const int w1 = (int)(((long long)(r + 1) * V + nruns - 1) / nruns);
    return r * P + (int)((long long)(v - w0) * P / (w1 - w0));
}

// The first task of worker v of V when the `per` tasks of touched slot i
// (KC tiles each) cost KC * (kTileCost + c_i) each, c_i = toff[i + 1] -
// toff[i] bucket rows: the task whose cost range holds the position
// floor(v * total / V).  Monotone in v; bound(0) = 0 and bound(V) = nt * per.
// The whole warp calls it: a ballot over the slots finds the one whose cost
// range holds the position (the prefixes rise with i), one division places
// the position within that slot.
__device__ __forceinline__ int split_bound_warp(int v, int V, int nt, int Tk, int per, int KC,
                                                const int* toff, int lane) {
    using u64 = unsigned long long;
    const u64 U = (u64)per * KC;  // tiles of a touched slot
    const u64 tot = U * ((u64)kTileCost * nt + Tk);
    const u64 vt = (u64)v * tot;  // V times the position
    // slots 0..nt whose prefix U * (kTileCost * i + toff[i]) <= the position
    int cnt = 0;
    for (int i0 = 0; i0 <= nt; i0 += 32) {
        const int i = i0 + lane;
        const bool le = i <= nt && (u64)V * U * ((u64)kTileCost * i + toff[i]) <= vt;
        cnt += __popc(__ballot_sync(0xffffffffu, le));
    }
    const int lo = cnt - 1;
    if (lo >= nt) return nt * per;
    // floor((position - prefix) / (KC * w)), w = kTileCost + c_lo, scaled by V
    const u64 num = vt - (u64)V * U * ((u64)kTileCost * lo + toff[lo]);
    const u64 den = (u64)V * KC * (kTileCost + toff[lo + 1] - toff[lo]);
    const u64 j = (num >> 32) == 0 && (den >> 32) == 0 ? (u64)((unsigned)num / (unsigned)den) : num / den;
    return lo * per + (int)(j < (u64)per ? j : (u64)per);
}

// The layer's shared state outside the dynamic plan.
struct LayerShared {
    int idx[kMaxTk];
    float w[kMaxTk];
    int btok[kMaxTk];    // bucket row -> token
    uint8_t bslot[kMaxTk];  // bucket row -> the token's choice (0 .. k-1)
    float bsw[kMaxTk];   // bucket row -> routing weight
    int slotpos[kMaxTk]; // (t, j) -> bucket row
    uint32_t mask[kMaxExperts];
    int off[kMaxExperts + 1];
    int touched[kMaxExperts];
    int toff[kMaxExperts + 1];  // touched slot -> its first bucket row (+ total)
    int slot_chunk[kMaxSlots];  // the latest chunk issued into each slot (both rings)
    const uint8_t* ctab_p[kGroups][32];  // producer: the next chunks' sources
    int ctab_n[kGroups][32];             // and sizes in tiles
    int nt, nsg, nsd;
    int eqc;                    // every touched slot has the same bucket size
    int bnd[kGroups][4];        // group g: gate/up tasks [0], [1]; down tasks [2], [3]
    int cmax;                   // clustered kernel: the largest slice
    int sto[kMaxSlices + 1];    // clustered kernel: slice -> its first bucket row (+ total)
    uint8_t sslot[kMaxSlices];  // clustered kernel: slice -> its touched slot
    int rns;                    // clustered kernel: slots of each group's ring
    volatile int abort;
    volatile int flag[kGroups];
};

// A thread's position in its group's ring (the chunk sequence continues
// from layer to layer within a launch).
struct Pipe {
    int slot, phase, cidx;
    int units;  // clustered kernel: units exchanged so far (the exchange barriers' phases)
    int armok;  // clustered kernel: the arming warp has met every phase in time
};

// What changes from layer to layer: the input (also the residual), the
// expert weights and the output.
struct LayerIO {
    const uint16_t* x_res;
    const uint8_t* wgu;
    const uint8_t* wd;
    void* out;
    int out_fp32;
};

// Full and empty barriers of slot s of group g's ring: kMaxSlots of each
// at off_bar, kRingStride a group, whatever number of slots a launch uses.
__device__ __forceinline__ uint32_t ring_bar(const LayerArgs& a, uint32_t sbase, bool full, int g, int s) {
    return sbase + a.off_bar + 8u * ((full ? 0 : kMaxSlots) + g * kRingStride + s);
}

// Once per launch: the ring barriers, no chunk issued yet, no failure.
__device__ __forceinline__ void ring_init(const LayerArgs& a, LayerShared& S, uint8_t* dsm) {
    const uint32_t sbase = smem_u32(dsm);
    if (threadIdx.x == 0) {
        for (int g = 0; g < kGroups; ++g) {
            for (int s = 0; s < kRingStride; ++s) {
                mbar_init(ring_bar(a, sbase, true, g, s), 1);
                mbar_init(ring_bar(a, sbase, false, g, s), kGroupWarps);
            }
        }
        S.abort = 0;
        fence_mbar_init();
    }
    for (int s = threadIdx.x; s < kMaxSlots; s += kLayerThreads) S.slot_chunk[s] = -1;
}

// Before the CTA exits, every copy it issued has landed: the producer warps
// wait for the latest chunk of each slot (earlier ones completed before it).
__device__ __forceinline__ void ring_drain(const LayerArgs& a, LayerShared& S, uint8_t* dsm, int ns) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp < kWarpProducer0) return;
    const int g = warp - kWarpProducer0;
    const uint32_t sbase = smem_u32(dsm);
    __syncwarp();
    for (int s = lane; s < ns; s += 32) {
        const int c = S.slot_chunk[g * kRingStride + s];
        if (c >= 0) mbar_wait(ring_bar(a, sbase, true, g, s), (c / ns) & 1);
    }
}

// Routing, taken by every CTA from the same logits: each token's top k
// (larger logit first, the lower expert index on a tie) with softmax weights
// over them, a token bitmask per expert, the buckets (a scan over experts),
// the K splits of the task kernel.  CTA 0 stores the routing results.  The
// logits and their order keys sit in the still idle dynamic shared memory
// below the codes of x.  split(warp, lane) runs on warps 0 .. 4*kGroups - 1
// (the work split of the caller) while the other warps fill the buckets.
// ROUTE: kRouteGeneral, kRouteOneTokenFast (a single token is routed by four
// warps instead) or kRouteOneTokenOnly (T == 1 always: only that path is
// built).
template <int ROUTE, typename Split>
__device__ __forceinline__ void route_layer(const LayerArgs& a, LayerShared& S, uint8_t* dsm,
                                            Split&& split) {
    constexpr bool ONE_TOKEN_PATH = ROUTE != kRouteGeneral;
    int* s_idx = S.idx;
    float* s_w = S.w;
    int* s_btok = S.btok;
    float* s_bsw = S.bsw;
    int* s_slotpos = S.slotpos;
    uint32_t* s_mask = S.mask;
    int* s_off = S.off;
    int* s_touched = S.touched;
    int* s_toff = S.toff;
    int& s_nt = S.nt;
    int& s_nsg = S.nsg;
    int& s_nsd = S.nsd;
    int& s_eqc = S.eqc;
    const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k;
    const int RBg = 2 * I / kTileRows, RBd = H / kTileRows;
    const int Tk = T * k;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const bool b0 = blockIdx.x == 0;  // CTA 0 stores the routing results
    if (ROUTE == kRouteOneTokenOnly || (ONE_TOKEN_PATH && T == 1)) {
        // One token: warps 0..3 (expert e on thread e % 128) rank every
        // expert's logit against all E (larger first, the lower index on a
        // tie: the order of the general path); rank < k places it.  Warp 0
        // then forms the softmax weights over the k choices exactly as the
        // general path, and each choice's bucket row (the choices of lower
        // index); every thread of the four warps forms the offsets of its
        // experts (the choices below them).
        if (warp < 4) {
            float* s_lg = reinterpret_cast<float*>(dsm);
            uint32_t* s_key = reinterpret_cast<uint32_t*>(s_lg + kMaxExperts);
            uint32_t mk[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int e = tid + 128 * r;
                const float v = e < E ? __ldcg(a.logits + e) : 0.f;
                mk[r] = float_order_key(v);
                if (e < E) {
                    s_lg[e] = v;
                    s_key[e] = mk[r];
                } else if (e < ((E + 3) & ~3)) {
                    s_key[e] = 0u;  // padding: never greater, never ranked before e < E
                }
            }
            named_sync(kRouteBarId, 128);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int e = tid + 128 * r;
                if (e < E) {
                    int rank = 0;
                    for (int q = 0; q < E; q += 4) {
                        const uint4 kq = *reinterpret_cast<const uint4*>(s_key + q);
                        rank += (kq.x > mk[r] || (kq.x == mk[r] && q < e)) ? 1 : 0;
                        rank += (kq.y > mk[r] || (kq.y == mk[r] && q + 1 < e)) ? 1 : 0;
                        rank += (kq.z > mk[r] || (kq.z == mk[r] && q + 2 < e)) ? 1 : 0;
                        rank += (kq.w > mk[r] || (kq.w == mk[r] && q + 3 < e)) ? 1 : 0;
                    }
                    if (rank < k) s_idx[rank] = e;
                }
            }
            named_sync(kRouteBarId, 128);
            if (warp == 0) {
                const int si = lane < k ? s_idx[lane] : 0;
                const float v = lane < k ? s_lg[si] : 0.f;
                const float m = __shfl_sync(0xffffffffu, v, 0);  // the largest
                const float z = lane < k ? expf(v - m) : 0.f;
                const float zs = warp_sum(z);
                int pos = 0;  // choice j's bucket row: the choices of lower index
                for (int q = 0; q < k; ++q) pos += __shfl_sync(0xffffffffu, si, q) < si ? 1 : 0;
                if (lane < k) {
                    const float sw = z / zs;
                    s_w[lane] = sw;
                    s_slotpos[lane] = pos;
                    s_btok[pos] = 0;
                    S.bslot[pos] = lane;
                    s_bsw[pos] = sw;
                    s_touched[pos] = si;
                    s_toff[pos] = pos;
                    if (b0) {
                        a.topk_idx[lane] = si;
                        a.topk_w[lane] = sw;
                        a.bucket_token[pos] = 0;
                        a.bucket_slot[pos] = lane;
                        a.touched[pos] = si;
                    }
                }
                if (lane == 0) {
                    s_off[E] = k;
                    s_toff[k] = k;
                    s_nt = k;
                    s_eqc = 1;
                    if (b0) {
                        a.offsets[E] = k;
                        a.counters[kCntTouched] = k;
                    }
                }
            }
            for (int e = tid; e < E; e += 128) {
                int c = 0;
                for (int q = 0; q < k; ++q) c += s_idx[q] < e ? 1 : 0;
                s_off[e] = c;
                if (b0) a.offsets[e] = c;
            }
        }
        __syncthreads();
        if (warp < 4 * kGroups) split(warp, lane);
        fence_proxy_async_smem();
        __syncthreads();
        return;
    }
    if constexpr (ROUTE != kRouteOneTokenOnly) {
    float* s_lg = reinterpret_cast<float*>(dsm);                  // [T][E] logits, and
    uint32_t* s_key = reinterpret_cast<uint32_t*>(s_lg + T * E);  // their order keys, in
    for (int i = tid; i < T * E; i += kLayerThreads) {            // the still idle ring
        const float v = __ldcg(a.logits + i);
        s_lg[i] = v;
        s_key[i] = float_order_key(v);
    }
    for (int e = tid; e < E; e += kLayerThreads) s_mask[e] = 0u;
    __syncthreads();
    // a warp a token (warp_topk) while every token has its warp; beyond
    // that, few experts: every thread ranks elements
    const bool rank_path = T > kConsumerWarps && T * E <= kLayerThreads &&
                           (long long)T * E * E <= (long long)kLayerThreads * kRankCompares;
    if (rank_path) {
        // every thread ranks (t, e) against a share of the token's keys
        // (nsub threads an element, interleaved; every element has a
        // thread), the shares are added; rank < k places e in t's choices
        int nsub = 1;
        while (nsub < 32 && T * E * 2 * nsub <= kLayerThreads) nsub *= 2;
        const int el = tid / nsub, sub = tid % nsub;
        const bool mine = el < T * E;
        const int t = mine ? el / E : 0, e = mine ? el - t * E : 0;
        int rank = 0;
        if (mine) {
            const uint32_t* kr = s_key + t * E;
            const uint32_t mk = kr[e];
            for (int q = sub; q < E; q += nsub) {
                const uint32_t kq = kr[q];
                rank += (kq > mk || (kq == mk && q < e)) ? 1 : 0;
            }
        }
        for (int o = 1; o < nsub; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (mine && sub == 0 && rank < k) {
            s_idx[t * k + rank] = e;
            atomicOr(&s_mask[e], 1u << t);
        }
    } else if (warp < kConsumerWarps) {
        // the choices, their softmax weights and token t's bit in the mask
        // of each expert it chose (T <= 32)
        for (int t = warp; t < T; t += kConsumerWarps) {
            int si;
            float sw;
            warp_topk(s_lg + t * E, E, k, si, sw);
            if (lane < k) {
                s_idx[t * k + lane] = si;
                s_w[t * k + lane] = sw;
                atomicOr(&s_mask[si], 1u << t);
            }
        }
    }
    __syncthreads();
    if (warp < kConsumerWarps) {
        // the softmax weights over each token's k choices (the rank path)
        for (int t = warp; t < T && rank_path; t += kConsumerWarps) {
            const float v = lane < k ? s_lg[t * E + s_idx[t * k + lane]] : 0.f;
            const float m = __shfl_sync(0xffffffffu, v, 0);  // the largest
            const float z = lane < k ? expf(v - m) : 0.f;
            const float zs = warp_sum(z);
            if (lane < k) s_w[t * k + lane] = z / zs;
        }
    } else if (warp == kWarpProducer0) {
        // experts 8*lane .. 8*lane+7 (E <= 256): bucket offsets, the touched
        // list (ascending expert order) and its offsets by a warp scan; the
        // K splits
        int cnt[8], tot = 0, tch = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = 8 * lane + i;
            cnt[i] = e < E ? __popc(s_mask[e]) : 0;
            tot += cnt[i];
            tch += cnt[i] > 0 ? 1 : 0;
        }
        int itot = tot, itch = tch;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a1 = __shfl_up_sync(0xffffffffu, itot, o);
            const int a2 = __shfl_up_sync(0xffffffffu, itch, o);
            if (lane >= o) {
                itot += a1;
                itch += a2;
            }
        }
        int off = itot - tot, pos = itch - tch;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = 8 * lane + i;
            if (e < E) {
                s_off[e] = off;
                if (cnt[i] > 0) {
                    s_toff[pos] = off;
                    s_touched[pos++] = e;
                }
                off += cnt[i];
            }
        }
        const int nt_ = __shfl_sync(0xffffffffu, itch, 31);
        // K splits: the smallest divisor of the row's 64-column blocks (listed
        // by the host, ascending, within the caps) that gives enough tasks,
        // else the largest
        const unsigned okg = __ballot_sync(
            0xffffffffu, lane < a.ndiv_g && nt_ * RBg * a.div_g[lane < a.ndiv_g ? lane : 0] >= kTargetTasks);
        const unsigned okd = __ballot_sync(
            0xffffffffu, lane < a.ndiv_d && nt_ * RBd * a.div_d[lane < a.ndiv_d ? lane : 0] >= kTargetTasks);
        const int ceq = Tk / nt_;  // every bucket of this size?
        bool eq_l = Tk % nt_ == 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) eq_l = eq_l && (cnt[i] == 0 || cnt[i] == ceq);
        const bool eqc = __all_sync(0xffffffffu, eq_l);
        if (lane == 31) {
            s_off[E] = itot;
            s_nt = itch;
            s_toff[itch] = itot;
            s_nsg = okg ? a.div_g[__ffs(okg) - 1] : a.div_g[a.ndiv_g - 1];
            s_nsd = okd ? a.div_d[__ffs(okd) - 1] : a.div_d[a.ndiv_d - 1];
            s_eqc = eqc ? 1 : 0;
        }
    }
    __syncthreads();
    const int nt = s_nt;
    if (warp < 4 * kGroups) {
        split(warp, lane);
    } else {
        const int tid2 = tid - 4 * kGroups * 32, nthr2 = kLayerThreads - 4 * kGroups * 32;
        for (int p = tid2; p < Tk; p += nthr2) {
            const int t = p / k, e = s_idx[p];
            const int pos = s_off[e] + __popc(s_mask[e] & ((1u << t) - 1u));
            s_btok[pos] = t;
            S.bslot[pos] = p % k;
            s_bsw[pos] = s_w[p];
            s_slotpos[p] = pos;
            if (b0) {
                a.topk_idx[p] = e;
                a.topk_w[p] = s_w[p];
                a.bucket_token[pos] = t;
                a.bucket_slot[pos] = p % k;
            }
        }
        if (b0) {
            for (int i = tid2; i <= E; i += nthr2) a.offsets[i] = s_off[i];
            for (int i = tid2; i < nt; i += nthr2) a.touched[i] = s_touched[i];
            if (tid2 == 0) a.counters[kCntTouched] = nt;
        }
    }
    // the logits were held through generic accesses; bulk copies refill
    // that memory
    fence_proxy_async_smem();
    __syncthreads();
    }
}

// One decode layer (everything after the prep kernel's work) by one CTA of
// the cooperative grid.  MAXNT: the most tokens an expert's bucket may hold
// (T <= MAXNT).  DOTS: also store every int32 group dot (stage outputs; the
// variant that does not is the one calls run without them).
template <int MAXNT, bool DOTS>
__device__ __forceinline__ void layer_body(const LayerArgs& a, const LayerIO& io, LayerShared& S,
                                           uint8_t* dsm, Pipe& pp) {
    int* s_btok = S.btok;
    float* s_bsw = S.bsw;
    int* s_slotpos = S.slotpos;
    int* s_off = S.off;
    int* s_touched = S.touched;
    int* s_toff = S.toff;
    int* s_slot_chunk = S.slot_chunk;
    int& s_nt = S.nt;
    int& s_nsg = S.nsg;
    int& s_nsd = S.nsd;
    int& s_eqc = S.eqc;
    auto& s_bnd = S.bnd;
    volatile int& s_abort = S.abort;
    volatile int* s_flag = S.flag;

    const int T = a.T, H = a.H, I = a.I, k = a.k;
    const int KBg = H / kTileK, KBd = I / kTileK;
    const int RBg = 2 * I / kTileRows, RBd = H / kTileRows, RBh = I / kTileRows;
    const int Gx = H / kGroup, Gh = I / kGroup;
    const int Tk = T * k, ns = a.ns;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int G = gridDim.x, b = blockIdx.x;
    const uint32_t sbase = smem_u32(dsm);
    // group g's ring: slots g*ns .. g*ns + ns - 1
    auto full_bar = [&](int g, int s) { return ring_bar(a, sbase, true, g, s); };
    auto empty_bar = [&](int g, int s) { return ring_bar(a, sbase, false, g, s); };
    const int st = a.st;
    auto slot_addr = [&](int g, int s) { return (uint32_t)((g * ns + s) * st * kTileBytes); };
    auto fail = [&]() {
        record_status(a.status, kStatusTimeout);
        s_abort = 1;
    };
    if (warp < kConsumerWarps) {
        // the int8 codes of x and their scales (written by the prep kernel)
        // start on their way to shared memory while the CTA routes
        const int n16 = (T * H + T * Gx * 8) / 16;
        const uint8_t* src = a.xq;
        for (int i = tid; i < n16; i += kConsumerThreads)
            cp_async16(sbase + a.off_ax + 16 * i, src + 16 * (size_t)i);
    }

    // ---------------------------------------------- routing (every CTA)
    route_layer<kRouteGeneral>(a, S, dsm, [&](int warp, int lane) {
        // Tasks are shared out by cost, a tile of touched slot i weighing
        // kTileCost + c_i: worker v = 2b + g (consumer group g of CTA b)
        // runs the gate/up tasks [bound(v), bound(v + 1)) and the down tasks
        // likewise.  With equal buckets and no more runs (gate/up: slot and
        // row block; down: slot and K part) than workers, the shares follow
        // the runs instead (run_bound).  Warp 4g + j finds group g's bound j.
        const int nt = s_nt;
        const int g = warp >> 2, j = warp & 3;
        const bool gu = j < 2;
        const int nsg_ = s_nsg, nsd_ = s_nsd;
        const int per = gu ? RBg * nsg_ : RBd * nsd_;
        const int KC = gu ? KBg / nsg_ : KBd / nsd_;
        const int nruns = gu ? nt * RBg : nt * nsd_, P = gu ? nsg_ : RBd;
        const int v = 2 * b + g + (j & 1);
        const int bnd = s_eqc && nruns <= 2 * G ? run_bound(v, 2 * G, nruns, P)
                                                 : split_bound_warp(v, 2 * G, nt, Tk, per, KC, s_toff, lane);
        if (lane == 0) s_bnd[g][j] = bnd;
    });
    const int nt = s_nt;

    // ------------------------------------------------------- work split
    const int nsg = s_nsg, nsd = s_nsd;
    const int KCg = KBg / nsg, KCd = KBd / nsd;
    const int per_g = RBg * nsg, per_d = RBd * nsd;  // tasks of a touched slot

    // A walk over one group's tasks in order: gate/up tasks (expert slot i,
    // row block rb, K part kc: kc fastest), then down tasks (i, K part kc,
    // row block rb: rb fastest, so that a run of down tasks shares its h),
    // advanced by counting (no division per step).
    struct Walk {
        int left_g, left_d;  // tasks left in each phase
        int i, rb, kc;       // the current task
        bool gu;
    };
    auto walk_down_at = [&](Walk& w, int t) {
        w.gu = false;
        w.i = t / per_d;
        const int r = t - w.i * per_d;
        w.kc = r / RBd;
        w.rb = r - w.kc * RBd;
    };
    auto walk_start = [&](int g) {
        Walk w;
        w.left_g = s_bnd[g][1] - s_bnd[g][0];
        w.left_d = s_bnd[g][3] - s_bnd[g][2];
        if (w.left_g > 0) {
            w.gu = true;
            const int t = s_bnd[g][0];
            w.i = t / per_g;
            const int r = t - w.i * per_g;
            w.rb = r / nsg;
            w.kc = r - w.rb * nsg;
        } else {
            walk_down_at(w, s_bnd[g][2]);
        }
        return w;
    };
    auto walk_next = [&](Walk w, int g) {
        if (w.gu) {
            if (--w.left_g > 0) {
                if (++w.kc == nsg) { w.kc = 0; if (++w.rb == RBg) { w.rb = 0; ++w.i; } }
            } else if (w.left_d > 0) {  // on to the group's first down task
                walk_down_at(w, s_bnd[g][2]);
            }
        } else {
            --w.left_d;
            if (++w.rb == RBd) { w.rb = 0; if (++w.kc == nsd) { w.kc = 0; ++w.i; } }
        }
        return w;
    };
    auto walk_live = [&](const Walk& w) { return w.gu ? w.left_g > 0 : w.left_d > 0; };

    // Chunks: each task's tiles are cut into runs of up to st tiles (one bulk
    // copy, one ring slot each), chunk after chunk in the group's task order.
    // Producer and consumers walk the same chunks; slot and phase advance by
    // counting.
    if (warp >= kWarpProducer0) {
        // ---------------------------------------------------------- producer
        // The group's chunks, 32 at a time: each lane finds one chunk's
        // source from its index (task = index / chunks a task, in the walk's
        // order), then lane 0 issues them in order; chunk c's slot held
        // chunk c - ns, issued before it, so a parity wait never aliases.
        const int g = warp - kWarpProducer0;
        const int ngu = s_bnd[g][1] - s_bnd[g][0], ndn = s_bnd[g][3] - s_bnd[g][2];
        const int cptg = (KCg + st - 1) / st, cptd = (KCd + st - 1) / st;  // chunks a task
        const int nch = ngu * cptg + ndn * cptd;
        bool ok = !s_abort;
        for (int c0 = 0; c0 < nch && ok; c0 += 32) {
            const int c = c0 + lane;
            if (c < nch) {
                const uint8_t* src;
                int n;
                if (c < ngu * cptg) {
                    const int tl = c / cptg, u0 = (c - tl * cptg) * st;
                    const int t = s_bnd[g][0] + tl;
                    const int i = t / per_g, r = t - i * per_g, rb = r / nsg, kc = r - rb * nsg;
                    src = io.wgu + (((size_t)s_touched[i] * RBg + rb) * KBg + (size_t)kc * KCg + u0) * kTileBytes;
                    n = KCg - u0 < st ? KCg - u0 : st;
                } else {
                    const int c2 = c - ngu * cptg, tl = c2 / cptd, u0 = (c2 - tl * cptd) * st;
                    const int t = s_bnd[g][2] + tl;
                    const int i = t / per_d, r = t - i * per_d, kc = r / RBd, rb = r - kc * RBd;
                    src = io.wd + (((size_t)s_touched[i] * RBd + rb) * KBd + (size_t)kc * KCd + u0) * kTileBytes;
                    n = KCd - u0 < st ? KCd - u0 : st;
                }
                S.ctab_p[g][lane] = src;
                S.ctab_n[g][lane] = n;
            }
            __syncwarp();
            if (lane == 0) {
                int& slot = pp.slot;
                int& phase = pp.phase;
                int& cidx = pp.cidx;
                const int m = nch - c0 < 32 ? nch - c0 : 32;
                for (int j = 0; j < m; ++j) {
                    ++cidx;
                    if (++slot == ns) {
                        slot = 0;
                        phase ^= 1;
                    }
                    // (the first ns chunks of the launch go to slots never used)
                    if (s_abort || (cidx >= ns && !mbar_wait(empty_bar(g, slot), phase ^ 1)) || s_abort) {
                        fail();
                        ok = false;
                        break;
                    }
                    const uint32_t bytes = (uint32_t)(S.ctab_n[g][j] * kTileBytes);
                    s_slot_chunk[g * kRingStride + slot] = cidx;
                    mbar_arrive_expect_tx(full_bar(g, slot), bytes);
                    bulk_g2s(sbase + slot_addr(g, slot), S.ctab_p[g][j], bytes, full_bar(g, slot));
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);  // (the table is rewritten next round)
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int grp = warp / kGroupWarps, w8 = warp % kGroupWarps;
    const int gtid = tid - grp * kGroupThreads;
    auto group_sync = [&]() { named_sync(2 + grp, kGroupThreads); };
    uint8_t* ax_q = dsm + a.off_ax;                                          // [T][H]
    const int2* ax_s = reinterpret_cast<const int2*>(ax_q + (size_t)T * H);  // [T][Gx]
    uint8_t* ah_q = dsm + a.off_ah + grp * a.ah_bytes;                       // [c][I]
    int2* ah_s = reinterpret_cast<int2*>(ah_q + (size_t)T * I);              // [c][Gh]
    uint8_t* red_buf = dsm + a.off_red + grp * kRedBytes;                     // K-part sums of h
    cp_async_wait_all();  // this thread's copies of the codes of x
    named_sync(1, kConsumerThreads);
    // Control flow must stay uniform within a group (it shares named
    // barriers): a failed wait only skips work; decisions the group shares
    // are taken by its thread 0 and read after a group barrier.
    bool live = !s_abort;  // this warp has not given up
    int& slot = pp.slot;   // the current chunk's slot (same walk as the producer)
    int& phase = pp.phase;
    const int r_lane = lane >> 1, h_lane = lane & 1;
    const int lrow = w8 * 16 + r_lane;  // this lane's row in the 128-row block

    // One run: the group's consecutive tasks of touched slot i that share a
    // row block (gate/up: so one h block) or a K part (down: so one h
    // range), from w on; returns the number of tasks and leaves w at the
    // next one.  Bucket rows off .. off + c - 1 (NT >= c).  A task is rows
    // rb*128 + lrow and the K part's KC 64-column blocks; its tiles arrive
    // in chunks of up to st tiles.  At its end the lane pair's sum for bucket
    // row off + n is stored in the K part's slot (down: times the row's
    // routing weight).  GU: gate/up (activations x, bucket row -> token) or
    // down (activations h, one row per bucket row).
    auto run_tasks = [&](auto ntc, auto guc, int off, int c, Walk& w) -> int {
        constexpr int NT = decltype(ntc)::value;
        constexpr bool GU = decltype(guc)::value;
        const uint8_t* aq = GU ? ax_q : ah_q;
        const int2* as = GU ? ax_s : ah_s;
        const int K = GU ? H : I, Gk = GU ? Gx : Gh, KC = GU ? KCg : KCd;
        int32_t* dots = DOTS ? (GU ? a.dots_gu : a.dots_d) : nullptr;
        const size_t dots_ld = GU ? (size_t)2 * I : (size_t)H;
        const size_t ld = GU ? (size_t)2 * I : (size_t)H;
        const int code_off = w8 * 512 + lane * 16;                  // this lane's 16 code bytes
        const int scale_off = kTileCodeBytes + w8 * 64 + lane * 2;  // and its group's scale
        const int i = w.i;
        // the bucket rows' activation rows and scale rows (fixed for the run;
        // held in registers for small buckets)
        constexpr int NH = NT <= 4 ? NT : 1;
        int arow[NH], srow[NH];
#pragma unroll
        for (int n = 0; n < NH; ++n) {
            const int ar = GU ? s_btok[off + (n < c ? n : 0)] : n;
            arow[n] = ar * K;
            srow[n] = ar * Gk;
        }
        int ntask = 0;
        while (true) {
            const int rb = w.rb, kc = w.kc, kb0 = kc * KC, row = rb * kTileRows + lrow;
            float acc[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[n] = 0.f;
            for (int u0 = 0; u0 < KC; u0 += st) {
                const int nu = KC - u0 < st ? KC - u0 : st;
                if (++slot == ns) {
                    slot = 0;
                    phase ^= 1;
                }
                if (live && (s_abort || !mbar_wait(full_bar(grp, slot), phase))) {
                    fail();
                    live = false;
                }
                const uint8_t* chunk = dsm + slot_addr(grp, slot);
                if (live) {
                    for (int uu = 0; uu < nu; ++uu) {
                        const uint8_t* tile = chunk + uu * kTileBytes;
                        const uint4 wv = *reinterpret_cast<const uint4*>(tile + code_off);
                        const float dw =
                            half_bits_to_float(*reinterpret_cast<const uint16_t*>(tile + scale_off));
                        const uint32_t wl[4] = {wv.x & 0x0F0F0F0Fu, wv.y & 0x0F0F0F0Fu, wv.z & 0x0F0F0F0Fu,
                                                wv.w & 0x0F0F0F0Fu};
                        const uint32_t wh[4] = {(wv.x >> 4) & 0x0F0F0F0Fu, (wv.y >> 4) & 0x0F0F0F0Fu,
                                                (wv.z >> 4) & 0x0F0F0F0Fu, (wv.w >> 4) & 0x0F0F0F0Fu};
                        const int g = 2 * (kb0 + u0 + uu) + h_lane;
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            if (n < c) {
                                int ao, so;
                                if constexpr (NT <= 4) {
                                    ao = arow[n];
                                    so = srow[n];
                                } else {
                                    const int ar = GU ? s_btok[off + n] : n;
                                    ao = ar * K;
                                    so = ar * Gk;
                                }
                                const int2 sc = as[so + g];
                                const int dot = group_dot(wl, wh, aq + ao + g * kGroup, sc.y);
                                acc[n] = fmaf((float)dot, dw * __int_as_float(sc.x), acc[n]);
                                if (DOTS) dots[((size_t)(off + n) * dots_ld + row) * Gk + g] = dot;
                            }
                        }
                    }
                }
                // the chunk's slot is free again
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(grp, slot));
            }
            float* dst = (GU ? a.gu_part + ((size_t)kc * Tk + off) * 2 * I
                             : a.y_part + ((size_t)kc * Tk + off) * H) + row;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const float v = acc[n] + __shfl_xor_sync(0xffffffffu, acc[n], 1);
                if (n < c && h_lane == 0 && live) dst[n * ld] = GU ? v : v * s_bsw[off + n];
            }
            ++ntask;
            const Walk nx = walk_next(w, grp);
            const bool more = walk_live(nx) && nx.gu == GU && nx.i == i && (GU ? nx.rb == rb : nx.kc == kc);
            w = nx;
            if (!more) return ntask;
        }
    };
    auto dispatch = [&](auto guc, int off, int c, Walk& w) -> int {
        if (c <= 1) return run_tasks(IntC<1>{}, guc, off, c, w);
        if (c <= 2) return run_tasks(IntC<2>{}, guc, off, c, w);
        if (c <= 4) return run_tasks(IntC<4>{}, guc, off, c, w);
        if (c <= 8) return run_tasks(IntC<8>{}, guc, off, c, w);
        if (MAXNT <= 16 || c <= 16) return run_tasks(IntC<16>{}, guc, off, c, w);
        return run_tasks(IntC<MAXNT>{}, guc, off, c, w);
    };
    // The h of a run of down tasks, from the gate/up K parts of its expert:
    // features f0 .. f0 + nf - 1 of bucket rows off .. off + c - 1, into this
    // group's buffer (int8 codes in dp4a order, {scale, -8 * sum} per 32).
    // The group's warps split the K parts into ps subsets (as many as still
    // cover every feature quad in one pass) and the quads; a lane keeps two
    // K parts in flight, the subsets' sums meet in shared memory and are
    // added in subset order.
    auto compute_h = [&](int off, int c, int f0, int nf, int nsg_, bool store) {
        const int nq4 = c * nf / 4, q4_per_tok = nf / 4;
        int ps = 1;
        while (ps < kGroupWarps && 2 * ps <= nsg_ && 32 * (kGroupWarps / (2 * ps)) >= nq4) ps *= 2;
        const int sub = w8 % ps, blk = w8 / ps, nblk = kGroupWarps / ps;
        float4* red = reinterpret_cast<float4*>(red_buf);  // [8 warps][32 lanes][2]
        for (int qb = 0; qb < nq4; qb += 32 * nblk) {
            const int quad = qb + blk * 32 + lane;
            const bool ok = quad < nq4;
            const int n = ok ? quad / q4_per_tok : 0, f = f0 + (ok ? quad % q4_per_tok : 0) * 4;
            float gv[4] = {0.f, 0.f, 0.f, 0.f}, uv[4] = {0.f, 0.f, 0.f, 0.f};
            if (ok) {
                for (int p0 = sub; p0 < nsg_; p0 += 2 * ps) {
                    float4 g4[2], u4[2];
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const int p = p0 + z * ps;
                        if (p < nsg_) {
                            const float* src = a.gu_part + ((size_t)p * Tk + off + n) * 2 * I + f;
                            g4[z] = __ldcg(reinterpret_cast<const float4*>(src));
                            u4[z] = __ldcg(reinterpret_cast<const float4*>(src + I));
                        }
                    }
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        if (p0 + z * ps < nsg_) {
                            gv[0] += g4[z].x; gv[1] += g4[z].y; gv[2] += g4[z].z; gv[3] += g4[z].w;
                            uv[0] += u4[z].x; uv[1] += u4[z].y; uv[2] += u4[z].z; uv[3] += u4[z].w;
                        }
                    }
                }
            }
            if (ps > 1) {
                red[(w8 * 32 + lane) * 2] = make_float4(gv[0], gv[1], gv[2], gv[3]);
                red[(w8 * 32 + lane) * 2 + 1] = make_float4(uv[0], uv[1], uv[2], uv[3]);
                group_sync();
            }
            if (sub == 0) {  // whole warps: the first warp of each quad block
                if (ps > 1) {
#pragma unroll
                    for (int z = 0; z < 4; ++z) gv[z] = uv[z] = 0.f;
                    for (int s = 0; s < ps; ++s) {
                        const float4 g4 = red[((w8 + s) * 32 + lane) * 2];
                        const float4 u4 = red[((w8 + s) * 32 + lane) * 2 + 1];
                        gv[0] += g4.x; gv[1] += g4.y; gv[2] += g4.z; gv[3] += g4.w;
                        uv[0] += u4.x; uv[1] += u4.y; uv[2] += u4.z; uv[3] += u4.w;
                    }
                }
                // h = silu(g) * u; eight lanes hold one 32-feature group
                float h[4], amax = 0.f;
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    h[z] = gv[z] / (1.0f + __expf(-gv[z])) * uv[z];
                    amax = fmaxf(amax, fabsf(h[z]));
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const uint16_t db = act_scale_bits(amax);
                const float d = half_bits_to_float(db);
                uint32_t w4 = 0u;
                int sum = 0;
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    const int qv = act_code(h[z], d);
                    sum += qv;
                    w4 |= ((uint32_t)qv & 0xffu) << (8 * z);
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                // lanes 2m and 2m+1 hold columns 8m..8m+3 and 8m+4..8m+7 of
                // the group: the even lane stores the chunk in dp4a order
                const uint32_t w4o = __shfl_xor_sync(0xffffffffu, w4, 1);
                if (ok) {
                    if ((lane & 1) == 0)
                        *reinterpret_cast<uint2*>(ah_q + (size_t)n * I + f) = permute_chunk(w4, w4o);
                    if ((lane & 7) == 0) ah_s[n * Gh + f / kGroup] = make_int2(__float_as_int(d), -8 * sum);
                    if (store) {
                        const size_t prow = (size_t)(off + n);
                        *reinterpret_cast<uint32_t*>(a.q_h + prow * I + f) = w4;
                        if ((lane & 7) == 0) a.d_h[prow * Gh + f / kGroup] = db;
                    }
                }
            }
            if (ps > 1) group_sync();  // the sums buffer is reused
        }
    };

    // Items it0 .. it1 - 1 (item = token * 128 + column) of output columns
    // rbd*128 .. +127, once every down task of the block is stored: residual
    // plus every slot's parts, slots in order, K parts in order.  sp threads
    // share an item when the piece has fewer items than the group has
    // threads; each takes a contiguous range of the parts (the first also
    // the residual), loading eight at a time, and the ranges' sums are added
    // in order.
    auto combine = [&](int rbd, int it0, int it1) {
        const int c0 = rbd * kTileRows, n_it = it1 - it0, P = k * nsd;
        int sp = 1;
        while (sp < 8 && n_it * 2 * sp <= kGroupThreads && 2 * sp <= P) sp *= 2;
        const int sub = gtid % sp;
        const int pa = P * sub / sp, pb = P * (sub + 1) / sp;
        const int ja = pa / nsd, kpa = pa % nsd;
        float* cred = reinterpret_cast<float*>(red_buf);  // [n_it][sp] range sums (sp > 1)
        auto store_out = [&](int it, float v) {
            const size_t o = (size_t)(it / kTileRows) * H + c0 + it % kTileRows;
            if (io.out_fp32) static_cast<float*>(io.out)[o] = v;
            else static_cast<uint16_t*>(io.out)[o] = float_to_bf16_bits(v);
        };
#pragma unroll 1
        for (int it = it0 + gtid / sp; it < it1; it += kGroupThreads / sp) {
            const int t = it / kTileRows, col = c0 + it % kTileRows;
            float v = sub == 0 ? bf16_bits_to_float(io.x_res[(size_t)t * H + col]) : 0.f;
            const float* yc = a.y_part + col;
            const int* sp_t = s_slotpos + t * k;
            int j = ja, kp = kpa;
#pragma unroll 1
            for (int p0 = pa; p0 < pb; p0 += 8) {
                float part[8];
#pragma unroll
                for (int z = 0; z < 8; ++z) {
                    part[z] = 0.f;
                    if (p0 + z < pb) {
                        part[z] = __ldcg(yc + ((size_t)kp * Tk + sp_t[j]) * H);
                        if (++kp == nsd) {
                            kp = 0;
                            ++j;
                        }
                    }
                }
#pragma unroll
                for (int z = 0; z < 8; ++z) v += part[z];  // (the padding adds 0)
            }
            if (sp > 1) cred[(it - it0) * sp + sub] = v;
            else store_out(it, v);
        }
        if (sp > 1) {
            group_sync();
#pragma unroll 1
            for (int it = it0 + gtid; it < it1; it += kGroupThreads) {
                float v = cred[(it - it0) * sp];
                for (int q = 1; q < sp; ++q) v += cred[(it - it0) * sp + q];
                store_out(it, v);
            }
            group_sync();  // the buffer is shared with compute_h
        }
    };

    Walk w = walk_start(grp);
    while (walk_live(w)) {
        const int i = w.i, rb = w.rb, kc = w.kc;
        const int e = s_touched[i], off = s_off[e], c = s_off[e + 1] - off;
        if (w.gu) {
            // ------------------------------------------ gate/up run
            const int n = dispatch(BoolC<true>{}, off, c, w);
            // count the run's K parts of h block rb % RBh (gate rows rb and
            // up rows rb + RBh feed it) once they are stored
            const int hb = rb < RBh ? rb : rb - RBh;
            group_sync();
            if (gtid == 0) red_release_add(&a.cnt_h[i * RBh + hb], n);
        } else {
            // --------------------------------------------- down run
            // (slot i, K part kc, row blocks rb, rb + 1, ...): wait until
            // every gate/up K part of the h blocks the K range overlaps is
            // stored, then form h for the range
            const int f0 = kc * KCd * kTileK, nf = KCd * kTileK;
            if (gtid == 0) {
                bool got = !s_abort;
                for (int hb = f0 / kTileRows; hb <= (f0 + nf - 1) / kTileRows && got; ++hb) {
                    const int* cnt = &a.cnt_h[i * RBh + hb];
                    if (ld_acquire(cnt) < 2 * nsg) {
                        const unsigned long long t0 = globaltimer_ns();
                        while (ld_acquire(cnt) < 2 * nsg) {
                            if (s_abort || globaltimer_ns() - t0 > kWaitLimitNs) {
                                got = false;
                                break;
                            }
                        }
                    }
                }
                if (!got) fail();
                s_flag[grp] = got ? 1 : 0;
            }
            group_sync();
            if (s_flag[grp]) {
                compute_h(off, c, f0, nf, nsg, a.write_qh && rb == 0);
            } else {
                live = false;  // nothing valid to multiply: skip the rest
            }
            group_sync();
            const int n = dispatch(BoolC<false>{}, off, c, w);
            // count the run's tasks (one per column block rb .. rb + n - 1):
            // a release add per block after the barrier that orders the
            // run's stores
            group_sync();
            for (int r = gtid; r < n; r += kGroupThreads) red_release_add(&a.cnt_y[rb + r], 1);
        }
    }

    // ------------------------------------------------------------ combine
    // The items of each output column block are cut into np pieces; piece q
    // of block r (unit u = r * np + q) belongs to worker u * V / (RBd * np),
    // which combines it after its own tasks, once the block's count shows
    // every down task stored.  With no more blocks than workers, no worker
    // holds more than one unit.
    {
        // np: enough pieces that a thread loads at most eight parts (sp
        // threads an item), while there are workers for them and a piece
        // keeps 32 items
        const int V = 2 * G, v = 2 * b + grp, items = kTileRows * T, P = k * nsd;
        int np = 1;
        while (np * 2 <= items / 32 && RBd * np * 2 <= V && (long long)items * P > 2048ll * np) np *= 2;
        const int nu = RBd * np;
        const int u0 = (v * nu + V - 1) / V, u1 = ((v + 1) * nu + V - 1) / V;
        for (int u = u0; u < u1; ++u) {
            const int r = u / np, q = u - r * np;
            if (gtid == 0) {
                const int* cnt = &a.cnt_y[r];
                bool got = !s_abort;
                if (got && ld_acquire(cnt) < nt * nsd) {
                    const unsigned long long t0 = globaltimer_ns();
                    while (ld_acquire(cnt) < nt * nsd) {
                        if (s_abort || globaltimer_ns() - t0 > kWaitLimitNs) {
                            got = false;
                            break;
                        }
                    }
                }
                if (!got) fail();
                s_flag[grp] = got ? 1 : 0;
            }
            group_sync();
            if (s_flag[grp]) combine(r, q * items / np, (q + 1) * items / np);
            group_sync();  // s_flag is reused
        }
    }
}

// One decode layer: one CTA per SM, launched cooperatively (all CTAs
// resident: they wait on one another's results).  At most 96 registers a
// thread, which leaves room on the SM for the next call's prep CTA; the
// MAXNT = 32 variant spills a little instead (it only runs when more than
// 16 tokens are decoded at once).
template <int MAXNT, bool DOTS>
__global__ void __maxnreg__(96) decode_layer_kernel(const LayerArgs a) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ LayerShared S;
    ring_init(a, S, dsm);
    __syncthreads();
    pdl_wait();     // the prep kernel's logits, codes and cleared counters
    pdl_trigger();  // the next call's prep may be scheduled; it waits for our end
    Pipe pp{-1, 0, -1, 0, 1};
    const LayerIO io{a.x_res, a.wgu, a.wd, a.out, a.out_fp32};
    layer_body<MAXNT, DOTS>(a, io, S, dsm, pp);
    ring_drain(a, S, dsm, a.ns);
}

// ------------------------------------------------------ clustered layer
// A second form of the layer kernel for a few tokens.  Pairs of CTAs form
// thread-block clusters; a cluster's kUnitWorkers consumer groups share each
// unit = (touched slot i, 128-feature block hb of h), so that a unit's h
// never leaves the cluster:
//   gate/up  worker w = 2 * rank + g (CTA rank of the cluster, group g):
//            rows of block hb of the gate (g = 0) or up (g = 1) half of
//            W_gu, K part `rank` of kClusterCTAs; its per-token row sums go
//            to every CTA of the cluster (st.async into distributed shared
//            memory, counted as transaction bytes on the receiver's mbarrier)
//   h        each group adds the K parts of gate and of up (part order),
//            h = silu(g) * u, int8 codes per 32 features
//   down     worker w: row blocks w, w + kUnitWorkers, ... of W_d over the
//            block's 128 columns: routing weight * row sums, the parts hb of
//            y (one per h block)
// and a third kernel (decode_combine_kernel) adds, per output element, the
// residual and the k * I/128 parts (slot order, then block order).
// A unit is (slice, h block): each touched expert's bucket of c rows is cut
// into n = ceil(c / cap) slices, rows s cap .. min(c, (s + 1) cap) - 1 of
// slice s: cap = 1 row for T <= 4, else 2 rows for 4-bit and 4 for 8-bit
// weights.  (Measured on the 16-layer decode chain, 4-bit: cap 1 / 2 / 4
// gave T=4 32.9 / 34.1 / 37.6 us and T=16 92.2 / 78.4 / 79.7 us a layer;
// 8-bit at T=16: cap 2 94.1, cap 4 89.3 us, the re-read slices cost more
// with weights 1.89 times as large.)  The slices of one expert read the
// same weights; they sit next to each other in the unit order, so their
// clusters run at about the same time and the later reads find the weights
// in L2.  Units go to clusters in contiguous ranges of equal cost (a unit of
// slice i weighs w0 + c_i, all units have the same tiles).  No CTA
// waits for a CTA outside its cluster, so the launch need not be
// cooperative (a cooperative launch would not start before the prep kernel
// has drained, and costs ~3 us a layer).
constexpr int kClusterCTAs = 2;
constexpr int kUnitWorkers = kClusterCTAs * kGroups;
constexpr int kClusterMaxT = 16;  // tokens per call of the clustered kernel
// Weight of a unit in the clustered kernel's split: w0 + c for a slice of c
// rows (all units have the same tiles).  4-bit weights: w0 = kUnitTileCost;
// measured units take ~6.2 us with one row and ~7.2 us with two (T=16), a
// ratio of 7/6: most of a unit's time does not grow with its rows.  8-bit
// weights (slices of up to 4 rows): w0 = kTileCost, as measured best there.
constexpr int kUnitTileCost = 5;
static_assert(kClusterMaxT * MOE_MAX_TOPK <= kMaxSlices, "a slice holds at least one bucket row");

__device__ __forceinline__ int unit_bound_at(unsigned qt, int cnt, int nt, int NC, int RBh, unsigned ncr,
                                             const int* toff, int w0) {
    if (cnt == 0) return 0;
    const int i = cnt - 1;
    if (i >= nt) return nt * RBh;
    const unsigned base = ncr * (unsigned)(w0 * i + toff[i]);
    const unsigned wn = (unsigned)NC * (unsigned)(w0 + toff[i + 1] - toff[i]);
    const unsigned j = (qt - base + wn - 1) / wn;
    return i * RBh + (int)(j < (unsigned)RBh ? j : (unsigned)RBh);
}

// The first units of clusters q and q + 1 of NC (their range [*u0, *u1)):
// the unit whose cost range holds the position q * total / NC (units of
// slice i, RBh of them, weigh w0 + c_i each, c_i = toff[i + 1] - toff[i]).
// Monotone in q; bound(0) = 0 and bound(NC) = nt * RBh.  The whole warp
// calls it.  Every product stays below 2^31 (NC * RBh * (w0 * nt + Tk),
// w0 <= kUnitTileCost, checked by the host plan), so the arithmetic is
// 32-bit.
__device__ __forceinline__ void unit_bounds_warp(int q, int NC, int nt, int Tk, int RBh, const int* toff,
                                                 int lane, bool equal, int w0, int* u0, int* u1) {
    if (equal) {  // (all units weigh the same)
        *u0 = (q * nt * RBh + NC - 1) / NC;
        *u1 = ((q + 1) * nt * RBh + NC - 1) / NC;
        return;
    }
    const unsigned tot = (unsigned)RBh * (unsigned)(w0 * nt + Tk);
    const unsigned qt0 = (unsigned)q * tot, qt1 = qt0 + tot;  // NC times the positions
    const unsigned ncr = (unsigned)(NC * RBh);
    int cnt0 = 0, cnt1 = 0;  // slices whose first unit starts before each
    for (int i0 = 0; i0 <= nt; i0 += 32) {
        const int i = i0 + lane;
        const unsigned pos = i <= nt ? ncr * (unsigned)(w0 * i + toff[i]) : 0xffffffffu;
        cnt0 += __popc(__ballot_sync(0xffffffffu, pos < qt0));
        cnt1 += __popc(__ballot_sync(0xffffffffu, pos < qt1));
    }
    *u0 = unit_bound_at(qt0, cnt0, nt, NC, RBh, ncr, toff, w0);
    *u1 = unit_bound_at(qt1, cnt1, nt, NC, RBh, ncr, toff, w0);
}

template <int MAXNT, bool DOTS, int WB>
__device__ __forceinline__ void cluster_body(const LayerArgs& a, const LayerIO& io, LayerShared& S,
                                             uint8_t* dsm, Pipe& pp) {
    // WB: weight bits (4: Q4_0 tiles; 8: 8-bit tiles, same layout of rows and
    // scales, one byte a code)
    constexpr int TB = WB == 8 ? kTileBytes8 : kTileBytes;
    constexpr int TCB = WB == 8 ? kTileCodeBytes8 : kTileCodeBytes;
    volatile int& s_abort = S.abort;
    const int T = a.T, H = a.H, I = a.I, k = a.k;
    const int KBg = H / kTileK, KBd = I / kTileK;
    const int RBg = 2 * I / kTileRows, RBd = H / kTileRows, RBh = I / kTileRows;
    const int Gx = H / kGroup, Gh = I / kGroup;
    const int Tk = T * k;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int rank = (int)cluster_ctarank(), cq = (int)cluster_id_x(), NC = (int)cluster_count_x();
    const int Hh = H / kClusterCTAs, Gxh = Gx / kClusterCTAs;  // this CTA's K part of x
    const uint32_t sbase = smem_u32(dsm);
    auto fail = [&]() {
        record_status(a.status, kStatusTimeout);
        s_abort = 1;
    };
    if (warp < kConsumerWarps) {
        // the codes of x and their scales over this CTA's K part: [T][H/2]
        // codes, then [T][Gx/2] scales
        const int nc16 = Hh / 16, ns16 = Gxh * 8 / 16, per = nc16 + ns16;
        const uint8_t* xs_g = a.xq + (size_t)T * H;
        for (int i = tid; i < T * per; i += kConsumerThreads) {
            const int t = i / per, j = i - t * per;
            if (j < nc16)
                cp_async16(sbase + a.off_ax + t * Hh + 16 * j, a.xq + (size_t)t * H + rank * Hh + 16 * j);
            else
                cp_async16(sbase + a.off_ax + T * Hh + t * Gxh * 8 + 16 * (j - nc16),
                           xs_g + ((size_t)t * Gx + rank * Gxh) * 8 + 16 * (j - nc16));
        }
    }
    route_layer<MAXNT == 1 ? kRouteOneTokenOnly : kRouteOneTokenFast>(a, S, dsm, [&](int warp, int lane) {
        if (warp == 0) {
            // the slices of the touched slots' buckets (a warp scan of their
            // counts), the largest and the smallest slice
            const int nt = S.nt;
            const int cap = T <= 4 ? 1 : (WB == 8 ? 4 : 2);  // bucket rows a slice may hold
            int nsl = 0, cm = 0, cmin = kSliceRows;
            if (T == 1) {  // every bucket holds one row: a slice per slot
                for (int i = lane; i < nt; i += 32) {
                    S.sto[i] = S.toff[i];
                    S.sslot[i] = (uint8_t)i;
                }
                nsl = nt;
                cm = cmin = 1;
            }
            for (int i0 = 0; i0 < nt && T > 1; i0 += 32) {
                const int i = i0 + lane;
                const int c = i < nt ? S.toff[i + 1] - S.toff[i] : 0;
                const int lc = cap == 4 ? 2 : cap == 2 ? 1 : 0;  // log2(cap)
                const int n = (c + cap - 1) >> lc;
                int incl = n;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                const int first = nsl + incl - n;
                for (int q = 0; q < n; ++q) {  // runs of cap rows, the last one shorter
                    S.sto[first + q] = S.toff[i] + (q << lc);
                    S.sslot[first + q] = (uint8_t)i;
                }
                if (n > 0) {
                    cm = max(cm, min(c, cap));
                    cmin = min(cmin, c - ((n - 1) << lc));
                }
                nsl += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) S.sto[nsl] = Tk;
            __syncwarp();
            if (T > 1) {
                cm = __reduce_max_sync(0xffffffffu, cm);
                cmin = __reduce_min_sync(0xffffffffu, cmin);
            }
            const bool equal = cmin == cm;
            constexpr int w0 = WB == 8 ? kTileCost : kUnitTileCost;  // a unit's weight: w0 + rows
            static_assert(w0 <= kUnitTileCost, "the host's 32-bit bound");
            int u0, u1;
            unit_bounds_warp(cq, NC, nsl, Tk, RBh, S.sto, lane, equal, w0, &u0, &u1);
            if (lane == 0) {
                S.bnd[0][0] = u0;
                S.bnd[0][1] = u1;
                S.cmax = cm;
            }
        }
    });
    const int ub0 = S.bnd[0][0], nu = S.bnd[0][1] - ub0;
    // The rings and the exchange buffers share ring_bytes: the exchange
    // buffers take what the largest bucket needs, the rings the rest (every
    // CTA lays them out alike from the same routing).
    const int cmax = S.cmax;
    const int pbytes = (2 * kUnitWorkers * cmax * kTileRows * 4 + 127) & ~127;
    const int rbytes = a.ring_bytes - pbytes;
    const int st = T >= 4 && rbytes >= kGroups * 3 * kSlotTiles * TB ? kSlotTiles : 2;
    const int ns = min(kRingStride, rbytes / (st * TB) / kGroups);
    const int off_p = kGroups * ns * st * TB;
    S.rns = ns;  // (every thread stores the same value)
    auto full_bar = [&](int g, int s) { return ring_bar(a, sbase, true, g, s); };
    auto empty_bar = [&](int g, int s) { return ring_bar(a, sbase, false, g, s); };
    auto slot_addr = [&](int g, int s) { return (uint32_t)((g * ns + s) * st * TB); };
    auto pbar = [&](int pb) { return sbase + a.off_bar + 8u * (2 * kMaxSlots + pb); };
    const int KCg = KBg / kClusterCTAs, kb0 = rank * KCg;  // this CTA's K part of gate/up
    const int cptg = (KCg + st - 1) / st;                    // gate/up chunks of a unit

    if (warp >= kWarpProducer0) {
        // ---------------------------------------------------------- producer
        // Worker w's chunks in its consumers' order: per unit, the gate/up
        // K part in runs of st tiles, then its down row blocks (two tiles
        // each: the block's 128 columns).
        const int g = warp - kWarpProducer0, w = 2 * rank + g;
        const int ndn = w < RBd ? (RBd - w + kUnitWorkers - 1) / kUnitWorkers : 0;
        const int cpu = cptg + ndn, nch = nu * cpu;
        bool ok = !s_abort;
        for (int c0 = 0; c0 < nch && ok; c0 += 32) {
            const int c = c0 + lane;
            if (c < nch) {
                const int ul = c / cpu, j = c - ul * cpu;
                const int u = ub0 + ul, i = u / RBh, hb = u - i * RBh;
                const size_t e = (size_t)S.touched[S.sslot[i]];
                const uint8_t* src;
                int n;
                if (j < cptg) {
                    const int rb = g ? RBh + hb : hb, u0 = j * st;
                    src = io.wgu + ((e * RBg + rb) * KBg + kb0 + u0) * TB;
                    n = KCg - u0 < st ? KCg - u0 : st;
                } else {
                    const int rbd = w + (j - cptg) * kUnitWorkers;
                    src = io.wd + ((e * RBd + rbd) * KBd + 2 * hb) * TB;
                    n = 2;
                }
                S.ctab_p[g][lane] = src;
                S.ctab_n[g][lane] = n;
            }
            __syncwarp();
            if (lane == 0) {
                int& slot = pp.slot;
                int& phase = pp.phase;
                int& cidx = pp.cidx;
                const int m = nch - c0 < 32 ? nch - c0 : 32;
                for (int j = 0; j < m; ++j) {
                    ++cidx;
                    if (++slot == ns) {
                        slot = 0;
                        phase ^= 1;
                    }
                    if (s_abort || (cidx >= ns && !mbar_wait(empty_bar(g, slot), phase ^ 1)) || s_abort) {
                        fail();
                        ok = false;
                        break;
                    }
                    const uint32_t bytes = (uint32_t)(S.ctab_n[g][j] * TB);
                    S.slot_chunk[g * kRingStride + slot] = cidx;
                    mbar_arrive_expect_tx(full_bar(g, slot), bytes);
                    bulk_g2s(sbase + slot_addr(g, slot), S.ctab_p[g][j], bytes, full_bar(g, slot));
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int grp = warp / kGroupWarps, w8 = warp % kGroupWarps;
    const int w = 2 * rank + grp;
    const int ndn = w < RBd ? (RBd - w + kUnitWorkers - 1) / kUnitWorkers : 0;
    auto group_sync = [&]() { named_sync(2 + grp, kGroupThreads); };
    const uint8_t* ax_q = dsm + a.off_ax;                                     // [T][H/2]
    const int2* ax_s = reinterpret_cast<const int2*>(ax_q + (size_t)T * Hh);  // [T][Gx/2]
    uint8_t* hq = dsm + a.off_h + grp * a.h_bytes;                           // [T][128] codes
    int2* hs = reinterpret_cast<int2*>(hq + (size_t)T * kTileRows);          // [T][4]
    const float* pbuf = reinterpret_cast<const float*>(dsm + off_p);  // [2][workers][cmax][128]
    cp_async_wait_all();
    named_sync(1, kConsumerThreads);
    bool live = !s_abort;
    // warp 0 of group 0 keeps this CTA's exchange barriers armed (its lane 0
    // arms them); it waits on every phase, even after a failure elsewhere,
    // so that it never arms a phase twice.  armok is uniform in the warp.
    const bool arm_warp = grp == 0 && w8 == 0;
    int& armok = pp.armok;
    int& slot = pp.slot;
    int& phase = pp.phase;
    const int r_lane = lane >> 1, h_lane = lane & 1;
    const int lrow = w8 * 16 + r_lane;
    const int code_off = WB == 8 ? w8 * 1024 + lane * 32 : w8 * 512 + lane * 16;
    const int scale_off = TCB + w8 * 64 + lane * 2;
    auto next_chunk = [&]() -> const uint8_t* {
        if (++slot == ns) {
            slot = 0;
            phase ^= 1;
        }
        if (live && (s_abort || !mbar_wait(full_bar(grp, slot), phase))) {
            fail();
            live = false;
        }
        return dsm + slot_addr(grp, slot);
    };
    auto free_chunk = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(grp, slot));
    };

    auto unit = [&](auto ntc, int ul) {
        constexpr int NT = decltype(ntc)::value;
        const int u = ub0 + ul, i = u / RBh, hb = u - i * RBh;  // (slice, h block)
        const int off = S.sto[i], c = S.sto[i + 1] - off;         // its bucket rows
        const int ux = pp.units + ul;  // the exchange's ordinal in the launch
        const int pb = ux & 1;
        const uint32_t ppar = (uint32_t)((ux >> 1) & 1);
        if (arm_warp && armok && lane == 0)
            mbar_arrive_expect_tx(pbar(pb), (uint32_t)(kUnitWorkers * c * kTileRows * 4));
        // ------------------------------------------------ gate/up K part
        const int rb = grp ? RBh + hb : hb;
        const int row = rb * kTileRows + lrow;
        constexpr int NH = NT <= 4 ? NT : 1;
        constexpr int NB = NT < 4 ? NT : 4;  // bucket rows per block of dot chains
        int arow[NH], srow[NH];
#pragma unroll
        for (int n = 0; n < NH; ++n) {
            const int ar = S.btok[off + (n < c ? n : 0)];
            arow[n] = ar * Hh;
            srow[n] = ar * Gxh;
        }
        float acc[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n] = 0.f;
        for (int jc = 0; jc < cptg; ++jc) {
            const int u0 = jc * st, nuj = KCg - u0 < st ? KCg - u0 : st;
            const uint8_t* chunk = next_chunk();
            if (live) {
                for (int uu = 0; uu < nuj; ++uu) {
                    const uint8_t* tile = chunk + uu * TB;
                    const float dw = half_bits_to_float(*reinterpret_cast<const uint16_t*>(tile + scale_off));
                    uint32_t wl[4], wh[4];
                    unpack_codes<WB>(tile + code_off, wl, wh);
                    const int gl = 2 * (u0 + uu) + h_lane, g = 2 * kb0 + gl;  // (local, absolute)
                    // blocks of NB bucket rows as independent dot chains; rows
                    // past c repeat an earlier row (in bounds) and their sums
                    // are never sent
#pragma unroll
                    for (int n0 = 0; n0 < NT; n0 += NB) {
                        if (n0 < c) {
                            int2 sc[NB];
                            int dot[NB];
#pragma unroll
                            for (int j = 0; j < NB; ++j) {
                                int ao, so;
                                if constexpr (NT <= 4) {
                                    ao = arow[n0 + j];
                                    so = srow[n0 + j];
                                } else {
                                    const int ar = S.btok[off + (n0 + j < c ? n0 + j : c - 1)];
                                    ao = ar * Hh;
                                    so = ar * Gxh;
                                }
                                sc[j] = ax_s[so + gl];
                                dot[j] = group_dot_w<WB>(wl, wh, ax_q + ao + gl * kGroup, sc[j].y);
                            }
#pragma unroll
                            for (int j = 0; j < NB; ++j) {
                                acc[n0 + j] = fmaf((float)dot[j], dw * __int_as_float(sc[j].x), acc[n0 + j]);
                                if (DOTS && n0 + j < c)
                                    a.dots_gu[((size_t)(off + n0 + j) * 2 * I + row) * Gx + g] = dot[j];
                            }
                        }
                    }
                }
            }
            free_chunk();
        }
        // the K part's row sums to every CTA of the cluster: lane 8q sends
        // rows 4q' .. 4q' + 3 of its warp (the lane pairs' sums)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            if (n < c) {
                const float v = acc[n] + __shfl_xor_sync(0xffffffffu, acc[n], 1);
                const float v1 = __shfl_down_sync(0xffffffffu, v, 2);
                const float v2 = __shfl_down_sync(0xffffffffu, v, 4);
                const float v3 = __shfl_down_sync(0xffffffffu, v, 6);
                if ((lane & 7) == 0) {
                    const uint32_t la =
                        sbase + off_p + 4u * ((((pb * kUnitWorkers + w) * cmax + n) * kTileRows) + lrow);
#pragma unroll
                    for (int d = 0; d < kClusterCTAs; ++d)
                        st_async_v4(mapa_shared(la, d), v, v1, v2, v3, mapa_shared(pbar(pb), d));
                }
            }
        }
        // ------------------------------------- h (every K part has arrived)
        if (arm_warp ? armok : live) {
            const bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(pbar(pb), ppar));
            if (!ok) {
                armok = 0;
                if (live) fail();
                live = false;
            } else if (live && s_abort) {
                live = false;
            }
        }
        for (int n = w8; n < c; n += kGroupWarps) {  // warp n: bucket row n, lane: 4 features
            const int f = 4 * lane;
            float gv[4] = {0.f, 0.f, 0.f, 0.f}, uv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int r = 0; r < kClusterCTAs; ++r) {
                const float4 g4 = *reinterpret_cast<const float4*>(
                    pbuf + (((pb * kUnitWorkers + 2 * r) * cmax + n) * kTileRows + f));
                const float4 u4 = *reinterpret_cast<const float4*>(
                    pbuf + (((pb * kUnitWorkers + 2 * r + 1) * cmax + n) * kTileRows + f));
                gv[0] += g4.x; gv[1] += g4.y; gv[2] += g4.z; gv[3] += g4.w;
                uv[0] += u4.x; uv[1] += u4.y; uv[2] += u4.z; uv[3] += u4.w;
            }
            float h[4], amax = 0.f;
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                h[z] = gv[z] / (1.0f + __expf(-gv[z])) * uv[z];
                amax = fmaxf(amax, fabsf(h[z]));
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const uint16_t db = act_scale_bits(amax);
            const float d = half_bits_to_float(db);
            uint32_t w4 = 0u;
            int sum = 0;
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const int qv = act_code(h[z], d);
                sum += qv;
                w4 |= ((uint32_t)qv & 0xffu) << (8 * z);
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            const uint32_t w4o = __shfl_xor_sync(0xffffffffu, w4, 1);
            if ((lane & 1) == 0) *reinterpret_cast<uint2*>(hq + n * kTileRows + f) = permute_chunk(w4, w4o);
            if ((lane & 7) == 0) hs[n * 4 + lane / 8] = make_int2(__float_as_int(d), -8 * sum);
            if (a.write_qh && w == 0) {
                const size_t prow = (size_t)(off + n);
                *reinterpret_cast<uint32_t*>(a.q_h + prow * I + hb * kTileRows + f) = w4;
                if ((lane & 7) == 0) a.d_h[prow * Gh + hb * 4 + lane / 8] = db;
            }
        }
        group_sync();
        // ------------------------------------------- down row blocks
        for (int dd = 0; dd < ndn; ++dd) {
            const int rbd = w + dd * kUnitWorkers;
            const uint8_t* chunk = next_chunk();
            float accd[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) accd[n] = 0.f;
            if (live) {
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const uint8_t* tile = chunk + kt * TB;
                    const float dw = half_bits_to_float(*reinterpret_cast<const uint16_t*>(tile + scale_off));
                    uint32_t wl[4], wh[4];
                    unpack_codes<WB>(tile + code_off, wl, wh);
                    const int gl = 2 * kt + h_lane;
#pragma unroll
                    for (int n0 = 0; n0 < NT; n0 += NB) {
                        if (n0 < c) {
                            int2 sc[NB];
                            int dot[NB];
#pragma unroll
                            for (int j = 0; j < NB; ++j) {
                                const int n = n0 + j < c ? n0 + j : c - 1;  // rows past c: in bounds, unused
                                sc[j] = hs[n * 4 + gl];
                                dot[j] = group_dot_w<WB>(wl, wh, hq + n * kTileRows + gl * kGroup, sc[j].y);
                            }
#pragma unroll
                            for (int j = 0; j < NB; ++j) {
                                accd[n0 + j] = fmaf((float)dot[j], dw * __int_as_float(sc[j].x), accd[n0 + j]);
                                if (DOTS && n0 + j < c)
                                    a.dots_d[((size_t)(off + n0 + j) * H + rbd * kTileRows + lrow) * Gh +
                                             hb * 4 + gl] = dot[j];
                            }
                        }
                    }
                }
            }
            free_chunk();
#pragma unroll
            for (int n0 = 0; n0 < NT; n0 += NB) {
                if (n0 < c) {  // warp-uniform: every lane takes the shuffles
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        const int n = n0 + j;
                        const float v = accd[n] + __shfl_xor_sync(0xffffffffu, accd[n], 1);
                        if (n < c && h_lane == 0 && live) {
                            const int tj = S.btok[off + n] * k + S.bslot[off + n];  // (token, choice)
                            a.y_part[((size_t)hb * Tk + tj) * H + rbd * kTileRows + lrow] = v * S.bsw[off + n];
                        }
                    }
                }
            }
        }
        group_sync();  // the h buffer is rewritten by the next unit
    };

    for (int ul = 0; ul < nu; ++ul) {
        static_assert(kSliceRows == 4, "units hold at most 4 bucket rows");
        if constexpr (MAXNT == 1) {
            unit(IntC<1>{}, ul);
        } else {
            const int i = (ub0 + ul) / RBh, c = S.sto[i + 1] - S.sto[i];
            if (c <= 1) unit(IntC<1>{}, ul);
            else if (c <= 2) unit(IntC<2>{}, ul);
            else if constexpr (WB == 8) unit(IntC<4>{}, ul);  // (4-bit units hold at most 2 rows)
        }
    }
    pp.units += nu;
    // every byte sent to this CTA has arrived before it may leave (the
    // arming warp waited on every phase unless one ran out of time)
    if (arm_warp && !armok && lane == 0) fail();
}

// The experts of one decode layer by clusters of kClusterCTAs CTAs, one CTA
// per SM.  MAXNT: the most tokens a bucket may hold (T <= MAXNT).
template <int MAXNT, bool DOTS, int WB>
__global__ void __maxnreg__(96) decode_cluster_kernel(const LayerArgs a) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ LayerShared S;
    if (threadIdx.x == 0) {
        const uint32_t sbase = smem_u32(dsm);
        for (int pb = 0; pb < 2; ++pb) mbar_init(sbase + a.off_bar + 8u * (2 * kMaxSlots + pb), 1);
    }
    ring_init(a, S, dsm);  // (its thread 0 fences the barrier inits for the cluster)
    __syncthreads();
    cluster_sync_all();  // the peers' exchange barriers exist before anyone sends
    pdl_wait();          // the prep kernel's logits, codes and cleared tickets
    pdl_trigger();
    Pipe pp{-1, 0, -1, 0, 1};
    const LayerIO io{a.x_res, a.wgu, a.wd, a.out, a.out_fp32};
    cluster_body<MAXNT, DOTS, WB>(a, io, S, dsm, pp);
    ring_drain(a, S, dsm, S.rns);
    __syncwarp();
    cluster_sync_all();  // no CTA leaves while its peer may still address it
}

// ------------------------------------------------------------- combine
// After the clustered layer kernel: out[t][col] = x[t][col] plus the k
// choices' parts (choice j = 0 .. k-1, then h block 0 .. nparts-1, in that
// order; the parts are stored by (token, choice)).  A CTA takes 32 consecutive columns of one token; warp w adds the
// w-th eighth of the parts (warp 0 starting from the residual), the eighths
// are added in warp order.
constexpr int kCombineWarps = 8;
struct CombineArgs {
    const uint16_t* x_res;
    const float* y_part;     // [nparts][T*k][H], row t*k + j
    int T, H, k, nparts;
    void* out;
    int out_fp32;
};

// Output columns 32*blk .. +31 (of the T x H output, row-major) by warps
// 0 .. kCombineWarps-1 of the calling CTA.
__device__ __forceinline__ void combine_cols32(const CombineArgs& c, int blk, float (*s_part)[32]) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int it = blk * 32 + lane;  // (H is a multiple of 32)
    const int t = it / c.H, col = it - t * c.H;
    const int Tk = c.T * c.k, P = c.k * c.nparts;
    const int pa = P * warp / kCombineWarps, pe = P * (warp + 1) / kCombineWarps;
    const bool mine = t < c.T;
    float v = mine && warp == 0 ? bf16_bits_to_float(c.x_res[(size_t)t * c.H + col]) : 0.f;
    int j = pa / c.nparts, hb = pa - (pa / c.nparts) * c.nparts;
#pragma unroll 1
    for (int p0 = pa; p0 < pe; p0 += 8) {
        float part[8];
#pragma unroll
        for (int z = 0; z < 8; ++z) {
            part[z] = 0.f;
            if (mine && p0 + z < pe) {
                part[z] = __ldcg(c.y_part + ((size_t)hb * Tk + t * c.k + j) * c.H + col);
                if (++hb == c.nparts) {
                    hb = 0;
                    ++j;
                }
            }
        }
#pragma unroll
        for (int z = 0; z < 8; ++z) v += part[z];
    }
    s_part[warp][lane] = v;
    named_sync(kCombineBarId, kCombineWarps * 32);
    if (warp == 0 && mine) {
        for (int w = 1; w < kCombineWarps; ++w) v += s_part[w][lane];
        const size_t o = (size_t)t * c.H + col;
        if (c.out_fp32) static_cast<float*>(c.out)[o] = v;
        else static_cast<uint16_t*>(c.out)[o] = float_to_bf16_bits(v);
    }
    named_sync(kCombineBarId, kCombineWarps * 32);  // s_part is reused
}

__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(const CombineArgs c) {
    __shared__ float s_part[kCombineWarps][32];
    pdl_wait();  // the layer kernel's parts
    pdl_trigger();
    combine_cols32(c, blockIdx.x, s_part);
}

// ---------------------------------------------------------------- launch
int g_layer_pdl[64] = {};  // 0 unknown, 1 cooperative + PDL accepted, 2 cooperative only
// clustered kernel: 0 unknown, 1 clusters + PDL accepted, 2 clusters without
// PDL, 3 not accepted (the task kernel runs instead)
int g_cluster_mode[64] = {};
int g_prep_carveout[64] = {};

struct Plan {
    int ns, st, off_bar, off_ax, off_ah, ah_bytes, off_red, smem;
    int ring_bytes, off_h, h_bytes;  // clustered kernel
};

int al128(long long v) { return (int)((v + 127) & ~127ll); }

// Shared-memory plan of the layer kernel; false if it does not fit.
// Layout: the two rings, the two groups' h buffers and K-part sum buffers
// (all idle while the CTA routes, when they hold the logits), then the
// codes of x (filled by cp.async during routing) and the ring barriers.
bool plan_layer(int T, int H, int I, int E, long long budget, Plan* p) {
    const long long ax = al128((long long)T * H + (long long)T * (H / kGroup) * 8);
    const long long ah = al128((long long)T * I + (long long)T * (I / kGroup) * 8);
    const long long rest = budget - ax - 2 * ah - 2 * kRedBytes - 2 * kMaxSlots * 8 - 256;
    // slots of four tiles for several tokens while each group's ring keeps
    // three of them (fewer chunk hand-offs), else two-tile slots (one token:
    // short tasks, deeper ring), else the largest slot that still gives each
    // group's ring two slots, else one
    int st = T >= 4 && rest >= (long long)kGroups * 3 * kSlotTiles * kTileBytes ? kSlotTiles : 2;
    while (st > 1 && rest < (long long)kGroups * 2 * st * kTileBytes) st /= 2;
    int ns = (int)(rest / ((long long)st * kTileBytes)) / kGroups;  // slots of each group's ring
    ns = ns > kMaxSlots / kGroups ? kMaxSlots / kGroups : ns;
    if (ns < 1) return false;
    p->ns = ns;
    p->st = st;
    p->off_ah = kGroups * ns * st * kTileBytes;
    p->ah_bytes = (int)ah;
    p->off_red = p->off_ah + 2 * (int)ah;
    p->off_ax = al128(p->off_red + 2 * kRedBytes);
    p->off_bar = al128(p->off_ax + ax);
    p->smem = p->off_bar + 2 * kMaxSlots * 8;
    // the routing phase keeps all T x E logits and their order keys below
    // the codes of x
    return (long long)T * E * 8 <= p->off_ax;
}

// Shared-memory plan of the clustered layer kernel; false if it does not
// fit (or T exceeds kClusterMaxT).  Layout: the rings and the K-part
// exchange buffers [2][workers][cmax][128] fp32 (ring_bytes, laid out by the
// kernel once the largest bucket cmax is known), the groups' h buffers, the
// codes of x over the CTA's K part, the barriers (rings, then the two
// exchange barriers).  ring_bytes must hold the exchange buffers of T tokens
// and two two-tile slots a group.
bool plan_cluster(int T, int H, int I, int E, long long budget, Plan* p, int wbits = 4) {
    const int tile_bytes = wbits == 8 ? kTileBytes8 : kTileBytes;
    if (T < 1 || T > kClusterMaxT) return false;
    // the unit split's 32-bit products: NC * RBh * (kUnitTileCost * slices +
    // Tk) with at most 1024 clusters and kMaxSlices slices
    if ((long long)(I / kTileRows) * 1024 * (kUnitTileCost + 1) * kMaxSlices >= (1ll << 31)) return false;
    if ((H / kTileK) % kClusterCTAs) return false;
    const long long ax = al128((long long)T * (H / kClusterCTAs) + (long long)T * (H / kGroup / kClusterCTAs) * 8);
    const long long hbytes = al128((long long)T * kTileRows + (long long)T * 4 * 8);
    const long long bars = (2ll * kMaxSlots + 2) * 8;
    const long long rb = (budget - ax - 2 * hbytes - bars - 256) & ~127ll;
    const long long pmax = al128(2ll * kUnitWorkers * T * kTileRows * 4);
    const long long ring_min = (long long)kGroups * 2 * 2 * tile_bytes;
    if (rb < pmax + ring_min) return false;
    // the routing scratch (logits and keys) stays below the exchange
    // buffers, which a peer may fill while this CTA still routes
    if ((long long)T * E * 8 > ring_min) return false;
    p->ns = p->st = 0;
    p->ring_bytes = (int)rb;
    p->off_h = (int)rb;
    p->h_bytes = (int)hbytes;
    p->off_ax = al128(p->off_h + 2 * hbytes);
    p->off_bar = al128(p->off_ax + ax);
    p->smem = p->off_bar + (int)bars;
    p->off_ah = p->off_red = p->ah_bytes = 0;
    return true;
}

__global__ void coop_pdl_probe_kernel(int* p) {
    pdl_wait();
    if (p && threadIdx.x == 0 && blockIdx.x == 0) *p = 1;
}

__global__ void cluster_probe_kernel(int* p) {
    cluster_sync_all();
    pdl_wait();
    if (p && threadIdx.x == 0 && blockIdx.x == 0) *p = 1;
}

}  // namespace

// Decides once per device (outside any capture) whether a cooperative launch
// may also carry the programmatic-dependent-launch attribute.
cudaError_t decode_prepare_device(int dev) {
    int& mode = g_layer_pdl[dev & 63];
    if (mode != 0) return cudaSuccess;
    cudaStream_t st;
    cudaError_t err = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[2];
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(32);
    cfg.stream = st;
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, coop_pdl_probe_kernel, (int*)nullptr);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&cfg, coop_pdl_probe_kernel, (int*)nullptr);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err == cudaSuccess) {
        mode = 1;
    } else {
        cudaGetLastError();  // refused: a launch error only, the context is intact
        mode = 2;
    }
    // a launch in clusters of kClusterCTAs, with PDL, else without
    cudaLaunchAttribute ac[2];
    ac[0].id = cudaLaunchAttributeClusterDimension;
    ac[0].val.clusterDim.x = kClusterCTAs;
    ac[0].val.clusterDim.y = 1;
    ac[0].val.clusterDim.z = 1;
    ac[1] = at[1];
    cfg.gridDim = dim3(2 * kClusterCTAs);
    cfg.attrs = ac;
    int& cm = g_cluster_mode[dev & 63];
    for (int na = 2; na >= 1 && cm == 0; --na) {
        cfg.numAttrs = na;
        err = cudaLaunchKernelEx(&cfg, cluster_probe_kernel, (int*)nullptr);
        if (err == cudaSuccess) err = cudaLaunchKernelEx(&cfg, cluster_probe_kernel, (int*)nullptr);
        if (err == cudaSuccess) err = cudaStreamSynchronize(st);
        if (err == cudaSuccess) cm = na == 2 ? 1 : 2;
        else cudaGetLastError();
    }
    if (cm == 0) cm = 3;
    cudaStreamDestroy(st);
    return cudaSuccess;
}

int cooperative_pdl_mode(int dev) { return g_layer_pdl[dev & 63]; }

bool decode_shape_fits(int T, int H, int I, int E) {
    Plan p;
    return plan_layer(T, H, I, E, kLayerSmemBudget, &p);
}

void decode_split_bounds(int T, int H, int I, int E, int k, int* cap_g, int* cap_d, int* nsg_max,
                         int* nsd_max) {
    const size_t Tk = (size_t)T * k;
    const int KBg = H / kTileK, KBd = I / kTileK;
    auto cap = [](size_t budget, size_t part_bytes) {
        size_t c = part_bytes ? budget / part_bytes : kMaxSplit;
        return (int)std::max<size_t>(1, std::min<size_t>(c, kMaxSplit));
    };
    *cap_g = cap(kPartBudgetGU, Tk * 2 * I * 4);
    *cap_d = cap(kPartBudgetD, Tk * H * 4);
    // the split only shrinks as more experts are touched, and at least k are
    const int nt_min = std::max(1, std::min(k, E));
    *nsg_max = decode_split_for(nt_min * (2 * I / kTileRows), KBg, kTargetTasks, *cap_g);
    *nsd_max = decode_split_for(nt_min * (H / kTileRows), KBd, kTargetTasks, *cap_d);
}

int decode_sync_ints(int T, int H, int I, int E, int k) {
    const int nslot = std::min(E, T * k);
    return nslot * (I / kTileRows) + H / kTileRows;
}

bool decode_w8_fits(int T, int H, int I, int E) {
    Plan p;
    return T <= MOE_W8_DECODE_MAX_T && plan_cluster(T, H, I, E, kLayerSmemBudget, &p, 8);
}

int decode_cluster_parts(int T, int H, int I, int E) {
    Plan p;
    return plan_cluster(T, H, I, E, kLayerSmemBudget, &p) ? I / kTileRows : 0;
}

namespace {

PrepArgs make_prep_args(int T, int H, int I, int E, int k, bool prenorm, const Workspace& ws,
                        int* status) {
    PrepArgs p{};
    p.T = T;
    p.H = H;
    p.E = E;
    p.prenorm = prenorm ? 1 : 0;
    p.logits = ws.logits;
    p.xq = ws.xq;
    p.xs = ws.xs;
    p.q_x = ws.q_x;
    p.d_x = ws.d_x;
    p.sync = ws.sync;
    p.nsync = decode_sync_ints(T, H, I, E, k);
    p.status = status;
    return p;
}

LayerArgs make_layer_args(int T, int H, int I, int E, int k, const Workspace& ws, const Plan& plan,
                          int* status) {
    LayerArgs a{};
    a.T = T;
    a.H = H;
    a.I = I;
    a.E = E;
    a.k = k;
    a.logits = ws.logits;
    a.xq = ws.xq;
    a.xs = ws.xs;
    a.topk_idx = ws.topk_idx;
    a.topk_w = ws.topk_w;
    a.offsets = ws.offsets;
    a.touched = ws.touched;
    a.counters = ws.counters;
    a.bucket_token = ws.bucket_token;
    a.bucket_slot = ws.bucket_slot;
    a.gu_part = ws.gu_part;
    a.q_h = ws.q_h;
    a.d_h = ws.d_h;
    a.y_part = ws.y_part;
    const int nslot = std::min(E, T * k);
    a.cnt_h = ws.sync;
    a.cnt_y = ws.sync + nslot * (I / kTileRows);
    a.cap_g = ws.cap_g;
    a.cap_d = ws.cap_d;
    // the K splits the kernel may choose: divisors of the row's 64-column
    // blocks within the cap, at least two tiles a task (the rule of
    // decode_split_for)
    auto divisors = [](int KB, int cap, int* list, int* n) {
        const int dmax = KB > 1 ? KB / 2 : 1;
        for (int d = 1; d <= dmax && d <= cap && *n < 16; ++d)
            if (KB % d == 0) list[(*n)++] = d;
    };
    divisors(H / kTileK, ws.cap_g, a.div_g, &a.ndiv_g);
    divisors(I / kTileK, ws.cap_d, a.div_d, &a.ndiv_d);
    a.status = status;
    a.ns = plan.ns;
    a.st = plan.st;
    a.off_bar = plan.off_bar;
    a.off_ax = plan.off_ax;
    a.off_ah = plan.off_ah;
    a.ah_bytes = plan.ah_bytes;
    a.off_red = plan.off_red;
    return a;
}

// A cooperative launch of one CTA per SM, with programmatic dependent launch
// where the device accepts both.
template <typename Args>
cudaError_t launch_coop(void (*kern)(Args), const Args& args, int num_sms, int smem, int dev,
                        cudaStream_t s) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[2];
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kLayerThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = (g_layer_pdl[dev & 63] == 2) ? 1 : 2;
    if ((err = cudaLaunchKernelEx(&cfg, kern, args)) != cudaSuccess) {
        cudaGetLastError();  // a refused launch: clear it, the context is intact
        return err;
    }
    return cudaSuccess;
}

int g_cluster_max[64] = {};  // co-resident clusters of the clustered kernel (0: not asked yet)

// A launch of the clustered layer kernel: clusters of kClusterCTAs CTAs, as
// many as the device holds at once (at most one CTA per SM), with
// programmatic dependent launch where the device accepts it.
cudaError_t launch_cluster(void (*kern)(LayerArgs), const LayerArgs& args, int num_sms, int smem, int dev,
                           cudaStream_t s) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[2];
    cfg.blockDim = dim3(kLayerThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kClusterCTAs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    int ncl = num_sms / kClusterCTAs;
    int& mx = g_cluster_max[dev & 63];
    if (mx == 0) {
        cfg.gridDim = dim3(ncl * kClusterCTAs);
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) {
            mx = n;
        } else {
            cudaGetLastError();
            mx = ncl;
        }
    }
    ncl = std::min(std::min(ncl, mx), 1024);  // (the unit split's 32-bit bound)
    if (ncl < 1) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(ncl * kClusterCTAs);
    cfg.numAttrs = g_cluster_mode[dev & 63] == 1 ? 2 : 1;
    if ((err = cudaLaunchKernelEx(&cfg, kern, args)) != cudaSuccess) {
        cudaGetLastError();
        return err;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_decode(const uint16_t* x, const float* wr, const void* wgu, const void* wd,
                          int T, int H, int I, int E, int k, bool prenorm, bool out_fp32,
                          void* out, const Workspace& ws, int32_t* dots_gu, int32_t* dots_d,
                          bool write_qh, int* status, int num_sms, void** ev, bool capturing,
                          cudaStream_t s, int wbits) {
    if (T == 0) return cudaSuccess;
    Plan plan;
    if (!plan_layer(T, H, I, E, kLayerSmemBudget, &plan)) return cudaErrorInvalidValue;
    cudaError_t err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    auto mark = [&](int i) -> cudaError_t {
        return (ev && ev[i]) ? record_stage(ev[i], s, capturing) : cudaSuccess;
    };
    // ---- prep ----
    PrepArgs p = make_prep_args(T, H, I, E, k, prenorm, ws, status);
    p.x = x;
    p.wr = wr;
    const int psmem = H * 4;
    if (psmem > 48 * 1024 &&
        (err = cudaFuncSetAttribute(decode_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    psmem)) != cudaSuccess)
        return err;
    // the SM's largest shared-memory split for the prep kernel too, so that a
    // layer CTA of the same call can be placed beside a running prep CTA
    if (!g_prep_carveout[dev & 63]) {
        if ((err = cudaFuncSetAttribute(decode_prep_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                        (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return err;
        g_prep_carveout[dev & 63] = 1;
    }
    // E router-row CTAs and the CTAs coding x, 32 groups each
    const int ncode = (T * (H / kGroup) + kPrepThreads / 4 - 1) / (kPrepThreads / 4);
    if ((err = launch_pdl(decode_prep_kernel, dim3(E + ncode), dim3(kPrepThreads), psmem, s, p)) !=
        cudaSuccess) {
        cudaGetLastError();
        return err;
    }
    if ((err = mark(1)) != cudaSuccess) return err;
    // ---- layer ----
    LayerArgs a = make_layer_args(T, H, I, E, k, ws, plan, status);
    a.x_res = x;
    a.wgu = static_cast<const uint8_t*>(wgu);
    a.wd = static_cast<const uint8_t*>(wd);
    a.out = out;
    a.out_fp32 = out_fp32 ? 1 : 0;
    a.dots_gu = dots_gu;
    a.dots_d = dots_d;
    a.write_qh = write_qh ? 1 : 0;
    const bool dots = dots_gu || dots_d;
    Plan cplan;
    const bool clustered = g_cluster_mode[dev & 63] <= 2 && plan_cluster(T, H, I, E, kLayerSmemBudget, &cplan, wbits);
    if (wbits == 8 && !clustered) return cudaErrorNotSupported;  // (8-bit weights: the clustered kernel only)
    if (clustered) {
        a.ns = a.st = 0;  // (the kernel lays out its rings)
        a.off_bar = cplan.off_bar;
        a.off_ax = cplan.off_ax;
        a.ring_bytes = cplan.ring_bytes;
        a.off_h = cplan.off_h;
        a.h_bytes = cplan.h_bytes;
        a.y_part = ws.y_unit;
        void (*kern)(LayerArgs);
        if (wbits == 8)
            kern = T <= 8 ? (dots ? decode_cluster_kernel<8, true, 8> : decode_cluster_kernel<8, false, 8>)
                          : (dots ? decode_cluster_kernel<kClusterMaxT, true, 8>
                                  : decode_cluster_kernel<kClusterMaxT, false, 8>);
        else
            kern = T <= 8 ? (dots ? decode_cluster_kernel<8, true, 4> : decode_cluster_kernel<8, false, 4>)
                          : (dots ? decode_cluster_kernel<kClusterMaxT, true, 4>
                                  : decode_cluster_kernel<kClusterMaxT, false, 4>);
        if ((err = launch_cluster(kern, a, num_sms, cplan.smem, dev, s)) != cudaSuccess) return err;
        for (int i = 2; i <= 5; ++i)
            if ((err = mark(i)) != cudaSuccess) return err;
        CombineArgs c{x, a.y_part, T, H, k, I / kTileRows, out, out_fp32 ? 1 : 0};
        if ((err = launch_pdl(decode_combine_kernel, dim3((T * H) / 32), dim3(kCombineWarps * 32), 0, s, c)) !=
            cudaSuccess) {
            cudaGetLastError();
            return err;
        }
        if ((err = mark(6)) != cudaSuccess) return err;
        return cudaGetLastError();
    }
    void (*kern)(LayerArgs) =
        T <= 16 ? (dots ? decode_layer_kernel<16, true> : decode_layer_kernel<16, false>)
                : (dots ? decode_layer_kernel<MOE_DECODE_MAX_T, true> : decode_layer_kernel<MOE_DECODE_MAX_T, false>);
    if ((err = launch_coop(kern, a, num_sms, plan.smem, dev, s)) != cudaSuccess) return err;
    for (int i = 2; i <= 6; ++i)
        if ((err = mark(i)) != cudaSuccess) return err;
    return cudaGetLastError();
}

cudaError_t launch_decode_stack(const uint16_t* x, int L, const float* const* wr,
                                const void* const* wgu, const void* const* wd, int T, int H, int I,
                                int E, int k, bool prenorm, bool out_fp32, void* out,
                                const Workspace& ws, int* status, int num_sms, cudaStream_t s) {
    if (T == 0 || L == 0) return cudaSuccess;
    if (L > MOE_DECODE_MAX_LAYERS) return cudaErrorInvalidValue;

    // layer l reads layer l - 1's bf16 output from one workspace buffer and
    // writes the other; each layer's prep kernel waits for the layer before
    const uint16_t* cur = x;
    for (int l = 0; l < L; ++l) {
        const bool last = l == L - 1;
        void* dst = last ? out : static_cast<void*>(l % 2 ? ws.xbuf1 : ws.xbuf0);
        cudaError_t err = launch_decode(cur, wr[l], wgu[l], wd[l], T, H, I, E, k, prenorm, last && out_fp32,
                                        dst, ws, nullptr, nullptr, false, status, num_sms, nullptr, false, s, 4);
        if (err != cudaSuccess) return err;
        cur = static_cast<const uint16_t*>(dst);
    }
    return cudaSuccess;
}

}  // namespace moeq4
