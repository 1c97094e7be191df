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
constexpr int kMaxRing = 48;                            // tile slots of both groups' rings
// Dynamic shared memory of the layer kernel: leaves room on the SM for a
// prep CTA of the next call (its router row) next to it.
constexpr int kLayerSmemBudget = 184 * 1024;
constexpr int kPrepThreads = 128;
constexpr int kMaxTk = MOE_DECODE_MAX_T * MOE_MAX_TOPK;
// Tasks the K split aims for (gate/up, down); the split depends only on the
// number of touched experts and the shape, so results are reproducible.
constexpr int kTargetGU = 152 * 8;
constexpr int kTargetD = 152 * 4;
constexpr int kMaxSplit = 16;
// Bytes of K-part sums (each of gate/up and down) the split may use; beyond
// it the split is capped.
constexpr size_t kPartBudget = 1u << 20;

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
    uint8_t* hq;        // [T*k, I] int8 codes of h, dp4a order
    int2* hs;           // [T*k, I/32] {fp32 bits of the scale, -8 * sum}
    int8_t* q_h;        // [T*k, I] stage output (column order), when write_qh
    uint16_t* d_h;      // [T*k, I/32]
    float* y_part;      // [nsd, T*k, H] K parts of the weighted expert outputs
    int* cnt_h;         // [nslot, I/128] finished gate/up tasks per h block
    int* done_h;        // [nslot] h blocks done per touched expert
    int* cnt_y;         // [H/128] finished down tasks per output column block
    int cap_g, cap_d;   // upper bounds of the K splits (size of the part buffers)
    void* out;
    int out_fp32;
    int32_t* dots_gu;   // optional stage outputs
    int32_t* dots_d;
    int write_qh;
    int* status;
    // shared-memory plan (bytes from the dynamic base)
    int ns;             // slots (one tile each) of each group's ring
    int off_bar, off_ax, off_ah, ah_bytes;
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

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int N>
struct IntC {
    static constexpr int value = N;
};

}  // namespace

// Smallest divisor d of KB (d <= cap) with units * d >= target; if there is
// none, the largest divisor <= cap.  Non-increasing in `units`.
__host__ __device__ inline int decode_split_for(int units, int KB, int target, int cap) {
    int best = 1;
    for (int d = 1; d <= KB && d <= cap; ++d) {
        if (KB % d) continue;
        best = d;
        if ((long long)units * d >= target) return d;
    }
    return best;
}

namespace {

// ------------------------------------------------------------------ prep
// One warp per token (tokens w, w + 4, ...), no block barriers after the
// router row has landed.  Lane l holds the row's 8-column units u0 + l +
// 32 i, i < 8, of a 2048-column chunk; with one chunk (H <= 2048) the row is
// read once, otherwise each chunk is read in turn (twice with the pre-norm:
// once for the norm).  At most 80 registers a thread: next to a layer kernel
// of the previous call (576 threads x 96) the SM has 128 x 80 left, so the
// next layer's prep can stage its router row while that kernel runs.
constexpr int kPrepUnits = 8;            // units per lane per chunk
constexpr int kChunkUnits = kPrepUnits * 32;

__device__ __forceinline__ void prep_load(const uint16_t* xr, int u0, int H8, int lane,
                                          uint4 (&v)[kPrepUnits]) {
#pragma unroll
    for (int i = 0; i < kPrepUnits; ++i) {
        const int u = u0 + lane + 32 * i;
        v[i] = u < H8 ? __ldcg(reinterpret_cast<const uint4*>(xr) + u) : make_uint4(0u, 0u, 0u, 0u);
    }
}

__device__ __forceinline__ void unpack8(const uint4 v, float (&xf)[8]) {
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        xf[2 * p] = __uint_as_float(wv[p] << 16);
        xf[2 * p + 1] = __uint_as_float(wv[p] & 0xffff0000u);
    }
}

__global__ void __maxnreg__(80) decode_prep_kernel(const PrepArgs a) {
    extern __shared__ __align__(128) uint8_t psm[];  // this CTA's router row [H] fp32
    __shared__ __align__(8) uint64_t s_bar;
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int e = blockIdx.x, H = a.H, T = a.T;
    const uint32_t bar = smem_u32(&s_bar);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, (uint32_t)(H * 4));
        bulk_g2s(smem_u32(psm), a.wr + (size_t)e * H, (uint32_t)(H * 4), bar);
    }
    __syncthreads();
    pdl_wait();     // x and the workspace belong to this call from here on
    pdl_trigger();  // the layer kernel may be scheduled; it waits for our end
    for (int i = e * kPrepThreads + tid; i < a.nsync; i += gridDim.x * kPrepThreads) a.sync[i] = 0;
    const int H8 = H / 8, G32 = H / kGroup;
    const int nw = kPrepThreads / 32, nchunk = (H8 + kChunkUnits - 1) / kChunkUnits;
    const bool one = nchunk == 1;
    uint4 cur[kPrepUnits];
    if (!mbar_wait(bar, 0)) record_status(a.status, kStatusTimeout);
    const float* w = reinterpret_cast<const float*>(psm);
    for (int t = warp; t < T; t += nw) {
        const uint16_t* xr = a.x + (size_t)t * H;
        if (one) prep_load(xr, 0, H8, lane, cur);
        float r = 1.0f;
        if (a.prenorm) {
            // the same order and rounding as the prefill RMSNorm: each lane
            // over its columns in order, then a butterfly
            float ss = 0.f;
            for (int ch = 0; ch < nchunk; ++ch) {
                if (!one) prep_load(xr, ch * kChunkUnits, H8, lane, cur);
#pragma unroll
                for (int i = 0; i < kPrepUnits; ++i) {
                    float xf[8];
                    unpack8(cur[i], xf);
#pragma unroll
                    for (int q = 0; q < 8; ++q) ss = fmaf(xf[q], xf[q], ss);
                }
            }
            ss = warp_sum(ss);
            r = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, (float)H) + 1e-6f));
        }
        const bool duty = (t % (int)gridDim.x) == e;  // this CTA writes token t's codes
        float acc = 0.f;
        for (int ch = 0; ch < nchunk; ++ch) {
            if (!one) prep_load(xr, ch * kChunkUnits, H8, lane, cur);
#pragma unroll
            for (int i = 0; i < kPrepUnits; ++i) {
                const int u = ch * kChunkUnits + lane + 32 * i;
                const bool valid = u < H8;
                float xf[8];
                unpack8(cur[i], xf);
                if (a.prenorm) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) xf[q] = bf16_bits_to_float(float_to_bf16_bits(xf[q] * r));
                }
                if (valid) {
                    const float4 w0 = *reinterpret_cast<const float4*>(w + u * 8);
                    const float4 w1 = *reinterpret_cast<const float4*>(w + u * 8 + 4);
                    acc = fmaf(xf[0], w0.x, acc);
                    acc = fmaf(xf[1], w0.y, acc);
                    acc = fmaf(xf[2], w0.z, acc);
                    acc = fmaf(xf[3], w0.w, acc);
                    acc = fmaf(xf[4], w1.x, acc);
                    acc = fmaf(xf[5], w1.y, acc);
                    acc = fmaf(xf[6], w1.z, acc);
                    acc = fmaf(xf[7], w1.w, acc);
                }
                if (duty) {
                    // int8 codes per 32 columns: lanes 4m..4m+3 hold one group
                    float amax = 0.f;
#pragma unroll
                    for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(xf[q]));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
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
                    gsum += __shfl_xor_sync(0xffffffffu, gsum, 1);
                    gsum += __shfl_xor_sync(0xffffffffu, gsum, 2);
                    if (valid) {
                        *reinterpret_cast<uint2*>(a.xq + (size_t)t * H + u * 8) = permute_chunk(lo, hi);
                        *reinterpret_cast<uint2*>(a.q_x + (size_t)t * H + u * 8) = make_uint2(lo, hi);
                        if ((lane & 3) == 0) {
                            a.xs[t * G32 + u / 4] = make_int2(__float_as_int(d), -8 * gsum);
                            a.d_x[t * G32 + u / 4] = db;
                        }
                    }
                }
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) a.logits[(size_t)t * a.E + e] = acc;
    }
}

// ----------------------------------------------------------------- layer
__global__ void __maxnreg__(96) decode_layer_kernel(const LayerArgs a) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ int s_idx[kMaxTk];
    __shared__ float s_w[kMaxTk];
    __shared__ int s_btok[kMaxTk];    // bucket row -> token
    __shared__ float s_bsw[kMaxTk];   // bucket row -> routing weight
    __shared__ int s_slotpos[kMaxTk]; // (t, j) -> bucket row
    __shared__ uint32_t s_mask[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_touched[kMaxExperts];
    __shared__ int s_slot_tile[kMaxRing];  // the latest tile issued into each slot (both rings)
    __shared__ int s_nt;
    __shared__ volatile int s_abort;
    __shared__ volatile int s_flag[kGroups];

    const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k;
    const int KBg = H / kTileK, KBd = I / kTileK;
    const int RBg = 2 * I / kTileRows, RBd = H / kTileRows, RBh = I / kTileRows;
    const int Gx = H / kGroup, Gh = I / kGroup;
    const int Tk = T * k, ns = a.ns;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int G = gridDim.x, b = blockIdx.x;
    const uint32_t sbase = smem_u32(dsm);
    const uint32_t bar0 = sbase + a.off_bar;
    // group g's ring: slots g*ns .. g*ns + ns - 1
    auto full_bar = [&](int g, int s) { return bar0 + 8u * (g * ns + s); };
    auto empty_bar = [&](int g, int s) { return bar0 + 8u * (2 * ns + g * ns + s); };
    auto slot_addr = [&](int g, int s) { return (uint32_t)((g * ns + s) * kTileBytes); };
    auto fail = [&]() {
        record_status(a.status, kStatusTimeout);
        s_abort = 1;
    };
    if (tid == 0) {
        for (int g = 0; g < kGroups; ++g) {
            for (int s = 0; s < ns; ++s) {
                mbar_init(full_bar(g, s), 1);
                mbar_init(empty_bar(g, s), kGroupWarps);
            }
        }
        s_abort = 0;
        fence_mbar_init();
    }
    for (int s = tid; s < kMaxRing; s += kLayerThreads) s_slot_tile[s] = -1;
    __syncthreads();
    pdl_wait();     // the prep kernel's logits, codes and cleared counters
    pdl_trigger();  // the next call's prep may be scheduled; it waits for our end

    // ---------------------------------------------- routing (every CTA)
    float* s_lg = reinterpret_cast<float*>(dsm);  // [T][E], in the (still unused) ring
    for (int i = tid; i < T * E; i += kLayerThreads) s_lg[i] = __ldcg(a.logits + i);
    for (int e = tid; e < E; e += kLayerThreads) s_mask[e] = 0u;
    __syncthreads();
    if (warp < kConsumerWarps) {
        for (int t = warp; t < T; t += kConsumerWarps) {
            int si;
            float sw;
            warp_topk(s_lg + t * E, E, k, si, sw);
            if (lane < k) {
                s_idx[t * k + lane] = si;
                s_w[t * k + lane] = sw;
            }
        }
    }
    __syncthreads();
    // token t's bit in the mask of each expert it chose (T <= 32)
    for (int p = tid; p < Tk; p += kLayerThreads) atomicOr(&s_mask[s_idx[p]], 1u << (p / k));
    __syncthreads();
    if (warp == 0) {
        // experts 8*lane .. 8*lane+7 (E <= 256): bucket offsets and the
        // touched list (ascending expert order) by a warp scan
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
                if (cnt[i] > 0) s_touched[pos++] = e;
                off += cnt[i];
            }
        }
        if (lane == 31) {
            s_off[E] = itot;
            s_nt = itch;
        }
    }
    __syncthreads();
    const int nt = s_nt;
    for (int p = tid; p < Tk; p += kLayerThreads) {
        const int t = p / k, e = s_idx[p];
        const int pos = s_off[e] + __popc(s_mask[e] & ((1u << t) - 1u));
        s_btok[pos] = t;
        s_bsw[pos] = s_w[p];
        s_slotpos[p] = pos;
        if (b == 0) {
            a.topk_idx[p] = e;
            a.topk_w[p] = s_w[p];
            a.bucket_token[pos] = t;
            a.bucket_slot[pos] = p % k;
        }
    }
    if (b == 0) {
        for (int i = tid; i <= E; i += kLayerThreads) a.offsets[i] = s_off[i];
        for (int i = tid; i < nt; i += kLayerThreads) a.touched[i] = s_touched[i];
        if (tid == 0) a.counters[kCntTouched] = nt;
    }
    // the ring held the logits through generic accesses; bulk copies refill it
    fence_proxy_async_smem();
    __syncthreads();

    // ------------------------------------------------------- work split
    const int nsg = decode_split_for(nt * RBg, KBg, kTargetGU, a.cap_g);
    const int nsd = decode_split_for(nt * RBd, KBd, kTargetD, a.cap_d);
    const int KCg = KBg / nsg, KCd = KBd / nsd;
    const int n_gu = nt * RBg * nsg, n_dn = nt * RBd * nsd;
    const int gu0 = (int)((long long)b * n_gu / G), gu1 = (int)((long long)(b + 1) * n_gu / G);
    const int dn0 = (int)((long long)b * n_dn / G), dn1 = (int)((long long)(b + 1) * n_dn / G);
    const int ngl = gu1 - gu0, ndl = dn1 - dn0;  // this CTA's tasks: gate/up, then down
    // The CTA's task list (local index j: gate/up tasks j < ngl, then down
    // tasks) is cut in two contiguous halves of about equal tile count, one
    // per consumer group, so that each group meets runs of tasks that share a
    // counter (consecutive K parts of one row block) and counts a run once.
    auto tile0 = [&](int j) { return j < ngl ? j * KCg : ngl * KCg + (j - ngl) * KCd; };
    const int nloc = ngl + ndl, half = (tile0(nloc) + 1) / 2;
    int jm = half <= ngl * KCg ? (half + KCg - 1) / KCg
                               : ngl + (half - ngl * KCg + KCd - 1) / KCd;
    jm = jm > nloc ? nloc : jm;
    // the cut nearest the middle: one task earlier if that splits more evenly
    if (jm > 0 && 2 * tile0(jm - 1) >= 2 * tile0(nloc) - 2 * tile0(jm)) --jm;
    auto jbeg = [&](int g) { return g == 0 ? 0 : jm; };
    auto jend = [&](int g) { return g == 0 ? jm : nloc; };

    if (warp >= kWarpProducer0) {
        // ---------------------------------------------------------- producer
        // The group's tiles in its consumption order: the first ring's worth
        // by all lanes at once (every slot starts free), then the rest in
        // order by one lane, each waiting for its slot, which held the tile
        // ns earlier (already issued), so a parity wait never aliases.
        const int g = warp - kWarpProducer0;
        const int t0 = tile0(jbeg(g)), nq = tile0(jend(g)) - t0;
        auto issue = [&](int q) -> bool {
            const int t = t0 + q;
            const uint8_t* src;
            if (t < ngl * KCg) {
                const int task = gu0 + t / KCg, u = t % KCg;
                const int i = task / (RBg * nsg), rem = task % (RBg * nsg);
                src = a.wgu + (((size_t)s_touched[i] * RBg + rem / nsg) * KBg + (rem % nsg) * KCg + u) *
                                  kTileBytes;
            } else {
                const int td = t - ngl * KCg;
                const int task = dn0 + td / KCd, u = td % KCd;
                const int i = task / (RBd * nsd), rem = task % (RBd * nsd);
                src = a.wd + (((size_t)s_touched[i] * RBd + rem / nsd) * KBd + (rem % nsd) * KCd + u) *
                                 kTileBytes;
            }
            const int s = q % ns;
            if (s_abort || !mbar_wait(empty_bar(g, s), ((q / ns) & 1) ^ 1) || s_abort) {
                fail();
                return false;
            }
            s_slot_tile[g * ns + s] = q;
            mbar_arrive_expect_tx(full_bar(g, s), (uint32_t)kTileBytes);
            bulk_g2s(sbase + slot_addr(g, s), src, (uint32_t)kTileBytes, full_bar(g, s));
            return true;
        };
        const int nfirst = nq < ns ? nq : ns;
        bool ok = true;
        for (int q = lane; q < nfirst; q += 32) ok = ok && issue(q);
        if (__all_sync(0xffffffffu, ok) && lane == 0)
            for (int q = nfirst; q < nq; ++q)
                if (!issue(q)) break;
        // every copy issued lands before the CTA can go away: wait for the
        // latest use of each slot (earlier uses completed before it)
        __syncwarp();
        for (int s = lane; s < ns; s += 32) {
            const int q = s_slot_tile[g * ns + s];
            if (q >= 0) mbar_wait(full_bar(g, s), (q / ns) & 1);
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
    {
        // the int8 codes of x (and their scales), written by the prep kernel
        const int n16 = (T * H + T * Gx * 8) / 16;
        const uint4* src = reinterpret_cast<const uint4*>(a.xq);
        uint4* dst = reinterpret_cast<uint4*>(ax_q);
        for (int i = tid; i < n16; i += kConsumerThreads) dst[i] = __ldcg(src + i);
        named_sync(1, kConsumerThreads);
    }
    // Control flow must stay uniform within a group (it shares named
    // barriers): a failed wait only skips work; decisions the group shares
    // are taken by its thread 0 and read after a group barrier.
    bool live = true;  // this warp has not given up
    auto slot_ready = [&](int q) -> bool {
        if (!live) return false;
        if (s_abort || !mbar_wait(full_bar(grp, q % ns), (q / ns) & 1)) {
            fail();
            live = false;
        }
        return live;
    };
    const int r_lane = lane >> 1, h_lane = lane & 1;
    const int lrow = w8 * 16 + r_lane;  // this lane's row in the 128-row block

    // One task: rows rb*128 + lrow, 64-column blocks kb0 .. kb0 + KC - 1 of
    // the current expert (bucket rows off .. off + c - 1, NT >= c), tiles q0 ..
    // of the group's sequence.  The lane pair's sum for bucket row off + n is stored at
    // dst[n * ld] (down: times the row's routing weight).
    auto run_tiles = [&](auto ntc, bool gu, int off, int c, int q0, int kb0, int KC, int row,
                         float* dst, size_t ld) {
        constexpr int NT = decltype(ntc)::value;
        const uint8_t* aq = gu ? ax_q : ah_q;
        const int2* as = gu ? ax_s : ah_s;
        const int K = gu ? H : I, Gk = gu ? Gx : Gh;
        int32_t* dots = gu ? a.dots_gu : a.dots_d;
        const size_t dots_ld = gu ? (size_t)2 * I : (size_t)H;
        float acc[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n] = 0.f;
        for (int u = 0; u < KC; ++u) {
            const int q = q0 + u;
            if (!slot_ready(q)) continue;
            const uint8_t* tile = dsm + slot_addr(grp, q % ns);
            const uint4 wv = *reinterpret_cast<const uint4*>(tile + w8 * 512 + lane * 16);
            const float dw = half_bits_to_float(
                *reinterpret_cast<const uint16_t*>(tile + kTileCodeBytes + w8 * 64 + lane * 2));
            const uint32_t wl[4] = {wv.x & 0x0F0F0F0Fu, wv.y & 0x0F0F0F0Fu, wv.z & 0x0F0F0F0Fu,
                                    wv.w & 0x0F0F0F0Fu};
            const uint32_t wh[4] = {(wv.x >> 4) & 0x0F0F0F0Fu, (wv.y >> 4) & 0x0F0F0F0Fu,
                                    (wv.z >> 4) & 0x0F0F0F0Fu, (wv.w >> 4) & 0x0F0F0F0Fu};
            const int g = 2 * (kb0 + u) + h_lane;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (n < c) {
                    const int ar = gu ? s_btok[off + n] : n;
                    const int2 sc = as[ar * Gk + g];
                    const int dot = group_dot(wl, wh, aq + (size_t)ar * K + g * kGroup, sc.y);
                    acc[n] = fmaf((float)dot, dw * __int_as_float(sc.x), acc[n]);
                    if (dots) dots[((size_t)(off + n) * dots_ld + row) * Gk + g] = dot;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(grp, q % ns));  // the tile is consumed
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const float v = acc[n] + __shfl_xor_sync(0xffffffffu, acc[n], 1);
            if (n < c && h_lane == 0 && live) dst[n * ld] = gu ? v : v * s_bsw[off + n];
        }
    };
    auto dispatch = [&](bool gu, int off, int c, int q0, int kb0, int KC, int row, float* dst,
                        size_t ld) {
        if (c <= 1) run_tiles(IntC<1>{}, gu, off, c, q0, kb0, KC, row, dst, ld);
        else if (c <= 2) run_tiles(IntC<2>{}, gu, off, c, q0, kb0, KC, row, dst, ld);
        else if (c <= 4) run_tiles(IntC<4>{}, gu, off, c, q0, kb0, KC, row, dst, ld);
        else if (c <= 8) run_tiles(IntC<8>{}, gu, off, c, q0, kb0, KC, row, dst, ld);
        else if (c <= 16) run_tiles(IntC<16>{}, gu, off, c, q0, kb0, KC, row, dst, ld);
        else run_tiles(IntC<MOE_DECODE_MAX_T>{}, gu, off, c, q0, kb0, KC, row, dst, ld);
    };
    // Adds a run's `add` finished tasks to `counter` (one release + acquire
    // atomic by one thread, after the group barrier that orders the run's
    // stores) and tells the group whether the run completed the `target`:
    // then the group goes on with the follow-up work, reading what the other
    // tasks stored.
    auto flush = [&](int* counter, int add, int target) -> bool {
        group_sync();
        if (gtid == 0) s_flag[grp] = (atom_add_acq_rel_gpu(counter, add) + add == target) ? 1 : 0;
        group_sync();
        return s_flag[grp] != 0;
    };

    const int jb = jbeg(grp), je = jend(grp), qb = tile0(jb);
    int h_expert = -1;  // touched slot whose h is in this group's buffer
    int run = 0;        // tasks of the current run counted so far
    for (int j = jb; j < je; ++j) {
        if (j < ngl) {
            // ------------------------------------------ gate/up task
            const int task = gu0 + j;
            const int i = task / (RBg * nsg), rem = task % (RBg * nsg);
            const int rb = rem / nsg, kc = rem % nsg;
            const int e = s_touched[i], off = s_off[e], c = s_off[e + 1] - off;
            const int row = rb * kTileRows + lrow;
            dispatch(true, off, c, tile0(j) - qb, kc * KCg, KCg, row,
                     a.gu_part + ((size_t)kc * Tk + off) * 2 * I + row, (size_t)2 * I);
            ++run;
            // the run goes on while the next task counts toward the same h block
            const int hb = rb % RBh;
            if (j + 1 < je && j + 1 < ngl && (task + 1) / (RBg * nsg) == i &&
                ((task + 1) % (RBg * nsg)) / nsg % RBh == hb)
                continue;
            const int add = run;
            run = 0;
            if (!flush(&a.cnt_h[i * RBh + hb], add, 2 * nsg)) continue;
            // the last run of h block hb: h = silu(g) * u over the K parts in
            // order, int8 per 32 features.  A warp takes four groups at once,
            // eight lanes a group, four features a lane.
            const int sub = lane / 8, l8 = lane % 8;
            for (int q0 = w8 * 4; q0 < 4 * c; q0 += 4 * kGroupWarps) {
                const int q = q0 + sub;
                const bool ok = q < 4 * c;
                const int n = ok ? q / 4 : 0, gg = ok ? q % 4 : 0;
                const int f0 = hb * kTileRows + gg * kGroup + l8 * 4;
                float gv[4] = {0.f, 0.f, 0.f, 0.f}, uv[4] = {0.f, 0.f, 0.f, 0.f};
                if (ok) {
                    for (int p = 0; p < nsg; ++p) {
                        const float* src = a.gu_part + ((size_t)p * Tk + off + n) * 2 * I + f0;
                        const float4 g4 = __ldcg(reinterpret_cast<const float4*>(src));
                        const float4 u4 = __ldcg(reinterpret_cast<const float4*>(src + I));
                        gv[0] += g4.x; gv[1] += g4.y; gv[2] += g4.z; gv[3] += g4.w;
                        uv[0] += u4.x; uv[1] += u4.y; uv[2] += u4.z; uv[3] += u4.w;
                    }
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
                // lanes 2m and 2m+1 hold columns 8m..8m+3 and 8m+4..8m+7 of
                // the group: the even lane stores the chunk in dp4a order
                const uint32_t w4o = __shfl_xor_sync(0xffffffffu, w4, 1);
                if (ok) {
                    const size_t prow = (size_t)(off + n);
                    if ((l8 & 1) == 0)
                        *reinterpret_cast<uint2*>(a.hq + prow * I + f0) = permute_chunk(w4, w4o);
                    if (l8 == 0) a.hs[prow * Gh + f0 / kGroup] = make_int2(__float_as_int(d), -8 * sum);
                    if (a.write_qh) {
                        *reinterpret_cast<uint32_t*>(a.q_h + prow * I + f0) = w4;
                        if (l8 == 0) a.d_h[prow * Gh + f0 / kGroup] = db;
                    }
                }
            }
            group_sync();
            if (gtid == 0) red_release_add(&a.done_h[i], 1);
        } else {
            // --------------------------------------------- down task
            const int task = dn0 + (j - ngl);
            const int i = task / (RBd * nsd), rem = task % (RBd * nsd);
            const int rbd = rem / nsd, kc = rem % nsd;
            const int e = s_touched[i], off = s_off[e], c = s_off[e + 1] - off;
            if (i != h_expert) {
                // wait until every h block of the expert is done, then load h
                if (gtid == 0) {
                    bool got = !s_abort;
                    if (got && ld_acquire(&a.done_h[i]) < RBh) {
                        const unsigned long long t0 = globaltimer_ns();
                        while (ld_acquire(&a.done_h[i]) < RBh) {
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
                if (s_flag[grp]) {
                    const int nq = c * I / 16, ns16 = c * Gh * 8 / 16;
                    const uint4* srcq = reinterpret_cast<const uint4*>(a.hq + (size_t)off * I);
                    const uint4* srcs = reinterpret_cast<const uint4*>(a.hs + (size_t)off * Gh);
                    for (int z = gtid; z < nq; z += kGroupThreads)
                        reinterpret_cast<uint4*>(ah_q)[z] = __ldcg(srcq + z);
                    for (int z = gtid; z < ns16; z += kGroupThreads)
                        reinterpret_cast<uint4*>(ah_s)[z] = __ldcg(srcs + z);
                } else {
                    live = false;  // nothing valid to multiply: skip the rest
                }
                group_sync();
                h_expert = i;
            }
            const int row = rbd * kTileRows + lrow;
            dispatch(false, off, c, tile0(j) - qb, kc * KCd, KCd, row,
                     a.y_part + ((size_t)kc * Tk + off) * H + row, (size_t)H);
            ++run;
            // the run goes on while the next task counts toward the same columns
            if (j + 1 < je && (task + 1) % (RBd * nsd) / nsd == rbd && (task + 1) / (RBd * nsd) == i)
                continue;
            const int add = run;
            run = 0;
            if (!flush(&a.cnt_y[rbd], add, nt * nsd)) continue;
            // the last run of output columns rbd*128 .. +127: residual plus
            // every slot's parts, slots in order, K parts in order
            const int c0 = rbd * kTileRows;
            for (int it = gtid; it < kTileRows * T; it += kGroupThreads) {
                const int t = it / kTileRows, col = c0 + it % kTileRows;
                float v = bf16_bits_to_float(a.x_res[(size_t)t * H + col]);
                for (int jj = 0; jj < k; ++jj) {
                    const int p = s_slotpos[t * k + jj];
                    for (int kp = 0; kp < nsd; ++kp) v += __ldcg(a.y_part + ((size_t)kp * Tk + p) * H + col);
                }
                if (a.out_fp32)
                    static_cast<float*>(a.out)[(size_t)t * H + col] = v;
                else
                    static_cast<uint16_t*>(a.out)[(size_t)t * H + col] = float_to_bf16_bits(v);
            }
        }
    }
}

// ---------------------------------------------------------------- launch
int g_layer_pdl[64] = {};  // 0 unknown, 1 cooperative + PDL accepted, 2 cooperative only

struct Plan {
    int ns, off_bar, off_ax, off_ah, ah_bytes, smem;
};

int al128(long long v) { return (int)((v + 127) & ~127ll); }

// Shared-memory plan of the layer kernel; false if it does not fit.
bool plan_layer(int T, int H, int I, int E, Plan* p) {
    const long long ax = al128((long long)T * H + (long long)T * (H / kGroup) * 8);
    const long long ah = al128((long long)T * I + (long long)T * (I / kGroup) * 8);
    const long long rest = kLayerSmemBudget - ax - 2 * ah - 2 * kMaxRing * 8 - 128;
    if (rest < 2ll * kGroups * kTileBytes) return false;
    int ns = (int)(rest / kTileBytes) / kGroups;  // slots of each group's ring
    ns = ns > kMaxRing / kGroups ? kMaxRing / kGroups : ns;
    // the routing phase keeps all T x E logits in the rings
    if ((long long)T * E * 4 > (long long)kGroups * ns * kTileBytes) return false;
    p->ns = ns;
    p->off_bar = kGroups * ns * kTileBytes;
    p->off_ax = al128(p->off_bar + 2 * kGroups * ns * 8);
    p->off_ah = p->off_ax + (int)ax;
    p->ah_bytes = (int)ah;
    p->smem = p->off_ah + 2 * (int)ah;
    return true;
}

__global__ void coop_pdl_probe_kernel(int* p) {
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
    cudaStreamDestroy(st);
    return cudaSuccess;
}

int cooperative_pdl_mode(int dev) { return g_layer_pdl[dev & 63]; }

bool decode_shape_fits(int T, int H, int I, int E) {
    Plan p;
    return plan_layer(T, H, I, E, &p);
}

void decode_split_bounds(int T, int H, int I, int E, int k, int* cap_g, int* cap_d, int* nsg_max,
                         int* nsd_max) {
    const size_t Tk = (size_t)T * k;
    const int KBg = H / kTileK, KBd = I / kTileK;
    auto cap = [](size_t row_bytes) {
        size_t c = row_bytes ? kPartBudget / row_bytes : kMaxSplit;
        return (int)std::max<size_t>(1, std::min<size_t>(c, kMaxSplit));
    };
    *cap_g = cap(Tk * 2 * I * 4);
    *cap_d = cap(Tk * H * 4);
    // the split only shrinks as more experts are touched, and at least k are
    const int nt_min = std::max(1, std::min(k, E));
    *nsg_max = decode_split_for(nt_min * (2 * I / kTileRows), KBg, kTargetGU, *cap_g);
    *nsd_max = decode_split_for(nt_min * (H / kTileRows), KBd, kTargetD, *cap_d);
}

int decode_sync_ints(int T, int H, int I, int E, int k) {
    const int nslot = std::min(E, T * k);
    return nslot * (I / kTileRows) + nslot + H / kTileRows;
}

cudaError_t launch_decode(const uint16_t* x, const float* wr, const void* wgu, const void* wd,
                          int T, int H, int I, int E, int k, bool prenorm, bool out_fp32,
                          void* out, const Workspace& ws, int32_t* dots_gu, int32_t* dots_d,
                          bool write_qh, int* status, int num_sms, void** ev, bool capturing,
                          cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    Plan plan;
    if (!plan_layer(T, H, I, E, &plan)) return cudaErrorInvalidValue;
    cudaError_t err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    auto mark = [&](int i) -> cudaError_t {
        return (ev && ev[i]) ? record_stage(ev[i], s, capturing) : cudaSuccess;
    };
    const int nslot = std::min(E, T * k);
    // ---- prep ----
    PrepArgs p{};
    p.x = x;
    p.wr = wr;
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
    const int psmem = H * 4;
    if (psmem > 48 * 1024 &&
        (err = cudaFuncSetAttribute(decode_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    psmem)) != cudaSuccess)
        return err;
    if ((err = launch_pdl(decode_prep_kernel, dim3(E), dim3(kPrepThreads), psmem, s, p)) != cudaSuccess)
        return err;
    if ((err = mark(1)) != cudaSuccess) return err;
    // ---- layer ----
    LayerArgs a{};
    a.x_res = x;
    a.wgu = static_cast<const uint8_t*>(wgu);
    a.wd = static_cast<const uint8_t*>(wd);
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
    a.hq = ws.hq;
    a.hs = ws.hs;
    a.q_h = ws.q_h;
    a.d_h = ws.d_h;
    a.y_part = ws.y_part;
    a.cnt_h = ws.sync;
    a.done_h = ws.sync + nslot * (I / kTileRows);
    a.cnt_y = a.done_h + nslot;
    a.cap_g = ws.cap_g;
    a.cap_d = ws.cap_d;
    a.out = out;
    a.out_fp32 = out_fp32 ? 1 : 0;
    a.dots_gu = dots_gu;
    a.dots_d = dots_d;
    a.write_qh = write_qh ? 1 : 0;
    a.status = status;
    a.ns = plan.ns;
    a.off_bar = plan.off_bar;
    a.off_ax = plan.off_ax;
    a.off_ah = plan.off_ah;
    a.ah_bytes = plan.ah_bytes;
    // (32-bit task indices: the api checks T * k * max(H, I) < 2^31, which
    // bounds touched experts x row blocks x splits far below it)
    err = cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               plan.smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[2];
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kLayerThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = (g_layer_pdl[dev & 63] == 2) ? 1 : 2;
    if ((err = cudaLaunchKernelEx(&cfg, decode_layer_kernel, a)) != cudaSuccess) return err;
    for (int i = 2; i <= 6; ++i)
        if ((err = mark(i)) != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moeq4
