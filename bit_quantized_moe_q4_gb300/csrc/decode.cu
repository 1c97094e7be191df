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
constexpr int kMaxSlots = 12;                           // slots of both groups' rings
constexpr int kRedBytes = kGroupWarps * 32 * 32;        // per group: 8 warps x 32 lanes x 8 floats
// Dynamic shared memory of the layer kernel: leaves room on the SM (228 KB)
// for its static part (13.1 KB) and a prep CTA of the next call (its router
// row, 8 KB at H = 2048) next to it.
constexpr int kLayerSmemBudget = 200 * 1024;
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
// MAXNT: the most tokens an expert's bucket may hold (T <= MAXNT).  At most
// 96 registers a thread, which leaves room on the SM for the next call's
// prep CTA; the MAXNT = 32 variant spills a little instead (it only runs
// when more than 16 tokens are decoded at once).
template <int MAXNT>
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
    __shared__ int s_slot_chunk[kMaxSlots];  // the latest chunk issued into each slot (both rings)
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
    const int st = a.st;
    auto slot_addr = [&](int g, int s) { return (uint32_t)((g * ns + s) * st * kTileBytes); };
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
    for (int s = tid; s < kMaxSlots; s += kLayerThreads) s_slot_chunk[s] = -1;
    __syncthreads();
    pdl_wait();     // the prep kernel's logits, codes and cleared counters
    pdl_trigger();  // the next call's prep may be scheduled; it waits for our end
    if (warp < kConsumerWarps) {
        // the int8 codes of x and their scales (written by the prep kernel)
        // start on their way to shared memory while the CTA routes
        const int n16 = (T * H + T * Gx * 8) / 16;
        const uint8_t* src = a.xq;
        for (int i = tid; i < n16; i += kConsumerThreads)
            cp_async16(sbase + a.off_ax + 16 * i, src + 16 * (size_t)i);
    }

    // ---------------------------------------------- routing (every CTA)
    float* s_lg = reinterpret_cast<float*>(dsm);  // [T][E], in the (still idle) rings and buffers
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
    // K splits: the smallest divisor of the row's 64-column blocks (up to
    // the cap, listed by the host in ascending order) that gives enough
    // tasks, else the largest.
    int nsg = a.div_g[a.ndiv_g - 1], nsd = a.div_d[a.ndiv_d - 1];
    for (int q = 0; q < a.ndiv_g; ++q)
        if (nt * RBg * a.div_g[q] >= kTargetGU) { nsg = a.div_g[q]; break; }
    for (int q = 0; q < a.ndiv_d; ++q)
        if (nt * RBd * a.div_d[q] >= kTargetD) { nsd = a.div_d[q]; break; }
    const int KCg = KBg / nsg, KCd = KBd / nsd;
    const int n_gu = nt * RBg * nsg, n_dn = nt * RBd * nsd;  // (x G fits in 32 bits: checked at launch)
    const int gu0 = b * n_gu / G, gu1 = (b + 1) * n_gu / G;
    const int dn0 = b * n_dn / G, dn1 = (b + 1) * n_dn / G;
    const int ngl = gu1 - gu0, ndl = dn1 - dn0;  // this CTA's tasks: gate/up, then down
    // Each group takes a contiguous half of the gate/up tasks, then a
    // contiguous half of the down tasks, so both groups are in the same
    // phase and each meets runs of tasks that share a counter.
    const int gh = (ngl + 1) / 2, dh = ndl / 2;

    // A walk over one group's tasks in order: gate/up tasks (expert slot i,
    // row block rb, K part kc), then down tasks (i, row block rb, K part kc),
    // advanced by counting (no division per step).
    struct Walk {
        int left_g, left_d;  // tasks left in each phase
        int i, rb, kc;       // the current task
        bool gu;
    };
    auto walk_start = [&](int g) {
        Walk w;
        w.left_g = g == 0 ? gh : ngl - gh;
        w.left_d = g == 0 ? dh : ndl - dh;
        w.gu = w.left_g > 0;
        const int t = w.gu ? gu0 + (g == 0 ? 0 : gh) : dn0 + (g == 0 ? 0 : dh);
        const int per = w.gu ? RBg * nsg : RBd * nsd, ns_ = w.gu ? nsg : nsd;
        w.i = t / per;
        w.rb = (t % per) / ns_;
        w.kc = t % ns_;
        return w;
    };
    auto walk_next = [&](Walk w, int g) {
        if (w.gu) {
            if (--w.left_g > 0) {
                if (++w.kc == nsg) { w.kc = 0; if (++w.rb == RBg) { w.rb = 0; ++w.i; } }
            } else if (w.left_d > 0) {  // on to the group's first down task
                w.gu = false;
                const int t = dn0 + (g == 0 ? 0 : dh);
                w.i = t / (RBd * nsd);
                w.rb = (t % (RBd * nsd)) / nsd;
                w.kc = t % nsd;
            }
        } else {
            --w.left_d;
            if (++w.kc == nsd) { w.kc = 0; if (++w.rb == RBd) { w.rb = 0; ++w.i; } }
        }
        return w;
    };
    auto walk_live = [&](const Walk& w) { return w.gu ? w.left_g > 0 : w.left_d > 0; };
    auto walk_base = [&](const Walk& w) -> const uint8_t* {
        return w.gu ? a.wgu + (((size_t)s_touched[w.i] * RBg + w.rb) * KBg + (size_t)w.kc * KCg) * kTileBytes
                    : a.wd + (((size_t)s_touched[w.i] * RBd + w.rb) * KBd + (size_t)w.kc * KCd) * kTileBytes;
    };

    // Chunks: the group's tiles, in sequence order, are cut into runs of up
    // to st tiles that lie back to back in memory (one bulk copy, one ring
    // slot each).  Producer and consumers apply the same rule to the same
    // sequence: a tile opens a new chunk unless it directly follows the
    // open chunk's last tile and the chunk has room.  Slot and phase advance
    // by counting.
    if (warp >= kWarpProducer0) {
        // ---------------------------------------------------------- producer
        // One lane issues the chunks in order; chunk c's slot held chunk
        // c - ns, issued before it, so a parity wait never aliases.
        const int g = warp - kWarpProducer0;
        if (lane == 0) {
            int slot = -1, phase = 0, clen = 0, cidx = -1;
            const uint8_t* caddr = nullptr;
            bool ok = true;
            auto issue = [&]() -> bool {
                if (s_abort || !mbar_wait(empty_bar(g, slot), phase ^ 1) || s_abort) {
                    fail();
                    return false;
                }
                s_slot_chunk[g * ns + slot] = cidx;
                mbar_arrive_expect_tx(full_bar(g, slot), (uint32_t)(clen * kTileBytes));
                bulk_g2s(sbase + slot_addr(g, slot), caddr, (uint32_t)(clen * kTileBytes), full_bar(g, slot));
                return true;
            };
            for (Walk w = walk_start(g); walk_live(w) && ok; w = walk_next(w, g)) {
                const uint8_t* base = walk_base(w);
                const int KC = w.gu ? KCg : KCd;
                for (int u = 0; u < KC; ++u) {
                    const uint8_t* t = base + (size_t)u * kTileBytes;
                    if (cidx < 0 || clen == st || t != caddr + (size_t)clen * kTileBytes) {
                        if (cidx >= 0 && !(ok = issue())) break;
                        ++cidx;
                        if (++slot == ns) { slot = 0; phase ^= 1; }
                        clen = 0;
                        caddr = t;
                    }
                    ++clen;
                }
            }
            if (ok && cidx >= 0) issue();
        }
        // every copy issued lands before the CTA can go away: wait for the
        // latest chunk of each slot (earlier ones completed before it)
        __syncwarp();
        for (int s = lane; s < ns; s += 32) {
            const int c = s_slot_chunk[g * ns + s];
            if (c >= 0) mbar_wait(full_bar(g, s), (c / ns) & 1);
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
    bool live = true;  // this warp has not given up
    int slot = -1, phase = 0, clen = 0, cidx = -1;  // the open chunk (same walk as the producer)
    const uint8_t* caddr = nullptr;
    const int r_lane = lane >> 1, h_lane = lane & 1;
    const int lrow = w8 * 16 + r_lane;  // this lane's row in the 128-row block

    // One task: rows rb*128 + lrow, 64-column blocks kb0 .. kb0 + KC - 1 of
    // the current expert (bucket rows off .. off + c - 1, NT >= c), packed
    // tiles base .. base + KC - 1; `next_contig`: the group's next tile lies
    // right after this task's last.  The lane pair's sum for bucket row
    // off + n is stored at dst[n * ld] (down: times the row's routing weight).
    auto run_tiles = [&](auto ntc, bool gu, int off, int c, const uint8_t* base, bool next_contig,
                         int kb0, int KC, int row, float* dst, size_t ld) {
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
            const uint8_t* tg = base + (size_t)u * kTileBytes;
            if (cidx < 0 || clen == st || tg != caddr + (size_t)clen * kTileBytes) {
                ++cidx;
                if (++slot == ns) { slot = 0; phase ^= 1; }
                clen = 0;
                caddr = tg;
                if (live && (s_abort || !mbar_wait(full_bar(grp, slot), phase))) {
                    fail();
                    live = false;
                }
            }
            const uint8_t* tile = dsm + slot_addr(grp, slot) + clen * kTileBytes;
            ++clen;
            if (live) {
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
            }
            // the chunk's last tile frees its slot
            if (clen == st || (u + 1 == KC && !next_contig)) {
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(grp, slot));
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const float v = acc[n] + __shfl_xor_sync(0xffffffffu, acc[n], 1);
            if (n < c && h_lane == 0 && live) dst[n * ld] = gu ? v : v * s_bsw[off + n];
        }
    };
    auto dispatch = [&](bool gu, int off, int c, const uint8_t* base, bool next_contig, int kb0,
                        int KC, int row, float* dst, size_t ld) {
        if (c <= 1) run_tiles(IntC<1>{}, gu, off, c, base, next_contig, kb0, KC, row, dst, ld);
        else if (c <= 2) run_tiles(IntC<2>{}, gu, off, c, base, next_contig, kb0, KC, row, dst, ld);
        else if (c <= 4) run_tiles(IntC<4>{}, gu, off, c, base, next_contig, kb0, KC, row, dst, ld);
        else if (c <= 8) run_tiles(IntC<8>{}, gu, off, c, base, next_contig, kb0, KC, row, dst, ld);
        else if (MAXNT <= 16 || c <= 16) run_tiles(IntC<16>{}, gu, off, c, base, next_contig, kb0, KC, row, dst, ld);
        else run_tiles(IntC<MAXNT>{}, gu, off, c, base, next_contig, kb0, KC, row, dst, ld);
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

    // The h of a down task's K range, from the gate/up K parts of its expert:
    // features f0 .. f0 + nf - 1 of bucket rows off .. off + c - 1, into this
    // group's buffer (int8 codes in dp4a order, {scale, -8 * sum} per 32).
    // The group's warps split the K parts (ps subsets) and the feature
    // quads, two K parts in flight a lane; the subsets' sums meet in shared
    // memory and are added in subset order.  Every down task of the range
    // computes the same codes.
    auto compute_h = [&](int off, int c, int f0, int nf, int nsg_, bool store) {
        const int ps = nsg_ >= 8 ? 8 : nsg_ >= 4 ? 4 : nsg_ >= 2 ? 2 : 1;
        const int sub = w8 % ps, blk = w8 / ps, nblk = kGroupWarps / ps;
        const int nq4 = c * nf / 4, q4_per_tok = nf / 4;
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

    int h_key = -1;  // (touched slot, K part) whose h is in this group's buffer
    int run = 0;     // tasks of the current run counted so far
    Walk w = walk_start(grp);
    while (walk_live(w)) {
        const Walk nx = walk_next(w, grp);
        const bool has_next = walk_live(nx);
        const uint8_t* base = walk_base(w);
        const int KC = w.gu ? KCg : KCd;
        const bool next_contig = has_next && walk_base(nx) == base + (size_t)KC * kTileBytes;
        const int i = w.i, rb = w.rb, kc = w.kc;
        const Walk cur = w;
        w = nx;
        const int e = s_touched[i], off = s_off[e], c = s_off[e + 1] - off;
        if (cur.gu) {
            // ------------------------------------------ gate/up task
            const int row = rb * kTileRows + lrow;
            dispatch(true, off, c, base, next_contig, kc * KCg, KCg, row,
                     a.gu_part + ((size_t)kc * Tk + off) * 2 * I + row, (size_t)2 * I);
            ++run;
            // the run goes on while the next task counts toward the same h
            // block (gate rows rb and up rows rb + RBh feed h block rb % RBh)
            const int hb = rb < RBh ? rb : rb - RBh;
            if (has_next && nx.gu && nx.i == i && (nx.rb < RBh ? nx.rb : nx.rb - RBh) == hb) continue;
            // count the run's K parts of h block hb (they are stored)
            group_sync();
            if (gtid == 0) red_release_add(&a.cnt_h[i * RBh + hb], run);
            run = 0;
        } else {
            // --------------------------------------------- down task
            const int rbd = rb;
            if (i * nsd + kc != h_key) {
                // wait until every gate/up K part of the h blocks this K range
                // overlaps is stored, then form h for the range
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
                    compute_h(off, c, f0, nf, nsg, a.write_qh && rbd == 0);
                } else {
                    live = false;  // nothing valid to multiply: skip the rest
                }
                group_sync();
                h_key = i * nsd + kc;
            }
            const int row = rbd * kTileRows + lrow;
            dispatch(false, off, c, base, next_contig, kc * KCd, KCd, row,
                     a.y_part + ((size_t)kc * Tk + off) * H + row, (size_t)H);
            ++run;
            // the run goes on while the next task counts toward the same columns
            if (has_next && nx.i == i && nx.rb == rbd) continue;
            const int add = run;
            run = 0;
            if (!flush(&a.cnt_y[rbd], add, nt * nsd)) continue;
            // the last run of output columns rbd*128 .. +127: residual plus
            // every slot's parts, slots in order, K parts in order (loaded
            // eight at a time before they are added)
            const int c0 = rbd * kTileRows;
            for (int it = gtid; it < kTileRows * T; it += kGroupThreads) {
                const int t = it / kTileRows, col = c0 + it % kTileRows;
                float v = bf16_bits_to_float(a.x_res[(size_t)t * H + col]);
                const float* yc = a.y_part + col;
                int jj = 0, kp = 0;  // slot and K part of the next load
                for (int q0 = 0; q0 < k * nsd; q0 += 8) {
                    float part[8];
#pragma unroll
                    for (int z = 0; z < 8; ++z) {
                        part[z] = 0.f;
                        if (jj < k) {
                            part[z] = __ldcg(yc + ((size_t)kp * Tk + s_slotpos[t * k + jj]) * H);
                            if (++kp == nsd) { kp = 0; ++jj; }
                        }
                    }
#pragma unroll
                    for (int z = 0; z < 8; ++z) v += part[z];  // (the padding adds 0)
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
    int ns, st, off_bar, off_ax, off_ah, ah_bytes, off_red, smem;
};

int al128(long long v) { return (int)((v + 127) & ~127ll); }

// Shared-memory plan of the layer kernel; false if it does not fit.
// Layout: the two rings, the two groups' h buffers and K-part sum buffers
// (all idle while the CTA routes, when they hold the logits), then the
// codes of x (filled by cp.async during routing) and the ring barriers.
bool plan_layer(int T, int H, int I, int E, Plan* p) {
    const long long ax = al128((long long)T * H + (long long)T * (H / kGroup) * 8);
    const long long ah = al128((long long)T * I + (long long)T * (I / kGroup) * 8);
    const long long rest = kLayerSmemBudget - ax - 2 * ah - 2 * kRedBytes - 2 * kMaxSlots * 8 - 256;
    // the largest slot (up to kSlotTiles tiles) that still gives each group's
    // ring two slots, else one
    int st = kSlotTiles;
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
    p->smem = p->off_bar + 2 * kGroups * ns * 8;
    // the routing phase keeps all T x E logits below the codes of x
    return (long long)T * E * 4 <= p->off_ax;
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
    return nslot * (I / kTileRows) + H / kTileRows;
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
    if ((err = launch_pdl(decode_prep_kernel, dim3(E), dim3(kPrepThreads), psmem, s, p)) != cudaSuccess) {
        cudaGetLastError();
        return err;
    }
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
    a.q_h = ws.q_h;
    a.d_h = ws.d_h;
    a.y_part = ws.y_part;
    a.cnt_h = ws.sync;
    a.cnt_y = ws.sync + nslot * (I / kTileRows);
    a.cap_g = ws.cap_g;
    a.cap_d = ws.cap_d;
    for (int d = 1; d <= H / kTileK && d <= ws.cap_g && a.ndiv_g < 16; ++d)
        if ((H / kTileK) % d == 0) a.div_g[a.ndiv_g++] = d;
    for (int d = 1; d <= I / kTileK && d <= ws.cap_d && a.ndiv_d < 16; ++d)
        if ((I / kTileK) % d == 0) a.div_d[a.ndiv_d++] = d;
    // 32-bit task indices: b x (tasks) must fit
    {
        const long long nt_max = std::min(E, T * k);
        const long long per = std::max((long long)(2 * I / kTileRows) * a.div_g[a.ndiv_g - 1],
                                       (long long)(H / kTileRows) * a.div_d[a.ndiv_d - 1]);
        if ((long long)(num_sms + 1) * nt_max * per >= (1ll << 31)) return cudaErrorInvalidValue;
    }
    a.out = out;
    a.out_fp32 = out_fp32 ? 1 : 0;
    a.dots_gu = dots_gu;
    a.dots_d = dots_d;
    a.write_qh = write_qh ? 1 : 0;
    a.status = status;
    a.ns = plan.ns;
    a.st = plan.st;
    a.off_bar = plan.off_bar;
    a.off_ax = plan.off_ax;
    a.off_ah = plan.off_ah;
    a.ah_bytes = plan.ah_bytes;
    a.off_red = plan.off_red;
    void (*kern)(LayerArgs) = T <= 16 ? decode_layer_kernel<16> : decode_layer_kernel<MOE_DECODE_MAX_T>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem);
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
    if ((err = cudaLaunchKernelEx(&cfg, kern, a)) != cudaSuccess) {
        cudaGetLastError();  // a refused launch: clear it, the context is intact
        return err;
    }
    for (int i = 2; i <= 6; ++i)
        if ((err = mark(i)) != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moeq4
