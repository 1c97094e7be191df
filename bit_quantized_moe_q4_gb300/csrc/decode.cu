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
// (each next grid is scheduled, and waits, before its predecessor ends):
//
//   layer    one CTA per SM, launched cooperatively (all CTAs resident: they
//            wait on one another).  It starts with the routing:
//              - CTA b owns router rows [bE/G, (b+1)E/G) (at most two); it
//                stages them into shared memory with one bulk copy before
//                waiting for the preceding work (the router does not depend
//                on it), then forms their logits for every token (fixed
//                summation order: per thread over its columns, then over the
//                lanes, then over the warps) and writes them to global memory;
//              - every CTA quantises x to int8 per 32 columns straight into
//                its own shared memory (the activations every gate/up task
//                reads), so no CTA waits for another's codes;
//              - one grid barrier (an arrival counter, bounded wait)
//                publishes the logits; the codes of x are formed meanwhile;
//              - every CTA then reads all T x E logits and takes the same
//                decisions itself: top-k and softmax weights (one token:
//                each expert's rank among the logits; more: one warp per
//                token), the expert buckets (a token bitmask per expert,
//                block scans for the offsets and the touched list).  CTA 0
//                also stores the routing results for the combine and the
//                debug outputs.
//            Then the expert work:
//            The packed weights of every touched expert
//            are cut into tasks of whole 4608-byte tiles: one 128-row block
//            times a range of 64-column blocks (the K range is split in
//            `ns` parts when there are too few row blocks to keep every SM
//            busy, e.g. for one token).  A task's tiles are contiguous in the
//            packed layout, so one producer warp streams them with 1-D bulk
//            copies (TMA) of up to four tiles into a shared-memory ring:
//            first the CTA's equal contiguous share of the gate/up tasks,
//            then its share of the down tasks, so down weights arrive while
//            gate/up is still being computed.  Eight consumer warps form the
//            dp4a group dots from shared memory (warp w: rows 16w..16w+15;
//            lane: one row and one 32-column half of each 64-column block)
//            and keep per-token fp32 row sums over the task's K range.
//            Gate/up tasks store the sums of g and u (with a K split the parts
//            are added with fp32 reductions into one buffer, so their order
//            of addition follows arrival) and raise a per-expert counter.  A
//            down task waits until every gate/up task of its expert is done,
//            then forms h = silu(g) * u and quantises it to int8 per 32
//            features; every CTA that needs an expert's h computes the same
//            codes.  Down tasks store partial sums of y = routing weight *
//            (W_d h).
//
//   combine  one thread per output: the residual plus every token's k expert
//            rows (slot order, partial sums in K order).
//
// Every weight byte of a touched expert is read once, by one CTA, from
// contiguous 4608-byte tiles.  Every wait is bounded; on expiry the kernel
// records MOE_ERR_TIMEOUT and stops.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int kMaxRouteRows = 2;              // router rows per CTA (E <= 2 x CTAs)
constexpr int kConsumerWarps = 8;             // 8 warps x 16 rows = one 128-row block
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kExpertThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kWarpProducer = kConsumerWarps;
constexpr int kChunkTiles = 4;                 // tiles per bulk copy / ring slot
constexpr int kSlotBytes = kChunkTiles * kTileBytes;
constexpr int kMaxSlots = 12;
constexpr int kExpertSmemBudget = 176 * 1024;
// Row blocks per SM the K split aims for (tasks = touched experts x row
// blocks x split); the split depends only on the shape, so results are
// reproducible.
constexpr int kTaskTarget = 152 * 5;
constexpr int kMaxSplit = 8;   // K parts of a gate/up task
constexpr int kMaxSplitD = 4;  // K parts of a down task

// Bytes of the fp16 activation scales of T tokens staged by one bulk copy
// (rounded up to 16; the workspace slot behind d_x is at least that long).
__host__ __device__ constexpr int act_scale_bytes(int T, int G) { return (T * G * 2 + 15) & ~15; }


struct DecodeArgs {
    const uint16_t* x;      // layer input as routed and multiplied
    const uint16_t* x_res;  // residual added by the combine (x, or the un-normalised input)
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
    int32_t* done;      // [E] finished gate/up tasks per touched expert
    int32_t* bucket_token;
    int32_t* bucket_slot;
    float* slot_w;
    int32_t* slot_pos;
    int8_t* q_x;
    uint16_t* d_x;
    int8_t* q_h;
    uint16_t* d_h;
    float* gu_sum;      // [T*k, 2I] fp32 sums of gate (0..I-1) and up (I..2I-1) rows;
                        // with a K split the parts are added into it (zeroed first)
    float* y_part;      // [nsd, T*k, H] fp32 partial sums of the weighted expert outputs
    int nsg, nsd;       // K splits of the gate/up and down tasks
    void* out;
    int out_fp32;
    int32_t* dots_gu;   // optional debug outputs
    int32_t* dots_d;
    int write_qh;       // 1: the CTA that owns down task (expert, 0) stores q_h / d_h
    int* status;
    int* gbar;          // [2] grid barrier: arrival count (0 between calls; the combine clears it)
    // expert-kernel shared-memory plan (bytes from the dynamic base)
    int nslot;          // ring slots of kSlotBytes
    int off_bar, off_ax, off_ah;
};

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Rearranges 8 int8 activations (x0..x7, one 8-column chunk) so that the two
// words line up with the packed code nibbles: the low nibbles of a code word
// (mask 0x0F0F0F0F) are columns 0,4,1,5 and the high nibbles 2,6,3,7.
__device__ __forceinline__ uint2 permute_chunk(uint32_t a, uint32_t b) {
    return make_uint2(__byte_perm(a, b, 0x5140), __byte_perm(a, b, 0x7362));
}

// Group dot of one packed 32-code group (4 words) with one staged activation
// group (8 permuted words in shared memory).
__device__ __forceinline__ int group_dot(const uint4 w, const uint8_t* a, int asum) {
    const uint4 a0 = *reinterpret_cast<const uint4*>(a);
    const uint4 a1 = *reinterpret_cast<const uint4*>(a + 16);
    // two independent chains (exact integer sums in any order)
    int p = -8 * asum, q = 0;
    p = dp4a_us(w.x & 0x0F0F0F0Fu, a0.x, p);
    q = dp4a_us((w.x >> 4) & 0x0F0F0F0Fu, a0.y, q);
    p = dp4a_us(w.y & 0x0F0F0F0Fu, a0.z, p);
    q = dp4a_us((w.y >> 4) & 0x0F0F0F0Fu, a0.w, q);
    p = dp4a_us(w.z & 0x0F0F0F0Fu, a1.x, p);
    q = dp4a_us((w.z >> 4) & 0x0F0F0F0Fu, a1.y, q);
    p = dp4a_us(w.w & 0x0F0F0F0Fu, a1.z, p);
    q = dp4a_us((w.w >> 4) & 0x0F0F0F0Fu, a1.w, q);
    return p + q;
}

// Barrier of the consumer warps only (named barrier 1).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// Exclusive prefix sum over the 256 consumer threads (thread order); `wt` is
// eight ints of shared memory.  Every consumer thread calls it.
__device__ __forceinline__ int consumers_exclusive_scan(int v, int* total, int* wt) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) wt[warp] = incl;
    consumers_sync();
    int base = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        if (w < warp) base += wt[w];
        all += wt[w];
    }
    consumers_sync();
    *total = all;
    return base + incl - v;
}

// -------------------------------------------------------------- experts
template <int N>
struct IntC {
    static constexpr int value = N;
};

// At most 128 registers a thread.
__global__ void __maxnreg__(128)
    decode_experts_kernel(const DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ int s_touched[kMaxExperts];
    __shared__ int s_tok[MOE_DECODE_MAX_T];
    __shared__ float s_sw[MOE_DECODE_MAX_T];
    __shared__ int s_route[2];  // off, c of the consumers' current expert
    __shared__ int s_nt;
    __shared__ volatile int s_cok[2];
    __shared__ volatile int s_abort;
    __shared__ __align__(8) uint64_t s_actbar;
    // routing (every CTA holds the whole decision)
    __shared__ float s_part[MOE_DECODE_MAX_T * kConsumerWarps * kMaxRouteRows];
    __shared__ int s_idx[MOE_DECODE_MAX_T * MOE_MAX_TOPK];
    __shared__ float s_w[MOE_DECODE_MAX_T * MOE_MAX_TOPK];
    __shared__ int s_btok[MOE_DECODE_MAX_T * MOE_MAX_TOPK];   // bucket rows: token
    __shared__ float s_bsw[MOE_DECODE_MAX_T * MOE_MAX_TOPK];  // bucket rows: routing weight
    __shared__ uint32_t s_mask[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_wt[kConsumerWarps];

    const int T = a.T, H = a.H, I = a.I, k = a.k;
    const int KBg = H / kTileK, KBd = I / kTileK;  // 64-column blocks per row
    const int RBg = 2 * I / kTileRows, RBd = H / kTileRows;  // 128-row blocks per expert
    const int Gx = H / kGroup, Gh = I / kGroup;
    const int nsg = a.nsg, nsd = a.nsd;
    const int KCg = KBg / nsg, KCd = KBd / nsd;  // blocks per task
    const int Tk = T * k;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, tid = threadIdx.x;
    const uint32_t sbase = smem_u32(dsm);
    const uint32_t bar0 = sbase + a.off_bar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxSlots + s); };
    uint8_t* ax_q = dsm + a.off_ax;                                   // [T][H] permuted int8
    uint16_t* ax_dh = reinterpret_cast<uint16_t*>(ax_q + (size_t)T * H);  // [T][Gx] fp16 (+pad)
    int* ax_s = reinterpret_cast<int*>(ax_q + (size_t)T * H + act_scale_bytes(T, Gx));  // [T][Gx]
    uint8_t* ah_q = dsm + a.off_ah;                                   // [T][I] permuted int8
    float* ah_d = reinterpret_cast<float*>(ah_q + (size_t)T * I);
    int* ah_s = reinterpret_cast<int*>(ah_d + T * Gh);

    const int E = a.E, G = gridDim.x, b = blockIdx.x;
    auto fail = [&]() {
        record_status(a.status, kStatusTimeout);
        s_abort = 1;
    };
    const uint32_t actbar = smem_u32(&s_actbar);
    // router rows of this CTA, staged in the (still unused) ring area
    const int eb0 = (int)((long long)b * E / G), eb1 = (int)((long long)(b + 1) * E / G);
    const int ne = eb1 - eb0;  // <= kMaxRouteRows (checked at launch)
    const float* s_wr = reinterpret_cast<const float*>(dsm);
    if (tid == 0) {
        for (int s = 0; s < kMaxSlots; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        mbar_init(actbar, 1);
        s_abort = 0;
        fence_mbar_init();
        if (ne > 0) {
            mbar_arrive_expect_tx(actbar, (uint32_t)(ne * H * 4));
            bulk_g2s(sbase, a.wr + (size_t)eb0 * H, (uint32_t)(ne * H * 4), actbar);
        }
    }
    __syncthreads();
    pdl_wait();     // x and the workspace belong to this call from here on
    pdl_trigger();  // the combine may be scheduled; it waits for our end
    // this CTA's share of the completion counters and of the K-split sums
    for (int i = eb0 + tid; i < eb1; i += kExpertThreads) a.done[i] = 0;
    if (nsg > 1) {
        const int n4 = Tk * 2 * I / 4;
        float4* z = reinterpret_cast<float4*>(a.gu_sum);
        for (int i = (int)((long long)b * n4 / G) + tid; i < (int)((long long)(b + 1) * n4 / G);
             i += kExpertThreads)
            z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int H8 = H / 8, nU = (H8 + 31) & ~31;  // 8-column units of a token, whole warps
    if (warp != kWarpProducer) {
        // logits of the CTA's router rows: thread unit u = 8 consecutive
        // columns of one token
        if (ne > 0 && !mbar_wait(actbar, 0)) fail();
        for (int t = 0; t < T && ne > 0; ++t) {
            float acc[kMaxRouteRows] = {0.f, 0.f};
            for (int u = tid; u < nU; u += kConsumerThreads) {  // warp-uniform bound
                if (u < H8) {
                    const uint4 xv = __ldcg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H) + u);
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                    float xf[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        xf[2 * i] = __uint_as_float(xw[i] << 16);
                        xf[2 * i + 1] = __uint_as_float(xw[i] & 0xffff0000u);
                    }
#pragma unroll
                    for (int r = 0; r < kMaxRouteRows; ++r) {
                        if (r < ne) {
                            const float4 w0 = *reinterpret_cast<const float4*>(s_wr + r * H + u * 8);
                            const float4 w1 = *reinterpret_cast<const float4*>(s_wr + r * H + u * 8 + 4);
                            float v = acc[r];
                            v = fmaf(xf[0], w0.x, v);
                            v = fmaf(xf[1], w0.y, v);
                            v = fmaf(xf[2], w0.z, v);
                            v = fmaf(xf[3], w0.w, v);
                            v = fmaf(xf[4], w1.x, v);
                            v = fmaf(xf[5], w1.y, v);
                            v = fmaf(xf[6], w1.z, v);
                            v = fmaf(xf[7], w1.w, v);
                            acc[r] = v;
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kMaxRouteRows; ++r) {
                const float v = warp_sum(acc[r]);
                if (lane == 0) s_part[(t * kConsumerWarps + warp) * kMaxRouteRows + r] = v;
            }
        }
        consumers_sync();
        for (int q = tid; q < T * ne; q += kConsumerThreads) {
            const int t = q / ne, r = q % ne;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) v += s_part[(t * kConsumerWarps + w) * kMaxRouteRows + r];
            a.logits[(size_t)t * E + eb0 + r] = v;
        }
    }
    // grid barrier: every CTA's logits and zeroed counters are published.
    // The count is zero when the call starts (the combine of the previous
    // call cleared it) and reaches G once every CTA has arrived.  The
    // producer warp arrives and waits; meanwhile the consumers quantise x.
    __syncthreads();
    if (warp == kWarpProducer) {
        if (lane == 0) {
            __threadfence();
            red_release_add(a.gbar, 1);
            const unsigned long long t0 = globaltimer_ns();
            while (ld_acquire(a.gbar) < G) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    fail();
                    break;
                }
            }
        }
    } else {
        // the int8 codes of x: unit u = 8 columns of one token, four
        // consecutive lanes one 32-column group
        for (int t = 0; t < T; ++t) {
            for (int u = tid; u < nU; u += kConsumerThreads) {  // warp-uniform bound
                const bool valid = u < H8;
                const uint4 xv = valid ? __ldcg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H) + u)
                                       : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                float xf[8];
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xf[2 * i] = __uint_as_float(xw[i] << 16);
                    xf[2 * i + 1] = __uint_as_float(xw[i] & 0xffff0000u);
                    amax = fmaxf(amax, fmaxf(fabsf(xf[2 * i]), fabsf(xf[2 * i + 1])));
                }
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                const uint16_t db = act_scale_bits(amax);
                const float d = half_bits_to_float(db);
                uint32_t lo = 0u, hi = 0u;
                int gsum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int qc = act_code(xf[i], d);
                    gsum += qc;
                    if (i < 4) lo |= ((uint32_t)qc & 0xffu) << (8 * i);
                    else hi |= ((uint32_t)qc & 0xffu) << (8 * (i - 4));
                }
                gsum += __shfl_xor_sync(0xffffffffu, gsum, 1);
                gsum += __shfl_xor_sync(0xffffffffu, gsum, 2);
                if (valid) {
                    *reinterpret_cast<uint2*>(ax_q + (size_t)t * H + u * 8) = permute_chunk(lo, hi);
                    if ((lane & 3) == 0) {
                        ax_dh[t * Gx + u / 4] = db;
                        ax_s[t * Gx + u / 4] = gsum;
                    }
                    if (b == 0) {  // the codes as stage outputs
                        *reinterpret_cast<uint2*>(a.q_x + (size_t)t * H + u * 8) = make_uint2(lo, hi);
                        if ((lane & 3) == 0) a.d_x[t * Gx + u / 4] = db;
                    }
                }
            }
        }
    }
    __syncthreads();
    // every CTA: all logits -> top-k, weights and buckets (the same in every CTA)
    float* s_lg = reinterpret_cast<float*>(dsm);  // [T][E], over the staged router rows
    for (int i = tid; i < T * E; i += kExpertThreads) s_lg[i] = __ldcg(a.logits + i);
    __syncthreads();
    if (T == 1) {
        // One token: expert e's rank among the E logits (larger first, equal
        // logits by lower index); ranks below k are the choices.  Its k
        // experts are distinct, so an expert's bucket offset is the number of
        // chosen experts below it, which is also a chosen expert's row.
        // Order keys rank every bit pattern (NaN included), so the ranks are
        // a permutation of 0..E-1.
        __shared__ float s_val[MOE_MAX_TOPK];
        __shared__ float s_ex[MOE_MAX_TOPK];
        // keys padded with 0 to a multiple of 8 (a padding key, index >= E,
        // never ranks above a real one)
        __shared__ __align__(16) uint32_t s_key[kMaxExperts];
        const int E8 = (E + 7) & ~7;
        for (int e = tid; e < E8; e += kExpertThreads) s_key[e] = e < E ? float_order_key(s_lg[e]) : 0u;
        __syncthreads();
        const int P = (2 * E <= kExpertThreads) ? 2 : 1;  // threads per expert
        const int half4 = E8 / 8;                           // uint4 groups per half
        const uint4* key4 = reinterpret_cast<const uint4*>(s_key);
        for (int base = 0; base < P * E; base += kExpertThreads) {  // warp-uniform
            const int q = base + tid;
            const bool act = q < P * E;
            const int e = act ? q / P : 0, part = q % P;
            const uint32_t kv = s_key[e];
            const int lo = (P == 2 && part == 1) ? half4 : 0;
            const int hi = !act ? 0 : (P == 2 && part == 0) ? half4 : 2 * half4;
            int rank = 0;
#pragma unroll 4
            for (int c4 = lo; c4 < hi; ++c4) {
                const uint4 k4 = key4[c4];
                const int e2 = 4 * c4;
                rank += (k4.x > kv) | ((k4.x == kv) & (e2 < e));
                rank += (k4.y > kv) | ((k4.y == kv) & (e2 + 1 < e));
                rank += (k4.z > kv) | ((k4.z == kv) & (e2 + 2 < e));
                rank += (k4.w > kv) | ((k4.w == kv) & (e2 + 3 < e));
            }
            if (P == 2) rank += __shfl_xor_sync(0xffffffffu, rank, 1);  // the pair (2m, 2m + 1)
            if (act && part == 0 && rank < k) {
                s_idx[rank] = e;
                s_val[rank] = s_lg[e];
            }
        }
        __syncthreads();
        if (tid < k) s_ex[tid] = expf(s_val[tid] - s_val[0]);
        for (int e = tid; e <= E; e += kExpertThreads) {
            int lt = 0;
            for (int j = 0; j < k; ++j) lt += s_idx[j] < e;
            s_off[e] = lt;
            if (b == 0) a.offsets[e] = lt;
        }
        __syncthreads();
        if (tid < k) {
            float den = 0.f;
            for (int j = 0; j < k; ++j) den += s_ex[j];
            const float w = s_ex[tid] / den;
            const int ex = s_idx[tid], pos = s_off[ex];
            s_touched[pos] = ex;
            s_btok[pos] = 0;
            s_bsw[pos] = w;
            if (b == 0) {
                a.topk_idx[tid] = ex;
                a.topk_w[tid] = w;
                a.touched[pos] = ex;
                a.bucket_token[pos] = 0;
                a.bucket_slot[pos] = tid;
                a.slot_w[pos] = w;
                a.slot_pos[tid] = pos;
            }
        }
        if (tid == 0) {
            s_nt = k;
            if (b == 0) a.counters[kCntTouched] = k;
        }
    } else if (warp != kWarpProducer) {
        for (int t = warp; t < T; t += kConsumerWarps) {
            int si;
            float sw;
            warp_topk(s_lg + t * E, E, k, si, sw);
            if (lane < k) {
                s_idx[t * k + lane] = si;
                s_w[t * k + lane] = sw;
            }
        }
        s_mask[tid] = 0u;  // kMaxExperts == kConsumerThreads
        consumers_sync();
        // token t's bit in the mask of each expert it chose (T <= 32)
        for (int p = tid; p < Tk; p += kConsumerThreads) atomicOr(&s_mask[s_idx[p]], 1u << (p / k));
        consumers_sync();
        const int e = tid;  // one thread per expert (E <= 256)
        const int cnt = (e < E) ? __popc(s_mask[e]) : 0;
        int total, ntouched;
        const int off = consumers_exclusive_scan(cnt, &total, s_wt);
        const int tpos = consumers_exclusive_scan(cnt > 0 ? 1 : 0, &ntouched, s_wt);
        if (e < E) {
            s_off[e] = off;
            if (cnt > 0) s_touched[tpos] = e;
        }
        if (tid == 0) {
            s_off[E] = total;
            s_nt = ntouched;
        }
        consumers_sync();
        for (int p = tid; p < Tk; p += kConsumerThreads) {
            const int t = p / k, ex = s_idx[p];
            const int pos = s_off[ex] + __popc(s_mask[ex] & ((1u << t) - 1u));
            s_btok[pos] = t;
            s_bsw[pos] = s_w[p];
            if (b == 0) {
                a.topk_idx[p] = ex;
                a.topk_w[p] = s_w[p];
                a.bucket_token[pos] = t;
                a.bucket_slot[pos] = p % k;
                a.slot_w[pos] = s_w[p];
                a.slot_pos[p] = pos;
            }
        }
        if (b == 0) {
            for (int i = tid; i <= E; i += kConsumerThreads) a.offsets[i] = s_off[i];
            for (int i = tid; i < ntouched; i += kConsumerThreads) a.touched[i] = s_touched[i];
            if (tid == 0) a.counters[kCntTouched] = ntouched;
        }
    }
    // the ring area was used through generic accesses; bulk copies refill it next
    fence_proxy_async_smem();
    __syncthreads();
    const int nt = s_nt;
    const int per_g = RBg * nsg, per_d = RBd * nsd;  // tasks per touched expert
    const int n_gu = nt * per_g, n_dn = nt * per_d;
    // (32-bit products: launch_decode checks that G x the task counts fits)
    const int gu0 = b * n_gu / G, gu1 = (b + 1) * n_gu / G;
    const int dn0 = b * n_dn / G, dn1 = (b + 1) * n_dn / G;

    if (warp == kWarpProducer) {
        // ----------------------------------------------------------- producer
        // gate/up tasks, then down tasks; each task's tiles in chunks of up to
        // kChunkTiles contiguous tiles, one bulk copy per chunk.  The down
        // weights are requested once this CTA's gate/up weights have landed:
        // every CTA's gate/up bytes then have the memory system to
        // themselves, and the down bytes arrive while gate/up is computed
        // and handed over.
        if (lane == 0) {
            int j = 0;  // ring position
            bool ok = true;
            for (int pass = 0; pass < 2 && ok; ++pass) {
                const bool gu = pass == 0;
                if (!gu && j > 0 && dn1 > dn0 &&
                    (s_abort || !mbar_wait(full_bar((j - 1) % a.nslot), ((j - 1) / a.nslot) & 1))) {
                    fail();
                    break;
                }
                const int t0 = gu ? gu0 : dn0, t1 = gu ? gu1 : dn1;
                const int per = gu ? per_g : per_d, ns = gu ? nsg : nsd;
                const int KB = gu ? KBg : KBd, KC = gu ? KCg : KCd, RB = gu ? RBg : RBd;
                const uint8_t* wbase = gu ? a.wgu : a.wd;
                for (int task = t0; task < t1 && ok; ++task) {
                    const int slot_i = task / per, rem = task % per;
                    const int rb = rem / ns, kc = rem % ns;
                    const uint8_t* src = wbase + (((size_t)s_touched[slot_i] * RB + rb) * KB +
                                                  (size_t)kc * KC) * kTileBytes;
                    for (int c0 = 0; c0 < KC; c0 += kChunkTiles, ++j) {
                        const int s = j % a.nslot;
                        const int nb = min(kChunkTiles, KC - c0) * kTileBytes;
                        if (s_abort || !mbar_wait(empty_bar(s), ((j / a.nslot) & 1) ^ 1)) {
                            fail();
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full_bar(s), (uint32_t)nb);
                        bulk_g2s(sbase + s * kSlotBytes, src + (size_t)c0 * kTileBytes, (uint32_t)nb,
                                 full_bar(s));
                    }
                }
            }
            // the copies already issued land before the CTA can go away
            for (int q = (j > a.nslot ? j - a.nslot : 0); q < j; ++q)
                mbar_wait(full_bar(q % a.nslot), (q / a.nslot) & 1);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    // (the int8 codes of x are in shared memory since the routing phase)
    // Consumer control flow must stay uniform (the consumers share named
    // barriers): the task loops always run to their end, and a decision that
    // can differ between threads (a timed wait, the abort flag the producer
    // may raise at any time) only skips work, never a barrier.  Decisions the
    // whole CTA must share are taken by thread 0 and handed to all consumers
    // through a barrier (double-buffered so a late reader never sees the next
    // decision).
    int round = 0;
    auto agree = [&](bool v0) -> bool {
        const int slot = round & 1;
        ++round;
        if (tid == 0) s_cok[slot] = (v0 && !s_abort) ? 1 : 0;
        consumers_sync();
        return s_cok[slot] != 0;
    };
    // Each warp waits (bounded) for a ring slot's copy itself; observing the
    // completed phase makes the copied bytes visible to its lanes.
    bool live = true;  // this warp has not given up
    auto slot_ready = [&](int j) -> bool {
        if (!live) return false;
        if (s_abort || !mbar_wait(full_bar(j % a.nslot), (j / a.nslot) & 1)) {
            fail();
            live = false;
        }
        return live;
    };
    // routing of one touched expert into shared memory (all consumers call it)
    auto load_routing = [&](int slot_i) {
        consumers_sync();
        const int ex = s_touched[slot_i];
        if (tid == 0) {
            s_route[0] = s_off[ex];
            s_route[1] = s_off[ex + 1] - s_off[ex];
        }
        consumers_sync();
        const int off = s_route[0], c = s_route[1];
        if (tid < c) {
            s_tok[tid] = s_btok[off + tid];
            s_sw[tid] = s_bsw[off + tid];
        }
        consumers_sync();
    };

    const int r_lane = lane >> 1, h_lane = lane & 1;
    const int lrow = warp * 16 + r_lane;  // this lane's row in the 128-row block
    int j = 0;                            // ring position (same order as the producer)

    // One task: rows rb*128 + lrow, 64-column blocks [kb0, kb0 + KC), for the
    // c bucket rows of the current expert; NT >= c is a compile-time bound.
    // Per token the lane pair's fp32 sum over the task's blocks is written
    // (times the routing weight for down) to dst[(off + n) * ld + row].
    auto run_task = [&](auto ntc, bool gu, int kb0, int KC, int row, float* dst, size_t ld) {
        constexpr int NT = decltype(ntc)::value;
        const int off = s_route[0], c = s_route[1];
        const uint8_t* aq = gu ? ax_q : ah_q;
        const int* as = gu ? ax_s : ah_s;
        const int K = gu ? H : I, Gk = gu ? Gx : Gh;
        int32_t* dots = gu ? a.dots_gu : a.dots_d;
        const size_t dots_ld = gu ? (size_t)2 * I : (size_t)H;
        float acc[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n] = 0.f;
        for (int c0 = 0; c0 < KC; c0 += kChunkTiles, ++j) {
            if (!slot_ready(j)) continue;
            const uint8_t* slot = dsm + (j % a.nslot) * kSlotBytes;
            const int nb = min(kChunkTiles, KC - c0);
            constexpr int UT = NT <= 8 ? kChunkTiles : 1;  // tiles in flight (registers)
#pragma unroll UT
            for (int t = 0; t < kChunkTiles; ++t) {
                if (t >= nb) break;
                const uint8_t* tile = slot + t * kTileBytes;
                const int g = 2 * (kb0 + c0 + t) + h_lane;
                const uint4 wv = *reinterpret_cast<const uint4*>(tile + warp * 512 + lane * 16);
                const float dw = half_bits_to_float(
                    *reinterpret_cast<const uint16_t*>(tile + kTileCodeBytes + warp * 64 + lane * 2));
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if (n < c) {
                        const int ar = gu ? s_tok[n] : n;
                        const int dot = group_dot(wv, aq + (size_t)ar * K + g * kGroup, as[ar * Gk + g]);
                        const float da = gu ? half_bits_to_float(ax_dh[ar * Gk + g]) : ah_d[ar * Gk + g];
                        acc[n] = fmaf((float)dot, dw * da, acc[n]);
                        if (dots) dots[((size_t)(off + n) * dots_ld + row) * Gk + g] = dot;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(j % a.nslot));
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], 1);
        if (h_lane == 0 && live) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (n >= c) continue;
                float* d = dst + (size_t)(off + n) * ld + row;
                if (!gu)
                    *d = acc[n] * s_sw[n];
                else if (nsg > 1)
                    atomicAdd(d, acc[n]);  // K parts meet here (order of arrival)
                else
                    *d = acc[n];
            }
        }
    };
    auto dispatch = [&](bool gu, int kb0, int KC, int row, float* dst, size_t ld) {
        const int c = s_route[1];
        if (c <= 1) run_task(IntC<1>{}, gu, kb0, KC, row, dst, ld);
        else if (c <= 2) run_task(IntC<2>{}, gu, kb0, KC, row, dst, ld);
        else if (c <= 4) run_task(IntC<4>{}, gu, kb0, KC, row, dst, ld);
        else if (c <= 8) run_task(IntC<8>{}, gu, kb0, KC, row, dst, ld);
        else if (c <= 16) run_task(IntC<16>{}, gu, kb0, KC, row, dst, ld);
        else run_task(IntC<MOE_DECODE_MAX_T>{}, gu, kb0, KC, row, dst, ld);
    };

    // 2. gate/up tasks -> partial sums of g and u
    int cur = -1, pending = 0;
    auto publish = [&](int slot_i, int count) {
        __threadfence();
        consumers_sync();  // every partial sum of these tasks is written
        if (tid == 0 && count > 0) atomicAdd(&a.done[slot_i], count);
    };
    for (int task = gu0; task < gu1; ++task) {
        const int slot_i = task / per_g, rem = task % per_g;
        const int rb = rem / nsg, kc = rem % nsg;
        if (slot_i != cur) {
            if (cur >= 0) publish(cur, pending);
            load_routing(slot_i);
            cur = slot_i;
            pending = 0;
        }
        dispatch(true, kc * KCg, KCg, rb * kTileRows + lrow, a.gu_sum, (size_t)2 * I);
        ++pending;
    }
    if (cur >= 0) publish(cur, pending);

    // 3. down tasks -> partial sums of y
    int h_slot = -1;
    bool have_h = true;
    for (int task = dn0; task < dn1; ++task) {
        const int slot_i = task / per_d, rem = task % per_d;
        const int rb = rem / nsd, kc = rem % nsd;
        if (slot_i != h_slot) {
            load_routing(slot_i);
            // wait until every gate/up task of this expert is done
            bool got = true;
            if (tid == 0) {
                if (ld_acquire(&a.done[slot_i]) < per_g) {
                    const unsigned long long t0 = globaltimer_ns();
                    while (ld_acquire(&a.done[slot_i]) < per_g) {
                        if (s_abort || globaltimer_ns() - t0 > kWaitLimitNs) {
                            got = false;
                            break;
                        }
                    }
                }
                if (!got) fail();
                __threadfence();
            }
            have_h = agree(got);
            // h = silu(g) * u (partial sums added in K order), int8 per 32
            // features: a warp takes four groups at once, eight lanes a group,
            // four consecutive features a lane
            const int off = s_route[0], c = s_route[1];
            const bool store = a.write_qh && rb == 0 && kc == 0;
            const int sub = lane / 8, l8 = lane % 8;
            for (int q0 = warp * 4; q0 < (have_h ? c * Gh : 0); q0 += 4 * kConsumerWarps) {
                const int q = q0 + sub;
                const bool ok = q < c * Gh;
                const int n = ok ? q / Gh : 0, gg = ok ? q % Gh : 0, f0 = gg * kGroup + l8 * 4;
                const float* gs = a.gu_sum + (size_t)(off + n) * 2 * I + f0;
                const float4 g4 = ok ? __ldcg(reinterpret_cast<const float4*>(gs)) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 u4 = ok ? __ldcg(reinterpret_cast<const float4*>(gs + I)) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
                float h[4];
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    h[i] = gv[i] / (1.0f + __expf(-gv[i])) * uv[i];
                    amax = fmaxf(amax, fabsf(h[i]));
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const uint16_t db = act_scale_bits(amax);
                const float d = half_bits_to_float(db);
                uint32_t w4 = 0u;
                int sum = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int qv = act_code(h[i], d);
                    sum += qv;
                    w4 |= ((uint32_t)qv & 0xffu) << (8 * i);
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                // lanes 2m and 2m+1 hold columns 8m..8m+3 and 8m+4..8m+7 of the
                // group: the even lane stores the chunk in the permuted order
                const uint32_t w4o = __shfl_xor_sync(0xffffffffu, w4, 1);
                if (ok) {
                    if ((l8 & 1) == 0)
                        *reinterpret_cast<uint2*>(ah_q + (size_t)n * I + gg * kGroup + l8 * 4) =
                            permute_chunk(w4, w4o);
                    if (l8 == 0) {
                        ah_d[n * Gh + gg] = d;
                        ah_s[n * Gh + gg] = sum;
                    }
                    if (store) {
                        *reinterpret_cast<uint32_t*>(a.q_h + (size_t)(off + n) * I + f0) = w4;
                        if (l8 == 0) a.d_h[(size_t)(off + n) * Gh + gg] = db;
                    }
                }
            }
            consumers_sync();
            h_slot = slot_i;
        }
        if (!have_h) live = false;  // nothing valid to multiply: skip the rest
        dispatch(false, kc * KCd, KCd, rb * kTileRows + lrow, a.y_part + (size_t)kc * Tk * H,
                 (size_t)H);
    }

}

// ---------------------------------------------------------------- combine
// out[t] = x[t] + sum over slots j (in order) of sum over the K parts of the
// down tasks (in order) of y_part[part][slot_pos[t, j]].  One output per
// thread; all of a thread's loads are issued before the first add.
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeArgs a) {
    pdl_wait();     // the layer kernel's y parts
    pdl_trigger();  // the next layer may be scheduled
    // the layer kernel has ended: its grid barrier count is zero again (also
    // after a timed-out call)
    if (blockIdx.x == 0 && threadIdx.x == 0) a.gbar[0] = 0;
    const int H = a.H, k = a.k, nsd = a.nsd, Tk = a.T * a.k;
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= a.T * H) return;
    const int t = q / H, col = q % H;
    float v = bf16_bits_to_float(a.x_res[q]);
    for (int j0 = 0; j0 < k; j0 += 8) {
        int rows[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) rows[u] = (j0 + u < k) ? a.slot_pos[t * k + j0 + u] : 0;
        float part[8][kMaxSplitD];
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int p = 0; p < kMaxSplitD; ++p)
                part[u][p] = (j0 + u < k && p < nsd)
                                 ? __ldcg(a.y_part + ((size_t)p * Tk + rows[u]) * H + col)
                                 : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int p = 0; p < kMaxSplitD; ++p) v += part[u][p];  // adding 0 is exact
    }
    if (a.out_fp32)
        static_cast<float*>(a.out)[q] = v;
    else
        static_cast<uint16_t*>(a.out)[q] = float_to_bf16_bits(v);
}

// ---------------------------------------------------------------- launch
int g_expert_pdl[64] = {};  // 0 unknown, 1 cooperative + PDL accepted, 2 cooperative only
int* g_gbar_seen[64] = {};  // per device: the last workspace whose barrier words were cleared
std::mutex g_gbar_mu;

// Smallest divisor of KB that is >= want; if that exceeds cap, the largest
// divisor of KB that is <= cap.
int split_at_least(int KB, int want, int cap) {
    if (want > cap) want = cap;
    for (int d = want < 1 ? 1 : want; d <= KB && d <= cap; ++d)
        if (KB % d == 0) return d;
    for (int d = cap; d > 1; --d)
        if (KB % d == 0) return d;
    return 1;
}

// K splits of the gate/up and down tasks for a shape: enough tasks that
// every SM gets several even when few experts are touched (one token).
void choose_splits(int T, int H, int I, int E, int k, int* nsg, int* nsd) {
    const int nt_est = min(E, T * k);
    const int rbg = 2 * I / kTileRows, rbd = H / kTileRows;
    if (nt_est <= 0 || rbg <= 0 || rbd <= 0 || H < kTileK || I < kTileK) {
        *nsg = *nsd = 1;
        return;
    }
    *nsg = split_at_least(H / kTileK, (kTaskTarget + nt_est * rbg - 1) / (nt_est * rbg), kMaxSplit);
    *nsd = split_at_least(I / kTileK, (kTaskTarget / 2 + nt_est * rbd - 1) / (nt_est * rbd),
                          kMaxSplitD);
}

// Shared-memory plan of the expert kernel; returns false if it does not fit.
bool plan_experts(DecodeArgs& a) {
    auto al = [](int v) { return (v + 127) & ~127; };
    const int ax = al(a.T * a.H + act_scale_bytes(a.T, a.H / kGroup) + a.T * (a.H / kGroup) * 4);
    const int ah = al(a.T * a.I + a.T * (a.I / kGroup) * 8);
    const int bars = 2 * kMaxSlots * 8;
    int ns = (kExpertSmemBudget - ax - ah - bars) / kSlotBytes;
    ns = ns > kMaxSlots ? kMaxSlots : ns;
    if (ns < 2) return false;
    // the routing phase keeps the CTA's router rows, then all logits, in the ring
    if (kMaxRouteRows * a.H * 4 > ns * kSlotBytes || a.T * a.E * 4 > ns * kSlotBytes) return false;
    a.nslot = ns;
    a.off_bar = ns * kSlotBytes;
    a.off_ax = al(a.off_bar + bars);
    a.off_ah = a.off_ax + ax;
    return true;
}

int expert_smem_bytes(const DecodeArgs& a) {
    return a.off_ah + ((a.T * a.I + a.T * (a.I / kGroup) * 8 + 127) & ~127);
}

cudaError_t launch_all(DecodeArgs& a, int num_sms, void** ev, bool capturing, cudaStream_t s) {
    cudaError_t err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    auto mark = [&](int i) -> cudaError_t {
        return (ev && ev[i]) ? record_stage(ev[i], s, capturing) : cudaSuccess;
    };
    cudaLaunchAttribute pdl{};
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    // ---- layer: routing and experts ----
    const int smem = expert_smem_bytes(a);
    err = cudaFuncSetAttribute(decode_experts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
    if (err != cudaSuccess) return err;
    const int mode = g_expert_pdl[dev & 63];
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[2];
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kExpertThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1] = pdl;
    cfg.attrs = at;
    cfg.numAttrs = (mode == 2) ? 1 : 2;
    err = cudaLaunchKernelEx(&cfg, decode_experts_kernel, a);
    if (err != cudaSuccess) return err;
    for (int i = 1; i <= 5; ++i)
        if ((err = mark(i)) != cudaSuccess) return err;
    // ---- combine ----
    {
        cudaLaunchConfig_t cc{};
        cc.gridDim = dim3((unsigned)((a.T * a.H + 255) / 256));
        cc.blockDim = dim3(256);
        cc.stream = s;
        cc.attrs = &pdl;
        cc.numAttrs = 1;
        err = cudaLaunchKernelEx(&cc, decode_combine_kernel, a);
        if (err != cudaSuccess) return err;
    }
    if ((err = mark(6)) != cudaSuccess) return err;
    return cudaGetLastError();
}

__global__ void coop_pdl_probe_kernel(int* p) {
    pdl_wait();
    if (p && threadIdx.x == 0 && blockIdx.x == 0) *p = 1;
}

}  // namespace

// Decides once per device (outside any capture) whether a cooperative launch
// may also carry the programmatic-dependent-launch attribute.
cudaError_t decode_prepare_device(int dev) {
    int& mode = g_expert_pdl[dev & 63];
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

bool decode_shape_fits(int T, int H, int I) {
    DecodeArgs a{};
    a.T = T;
    a.H = H;
    a.I = I;
    return plan_experts(a);
}

void decode_splits(int T, int H, int I, int E, int k, int* nsg, int* nsd) {
    choose_splits(T, H, I, E, k, nsg, nsd);
}

cudaError_t launch_decode(const uint16_t* x, const uint16_t* x_res, const float* wr,
                          const void* wgu, const void* wd,
                          int T, int H, int I, int E, int k, bool out_fp32, void* out,
                          const Workspace& ws, int32_t* dots_gu, int32_t* dots_d, bool write_qh,
                          int* status, int num_sms, void** events, bool capturing,
                          cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    DecodeArgs a{};
    a.x = x;
    a.x_res = x_res;
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
    a.done = ws.done;
    a.bucket_token = ws.bucket_token;
    a.bucket_slot = ws.bucket_slot;
    a.slot_w = ws.slot_w;
    a.slot_pos = ws.slot_pos;
    a.q_x = ws.q_x;
    a.d_x = ws.d_x;
    a.q_h = ws.q_h;
    a.d_h = ws.d_h;
    a.gu_sum = ws.gu_sum;
    a.y_part = ws.y_part;
    choose_splits(T, H, I, E, k, &a.nsg, &a.nsd);
    a.out = out;
    a.out_fp32 = out_fp32 ? 1 : 0;
    a.dots_gu = dots_gu;
    a.dots_d = dots_d;
    a.write_qh = write_qh ? 1 : 0;
    a.status = status;
    a.gbar = ws.gbar;
    if (!plan_experts(a)) return cudaErrorInvalidValue;
    if ((E + num_sms - 1) / num_sms > kMaxRouteRows) return cudaErrorInvalidValue;
    {
        const long long nt_max = E < T * k ? E : T * k;
        const long long per = std::max((long long)(2 * I / kTileRows) * a.nsg,
                                       (long long)(H / kTileRows) * a.nsd);
        if ((long long)(num_sms + 1) * nt_max * per >= (1ll << 31)) return cudaErrorInvalidValue;
    }
    // The grid barrier's count must start at zero; every call leaves it
    // there.  A workspace not seen before gets it cleared once.
    {
        std::lock_guard<std::mutex> lock(g_gbar_mu);
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        if (g_gbar_seen[dev & 63] != ws.gbar) {
            err = cudaMemsetAsync(ws.gbar, 0, 2 * sizeof(int), s);
            if (err != cudaSuccess) return err;
            g_gbar_seen[dev & 63] = ws.gbar;
        }
    }
    return launch_all(a, num_sms, events, capturing, s);
}

}  // namespace moeq4
