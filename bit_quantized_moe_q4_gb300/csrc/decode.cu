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
// One decode layer is three kernels chained with programmatic dependent launch
// (each next grid is resident, and has issued its weight-only loads, before
// its predecessor ends):
//
//   route    a thread-block cluster.  Each warp reads one router row into
//            registers before waiting for the preceding work (the router does
//            not depend on it), then forms that expert's logits for all tokens
//            and writes them into the leader CTA's shared memory (distributed
//            shared memory).  The cluster also quantises x to int8 per 32.
//            After a cluster barrier the leader picks the top-k and the
//            softmax weights (one warp per token), builds the expert buckets
//            (one thread per expert: bitmask, popcount, block scan) and clears
//            the completion counters the expert kernel uses.  With few
//            (token, slot) pairs one warp does the bucketing with shuffles.
//
//   experts  one CTA per SM, launched cooperatively (all CTAs resident: they
//            wait on one another).  The packed weights of every touched expert
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
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int kRouteThreads = 256;            // 8 warps per cluster CTA
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

__host__ __device__ constexpr int align128(int v) { return (v + 127) & ~127; }

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
                        // with a K split the parts are added into it (zeroed by route)
    float* y_part;      // [nsd, T*k, H] fp32 partial sums of the weighted expert outputs
    int nsg, nsd;       // K splits of the gate/up and down tasks
    void* out;
    int out_fp32;
    int32_t* dots_gu;   // optional debug outputs
    int32_t* dots_d;
    int write_qh;       // 1: the CTA that owns down task (expert, 0) stores q_h / d_h
    int* status;
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
// Byte position of column c (0..31) of a group in that permuted order.
__device__ __forceinline__ int permuted_pos(int c) {
    const int cc = c & 7;
    return (c & ~7) + (cc & 3) * 2 + (cc >> 2);
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

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---------------------------------------------------------------- route
// For T <= 8 at most 104 registers a thread (256 x 104 = 26,624): the CTA fits beside
// an expert CTA (288 threads x 128 registers) on the same SM, so the next
// layer's router becomes resident while the current layer streams its
// weights.
template <int TM>
__global__ void __maxnreg__(TM <= 8 ? 104 : 224) decode_route_kernel(const DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t dsm[];  // x bf16 [T][H], then logits [T][E] fp32
    __shared__ int s_idx[MOE_DECODE_MAX_T * MOE_MAX_TOPK];
    __shared__ float s_w[MOE_DECODE_MAX_T * MOE_MAX_TOPK];
    __shared__ uint32_t s_mask[kMaxExperts];
    __shared__ int s_off[kMaxExperts];
    __shared__ __align__(8) uint64_t s_xbar;
    const int T = a.T, H = a.H, E = a.E, k = a.k;
    uint16_t* sx = reinterpret_cast<uint16_t*>(dsm);
    float* s_logits = reinterpret_cast<float*>(dsm + (size_t)T * H * 2);  // used in the leader
    const uint32_t rank = cluster_ctarank(), ncta = cluster_nctarank();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int W = (int)ncta * (kRouteThreads / 32);
    const int gw = (int)rank * (kRouteThreads / 32) + warp;
    const uint32_t xbar = smem_u32(&s_xbar);
    if (threadIdx.x == 0) {
        mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // This warp's first router row (its first 2048 columns) does not depend
    // on the preceding work: request it before waiting.
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
    pdl_wait();     // x and the workspace belong to this call from here on
    pdl_trigger();  // the expert grid may be scheduled; it waits for our end
    // the gate/up sums are accumulated over K parts by the expert kernel
    if (a.nsg > 1) {
        float4* z = reinterpret_cast<float4*>(a.gu_sum);
        const int n4 = T * k * 2 * a.I / 4;
        for (int i = (int)rank * kRouteThreads + threadIdx.x; i < n4; i += (int)ncta * kRouteThreads)
            z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // x into shared memory with one bulk copy
    if (threadIdx.x == 0) {
        fence_proxy_async_global();
        mbar_arrive_expect_tx(xbar, (uint32_t)(T * H * 2));
        bulk_g2s(smem_u32(sx), a.x, (uint32_t)(T * H * 2), xbar);
    }
    if (!mbar_wait(xbar, 0)) record_status(a.status, kStatusTimeout);

    const uint32_t leader_logits = mapa_shared(smem_u32(s_logits), 0);
    for (int e = gw; e < E; e += W) {
        float acc[TM], acc2[TM];  // two chains per token (columns 4c..4c+1 and 4c+2..4c+3)
#pragma unroll
        for (int t = 0; t < TM; ++t) acc[t] = acc2[t] = 0.f;
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
                            acc2[t] = fmaf(__uint_as_float(xv.y << 16), wv.z, acc2[t]);
                            acc2[t] = fmaf(__uint_as_float(xv.y & 0xffff0000u), wv.w, acc2[t]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            if (t < T) {
                const float v = warp_sum(acc[t] + acc2[t]);
                if (lane == 0) st_cluster_f32(leader_logits + (uint32_t)(t * E + e) * 4u, v);
            }
        }
    }
    // The logits are in the leader's shared memory once every CTA has
    // arrived (release); the int8 quantisation of x runs while the barrier
    // completes (its results are read only by the next kernel).
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    const int G = H / kGroup;
    for (int q = gw; q < T * G; q += W) {
        const int t = q / G, g = q % G;
        const float v = bf16_bits_to_float(sx[t * H + g * kGroup + lane]);
        const float amax = warp_max(fabsf(v));
        const uint16_t db = act_scale_bits(amax);
        a.q_x[(size_t)t * H + g * kGroup + lane] = (int8_t)act_code(v, half_bits_to_float(db));
        if (lane == 0) a.d_x[(size_t)t * G + g] = db;
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (rank != 0) return;

    // ---- leader CTA: top-k, weights, buckets, counters ----
    const int tid = threadIdx.x;
    const int Tk = T * k;
    if (T <= 2) {
        // Every thread: the rank of (token, expert) pairs among the token's
        // E logits (two threads per pair, half the experts each); the pairs
        // of rank < k are the choices, in rank order.  Then one thread per
        // (token, slot) pair and one per expert build the buckets; no loop
        // carries a dependence from one expert or pair to the next.
        __shared__ float s_val[2 * MOE_MAX_TOPK];
        for (int base = 0; base < 2 * T * E; base += kRouteThreads) {  // whole warps take part
            const int p2 = base + tid;
            const bool act = p2 < 2 * T * E;
            const int p = act ? p2 >> 1 : 0, half = p2 & 1;
            const int t = p / E, e = p % E;
            const float* lg = s_logits + t * E;
            const float v = lg[e];
            int rank = 0;
            const int e0 = half ? E / 2 : 0, e1 = act ? (half ? E : E / 2) : 0;
#pragma unroll 16
            for (int e2 = e0; e2 < e1; ++e2) {
                const float v2 = lg[e2];
                rank += (v2 > v) || (v2 == v && e2 < e);
            }
            rank += __shfl_xor_sync(0xffffffffu, rank, 1);  // pair of threads
            if (act && !half && rank < k) {
                s_idx[t * k + rank] = e;
                s_val[t * k + rank] = v;
            }
        }
        for (int e = tid; e < E; e += kRouteThreads) a.done[e] = 0;
        __syncthreads();
        // weights: softmax over the token's k chosen logits; bucket rows
        if (tid < Tk) {
            const int t = tid / k;
            const float m = s_val[t * k];
            float den = 0.f;
            for (int j = 0; j < k; ++j) den += expf(s_val[t * k + j] - m);
            const float w = expf(s_val[tid] - m) / den;
            s_w[tid] = w;
            a.topk_idx[tid] = s_idx[tid];
            a.topk_w[tid] = w;
        }
        for (int i = tid; i < T * E; i += kRouteThreads) a.logits[i] = s_logits[i];
        __syncthreads();
        if (T == 1) {
            // One token: its k experts are distinct, so an expert's bucket
            // offset is the number of chosen experts below it, which is also
            // a chosen expert's index in the touched list and its bucket row.
            for (int e = tid; e <= E; e += kRouteThreads) {
                int lt = 0;
#pragma unroll
                for (int j = 0; j < MOE_MAX_TOPK; ++j) lt += (j < k) && s_idx[j] < e;
                a.offsets[e] = lt;
            }
            if (tid < k) {
                const int ex = s_idx[tid];
                int pos = 0;
#pragma unroll
                for (int j = 0; j < MOE_MAX_TOPK; ++j) pos += (j < k) && s_idx[j] < ex;
                a.touched[pos] = ex;
                a.bucket_token[pos] = 0;
                a.bucket_slot[pos] = tid;
                a.slot_w[pos] = s_w[tid];
                a.slot_pos[tid] = pos;
            }
            if (tid == 0) a.counters[kCntTouched] = k;
            return;
        }
        __syncthreads();
    } else {
        for (int t = warp; t < T; t += kRouteThreads / 32) {
            int si;
            float sw;
            warp_topk(s_logits + t * E, E, k, si, sw);
            if (lane < k) {
                s_idx[t * k + lane] = si;
                s_w[t * k + lane] = sw;
                a.topk_idx[t * k + lane] = si;
                a.topk_w[t * k + lane] = sw;
            }
        }
        for (int i = tid; i < T * E; i += kRouteThreads) a.logits[i] = s_logits[i];
        for (int e = tid; e < E; e += kRouteThreads) a.done[e] = 0;
        __syncthreads();
    }
    if (Tk <= 32) {
        // One warp: counts per expert, a warp scan over the experts (eight
        // per lane) for the offsets and the list of touched experts, and each
        // (token, slot) pair's row: its expert's offset plus the number of
        // lower lanes (= earlier tokens) that chose the same expert.
        if (warp != 0) return;
        for (int e = lane; e < kMaxExperts; e += 32) s_off[e] = 0;
        __syncwarp();
        const bool act = lane < Tk;
        const int ex = act ? s_idx[lane] : 0;
        if (act) atomicAdd(&s_off[ex], 1);
        __syncwarp();
        constexpr int EPL = kMaxExperts / 32;
        int cnt[EPL];
        int tot = 0, ntl = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane * EPL + i;
            cnt[i] = e < E ? s_off[e] : 0;
            tot += cnt[i];
            ntl += cnt[i] > 0;
        }
        int inc = tot, incn = ntl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            const int vn = __shfl_up_sync(0xffffffffu, incn, o);
            if (lane >= o) {
                inc += v;
                incn += vn;
            }
        }
        int base = inc - tot, nbase = incn - ntl;
        __syncwarp();
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
        if (lane == 31) {
            a.offsets[E] = inc;
            a.counters[kCntTouched] = incn;
        }
        __syncwarp();
        const unsigned same = __match_any_sync(0xffffffffu, act ? ex : -1 - lane);
        if (act) {
            const int pos = s_off[ex] + __popc(same & ((1u << lane) - 1u));
            a.bucket_token[pos] = lane / k;
            a.bucket_slot[pos] = lane % k;
            a.slot_w[pos] = s_w[lane];
            a.slot_pos[lane] = pos;
        }
        return;
    }
    for (int e = tid; e < kMaxExperts; e += kRouteThreads) s_mask[e] = 0u;
    __syncthreads();
    // token t's bit in the mask of each expert it chose (T <= 32)
    for (int p = tid; p < Tk; p += kRouteThreads) atomicOr(&s_mask[s_idx[p]], 1u << (p / k));
    __syncthreads();
    const int e = tid;  // one thread per expert (E <= 256)
    const int cnt = (e < E) ? __popc(s_mask[e]) : 0;
    int total, ntouched;
    const int off = block256_exclusive_scan(cnt, &total);
    const int tpos = block256_exclusive_scan(cnt > 0 ? 1 : 0, &ntouched);
    if (e < E) {
        s_off[e] = off;
        a.offsets[e] = off;
        if (cnt > 0) a.touched[tpos] = e;
    }
    if (tid == 0) {
        a.offsets[E] = total;
        a.counters[kCntTouched] = ntouched;
    }
    __syncthreads();
    for (int p = tid; p < Tk; p += kRouteThreads) {
        const int t = p / k, j = p % k, ex = s_idx[p];
        const int pos = s_off[ex] + __popc(s_mask[ex] & ((1u << t) - 1u));
        a.bucket_token[pos] = t;
        a.bucket_slot[pos] = j;
        a.slot_w[pos] = s_w[p];
        a.slot_pos[p] = pos;
    }
}

// -------------------------------------------------------------- experts
template <int N>
struct IntC {
    static constexpr int value = N;
};

// At most 128 registers a thread, so that a route CTA of the next layer fits
// beside this CTA on its SM.
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

    const uint32_t actbar = smem_u32(&s_actbar);
    if (tid == 0) {
        for (int s = 0; s < kMaxSlots; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        mbar_init(actbar, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    pdl_wait();     // routing, buckets, x codes and cleared counters of this call
    pdl_trigger();  // the next layer's router may be scheduled
    for (int i = tid; i < kMaxExperts; i += kExpertThreads)
        s_touched[i] = (i < a.E) ? a.touched[i] : 0;  // entries past n_touched are unused
    if (tid == 0) s_nt = a.counters[kCntTouched];
    __syncthreads();
    const int nt = s_nt;
    const int G = gridDim.x, b = blockIdx.x;
    const int per_g = RBg * nsg, per_d = RBd * nsd;  // tasks per touched expert
    const int n_gu = nt * per_g, n_dn = nt * per_d;
    const int gu0 = (int)((long long)b * n_gu / G), gu1 = (int)((long long)(b + 1) * n_gu / G);
    const int dn0 = (int)((long long)b * n_dn / G), dn1 = (int)((long long)(b + 1) * n_dn / G);

    auto fail = [&]() {
        record_status(a.status, kStatusTimeout);
        s_abort = 1;
    };

    if (warp == kWarpProducer) {
        // ----------------------------------------------------------- producer
        // gate/up tasks, then down tasks; each task's tiles in chunks of up to
        // kChunkTiles contiguous tiles, one bulk copy per chunk.
        if (lane == 0) {
            int j = 0;  // ring position
            bool ok = true;
            for (int pass = 0; pass < 2 && ok; ++pass) {
                const bool gu = pass == 0;
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
    // 1. the int8 codes of x (every token) and their fp16 scales: two bulk
    //    copies, then the codes are permuted in place and summed per group
    if (tid == 0) {
        fence_proxy_async_global();
        const uint32_t sb = (uint32_t)act_scale_bytes(T, Gx);  // rounded up to 16 bytes
        mbar_arrive_expect_tx(actbar, (uint32_t)(T * H) + sb);
        bulk_g2s(smem_u32(ax_q), a.q_x, (uint32_t)(T * H), actbar);
        bulk_g2s(smem_u32(ax_dh), a.d_x, sb, actbar);
    }
    if (!mbar_wait(actbar, 0)) fail();
    for (int i = tid; i < T * Gx; i += kConsumerThreads) {
        uint2* g = reinterpret_cast<uint2*>(ax_q + (size_t)i * kGroup);
        int sum = 0;
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
            const uint2 v = g[c8];
            sum = __dp4a((int)v.x, 0x01010101, sum);  // signed byte sum
            sum = __dp4a((int)v.y, 0x01010101, sum);
            g[c8] = permute_chunk(v.x, v.y);
        }
        ax_s[i] = sum;
    }
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
            s_route[0] = a.offsets[ex];
            s_route[1] = a.offsets[ex + 1] - s_route[0];
        }
        consumers_sync();
        const int off = s_route[0], c = s_route[1];
        if (tid < c) {
            s_tok[tid] = a.bucket_token[off + tid];
            s_sw[tid] = a.slot_w[off + tid];
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
            const int off = s_route[0], c = s_route[1];
            const bool store = a.write_qh && rb == 0 && kc == 0;
            // four groups per warp at a time, every load first
            for (int q0 = warp; q0 < (have_h ? c * Gh : 0); q0 += 4 * kConsumerWarps) {
                float gv[4], uv[4];
#pragma unroll
                for (int o = 0; o < 4; ++o) {
                    const int q = q0 + o * kConsumerWarps;
                    const bool ld = q < c * Gh;
                    const float* gs = a.gu_sum + (size_t)(off + (ld ? q / Gh : 0)) * 2 * I +
                                      (ld ? q % Gh : 0) * kGroup + lane;
                    gv[o] = ld ? __ldcg(gs) : 0.f;
                    uv[o] = ld ? __ldcg(gs + I) : 0.f;
                }
#pragma unroll
                for (int o = 0; o < 4; ++o) {
                    const int q = q0 + o * kConsumerWarps;
                    if (q >= c * Gh) continue;  // warp-uniform
                    const int n = q / Gh, gg = q % Gh, f = gg * kGroup + lane;
                    const float h = gv[o] / (1.0f + __expf(-gv[o])) * uv[o];
                    const float amax = warp_max(fabsf(h));
                    const uint16_t db = act_scale_bits(amax);
                    const int qv = act_code(h, half_bits_to_float(db));
                    ah_q[(size_t)n * I + gg * kGroup + permuted_pos(lane)] = (uint8_t)(int8_t)qv;
                    int sum = qv;
#pragma unroll
                    for (int o2 = 16; o2 > 0; o2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
                    if (lane == 0) {
                        ah_d[n * Gh + gg] = half_bits_to_float(db);
                        ah_s[n * Gh + gg] = sum;
                    }
                    if (store) {
                        a.q_h[(size_t)(off + n) * I + f] = (int8_t)qv;
                        if (lane == 0) a.d_h[(size_t)(off + n) * Gh + gg] = db;
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
    pdl_wait();     // the expert kernel's y parts
    pdl_trigger();  // the next layer's router may be scheduled
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

// Cluster size of the route kernel: 16 CTAs where the device can place such a
// cluster, else the portable 8.  Cached per device and shared-memory size.
template <int TM>
int route_cluster_size(int dev, size_t smem) {
    static int cache[64] = {};
    static size_t cache_smem[64] = {};
    int& cs = cache[dev & 63];
    if (cs != 0 && cache_smem[dev & 63] == smem) return cs;
    cache_smem[dev & 63] = smem;
    cudaFuncSetAttribute(decode_route_kernel<TM>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaFuncSetAttribute(decode_route_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
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
    a.nslot = ns;
    a.off_bar = ns * kSlotBytes;
    a.off_ax = al(a.off_bar + bars);
    a.off_ah = a.off_ax + ax;
    return true;
}

int expert_smem_bytes(const DecodeArgs& a) {
    return a.off_ah + ((a.T * a.I + a.T * (a.I / kGroup) * 8 + 127) & ~127);
}

template <int TM>
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
    // ---- route ----
    const size_t rsm = (size_t)a.T * a.H * 2 + (size_t)a.T * a.E * 4;
    const int cs = route_cluster_size<TM>(dev, rsm);
    if (cs > 8) {
        err = cudaFuncSetAttribute(decode_route_kernel<TM>,
                                   cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess) return err;
    }
    err = cudaFuncSetAttribute(decode_route_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)rsm);
    if (err != cudaSuccess) return err;
    {
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute at[2];
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = rsm;
        cfg.stream = s;
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = cs;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        at[1] = pdl;
        cfg.attrs = at;
        cfg.numAttrs = 2;
        err = cudaLaunchKernelEx(&cfg, decode_route_kernel<TM>, a);
        if (err != cudaSuccess) return err;
    }
    for (int i = 1; i <= 3; ++i)
        if ((err = mark(i)) != cudaSuccess) return err;
    // ---- experts ----
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
    if ((err = mark(4)) != cudaSuccess || (err = mark(5)) != cudaSuccess) return err;
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
    if (!plan_experts(a)) return cudaErrorInvalidValue;
    if (T <= 1) return launch_all<1>(a, num_sms, events, capturing, s);
    if (T <= 2) return launch_all<2>(a, num_sms, events, capturing, s);
    if (T <= 4) return launch_all<4>(a, num_sms, events, capturing, s);
    if (T <= 8) return launch_all<8>(a, num_sms, events, capturing, s);
    if (T <= 16) return launch_all<16>(a, num_sms, events, capturing, s);
    return launch_all<32>(a, num_sms, events, capturing, s);
}

}  // namespace moeq4
