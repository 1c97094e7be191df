// Prefill grouped GEMM on the 5th-generation tensor cores (tcgen05).
//
// Page "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU",
// Methodology 1 "Prefill (GPU)": a grouped 4-bit GEMM over the tokens routed
// to each expert, run over the whole prompt in one pass (Methodology 4,
// "Single-Pass Prefill": the batch is as large as possible).  There it ran on
// a Fermi GPU without tensor cores; here each expert's token bucket is one
// operand of tcgen05.mma with fp16 inputs and fp32 accumulators in tensor
// memory.  fp16 rather than bf16: the dequantised weights d(q - 8), the bf16
// hidden states (exact in fp16 within its range) and h keep 3 more mantissa
// bits, which cuts the layer's error against exact arithmetic about tenfold
// at the same tensor-core rate.
//
// Weights sit on the MMA's M side (128 rows per tile) and tokens on N (up to
// 160 per tile, padded to a multiple of 16; larger buckets are cut into
// tiles of near-equal size), so an expert's bucket of ~128 tokens is one
// tile and every weight is dequantised once.  160 is the widest accumulator
// that leaves each matrix's 256 tensor-memory columns room for three A
// stages; the operand stream costs about the same per K-block whatever the
// tile's width, so fewer, wider tiles are faster.  Per 64-column
// K-block, three decoupled rings:
//   raw    the packed 4-bit tiles (4608 bytes each), two K-blocks of each
//          weight block per bulk copy (contiguous in the packed layout), by
//          the weight producer warp ten K-blocks ahead (these come from HBM);
//   A      the dequantised fp16 weights, in tensor memory (one weight row per
//          TMEM lane, written by eight dequant warps with tcgen05.st; the MMA
//          reads A from TMEM), which leaves shared memory to the two rings
//          that wait on memory;
//   B      the bucket's token rows, brought in by four token-loader warps
//          with 16-byte cp.async copies straight into the 128-byte-swizzled
//          layout (gate/up: rows of x picked by token id; down: consecutive
//          rows of h), six K-blocks deep; they mostly hit L2.  (Many small
//          TMA copies - gather4 or 16-row boxes - proved slower here: the
//          copy engine spent ~40 ns on each.)
// A K-block costs ~0.63 us per CTA against 0.3 us for its MMAs alone; the
// difference is spread over the hand-offs between these roles (each ring
// is released by MMA completions) rather than set by one operand stream.
// The weight copies carry an L2 evict-first hint: they are read once, and
// should not push the reused token rows out of L2.
// One thread of the MMA warp issues 4 x K=16 MMAs per matrix into TMEM; twelve
// epilogue warps (the tensor pipe waits while they drain the accumulators)
// read TMEM: gate/up -> h = silu(g) * u, down -> y = routing
// weight * acc, both fp16 (saturating at +-65504), in bucket order.
// Both GEMMs run in one launch: one persistent CTA per SM walks a static
// round-robin list of work items, first every gate/up item (token tile, 128
// rows of h), then every down item (token tile, 256 rows of y).  A down item
// reads the h rows of its token tile, so its token loaders wait until the
// tile's gate/up items have all published theirs (a per-tile count each
// epilogue warp raises with release semantics after storing its rows; a
// bounded acquire spin).  The launch is cooperative, so every CTA is
// resident, and every CTA finishes its gate/up items before its down items,
// so the waits always end; the CTAs
// that finish the gate/up items early go on to down items instead of idling
// until the last gate/up item is done.  The kernel is launched with
// programmatic dependent launch:
// the weight producer and the dequant warps start on their first weight
// tiles (which depend only on the tile list, two kernels back) while the
// preceding kernel drains; the token loaders, the MMA and the epilogue wait
// for it first.  Every wait is bounded; on expiry the CTA records
// MOE_ERR_TIMEOUT in the status word, stops, drains its copies, frees TMEM
// and exits.
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int BN = 160;                 // max tokens per tile (buckets are cut evenly)
constexpr int B_BYTES = BN * 128;       // BN rows x 64 fp16
constexpr int NUM_EPI_WARPS = 12, NUM_DEQ_WARPS = 8, NUM_B_WARPS = 4;
constexpr int WARP_WPROD = 0, WARP_MMA = 1, WARP_B0 = 2;
constexpr int WARP_EPI0 = WARP_B0 + NUM_B_WARPS;
constexpr int WARP_DEQ0 = WARP_EPI0 + NUM_EPI_WARPS;
constexpr int NUM_THREADS = (WARP_DEQ0 + NUM_DEQ_WARPS) * 32;  // 26 warps
constexpr int B_ROWS_PER_THREAD = BN * 8 / (NUM_B_WARPS * 32);  // 16-byte chunks: 10
static_assert(BN * 8 % (NUM_B_WARPS * 32) == 0, "B chunks per loader thread");

// Both GEMMs multiply two 128-row weight blocks by the same token tile:
// gate/up the gate rows and the matching up rows, down two adjacent row
// blocks of W_d (so each token row is read from L2 once per 256 output rows).
struct Cfg {
    static constexpr int NMAT = 2;
    static constexpr int RK = 2;  // K-blocks per weight copy (contiguous tiles)
    static constexpr int RAW_STAGES = 5;
    static constexpr int A_STAGES = 3;  // in tensor memory
    static constexpr int B_STAGES = 6;
    static constexpr int RAW_BYTES = NMAT * RK * kTileBytes;
    // tensor memory: accumulator m at column m * 256 (BN columns); A stage s
    // of matrix m at column m * 256 + A_COL0 + s * 32 (64 fp16 per row, two
    // per column), in the columns the accumulator leaves free
    static constexpr int A_COL0 = 160;
    static constexpr int TMEM_COLS = NMAT * 256;
    static_assert(BN <= A_COL0 && A_COL0 + A_STAGES * 32 <= 256, "tensor memory budget");
    // shared memory carve-up (offsets from a 1024-aligned base)
    static constexpr int OFF_B = 0;
    static constexpr int OFF_RAW = OFF_B + B_STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_RAW + RAW_STAGES * RAW_BYTES;
    static constexpr int NUM_BARS = 2 * RAW_STAGES + A_STAGES + 2 * B_STAGES + 3;
    static_assert(B_STAGES > A_STAGES, "A stages are freed through the token-stage barriers");
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    // per epilogue warp: a 16-token x 32-feature fp16 transpose buffer
    static constexpr int OFF_STAGE = (OFF_TMEM + 16 + 127) & ~127;
    static_assert(OFF_STAGE % 128 == 0, "16-byte vector access into the transpose buffers");
    static constexpr int SMEM_BYTES = OFF_STAGE + NUM_EPI_WARPS * 1024 + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// One of the two GEMMs (0: gate/up, 1: down).
struct GemmOp {
    const uint8_t* wpk;        // packed weights
    const uint16_t* bsrc;      // fp16 token rows: x16 [T, H] (gate/up) or h [T*k, I] (down)
    uint16_t* out;             // h [T*k, I] (gate/up) or y [T*k, H] (down)
    int K;                     // reduction length: H (gate/up) or I (down)
    int rows_per_e;            // packed rows per expert: 2I (gate/up) or H (down)
    int rb_items;              // work items per token tile: I/128 or H/256
    int rb_mul;                // first row block of item i: i * rb_mul (1 or 2)
    int rb_second;             // second row block = first + rb_second (I/128 or 1)
    int out_ld;                // leading dimension of out
};

struct GemmArgs {
    GemmOp op[2];
    const int32_t* counters;   // kCntTiles
    const int32_t* tile_e;
    const int32_t* tile_n0;
    const int32_t* tile_nn;
    const int32_t* bucket_token;
    const float* slot_w;
    int* tile_done;            // [max_tiles] gate/up epilogue warps done per token tile
                               // (zeroed by the bucket scan before every call)
    int* status;
};

// Work item w of the combined list: its GEMM, token tile, row-block index
// and K-blocks.
struct Item {
    int op, tile, ri, KB;
};
__device__ __forceinline__ Item item_of(const GemmOp* ops, int w, int n_gu) {
    Item it;
    it.op = w < n_gu ? 0 : 1;
    const int wl = it.op ? w - n_gu : w;
    it.tile = wl / ops[it.op].rb_items;
    it.ri = wl % ops[it.op].rb_items;
    it.KB = ops[it.op].K / kTileK;
    return it;
}

// Eight 4-bit codes of one packed word (columns 8c..8c+7: even columns in the
// low 16 bits, odd in the high, nibble m = column pair m) to fp16 d(q - 8).
// 0x6400 is fp16 1024 with ulp 1, so (0x6400 | q) is 1024 + q and
// (0x6400 | q << 4) is 1024 + 16 q: q - 8 comes out exactly as
// (1024 + q) - 1032 or (1024 + 16 q) / 16 - 72, and one rounding of (q - 8) d
// follows.
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t d2) {
    const uint32_t w8 = w >> 8;
    uint32_t t[4];
    asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(t[0]) : "r"(w));
    asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(t[1]) : "r"(w));
    asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(t[2]) : "r"(w8));
    asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(t[3]) : "r"(w8));
    const __half2 k1032 = __floats2half2_rn(1032.0f, 1032.0f);
    const __half2 k16th = __floats2half2_rn(0.0625f, 0.0625f);
    const __half2 km72 = __floats2half2_rn(-72.0f, -72.0f);
    const __half2 d = *reinterpret_cast<const __half2*>(&d2);
    __half2 v[4];
    v[0] = __hsub2(*reinterpret_cast<const __half2*>(&t[0]), k1032);
    v[1] = __hfma2(*reinterpret_cast<const __half2*>(&t[1]), k16th, km72);
    v[2] = __hsub2(*reinterpret_cast<const __half2*>(&t[2]), k1032);
    v[3] = __hfma2(*reinterpret_cast<const __half2*>(&t[3]), k16th, km72);
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 r = __hmul2(v[i], d);
        op[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
    return o;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_q4_gemm_kernel(const GemmArgs args) {
    using C = Cfg;
    constexpr int SR = C::RAW_STAGES, SA = C::A_STAGES, SB = C::B_STAGES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ GemmOp ops[2];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw_base);

    const int n_tiles = args.counters[kCntTiles];
    const int n_gu = n_tiles * args.op[0].rb_items;
    const int n_items = n_gu + n_tiles * args.op[1].rb_items;
    if ((int)blockIdx.x >= n_items) return;
    // a down item's h rows are complete once every epilogue warp of each of
    // the tile's gate/up items has counted itself
    const int tile_ready = NUM_EPI_WARPS * args.op[0].rb_items;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const uint32_t bar0 = base + C::OFF_BAR;
    auto raw_full = [&](int s) { return bar0 + 8u * s; };
    auto raw_empty = [&](int s) { return bar0 + 8u * (SR + s); };
    // (no "A empty" barriers: the MMA commits once per K-block, to its
    // token-row stage, and A stage it % SA is free again once K-block it - SA
    // has completed, which that commit shows; SB > SA keeps the phase of
    // K-block it - SA the latest one the dequant can see on that barrier)
    auto a_full = [&](int s) { return bar0 + 8u * (2 * SR + s); };
    auto b_full = [&](int s) { return bar0 + 8u * (2 * SR + SA + s); };
    auto b_empty = [&](int s) { return bar0 + 8u * (2 * SR + SA + SB + s); };
    const uint32_t acc_full = bar0 + 8u * (2 * SR + SA + 2 * SB);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t mma_done = acc_full + 16u;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + C::OFF_TMEM + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + C::OFF_TMEM);

    if (threadIdx.x == 0) {
        ops[0] = args.op[0];
        ops[1] = args.op[1];
        for (int s = 0; s < SR; ++s) {
            mbar_init(raw_full(s), 1);
            mbar_init(raw_empty(s), NUM_DEQ_WARPS);
        }
        for (int s = 0; s < SA; ++s) mbar_init(a_full(s), NUM_DEQ_WARPS);
        for (int s = 0; s < SB; ++s) {
            mbar_init(b_full(s), NUM_B_WARPS * 32);
            mbar_init(b_empty(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, NUM_EPI_WARPS);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(base + C::OFF_TMEM, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        record_status(args.status, kStatusTimeout);
        *abort_flag = 1;
    };

    if (warp == WARP_WPROD) {
        // ------------------------------------------------ weight (raw) producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int it = 0;  // global K-block counter
            bool ok = true;
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
                const Item im = item_of(ops, w, n_gu);
                const GemmOp& o = ops[im.op];
                const int e = args.tile_e[im.tile];
                const int rbs_per_e = o.rows_per_e / kTileRows;
                const int rb0 = im.ri * o.rb_mul;
                // an odd last block of W_d has no partner: load it twice (the
                // epilogue drops the copy)
                const int rb1 = (rb0 + o.rb_second < rbs_per_e) ? rb0 + o.rb_second : rb0;
                // im.KB packed tiles per (expert, row block)
                const uint8_t* wt0 = o.wpk + ((size_t)e * rbs_per_e + rb0) * im.KB * kTileBytes;
                const uint8_t* wt1 = o.wpk + ((size_t)e * rbs_per_e + rb1) * im.KB * kTileBytes;
                for (int kb = 0; kb < im.KB; kb += C::RK, ++it) {
                    const int s = it % SR;
                    if (*abort_flag || !mbar_wait(raw_empty(s), ((it / SR) & 1) ^ 1)) {
                        fail();
                        ok = false;
                        break;
                    }
                    const uint32_t raw = base + C::OFF_RAW + s * C::RAW_BYTES;
                    constexpr uint32_t half = C::RK * kTileBytes;
                    mbar_arrive_expect_tx(raw_full(s), C::RAW_BYTES);
                    bulk_g2s_hint(raw, wt0 + (size_t)kb * kTileBytes, half, raw_full(s), pol);
                    bulk_g2s_hint(raw + half, wt1 + (size_t)kb * kTileBytes, half, raw_full(s), pol);
                }
            }
            // the copies already issued land before the CTA can go away
            for (int j = (it > SR ? it - SR : 0); j < it; ++j) mbar_wait(raw_full(j % SR), (j / SR) & 1);
        }
    } else if (warp >= WARP_B0 && warp < WARP_B0 + NUM_B_WARPS) {
        // ----------------------------------------------- token-row loaders
        // thread bt: 16-byte chunk c = bt % 8 of rows bt / 8 + 16 i
        pdl_wait();  // the token rows and bucket lists of the preceding kernels
        pdl_trigger();
        const int bt = threadIdx.x - WARP_B0 * 32;
        const int c = bt % 8, r0 = bt / 8;
        int it = 0, issued = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
            const Item im = item_of(ops, w, n_gu);
            const GemmOp& o = ops[im.op];
            const int n0 = args.tile_n0[im.tile], nn = args.tile_nn[im.tile];
            const int npad = (nn + 15) & ~15;
            if (im.op == 1) {  // the tile's h rows: wait for its gate/up items
                const int* done = args.tile_done + im.tile;
                if (ld_acquire(done) < tile_ready) {
                    const unsigned long long t0 = globaltimer_ns();
                    while (ld_acquire(done) < tile_ready) {
                        if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) {
                    fail();
                    break;
                }
            }
            const uint16_t* src[B_ROWS_PER_THREAD];
#pragma unroll
            for (int i = 0; i < B_ROWS_PER_THREAD; ++i) {
                const int r = r0 + 16 * i;
                const int rr = r < nn ? r : 0;  // padding rows repeat row 0
                const size_t row = im.op == 0 ? (size_t)args.bucket_token[n0 + rr] : (size_t)(n0 + rr);
                src[i] = o.bsrc + row * o.K + c * 8;
            }
            for (int kb = 0; kb < im.KB; ++kb, ++it) {
                const int s = it % SB;
                if (*abort_flag || !mbar_wait(b_empty(s), ((it / SB) & 1) ^ 1)) {
                    fail();
                    ok = false;
                    break;
                }
                const uint32_t bsm = base + C::OFF_B + s * B_BYTES;
#pragma unroll
                for (int i = 0; i < B_ROWS_PER_THREAD; ++i) {
                    const int r = r0 + 16 * i;
                    if (r < npad)
                        cp_async16(bsm + r * 128 + ((c ^ (r & 7)) * 16), src[i] + kb * kTileK);
                }
                cp_async_arrive_noinc(b_full(s));
                ++issued;
            }
        }
        // the copies already issued land before the CTA can go away
        for (int j = (issued > SB ? issued - SB : 0); j < issued; ++j)
            mbar_wait(b_full(j % SB), (j / SB) & 1);
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------------------------- MMA
        pdl_wait();
        pdl_trigger();
        int it = 0, item = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++item) {
            const Item im = item_of(ops, w, n_gu);
            const int nn = args.tile_nn[im.tile];
            const int npad = (nn + 15) & ~15;
            const uint32_t idesc = idesc_f16_f32(128, npad);
            if (*abort_flag || !mbar_wait(acc_empty, (item & 1) ^ 1)) {
                fail();
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kb = 0; kb < im.KB; ++kb, ++it) {
                const int sa = it % SA, sb = it % SB;
                if (*abort_flag || !mbar_wait(b_full(sb), (it / SB) & 1) ||
                    !mbar_wait(a_full(sa), (it / SA) & 1)) {
                    fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
                fence_proxy_async_smem();  // token rows were written by cp.async (generic proxy)
                if (lane == 0) {
                    const uint32_t b_sm = base + C::OFF_B + sb * B_BYTES;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bdesc = sw128_kmajor_desc(b_sm + kk * 32);
#pragma unroll
                        for (int m = 0; m < C::NMAT; ++m) {
                            const uint32_t a_t = tmem + m * 256 + C::A_COL0 + sa * 32 + kk * 8;
                            mma_f16_ta(tmem + m * 256, a_t, bdesc, idesc, (kb | kk) != 0);
                        }
                    }
                    mma_commit(b_empty(sb));  // frees token stage sb and A stage sa
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) mma_commit(acc_full);
            __syncwarp();
        }
        // wait for every MMA issued here before TMEM can be released
        if (lane == 0) {
            mma_commit(mma_done);
            mbar_wait(mma_done, 0);
        }
        __syncwarp();
    } else if (warp >= WARP_DEQ0) {
        // ------------------------------------------------------------ dequant
        // thread = one weight row: warp w handles rows 32 (w % 4) .. +31 (its
        // TMEM lane quarter) of matrix (w - WARP_DEQ0) / 4; per K-block it
        // reads the row's 32 code bytes and 2 scales and writes its 64 fp16
        // weights to the A stage in tensor memory (32 columns)
        const int quad = warp % 4, mm = (warp - WARP_DEQ0) / 4;
        const int r = quad * 32 + lane;
        const uint32_t tlane = (uint32_t)(quad * 32) << 16;
        int it = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
            const int KB = item_of(ops, w, n_gu).KB;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int ir = it / C::RK, sub = it % C::RK;  // weight copy and its K-block
                const int sr = ir % SR, sa = it % SA;
                const bool bad =
                    *abort_flag || !mbar_wait(raw_full(sr), (ir / SR) & 1) ||
                    (it >= SA && !mbar_wait(b_empty((it - SA) % SB), ((it - SA) / SB) & 1));
                if (__any_sync(0xffffffffu, bad)) {  // tcgen05.st below needs the whole warp
                    fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* t = sbase + C::OFF_RAW + sr * C::RAW_BYTES +
                                   mm * (C::RK * kTileBytes) + sub * kTileBytes;
                const uint4 c0 = *reinterpret_cast<const uint4*>(t + r * 32);
                const uint4 c1 = *reinterpret_cast<const uint4*>(t + r * 32 + 16);
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(t + kTileCodeBytes + r * 4);
                __syncwarp();
                if (lane == 0 && sub == C::RK - 1) mbar_arrive(raw_empty(sr));  // copy read
                const uint32_t d0 = (sc & 0xFFFFu) * 0x10001u, d1 = (sc >> 16) * 0x10001u;
                const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint32_t o[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 v = dequant8(words[i], i < 4 ? d0 : d1);
                    o[4 * i] = v.x;
                    o[4 * i + 1] = v.y;
                    o[4 * i + 2] = v.z;
                    o[4 * i + 3] = v.w;
                }
                tmem_st32(tmem + tlane + mm * 256 + C::A_COL0 + sa * 32, o);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_full(sa));
            }
        }
    } else {
        // ----------------------------------------------------------- epilogue
        // warp w reads TMEM lanes 32 (w % 4) .. +31 (one accumulator row per
        // thread); the three warps of a lane quarter take every third
        // 16-column chunk, each loading 2 x 16 columns before one wait
        constexpr int kEpiPerQuad = NUM_EPI_WARPS / 4;
        static_assert(NUM_EPI_WARPS % 4 == 0, "whole lane quarters");
        const int quad = warp % 4, half = (warp - WARP_EPI0) / 4;  // 0 .. kEpiPerQuad - 1
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        pdl_wait();  // the output buffer and routing weights of the preceding kernels
        pdl_trigger();
        int item = 0;
        for (int w = blockIdx.x; w < n_items; w += gridDim.x, ++item) {
            const Item im = item_of(ops, w, n_gu);
            const GemmOp& o = ops[im.op];
            const bool gateup = im.op == 0;
            const int tile = im.tile, ri = im.ri;
            const int rbs_per_e = o.rows_per_e / kTileRows;
            const int n0 = args.tile_n0[tile], nn = args.tile_nn[tile];
            const bool bad = *abort_flag || !mbar_wait(acc_full, item & 1);
            if (__any_sync(0xffffffffu, bad)) {  // tcgen05.ld below needs the whole warp
                fail();
                break;
            }
            tc_fence_after();
            const bool second = ri * o.rb_mul + o.rb_second < rbs_per_e;  // down: partner exists
            // 16 columns (tokens) x 32 rows (features) go through the warp's
            // transpose buffer so that each lane stores 8 consecutive features
            // of one token (16 bytes): two 16-byte stores per lane instead of
            // sixteen 2-byte ones
            uint16_t* stg = reinterpret_cast<uint16_t*>(sbase + C::OFF_STAGE) + (warp - WARP_EPI0) * 512;
            const int fbase = ri * o.rb_mul * kTileRows + quad * 32;
            auto flush = [&](int c0, int fo) {
                __syncwarp();
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int tok = r * 8 + lane / 4, ch = lane % 4;
                    const uint4 v = *reinterpret_cast<const uint4*>(stg + tok * 32 + ch * 8);
                    if (c0 + tok < nn)
                        *reinterpret_cast<uint4*>(o.out + (size_t)(n0 + c0 + tok) * o.out_ld +
                                                  fbase + fo + ch * 8) = v;
                }
                __syncwarp();
            };
            for (int c0 = half * 16; c0 < nn; c0 += 16 * kEpiPerQuad) {
                uint32_t g[16], u[16];
                tmem_ld16(trow + c0, g);
                tmem_ld16(trow + 256 + c0, u);
                tmem_ld_wait();
                if (gateup) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
                        // silu(g) u; the result is rounded to fp16 next, so the
                        // fast reciprocal division is ample
                        const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                        stg[j * 32 + lane] = float_to_half_bits_sat(hv);
                    }
                    flush(c0, 0);
                } else {
                    float sw[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        sw[j] = (c0 + j < nn) ? __ldg(args.slot_w + n0 + c0 + j) : 0.0f;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        stg[j * 32 + lane] = float_to_half_bits_sat(__uint_as_float(g[j]) * sw[j]);
                    flush(c0, 0);
                    if (second) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            stg[j * 32 + lane] = float_to_half_bits_sat(__uint_as_float(u[j]) * sw[j]);
                        flush(c0, kTileRows);
                    }
                }
            }
            tc_fence_before();
            if (gateup) {  // this warp's rows of h are stored: count them for the tile
                __threadfence();
                __syncwarp();
                if (lane == 0) red_release_add(args.tile_done + tile, 1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace

cudaError_t launch_prefill_experts(const void* wgu, const void* wd, const Workspace& ws, int H,
                                   int I, int* status, int num_sms, cudaStream_t s) {
    GemmArgs a{};
    GemmOp& g = a.op[0];
    g.wpk = static_cast<const uint8_t*>(wgu);
    g.bsrc = ws.x16;
    g.out = ws.h;
    g.K = H;
    g.rows_per_e = 2 * I;
    g.rb_items = I / kTileRows;
    g.rb_mul = 1;
    g.rb_second = I / kTileRows;  // the matching up rows
    g.out_ld = I;
    GemmOp& d = a.op[1];
    d.wpk = static_cast<const uint8_t*>(wd);
    d.bsrc = ws.h;
    d.out = static_cast<uint16_t*>(ws.y);
    d.K = I;
    d.rows_per_e = H;
    d.rb_items = (H / kTileRows + 1) / 2;
    d.rb_mul = 2;
    d.rb_second = 1;  // the next row block
    d.out_ld = H;
    a.counters = ws.counters;
    a.tile_e = ws.tile_e;
    a.tile_n0 = ws.tile_n0;
    a.tile_nn = ws.tile_nn;
    a.bucket_token = ws.bucket_token;
    a.slot_w = ws.slot_w;
    a.tile_done = ws.tile_done;
    a.status = status;
    cudaError_t err = cudaFuncSetAttribute(grouped_q4_gemm_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    // Cooperative: the down items wait on gate/up items of other CTAs, so
    // every CTA must be resident at once, also when other work holds SMs.
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[2];
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = (cooperative_pdl_mode(dev) == 2) ? 1 : 2;
    return cudaLaunchKernelEx(&cfg, grouped_q4_gemm_kernel, a);
}

}  // namespace moeq4
