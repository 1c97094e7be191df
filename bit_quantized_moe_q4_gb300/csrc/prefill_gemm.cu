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
// 256 per tile, padded to a multiple of 16), so a bucket of ~128 tokens wastes
// little.  Per 64-column K-block:
//   producer warp   bulk-copies the packed 4-bit tile(s) (4608 bytes each)
//                   and brings the bucket's token rows in: gate/up gathers
//                   rows of x by token id (TMA gather4), down loads
//                   consecutive rows of h (2-D TMA tiles);
//   dequant warps   turn codes and fp16 scales into fp16 w = d (q - 8) in the
//                   128-byte-swizzled K-major layout the MMA reads;
//   MMA warp        one thread issues 4 x K=16 MMAs per matrix into TMEM;
//   epilogue warps  read TMEM: gate/up -> h = silu(g) * u, down ->
//                   y = w_route * acc, both fp16 (saturating at +-65504), in
//                   bucket order.
// One persistent CTA per SM walks a static list of (token tile, row block)
// work items.  Every wait is bounded; on expiry the CTA records
// MOE_ERR_TIMEOUT in the status word, drains its copies, frees TMEM and exits.
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

constexpr int BN = 256;           // max tokens per tile
constexpr int A_MAT_BYTES = 128 * 128;  // 128 rows x 64 fp16
constexpr int B_BYTES = BN * 128;       // BN rows x 64 fp16
constexpr int NUM_THREADS = 448;  // 14 warps
constexpr int WARP_PRODUCER = 0, WARP_MMA = 1, WARP_EPI0 = 2, WARP_DEQ0 = 6;
constexpr int NUM_EPI_WARPS = 4, NUM_DEQ_WARPS = 8;

template <bool GATEUP>
struct Cfg {
    static constexpr int NMAT = GATEUP ? 2 : 1;
    static constexpr int STAGES = GATEUP ? 3 : 4;
    static constexpr int RAW_BYTES = NMAT * kTileBytes;
    static constexpr int A_BYTES = NMAT * A_MAT_BYTES;
    static constexpr int TMEM_COLS = NMAT * 256;
    // shared memory carve-up (offsets from a 1024-aligned base)
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_RAW = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_RAW + STAGES * RAW_BYTES;
    static constexpr int NUM_BARS = 4 * STAGES + 3;
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_TMEM + 16 + 1024;  // + alignment slack
};

struct GemmArgs {
    const uint8_t* wpk;        // packed weights
    const int32_t* counters;   // kCntTiles
    const int32_t* tile_e;
    const int32_t* tile_n0;
    const int32_t* tile_nn;
    const int32_t* bucket_token;
    const float* slot_w;
    uint16_t* out;             // h [T*k, I] (gate/up) or y [T*k, H] (down)
    int K;                     // reduction length: H (gate/up) or I (down)
    int rows_per_e;            // packed rows per expert: 2I (gate/up) or H (down)
    int out_rows;              // output features per expert: I or H
    int out_ld;                // leading dimension of out
    int* status;
};

__device__ __forceinline__ uint32_t f16x2_dequant(uint32_t nib2, uint32_t d2) {
    // nib2 holds two codes at bits 0..3 and 16..19; 0x6400 is fp16 1024.0 and
    // its ulp is 1, so (0x6400 | q) is exactly 1024 + q.
    const uint32_t v = nib2 | 0x64006400u;
    __half2 b = *reinterpret_cast<const __half2*>(&v);
    const __half2 off = __floats2half2_rn(1032.0f, 1032.0f);  // 1024 + 8
    const __half2 d = *reinterpret_cast<const __half2*>(&d2);
    b = __hmul2(__hsub2(b, off), d);  // (q - 8) exact, then one rounding of d(q-8)
    return *reinterpret_cast<uint32_t*>(&b);
}

template <bool GATEUP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_q4_gemm_kernel(const __grid_constant__ CUtensorMap bmap, const GemmArgs args) {
    using C = Cfg<GATEUP>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw_base);

    const int n_items_tiles = args.counters[kCntTiles];
    const int rb_count = args.out_rows / kTileRows;
    const int n_items = n_items_tiles * rb_count;
    if ((int)blockIdx.x >= n_items) return;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int KB = args.K / kTileK;
    const int tiles_per_rb = KB;  // packed tiles per (expert, row block)
    const int rbs_per_e = args.rows_per_e / kTileRows;

    const uint32_t bar0 = base + C::OFF_BAR;
    auto full_raw = [&](int s) { return bar0 + 8u * s; };
    auto full_b = [&](int s) { return bar0 + 8u * (S + s); };
    auto full_a = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto empty = [&](int s) { return bar0 + 8u * (3 * S + s); };
    const uint32_t acc_full = bar0 + 8u * (4 * S);
    const uint32_t acc_empty = bar0 + 8u * (4 * S + 1);
    const uint32_t mma_done = bar0 + 8u * (4 * S + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + C::OFF_TMEM + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + C::OFF_TMEM);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_raw(s), 1);
            mbar_init(full_b(s), 1);
            mbar_init(full_a(s), NUM_DEQ_WARPS);
            mbar_init(empty(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, NUM_EPI_WARPS);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_PRODUCER && lane == 0) prefetch_tensormap(&bmap);
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

    if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ producer
        int it = 0;  // global K-block counter
        int issued = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
            const int tile = w / rb_count, rb = w % rb_count;
            const int e = args.tile_e[tile], n0 = args.tile_n0[tile], nn = args.tile_nn[tile];
            const int npad = (nn + 15) & ~15;
            // token rows for the gathers: lane handles 4-row groups lane, lane+32
            int rows[8];
            if (GATEUP) {
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = (lane + 32 * q) * 4 + i;
                        rows[q * 4 + i] = args.bucket_token[n0 + (r < nn ? r : 0)];
                    }
            }
            const uint8_t* wtile =
                args.wpk + ((size_t)e * rbs_per_e + rb) * tiles_per_rb * kTileBytes;
            const uint8_t* wtile_up =
                args.wpk + ((size_t)e * rbs_per_e + rb + rb_count) * tiles_per_rb * kTileBytes;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % S;
                const uint32_t ph = (it / S) & 1;
                if (*abort_flag || !mbar_wait(empty(s), ph ^ 1)) {
                    fail();
                    ok = false;
                    break;
                }
                const uint32_t raw = base + C::OFF_RAW + s * C::RAW_BYTES;
                const uint32_t bsm = base + C::OFF_B + s * B_BYTES;
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_raw(s), C::RAW_BYTES);
                    bulk_g2s(raw, wtile + (size_t)kb * kTileBytes, kTileBytes, full_raw(s));
                    if (GATEUP)
                        bulk_g2s(raw + kTileBytes, wtile_up + (size_t)kb * kTileBytes, kTileBytes,
                                 full_raw(s));
                    mbar_arrive_expect_tx(full_b(s), npad * 128);
                }
                __syncwarp();
                if (GATEUP) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int g4 = lane + 32 * q;
                        if (g4 * 4 < npad)
                            tma_gather4(bsm + g4 * 512, &bmap, kb * kTileK, rows[q * 4 + 0],
                                        rows[q * 4 + 1], rows[q * 4 + 2], rows[q * 4 + 3],
                                        full_b(s));
                    }
                } else {
                    if (lane * 16 < npad)
                        tma_load_2d(bsm + lane * 16 * 128, &bmap, kb * kTileK, n0 + lane * 16,
                                    full_b(s));
                }
                ++issued;
            }
        }
        if (!ok) {
            // let the copies already issued land before the CTA goes away
            const int first = issued > S ? issued - S : 0;
            for (int j = first; j < issued; ++j) {
                mbar_wait(full_raw(j % S), (j / S) & 1);
                mbar_wait(full_b(j % S), (j / S) & 1);
            }
        }
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------------------------- MMA
        int it = 0, item = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++item) {
            const int tile = w / rb_count;
            const int nn = args.tile_nn[tile];
            const int npad = (nn + 15) & ~15;
            const uint32_t idesc = idesc_f16_f32(128, npad);
            if (*abort_flag || !mbar_wait(acc_empty, (item & 1) ^ 1)) {
                fail();
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % S;
                const uint32_t ph = (it / S) & 1;
                if (*abort_flag || !mbar_wait(full_b(s), ph) || !mbar_wait(full_a(s), ph)) {
                    fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a_sm = base + C::OFF_A + s * C::A_BYTES;
                    const uint32_t b_sm = base + C::OFF_B + s * B_BYTES;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bdesc = sw128_kmajor_desc(b_sm + kk * 32);
#pragma unroll
                        for (int m = 0; m < C::NMAT; ++m) {
                            const uint64_t adesc =
                                sw128_kmajor_desc(a_sm + m * A_MAT_BYTES + kk * 32);
                            mma_f16(tmem + m * 256, adesc, bdesc, idesc, (kb | kk) != 0);
                        }
                    }
                    mma_commit(empty(s));
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
        const int dt = threadIdx.x - WARP_DEQ0 * 32;  // 0..255
        int it = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % S;
                const uint32_t ph = (it / S) & 1;
                if (*abort_flag || !mbar_wait(full_raw(s), ph)) {
                    fail();
                    ok = false;
                    break;
                }
                const uint8_t* raw = sbase + C::OFF_RAW + s * C::RAW_BYTES;
                uint8_t* a = sbase + C::OFF_A + s * C::A_BYTES;
#pragma unroll
                for (int q = dt; q < C::NMAT * 1024; q += NUM_DEQ_WARPS * 32) {
                    const int m = q / 1024, r = (q / 8) % 128, c = q % 8;
                    const uint8_t* t = raw + m * kTileBytes;
                    const uint32_t word = *reinterpret_cast<const uint32_t*>(t + r * 32 + c * 4);
                    const uint16_t dh =
                        *reinterpret_cast<const uint16_t*>(t + kTileCodeBytes + r * 4 + (c / 4) * 2);
                    const uint32_t d2 = (uint32_t)dh | ((uint32_t)dh << 16);
                    uint4 o;
                    o.x = f16x2_dequant(word & 0x000F000Fu, d2);
                    o.y = f16x2_dequant((word >> 4) & 0x000F000Fu, d2);
                    o.z = f16x2_dequant((word >> 8) & 0x000F000Fu, d2);
                    o.w = f16x2_dequant((word >> 12) & 0x000F000Fu, d2);
                    *reinterpret_cast<uint4*>(a + m * A_MAT_BYTES + r * 128 + ((c ^ (r & 7)) * 16)) = o;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_a(s));
            }
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int quad = warp % 4;
        const int row = quad * 32 + lane;
        int item = 0;
        for (int w = blockIdx.x; w < n_items; w += gridDim.x, ++item) {
            const int tile = w / rb_count, rb = w % rb_count;
            const int n0 = args.tile_n0[tile], nn = args.tile_nn[tile];
            if (*abort_flag || !mbar_wait(acc_full, item & 1)) {
                fail();
                break;
            }
            tc_fence_after();
            const int feat = rb * kTileRows + row;
            for (int c0 = 0; c0 < nn; c0 += 16) {
                uint32_t g[16];
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c0, g);
                if (GATEUP) {
                    uint32_t u[16];
                    tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + 256 + c0, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < nn) {
                            const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
                            const float h = gv / (1.0f + __expf(-gv)) * uv;
                            args.out[(size_t)(n0 + c0 + j) * args.out_ld + feat] =
                                float_to_half_bits_sat(h);
                        }
                    }
                } else {
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < nn) {
                            const float yv = __uint_as_float(g[j]) * args.slot_w[n0 + c0 + j];
                            args.out[(size_t)(n0 + c0 + j) * args.out_ld + feat] =
                                float_to_half_bits_sat(yv);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <bool GATEUP>
cudaError_t launch_gemm(const CUtensorMap* map, const GemmArgs& a, int num_sms, cudaStream_t s) {
    using C = Cfg<GATEUP>;
    cudaError_t err = cudaFuncSetAttribute(grouped_q4_gemm_kernel<GATEUP>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    grouped_q4_gemm_kernel<GATEUP><<<num_sms, NUM_THREADS, C::SMEM_BYTES, s>>>(*map, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_gateup(const CUtensorMap* x_map, const void* wgu, const Workspace& ws,
                                  int T, int H, int I, int E, int k, int* status, int num_sms,
                                  cudaStream_t s) {
    (void)T; (void)E; (void)k;
    GemmArgs a{};
    a.wpk = static_cast<const uint8_t*>(wgu);
    a.counters = ws.counters;
    a.tile_e = ws.tile_e;
    a.tile_n0 = ws.tile_n0;
    a.tile_nn = ws.tile_nn;
    a.bucket_token = ws.bucket_token;
    a.slot_w = ws.slot_w;
    a.out = ws.h;
    a.K = H;
    a.rows_per_e = 2 * I;
    a.out_rows = I;
    a.out_ld = I;
    a.status = status;
    return launch_gemm<true>(x_map, a, num_sms, s);
}

cudaError_t launch_prefill_down(const CUtensorMap* h_map, const void* wd, const Workspace& ws,
                                int T, int H, int I, int E, int k, int* status, int num_sms,
                                cudaStream_t s) {
    (void)T; (void)E; (void)k;
    GemmArgs a{};
    a.wpk = static_cast<const uint8_t*>(wd);
    a.counters = ws.counters;
    a.tile_e = ws.tile_e;
    a.tile_n0 = ws.tile_n0;
    a.tile_nn = ws.tile_nn;
    a.bucket_token = ws.bucket_token;
    a.slot_w = ws.slot_w;
    a.out = static_cast<uint16_t*>(ws.y);
    a.K = I;
    a.rows_per_e = H;
    a.out_rows = H;
    a.out_ld = H;
    a.status = status;
    return launch_gemm<false>(h_map, a, num_sms, s);
}

}  // namespace moeq4
