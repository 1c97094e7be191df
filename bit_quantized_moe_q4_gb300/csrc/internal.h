// Host-side declarations shared by the moeq4 translation units (not part of
// the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moeq4.h"

#include <utility>

namespace moeq4 {

// Workspace pieces of one forward call; every pointer is a device address
// carved out of the caller's workspace (see api.cu).
struct Workspace {
    float* logits;          // [T, E]
    int32_t* topk_idx;      // [T, k]
    float* topk_w;          // [T, k]
    int32_t* chunk_count;   // [nchunk, E]   bucket counts per 32-token chunk
    int32_t* entry_rank;    // [T*k]         rank inside the chunk
    int32_t* offsets;       // [E+1]
    int32_t* touched;       // [E]           experts with a non-empty bucket
    int32_t* counters;      // [8]           n_touched, n_tiles, n_items, ...
    int32_t* bucket_token;  // [T*k]
    int32_t* bucket_slot;   // [T*k]
    float* slot_w;          // [T*k]         routing weight of each bucket row
    int32_t* slot_pos;      // [T*k]         bucket row of (t, j)
    int32_t* tile_e;        // [max_tiles]   expert of each token tile
    int32_t* tile_n0;       // [max_tiles]   first bucket row of the tile
    int32_t* tile_nn;       // [max_tiles]   rows in the tile
    uint16_t* xn;           // [T, H] bf16 RMSNorm(x) (stacked pre-norm layers)
    uint16_t* x16;          // [T, H] fp16 copy of x (prefill GEMM operand)
    float* route_parts;     // [ksplit, T, E] router K-slice sums (prefill)
    uint16_t* wr_planes;    // [3, E, H] bf16 parts of W_r (prefill, tensor-core router)
    uint16_t* h;            // [T*k, I] fp16 (prefill)
    int32_t* tile_done;     // [max_tiles] (prefill) gate/up epilogue warps done per token tile
    void* y;                // [T*k, H] (prefill) fp16 weighted expert outputs, bucket order
    // decode
    uint8_t* xq;            // [T, H]        int8 codes of x, dp4a order; xs follows directly
    int2* xs;               // [T, H/32]     {fp32 bits of the scale, -8 * sum of the codes}
    int8_t* q_x;            // [T, H]        codes of x, column order (stage output)
    uint16_t* d_x;          // [T, H/32]     fp16 scales of x (stage output)
    float* gu_part;         // [nsg, T*k, 2I] K parts of the gate/up row sums, bucket order
    int8_t* q_h;            // [T*k, I]      (stage output)
    uint16_t* d_h;          // [T*k, I/32]
    float* y_part;          // [nsd, T*k, H] K parts of the weighted expert outputs (task kernel)
    float* y_unit;          // [I/128, T*k, H] h-block parts (clustered kernel; shares memory
                            // with gu_part and y_part)
    int32_t* sync;          // counters of the layer kernel, cleared by its prep kernel
    uint16_t* xbuf0;        // [T, H] decode stack: layer outputs inside the stack (ping-pong)
    uint16_t* xbuf1;
    int cap_g, cap_d;       // bounds of the K splits (part buffers hold that many)
    int max_tiles;
    int tile_n;             // tokens per GEMM tile (prefill)
};

// Launches kernel<<<grid, block, smem, s>>>(args...) with programmatic
// dependent launch allowed: the grid may be scheduled before the preceding
// kernel on s has finished; the kernel orders itself after it with
// griddepcontrol.wait before touching that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[1];
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// counters[] slots
enum { kCntTouched = 0, kCntTiles = 1 };


// Records a stage event on s (as an external graph node while s is capturing).
cudaError_t record_stage(void* event, cudaStream_t s, bool capturing);

int nchunks(int T);

// Sets the thread's error string (moe_last_error_string) and returns code.
int record_error(int code, const char* msg);

// launchers; each returns cudaGetLastError() of its launch
// 8-bit codes int8 [E, N, K] and fp16 scales [E, N, K/32] -> 8-bit tiles.
cudaError_t launch_pack8(const void* codes, const void* scales, int E, int N, int K, void* dst,
                         cudaStream_t s);
cudaError_t launch_pack(int fmt, const void* src, const void* src_scales, int E, int N, int K,
                        void* dst, cudaStream_t s);
cudaError_t launch_quantize(int src_type, const void* src, long long rows, int K, int fmt,
                            void* dst, void* dst_scales, cudaStream_t s);
cudaError_t launch_route(const uint16_t* x, const float* wr, int T, int H, int E, int k,
                         float* logits, int32_t* idx, float* w, uint16_t* x16, cudaStream_t s);
// Router as a K-sliced fp32 GEMM into `parts` (route_parts_floats floats; H %
// 16 == 0), then top-k; optionally writes the logits and the fp16 copy of x.
// With `planes` (route_planes_bytes bytes; non-zero for prefill token
// counts the tensor-core router takes) the product runs on the tensor cores.
int route_ksplit(int T, int H, int E);
size_t route_parts_floats(int T, int H, int E);
size_t route_planes_bytes(int T, int H, int E);
// With `chunk_count` and `entry_rank` (the bucketing's per-32-token-chunk
// arrays) the top-k kernel also counts the chunks, the first pass of the
// bucketing that launch_bucket completes.
cudaError_t launch_route_gemm(const uint16_t* x, const float* wr, int T, int H, int E, int k,
                              float* parts, float* logits, int32_t* idx, float* w, uint16_t* x16,
                              uint16_t* planes, int* status, int32_t* chunk_count,
                              int32_t* entry_rank, cudaStream_t s);
// Bucketing from the chunk counts and ranks the router's top-k kernel left in
// ws (chunk bases, offsets, tile list, touched list, then the scatter).
cudaError_t launch_bucket(const int32_t* idx, const float* w, int T, int E, int k, int tile_n,
                          const Workspace& ws, cudaStream_t s);
// Both expert GEMMs of the prefill layer in one launch: gate/up + SwiGLU -> h,
// then down x routing weight -> y (bucket order).
cudaError_t launch_prefill_experts(const void* wgu, const void* wd, const Workspace& ws, int H,
                                   int I, int* status, int num_sms, cudaStream_t s);
// The whole W4A8 decode layer: a prep kernel (counters cleared, optional
// pre-norm, router logits, int8 codes of x) and a cooperative layer kernel
// (top-k and buckets in every CTA, gate/up, h, down, combine).  `events` is
// null or the caller's MOE_NUM_STAGE_EVENTS events; boundary 1 is recorded
// after the prep kernel and 2..6 after the layer kernel.
cudaError_t launch_decode(const uint16_t* x, const float* wr, const void* wgu, const void* wd,
                          int T, int H, int I, int E, int k, bool prenorm, bool out_fp32,
                          void* out, const Workspace& ws, int32_t* dots_gu, int32_t* dots_d,
                          bool write_qh, int* status, int num_sms, void** events, bool capturing,
                          cudaStream_t s, int wbits = 4);
// L chained decode layers: per layer the prep and layer kernels, linked by
// programmatic dependent launch; layer l + 1 reads layer l's bf16 output.
cudaError_t launch_decode_stack(const uint16_t* x, int L, const float* const* wr,
                                const void* const* wgu, const void* const* wd, int T, int H, int I,
                                int E, int k, bool prenorm, bool out_fp32, void* out,
                                const Workspace& ws, int* status, int num_sms, cudaStream_t s);
// Once per device, outside any stream capture: decides whether a cooperative
// launch may also carry the programmatic-dependent-launch attribute.
cudaError_t decode_prepare_device(int dev);
// 1: cooperative launches may carry the PDL attribute; 2: they may not.
int cooperative_pdl_mode(int dev);
// Whether the decode layer kernel's on-chip staging fits this shape.
bool decode_shape_fits(int T, int H, int I, int E);
// Bounds of the decode K splits for a shape: the caps (part-buffer budget)
// and the largest split any routing can pick (the part buffers' size).
void decode_split_bounds(int T, int H, int I, int E, int k, int* cap_g, int* cap_d, int* nsg_max,
                         int* nsd_max);
// Counters the decode prep kernel clears.
int decode_sync_ints(int T, int H, int I, int E, int k);
// Whether the clustered decode kernel takes this shape with 8-bit weights.
bool decode_w8_fits(int T, int H, int I, int E);
// Parts of the weighted expert outputs the clustered decode kernel stores
// (I/128 planes of [T*k, H]), or 0 when the shape never takes that kernel.
int decode_cluster_parts(int T, int H, int I, int E);
// xn[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps)), one warp per token.
cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps, uint16_t* xn,
                           cudaStream_t s);
cudaError_t launch_combine(const uint16_t* x, const void* y, bool y_fp32, const int32_t* slot_pos,
                           int T, int H, int k, bool out_fp32, void* out, cudaStream_t s);

// tensor maps
// 2-D map over a row-major [rows, cols] tensor of 16-bit elements (fp16).
bool encode_tmap_2d_f16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_cols, uint32_t box_rows, bool swizzle128);
// 2-D map over packed Q4 weights seen as [ntiles, 1152] 32-bit words (one row
// per 4608-byte tile); box of box_words x box_tiles.
bool encode_tmap_packed(CUtensorMap* map, const void* packed, uint64_t ntiles, uint32_t box_words,
                        uint32_t box_tiles);

}  // namespace moeq4
