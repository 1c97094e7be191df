// Expert bucketing: histogram -> exclusive prefix scan -> stable scatter.
//
// The grouped GEMM of the page "A 35B Hybrid-Attention Mixture-of-Experts
// Model on a 6GB 2011 GPU" (Methodology 1, prefill) needs each expert's tokens
// side by side.  Bucket e lists the (token, slot) pairs that chose e in
// ascending token order; buckets follow each other in expert order.  The
// result is deterministic: no atomics decide an order.
//
//   1. count:   per chunk of 32 consecutive tokens, a per-expert bitmask of
//               the tokens that chose it gives, by popcount, the chunk's
//               count per expert and each pair's rank inside the chunk.  The
//               router's top-k kernel does this (route.cu, one CTA per
//               chunk), so the bucketing starts from its chunk counts.
//   2. scan:    per expert, an exclusive scan over chunks (chunk bases; four
//               threads per expert, each over a quarter of the chunks), then
//               one over experts (offsets); the same pass lists the token
//               tiles of the grouped GEMM and the non-empty experts.
//   3. scatter: row = offsets[e] + chunk base + rank.
#include "common.cuh"
#include "internal.h"

namespace moeq4 {

int nchunks(int T) { return (T + 31) / 32; }

namespace {

// Exclusive prefix sum over a 1024-thread block (thread order).
__device__ __forceinline__ int block1024_exclusive_scan(int v, int* total) {
    __shared__ int warp_tot[32];
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int wv = lane < 32 ? warp_tot[lane] : 0;
    int wincl = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o) wincl += n;
    }
    const int base = __shfl_sync(0xffffffffu, wincl - wv, warp);  // warps before this one
    const int all = __shfl_sync(0xffffffffu, wincl, 31);
    __syncthreads();
    *total = all;
    return base + incl - v;
}

constexpr int kScanParts = 4;  // threads per expert in the chunk scan

__global__ void __launch_bounds__(1024) bucket_scan_kernel(int32_t* __restrict__ chunk_count,
                                                           int nchunk, int E, int tile_n,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ touched,
                                                           int32_t* __restrict__ counters,
                                                           int32_t* __restrict__ tile_e,
                                                           int32_t* __restrict__ tile_n0,
                                                           int32_t* __restrict__ tile_nn,
                                                           int32_t* __restrict__ tile_done,
                                                           int max_tiles) {
    __shared__ int part_tot[kScanParts][kMaxExperts];
    pdl_wait();  // the chunk counts of the top-k kernel
    pdl_trigger();
    // the expert GEMMs count finished gate/up items per token tile from zero
    // (the previous call's GEMMs completed before the top-k kernel did)
    for (int i = threadIdx.x; i < max_tiles; i += blockDim.x) tile_done[i] = 0;
    const int e = threadIdx.x % kMaxExperts, part = threadIdx.x / kMaxExperts;
    const int c0 = part * nchunk / kScanParts, c1 = (part + 1) * nchunk / kScanParts;
    // this quarter's total, 16 chunk counts in flight at a time
    int tot = 0;
    if (e < E) {
        for (int c = c0; c < c1; c += 16) {
            int n[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) n[u] = (c + u < c1) ? chunk_count[(size_t)(c + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 16; ++u) tot += n[u];
        }
        part_tot[part][e] = tot;
    }
    __syncthreads();
    // each count becomes its chunk's base: the expert's tokens in earlier chunks
    int count = 0;
    if (e < E) {
        int run = 0;
        for (int p = 0; p < kScanParts; ++p) {
            if (p < part) run += part_tot[p][e];
            count += part_tot[p][e];
        }
        for (int c = c0; c < c1; c += 16) {
            int n[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) n[u] = (c + u < c1) ? chunk_count[(size_t)(c + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (c + u < c1) chunk_count[(size_t)(c + u) * E + e] = run;
                run += n[u];
            }
        }
    }
    // experts in order (threads of part 0 carry them; the others add 0)
    const bool lead = part == 0 && e < E;
    int total;
    const int off = block1024_exclusive_scan(lead ? count : 0, &total);
    if (lead) offsets[e] = off;
    if (threadIdx.x == 0) offsets[E] = total;
    const int ntiles = lead ? (count + tile_n - 1) / tile_n : 0;
    int all_tiles;
    const int toff = block1024_exclusive_scan(ntiles, &all_tiles);
    // a bucket is cut into ntiles tiles of near-equal size (the first
    // count % ntiles tiles one row longer), each at most tile_n rows
    const int tbase = ntiles ? count / ntiles : 0, textra = ntiles ? count % ntiles : 0;
    for (int i = 0, r0 = 0; i < ntiles; ++i) {
        const int nn = tbase + (i < textra ? 1 : 0);
        tile_e[toff + i] = e;
        tile_n0[toff + i] = off + r0;
        tile_nn[toff + i] = nn;
        r0 += nn;
    }
    int ntouched;
    const int pos = block1024_exclusive_scan(lead && count > 0 ? 1 : 0, &ntouched);
    if (lead && count > 0) touched[pos] = e;
    if (threadIdx.x == 0) {
        counters[kCntTouched] = ntouched;
        counters[kCntTiles] = all_tiles;
    }
}

__global__ void bucket_scatter_kernel(const int32_t* __restrict__ idx,
                                      const float* __restrict__ w, int T, int E, int k,
                                      const int32_t* __restrict__ chunk_base,
                                      const int32_t* __restrict__ entry_rank,
                                      const int32_t* __restrict__ offsets,
                                      int32_t* __restrict__ bucket_token,
                                      int32_t* __restrict__ bucket_slot,
                                      float* __restrict__ slot_w, int32_t* __restrict__ slot_pos) {
    pdl_wait();  // the chunk bases and offsets of the scan
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T * k) return;
    const int t = i / k, j = i % k;
    const int e = idx[i];
    const int pos = offsets[e] + chunk_base[(size_t)(t / 32) * E + e] + entry_rank[i];
    bucket_token[pos] = t;
    bucket_slot[pos] = j;
    slot_w[pos] = w[i];
    slot_pos[i] = pos;
}

}  // namespace

cudaError_t launch_bucket(const int32_t* idx, const float* w, int T, int E, int k, int tile_n,
                          const Workspace& ws, cudaStream_t s) {
    const int nc = nchunks(T);
    cudaError_t err = launch_pdl(bucket_scan_kernel, dim3(1), dim3(1024), 0, s, ws.chunk_count, nc,
                                 E, tile_n, ws.offsets, ws.touched, ws.counters, ws.tile_e,
                                 ws.tile_n0, ws.tile_nn, ws.tile_done, ws.max_tiles);
    if (err != cudaSuccess) return err;
    if (T > 0)
        err = launch_pdl(bucket_scatter_kernel, dim3((T * k + 255) / 256), dim3(256), 0, s, idx, w,
                         T, E, k, (const int32_t*)ws.chunk_count, (const int32_t*)ws.entry_rank,
                         (const int32_t*)ws.offsets, ws.bucket_token, ws.bucket_slot, ws.slot_w,
                         ws.slot_pos);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moeq4
