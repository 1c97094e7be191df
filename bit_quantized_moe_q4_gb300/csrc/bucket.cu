// Expert bucketing: histogram -> exclusive prefix scan -> stable scatter.
//
// The grouped GEMM of the page "A 35B Hybrid-Attention Mixture-of-Experts
// Model on a 6GB 2011 GPU" (Methodology 1, prefill) needs each expert's tokens
// side by side.  Bucket e lists the (token, slot) pairs that chose e in
// ascending token order; buckets follow each other in expert order.  The
// result is deterministic: no atomics decide an order.
//
//   1. count:   each warp takes 32 consecutive tokens; a per-expert bitmask of
//               the lanes that chose it gives, by popcount, the chunk's count
//               per expert and each pair's rank inside the chunk.
//   2. scan:    per expert, an exclusive scan over chunks (chunk bases), then
//               one over experts (offsets); the same pass lists the token
//               tiles of the grouped GEMM and the non-empty experts.
//   3. scatter: row = offsets[e] + chunk base + rank.
#include "common.cuh"
#include "internal.h"

namespace moeq4 {

int nchunks(int T) { return (T + 31) / 32; }

namespace {

__global__ void __launch_bounds__(256) bucket_count_kernel(const int32_t* __restrict__ idx, int T,
                                                           int E, int k,
                                                           int32_t* __restrict__ chunk_count,
                                                           int32_t* __restrict__ entry_rank) {
    __shared__ uint32_t bits[8][kMaxExperts];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int chunk = blockIdx.x * 8 + warp;
    if (chunk * 32 >= T) return;  // whole warp leaves together
    for (int e = lane; e < E; e += 32) bits[warp][e] = 0u;
    __syncwarp();
    const int t = chunk * 32 + lane;
    const bool valid = t < T;
    if (valid)
        for (int j = 0; j < k; ++j) atomicOr(&bits[warp][idx[(size_t)t * k + j]], 1u << lane);
    __syncwarp();
    if (valid) {
        const uint32_t below = (1u << lane) - 1u;
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            entry_rank[(size_t)t * k + j] = __popc(bits[warp][e] & below);
        }
    }
    for (int e = lane; e < E; e += 32) chunk_count[(size_t)chunk * E + e] = __popc(bits[warp][e]);
}

__global__ void __launch_bounds__(256) bucket_scan_kernel(int32_t* __restrict__ chunk_count,
                                                          int nchunk, int E, int tile_n,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ touched,
                                                          int32_t* __restrict__ counters,
                                                          int32_t* __restrict__ tile_e,
                                                          int32_t* __restrict__ tile_n0,
                                                          int32_t* __restrict__ tile_nn) {
    const int e = threadIdx.x;
    int count = 0;
    if (e < E) {
        // 16 chunk counts in flight at a time; each becomes its chunk's base
        for (int c0 = 0; c0 < nchunk; c0 += 16) {
            int n[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                n[u] = (c0 + u < nchunk) ? chunk_count[(size_t)(c0 + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (c0 + u < nchunk) chunk_count[(size_t)(c0 + u) * E + e] = count;
                count += n[u];
            }
        }
    }
    int total;
    const int off = block256_exclusive_scan(count, &total);
    if (e < E) offsets[e] = off;
    if (e == 0) offsets[E] = total;
    const int ntiles = (count + tile_n - 1) / tile_n;
    int all_tiles;
    const int toff = block256_exclusive_scan(ntiles, &all_tiles);
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
    const int pos = block256_exclusive_scan(count > 0 ? 1 : 0, &ntouched);
    if (count > 0) touched[pos] = e;
    if (e == 0) {
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
    if (T > 0)
        bucket_count_kernel<<<(nc + 7) / 8, 256, 0, s>>>(idx, T, E, k, ws.chunk_count,
                                                         ws.entry_rank);
    bucket_scan_kernel<<<1, 256, 0, s>>>(ws.chunk_count, nc, E, tile_n, ws.offsets, ws.touched,
                                         ws.counters, ws.tile_e, ws.tile_n0, ws.tile_nn);
    if (T > 0)
        bucket_scatter_kernel<<<(T * k + 255) / 256, 256, 0, s>>>(
            idx, w, T, E, k, ws.chunk_count, ws.entry_rank, ws.offsets, ws.bucket_token,
            ws.bucket_slot, ws.slot_w, ws.slot_pos);
    return cudaGetLastError();
}

}  // namespace moeq4
