// moe_q4_pack: canonical Q4_0-family weights -> the packed tile layout.
//
// Q4_0 family (page "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB
// 2011 GPU", Methodology 2 "Quantization": group-wise symmetric 4-bit
// weights): 32 consecutive codes of a row share one fp16 scale, w = d(q - 8).
// The packed layout (include/moeq4.h) keeps exactly that information and
// only reorders it: 128 x 64 tiles, 4608 bytes each, one bulk copy per tile.
#include "common.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

// Reads code `i` (0..K-1) of row `row` from either source format.
struct CodeSource {
    int fmt;
    const uint8_t* src;
    int K;
    __device__ __forceinline__ void load8(size_t row, int k0, uint32_t (&c)[8]) const {
        if (fmt == 0) {
            const uint8_t* p = src + row * (size_t)K + k0;
            const uint2 v = *reinterpret_cast<const uint2*>(p);
#pragma unroll
            for (int i = 0; i < 4; ++i) c[i] = (v.x >> (8 * i)) & 0xFu;
#pragma unroll
            for (int i = 0; i < 4; ++i) c[4 + i] = (v.y >> (8 * i)) & 0xFu;
        } else {
            // 18-byte block: 2 scale bytes, then byte j = element j (low
            // nibble) | element j+16 (high nibble)
            const uint8_t* blk = src + (row * (size_t)(K / kGroup) + k0 / kGroup) * 18;
            const int e0 = k0 % kGroup;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + i;
                const uint8_t b = blk[2 + (e & 15)];
                c[i] = (e < 16) ? (b & 0xFu) : (b >> 4);
            }
        }
    }
    __device__ __forceinline__ uint16_t scale(const uint16_t* scales, size_t row, int g) const {
        if (fmt == 0) return scales[row * (size_t)(K / kGroup) + g];
        const uint8_t* blk = src + (row * (size_t)(K / kGroup) + g) * 18;
        return (uint16_t)(blk[0] | (blk[1] << 8));
    }
};

// One thread per 32-bit word of packed codes (8 codes).
__global__ void pack_codes_kernel(CodeSource cs, int E, int N, int K, uint8_t* dst) {
    const int words_per_row = K / 8;
    const size_t total = (size_t)E * N * words_per_row;
    const int kb_per_row = K / kTileK;
    const int rb_per_e = N / kTileRows;
    for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < total;
         w += (size_t)gridDim.x * blockDim.x) {
        const size_t row = w / words_per_row;  // e * N + n
        const int c = (int)(w % words_per_row);
        const int e = (int)(row / N), n = (int)(row % N);
        uint32_t q[8];
        cs.load8(row, c * 8, q);
        // even columns -> nibbles 0..3, odd columns -> nibbles 4..7
        const uint32_t word = q[0] | (q[2] << 4) | (q[4] << 8) | (q[6] << 12) | (q[1] << 16) |
                              (q[3] << 20) | (q[5] << 24) | (q[7] << 28);
        const size_t tile = ((size_t)e * rb_per_e + n / kTileRows) * kb_per_row + c / 8;
        uint32_t* t = reinterpret_cast<uint32_t*>(dst + tile * kTileBytes);
        t[(n % kTileRows) * 8 + (c % 8)] = word;
    }
}

// One thread per (row, 64-column block): its two fp16 scales.
__global__ void pack_scales_kernel(CodeSource cs, const uint16_t* scales, int E, int N, int K,
                                   uint8_t* dst) {
    const int kb_per_row = K / kTileK;
    const int rb_per_e = N / kTileRows;
    const size_t total = (size_t)E * N * kb_per_row;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / kb_per_row;
        const int kb = (int)(i % kb_per_row);
        const int e = (int)(row / N), n = (int)(row % N);
        const size_t tile = ((size_t)e * rb_per_e + n / kTileRows) * kb_per_row + kb;
        uint16_t* t = reinterpret_cast<uint16_t*>(dst + tile * kTileBytes + kTileCodeBytes);
        t[(n % kTileRows) * 2 + 0] = cs.scale(scales, row, 2 * kb);
        t[(n % kTileRows) * 2 + 1] = cs.scale(scales, row, 2 * kb + 1);
    }
}

// 8-bit tiles: one thread per 8 codes of a row.  Row r's 64 codes take bytes
// r*64 .. r*64 + 63 of the tile; each 8-code chunk is stored in the order the
// int8 activations are (columns 0, 4, 1, 5, 2, 6, 3, 7), so that two dp4a
// of its two words with the activation chunk's two words give its dot.
__global__ void pack8_codes_kernel(const int8_t* src, int E, int N, int K, uint8_t* dst) {
    const int chunks_per_row = K / 8;
    const size_t total = (size_t)E * N * chunks_per_row;
    const int kb_per_row = K / kTileK;
    const int rb_per_e = N / kTileRows;
    for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < total;
         w += (size_t)gridDim.x * blockDim.x) {
        const size_t row = w / chunks_per_row;
        const int c = (int)(w % chunks_per_row);
        const int e = (int)(row / N), n = (int)(row % N);
        const uint2 v = *reinterpret_cast<const uint2*>(src + row * (size_t)K + c * 8);
        const uint2 o = make_uint2(__byte_perm(v.x, v.y, 0x5140), __byte_perm(v.x, v.y, 0x7362));
        const size_t tile = ((size_t)e * rb_per_e + n / kTileRows) * kb_per_row + c / 8;
        *reinterpret_cast<uint2*>(dst + tile * kTileBytes8 + (n % kTileRows) * 64 + (c % 8) * 8) = o;
    }
}

__global__ void pack8_scales_kernel(const uint16_t* scales, int E, int N, int K, uint8_t* dst) {
    const int kb_per_row = K / kTileK;
    const int rb_per_e = N / kTileRows;
    const size_t total = (size_t)E * N * kb_per_row;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / kb_per_row;
        const int kb = (int)(i % kb_per_row);
        const int e = (int)(row / N), n = (int)(row % N);
        const size_t tile = ((size_t)e * rb_per_e + n / kTileRows) * kb_per_row + kb;
        uint16_t* t = reinterpret_cast<uint16_t*>(dst + tile * kTileBytes8 + kTileCodeBytes8);
        t[(n % kTileRows) * 2 + 0] = scales[row * (size_t)(K / kGroup) + 2 * kb];
        t[(n % kTileRows) * 2 + 1] = scales[row * (size_t)(K / kGroup) + 2 * kb + 1];
    }
}

}  // namespace

cudaError_t launch_pack8(const void* codes, const void* scales, int E, int N, int K, void* dst,
                         cudaStream_t s) {
    pack8_codes_kernel<<<1184, 256, 0, s>>>(static_cast<const int8_t*>(codes), E, N, K,
                                            static_cast<uint8_t*>(dst));
    pack8_scales_kernel<<<592, 256, 0, s>>>(static_cast<const uint16_t*>(scales), E, N, K,
                                            static_cast<uint8_t*>(dst));
    return cudaGetLastError();
}

cudaError_t launch_pack(int fmt, const void* src, const void* src_scales, int E, int N, int K,
                        void* dst, cudaStream_t s) {
    CodeSource cs{fmt, static_cast<const uint8_t*>(src), K};
    const int threads = 256;
    pack_codes_kernel<<<1184, threads, 0, s>>>(cs, E, N, K, static_cast<uint8_t*>(dst));
    pack_scales_kernel<<<592, threads, 0, s>>>(cs, static_cast<const uint16_t*>(src_scales), E, N,
                                               K, static_cast<uint8_t*>(dst));
    return cudaGetLastError();
}

}  // namespace moeq4
