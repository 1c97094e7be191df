// moe_w4a8_forward_decode_noalloc: the W4A8 decode layer with its scratch
// memory in a fixed device array owned by this library, for callers that
// cannot allocate device memory themselves.
//
// Who needs it: code that runs inside a host application or plugin interface
// which owns the device memory and gives its components no way to allocate,
// and latency-critical decode loops that must not call cudaMalloc on their
// path (it can synchronise the device and its cost is unbounded).  Such
// callers still pass their inputs and outputs; only the scratch workspace of
// moe_w4a8_forward_decode moves into the array below.
//
// The array is a file-scope device variable, so every GPU that loads this
// library holds it (kNoAllocScratchBytes) until the process exits.  Host code
// must not pass the array's name to a kernel: on the host it is a stand-in
// symbol, not a device address.  Its device address is looked up once per
// device, with that device current, by cudaGetSymbolAddress on the first call
// made on that device; that first call should therefore come before any
// stream capture.  All calls share the one array: calls whose work overlaps
// on the GPU (different streams, or different host threads on one device)
// race on it.  The array keeps the last call's contents; nothing in it needs
// to start at zero: the decode path writes every scratch value it reads
// earlier in the same call, and its first kernel clears the counters the
// second one synchronises on, whatever shape the previous call had.
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

static_assert(MOE_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) uint8_t g_decode_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace moeq4 {
namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;

constexpr int kMaxDevicesNoAlloc = 64;
void* g_scratch_addr[kMaxDevicesNoAlloc] = {};
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device (looked up once).
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        char msg[160];
        snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
        return record_error(MOE_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevicesNoAlloc)
        return record_error(MOE_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            char msg[160];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress(decode scratch): %s",
                     cudaGetErrorString(e));
            return record_error(MOE_ERR_CUDA, msg);
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moeq4

extern "C" int moe_w4a8_forward_decode_noalloc(const uint16_t* x_bf16, const float* wr,
                                               const void* wgu_packed, const void* wd_packed,
                                               int T, int H, int I, int E, int k,
                                               unsigned flags, void* out, moe_debug* dbg,
                                               void* stream) {
    using namespace moeq4;
    const size_t need = moe_workspace_bytes(MOE_MODE_DECODE, T, H, I, E, k);
    if (need > kNoAllocScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "decode with T=%d H=%d I=%d E=%d k=%d needs %zu bytes of scratch; the static "
                 "array holds %zu",
                 T, H, I, E, k, need, kNoAllocScratchBytes);
        return record_error(MOE_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc) return rc;
    return moe_w4a8_forward_decode(x_bf16, wr, wgu_packed, wd_packed, T, H, I, E, k, flags, out,
                                   scratch, kNoAllocScratchBytes, dbg, stream);
}
