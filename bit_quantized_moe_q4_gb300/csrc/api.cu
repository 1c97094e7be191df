// C ABI of moeq4 (include/moeq4.h): argument checks, workspace carve-up,
// tensor-map set-up and the launch sequence of each forward path.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include <algorithm>

#include "internal.h"

namespace moeq4 {
namespace {

thread_local char g_err[512] = "";

int set_err(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

// Per-device status word written by kernels whose bounded wait ran out.
__device__ int g_device_status = 0;

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    int* status = nullptr;  // device address of g_device_status
    // the streamed prefill stack: its copy stream and events (created on
    // first use)
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_copied[2] = {nullptr, nullptr}, ev_done[2] = {nullptr, nullptr};
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Looks up (once per device, with that device current) the SM count, the
// architecture and the address of the status word.
int device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return set_err(MOE_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(cudaGetLastError()));
    if (dev < 0 || dev >= kMaxDevices) return set_err(MOE_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        d.supported = (major == 10 && minor == 3);
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess)
            return set_err(MOE_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
        d.status = static_cast<int*>(p);
        if (d.supported) {
            e = decode_prepare_device(dev);
            if (e != cudaSuccess)
                return set_err(MOE_ERR_CUDA, "decode set-up: %s", cudaGetErrorString(e));
        }
        d.ready = true;
        if (!d.supported)
            return set_err(MOE_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                           dev, major, minor);
    }
    if (!d.supported) return set_err(MOE_ERR_UNSUPPORTED, "device %d is not sm_103a", dev);
    *out = &d;
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_check(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return set_err(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return MOE_OK;
}

// ---- tensor maps (driver entry point fetched through the runtime) --------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

namespace {
EncodeTiledFn encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}
}  // namespace

bool encode_tmap_2d_f16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tmap_packed(CUtensorMap* map, const void* packed, uint64_t ntiles, uint32_t box_words,
                        uint32_t box_tiles) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(kTileBytes / 4), ntiles};
    const cuuint64_t strides[1] = {(cuuint64_t)kTileBytes};
    const cuuint32_t box[2] = {box_words, box_tiles};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(packed), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

constexpr int kPrefillTileN = 160;  // tokens per prefill GEMM tile (the GEMM's BN)

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Lays the workspace out; with base == nullptr only the size is computed.
size_t carve(int mode, int T, int H, int I, int E, int k, uint8_t* base, Workspace* ws) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> uint8_t* {
        uint8_t* p = base ? base + off : nullptr;
        off += align256(bytes ? bytes : 1);
        return p;
    };
    const size_t Tk = (size_t)T * k;
    const int nc = nchunks(T);
    const int tile_n = (mode == MOE_MODE_PREFILL) ? kPrefillTileN : 32;
    const int max_tiles = (int)((Tk + tile_n - 1) / tile_n) + E;
    Workspace w{};
    w.logits = reinterpret_cast<float*>(take((size_t)T * E * 4));
    w.topk_idx = reinterpret_cast<int32_t*>(take(Tk * 4));
    w.topk_w = reinterpret_cast<float*>(take(Tk * 4));
    w.chunk_count = reinterpret_cast<int32_t*>(take((size_t)nc * E * 4));
    w.entry_rank = reinterpret_cast<int32_t*>(take(Tk * 4));
    w.offsets = reinterpret_cast<int32_t*>(take((size_t)(E + 1) * 4));
    w.touched = reinterpret_cast<int32_t*>(take((size_t)E * 4));
    w.counters = reinterpret_cast<int32_t*>(take(8 * 4));
    w.bucket_token = reinterpret_cast<int32_t*>(take(Tk * 4));
    w.bucket_slot = reinterpret_cast<int32_t*>(take(Tk * 4));
    w.slot_w = reinterpret_cast<float*>(take(Tk * 4));
    w.slot_pos = reinterpret_cast<int32_t*>(take(Tk * 4));
    w.tile_e = reinterpret_cast<int32_t*>(take((size_t)max_tiles * 4));
    w.tile_n0 = reinterpret_cast<int32_t*>(take((size_t)max_tiles * 4));
    w.tile_nn = reinterpret_cast<int32_t*>(take((size_t)max_tiles * 4));
    if (mode == MOE_MODE_PREFILL) {
        w.xn = reinterpret_cast<uint16_t*>(take((size_t)T * H * 2));
        w.y = take(Tk * H * 2);
        w.x16 = reinterpret_cast<uint16_t*>(take((size_t)T * H * 2));
        w.route_parts = reinterpret_cast<float*>(take(route_parts_floats(T, H, E) * 4));
        w.wr_planes = reinterpret_cast<uint16_t*>(take(route_planes_bytes(T, H, E)));
        w.h = reinterpret_cast<uint16_t*>(take(Tk * I * 2));
        w.tile_done = reinterpret_cast<int32_t*>(take((size_t)max_tiles * 4));
    } else {
        int nsg = 1, nsd = 1;
        decode_split_bounds(T, H, I, E, k, &w.cap_g, &w.cap_d, &nsg, &nsd);
        // the codes of x and their scales back to back (one contiguous copy)
        const size_t xq_bytes = (size_t)T * H;
        w.xq = take(xq_bytes + (size_t)T * (H / kGroup) * 8);
        w.xs = base ? reinterpret_cast<int2*>(w.xq + xq_bytes) : nullptr;
        w.q_x = reinterpret_cast<int8_t*>(take((size_t)T * H));
        w.d_x = reinterpret_cast<uint16_t*>(take((size_t)T * (H / kGroup) * 2));
        // one region for the parts: the task kernel's gate/up K parts and
        // down K parts, or the clustered kernel's per-h-block parts
        const size_t gu_bytes = (size_t)nsg * Tk * 2 * I * 4, yd_bytes = (size_t)nsd * Tk * H * 4;
        const size_t yc_bytes = (size_t)decode_cluster_parts(T, H, I, E) * Tk * H * 4;
        uint8_t* parts = take(std::max(gu_bytes + yd_bytes, yc_bytes));
        w.gu_part = reinterpret_cast<float*>(parts);
        w.y_part = base ? reinterpret_cast<float*>(parts + gu_bytes) : nullptr;
        w.y_unit = reinterpret_cast<float*>(parts);
        w.q_h = reinterpret_cast<int8_t*>(take(Tk * I));
        w.d_h = reinterpret_cast<uint16_t*>(take(Tk * (I / kGroup) * 2));
        w.sync = reinterpret_cast<int32_t*>(take((size_t)decode_sync_ints(T, H, I, E, k) * 4));
        w.xbuf0 = reinterpret_cast<uint16_t*>(take((size_t)T * H * 2));
        w.xbuf1 = reinterpret_cast<uint16_t*>(take((size_t)T * H * 2));
    }
    w.max_tiles = max_tiles;
    w.tile_n = tile_n;
    if (ws) *ws = w;
    return off;
}

int check_layer_shape(int mode, int T, int H, int I, int E, int k) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0)
        return set_err(MOE_ERR_SHAPE, "non-positive dimension (T=%d H=%d I=%d E=%d k=%d)", T, H, I,
                       E, k);
    if (E > MOE_MAX_EXPERTS) return set_err(MOE_ERR_SHAPE, "E=%d exceeds %d", E, MOE_MAX_EXPERTS);
    if (k > E || k > MOE_MAX_TOPK)
        return set_err(MOE_ERR_SHAPE, "k=%d must satisfy 1 <= k <= min(E, %d)", k, MOE_MAX_TOPK);
    if (H % 128 || I % 128)
        return set_err(MOE_ERR_SHAPE, "H=%d and I=%d must be multiples of 128", H, I);
    const long long big = (long long)T * k * (H > I ? H : I);
    if (big >= (1ll << 31)) return set_err(MOE_ERR_SHAPE, "T*k*max(H,I) = %lld too large", big);
    if (mode == MOE_MODE_DECODE && T > MOE_DECODE_MAX_T)
        return set_err(MOE_ERR_SHAPE, "decode takes at most %d tokens (T=%d)", MOE_DECODE_MAX_T, T);
    if (mode == MOE_MODE_DECODE && T > 0 && !decode_shape_fits(T, H, I, E))
        return set_err(MOE_ERR_SHAPE,
                       "decode with T=%d H=%d I=%d E=%d does not fit the on-chip staging "
                       "(T*(H+I) or T*E too large)", T, H, I, E);
    return MOE_OK;
}

int copy_d2d(void* dst, const void* src, size_t bytes, cudaStream_t s) {
    if (!dst || bytes == 0) return MOE_OK;
    return cuda_check(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s),
                      "debug copy");
}

int forward(int mode, const uint16_t* x, const float* wr, const void* wgu, const void* wd, int T,
            int H, int I, int E, int k, unsigned flags, void* out, void* workspace,
            size_t ws_bytes, moe_debug* dbg, void* stream, int wbits = 4) {
    int rc = check_layer_shape(mode, T, H, I, E, k);
    if (rc) return rc;
    if (wbits == 8 && T > 0 && !decode_w8_fits(T, H, I, E))
        return set_err(MOE_ERR_SHAPE,
                       "8-bit decode takes at most %d tokens and must fit the on-chip staging "
                       "(T=%d H=%d I=%d E=%d)", MOE_W8_DECODE_MAX_T, T, H, I, E);
    if (flags & ~(MOE_OUT_FP32 | MOE_STACKED_PRENORM))
        return set_err(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    if (T == 0) return MOE_OK;
    if (!x || !wr || !wgu || !wd || !out)
        return set_err(MOE_ERR_INVALID_ARG, "null tensor argument");
    if (!aligned16(x) || !aligned16(wr) || !aligned16(wgu) || !aligned16(wd) || !aligned16(out) ||
        !aligned16(workspace))
        return set_err(MOE_ERR_ALIGN, "tensor arguments must be 16-byte aligned");
    if (out == static_cast<const void*>(x)) return set_err(MOE_ERR_INVALID_ARG, "out may not alias x");
    const size_t need = carve(mode, T, H, I, E, k, nullptr, nullptr);
    if (!workspace || ws_bytes < need)
        return set_err(MOE_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Workspace ws{};
    carve(mode, T, H, I, E, k, static_cast<uint8_t*>(workspace), &ws);
    const size_t Tk = (size_t)T * k;

    void** ev = dbg ? dbg->stage_events : nullptr;
    bool capturing = false;
    if (ev) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if ((rc = cuda_check(cudaStreamIsCapturing(s, &cs), "capture status"))) return rc;
        capturing = cs == cudaStreamCaptureStatusActive;
    }
    // Inside a stream capture the events become external event-record nodes of
    // the graph; otherwise they are plain records.
    auto mark = [&](int i) -> int {
        if (!ev || !ev[i]) return MOE_OK;
        return cuda_check(record_stage(ev[i], s, capturing), "stage event");
    };
    if ((rc = mark(0))) return rc;
    if (mode == MOE_MODE_DECODE) {
        // prep (counters, optional pre-norm, logits, x codes), then the layer
        // kernel (top-k, buckets, gate/up, h, down, combine)
        if ((rc = cuda_check(launch_decode(x, wr, wgu, wd, T, H, I, E, k,
                                           (flags & MOE_STACKED_PRENORM) != 0,
                                           (flags & MOE_OUT_FP32) != 0, out, ws,
                                           dbg ? dbg->dots_gu : nullptr,
                                           dbg ? dbg->dots_d : nullptr,
                                           dbg != nullptr && (dbg->q_h || dbg->d_h), dev->status,
                                           dev->num_sms, ev, capturing, s, wbits),
                             "decode")))
            return rc;
    } else {
        // the routed and multiplied input: x, or RMSNorm(x) for a stacked layer
        const uint16_t* xin = x;
        if (flags & MOE_STACKED_PRENORM) {
            if ((rc = cuda_check(launch_rmsnorm(x, T, H, 1e-6f, ws.xn, s), "rmsnorm"))) return rc;
            xin = ws.xn;
        }
        // 1. route (also writes the fp16 copy of x)
        float* logits = dbg ? dbg->logits : nullptr;
        if ((rc = cuda_check(launch_route_gemm(xin, wr, T, H, E, k, ws.route_parts, logits,
                                               ws.topk_idx, ws.topk_w, ws.x16,
                                               route_planes_bytes(T, H, E) ? ws.wr_planes : nullptr,
                                               dev->status, ws.chunk_count, ws.entry_rank, s),
                             "route")))
            return rc;
        if ((rc = mark(1))) return rc;
        // 2. bucket
        if ((rc = cuda_check(launch_bucket(ws.topk_idx, ws.topk_w, T, E, k, ws.tile_n, ws, s),
                             "bucket")))
            return rc;
        if ((rc = mark(2))) return rc;
        if ((rc = mark(3))) return rc;
        // 3. grouped GEMMs (gate/up, then down, in one launch; boundaries 4 and 5
        // both follow it)
        if ((rc = cuda_check(launch_prefill_experts(wgu, wd, ws, H, I, dev->status, dev->num_sms,
                                                    s), "prefill experts")))
            return rc;
        if ((rc = mark(4))) return rc;
        if ((rc = mark(5))) return rc;
        // 4. combine
        if ((rc = cuda_check(launch_combine(x, ws.y, false, ws.slot_pos, T, H, k,
                                            (flags & MOE_OUT_FP32) != 0, out, s), "combine")))
            return rc;
        if ((rc = mark(6))) return rc;
    }
    if (dbg) {
        if (mode == MOE_MODE_DECODE && (rc = copy_d2d(dbg->logits, ws.logits, (size_t)T * E * 4, s)))
            return rc;
        if ((rc = copy_d2d(dbg->topk_idx, ws.topk_idx, Tk * 4, s))) return rc;
        if ((rc = copy_d2d(dbg->topk_w, ws.topk_w, Tk * 4, s))) return rc;
        if ((rc = copy_d2d(dbg->expert_offsets, ws.offsets, (size_t)(E + 1) * 4, s))) return rc;
        if ((rc = copy_d2d(dbg->bucket_token, ws.bucket_token, Tk * 4, s))) return rc;
        if ((rc = copy_d2d(dbg->bucket_slot, ws.bucket_slot, Tk * 4, s))) return rc;
        if (mode == MOE_MODE_PREFILL) {
            if ((rc = copy_d2d(dbg->h, ws.h, Tk * I * 2, s))) return rc;
        } else {
            if ((rc = copy_d2d(dbg->q_x, ws.q_x, (size_t)T * H, s))) return rc;
            if ((rc = copy_d2d(dbg->d_x, ws.d_x, (size_t)T * (H / kGroup) * 2, s))) return rc;
            if ((rc = copy_d2d(dbg->q_h, ws.q_h, Tk * I, s))) return rc;
            if ((rc = copy_d2d(dbg->d_h, ws.d_h, Tk * (I / kGroup) * 2, s))) return rc;
        }
    }
    return MOE_OK;
}

}  // namespace

int record_error(int code, const char* msg) { return set_err(code, "%s", msg); }

cudaError_t record_stage(void* event, cudaStream_t s, bool capturing) {
    cudaEvent_t e = static_cast<cudaEvent_t>(event);
    return capturing ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
                     : cudaEventRecord(e, s);
}

}  // namespace moeq4

using namespace moeq4;

extern "C" {

int moe_version(void) { return 100; }

const char* moe_last_error_string(void) { return g_err; }

int moe_get_device_status(void* stream, int* status_out) {
    if (!status_out) return set_err(MOE_ERR_INVALID_ARG, "status_out is null");
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if ((rc = cuda_check(cudaMemcpyAsync(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost, s),
                         "read status")))
        return rc;
    if ((rc = cuda_check(cudaStreamSynchronize(s), "synchronize"))) return rc;
    *status_out = v;
    return MOE_OK;
}

int moe_clear_device_status(void* stream) {
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    return cuda_check(cudaMemsetAsync(dev->status, 0, sizeof(int), static_cast<cudaStream_t>(stream)),
                      "clear status");
}

size_t moe_q4_packed_bytes(int E, int N, int K) {
    if (E <= 0 || N <= 0 || K <= 0 || N % kTileRows || K % kTileK) return 0;
    return (size_t)E * (N / kTileRows) * (K / kTileK) * kTileBytes;
}

int moe_q4_pack(int fmt, const void* src, const void* src_scales, int E, int N, int K, void* dst,
                size_t dst_bytes, void* stream) {
    if (fmt != MOE_Q4_CODES && fmt != MOE_Q4_BLOCK18)
        return set_err(MOE_ERR_INVALID_ARG, "unknown pack format %d", fmt);
    if (E <= 0 || N <= 0 || K <= 0 || N % kTileRows || K % kTileK)
        return set_err(MOE_ERR_SHAPE, "pack needs E>0, N%%128==0, K%%64==0 (E=%d N=%d K=%d)", E, N, K);
    if (!src || !dst || (fmt == MOE_Q4_CODES && !src_scales))
        return set_err(MOE_ERR_INVALID_ARG, "null pointer");
    if (fmt == MOE_Q4_BLOCK18 && src_scales)
        return set_err(MOE_ERR_INVALID_ARG, "18-byte blocks carry their scales; src_scales must be NULL");
    if (!aligned16(src) || !aligned16(dst) || (src_scales && !aligned16(src_scales)))
        return set_err(MOE_ERR_ALIGN, "pointers must be 16-byte aligned");
    const size_t need = moe_q4_packed_bytes(E, N, K);
    if (dst_bytes < need)
        return set_err(MOE_ERR_INVALID_ARG, "dst holds %zu bytes, %zu needed", dst_bytes, need);
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    return cuda_check(launch_pack(fmt, src, src_scales, E, N, K, dst, static_cast<cudaStream_t>(stream)),
                      "pack");
}

int moe_q4_quantize(int src_type, const void* src, long long rows, int K, int fmt, void* dst,
                    void* dst_scales, void* stream) {
    if (src_type != MOE_SRC_F32 && src_type != MOE_SRC_BF16)
        return set_err(MOE_ERR_INVALID_ARG, "unknown source type %d", src_type);
    if (fmt != MOE_Q4_CODES && fmt != MOE_Q4_BLOCK18)
        return set_err(MOE_ERR_INVALID_ARG, "unknown output format %d", fmt);
    if (rows < 0 || K <= 0 || K % kGroup)
        return set_err(MOE_ERR_SHAPE, "quantize needs rows >= 0 and K %% 32 == 0 (rows=%lld K=%d)",
                       rows, K);
    if (rows == 0) return MOE_OK;
    if (!src || !dst || (fmt == MOE_Q4_CODES && !dst_scales))
        return set_err(MOE_ERR_INVALID_ARG, "null pointer");
    if (fmt == MOE_Q4_BLOCK18 && dst_scales)
        return set_err(MOE_ERR_INVALID_ARG, "18-byte blocks carry their scales; dst_scales must be NULL");
    if (!aligned16(src) || !aligned16(dst) || (reinterpret_cast<uintptr_t>(dst_scales) & 1u))
        return set_err(MOE_ERR_ALIGN, "src and dst must be 16-byte aligned, dst_scales 2-byte");
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    return cuda_check(launch_quantize(src_type, src, rows, K, fmt, dst, dst_scales,
                                      static_cast<cudaStream_t>(stream)),
                      "quantize");
}

int moe_route_topk(const uint16_t* x_bf16, const float* wr, int T, int H, int E, int k,
                   int32_t* topk_idx, float* topk_w, float* logits_or_null, void* stream) {
    if (T < 0 || H <= 0 || E <= 0 || E > MOE_MAX_EXPERTS || k <= 0 || k > E || k > MOE_MAX_TOPK ||
        H % 8)
        return set_err(MOE_ERR_SHAPE, "route shape T=%d H=%d E=%d k=%d outside limits", T, H, E, k);
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !wr || !topk_idx || !topk_w) return set_err(MOE_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(x_bf16) || !aligned16(wr) || !aligned16(topk_idx) || !aligned16(topk_w) ||
        (logits_or_null && !aligned16(logits_or_null)))
        return set_err(MOE_ERR_ALIGN, "pointers must be 16-byte aligned");
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    return cuda_check(launch_route(x_bf16, wr, T, H, E, k, logits_or_null, topk_idx, topk_w,
                                   nullptr, static_cast<cudaStream_t>(stream)),
                      "route");
}

// The streamed prefill stack's workspace: the prefill workspace, two staging
// buffers of one layer's packed experts (gate/up, then down), two [T, H]
// bf16 activations.
struct StreamedPlan {
    size_t prefill, gu, d, stage, act, total;
};
StreamedPlan streamed_plan(int T, int H, int I, int E, int k) {
    auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
    StreamedPlan p{};
    p.prefill = al(carve(MOE_MODE_PREFILL, T, H, I, E, k, nullptr, nullptr));
    p.gu = moe_q4_packed_bytes(E, 2 * I, H);
    p.d = moe_q4_packed_bytes(E, H, I);
    p.stage = al(p.gu) + al(p.d);
    p.act = al((size_t)T * H * 2);
    p.total = p.prefill + 2 * p.stage + 2 * p.act;
    return p;
}

size_t moe_workspace_bytes(int mode, int T, int H, int I, int E, int k) {
    if ((mode != MOE_MODE_PREFILL && mode != MOE_MODE_DECODE && mode != MOE_MODE_PREFILL_STREAMED) ||
        T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0)
        return 0;
    if (mode == MOE_MODE_PREFILL_STREAMED) return streamed_plan(T, H, I, E, k).total;
    return carve(mode, T, H, I, E, k, nullptr, nullptr);
}

int moe_q4_forward_prefill(const uint16_t* x_bf16, const float* wr, const void* wgu_packed,
                           const void* wd_packed, int T, int H, int I, int E, int k,
                           unsigned flags, void* out, void* workspace, size_t ws_bytes,
                           moe_debug* dbg, void* stream) {
    return forward(MOE_MODE_PREFILL, x_bf16, wr, wgu_packed, wd_packed, T, H, I, E, k, flags, out,
                   workspace, ws_bytes, dbg, stream);
}

int moe_w4a8_forward_decode(const uint16_t* x_bf16, const float* wr, const void* wgu_packed,
                            const void* wd_packed, int T, int H, int I, int E, int k,
                            unsigned flags, void* out, void* workspace, size_t ws_bytes,
                            moe_debug* dbg, void* stream) {
    return forward(MOE_MODE_DECODE, x_bf16, wr, wgu_packed, wd_packed, T, H, I, E, k, flags, out,
                   workspace, ws_bytes, dbg, stream);
}

int moe_w8a8_forward_decode(const uint16_t* x_bf16, const float* wr, const void* wgu_q8,
                            const void* wd_q8, int T, int H, int I, int E, int k, unsigned flags,
                            void* out, void* workspace, size_t ws_bytes, moe_debug* dbg,
                            void* stream) {
    return forward(MOE_MODE_DECODE, x_bf16, wr, wgu_q8, wd_q8, T, H, I, E, k, flags, out, workspace,
                   ws_bytes, dbg, stream, 8);
}

size_t moe_q8_packed_bytes(int E, int N, int K) {
    if (E <= 0 || N <= 0 || K <= 0 || N % kTileRows || K % kTileK) return 0;
    return (size_t)E * (N / kTileRows) * (K / kTileK) * kTileBytes8;
}

int moe_q8_pack(const void* codes, const void* scales, int E, int N, int K, void* dst,
                size_t dst_bytes, void* stream) {
    if (!codes || !scales || !dst) return set_err(MOE_ERR_INVALID_ARG, "null argument");
    if (E <= 0 || N <= 0 || K <= 0 || N % kTileRows || K % kTileK)
        return set_err(MOE_ERR_SHAPE, "E=%d N=%d K=%d: N must be a multiple of %d and K of %d", E, N, K,
                       kTileRows, kTileK);
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(dst))
        return set_err(MOE_ERR_ALIGN, "pointers must be 16-byte aligned");
    const size_t need = moe_q8_packed_bytes(E, N, K);
    if (dst_bytes < need)
        return set_err(MOE_ERR_INVALID_ARG, "dst holds %zu bytes, %zu needed", dst_bytes, need);
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    return cuda_check(launch_pack8(codes, scales, E, N, K, dst, static_cast<cudaStream_t>(stream)), "pack8");
}

int moe_q4_forward_prefill_stack_streamed(const uint16_t* x_bf16, int L, const float* const* wr,
                                          const void* const* wgu_host, const void* const* wd_host,
                                          int T, int H, int I, int E, int k, unsigned flags,
                                          void* out, void* workspace, size_t ws_bytes,
                                          void* stream) {
    int rc = check_layer_shape(MOE_MODE_PREFILL, T, H, I, E, k);
    if (rc) return rc;
    if (flags & ~(MOE_OUT_FP32 | MOE_STACKED_PRENORM))
        return set_err(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    if (L < 1 || L > MOE_DECODE_MAX_LAYERS)
        return set_err(MOE_ERR_SHAPE, "L=%d must satisfy 1 <= L <= %d", L, MOE_DECODE_MAX_LAYERS);
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !wr || !wgu_host || !wd_host || !out)
        return set_err(MOE_ERR_INVALID_ARG, "null argument");
    for (int l = 0; l < L; ++l) {
        if (!wr[l] || !wgu_host[l] || !wd_host[l])
            return set_err(MOE_ERR_INVALID_ARG, "null weight pointer of layer %d", l);
        if (!aligned16(wr[l]) || !aligned16(wgu_host[l]) || !aligned16(wd_host[l]))
            return set_err(MOE_ERR_ALIGN, "weights of layer %d must be 16-byte aligned", l);
    }
    if (!aligned16(x_bf16) || !aligned16(out) || !aligned16(workspace))
        return set_err(MOE_ERR_ALIGN, "tensor arguments must be 16-byte aligned");
    if (out == static_cast<const void*>(x_bf16))
        return set_err(MOE_ERR_INVALID_ARG, "out may not alias x");
    const StreamedPlan sp = streamed_plan(T, H, I, E, k);
    if (!workspace || ws_bytes < sp.total)
        return set_err(MOE_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", sp.total, ws_bytes);
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    // the expert weights must be page-locked host memory
    for (int l = 0; l < L; ++l) {
        for (const void* p : {wgu_host[l], wd_host[l]}) {
            cudaPointerAttributes at{};
            if (cudaPointerGetAttributes(&at, p) != cudaSuccess || at.type != cudaMemoryTypeHost) {
                cudaGetLastError();
                return set_err(MOE_ERR_INVALID_ARG,
                               "expert weights of layer %d must be pinned host memory", l);
            }
        }
    }
    {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (!dev->copy_stream) {
            if ((rc = cuda_check(cudaStreamCreateWithFlags(&dev->copy_stream, cudaStreamNonBlocking),
                                 "copy stream")))
                return rc;
            cudaEvent_t* evs[5] = {&dev->ev_fork, &dev->ev_copied[0], &dev->ev_copied[1], &dev->ev_done[0],
                                   &dev->ev_done[1]};
            for (cudaEvent_t* e : evs)
                if ((rc = cuda_check(cudaEventCreateWithFlags(e, cudaEventDisableTiming), "copy events")))
                    return rc;
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream), cs = dev->copy_stream;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    uint8_t* stage[2] = {base + sp.prefill, base + sp.prefill + sp.stage};
    uint16_t* act[2] = {reinterpret_cast<uint16_t*>(base + sp.prefill + 2 * sp.stage),
                        reinterpret_cast<uint16_t*>(base + sp.prefill + 2 * sp.stage + sp.act)};
    const size_t gu_off = 0, d_off = (sp.gu + 255) & ~(size_t)255;
    // the copies start after the work the caller enqueued before this call
    if ((rc = cuda_check(cudaEventRecord(dev->ev_fork, s), "fork"))) return rc;
    if ((rc = cuda_check(cudaStreamWaitEvent(cs, dev->ev_fork, 0), "fork"))) return rc;
    auto copy_layer = [&](int l) -> int {
        uint8_t* st = stage[l & 1];
        int r;
        if ((r = cuda_check(cudaMemcpyAsync(st + gu_off, wgu_host[l], sp.gu, cudaMemcpyHostToDevice, cs),
                            "expert copy")))
            return r;
        if ((r = cuda_check(cudaMemcpyAsync(st + d_off, wd_host[l], sp.d, cudaMemcpyHostToDevice, cs),
                            "expert copy")))
            return r;
        return cuda_check(cudaEventRecord(dev->ev_copied[l & 1], cs), "copy event");
    };
    for (int l = 0; l < L && l < 2; ++l)
        if ((rc = copy_layer(l))) return rc;
    for (int l = 0; l < L; ++l) {
        const bool last = l == L - 1;
        if ((rc = cuda_check(cudaStreamWaitEvent(s, dev->ev_copied[l & 1], 0), "copy wait"))) return rc;
        const uint16_t* xin = l == 0 ? x_bf16 : act[(l - 1) & 1];
        void* dst = last ? out : static_cast<void*>(act[l & 1]);
        const unsigned f = (flags & MOE_STACKED_PRENORM) | (last ? (flags & MOE_OUT_FP32) : 0u);
        if ((rc = forward(MOE_MODE_PREFILL, xin, wr[l], stage[l & 1] + gu_off, stage[l & 1] + d_off, T, H,
                          I, E, k, f, dst, workspace, sp.prefill, nullptr, stream)))
            return rc;
        if (l + 2 < L) {
            // layer l + 2 refills the buffer once layer l has read it
            if ((rc = cuda_check(cudaEventRecord(dev->ev_done[l & 1], s), "layer event"))) return rc;
            if ((rc = cuda_check(cudaStreamWaitEvent(cs, dev->ev_done[l & 1], 0), "layer wait"))) return rc;
            if ((rc = copy_layer(l + 2))) return rc;
        }
    }
    return MOE_OK;
}

int moe_w4a8_forward_decode_stack(const uint16_t* x_bf16, int L, const float* const* wr,
                                  const void* const* wgu_packed, const void* const* wd_packed,
                                  int T, int H, int I, int E, int k, unsigned flags, void* out,
                                  void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_layer_shape(MOE_MODE_DECODE, T, H, I, E, k);
    if (rc) return rc;
    if (flags & ~(MOE_OUT_FP32 | MOE_STACKED_PRENORM))
        return set_err(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    if (L < 1 || L > MOE_DECODE_MAX_LAYERS)
        return set_err(MOE_ERR_SHAPE, "L=%d must satisfy 1 <= L <= %d", L, MOE_DECODE_MAX_LAYERS);
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !wr || !wgu_packed || !wd_packed || !out)
        return set_err(MOE_ERR_INVALID_ARG, "null argument");
    for (int l = 0; l < L; ++l) {
        if (!wr[l] || !wgu_packed[l] || !wd_packed[l])
            return set_err(MOE_ERR_INVALID_ARG, "null weight pointer of layer %d", l);
        if (!aligned16(wr[l]) || !aligned16(wgu_packed[l]) || !aligned16(wd_packed[l]))
            return set_err(MOE_ERR_ALIGN, "weights of layer %d must be 16-byte aligned", l);
    }
    if (!aligned16(x_bf16) || !aligned16(out) || !aligned16(workspace))
        return set_err(MOE_ERR_ALIGN, "tensor arguments must be 16-byte aligned");
    if (out == static_cast<const void*>(x_bf16))
        return set_err(MOE_ERR_INVALID_ARG, "out may not alias x");
    const size_t need = carve(MOE_MODE_DECODE, T, H, I, E, k, nullptr, nullptr);
    if (!workspace || ws_bytes < need)
        return set_err(MOE_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    Workspace ws{};
    carve(MOE_MODE_DECODE, T, H, I, E, k, static_cast<uint8_t*>(workspace), &ws);
    return cuda_check(launch_decode_stack(x_bf16, L, wr, wgu_packed, wd_packed, T, H, I, E, k,
                                          (flags & MOE_STACKED_PRENORM) != 0,
                                          (flags & MOE_OUT_FP32) != 0, out, ws, dev->status,
                                          dev->num_sms, static_cast<cudaStream_t>(stream)),
                      "decode stack");
}

}  // extern "C"
