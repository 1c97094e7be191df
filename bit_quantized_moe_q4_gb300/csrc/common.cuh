// Shared device helpers for the moeq4 kernels (sm_103a): constants of the
// packed Q4_0 layout, bf16/fp16 bit helpers, bounded mbarrier waits, bulk and
// tensor copies, and the tcgen05 (5th-generation tensor core) primitives.
// Everything here is inline PTX written against the public PTX ISA.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moeq4 {

// ---- packed Q4_0 layout (see include/moeq4.h) ----------------------------
constexpr int kGroup = 32;            // codes per fp16 scale
constexpr int kTileRows = 128;        // rows per packed tile
constexpr int kTileK = 64;            // columns per packed tile
constexpr int kTileCodeBytes = 4096;  // 128 rows x 32 bytes
constexpr int kTileBytes = 4608;      // codes + 128 rows x 2 fp16 scales
// 8-bit weight tiles (the decode path's 8-bit variant): 128 rows x 64 int8
// codes, then the same 128 x 2 fp16 scales
constexpr int kTileCodeBytes8 = 8192;
constexpr int kTileBytes8 = 8704;
constexpr int kMaxExperts = 256;

// ---- device status word: kernels record a timed-out wait here -------------
constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = -6;
// Upper bound on any single device-side wait, in nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, kStatusOk, code);
}

// ---- number formats --------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}
// fp32 -> fp16 (round to nearest even), saturating at +-65504 instead of
// overflowing to infinity.
__device__ __forceinline__ uint16_t float_to_half_bits_sat(float f) {
    f = fminf(fmaxf(f, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(f));
}

// ---- shared-memory addresses and fences ------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Orders this thread's earlier generic-proxy accesses to global memory before
// its later bulk copies (async proxy) that read global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---- gpu-scope flags between CTAs ------------------------------------------
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Atomic add that releases this thread's (and, after a barrier, its CTA's)
// earlier writes and acquires what the earlier adders released; returns the
// old value.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// A thread that finds the phase incomplete is suspended until it completes
// or kSuspendHintNs pass (then the caller checks its own time limit), so
// waiting warps take no issue slots from the working ones.
constexpr uint32_t kSuspendHintNs = 1000000u;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity to complete, for at most
// kWaitLimitNs.  Returns false (and the caller must give up) on expiry.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ---- bulk copies (TMA) -----------------------------------------------------
// Contiguous global -> shared copy; both addresses 16-byte aligned, size a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// An L2 cache policy for data read once: evict it first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}
// 2-D tiled tensor load: box at (x = column, y = row).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// 2-D gather of four rows (y0..y3) of one box width starting at column x;
// the tensor map's box is one row high.  Rows land at 4 consecutive box rows.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0,
                                            int y1, int y2, int y3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
        : "memory");
}
// 16-byte asynchronous copy global -> shared (L2 only), and an arrival on
// `bar` once every such copy of this thread has landed (the barrier's count
// must include this thread; the arrival does not add to it).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Waits until every cp.async of this thread has landed (in its shared memory).
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---- tcgen05: tensor memory and MMA ----------------------------------------
// Allocation is done by one full warp; the TMEM base address is written to
// shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit inputs (kind::f16), fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Same, with A read from tensor memory: a_tmem addresses lane 0 of the A
// tile (row i of A in lane i, two 16-bit elements per 32-bit column).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// 32 lanes x 32 bits, 32 consecutive columns per thread (this warp's lanes).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes (64 bf16), 8-row atoms of 1024 bytes.
// The leading-byte offset is unused by this layout (set to 1); the stride
// byte offset is 1024 (the distance between 8-row atoms).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address, bits 0..13
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset
    d |= (uint64_t)1 << 46;                    // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                    // swizzle: 128 bytes
    return d;
}
// Instruction descriptor for kind::f16 with fp16 A and B (both K-major) and an
// fp32 accumulator of M x N.  (Format code 0 is fp16, 1 would be bf16.)
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4)                          // D format: f32
           | (0u << 7)                        // A format: f16
           | (0u << 10)                       // B format: f16
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// ---- thread-block clusters and programmatic dependent launch ---------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// All threads of all CTAs of the cluster; release/acquire orders shared and
// distributed-shared memory.  Cluster CTAs are co-scheduled, so it completes.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// 16 bytes into the shared memory of a CTA of this cluster (raddr and rbar
// from mapa_shared): an asynchronous store whose bytes count as transaction
// bytes on that CTA's mbarrier rbar, so the receiver's wait on the barrier
// also covers the data.
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float a, float b, float c, float d,
                                            uint32_t rbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
            raddr),
        "f"(a), "f"(b), "f"(c), "f"(d), "r"(rbar)
        : "memory");
}
// mbar_try_wait / mbar_wait with cluster-scope acquire: the phase's bytes
// were written by other CTAs of the cluster.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}
// Programmatic dependent launch: wait for the prerequisite grid's completion
// (and its memory), or let the dependent grid start being scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- warp helpers ------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 256); the
// block total lands in *total.  Every thread of the block must call it.
__device__ __forceinline__ int block256_exclusive_scan(int v, int* total) {
    __shared__ int warp_tot[8];
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0, all = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        if (w < warp) base += warp_tot[w];
        all += warp_tot[w];
    }
    __syncthreads();
    *total = all;
    return base + incl - v;
}

// ---- router top-k ----------------------------------------------------------
// Order-preserving 32-bit key of a float: larger float -> larger unsigned key.
// -0.0 is first turned into +0.0 so the two compare equal, as floats do.
__device__ __forceinline__ uint32_t float_order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token's logits (row of `E` floats readable by the whole warp);
// lane j < k returns the j-th choice in (sel_i, weight).  Order: larger logit
// first; equal logits -> lower expert index first.
//
// Lane l owns the contiguous experts [l*P, l*P + P), P = ceil(E/32) <= 8, and
// sorts them once (a sorting network on (key descending, index ascending), in
// PM >= P registers).  Each of the k rounds takes the warp maximum of the
// lanes' heads (redux.sync), and among the lanes holding it the lowest one,
// which owns the lowest index because lanes own ascending index ranges.  That
// lane drops its head by shifting its list (predicated moves, no branch).
// The weights are a softmax over the k chosen logits.
template <int PM>
__device__ __forceinline__ void warp_topk_sorted(const float* row, int E, int k, int& sel_i, float& weight) {
    const int lane = threadIdx.x % 32;
    const int P = (E + 31) / 32;
    uint32_t kk[PM];
    int ii[PM];
#pragma unroll
    for (int i = 0; i < PM; ++i) {
        const int e = lane * P + i;
        const bool have = i < P && e < E;
        kk[i] = have ? float_order_key(row[e]) : 0u;  // key 0: absent
        ii[i] = have ? e : 0;
    }
    auto cs = [&](int a, int b) {  // (a, b) into order: a first
        const bool sw = kk[b] > kk[a] || (kk[b] == kk[a] && ii[b] < ii[a]);
        const uint32_t ka = kk[a];
        const int ia = ii[a];
        kk[a] = sw ? kk[b] : ka;
        ii[a] = sw ? ii[b] : ia;
        kk[b] = sw ? ka : kk[b];
        ii[b] = sw ? ia : ii[b];
    };
    if constexpr (PM == 2) {
        cs(0, 1);
    } else if constexpr (PM == 4) {
        cs(0, 1); cs(2, 3); cs(0, 2); cs(1, 3); cs(1, 2);
    } else if constexpr (PM == 8) {
        cs(0, 2); cs(1, 3); cs(4, 6); cs(5, 7); cs(0, 4); cs(1, 5); cs(2, 6); cs(3, 7); cs(0, 1); cs(2, 3);
        cs(4, 5); cs(6, 7); cs(2, 4); cs(3, 5); cs(1, 4); cs(3, 6); cs(1, 2); cs(3, 4); cs(5, 6);
    }
    sel_i = 0;
    for (int r = 0; r < k; ++r) {
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, kk[0]);
        const int wl = __ffs(__ballot_sync(0xffffffffu, kk[0] == kmax)) - 1;
        const int e = __shfl_sync(0xffffffffu, ii[0], wl);
        if (lane == r) sel_i = e;
        const bool win = lane == wl;
#pragma unroll
        for (int i = 0; i + 1 < PM; ++i) {
            kk[i] = win ? kk[i + 1] : kk[i];
            ii[i] = win ? ii[i + 1] : ii[i];
        }
        kk[PM - 1] = win ? 0u : kk[PM - 1];
    }
    const float sel_v = (lane < k) ? row[sel_i] : 0.f;
    const float m = __shfl_sync(0xffffffffu, sel_v, 0);  // the largest
    const float z = (lane < k) ? expf(sel_v - m) : 0.f;
    const float s = warp_sum(z);
    weight = z / s;
}

__device__ __forceinline__ void warp_topk(const float* row, int E, int k, int& sel_i, float& weight) {
    if (E <= 32) warp_topk_sorted<1>(row, E, k, sel_i, weight);
    else if (E <= 64) warp_topk_sorted<2>(row, E, k, sel_i, weight);
    else if (E <= 128) warp_topk_sorted<4>(row, E, k, sel_i, weight);
    else warp_topk_sorted<8>(row, E, k, sel_i, weight);
}

// Activation quantiser decision, taken in fp32 (see act-quant kernels):
// d = fp16(amax / 127) saturating at 65504; q = round-half-away(v / d)
// clamped to +-127; d == 0 gives q = 0.
__device__ __forceinline__ uint16_t act_scale_bits(float amax) {
    float quot = __fdiv_rn(amax, 127.0f);
    quot = fminf(quot, 65504.0f);
    return __half_as_ushort(__float2half_rn(quot));
}
__device__ __forceinline__ int act_code(float v, float d) {
    if (d == 0.0f) return 0;
    float r = roundf(__fdiv_rn(v, d));  // roundf: half away from zero
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int)r;
}

}  // namespace moeq4
