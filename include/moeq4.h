/*
 * moeq4 — a 4-bit (Q4_0 family) mixture-of-experts expert-FFN layer for one
 * NVIDIA GB300 (sm_103a).  C ABI.
 *
 * What the layer computes (the page "A 35B Hybrid-Attention Mixture-of-Experts
 * Model on a 6GB 2011 GPU: Hand-Written 4-bit CUDA Inference for Fermi",
 * Methodology 1 "Hybrid GPU-Prefill / CPU-Decode" and 2 "Memory and
 * Quantization"):
 *
 *   weights   group-wise symmetric 4-bit, Q4_0 family: blocks of 32 codes
 *             q in 0..15 along a row's input dimension share one fp16 scale d,
 *             and each weight is w = d * (q - 8)
 *   router    logits = x W_r^T (fp32 accumulation); the k largest are chosen
 *             (equal logits: lower expert index first); their weights are a
 *             softmax over the k chosen logits
 *   expert    h = silu(W_g x) * (W_u x), y = W_d h   (SwiGLU FFN)
 *   combine   out[t] = x[t] + sum_j w[t, j] * y(t, j), j = 0..k-1 in order
 *   prefill   ("grouped 4-bit GEMM"): bf16 activations; the tensor-core
 *             operands are fp16 (x converted exactly, weights d(q-8) rounded
 *             once, h rounded once) with fp32 accumulation; values beyond the
 *             fp16 range (|v| > 65504) saturate there
 *   decode    ("W4A8 integer kernel"): activations quantised to int8 per 32
 *             with an fp16 scale; exact int32 group dot products, scaled by
 *             d_w * d_x in fp32; h quantised the same way before the down
 *             projection
 *
 * Conventions for every entry point:
 *   - Tensor arguments are DEVICE pointers owned by the caller, row-major and
 *     contiguous, 16-byte aligned (MOE_ERR_ALIGN otherwise).  Nothing is
 *     allocated on the forward path: scratch lives in a caller-provided
 *     workspace sized by moe_workspace_bytes().
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream; outputs are valid once
 *     the stream has reached the point of the call.
 *   - The return value is MOE_OK (0) or a negative MOE_ERR_* code; the reason
 *     is available from moe_last_error_string() (thread-local).  No exception
 *     crosses the ABI; device code never traps.  A kernel whose bounded wait
 *     ran out records MOE_ERR_TIMEOUT in a per-device status word that
 *     moe_get_device_status() reads.
 *   - bf16 and fp16 tensors are passed as their 16-bit patterns.
 */
#ifndef MOEQ4_H
#define MOEQ4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MOE_OK                0
#define MOE_ERR_INVALID_ARG  -1  /* null pointer, bad enum, bad flag        */
#define MOE_ERR_SHAPE        -2  /* dimensions outside the supported limits */
#define MOE_ERR_ALIGN        -3  /* pointer not 16-byte aligned             */
#define MOE_ERR_UNSUPPORTED  -4  /* no sm_103a device / not built for it    */
#define MOE_ERR_CUDA         -5  /* a CUDA runtime or driver call failed    */
#define MOE_ERR_TIMEOUT      -6  /* a device-side bounded wait ran out      */
#define MOE_ERR_WORKSPACE    -7  /* workspace missing or too small          */

/* ---- limits -------------------------------------------------------------- */
#define MOE_GROUP         32     /* Q4_0 block / activation group           */
#define MOE_MAX_EXPERTS   256
#define MOE_MAX_TOPK      16
#define MOE_DECODE_MAX_T  32     /* decode path: tokens per call            */
#define MOE_W8_DECODE_MAX_T 16   /* 8-bit-weight decode: tokens per call    */
#define MOE_DECODE_MAX_LAYERS 64 /* decode stack: layers per call           */

/* ---- moe_q4_pack formats ------------------------------------------------- */
/* MOE_Q4_CODES:   src = uint8 codes [E, N, K] (values 0..15, one per byte),
 *                 src_scales = fp16 [E, N, K/32].
 * MOE_Q4_BLOCK18: src = 18-byte blocks [E, N, K/32]: fp16 scale
 *                 (little-endian) then 16 bytes, byte j holding element j in
 *                 its low nibble and element j+16 in its high nibble;
 *                 src_scales must be NULL.                                   */
#define MOE_Q4_CODES   0
#define MOE_Q4_BLOCK18 1

/* ---- forward flags ------------------------------------------------------- */
#define MOE_OUT_FP32  1u   /* out is fp32 [T, H]; otherwise bf16 [T, H]      */
/* MOE_STACKED_PRENORM: a pre-norm residual layer for stacking.  The router
 * and the experts read xn = RMSNorm(x) (per token: x / sqrt(mean(x^2) +
 * 1e-6), unit gain, computed in fp32 and rounded to bf16); the residual added
 * to the MoE term is x itself: out = x + sum_j w_j y_j(xn).  With bf16
 * output, layer l+1 takes layer l's out as its x.  The pages do not print
 * the layer's norm; this is the plainest pre-norm reading that keeps many
 * stacked residual layers finite. */
#define MOE_STACKED_PRENORM 2u

/* ---- forward modes for moe_workspace_bytes ------------------------------- */
#define MOE_MODE_PREFILL 0
#define MOE_MODE_DECODE  1
#define MOE_MODE_PREFILL_STREAMED 2  /* moe_q4_forward_prefill_stack_streamed */

/*
 * Optional stage outputs of a forward call (all DEVICE pointers, each may be
 * NULL).  Used to check each stage on its own.  "Bucket order" means the
 * (token, slot) pairs grouped by expert: expert 0's tokens in ascending order,
 * then expert 1's, and so on; row p of a bucket-order tensor belongs to
 * bucket_token[p], slot bucket_slot[p].
 */
typedef struct moe_debug {
    float*    logits;          /* [T, E] fp32 router logits                  */
    int32_t*  topk_idx;        /* [T, k] chosen experts, best first          */
    float*    topk_w;          /* [T, k] routing weights                     */
    int32_t*  expert_offsets;  /* [E+1] exclusive prefix sum of bucket sizes */
    int32_t*  bucket_token;    /* [T*k] token of each bucket-order row       */
    int32_t*  bucket_slot;     /* [T*k] slot j of each bucket-order row      */
    uint16_t* h;               /* prefill: [T*k, I] fp16 SwiGLU output,
                                  bucket order                               */
    int8_t*   q_x;             /* decode: [T, H] int8 activation codes       */
    uint16_t* d_x;             /* decode: [T, H/32] fp16 activation scales   */
    int32_t*  dots_gu;         /* decode: [T*k, 2I, H/32] int32 group dots of
                                  gate (rows 0..I-1) and up (I..2I-1),
                                  bucket order                               */
    int8_t*   q_h;             /* decode: [T*k, I] int8 codes of h           */
    uint16_t* d_h;             /* decode: [T*k, I/32] fp16 scales of h       */
    int32_t*  dots_d;          /* decode: [T*k, H, I/32] int32 group dots of
                                  the down projection, bucket order          */
    void**    stage_events;    /* NULL or MOE_NUM_STAGE_EVENTS cudaEvent_t
                                  handles (caller-created); the call records
                                  event i at stage boundary i on `stream`
                                  (as external events, so they also work
                                  inside a captured CUDA graph):
                                  prefill: 0 start, 1 routed, 2 bucketed,
                                  3 (= 2), 4 gate/up done, 5 down done
                                  (both expert GEMMs are one launch: 4 and
                                  5 both follow it), 6 combined (end);
                                  decode: 0 start, 1 logits and codes of x
                                  done (first kernel), 2..6 all after the
                                  second kernel (routing, experts and
                                  combine are one launch)                    */
} moe_debug;

#define MOE_NUM_STAGE_EVENTS 7

/* Library version (major*10000 + minor*100 + patch). */
int moe_version(void);

/* Reason for the last non-zero return on this thread ("" if none). */
const char* moe_last_error_string(void);

/* Reads the current device's status word: MOE_OK, or MOE_ERR_TIMEOUT if a
 * kernel's bounded wait ran out since the last moe_clear_device_status().
 * Synchronises `stream`. */
int moe_get_device_status(void* stream, int* status_out);
int moe_clear_device_status(void* stream);

/*
 * Packed weight layout.  A weight tensor [E, N, K] (N output rows, K input
 * columns, N % 128 == 0, K % 64 == 0) is cut into tiles of 128 rows x 64
 * columns, stored in (expert, row block, column block) order, 4608 bytes per
 * tile: 4096 bytes of codes (row r of the tile at byte 32*r) followed by 512
 * bytes of fp16 scales (row r: the scales of its two 32-blocks at 4096+4*r).
 * Within a row's 32 code bytes, 32-bit word c holds columns 8c..8c+7: the
 * even columns 8c, 8c+2, 8c+4, 8c+6 in nibbles 0..3 (bits 0..15) and the odd
 * columns 8c+1, 8c+3, 8c+5, 8c+7 in nibbles 4..7 (bits 16..31).  Each tile is
 * one 16-byte-aligned bulk copy.
 */
size_t moe_q4_packed_bytes(int E, int N, int K);

/*
 * moe_q4_pack — canonical Q4_0 weights (see the formats above) to the packed
 * layout.  Source and destination are device pointers; dst must hold
 * moe_q4_packed_bytes(E, N, K) bytes.  Codes above 15 are taken modulo 16.
 * For the gate/up projection pass the [E, 2I, H] tensor whose rows 0..I-1
 * are the gate and rows I..2I-1 the up projection; for the down projection
 * the [E, H, I] tensor.
 */
int moe_q4_pack(int fmt, const void* src, const void* src_scales,
                int E, int N, int K, void* dst, size_t dst_bytes, void* stream);

/* ---- moe_q4_quantize source types ---------------------------------------- */
#define MOE_SRC_F32  0   /* fp32 weights                                       */
#define MOE_SRC_BF16 1   /* bf16 weights (their 16-bit patterns)               */

/*
 * moe_q4_quantize — float weights to Q4_0-family blocks on the GPU (the page,
 * Methodology 2 "Quantization": group-wise symmetric 4-bit weights of the
 * Q4_0 family; the page prints no encoder, this is that family's usual
 * rule).  Per block of 32 consecutive weights of a row: m = the element of
 * largest magnitude (the first on a tie), sign kept; d = fp16(m / -8), round
 * to nearest even (d may be negative); q = min(15, max(0, floor(x/d + 8.5)))
 * against the stored d, taken exactly (the result equals the rounding of the
 * exact rational); d = 0 gives q = 8.  So w = d (q - 8) decodes it.
 *   src       [rows, K] fp32 or bf16 (src_type), device pointer
 *   fmt       MOE_Q4_CODES: dst = uint8 codes [rows, K] (0..15),
 *                           dst_scales = fp16 [rows, K/32];
 *             MOE_Q4_BLOCK18: dst = 18-byte blocks [rows, K/32] (the layout
 *                           above), dst_scales must be NULL
 * The output is what moe_q4_pack takes.  Limits: rows >= 0, K % 32 == 0,
 * src and dst 16-byte aligned (dst_scales 2-byte); inputs finite with
 * |m / 8| <= 65504 (beyond it d overflows to infinity and every code is 8).
 * One kernel on `stream`; nothing is allocated.
 */
int moe_q4_quantize(int src_type, const void* src, long long rows, int K, int fmt, void* dst,
                    void* dst_scales, void* stream);

/*
 * moe_route_topk — router logits, top-k selection and routing weights.
 *   x_bf16  [T, H] bf16 hidden states       wr [E, H] fp32 router weights
 *   topk_idx [T, k] int32 (descending logit; equal logits: lower index first)
 *   topk_w   [T, k] fp32 softmax over the k chosen logits
 *   logits_or_null [T, E] fp32 (optional)
 * Limits: 1 <= E <= 256, 1 <= k <= min(E, 16), H % 8 == 0, T >= 0.
 */
int moe_route_topk(const uint16_t* x_bf16, const float* wr, int T, int H, int E, int k,
                   int32_t* topk_idx, float* topk_w, float* logits_or_null, void* stream);

/* Workspace bytes needed by a forward call of the given mode and shape. */
size_t moe_workspace_bytes(int mode, int T, int H, int I, int E, int k);

/*
 * moe_q4_forward_prefill — one MoE layer with bf16 activations: route, bucket
 * by expert, grouped gate/up GEMM with SwiGLU, grouped down GEMM scaled by the
 * routing weight, combine with the residual.
 *   x_bf16     [T, H] bf16          wr [E, H] fp32
 *   wgu_packed moe_q4_pack of the [E, 2I, H] gate/up tensor
 *   wd_packed  moe_q4_pack of the [E, H, I] down tensor
 *   out        [T, H] fp32 if flags & MOE_OUT_FP32, else bf16; may not alias x
 *   workspace  >= moe_workspace_bytes(MOE_MODE_PREFILL, T, H, I, E, k) bytes
 *   dbg        NULL or stage outputs to fill
 * Limits: H % 128 == 0, I % 128 == 0, 1 <= E <= 256, 1 <= k <= min(E, 16),
 * 0 <= T, T * k * max(H, I) < 2^31.
 * The call's kernels are launched with programmatic dependent launch; the
 * first one reads `wr` before the work that precedes it on the stream has
 * finished, so `wr` must not be written by the kernel launched immediately
 * before this call on the same stream.  x, the output and the workspace are
 * touched only after that work has finished.
 */
int moe_q4_forward_prefill(const uint16_t* x_bf16, const float* wr,
                           const void* wgu_packed, const void* wd_packed,
                           int T, int H, int I, int E, int k, unsigned flags,
                           void* out, void* workspace, size_t ws_bytes,
                           moe_debug* dbg, void* stream);

/*
 * moe_w4a8_forward_decode — one MoE layer on the W4A8 integer path (the page,
 * Methodology 1 "Decode (CPU)" and Key Contributions 2: 4-bit weights times
 * 8-bit activations with integer dot products): same arguments and layouts
 * as the prefill call, T <= MOE_DECODE_MAX_T, and the on-chip staging must
 * fit: T * (H + I) * 1.25 bytes plus four weight tiles, and the T x E logits,
 * stay under ~180 KB (MOE_ERR_SHAPE otherwise; T = 32 at H = 2048, I = 768,
 * E = 256 fits).  The int32 group dots are exact; the float sums run in fp32
 * in a fixed order, so repeated calls give the same bits.
 *
 * The call launches kernels that let their successors start early
 * (programmatic dependent launch), first a prep kernel (router logits, int8
 * codes of x, and the clearing of the counters the layer kernel synchronises
 * on). For T <= 16 two follow: the experts kernel, in clusters of two CTAs
 * (top-k and buckets in every CTA; each bucket cut into slices of at most 2
 * rows, 1 for T <= 4 (8-bit weights: 4 and 1); units of (slice, 128-feature
 * block of h) shared by the cluster's CTAs through distributed shared
 * memory: gate/up, h, down), and a combine kernel (residual plus the parts
 * of every output). For larger T one cooperative layer kernel (one CTA per
 * SM: top-k, buckets, gate/up, h, down and the combine over all CTAs, the
 * experts' rows and K ranges split into tasks) follows. The prep kernel
 * reads `wr` before the work that precedes it on the stream has finished, so
 * `wr` must not be written by the kernel launched immediately before this
 * call on the same stream; x, the output and the workspace are touched only
 * after that work has finished.
 * Nothing in the workspace has to survive from one call to the next, and
 * any other call may use the same workspace in between.  Routing needs
 * E <= 256 (one prep CTA per expert).
 */
int moe_w4a8_forward_decode(const uint16_t* x_bf16, const float* wr,
                            const void* wgu_packed, const void* wd_packed,
                            int T, int H, int I, int E, int k, unsigned flags,
                            void* out, void* workspace, size_t ws_bytes,
                            moe_debug* dbg, void* stream);

/*
 * moe_w4a8_forward_decode_stack — L consecutive decode layers (each adds its
 * expert output to its input, the residual stream) from one call: the
 * pages' per-token decode loop over the MoE layers.  The call enqueues each
 * layer's two kernels on the stream, every kernel linked to the one before
 * by programmatic dependent launch (the next layer's router row is staged
 * while the layer before still runs).  Layer l + 1 reads layer l's output
 * rounded to bf16; the result equals, bit for bit, L moe_w4a8_forward_decode
 * calls chained through bf16 outputs with the same flags (MOE_OUT_FP32
 * applies to the last layer only).
 *   x_bf16     [T, H] input of layer 0 (not written)
 *   L          1 <= L <= MOE_DECODE_MAX_LAYERS
 *   wr, wgu_packed, wd_packed
 *              HOST arrays of L device pointers, one layer each, layouts as in
 *              moe_w4a8_forward_decode (the arrays are read during the call)
 *   out        the last layer's output; may not alias x
 *   workspace  >= moe_workspace_bytes(MOE_MODE_DECODE, T, H, I, E, k) bytes
 * Each layer clears its own counters in its first kernel, so nothing in the
 * workspace has to survive between calls; the layers' intermediate outputs
 * live in the workspace.  Shapes as for moe_w4a8_forward_decode.  Routing,
 * codes and sums follow the single-layer call exactly; no stage outputs are
 * written.
 */
int moe_w4a8_forward_decode_stack(const uint16_t* x_bf16, int L, const float* const* wr,
                                  const void* const* wgu_packed, const void* const* wd_packed,
                                  int T, int H, int I, int E, int k, unsigned flags, void* out,
                                  void* workspace, size_t ws_bytes, void* stream);

/*
 * 8-bit expert weights (the companion page "A Modern Multimodal Assistant
 * on a 6 GB 2011 GPU: Stage-Validated, All-GPU CUDA Inference for Fermi",
 * Abstract, runs 8-bit weights against 4-bit ones; its format is not
 * printed, this library takes the Q8_0-style reading): blocks of 32 int8 codes q in
 * -127..127 along a row share one fp16 scale d, w = d * q.
 *
 * moe_q8_packed_bytes / moe_q8_pack — int8 codes [E, N, K] and fp16 scales
 * [E, N, K/32] (DEVICE) to 8-bit tiles: 128 rows x 64 columns, 8704 bytes
 * (each row's 64 codes, 8-code chunks in the order 0,4,1,5,2,6,3,7, then the
 * 128 x 2 fp16 scales), tiles ordered as the Q4_0 ones.  N % 128 == 0,
 * K % 64 == 0.
 *
 * moe_w8a8_forward_decode — the decode layer of moe_w4a8_forward_decode with
 * 8-bit expert weights (both packed by moe_q8_pack): the same routing,
 * activation quantiser and combine; group dots sum q_w * q_a exactly.
 * T <= MOE_W8_DECODE_MAX_T (the clustered layer kernel); workspace as for
 * moe_w4a8_forward_decode (moe_workspace_bytes(MOE_MODE_DECODE, ...)).
 * Stage outputs as for the 4-bit call.
 */
size_t moe_q8_packed_bytes(int E, int N, int K);
int moe_q8_pack(const void* codes, const void* scales, int E, int N, int K, void* dst,
                size_t dst_bytes, void* stream);
int moe_w8a8_forward_decode(const uint16_t* x_bf16, const float* wr, const void* wgu_q8,
                            const void* wd_q8, int T, int H, int I, int E, int k, unsigned flags,
                            void* out, void* workspace, size_t ws_bytes, moe_debug* dbg,
                            void* stream);

/*
 * moe_q4_forward_prefill_stack_streamed — L consecutive prefill layers whose
 * packed expert weights stay in HOST memory and are streamed to the GPU layer
 * by layer, overlapped with the layers' compute.  This is the pages' prefill
 * mechanism (the page, Methodology 1 "Prefill (GPU)": the experts live in
 * host RAM and move to the GPU one layer at a time) on the host-to-GPU link
 * of this machine, for models whose experts do not fit in device memory.
 *
 * The call enqueues, on the caller's stream and a copy stream of the
 * library, per layer l:
 *   - one cudaMemcpyAsync for layer l's gate/up weights and one for its
 *     down weights, into staging buffer l % 2 of the workspace;
 *   - the layer itself (the kernels of moe_q4_forward_prefill) once that
 *     copy is done.
 * Layer l + 2's copies wait for layer l's kernels, which read the same
 * buffer.  Events link the two streams, so the call can be captured into a
 * CUDA graph.  Layer l + 1 reads layer l's output rounded to bf16 (kept in
 * the workspace); the result equals, bit for bit, L moe_q4_forward_prefill
 * calls chained through bf16 outputs with the same flags and the weights
 * in device memory.  MOE_OUT_FP32 applies to the last layer only.
 *   x_bf16     [T, H] DEVICE, input of layer 0 (not written)
 *   L          1 <= L <= MOE_DECODE_MAX_LAYERS
 *   wr         HOST array of L DEVICE pointers to the router weights
 *   wgu_host, wd_host
 *              HOST arrays of L HOST pointers to each layer's packed weights
 *              (layouts as in moe_q4_forward_prefill).  They must be pinned
 *              (page-locked: cudaHostAlloc or cudaHostRegister), else
 *              MOE_ERR_INVALID_ARG.  They must not change until the work
 *              the call enqueued has finished.
 *   out        the last layer's output [T, H]; may not alias x
 *   workspace  >= moe_workspace_bytes(MOE_MODE_PREFILL_STREAMED, T, H, I, E, k)
 *              bytes: the prefill workspace, two staging buffers of one
 *              layer's experts, and two [T, H] bf16 activations.
 * Shapes as for moe_q4_forward_prefill.  The first call on a device creates
 * the copy stream and its events; make that first call before any stream
 * capture.
 */
int moe_q4_forward_prefill_stack_streamed(const uint16_t* x_bf16, int L, const float* const* wr,
                                          const void* const* wgu_host, const void* const* wd_host,
                                          int T, int H, int I, int E, int k, unsigned flags,
                                          void* out, void* workspace, size_t ws_bytes,
                                          void* stream);

/*
 * moe_w4a8_forward_decode_noalloc — the same decode layer as
 * moe_w4a8_forward_decode, for callers that cannot allocate device memory:
 * components hosted by an application or plugin interface that owns all
 * device memory and offers no allocation, and latency-critical decode loops
 * that must not call cudaMalloc (it can synchronise the device).  The paper
 * has no counterpart; this is a convenience of this library.
 *
 * The caller passes inputs and outputs exactly as for
 * moe_w4a8_forward_decode; the scratch workspace is a fixed device array of
 * MOE_NOALLOC_SCRATCH_BYTES inside this library (every GPU that loads the
 * library holds it until the process exits).  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.
 *   - Shapes whose workspace (moe_workspace_bytes(MOE_MODE_DECODE, ...)) is
 *     larger than the array are rejected with MOE_ERR_WORKSPACE; 8 MiB covers
 *     T <= 32 at H = 2048, I = 768, E <= 256, k = 8 (6.4 MiB at most, at
 *     T = 16).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls share the array and it keeps the last call's contents.  No
 *     value in it has to start at zero: every call clears the counters it
 *     synchronises on (in its first kernel) and writes everything else it
 *     reads earlier in the same call, whatever shape the previous call had.
 *     Calls whose work overlaps on the GPU (several streams or host threads
 *     on one device) race on the array: serialise them.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (8u << 20)
int moe_w4a8_forward_decode_noalloc(const uint16_t* x_bf16, const float* wr,
                                    const void* wgu_packed, const void* wd_packed,
                                    int T, int H, int I, int E, int k, unsigned flags,
                                    void* out, moe_debug* dbg, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ4_H */
