/*
 * st_rope_attn — fused QK-RMSNorm + multi-axis RoPE + scaled-dot-product
 * attention (forward and backward) for NVIDIA GB300 (sm_103a).
 *
 * What the calls compute (sources by page title and section):
 *  - "Flux-family attention: flash-attn and other backends fail in an autocast
 *    context" (diffusers issue 14104), "Root cause" list: q and k pass through
 *    RMSNorm (norm_q / norm_k, torch.nn.RMSNorm over the head dimension, fp32
 *    compute) and then the rotary embedding before attention; v does not. Under
 *    autocast q/k reach attention as fp32 while v stays bf16; this library
 *    accepts that mix and casts on load.
 *  - "Metal Flash Attention" (SimpleTuner docs), section "Fused RoPE + SDPA":
 *    the entry point rope_scaled_dot_product_attention(query, key, value,
 *    rope_cos, rope_sin, attn_mask, is_causal, scale) rotates interleaved pairs
 *    (2i, 2i+1) of Q/K right before attention, with one angle per pair; its
 *    backward applies the inverse rotation (sin negated) so gradients are taken
 *    w.r.t. the pre-RoPE Q/K.
 *  - same page, section "Enable In SimpleTuner": bool masks (True = attend),
 *    additive float masks, batched [B,H,S_q,S_kv] and broadcast [B,1,1,S_kv]
 *    masks, causal calls; all-true bool masks are detected and skipped; work is
 *    encoded on the caller's stream with no per-call synchronisation; the
 *    dispatch counters (get_dispatch_stats) become st_get_stats().
 *
 * Differences from that entry point: tensors are [B, S, H, D] (any strides on
 * B/S/H, unit stride on D) instead of BHSD (a BHSD tensor passes as its
 * transpose(1, 2) view, without a copy); the rotation comes either from
 * per-token position ids, axis widths and theta (built on the device) or from
 * the entry point's own pair-duplicated cos/sin tables; the RMSNorm of q and k
 * is fused in; the backward also returns the two norm-weight gradients.
 *
 * Per token t and head h (D = 128):
 *   r      = 1 / sqrt(mean_d x[d]^2 + eps)                 (x = q or k row)
 *   n[d]   = x[d] * r * w[d]                              (w = q/k norm weight)
 *   axis a owns dims [o_a, o_a + d_a), o_a = d_0 + ... + d_{a-1}, sum d_a = D;
 *   pair j of axis a: phi = id[t, a] * theta^(-2j / d_a)
 *   (y[o_a+2j], y[o_a+2j+1]) = (n0 cos phi - n1 sin phi, n0 sin phi + n1 cos phi)
 *   s_ij   = scale * q'_i . k'_j  (+ additive mask; -inf where a bool mask is
 *            False, or where j > i when causal, top-left aligned)
 *   O_i    = sum_j softmax_j(s_ij) v_j,   LSE_i = ln sum_j exp(s_ij)
 * A row with no attended key gets O = 0, LSE = -inf and zero gradients.
 *
 * Conventions for every call:
 *  - Ownership: the caller owns every buffer, including the workspace. The
 *    library never allocates device memory and never synchronises the stream
 *    (except st_get_stats and st_check_status, which say so).
 *  - Asynchrony: work is enqueued on `stream` (a cudaStream_t, NULL = legacy
 *    default stream) and runs in stream order.
 *  - Errors: arguments are validated before anything is launched; a non-OK
 *    status means nothing was enqueued. st_last_error() gives a message. No C++
 *    exception crosses this boundary.
 *  - Device waits are bounded: a kernel that gives up waiting records a
 *    timeout, which the next st_check_status() returns as ST_ERR_TIMEOUT.
 *  - Pointers are device pointers unless stated otherwise; data pointers and
 *    the byte strides of the B/S/H dimensions must be multiples of 16 bytes.
 */
#ifndef ST_ROPE_ATTN_H
#define ST_ROPE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ST_API __attribute__((visibility("default")))
#else
#define ST_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ST_OK = 0,
  ST_ERR_INVALID_ARG = 1, /* null pointer, bad flag combination, bad rope spec */
  ST_ERR_DTYPE = 2,       /* unsupported dtype for that argument */
  ST_ERR_SHAPE = 3,       /* inconsistent or unsupported shapes */
  ST_ERR_ALIGN = 4,       /* pointer or stride not 16-byte aligned, D stride != 1 */
  ST_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required */
  ST_ERR_CUDA = 6,        /* a CUDA runtime call failed (message in st_last_error) */
  ST_ERR_TIMEOUT = 7,     /* a kernel's bounded wait ran out (from st_check_status) */
  ST_ERR_UNSUPPORTED = 8  /* valid request outside what this build implements */
} st_status;

typedef enum { ST_BF16 = 0, ST_F16 = 1, ST_F32 = 2, ST_BOOL = 3, ST_I32 = 4 } st_dtype;

/* A strided view. Strides are in elements. Unused trailing dims are ignored. */
typedef struct {
  void* data;
  int32_t dtype; /* st_dtype */
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];
} st_tensor;

/* Rotary specification: either position ids (the first five fields) or the
 * cos/sin tables of "Metal Flash Attention", section "Fused RoPE + SDPA"
 * (the last four fields); exactly one of `ids` and `cos` is set.
 * ids:   [B|1, S_q, n_axes], int32 or fp32, device; position id of each token
 *        on each axis (Flux: text (0,0,0), image (0,row,col)).
 * ids_k: the same for the keys ([B|1, S_kv, n_axes]); NULL means "same as ids"
 *        and requires S_q == S_kv.
 * axes_dim: width of each axis in head dims (even, summing to D); theta: base.
 * cos, sin: pair-duplicated tables (cos[..., 2j] == cos[..., 2j+1]) of shape
 *        [S_q, D], [1, S_q, D] or [B, S_q, D]; fp32, bf16 or fp16 (the same for
 *        both), any element strides, device. Entry 2j of each pair is read and
 *        converted to fp32 (entry 2j+1 is not read: the tables promise it is
 *        equal); n_axes, axes_dim and theta are then ignored.
 * cos_k, sin_k: the same for the keys ([S_kv, D], [1, S_kv, D] or
 *        [B, S_kv, D]); NULL means "same as cos/sin" and requires S_q == S_kv.
 * reuse_tables: read by st_rope_attn_bwd only. 1 states that the workspace
 *        passed to the backward already holds the device tables of exactly
 *        this rotation, the tile classes of exactly this mask and the
 *        normalised, rotated q rows (Q') of exactly these inputs, written by an
 *        st_rope_attn_fwd call on the same workspace pointer with a backward-
 *        sized workspace_bytes, stream-ordered before the backward (its first
 *        bytes have the forward's layout); the backward then skips rebuilding
 *        them, and relies on the forward having zeroed its dQ accumulator
 *        there, which it consumes: one reusing backward per forward. Anything
 *        else is undefined results (not a fault). 0: the backward rebuilds
 *        them. */
typedef struct {
  const st_tensor* ids;
  const st_tensor* ids_k;
  int32_t n_axes; /* 1..8 (ids form) */
  int32_t axes_dim[8];
  double theta;
  const st_tensor* cos;
  const st_tensor* sin;
  const st_tensor* cos_k;
  const st_tensor* sin_k;
  int32_t reuse_tables;
} st_rope;

/* Counters after the pages' dispatch statistics. Bumped only after a launch
 * was enqueued successfully. */
typedef struct {
  uint64_t fwd_calls;             /* st_rope_attn_fwd calls ("rope_instream") */
  uint64_t bwd_calls;             /* st_rope_attn_bwd calls ("rope_autograd") */
  uint64_t mask_all_true_skipped; /* calls whose bool mask was all True (device-detected) */
  uint64_t mixed_dtype_calls;     /* calls with fp32 q/k and bf16 v (cast on load) */
  uint64_t tiles_skipped;         /* key tiles skipped (all-False or causal-dead), device count */
  uint64_t tiles_total;           /* key tiles visited or skipped, device count */
  uint64_t timeouts;              /* kernels that recorded a bounded-wait timeout */
  uint64_t kernel_launches;       /* kernels this library enqueued (host count) */
} st_stats;

/* Kernel kinds reported by st_timing_read. */
enum {
  ST_K_TABLE = 0,     /* rotary (cos, sin) table */
  ST_K_CLASSIFY = 1,  /* bool mask tile classification */
  ST_K_FWD = 2,       /* forward attention */
  ST_K_BWD_PRE = 3,   /* Delta = rowsum(dO * O), zero the dQ accumulator */
  ST_K_BWD = 4,       /* backward attention: dV, dK (inverse rotation and RMSNorm
                         backward in its epilogue), dQ' accumulation */
  ST_K_DQ_POST = 5,   /* dQ: inverse rotation + RMSNorm backward */
  ST_K_DW = 6,        /* norm-weight gradient reduction */
  ST_K_QPRIME = 7,    /* Q' rows for a backward without a forward's workspace */
  ST_K_PROBE = 8,     /* bounded-wait self-test */
  ST_K_COUNT = 9
};

/* Per-kernel device time between two st_timing_read calls. */
typedef struct {
  uint64_t launches[ST_K_COUNT];
  double ms[ST_K_COUNT];
} st_kernel_times;

/* Bytes of device workspace a call needs (0 on invalid arguments; the error is
 * then in st_last_error). for_backward = 0 for st_rope_attn_fwd, 1 for
 * st_rope_attn_bwd. */
ST_API size_t st_rope_attn_workspace_size(const st_tensor* q, const st_tensor* k, const st_tensor* v,
                                   const st_tensor* mask, int causal, const st_rope* rope, int for_backward);

/* Forward.
 *  q, k:   [B, S_q, H, D] / [B, S_kv, H_kv, D], bf16, fp16 or fp32 (q and k
 *          of one dtype). D = 128; B, H <= 65535; S_q, S_kv <= 2^30
 *          (ST_ERR_SHAPE otherwise).
 *  v:      [B, S_kv, H_kv, D], bf16, fp16 or fp32.
 *          Dtype combinations ("Metal Flash Attention", section
 *          "Requirements": FP32 runs natively, FP16/BF16 on low-precision
 *          kernels):
 *          - bf16 (or fp16) q, k, v: tensor-core MMAs on bf16 (fp16)
 *            operands with fp32 accumulation, softmax and norm arithmetic;
 *          - fp32 q, k with bf16 or fp16 v (the autocast mix): q and k are
 *            normalised and rotated in fp32, then rounded to v's type for the
 *            MMAs, as an autocast SDPA would;
 *          - fp32 q, k, v: every product and sum in fp32 on the CUDA cores
 *            (exact-fp32 kernels, far slower than the tensor cores).
 *          16-bit q/k of a type other than v's are rejected (ST_ERR_DTYPE).
 *          H_kv divides H (grouped K/V heads; H_kv = H is plain multi-head
 *          attention): query head h attends with K/V head h / (H / H_kv), and
 *          k is normalised and rotated at the K/V head count ("Metal Flash
 *          Attention", section "Fused RoPE + SDPA": GQA inputs are rotated at
 *          the K/V head count and expanded afterwards).
 *  q_norm_w, k_norm_w: [D] fp32 RMSNorm weights; eps: RMSNorm epsilon.
 *  rope:   rotary specification (above).
 *  mask:   NULL, or [B|1, H|1, S_q|1, S_kv] bool (True = attend) or additive
 *          fp32/bf16 (added to the scaled scores); unit stride on S_kv.
 *  causal: 1 for top-left causal masking; must be 0 when mask != NULL.
 *  scale:  score scale; <= 0 selects 1/sqrt(D).
 *  o:      [B, S_q, H, D] output, dtype of v.  lse: [B, H, S_q] fp32 output,
 *          natural-log log-sum-exp of each row (contiguous).
 *  workspace: device buffer of at least st_rope_attn_workspace_size(..., 0)
 *          bytes, 256-byte aligned; its contents need no initialisation. When
 *          workspace_bytes also covers st_rope_attn_workspace_size(..., 1)
 *          (and q, k, v are not all fp32), the forward leaves its Q' rows
 *          ([B, S_q, H, D] in the 16-bit operand type, the bf16 or fp16 values
 *          its attention kernel multiplies) in the backward's part of the
 *          workspace and zeroes the backward's fp32 dQ accumulator there, for
 *          a backward with rope->reuse_tables = 1.
 *  stream: cudaStream_t. */
ST_API st_status st_rope_attn_fwd(const st_tensor* q, const st_tensor* k, const st_tensor* v, const st_tensor* q_norm_w,
                           const st_tensor* k_norm_w, float eps, const st_rope* rope, const st_tensor* mask,
                           int causal, float scale, st_tensor* o, st_tensor* lse, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Backward. Inputs as for the forward plus o and lse from it and d_o
 * ([B, S_q, H, D], dtype of v). Outputs:
 *  dq, dk: dtype of q / k; dv: dtype of v; same shapes as q / k / v (with
 *          grouped K/V heads, dk and dv of a K/V head sum the gradients of
 *          all the query heads that use it).
 *  d_q_norm_w, d_k_norm_w: [D] fp32 (overwritten, not accumulated).
 * dk/dv/dw are deterministic; dq is not bit-reproducible: its fp32
 * accumulation across key tiles is a sum of TMA bulk reduce-adds (fp32 adds in
 * L2) whose order varies from run to run. */
ST_API st_status st_rope_attn_bwd(const st_tensor* q, const st_tensor* k, const st_tensor* v, const st_tensor* q_norm_w,
                           const st_tensor* k_norm_w, float eps, const st_rope* rope, const st_tensor* mask,
                           int causal, float scale, const st_tensor* o, const st_tensor* lse, const st_tensor* d_o,
                           st_tensor* dq, st_tensor* dk, st_tensor* dv, st_tensor* d_q_norm_w,
                           st_tensor* d_k_norm_w, void* workspace, size_t workspace_bytes, void* stream);

/* Size of the library's built-in forward scratch, used by
 * st_rope_attn_fwd_noalloc. */
#define ST_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Forward without a caller-provided workspace (no counterpart in the paper;
 * an addition of this library). Some callers cannot allocate device memory:
 * code running while a CUDA graph is being captured into a fixed memory plan,
 * plugins hosted by inference runtimes that hand out only input and output
 * buffers, and serving processes that forbid allocation after start-up to keep
 * their memory footprint fixed. For them the scratch (rotary tables, mask tile
 * classes, control words) lives in one static device array of
 * ST_NOALLOC_SCRATCH_BYTES, held by every GPU that loads the library until the
 * process exits. Arguments and results are those of st_rope_attn_fwd.
 *  - A call whose scratch need exceeds ST_NOALLOC_SCRATCH_BYTES returns
 *    ST_ERR_WORKSPACE and launches nothing (the need is B_ids * S * 512 bytes
 *    of tables, doubled with separate key ids, plus the mask tile classes).
 *  - The first call on a device looks up the array's device address (a
 *    one-time set-up per device, which also loads the library's kernels on
 *    that device); make that first call before any stream capture begins.
 *  - Every call on a device shares the one array: calls that overlap on the
 *    GPU (on different streams, or from several threads without ordering)
 *    race on it. Calls in stream order are safe; each call re-initialises what
 *    must start from zero.
 *  - Nothing here calls cudaMalloc, cudaFree or any allocating routine. */
ST_API st_status st_rope_attn_fwd_noalloc(const st_tensor* q, const st_tensor* k, const st_tensor* v,
                                          const st_tensor* q_norm_w, const st_tensor* k_norm_w, float eps,
                                          const st_rope* rope, const st_tensor* mask, int causal, float scale,
                                          st_tensor* o, st_tensor* lse, void* stream);

/* Message of the last failing call on this thread ("" if none). */
ST_API const char* st_last_error(void);

/* Copies the counters into *out. Synchronises the device to read the device-
 * side counters. */
ST_API st_status st_get_stats(st_stats* out);
ST_API void st_reset_stats(void);

/* Kernel timing for measurement: while enabled, every kernel launch is
 * bracketed by two CUDA events recorded on its own stream. st_timing_read
 * waits for those events, returns the summed durations per kernel kind and
 * starts a new accumulation. Off by default. */
ST_API st_status st_timing_enable(int on);
ST_API st_status st_timing_read(st_kernel_times* out);

/* Self-test of the bounded-wait mechanism: enqueues one tiny kernel that waits
 * on an mbarrier nothing arrives on and gives up after `budget_cycles`
 * (clock64 cycles, 1..2^34), recording a timeout exactly as the attention
 * kernels do. The next st_check_status() then returns ST_ERR_TIMEOUT and the
 * CUDA context stays usable. */
ST_API st_status st_selftest_wait_timeout(long long budget_cycles, void* stream);

/* Synchronises `stream` and reports ST_ERR_TIMEOUT if any kernel recorded a
 * bounded-wait timeout since the previous check (the record is then cleared),
 * or ST_ERR_CUDA if the stream holds an error. For tests and debugging. */
ST_API st_status st_check_status(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* ST_ROPE_ATTN_H */
