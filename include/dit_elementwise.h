/*
 * dit_elementwise.h -- C ABI of libdit_elementwise.so, the GB300 (sm_103a)
 * kernels for the memory-bound elementwise hot path of LTX-2-style video
 * diffusion transformers.
 *
 * Operations, each one kernel launch on the caller's stream:
 *
 *   dit_residual_gate_add          out = hidden + update * gate
 *   dit_rmsnorm_modulate           out = rms_norm(x, eps) * (1 + scale) + shift
 *   dit_gate_add_rmsnorm_modulate  both in one pass: writes the new residual
 *                                  and the modulated input of the next site
 *   dit_*_fp8                      the modulation / fused op with an FP8
 *                                  (E4M3) modulated output
 *   dit_gelu_tanh                  the feed-forward's tanh-GELU, elementwise
 *   dit_grouped                    one of the first three over several
 *                                  problems (e.g. video and audio streams)
 *                                  in one launch
 *   dit_selfcheck                  bit-for-bit check of one runtime key
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Tensors.  Every tensor is contiguous, row-major [B, L, D] in device memory
 *   (or memory the device can address), all of one dtype.  A "row" is one
 *   (b, l) pair of D elements.  An operand of layout DIT_ROW_BCAST has shape
 *   [B, 1, D]: its row b is used for all L rows of batch b.
 * Arithmetic.  Every element is loaded exactly into fp32, computed with IEEE
 *   fp32 operations (round to nearest even, no fused multiply-add where the
 *   formula below writes two operations, no flush of subnormals) and rounded
 *   once to the output dtype (round to nearest even; overflow gives +-inf;
 *   NaN propagates).
 * Ownership.  The caller owns all memory.  The library allocates nothing,
 *   keeps no per-call state and never synchronises: each call validates its
 *   arguments on the host, enqueues one kernel on `stream` (0 = the legacy
 *   default stream; dit_grouped: one kernel, or one per problem as stated
 *   there) and returns.  Outputs are complete once the stream
 *   reaches that point.
 * Aliasing.  out == hidden (exactly the same pointer) is allowed, as is
 *   residual_out == hidden; any other overlap between an output and another
 *   tensor returns DIT_ERR_ALIAS.
 * Alignment.  Pointers must be aligned to the element size (2 bytes for
 *   bf16/fp16, 4 for fp32); otherwise DIT_ERR_MISALIGNED.  Any such pointer
 *   is accepted: the widest vector access that every pointer and the row
 *   pitch D * element_size allow is chosen per call (up to 32 bytes).  Rows
 *   whose pitch is not a multiple of 16 bytes, in tensors that start on
 *   16-byte boundaries, are still moved in 16-byte granules (the row-wise
 *   operations group the rows by their offset modulo 16 bytes); only
 *   sub-views that start off a 16-byte boundary fall back to narrower
 *   accesses.
 * Errors.  Argument errors are returned before any launch and leave outputs
 *   untouched.  B, L, D >= 0; a call with B * L * D == 0 returns DIT_OK and
 *   launches nothing.  A launch failure reported by the CUDA runtime returns
 *   DIT_ERR_LAUNCH; faults during execution surface at the caller's next
 *   synchronisation, as for any CUDA kernel.  There is no fallback path.
 * Threads.  Entry points may be called from several host threads; the only
 *   shared state is a per-device cache of launch limits, filled on first use.
 */
#ifndef DIT_ELEMENTWISE_H
#define DIT_ELEMENTWISE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The stream type of the CUDA runtime, without requiring its headers. */
typedef struct CUstream_st* dit_stream_t;

typedef enum { DIT_BF16 = 0, DIT_FP16 = 1, DIT_FP32 = 2 } dit_dtype;

typedef enum {
  DIT_FULL = 0,      /* [B, L, D]: one value per element            */
  DIT_ROW_BCAST = 1  /* [B, 1, D]: one vector per batch, reused over L */
} dit_layout;

typedef enum {
  DIT_OK = 0,
  DIT_ERR_NULL_PTR = 1,     /* a tensor pointer is NULL while B*L*D > 0      */
  DIT_ERR_BAD_SHAPE = 2,    /* B, L or D negative, or B*L*D overflows         */
  DIT_ERR_BAD_DTYPE = 3,    /* dtype is not a dit_dtype value                 */
  DIT_ERR_BAD_LAYOUT = 4,   /* layout is not a dit_layout value               */
  DIT_ERR_ALIAS = 5,        /* an output overlaps another tensor (other than
                               the allowed out == hidden)                     */
  DIT_ERR_BAD_EPS = 6,      /* eps is negative, infinite or NaN               */
  DIT_ERR_LAUNCH = 7,       /* the CUDA runtime rejected the launch           */
  DIT_ERR_MISALIGNED = 8,   /* a pointer is not aligned to the element size   */
  DIT_ERR_NO_DEVICE = 9,    /* no current CUDA device could be queried        */
  DIT_ERR_BAD_OP = 10,      /* op is not a dit_op value, or (dit_grouped) count
                               is outside [0, DIT_MAX_GROUP]                  */
  DIT_ERR_WORKSPACE = 11,   /* dit_selfcheck: workspace NULL, smaller than
                               dit_selfcheck_workspace_bytes or not 256-byte
                               aligned                                        */
  DIT_ERR_BAD_STATISTIC = 12  /* dit_set_statistic: not a dit_statistic value */
} dit_status;

/* Version of this interface; bumped on any incompatible change. */
#define DIT_ABI_VERSION 3
int dit_abi_version(void);

/* A static, human-readable name for a status code. */
const char* dit_status_string(dit_status status);

/*
 * The row statistic r = 1 / sqrt(mean(x^2) + eps) of the modulating
 * operations (dit_rmsnorm_modulate, dit_gate_add_rmsnorm_modulate, their
 * _strided, grouped and _fp8 forms), chosen for the whole process:
 *
 *   DIT_STATISTIC_FAST (default): the row's fp32 sum of squares, one FMA per
 *     element, merged in tree order; ms = S / D by a corrected quotient;
 *     r = rsqrtf(fl(ms + eps)) refined by one Newton-Raphson step.  r is
 *     within about seventeen fp32 ulps of the exact statistic's, so each
 *     output element is within one bf16/fp16 ulp of the exact definition's
 *     except where the final + shift cancels (|y| much smaller than
 *     |x r (1 + scale)|), where the difference stays below one dtype ulp of
 *     max(|t|, |y|), t = n (1 + scale); fp32 outputs within 2^-18 of
 *     max(|t|, |y|).  A row whose fp32 sum leaves [2^-100, 2^100] (a square
 *     that overflows fp32, infinities, squares below its normal range) is
 *     summed again with its elements scaled by 2^-64 or 2^64; a mean square
 *     in fp32's subnormal range with eps = 0 may then be one subnormal step
 *     off.
 *   DIT_STATISTIC_EXACT: ms = RN32(mean(x^2)), the exact mean of the row's
 *     squares rounded once to fp32, and r = RN32(1 / sqrt(fl(ms + eps))),
 *     correctly rounded: every output element equals the definition
 *     evaluated in fp32 with those values, bit for bit (NaN payloads aside),
 *     whatever kernel or launch shape computes it.  The squares are summed in
 *     compensated (TwoSum) pairs with a proven error bound and the rounding
 *     decided from it; rows the bound cannot decide (ties and near-ties) are
 *     summed exactly.  It costs time: on [1,32640,4096] bf16 the modulation
 *     takes about a third longer and the fused op an eighth (the compensated
 *     sum makes them issue-bound).
 *
 * Sources: the statistic is fp32 and the result is held to one bf16 ulp per
 * element (prhub summary of sglang PR #34172, "implementation breakdown"
 * item 2 and risks item 1).
 *
 * The mode is read when a call is made (host side) and selects the kernel
 * it launches -- a CUDA graph keeps the statistic its captured calls were
 * made with; set it before launching, not concurrently with calls from other
 * threads.  dit_set_statistic returns
 * DIT_ERR_BAD_STATISTIC for other values and leaves the mode unchanged.
 */
typedef enum {
  DIT_STATISTIC_FAST = 0,
  DIT_STATISTIC_EXACT = 1
} dit_statistic;
dit_status dit_set_statistic(dit_statistic statistic);
dit_statistic dit_get_statistic(void);

/*
 * Gated residual update:  out[b,l,d] = hidden[b,l,d] + update[b,l,d] * G
 * with G = gate[b,l,d] (gate_layout DIT_FULL) or gate[b,0,d] (DIT_ROW_BCAST),
 * evaluated as p = fl32(update * G), s = fl32(hidden + p), out = rnd(s).
 *
 * Source: sglang PR #29361 "Add diffusion residual-gate CUDA fast path for
 * LTX2", section Motivation (the hot pattern hidden + update * gate for
 * contiguous [B, L, D] tensors with a full gate or a [B, 1, D] gate) and
 * section Modifications (full and row-broadcast gates, dtype coverage, tail
 * shapes, rejection of unsupported inputs).
 *
 * out, hidden, update: [B, L, D].  gate: [B, L, D] or [B, 1, D].
 * out may be hidden (in-place update).
 */
dit_status dit_residual_gate_add(void* out, const void* hidden,
                                 const void* update, const void* gate,
                                 int64_t B, int64_t L, int64_t D,
                                 dit_dtype dtype, dit_layout gate_layout,
                                 dit_stream_t stream);

/*
 * adaLN modulation with a weightless RMSNorm over each row:
 *   r   = 1 / sqrt(mean_d(x[b,l,d]^2) + eps)     (fp32 statistic per row)
 *   out = rnd(fl32(fl32(fl32(x * r) * fl32(1 + S)) + H))
 * with S, H = scale, shift at [b,l,d] (mod_layout DIT_FULL) or [b,0,d]
 * (DIT_ROW_BCAST).  The statistic is computed as dit_set_statistic chose
 * (fast by default; exact: ms = RN32(mean(x^2)) and r = RN32(1/sqrt(fl(ms +
 * eps))), the same output bits whatever the launch shape).  A row holding a
 * NaN gives NaN; a row holding an infinity a zero statistic.
 *
 * Rows of at most 2^24 elements (D larger: DIT_ERR_BAD_SHAPE).
 *
 * Source: prhub summary of sglang PR #34172 (LTX-2 quality=high fused
 * RMSNorm+modulate), section "key source snippet" (the eager expression
 * rms_norm(x, eps) * (1 + scale) + shift of _ltx2_rms_norm_modulate, called
 * with the block's norm_eps) and section "implementation breakdown", item 2
 * (RMSNormNoWeight: the norm has no weight; one launch for the whole
 * expression).
 *
 * out, x: [B, L, D].  scale, shift: [B, L, D] or [B, 1, D].  eps >= 0.
 */
dit_status dit_rmsnorm_modulate(void* out, const void* x, const void* scale,
                                const void* shift, int64_t B, int64_t L,
                                int64_t D, float eps, dit_dtype dtype,
                                dit_layout mod_layout, dit_stream_t stream);

/*
 * Fused residual gate + modulation, one pass over the rows:
 *   residual_out = dit_residual_gate_add(hidden, update, gate)   (stored)
 *   modulated_out = dit_rmsnorm_modulate(residual_out, scale, shift, eps)
 * The statistic is taken over the residual as stored (rounded to the dtype),
 * so the two outputs are bitwise those of the two separate calls.  The
 * residual is never re-read from memory.  D at most 2^24.
 *
 * Source: the two operations above; the pages name the fused family member
 * (fused_gate_rmsnorm, prhub summary of sglang PR #34172, "implementation
 * breakdown" items 2 and 4) without describing it.
 *
 * residual_out, modulated_out, hidden, update: [B, L, D].
 * gate: per gate_layout.  scale, shift: per mod_layout.
 * residual_out may be hidden; modulated_out may not alias anything.
 */
dit_status dit_gate_add_rmsnorm_modulate(
    void* residual_out, void* modulated_out, const void* hidden,
    const void* update, const void* gate, const void* scale, const void* shift,
    int64_t B, int64_t L, int64_t D, float eps, dit_dtype dtype,
    dit_layout gate_layout, dit_layout mod_layout, dit_stream_t stream);

/*
 * Strided [B, 1, D] operands.  The same three operations, with one more
 * argument: vec_stride, the distance in elements between the vectors of
 * consecutive batches of every DIT_ROW_BCAST operand of the call (D for a
 * contiguous [B, 1, D] tensor).  It lets a caller pass rows of an adaLN
 * table directly: with a per-block table of shape [B, 9, D] (shift, scale,
 * gate for each of the block's three modulation sites -- self-attention,
 * prompt cross-attention, feed-forward: prhub summary of sglang PR #34172,
 * "implementation breakdown" item 3), the site's vectors are
 * table + i*D with vec_stride = 9*D, and no chunk is copied out.
 *
 * vec_stride must be >= D when B > 1 (DIT_ERR_BAD_SHAPE otherwise); it is
 * unused for DIT_FULL operands.  Aliasing is checked over the whole span
 * [p, p + ((B-1)*vec_stride + D) elements) of each strided operand.
 */
dit_status dit_residual_gate_add_strided(void* out, const void* hidden,
                                         const void* update, const void* gate,
                                         int64_t B, int64_t L, int64_t D,
                                         dit_dtype dtype, dit_layout gate_layout,
                                         int64_t vec_stride, dit_stream_t stream);

dit_status dit_rmsnorm_modulate_strided(void* out, const void* x,
                                        const void* scale, const void* shift,
                                        int64_t B, int64_t L, int64_t D,
                                        float eps, dit_dtype dtype,
                                        dit_layout mod_layout, int64_t vec_stride,
                                        dit_stream_t stream);

dit_status dit_gate_add_rmsnorm_modulate_strided(
    void* residual_out, void* modulated_out, const void* hidden,
    const void* update, const void* gate, const void* scale, const void* shift,
    int64_t B, int64_t L, int64_t D, float eps, dit_dtype dtype,
    dit_layout gate_layout, dit_layout mod_layout, int64_t vec_stride,
    dit_stream_t stream);

/*
 * tanh-approximated GELU, elementwise over n contiguous elements:
 *   out[i] = 0.5 * x[i] * (1 + tanh(z)),  z = sqrt(2/pi) * (x + 0.044715 x^3)
 * evaluated in fp32 as x * sigmoid(2z) (the same function: 1 + tanh(z) =
 * 2 / (1 + exp(-2z))), then rounded once to the dtype.  16-bit dtypes use
 * the hardware approximations of 2^v and 1/v (each within about 2^-22
 * relative); fp32 uses expf and an IEEE division.
 *
 * Source: prhub summary of sglang PR #34172, "implementation breakdown"
 * item 3 (LTX2FeedForward: proj_in, then the tanh-GELU act) and "functions
 * and motivation" (the FFN GELU is the second elementwise chain that
 * torch.compile fuses).
 *
 * out may be x (in place); any other overlap returns DIT_ERR_ALIAS.
 */
dit_status dit_gelu_tanh(void* out, const void* x, int64_t n, dit_dtype dtype,
                         dit_stream_t stream);

/*
 * Modulated output quantised to FP8 (OCP E4M3: 4 exponent bits, bias 7, 3
 * fraction bits, no infinities, largest finite 448), with a static
 * per-tensor scale:
 *   y   = the fp32 modulation value of dit_rmsnorm_modulate (before any
 *         rounding to the activation dtype)
 *   out = e4m3(fl32(y * fl32(1 / *quant_scale)))
 * rounded to nearest-even, saturating to +-448 (infinities included); NaN
 * stays NaN.  One byte per element, [B, L, D] row-major.
 *
 * Source: the prhub summary of sglang PR #34172 lists, among its related
 * PRs, the RMSNorm + FP8 quantisation fusion of the same fused-norm family;
 * the pages give neither the format nor the scaling, so the plainest
 * readings are taken: E4M3 (the activation FP8 format of such fusions), a
 * per-tensor scale that divides (applied as a multiplication by its
 * correctly rounded reciprocal), saturation instead of overflow.
 *
 * quant_scale: DEVICE pointer to one fp32 value, finite and > 0 (read by the
 * kernel, so it may change between graph replays; not checked on the host:
 * other values give defined but meaningless codes).  vec_stride: as in the
 * _strided calls.
 *
 * These calls take the staged row kernel only: every input pointer (and
 * residual_out) 16-byte aligned, D * element_size a multiple of 16 bytes (a
 * multiple of 16 elements is what FP8 GEMM inputs need anyway), the vector
 * stride in bytes a multiple of 16, and `out` aligned to 8 bytes (bf16/fp16)
 * or 4 (fp32) -- otherwise DIT_ERR_MISALIGNED; rows of at most 16 KB (D <=
 * 8192 for 16-bit, 4096 for fp32) -- otherwise DIT_ERR_BAD_SHAPE.  `out`
 * may not overlap any other tensor or *quant_scale.
 */
dit_status dit_rmsnorm_modulate_fp8(void* out, const void* x, const void* scale,
                                    const void* shift, int64_t B, int64_t L,
                                    int64_t D, float eps, dit_dtype dtype,
                                    dit_layout mod_layout, int64_t vec_stride,
                                    const float* quant_scale, dit_stream_t stream);

/* The fused op with its modulated output in E4M3 (residual_out keeps the
 * dtype, bitwise that of dit_residual_gate_add). */
dit_status dit_gate_add_rmsnorm_modulate_fp8(
    void* residual_out, void* out, const void* hidden, const void* update,
    const void* gate, const void* scale, const void* shift, int64_t B,
    int64_t L, int64_t D, float eps, dit_dtype dtype, dit_layout gate_layout,
    dit_layout mod_layout, int64_t vec_stride, const float* quant_scale,
    dit_stream_t stream);

/*
 * Grouped launches: one operation over up to DIT_MAX_GROUP independent
 * problems of one dtype and layout, each with its own pointers, B, L, D and
 * vec_stride.  An LTX-2 block applies each of its adaLN modulations to the
 * video stream (hidden size 4096) and to the audio stream (hidden size 2048)
 * -- prhub summary of sglang PR #34172, "implementation breakdown" item 3
 * (the six sites: video/audio self-attention, prompt cross-attention and
 * feed-forward) and the test section (hidden 4096 = video, 2048 = audio) --
 * so one grouped call covers both streams of a site.
 *
 * Each problem computes what the single call of the same operation
 * computes: the residual bit for bit; the modulated output bit for bit with
 * the exact statistic, and within the fast statistic's bound otherwise (its
 * sum may be taken in another tree order than a single call's).
 *
 * Launch: when every non-empty problem has 16-byte aligned pointers, pitch
 * and vec_stride and (for the modulating operations) rows of at most 8192
 * 16-bit or 4096 fp32 elements, the call enqueues ONE kernel on `stream`
 * that covers all of them, with the CTAs split in proportion to the
 * problems' sizes.  Otherwise, and for a DIT_FULL gate of the residual gate
 * (whose flat kernel has no rows), it enqueues one kernel per non-empty
 * problem, in order.  No problem may write memory that another problem
 * reads or writes (DIT_ERR_ALIAS), since they run concurrently.
 *
 * problems: a HOST array of `count` descriptors (0 <= count <= DIT_MAX_GROUP;
 * NULL allowed when count == 0), read during the call only.  Validation is
 * that of the single calls, per problem, before anything is launched; the
 * first failing problem's status is returned.
 */
#define DIT_MAX_GROUP 8

typedef enum {
  DIT_OP_RESIDUAL_GATE = 0,          /* out = hidden + update * gate */
  DIT_OP_RMSNORM_MODULATE = 1,       /* out = rms_norm(x) * (1 + scale) + shift */
  DIT_OP_GATE_ADD_RMSNORM_MODULATE = 2 /* both, fused */
} dit_op;

typedef struct {
  void* out;          /* residual gate: out; modulation: out; fused: residual_out */
  void* out2;         /* fused: modulated_out; NULL otherwise */
  const void* x;      /* residual gate, fused: hidden; modulation: x */
  const void* update; /* residual gate, fused */
  const void* gate;   /* residual gate, fused */
  const void* scale;  /* modulation, fused */
  const void* shift;  /* modulation, fused */
  int64_t B, L, D;
  int64_t vec_stride; /* as in the _strided calls (elements; D if contiguous) */
} dit_problem;

/* gate_layout is read by the residual gate and the fused op, mod_layout by
 * the modulation and the fused op; eps by the modulating operations. */
dit_status dit_grouped(dit_op op, const dit_problem* problems, int count,
                       float eps, dit_dtype dtype, dit_layout gate_layout,
                       dit_layout mod_layout, dit_stream_t stream);

/*
 * Self-check of one runtime key: (op, dtype, gate_layout, mod_layout, D).
 *
 * The pages' integration checks every runtime key of its pointwise fusions
 * bit for bit on first use and falls back to the model's math on a mismatch
 * or a launch failure (vllm-omni PR #7350, "[Kernel] Enable LTX DiffVAE
 * fusions on SM100 and SM103", section Purpose).  This library has no
 * fallback; dit_selfcheck gives the caller the check itself.  It enqueues on
 * `stream`, in order:
 *   1. seeded inputs of a [2, 7, D] problem, written into `workspace`;
 *   2. the operation, through the same validation and launch path as the
 *      public call of that op, dtype and layouts (so the kernel the library
 *      picks for 256-byte aligned tensors with rows of D elements);
 *   3. the expected outputs from plain one-thread-per-element kernels;
 *   4. the count of output words that differ from the expected ones, added
 *      to *mismatches after the call has set it to zero.
 * Every output has exactly one correct value: the residual gate is defined
 * to the bit, and the inputs of the modulating ops make the row statistic
 * exact in any summation order (every normalised value is +-1/2, eps = 3/4,
 * so r = 1).  Zero mismatches: the key's path computes the definition.
 *
 * workspace: device memory of at least dit_selfcheck_workspace_bytes(op,
 * dtype, D) bytes, 256-byte aligned, owned by the caller and free for the
 * call's duration; on return it holds, from offset 0, nine tensors of
 * N = 14 * D elements each starting on a 256-byte boundary -- x (hidden),
 * update, gate, scale, shift (a [2, 1, D] operand fills its first 2 * D
 * elements), out, out2, expected, expected2 -- then 14 fp32 row statistics.
 * mismatches: device pointer to one unsigned int (4-byte aligned).
 * eps is fixed (3/4) and not an argument.  The call does not synchronise:
 * read *mismatches after the stream has reached it.
 */
int64_t dit_selfcheck_workspace_bytes(dit_op op, dit_dtype dtype, int64_t D);

dit_status dit_selfcheck(dit_op op, dit_dtype dtype, dit_layout gate_layout,
                         dit_layout mod_layout, int64_t D, void* workspace,
                         int64_t workspace_bytes, unsigned int* mismatches,
                         dit_stream_t stream);

/*
 * dit_selfcheck_static: the same check, with no workspace argument and no
 * allocation.  The pages have no counterpart; this entry point exists for
 * callers that cannot allocate device memory when they want the check -- a
 * process whose device memory is all held by a framework's caching
 * allocator, or a latency-critical loop that must not call cudaMalloc or
 * cudaFree (both may synchronise the device).
 *
 * The workspace is a static device array of DIT_SELFCHECK_STATIC_BYTES
 * (4 MiB) inside the library, which every GPU that loads the library keeps
 * until the process exits.  That covers bf16/fp16 keys up to D = 16384 and
 * fp32 keys up to D = 8192; a key whose dit_selfcheck_workspace_bytes is
 * larger returns DIT_ERR_WORKSPACE.  The caller passes `mismatches` (device,
 * one unsigned int) as for dit_selfcheck; the call allocates nothing.
 *
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress, a host-side runtime query that allocates nothing;
 * the first one per context may load the library's device code).  All calls
 * share the one array, and nothing in it needs to start at zero; calls whose
 * work overlaps on the GPU (other streams, other host threads) race on its
 * contents, so order them -- one stream, or a synchronisation between them.
 * After the check the array holds dit_selfcheck's workspace layout: nine
 * slots of round_up(2 * 7 * D * element size, 256) bytes -- inputs hidden/x,
 * update, gate, scale, shift, outputs out (residual), modulated, and the
 * plain kernels' expected out and modulated -- then the row statistics.
 */
#define DIT_SELFCHECK_STATIC_BYTES (4u << 20)

dit_status dit_selfcheck_static(dit_op op, dit_dtype dtype,
                                dit_layout gate_layout, dit_layout mod_layout,
                                int64_t D, unsigned int* mismatches,
                                dit_stream_t stream);

/*
 * dit_selfcheck_static_workspace: the device address (*workspace) and size
 * (*bytes, DIT_SELFCHECK_STATIC_BYTES) of dit_selfcheck_static's array in
 * the current context, for reading back what a check left there.  The array
 * belongs to the library: the caller may read it (after the check's stream
 * is synchronised) and must not free it.  DIT_ERR_NULL_PTR for a NULL
 * argument; DIT_ERR_NO_DEVICE (with *workspace = NULL, *bytes = 0) when no
 * device is current or the runtime cannot give the address.
 */
dit_status dit_selfcheck_static_workspace(void** workspace, int64_t* bytes);

#ifdef __cplusplus
}
#endif
#endif /* DIT_ELEMENTWISE_H */
