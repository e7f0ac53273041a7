/*
 * moe.h -- C ABI of the GB300 MoE layer hot path (route -> permute -> grouped
 * SwiGLU expert GEMM -> combine, plus the static-shape pooled-wave layout).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Array arguments are DEVICE pointers to memory the caller owns and keeps
 *    alive until the work enqueued on `stream` has finished.  Nothing here
 *    allocates, frees or retains device memory; scratch space is passed in as
 *    a caller-owned workspace sized by the matching *_workspace_size() call.
 *  - moe_bf16 is the raw 16-bit pattern of a bfloat16 value.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronises the host, so a whole layer can be
 *    enqueued back to back or captured into a CUDA graph.
 *  - Arguments are validated on the host BEFORE anything is enqueued: a
 *    non-OK return means no work was launched.  MOE_ERR_CUDA means a launch
 *    itself failed (the CUDA error is left for cudaGetLastError()).
 *  - Data errors found on the device are OR-ed into *dev_status (a device
 *    uint32 the caller zeroes; may be NULL): the offending element is skipped,
 *    the kernel never traps.  Bits: MOE_DEV_*.
 *  - Row-major layouts throughout; [a,b] means b is contiguous.
 *
 * Vocabulary follows the pages' problem statement: T tokens of width d, E
 * experts, top-k routes per token (route id r = t*k + j, slot j = 0 is the
 * best expert), capacity C, SwiGLU intermediate width I.
 *
 * Sources (page title, section):
 *  [M6.6] "M6.6 - MoE Runtime Systems: Placement, Dispatch, Kernels, and Topology"
 *  [M6.2] "M6.2 - Expert Parallelism and DeepSeek MoE: Load Balancing, Shared
 *         Experts, and Fine-Grained Routing"
 *  [POOL] "Fixed pooled-wave all-to-all for the 8-of-384 MoE"
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;
typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */
typedef int32_t moe_status;

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null pointer, negative size, k > E, ...   */
  MOE_ERR_UNSUPPORTED = 2,          /* outside the shape limits stated per call  */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < the *_workspace_size() value   */
  MOE_ERR_CUDA = 4                  /* a CUDA launch or driver call failed       */
};

enum {
  MOE_DEV_NONFINITE_LOGIT = 1u, /* a NaN logit was met; it ranked below every number */
  MOE_DEV_BAD_EXPERT_ID = 2u,   /* an expert id outside [0,E); the route was skipped */
  MOE_DEV_BAD_HEADER_ID = 4u,   /* a pool header id >= n_local that is not EMPTY     */
  MOE_DEV_BAD_ROW = 8u,         /* a map entry outside the row space; skipped        */
  MOE_DEV_TIMEOUT = 16u,        /* a bounded pipeline wait gave up; output invalid   */
  MOE_DEV_NONFINITE_INPUT = 32u, /* a NaN/Inf activation met by moe_quantize_fp8     */
  MOE_DEV_BAD_MAP = 64u          /* a moe_validate_* call found a broken invariant    */
};

#define MOE_POOL_EMPTY 0xFFFFu /* header element of an unused pool row */
#define MOE_ROUTE_MASKED (-1)  /* topk_ids of a masked padding slot of a token bucket */

/* Library version (major*10000 + minor*100 + patch) and a status message. */
int32_t moe_version(void);
const char* moe_status_string(moe_status s);

/* ------------------------------------------------------------------------ */
/* Capacity                                                                 */
/* ------------------------------------------------------------------------ */
/* ceil(cf * assignments / slots) with cf = cf_num / cf_den, in exact integer
 * arithmetic.  [M6.2] 0x01C: per-expert capacity C = ceil(c_f * T*k / E)
 * (slots = E).  [POOL] 04: sender pool rows ceil(1.10 * 524288 / 64 / 3) and
 * receiver rows ceil(1.15 * 524288 / 6 / 3) (slots = n_dest*n_waves and
 * n_local*n_waves).  Returns -1 on a non-positive denominator or overflow.  */
int64_t moe_capacity(int64_t cf_num, int64_t cf_den, int64_t assignments, int64_t slots);

/* ------------------------------------------------------------------------ */
/* Route                                                                    */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t T, E, k;
  int32_t score_fn;   /* MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID_GROUP           */
  int32_t n_group;    /* sigmoid_group: contiguous logical groups (E % n_group == 0) */
  int32_t topk_group; /* sigmoid_group: groups kept before the expert top-k     */
  float route_scale;  /* sigmoid_group: gates sum to route_scale                */
} moe_route_params;

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID_GROUP = 1 };

/* Top-k routing of fp32 logits [T,E] -> topk_ids int32 [T,k], gates fp32 [T,k].
 *
 * MOE_SCORE_SOFTMAX ([M6.2] 0x06L1, Mixtral row): the k largest logits, slot 0
 * the largest, ties to the lower expert index; gate_j = exp(z_j - z_max) /
 * sum over the selected exp(z_i - z_max), i.e. the selected softmax
 * probabilities renormalised to one.  sel_bias must be NULL.
 *
 * MOE_SCORE_SIGMOID_GROUP ([M6.2] 0x06A-0x06D, 0x06I, DeepSeek-V3): s =
 * sigmoid(z) computed by a fixed fp32 recipe (see moe_sigmoid_det), corrected
 * score s~ = s + sel_bias[e] (sel_bias fp32 [E] or NULL = 0); group score =
 * sum of the two largest s~ in each of n_group contiguous groups; the
 * topk_group best groups stay eligible; the top-k experts by s~ among them are
 * selected; gate = route_scale * s_e / sum of s over the selected.  Ties to
 * the lower expert / group index.
 *
 * Limits (MOE_ERR_UNSUPPORTED): 1 <= E <= 512, 1 <= k <= min(E, 16); for
 * sigmoid_group also n_group <= 32, E/n_group >= 2, topk_group*E/n_group >= k.
 * NaN logits set MOE_DEV_NONFINITE_LOGIT and rank below every number.      */
moe_status moe_route(const moe_route_params* p, const float* logits, const float* sel_bias,
                     int32_t* topk_ids, float* gates, uint32_t* dev_status, moe_stream_t stream);

/* s[i] = sigmoid(z[i]) by the router's fixed fp32 recipe: e^x from a
 * Cody-Waite reduction (ln2 split at 16 bits), a degree-7 Taylor polynomial
 * and an exponent-bit scale, x clamped to [-87, 87], every operation a single
 * correctly rounded fp32 add/sub/mul/div with no fused multiply-add.  Exposed
 * so that its bit pattern can be checked over all inputs.                   */
moe_status moe_sigmoid_det(int64_t n, const float* z, float* s, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Permute: admission, count, prefix, stable scatter, row gather            */
/* ------------------------------------------------------------------------ */
/* [M6.2] 0x03B "Count, Prefix, Permute" and [M6.6] 0x03B.  Route r = t*k + j
 * goes to expert topk_ids[r]; it is ACCEPTED iff fewer than `capacity`
 * earlier routes (in route id order) chose the same expert (capacity < 0:
 * dropless).  Outputs:
 *   counts[E]          accepted routes per expert (c_e),
 *   offsets[E+1]       o_0 = 0, o_{e+1} = o_e + c_e (sentinel = accepted total),
 *   row_to_route[R]    rows [0, offsets[E]) hold accepted route ids ordered by
 *                      (expert, route id) -- the permutation pi; the rest of
 *                      the array is left untouched,
 *   route_to_row[R]    the inverse: row of route r, or -1 if r was dropped,
 *   n_dropped[1]       R - accepted,
 *   x_perm[R,d]        x_perm[row] = x[token of row_to_route[row]] (bit copy);
 *                      rows >= offsets[E] are left untouched.
 * x is [T,d].  x and x_perm may both be NULL: then only the maps, counts,
 * offsets and n_dropped are produced and no row is copied (for
 * moe_grouped_gate_up_gather, which reads the rows from token order itself).
 * Workspace: moe_permute_workspace_size(T,k,E) bytes.
 * Limits: 1 <= E <= 512, 1 <= k <= 16, 0 <= T, T*k < 2^31, d % 8 == 0,
 * 16-byte aligned x / x_perm.  Out-of-range ids set MOE_DEV_BAD_EXPERT_ID and
 * the route is treated as dropped.                                          */
size_t moe_permute_workspace_size(int32_t T, int32_t k, int32_t E);
moe_status moe_permute(int32_t T, int32_t d, int32_t E, int32_t k, int32_t capacity,
                       const int32_t* topk_ids, const moe_bf16* x, moe_bf16* x_perm,
                       int32_t* counts, int32_t* offsets, int32_t* row_to_route,
                       int32_t* route_to_row, int32_t* n_dropped, void* ws, size_t ws_bytes,
                       uint32_t* dev_status, moe_stream_t stream);

/* moe_permute for callers that cannot allocate device memory.  The pages have
 * no counterpart to this call: it exists for code that must not call
 * cudaMalloc and has no workspace to lend -- for example an inference
 * runtime's plugin hook that may only enqueue on the stream it is handed, or a
 * latency-critical loop where an allocation could synchronise the device.
 * Same arguments, outputs, limits and errors as moe_permute minus the
 * workspace: the per-tile histogram lives in a 64 KiB file-scope device array
 * of the library, which every GPU that loads the library holds until the
 * process exits.  Sizes whose moe_permute_workspace_size(T,k,E) exceeds 64 KiB
 * are rejected with MOE_ERR_UNSUPPORTED before anything is enqueued: beyond
 * 63,488 routes T*k for E = 512, 129,024 for E = 256, 260,096 for E = 128;
 * up to E = 127 every size fits.  Nothing is allocated or freed.
 * The first call on a device looks up the array's device address for that
 * device (cudaGetSymbolAddress, with the device current); make that first call
 * before any stream capture.  The address is kept for the life of the process:
 * after cudaDeviceReset (which unloads the library's module on that device) this
 * call must not be used again in the same process.  Every call on a device shares the one array and
 * it keeps the last call's contents (each call overwrites every entry it reads
 * before reading it, so nothing needs clearing).  Calls whose work overlaps on
 * the GPU -- other streams, other host threads -- race on the array: serialise
 * them.                                                                     */
moe_status moe_permute_noalloc(int32_t T, int32_t d, int32_t E, int32_t k, int32_t capacity,
                               const int32_t* topk_ids, const moe_bf16* x, moe_bf16* x_perm,
                               int32_t* counts, int32_t* offsets, int32_t* row_to_route,
                               int32_t* route_to_row, int32_t* n_dropped, uint32_t* dev_status,
                               moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Grouped SwiGLU expert GEMM over ragged row segments                      */
/* ------------------------------------------------------------------------ */
/* [M6.6] 0x04A and 0x04C "Variable Grouped GEMM": for every segment q with
 * rows [b, b+c), b = seg_begin[q], c = seg_count[q] (device arrays, read on the
 * device -- no host synchronisation):
 *   G = X_q W_gate[q],  U = X_q W_up[q]        (bf16 in, fp32 accumulate)
 *   H = bf16( SiLU(G) * U )                      (stored bf16, round to nearest even)
 *   y[b:b+c] = bf16( H W_down[q] )
 * with x, y [max_rows, d], W_gate / W_up [n_seg, d, I], W_down [n_seg, I, d].
 * Only segment rows of y are written.  Segments may be empty and need not be
 * contiguous, but must not overlap and must lie in [0, max_rows).  Runs on the
 * 5th-generation tensor cores (tcgen05, accumulators in tensor memory, operands
 * staged by TMA).
 * Workspace: moe_grouped_swiglu_workspace_size(max_rows, I) bytes; after the
 * stream reaches this call's end its first max_rows*I*2 bytes hold H in the
 * same row space as x.
 * Limits: d % 64 == 0, I % 64 == 0, d, I <= 65536, n_seg <= 1024; pointers
 * 16-byte aligned; n_seg >= 1.  Rows outside [0,max_rows) in a segment set
 * MOE_DEV_BAD_ROW and that segment is skipped.                              */
size_t moe_grouped_swiglu_workspace_size(int32_t max_rows, int32_t I);
moe_status moe_grouped_swiglu(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                              const moe_bf16* x, const int32_t* seg_begin,
                              const int32_t* seg_count, const moe_bf16* w_gate,
                              const moe_bf16* w_up, const moe_bf16* w_down, moe_bf16* y,
                              void* ws, size_t ws_bytes, uint32_t* dev_status,
                              moe_stream_t stream);

/* The two passes of moe_grouped_swiglu as separate calls (same segment rules,
 * limits and device-side error reporting; no workspace):
 *   moe_grouped_gate_up: h[b:b+c] = bf16(SiLU(X_q W_gate[q]) * (X_q W_up[q]))
 *                        x [max_rows, d], h [max_rows, I]   ([M6.6] 0x04C, "gate/up")
 *   moe_grouped_down:    y[b:b+c] = bf16(H_q W_down[q])
 *                        h [max_rows, I], y [max_rows, d]   ([M6.6] 0x04C, "down")  */
moe_status moe_grouped_gate_up(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                               const moe_bf16* x, const int32_t* seg_begin,
                               const int32_t* seg_count, const moe_bf16* w_gate,
                               const moe_bf16* w_up, moe_bf16* h, uint32_t* dev_status,
                               moe_stream_t stream);
/* moe_grouped_gate_up whose A rows are gathered from token order inside the
 * pass instead of read from a permuted copy: row i of the expert row space is
 * x[row_to_route[i] / k] of the token rows x [T, d] -- exactly the row
 * moe_permute copies to x_perm[i] -- so with moe_permute's row_to_route, counts
 * and offsets as the segment table h is bit-identical to moe_grouped_gate_up on
 * moe_permute's x_perm, and the permuted rows are never written to or read back
 * from HBM.  The loader issues one TMA gather per four rows: the permutation
 * of [M6.6] 0x03B is applied as a map of rows inside the pass rather than as a
 * copy.  Only row_to_route entries of rows inside segments are read; one
 * outside [0, T*k) sets MOE_DEV_BAD_ROW and that row reads token 0.  Limits
 * and errors as moe_grouped_gate_up, plus T*k < 2^31.                        */
moe_status moe_grouped_gate_up_gather(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                                      int32_t T, int32_t k, const moe_bf16* x,
                                      const int32_t* row_to_route, const int32_t* seg_begin,
                                      const int32_t* seg_count, const moe_bf16* w_gate,
                                      const moe_bf16* w_up, moe_bf16* h, uint32_t* dev_status,
                                      moe_stream_t stream);
moe_status moe_grouped_down(int32_t n_seg, int32_t I, int32_t d, int32_t max_rows,
                            const moe_bf16* h, const int32_t* seg_begin, const int32_t* seg_count,
                            const moe_bf16* w_down, moe_bf16* y, uint32_t* dev_status,
                            moe_stream_t stream);
/* moe_grouped_down for a call that directly follows this library's
 * moe_grouped_gate_up (or _gate_up_fp8 / _gate_up_gather) on the same stream,
 * with the same seg_begin / seg_count, and with h that pass's output.  It
 * computes the same y, bit for bit.  The gate/up pass lets the next kernel
 * launch early.  This call then reads the segment table and stages its first
 * tile's W_down atoms before that pass has finished.  It waits for the pass only
 * before its first read of h.  Precondition: nothing the gate/up pass or a kernel
 * enqueued after it writes seg_begin, seg_count or W_down.  If the precondition
 * is broken, the result is undefined.  The kernel still reads and writes only
 * inside the bounds the segment checks allow.  moe_grouped_swiglu issues its
 * down pass this way.  Arguments, limits and errors as moe_grouped_down.      */
moe_status moe_grouped_down_chained(int32_t n_seg, int32_t I, int32_t d, int32_t max_rows,
                                    const moe_bf16* h, const int32_t* seg_begin,
                                    const int32_t* seg_count, const moe_bf16* w_down,
                                    moe_bf16* y, uint32_t* dev_status, moe_stream_t stream);

/* Both passes of moe_grouped_swiglu in one persistent launch ([M6.6] 0x04C:
 * the gate/up pass, then the down pass, over the same segment table), for
 * decode-sized batches: h[b:b+c] as moe_grouped_gate_up, then y[b:b+c] as
 * moe_grouped_down on that h, bit for bit.  The units are the gate/up tiles,
 * then the down tiles, dealt to one CTA per SM; a down tile loads its W_down
 * atoms at once and waits (bounded) only before reading its h rows, until every
 * gate/up tile of its segment has stored them, so the weights of the two passes
 * stream back to back.  Taken when moe_grouped_swiglu_onepass_taken says so
 * (row boxes of at most 32 rows, d and I multiples of 128, and the two-launch
 * gate/up pass would take its narrow tiles too); otherwise this call issues
 * moe_grouped_gate_up and moe_grouped_down_chained and does not touch sync.
 * sync: int32 [2 * n_seg] device scratch, caller-owned, all zero before the
 * first call on it; every call that completes leaves it all zero again.  Calls
 * that overlap on the GPU must not share it.  After a MOE_DEV_TIMEOUT report its
 * contents are undefined: zero it before reuse.
 * Residency: the down tiles' waits end once every CTA of the launch has reached
 * an SM.  A kernel running beside it on another stream only delays that until it
 * ends; but a second launch of this call on another stream at the same time
 * (its units also dealt to CTAs in advance) can hold the SMs this one needs while
 * it waits in turn, and a wait then gives up with MOE_DEV_TIMEOUT (outputs
 * invalid).  Order such calls on one stream or by events.
 * h [max_rows, I] and y [max_rows, d] are outputs (only segment rows written).
 * Limits and errors as moe_grouped_gate_up and moe_grouped_down; sync 4-byte
 * aligned.                                                                 */
int32_t moe_grouped_swiglu_onepass_taken(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows);
moe_status moe_grouped_swiglu_onepass(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                                      const moe_bf16* x, const int32_t* seg_begin,
                                      const int32_t* seg_count, const moe_bf16* w_gate,
                                      const moe_bf16* w_up, const moe_bf16* w_down, moe_bf16* h,
                                      moe_bf16* y, int32_t* sync, uint32_t* dev_status,
                                      moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Combine                                                                  */
/* ------------------------------------------------------------------------ */
/* [M6.6] 0x03C3 and 0x0CD, [M6.2] 0x03C: weighted scatter-add back to token
 * order, gate applied exactly once and after the expert ([M6.6] 0x0AE), fp32
 * token accumulation:
 *   out[t] = (accumulate ? out[t] : 0)
 *            + sum_{j=0..k-1, route_to_row[t*k+j] >= 0} gates[t*k+j] * y[route_to_row[t*k+j]]
 *            + (shared_y ? shared_y[t] : 0)
 * summed in slot order in fp32.  Dropped routes contribute nothing and the
 * remaining gates are not renormalised.  y is [y_rows, d] bf16, shared_y
 * [T,d] bf16 or NULL, out [T,d] fp32.  Limits: d % 8 == 0, k <= 16.  Rows
 * >= y_rows set MOE_DEV_BAD_ROW and are skipped.                            */
moe_status moe_combine(int32_t T, int32_t k, int32_t d, const moe_bf16* y, int64_t y_rows,
                       const int32_t* route_to_row, const float* gates,
                       const moe_bf16* shared_y, int32_t accumulate, float* out,
                       uint32_t* dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* One-launch layer for small batches (decode)                              */
/* ------------------------------------------------------------------------ */
/* The whole layer -- moe_route, moe_permute, moe_grouped_swiglu and
 * moe_combine of [M6.6] 0x03-0x04 and 0x0AE -- as ONE kernel launch, for
 * decode-sized batches (at most 64 routes).  At that size the step is a stream
 * of the touched experts' weights ([M6.6] 0x05: decode is latency-bound), so one
 * launch whose every SM streams weights replaces six dependent kernels.
 * Arguments and outputs are those of the four calls, with:
 *   p            router parameters (p->T tokens; either score function);
 *   capacity     per-expert capacity, -1 for dropless (admission in route-id
 *                order, as moe_permute);
 *   valid_tokens NULL, or a device int32: tokens t >= *valid_tokens are padding
 *                slots of a fixed token bucket, as moe_route_bucket /
 *                moe_permute_bucket / moe_combine_bucket treat them;
 *   x [T,d] bf16 token rows; w_gate, w_up [E,d,I], w_down [E,I,d] bf16;
 *   topk_ids, gates [T,k]; counts [E]; offsets [E+1]; row_to_route,
 *   route_to_row [T*k]; n_dropped [1] -- exactly as moe_route / moe_permute;
 *   x_perm [T*k,d] the permuted rows (may be NULL: not written);
 *   h [T*k,I] the SwiGLU intermediate, y [T*k,d] the expert rows (row space of
 *   the permutation); out [T,d] fp32, accumulate = 0, no shared expert.
 * Integer outputs are identical to those calls'.  The expert arithmetic runs on
 * CUDA cores with fp32 accumulation (a segment holds a row or two) in a fixed
 * order, so h and y can differ from the tensor-core pass by a bf16 rounding
 * where the two fp32 sums straddle a rounding boundary; out is summed in slot
 * order in fp32 exactly like moe_combine.  Results are deterministic.
 * Workspace: moe_decode_workspace_size() bytes (0 = shape unsupported; a few
 * hundred bytes of counters), owned by the caller and ZERO-FILLED before its
 * first use; every call leaves the counters zero again, so it can be reused
 * (and the call replayed from a CUDA graph) without clearing.  Two calls whose work overlaps on the GPU
 * must not share one workspace.  A bounded wait inside the kernel that gives up
 * sets MOE_DEV_TIMEOUT (outputs then invalid).  Its units are claimed from a global
 * counter by running CTAs only, so its waits end whatever else runs beside it.
 * Limits (else MOE_ERR_UNSUPPORTED): 1 <= T <= 16, T*k <= 64, T*d <= 16384,
 * I <= 2048, d % 64 == 0, I % 64 == 0, E <= 512, k <= 16; grouped routers as moe_route
 * plus (E/n_group) a multiple of ceil-to-{1,2,4,8,12,16}(E/32) spanning a power
 * of two of lanes; pointers 16-byte aligned.                                 */
size_t moe_decode_workspace_size(int32_t T, int32_t d, int32_t E, int32_t k, int32_t I);
moe_status moe_decode_layer(const moe_route_params* p, int32_t d, int32_t I, int32_t capacity,
                            const int32_t* valid_tokens, const float* logits,
                            const float* sel_bias, const moe_bf16* x, const moe_bf16* w_gate,
                            const moe_bf16* w_up, const moe_bf16* w_down, int32_t* topk_ids,
                            float* gates, int32_t* counts, int32_t* offsets,
                            int32_t* row_to_route, int32_t* route_to_row, int32_t* n_dropped,
                            moe_bf16* x_perm, moe_bf16* h, moe_bf16* y, float* out, void* ws,
                            size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Pooled-wave static-shape layout (in-memory only; no communication)       */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t n_dest;         /* destinations; expert e lives on e / local_per_dest */
  int32_t local_per_dest; /* local experts per destination (local id = e % L)   */
  int32_t n_waves;
  int32_t pool_cap;       /* payload rows per destination pool per wave         */
  int32_t wave_policy;    /* MOE_WAVE_STRIPE or MOE_WAVE_DESTMOD                */
} moe_pool_params;

enum { MOE_WAVE_STRIPE = 0, MOE_WAVE_DESTMOD = 1 };

/* Sender side of one wave ([POOL] 02-04).  Routes to destination D, taken in
 * route id order, get ordinal j_D.  MOE_WAVE_STRIPE: wave = j_D % n_waves,
 * row = j_D / n_waves.  MOE_WAVE_DESTMOD: wave = D % n_waves, row = j_D.  A
 * route of `wave` with row < pool_cap is copied to pools[D][1+row] and its
 * local id written to header element pools[D][0][row]; one with row >=
 * pool_cap is a sender drop.  pools is [n_dest, pool_cap+1, d]: row 0 is the
 * header (elements < pool_cap: local id of that payload row or MOE_POOL_EMPTY;
 * elements >= pool_cap: MOE_POOL_EMPTY), payload rows fill from 0.  Unused
 * payload rows are not written.  Outputs: route_to_poolrow[T*k] =
 * D*pool_cap + row, or -1 (not in this wave, or dropped); pool_fill[n_dest];
 * sender_drops[1] = this wave's sender drops.
 * Workspace: moe_pool_pack_workspace_size(). Limits: pool_cap <= d (the header
 * fits one row), local_per_dest <= 65534, n_dest*local_per_dest <= 512,
 * k <= 16, d % 8 == 0.                                                       */
size_t moe_pool_pack_workspace_size(const moe_pool_params* p, int32_t T, int32_t k);
moe_status moe_pool_pack(const moe_pool_params* p, int32_t T, int32_t d, int32_t k, int32_t wave,
                         const int32_t* topk_ids, const moe_bf16* x, moe_bf16* pools,
                         int32_t* route_to_poolrow, int32_t* pool_fill, int32_t* sender_drops,
                         void* ws, size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream);

/* Receiver side of one wave ([POOL] 03 "Receiver compact", 05 "Carry expert IDs
 * in-band", 07 fixed source order).  Payload rows of n_src pools shaped
 * [n_src, pool_cap+1, d] are visited in (source, row) order; a row whose
 * header id is l < n_local takes the next free row of local expert l in
 * compact [n_local, local_cap, d], or is a receiver drop once that expert holds
 * local_cap rows.  Outputs: local_counts[n_local]; poolrow_to_row[n_src*pool_cap]
 * = l*local_cap + slot, or -1; receiver_drops[1] = this wave's receiver drops.
 * Header ids >= n_local other than MOE_POOL_EMPTY set MOE_DEV_BAD_HEADER_ID
 * and the row is skipped.  Unfilled compact rows are not written.
 * Workspace: moe_pool_compact_workspace_size().  Limits as moe_pool_pack.     */
size_t moe_pool_compact_workspace_size(int32_t n_src, int32_t pool_cap, int32_t n_local);
moe_status moe_pool_compact(int32_t n_src, int32_t pool_cap, int32_t d, int32_t n_local,
                            int32_t local_cap, const moe_bf16* pools, moe_bf16* compact,
                            int32_t* local_counts, int32_t* poolrow_to_row,
                            int32_t* receiver_drops, void* ws, size_t ws_bytes,
                            uint32_t* dev_status, moe_stream_t stream);

/* moe_pool_compact with a per-receiver rotation of the source order ([POOL] 07
 * names it as a proposal, so that overflow does not always fall on the same
 * last sources): sources are visited first_source, first_source + 1, ...,
 * n_src - 1, 0, ..., first_source - 1, each from row 0 up; 0 <= first_source
 * < n_src.  poolrow_to_row stays indexed by source * pool_cap + row.
 * first_source = 0 is moe_pool_compact.                                     */
moe_status moe_pool_compact_rotated(int32_t n_src, int32_t pool_cap, int32_t d, int32_t n_local,
                                    int32_t local_cap, int32_t first_source,
                                    const moe_bf16* pools, moe_bf16* compact,
                                    int32_t* local_counts, int32_t* poolrow_to_row,
                                    int32_t* receiver_drops, void* ws, size_t ws_bytes,
                                    uint32_t* dev_status, moe_stream_t stream);

/* out[i] = a[i] < 0 ? -1 : b[a[i]] for i < n (route -> pool row -> compact row;
 * the inverse composition of [M6.6] 0x03C3).  Entries a[i] >= b_len set
 * MOE_DEV_BAD_ROW and give -1.                                               */
moe_status moe_compose_map(int64_t n, const int32_t* a, const int32_t* b, int64_t b_len,
                           int32_t* out, uint32_t* dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Fixed token bucket (decode graphs)                                       */
/* ------------------------------------------------------------------------ */
/* [M6.6] 0x05C-0x05F: a decode graph keeps stable buffers for a bucket of T
 * token slots while the number of real tokens changes on the device each step.
 * These calls are moe_route / moe_permute / moe_combine with T = the bucket
 * capacity and one more argument, valid_tokens: a DEVICE int32 read by the
 * kernels, so a captured graph can be replayed with a new count.  Slots
 * t >= *valid_tokens (clamped to [0, T]) are padding and are masked before
 * they acquire an expert identity:
 *   moe_route_bucket    writes topk_ids = MOE_ROUTE_MASKED and gates = 0 there;
 *   moe_permute_bucket  never reads their ids, neither counts, admits nor drops
 *                       their routes (n_dropped counts real routes only) and
 *                       maps them to row -1; the real routes get exactly the
 *                       rows an unbucketed moe_permute of the real tokens gives;
 *   moe_combine_bucket  writes zero output rows for them (leaves them as they
 *                       are when accumulating).
 * The capacity argument of moe_permute_bucket is fixed at capture (it is part
 * of the graph's key).  Everything else as the unbucketed calls.            */
/* moe_bucket_stage: one step's inputs into a bucket's stable buffers, in one
 * launch.  Copies logits [T, E] fp32 and x [T, d] bf16 (token-major, contiguous)
 * into rows [0, T) of logits_dst [B, E] and x_dst [B, d], and writes T to the
 * DEVICE int32 *valid_tokens.  It waits for the previous kernel on the stream, so a
 * replay of the bucket's graph that still reads the buffers has finished.  The
 * caller keeps T <= B (the bucket's slot count; the buffers are not bounds
 * checked against B).  Rows [T, B) are left as they are: the bucketed calls mask
 * them.  T = 0 only writes the count.  Limits: d % 8 == 0, x and x_dst 16-byte
 * aligned (logits use 16-byte copies when both sides are aligned).             */
moe_status moe_bucket_stage(int32_t T, int32_t E, int32_t d, const float* logits,
                            const moe_bf16* x, float* logits_dst, moe_bf16* x_dst,
                            int32_t* valid_tokens, moe_stream_t stream);
moe_status moe_route_bucket(const moe_route_params* p, const int32_t* valid_tokens,
                            const float* logits, const float* sel_bias, int32_t* topk_ids,
                            float* gates, uint32_t* dev_status, moe_stream_t stream);
moe_status moe_permute_bucket(int32_t T, int32_t d, int32_t E, int32_t k, int32_t capacity,
                              const int32_t* valid_tokens, const int32_t* topk_ids,
                              const moe_bf16* x, moe_bf16* x_perm, int32_t* counts,
                              int32_t* offsets, int32_t* row_to_route, int32_t* route_to_row,
                              int32_t* n_dropped, void* ws, size_t ws_bytes, uint32_t* dev_status,
                              moe_stream_t stream);
moe_status moe_combine_bucket(int32_t T, int32_t k, int32_t d, const int32_t* valid_tokens,
                              const moe_bf16* y, int64_t y_rows, const int32_t* route_to_row,
                              const float* gates, const moe_bf16* shared_y, int32_t accumulate,
                              float* out, uint32_t* dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Backward of the transpose                                                */
/* ------------------------------------------------------------------------ */
/* [M6.2] 0x03D "Backward Is The Reverse Semantic Transpose".  For the combine
 * out[t] = sum_j g[t,j] * y[row(t,j)] and upstream gradient dout [T,d] fp32:
 *   dy[row(t,j)] = bf16(g[t,j] * dout[t])   for every accepted route (the
 *                  expert-output gradient, in the expert-major row space of y;
 *                  rows of no accepted route are left untouched),
 *   dgates[t,j]  = <dout[t], y[row(t,j)]>  fp32 (0 for dropped routes).
 * y and dy are [y_rows, d] bf16.  Limits: d % 8 == 0, k <= 16, 16-byte aligned
 * dout / y / dy.  Rows >= y_rows set MOE_DEV_BAD_ROW and are skipped.        */
moe_status moe_combine_backward(int32_t T, int32_t k, int32_t d, const float* dout,
                                const moe_bf16* y, int64_t y_rows, const int32_t* route_to_row,
                                const float* gates, moe_bf16* dy, float* dgates,
                                uint32_t* dev_status, moe_stream_t stream);

/* Route-input gradients back to their tokens through the saved inverse map
 * ([M6.2] 0x03D, "the inverse ownership path then sums route-input gradients
 * by origin token"): dx[t] = (accumulate ? dx[t] : 0) + sum over the token's
 * accepted routes of dx_perm[route_to_row[t*k+j]], fp32, slot order.  dx_perm
 * is [rows, d] bf16, dx [T,d] fp32.  Limits and errors as moe_combine.       */
moe_status moe_unpermute_grad(int32_t T, int32_t k, int32_t d, const moe_bf16* dx_perm,
                              int64_t rows, const int32_t* route_to_row, float* dx,
                              int32_t accumulate, uint32_t* dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Load telemetry and the delayed bias controller                          */
/* ------------------------------------------------------------------------ */
/* [M6.2] 0x01I skew summaries of a count vector n[U] (int32, e.g. the per-expert
 * counts written by moe_permute): with mu = R/U, R = sum n, q = n/R, 0 log 0 = 0,
 *   stats[0] = CV^2 = mean((n - mu)^2) / mu^2      stats[1] = rho_max = max n / mu
 *   stats[2] = H_norm = -sum q log q / log U      stats[3] = E_eff = exp(-sum q log q)
 *   stats[4] = MaxVio = (max n - mu) / mu         ([M6.2] 0x06J2)
 * in fp64 (device array of 5 doubles).  All five are 0 when R = 0; H_norm is 0
 * when U = 1.  Negative counts are read as 0.                                */
moe_status moe_load_stats(int32_t U, const int32_t* counts, double* stats, moe_stream_t stream);

enum { MOE_BIAS_SIGN = 0, MOE_BIAS_PROPORTIONAL = 1 };

/* One step of the loss-free selection-bias controller ([M6.2] 0x06E, 0x06J1,
 * 0x06J3) after a batch routed with the current bias: with c = counts[E] and
 * cbar = mean(c),
 *   MOE_BIAS_SIGN:         bias[e] += u * sign(cbar - c[e])
 *   MOE_BIAS_PROPORTIONAL: bias[e] += u * (cbar - c[e])
 * in place on the fp32 bias [E]; the increment is formed in fp64 and rounded to
 * fp32 once, then added with one fp32 rounding.                              */
moe_status moe_bias_update(int32_t E, const int32_t* counts, float* bias, float u, int32_t rule,
                           moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* FP8 dispatch payload with fp32 scales                                    */
/* ------------------------------------------------------------------------ */
/* [M6.6] 0x0AB-0x0AF: a dispatched activation row may travel as FP8 data plus
 * fp32 scale metadata.  The pair belongs together: the scales are permuted with
 * their rows (same route row) and the expert dequantizes each row with its own
 * scale; scales left in token order next to expert-major rows would give finite
 * but wrong expert inputs.
 *   Format: E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 *   infinities; 0x7F / 0xFF are NaN; largest finite value 448).
 *   Scale groups: group = MOE_SCALE_ROW (0): one scale per row, G = 1;
 *   group = MOE_SCALE_BLOCK128 (128): one scale per 128 consecutive values of a
 *   row, G = ceil(d / 128), the last group shorter when 128 does not divide d.
 *   Scales are fp32 [rows, G], row-major.
 *   Quantization of a group with largest magnitude amax: s = fp32(amax / 448)
 *   (s = 1 for an all-zero group) and code = E4M3(fp32(x / s)), to nearest with
 *   ties to even, saturated to +-448.
 *   Dequantization: xhat = bf16(fp32(decode(code) * s)), the bf16 operand of the
 *   expert GEMM (one fp32 rounding of the exact product, one bf16 rounding).
 *   The NaN codes, which moe_quantize_fp8 emits only for non-finite input, are
 *   outside the contract: they dequantize to +-480 * s.                      */
typedef uint8_t moe_fp8; /* raw E4M3 byte */

enum { MOE_SCALE_ROW = 0, MOE_SCALE_BLOCK128 = 128 };
enum { MOE_PAYLOAD_BF16 = 0, MOE_PAYLOAD_FP8_ROW = 1, MOE_PAYLOAD_FP8_BLOCK128 = 2 };

/* Logical payload bytes of `rows` dispatched rows of width d ([M6.6] 0x0AB):
 * BF16 rows*d*2; FP8_ROW rows*d + rows*4; FP8_BLOCK128 rows*d + rows*ceil(d/128)*4.
 * Alignment, metadata, headers and packetization are not included.  Host
 * function; returns -1 for rows < 0, d < 1 or an unknown payload.           */
int64_t moe_payload_bytes(int64_t rows, int32_t d, int32_t payload);

/* Quantize bf16 rows x [n,d] to E4M3 codes q [n,d] and fp32 scales [n,G] as
 * above.  Limits: d % 16 == 0, 16-byte aligned x and q, group 0 or 128.  A
 * non-finite input sets MOE_DEV_NONFINITE_INPUT; that group's codes and scale
 * are then unspecified.                                                      */
moe_status moe_quantize_fp8(int64_t n, int32_t d, int32_t group, const moe_bf16* x, moe_fp8* q,
                            float* scales, uint32_t* dev_status, moe_stream_t stream);

/* x[i] = bf16(fp32(decode(q[i]) * s)) over rows [n,d]: the operand that
 * moe_grouped_gate_up_fp8 builds in shared memory, written out.  Limits as
 * moe_quantize_fp8 (x and q 16-byte aligned).                                */
moe_status moe_dequantize_fp8(int64_t n, int32_t d, int32_t group, const moe_fp8* q,
                              const float* scales, moe_bf16* x, moe_stream_t stream);

/* moe_permute with an FP8 payload ([M6.6] 0x0AC row trace): the same admission,
 * counts, offsets, row_to_route, route_to_row and n_dropped as moe_permute,
 * and for every accepted route q_perm[row] = q[token] (d bytes) and
 * scales_perm[row] = scales[token] (G floats): the payload and its scales move
 * together.  q [T,d], scales [T,G], q_perm [T*k,d], scales_perm [T*k,G]; rows
 * >= offsets[E] are left untouched.  Workspace: moe_permute_workspace_size.
 * Limits as moe_permute with d % 16 == 0 and 16-byte aligned q / q_perm.     */
moe_status moe_permute_fp8(int32_t T, int32_t d, int32_t E, int32_t k, int32_t capacity,
                           int32_t group, const int32_t* topk_ids, const moe_fp8* q,
                           const float* scales, moe_fp8* q_perm, float* scales_perm,
                           int32_t* counts, int32_t* offsets, int32_t* row_to_route,
                           int32_t* route_to_row, int32_t* n_dropped, void* ws, size_t ws_bytes,
                           uint32_t* dev_status, moe_stream_t stream);

/* moe_grouped_gate_up with an FP8 A operand: the expert input rows arrive as
 * E4M3 codes xq [max_rows, d] with fp32 scales [max_rows, G]; the kernel's
 * loader dequantizes every staged tile with the scale of its own row (and
 * 128-value group) into the bf16 operand moe_dequantize_fp8 defines, so h is
 * bit-identical to moe_grouped_gate_up on moe_dequantize_fp8's output.  Limits
 * and errors as moe_grouped_gate_up; scales 4-byte aligned.                  */
moe_status moe_grouped_gate_up_fp8(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                                   int32_t group, const moe_fp8* xq, const float* scales,
                                   const int32_t* seg_begin, const int32_t* seg_count,
                                   const moe_bf16* w_gate, const moe_bf16* w_up, moe_bf16* h,
                                   uint32_t* dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert demand and map validators                                         */
/* ------------------------------------------------------------------------ */
/* Per-expert demand before capacity ([M6.2] 0x01I: n_e, the count of routes
 * that chose expert e, the quantity the skew summaries and the bias controller
 * read; with a capacity C the admitted count is min(n_e, C)).  demand[E] int32
 * is overwritten with the histogram of topk_ids[0 .. R_live), R_live = T*k, or
 * min(*valid_tokens, T)*k when valid_tokens (a device int32) is not NULL.  Ids
 * outside [0,E) -- including MOE_ROUTE_MASKED -- are not counted; ids other
 * than MOE_ROUTE_MASKED outside [0,E) set MOE_DEV_BAD_EXPERT_ID.  Limits: 1 <=
 * E <= 512, T*k < 2^31.                                                      */
moe_status moe_expert_demand(int32_t T, int32_t k, int32_t E, const int32_t* valid_tokens,
                             const int32_t* topk_ids, int32_t* demand, uint32_t* dev_status,
                             moe_stream_t stream);

/* Debug validators ([M6.6] 0x0CD "Route And Combine Assertions": accepted +
 * dropped = routes, the counts sum to the accepted routes, one inverse entry
 * per accepted route).  Each reads outputs of the calls named and sets
 * MOE_DEV_BAD_MAP in *dev_status when an invariant below fails; nothing else is
 * written (dev_status is never cleared; workspaces are scratch).  They are meant for tests
 * and for checking a pipeline once, not for every step.
 *
 * moe_validate_permutation -- after moe_permute / moe_permute_bucket /
 * moe_permute_fp8 with the same T, E, k, capacity and valid_tokens (NULL for
 * the unbucketed calls).  [M6.2] 0x03B and [M6.6] 0x03B, 0x03C3: offsets[0] =
 * 0 and offsets[e+1] - offsets[e] = counts[e] >= 0 (capacity >= 0: <=
 * capacity); accepted + n_dropped = R_live (no drops when dropless); every row
 * i < offsets[E] holds a live route r with route_to_row[r] = i, and every
 * route r with route_to_row[r] = i >= 0 has row_to_route[i] = r inside its
 * expert's segment (the two maps are inverse bijections between the accepted
 * routes and [0, offsets[E])); route ids increase along a segment (stable
 * order); a route is dropped (-1) only when its expert holds `capacity` rows,
 * all of routes with smaller ids (admission in route id order); padding routes
 * map to -1.  Routes with ids outside [0,E) are not checked against a segment.
 *
 * moe_validate_pools -- after moe_pool_pack of one wave.  [POOL] 02-05:
 * 0 <= pool_fill[D] <= pool_cap; header element r of pool D is a local id <
 * local_per_dest for r < pool_fill[D] and MOE_POOL_EMPTY otherwise; a placed
 * route (route_to_poolrow >= 0) points at a filled row of destination
 * topk_ids / local_per_dest whose header holds topk_ids % local_per_dest; every
 * filled row is pointed at by exactly one route (conservation of placed rows).
 * Workspace: moe_validate_pools_workspace_size(p) bytes.
 *
 * moe_validate_compact -- after moe_pool_compact(_rotated) of one wave with the
 * same first_source (0 for moe_pool_compact).  [POOL] 03, 05: 0 <=
 * local_counts[l] <= local_cap; a pool row whose header id l < n_local maps to
 * -1 (a receiver drop) or to l*local_cap + slot with slot < local_counts[l];
 * every other pool row maps to -1; every compact row below its expert's count
 * is the image of exactly one pool row, slots in the receiver's visiting order;
 * receiver drops happen only to experts that are full of rows visited earlier.
 * Workspace:
 * moe_validate_compact_workspace_size(n_local, local_cap) bytes.
 *
 * Limits as the calls they check.                                           */
moe_status moe_validate_permutation(int32_t T, int32_t E, int32_t k, int32_t capacity,
                                    const int32_t* valid_tokens, const int32_t* topk_ids,
                                    const int32_t* counts, const int32_t* offsets,
                                    const int32_t* row_to_route, const int32_t* route_to_row,
                                    const int32_t* n_dropped, uint32_t* dev_status,
                                    moe_stream_t stream);
size_t moe_validate_pools_workspace_size(const moe_pool_params* p);
moe_status moe_validate_pools(const moe_pool_params* p, int32_t T, int32_t d, int32_t k,
                              const int32_t* topk_ids, const moe_bf16* pools,
                              const int32_t* route_to_poolrow, const int32_t* pool_fill, void* ws,
                              size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream);
size_t moe_validate_compact_workspace_size(int32_t n_local, int32_t local_cap);
moe_status moe_validate_compact(int32_t n_src, int32_t pool_cap, int32_t d, int32_t n_local,
                                int32_t local_cap, int32_t first_source, const moe_bf16* pools,
                                const int32_t* local_counts, const int32_t* poolrow_to_row,
                                void* ws, size_t ws_bytes, uint32_t* dev_status,
                                moe_stream_t stream);

/* Self-test of the bounded pipeline wait used by the tensor-core kernels: one
 * CTA initialises an mbarrier that nothing arrives at and waits on it with the
 * same bounded-wait routine, giving up after limit_ns nanoseconds of global
 * time (1 <= limit_ns <= 10^9); it then sets MOE_DEV_TIMEOUT and returns.  The
 * kernel never traps and leaves the context usable.                          */
moe_status moe_debug_wait_timeout(int64_t limit_ns, uint32_t* dev_status, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
