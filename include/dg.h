/*
 * dg.h -- libdecodegemm: decode-time skinny linear layers on GB300 (sm_103a).
 *
 * One C ABI for the operations a decode step runs against large weight
 * matrices with few token rows (M = 1..128; the bf16 linear and gate/up also
 * take the mid-M range 129..512):
 *
 *   dg_gemv_bf16        y = x . W^T, bf16 weights, bf16 out
 *   dg_gate_up_silu     out = silu(x . W_gate^T) * (x . W_up^T), one launch
 *   dg_head_fp8_argmax  fp8-e4m3 vocabulary head with one per-tensor scale,
 *                       greedy (temperature 0) argmax fused into the same launch
 *   dg_moe_w1_silu      routed-expert W1 (gate+up) with SiLU.mul, N-split
 *   dg_moe_w2           routed-expert W2 with the gate-weighted combine, N-split
 *   dg_gemv_a8w8_blockscale
 *                       e4m3 weights with 128 x 128 block scales, the per-(token,
 *                       128-block) activation quantisation fused in (M <= 64)
 *
 * plus dg_select, which maps (op, M, N, K) to a kernel variant through a
 * per-device shape table written by an on-device sweep (dg_sweep), and a
 * process-wide numerics mode (dg_set_numerics) that can make every row's result
 * independent of the batch it is computed in.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers, row-major, densely packed, owned
 *   by the caller.  bf16 values travel as their 16-bit patterns, e4m3 values as
 *   their 8-bit codes (OCP 8-bit float E4M3, "fn" variant: no infinities,
 *   S.1111.111 is NaN, largest magnitude 448).
 * - Every pointer must be 16-byte aligned and K must be a multiple of 8
 *   (bf16 weights) or 16 (e4m3 weights); otherwise DG_ERR_ALIGNMENT /
 *   DG_ERR_UNSUPPORTED_SHAPE is returned before anything is launched.
 * - Calls are asynchronous on `stream` and make no host synchronisation.
 *   Argument errors are returned synchronously and launch nothing.
 * - `ws` is a caller-owned device workspace of at least
 *   dg_workspace_bytes(op, ...) bytes.  It must be zero-filled once when it is
 *   allocated (e.g. cudaMemsetAsync); every call leaves its counters at zero
 *   again (a grid barrier's generation word keeps counting; any value is fine).
 *   Calls that share one workspace must be ordered on one stream.  After a
 *   DG_DEVERR_WAIT_TIMEOUT the workspace must be zero-filled again, and the
 *   outputs of the call that set it are not valid (where a grid-wide combine
 *   gave up, the tensor-core MoE W2 writes NaN rather than leave older values).
 *   The first 16 bytes hold a sticky device status word (dg_device_status).
 * - `choice` may be NULL (dg_select picks); otherwise the given variant runs.
 * - Accumulation is fp32 in a fixed order that does not depend on the kernel
 *   variant, the launch geometry or the run: every variant dg_select can pick
 *   for one (op, M, N, K) gives bitwise identical outputs.
 * - The library allocates no device memory.  It keeps host-side state only:
 *   per-device properties and the loaded shape table.
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* dg_stream_t;

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1,         /* null pointer, negative or zero size, bad topk/E */
    DG_ERR_ALIGNMENT = 2,           /* a pointer is not 16-byte aligned */
    DG_ERR_UNSUPPORTED_SHAPE = 3,   /* K not a multiple of the vector width, M too large, ... */
    DG_ERR_WORKSPACE_TOO_SMALL = 4,
    DG_ERR_CUDA = 5,                /* a CUDA runtime call or a launch failed */
    DG_ERR_TABLE_REFUSED = 6,       /* a shape table failed its identity or knob checks */
    DG_ERR_NO_DEVICE = 7,           /* no usable sm_103 device is current */
    DG_ERR_BAD_VARIANT = 8          /* a dg_choice names a variant or params this op lacks */
} dg_status;

typedef enum {
    DG_OP_GEMV_BF16 = 0,
    DG_OP_GATE_UP_SILU = 1,
    DG_OP_HEAD_FP8_ARGMAX = 2,
    DG_OP_MOE_W1 = 3,
    DG_OP_MOE_W2 = 4,
    DG_OP_GEMV_A8W8 = 5,
    DG_OP_COUNT = 6
} dg_op;

/* Kernel families.  One family serves one (op, M) bucket; variants inside a
 * family differ only in launch geometry and staging, never in arithmetic. */
typedef enum {
    DG_VAR_DEFAULT = 0,      /* let the library choose (same as choice == NULL) */
    DG_VAR_CC_WARP = 1,      /* CUDA cores, each warp streams R weight rows through registers */
    DG_VAR_CC_BULK = 2,      /* CUDA cores, bulk-async (TMA) copies stage weight rows in shared memory */
    DG_VAR_TC = 3,           /* tcgen05 tensor cores, TMA tiles, TMEM accumulators */
    DG_VAR_MMA = 4           /* warp-level tensor cores (mma.sync), weights streamed through registers */
} dg_variant;

/* params[] meaning by variant:
 *   DG_VAR_CC_WARP: [0] rows per warp R (1, 2, 4, 8), [1] warps per CTA (1..8),
 *                   [2] CTAs per SM cap (0 = occupancy limit), [3] dense ops: warps
 *                   sharing one row group's K segments (1, 2, 4, 8 dividing [1];
 *                   0 = 1) -- the segment partials are folded in the same order
 *   DG_VAR_CC_BULK: [0] 0, [1] pipeline stages (0 = as many as fit), [2] CTAs per SM (0 = 1)
 *   DG_VAR_MMA:     bf16 linear and gate/up, 1..16 rows: [0] warps sharing one 16-row
 *                   group's 512-element K segments (1, 2, 4, 8; 0 = derived), [1] warps per
 *                   CTA (4 or 8; 0 = derived), [2] CTAs per SM cap (0 = occupancy limit),
 *                   [3] 32-element chunks per load round (2, 4, 8; 0 = 8 up to 8 rows,
 *                   4 above)
 *   DG_VAR_TC:      [0] pipeline stages (0 = derived from the shape); bf16 linear and
 *                   gate/up: [1] K-split rule, 0 = sized by the shape and the row
 *                   count, 1 = by the shape alone, on a given device (the
 *                   batch-invariant mode's choice;
 *                   the two agree up to 128 rows); A8W8: [1] 1 = quantise the activations
 *                   in a launch of its own into the workspace and stream the codes by TMA
 *                   (0 = the quantisation fused into the tensor-core kernel; same bits)
 * For the MoE ops (DG_VAR_CC_WARP), params[5] is the work order: 0 or 1 = persistent
 * CTAs walk (active expert, N-tile) units, params[3] the N-tile width in rows (0 =
 * derived); 2 = each CTA owns one contiguous row range of every active expert (W2:
 * output rows, folded over the slots inside the CTA; W1: an even share of the
 * (expert, column pair) list), params[1] warps per CTA 4 or 8, params[2] CTAs per SM
 * (0 = the occupancy limit, at most 4), params[3] 0; W2 in this order keeps all M *
 * topk activation rows in shared memory (M * topk * I * 2 bytes, at most 200 KiB, else
 * DG_ERR_UNSUPPORTED_SHAPE).  params[4] is, in both orders, the most
 * (token, slot) pairs of one expert per pass over its rows (1, 2, 4 or 8; 0 = 2).
 * Both orders give the same bits. */
typedef struct {
    int32_t variant;
    int32_t params[6];
    int32_t from_table;      /* 1 when the choice came from a loaded shape table */
    float table_us;          /* the table's measured time for this choice, else 0 */
} dg_choice;

/* Device status word values (sticky, OR-ed bits). */
#define DG_DEVERR_BAD_TOPK_ID 0x1   /* a topk id was out of range or repeated in its row */
#define DG_DEVERR_WAIT_TIMEOUT 0x2  /* a bounded pipeline wait gave up */

/* ---------------------------------------------------------------- setup */

/* Prepare the library for `device` (makes it current): checks for compute
 * capability 10.3 and caches its properties, then loads the table named by
 * the DG_TABLE environment variable, if any.  A refused table prints one line
 * to stderr and leaves the compiled defaults in effect (the call still returns
 * DG_OK).  Entry points call this lazily for the current device. */
dg_status dg_init(int device);

/* Human-readable name of a status code (static storage). */
const char* dg_status_str(dg_status s);

/* Workspace bytes an entry point needs.  N, K, topk by op:
 *   GEMV_BF16:       N rows of W, K
 *   GATE_UP_SILU:    N = N_half (output columns), K
 *   HEAD_FP8_ARGMAX: N = vocabulary rows, K
 *   MOE_W1:          N = I (expert intermediate), K = hidden, topk
 *   MOE_W2:          N = Nout (hidden), K = I, topk
 * Always >= 16 (the device status word). */
size_t dg_workspace_bytes(dg_op op, int M, int N, int K, int topk);

/* Copy the workspace's device status word to *host_out (synchronises `stream`;
 * meant for tests and health checks, not the decode loop). */
dg_status dg_device_status(const void* ws, int32_t* host_out, dg_stream_t stream);

/* Launch flags (process-wide).  DG_LAUNCH_PDL (on by default): every kernel is
 * launched with programmatic dependent launch, so it can be scheduled while the
 * preceding kernel on the stream finishes; before waiting for that kernel it
 * touches nothing but weights (streams them into L2 or shared memory), which this
 * library never writes.  A preceding kernel that does not signal early (any
 * kernel not from this library) still completes before this one starts its
 * dependent work.  Turn it off when a kernel of this library must wait for a
 * preceding launch that writes the weights it reads.
 * "Decode optimization round 3", "Profiling" / "Remaining headroom": decode steps
 * are bound by per-kernel launch latency, not bandwidth. */
#define DG_LAUNCH_PDL 0x1u
dg_status dg_set_launch_flags(unsigned flags);
unsigned dg_launch_flags(void);

/* Numerics mode (process-wide); it steers dg_select, and so every call made with a
 * NULL choice.
 *   DG_NUMERICS_FASTEST (default): each row bucket takes its fastest kernel family.
 *     The CUDA-core families (1 row for the bf16 linear, 1-2 for gate/up), the
 *     warp-level tensor-core family (2-12 and 3-8 rows) and the tcgen05 families
 *     reduce in different orders, so a row's bits can change when the same row is
 *     computed inside a larger batch (all meet the same error bound).
 *   DG_NUMERICS_BATCH_INVARIANT: every bucket of an op takes one family (the
 *     tensor cores; the fp8 head with K > 8192 the CUDA cores), so output row m is
 *     a function of input row m alone -- for the MoE ops, of token m's activations,
 *     ids and gate weights -- whatever M is and whatever the other rows hold.  A
 *     one-row draft pass and a many-row verify pass then give the same logits and
 *     the same argmax for the same row.  Table picks from another family are
 *     ignored in this mode; an explicit choice passed to a call is used as given.
 * The pages ask for bitwise-equal results per shape only (Strata PR #1297,
 * "Summary"; "Decode optimization round 3", "Validation"); this mode extends the
 * guarantee across row counts at the cost of the CUDA-core and warp-level speed
 * at 1-12 rows. */
#define DG_NUMERICS_FASTEST 0
#define DG_NUMERICS_BATCH_INVARIANT 1
dg_status dg_set_numerics(int mode);   /* DG_ERR_INVALID_ARG for an unknown mode */
int dg_numerics(void);

/* Clear the device status word (asynchronous on `stream`). */
dg_status dg_device_status_clear(void* ws, dg_stream_t stream);

/* Health check of the bounded waits (no counterpart on the pages): one CTA waits on a barrier that never completes, gives up
 * after timeout_us (1 .. 2,000,000) and sets DG_DEVERR_WAIT_TIMEOUT in the
 * workspace status word -- the same path every pipelined kernel takes when a wait
 * runs out.  Asynchronous on `stream`; the context stays usable. */
dg_status dg_selftest_wait_timeout(void* ws, int timeout_us, dg_stream_t stream);

/* Test export of the MoE routing step ("Decode optimization round 3", Retained
 * change 1: the active experts and their (token, slot) pairs): one CTA runs the
 * routing scan the MoE kernels run and writes, into the caller's device buffer
 * `out` of DG_ROUTE_DEBUG_INTS int32 (asynchronously on `stream`):
 *   [0] U active experts, [1] P valid pairs,
 *   [2 .. 2+128)          valid[t*topk + k] (1/0; 0 past M*topk),
 *   then 16               valid slots per token (0 past M),
 *   then 128              active experts ascending (-1 past U),
 *   then 129              pair offsets of each active expert, offs[U] = P (-1 past U),
 *   then 128 + 128        pair token / pair slot, by expert then token then slot (-1 past P).
 * topk_ids [M, topk] int32 device; 1 <= M <= 16, 1 <= topk <= 8, 1 <= E <= 1024;
 * ws a zero-filled workspace (its status word gets DG_DEVERR_BAD_TOPK_ID for
 * invalid slots).  Argument errors return before any launch. */
#define DG_ROUTE_DEBUG_INTS (2 + 128 + 16 + 128 + 129 + 128 + 128)
dg_status dg_moe_route_debug(const int32_t* topk_ids, int M, int topk, int E, int32_t* out, void* ws,
                             dg_stream_t stream);

/* ---------------------------------------------------------------- compute */

/* Decode linear, mstar PR #1104 (decode GEMM table), "Why" / "What changed":
 *   y[m, n] = bf16_rn( sum_k x[m, k] * W[n, k] )   fp32 accumulation
 * x [M, K] bf16, W [N, K] bf16, y [M, N] bf16.  1 <= M <= 512. */
dg_status dg_gemv_bf16(const void* x, const void* W, void* y, int M, int N, int K,
                       void* ws, size_t ws_bytes, dg_stream_t stream, const dg_choice* choice);

/* Fused gate/up projection with SiLU.mul, mstar PR #1104, "What changed"
 * (the fused gate/up entry):
 *   g = sum_k x[m,k] * W_gu[2j, k],  u = sum_k x[m,k] * W_gu[2j+1, k]   (fp32)
 *   out[m, j] = bf16_rn( silu(g) * u ),  silu(g) = g / (1 + exp(-g))     (fp32)
 * W_gu [2*N_half, K] bf16 stores gate row j at row 2j and up row j at 2j+1.
 * out [M, N_half] bf16.  1 <= M <= 512. */
dg_status dg_gate_up_silu(const void* x, const void* W_gu, void* out, int M, int N_half, int K,
                          void* ws, size_t ws_bytes, dg_stream_t stream, const dg_choice* choice);

/* fp8 vocabulary head with greedy pick, mstar PR #1102 (fused draft step and
 * fp8 draft head), "What changed" (one scale for all of the head; the pick at
 * temperature 0 in the graph):
 *   acc[m, n]   = sum_k x[m, k] * e4m3(Wq[n, k])        fp32
 *   logit[m, n] = acc[m, n] * scale                      fp32 (one multiply)
 *   logits[m,n] = bf16_rn(logit)                          (skipped if logits == NULL)
 *   argmax[m]   = lowest n with the largest fp32 logit; NaN is never picked
 *                 (a row of only NaN gives -1)
 * x [M, K] bf16, Wq [N, K] e4m3 codes, scale: device pointer to one fp32,
 * logits [M, N] bf16 or NULL, argmax [M] int32.  1 <= M <= 8.
 * The CUDA-core kernels (one row, or K > 8192) stage every row's activations in
 * shared memory: there M * K <= 49,152, else DG_ERR_UNSUPPORTED_SHAPE.
 * The argmax buffer is sized by this call's M. */
dg_status dg_head_fp8_argmax(const void* x, const void* Wq, const float* scale, void* logits,
                             int32_t* argmax, int M, int N, int K, void* ws, size_t ws_bytes,
                             dg_stream_t stream, const dg_choice* choice);

/* The same head and pick for callers that cannot allocate device memory (no
 * counterpart on the pages).  Engines whose device memory pool belongs to someone
 * else, plugins whose host forbids device allocation, or code that runs after its
 * memory budget is fixed cannot hand over a workspace; this entry point keeps the
 * scratch (status word, pick ticket, per-CTA partials) in a static device array of
 * 294,912 bytes inside the library instead, held by every GPU that loads the
 * library until the process exits.  It calls no allocator.
 * - Arguments and results as dg_head_fp8_argmax, without ws / ws_bytes.
 * - The first call on a device looks up the array's device address (with that
 *   device current); make that first call before any stream capture.
 * - Every check of the call runs first (the same code as dg_head_fp8_argmax): a
 *   refused call queues nothing.  An accepted call clears the status word and ticket
 *   with an asynchronous memset on `stream`, then launches.
 * - All calls share the one array: calls that may overlap on the GPU (different
 *   streams, or different host threads) race and must be serialised by the caller.
 *   The status word therefore describes the latest call only; read it with
 *   dg_head_fp8_argmax_noalloc_status before the next call clears it.
 * - A launch that would need more than 4096 CTA partial slots is rejected with
 *   DG_ERR_WORKSPACE_TOO_SMALL and one stderr line (no grid this library launches for
 *   the head on a 152-SM part comes near it). */
dg_status dg_head_fp8_argmax_noalloc(const void* x, const void* Wq, const float* scale, void* logits,
                                     int32_t* argmax, int M, int N, int K, dg_stream_t stream,
                                     const dg_choice* choice);

/* The device status word of the no-allocation head's static scratch, i.e. of its
 * latest call (DG_DEVERR_* bits; a bounded wait that gave up shows as
 * DG_DEVERR_WAIT_TIMEOUT): copied to *host_out after synchronising `stream`.  For
 * health checks, like dg_device_status (no counterpart on the pages). */
dg_status dg_head_fp8_argmax_noalloc_status(int32_t* host_out, dg_stream_t stream);

/* The static scratch's device address on the current device (a health-check hook,
 * e.g. to run dg_selftest_wait_timeout on it; no counterpart on the pages).  Looks
 * the address up on first use, like the first call of the no-allocation head. */
dg_status dg_head_fp8_argmax_noalloc_scratch(void** device_ptr);

/* Routed-expert W1 with SiLU.mul, "Decode optimization round 3", "Retained
 * change 1: N-split W1/W2 MoE kernels" (experts split along N at small M).
 * A slot (t, k) is valid when 0 <= topk_ids[t, k] < E and no earlier slot of
 * token t names the same expert.  For each valid slot, e = topk_ids[t, k]:
 *   g = s1[e, j]     * sum_i x[t, i] * e4m3(W1[e, j, i])        fp32
 *   u = s1[e, I + j] * sum_i x[t, i] * e4m3(W1[e, I + j, i])    fp32
 *   a[t, k, j] = bf16_rn( silu(g) * u )
 * Invalid slots write a = 0 and set DG_DEVERR_BAD_TOPK_ID in the status word.
 * x [M, K] bf16, topk_ids [M, topk] int32, W1 [E, 2I, K] e4m3 (gate rows
 * 0..I-1, up rows I..2I-1), s1 [E, 2I] fp32, a [M, topk, I] bf16.
 * 1 <= M <= 16, 1 <= topk <= 8. */
dg_status dg_moe_w1_silu(const void* x, const int32_t* topk_ids, const void* W1, const float* s1,
                         void* a, int M, int topk, int E, int I, int K, void* ws, size_t ws_bytes,
                         dg_stream_t stream, const dg_choice* choice);

/* Routed-expert W2 with the gate-weighted combine (same page and section):
 *   h[t, k, n] = s2[e, n] * sum_i a[t, k, i] * e4m3(W2[e, n, i])  fp32, e = topk_ids[t, k]
 *   y[t, n]    = bf16_rn( sum over valid k, ascending: h[t, k, n] * gw[t, k] )  fp32
 * a [M, topk, I] bf16, topk_ids [M, topk] int32, gw [M, topk] fp32,
 * W2 [E, Nout, I] e4m3, s2 [E, Nout] fp32, y [M, Nout] bf16.
 * 1 <= M <= 16, 1 <= topk <= 8; I must be a multiple of 16. */
dg_status dg_moe_w2(const void* a, const int32_t* topk_ids, const float* gw, const void* W2,
                    const float* s2, void* y, int M, int topk, int E, int I, int Nout, void* ws,
                    size_t ws_bytes, dg_stream_t stream, const dg_choice* choice);

/* A8W8 block-scaled linear with the activation quantisation fused in as its prologue
 * ("Decode optimization round 3", "Retained change 2: decode-M rows for the A8W8
 * bpreshuffle table" -- the A8W8 blockscale GEMM at decode rows -- and "Rejected
 * paths" / "Remaining headroom" -- quantisation kernels fused into the GEMM).
 * Blocks are 128 wide along K.  Per token m and K-block b, in binary32:
 *   amax    = max(max_{k in b} |x[m, k]|, 2^-32)
 *   q[m, k] = e4m3(x[m, k] * (448 / amax))     round to nearest even, saturating
 *   sx[m,b] = amax / 448
 *   y[m, n] = bf16_rn( sum_b  P_b * (sx[m, b] * sw[n / 128, b]) ),
 *             P_b = sum_{k in b} e4m3(q[m, k]) * e4m3(Wq[n, k])      fp32
 * x [M, K] bf16, Wq [N, K] e4m3 codes, sw [ceil(N/128), ceil(K/128)] fp32 (one scale
 * per 128 x 128 weight block, row-major), y [M, N] bf16.  1 <= M <= 64, K % 16 == 0.
 * Runs on the tensor cores only (DG_VAR_TC; params[0] pipeline stages); the K-split
 * is fixed by (N, K) on a given device, so output row m depends on input row m alone
 * at every M.
 * Non-finite activations give NaN outputs for their token.  ws: the status word, and
 * the codes and scales when the quantisation runs as a launch of its own. */
dg_status dg_gemv_a8w8_blockscale(const void* x, const void* Wq, const float* sw, void* y, int M, int N, int K,
                                  void* ws, size_t ws_bytes, dg_stream_t stream, const dg_choice* choice);

/* The quantisation step of dg_gemv_a8w8_blockscale on its own (the same device code):
 * q [M, K] e4m3 codes and sx [M, ceil(K/128)] fp32, as defined there.  M >= 1,
 * K % 16 == 0; asynchronous on `stream`; argument errors return before any launch. */
dg_status dg_quant_a8_blockscale(const void* x, void* q, float* sx, int M, int K, dg_stream_t stream);

/* ---------------------------------------------------------------- selection */

/* Kernel choice for (op, M, N, K): the loaded table's entry for M padded up to
 * the next row bucket (1 2 3 4 6 8 12 16 24 32 48 64 96 128 192 256 384 512), else the compiled
 * default for that bucket -- never a nearest-bucket guess.  mstar PR #1104
 * "What changed" (one per-device table; no table keeps the defaults);
 * "Decode optimization round 3", "Retained change 2" (padded-M lookup). */
dg_status dg_select(dg_op op, int M, int N, int K, dg_choice* out);

/* Load a shape table (JSON written by dg_sweep).  The table's identity (device
 * architecture, driver and runtime versions, library build id, selection-space
 * token) must match this build and device, and no dispatch knob (DG_FORCE_VARIANT)
 * may be set; otherwise DG_ERR_TABLE_REFUSED, one line on stderr, defaults stay.
 * Strata PR #1297, "The second commit: the seam rework", items 1 and 2. */
dg_status dg_table_load(const char* path);

/* Drop the loaded table (defaults again). */
void dg_table_clear(void);

/* Number of entries in the loaded table (0 when none). */
int dg_table_entries(void);

/* Content hash of this library build (sources and compiler); tables record it. */
const char* dg_build_id(void);

/* The selection-space token of this build: it changes whenever the set of
 * variants or their arithmetic changes, which makes older tables stale. */
int dg_selection_space(void);

/* Parse and check a table file without a GPU, against an explicit identity
 * (for host-side tests and offline tools).  Returns the entry count through
 * *entries and DG_OK, or DG_ERR_TABLE_REFUSED with a reason in reason[0..cap). */
dg_status dg_table_check(const char* path, const char* arch, int driver_version,
                         int runtime_version, int* entries, char* reason, size_t reason_cap);

/* On-device sweep: for every shape in the request list, time every candidate
 * variant of the bucket's kernel family the way the benchmark does (CUDA graphs
 * of back-to-back calls over weight copies that exceed the L2 cache), byte-compare
 * each candidate's output with the compiled default's on the same inputs, and
 * write a table that keeps every candidate's time and parameters beside the pick.
 * A candidate replaces the default only if it is bitwise equal and at least 2 %
 * faster, first in the sweep and then in the medians of three more timings of
 * each, taken alternately (pick_us / default_us are then those medians).  mstar PR #1104, "What changed" (the promotion rule, every candidate's
 * time kept beside the choice); Strata PR #1297, "Summary" (byte-compared
 * variants only) and "True-default baseline"; "Decode optimization round 3",
 * "Rejected paths" (re-measure every row against the incumbent in context).
 * Each record names the op and its sizes as dg_workspace_bytes does (N = N_half
 * for gate/up, N = I and K = hidden for MoE W1, N = Nout and K = I for MoE W2);
 * E is the expert count (0 = 128).  The table is written to out_path as JSON with
 * this build's identity.  The sweep allocates and frees its own device buffers
 * (it is an offline tool, not a decode-loop call) and synchronises the device.
 * Returns the first error met; shapes after it are not measured. */
typedef struct {
    int32_t op, M, N, K, topk, E;
} dg_shape;
dg_status dg_sweep(const dg_shape* shapes, int n_shapes, const char* out_path, int reps);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
