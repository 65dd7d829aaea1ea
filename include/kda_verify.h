/*
 * kda_verify.h -- C ABI of the fused causal-conv1d + Kimi Delta Attention
 * (gated delta rule) multi-token-prediction verify decode for GB300 (sm_103a).
 *
 * Operation ("[KDA] Fuse causal conv1d into MTP verify decode", cuLA pull
 * request 107: description section and both commit messages).  For every
 * sequence n and value head hv, with q/k head h = hv / (HV/H):
 *
 *   1. width-4 depthwise causal conv1d over [conv_state || T new tokens] of
 *      the packed pre-convolution mixed_qkv, then SiLU, on the q, k and v
 *      channels;
 *   2. q and k L2-normalised over K (eps = 1e-6 inside the root), q scaled
 *      by K^-1/2;
 *   3. the gate: softplus form g = -exp(A_log[hv]) * softplus(a + dt_bias),
 *      softplus linear above 20 (a real branch, as the review of that page
 *      requires), or the safe form g = min(a, 0); beta = sigmoid(b);
 *   4. the gated delta rule, token by token, on the fp32 K x V state:
 *        S <- diag(exp g) S ;  S <- S + beta k (v - S^T k)^T ;  o = S^T q ;
 *   5. outputs: o, the state after every token (inter_ssm), the raw conv
 *      window after every token (conv_snapshots), and conv_state rolled in
 *      place to the last W-1 raw inputs.  The persistent state S0 is read only.
 *
 * Layouts: every tensor is dense, row-major, contiguous; "act" is the
 * activation type of the call (fp32 or bf16); dim = 2*H*K + HV*V and the
 * channels of mixed_qkv / conv_w / conv_state / conv_snapshots are ordered
 * q (H heads x K) | k (H x K) | v (HV x V).  conv_w tap W-1 multiplies the
 * newest token; conv_state index 0 is the oldest raw input.
 *
 * Ownership: the caller allocates every buffer (device memory) and keeps
 * ownership; the library allocates nothing and keeps no pointer after a call
 * returns.  Calls are asynchronous on `stream` (NULL = legacy default
 * stream); no call synchronises except kda_read_status.  Stream order holds
 * as for any launch: every kernel the library launches is a programmatic
 * dependent of the kernel before it on the stream, so its CTAs may become
 * resident while that kernel finishes, but no thread of it touches global
 * memory before that kernel has completed and its writes are visible.
 *
 * Errors: 0 on success; a negative KDA_ERR_* code when the arguments are
 * rejected on the host (nothing is launched, no buffer is touched); a
 * positive value is a cudaError_t reported by the launch.
 */
#ifndef KDA_VERIFY_H
#define KDA_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle type as cudaStream_t. */
typedef struct CUstream_st* kda_stream_t;

typedef enum { KDA_GATE_SOFTPLUS = 0, KDA_GATE_SAFE = 1 } kda_gate_mode;
typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Kernel variants, named after the kernel they run.  An item is one
 * (sequence, v-head, v-tile) slice of a state.  AUTO picks ONE_ITEM (128- or
 * 64-column tiles) or ONE_ITEM_SMEM from N*HV, T, the v-heads per q/k head
 * and the SM count (kda_make_plan, kda_make_decode_plan); PIPELINED and SPLIT
 * measured slower at every point of the configuration sweep on GB300 and run
 * only when requested. */
typedef enum {
  KDA_VARIANT_AUTO = 0,
  KDA_VARIANT_ONE_ITEM = 1,      /* one CTA per item, the state in registers; every warp
                                    runs the item's producer arithmetic, then its recurrence */
  KDA_VARIANT_PIPELINED = 2,     /* persistent, warp-specialised CTAs: producer warps stage the
                                    next item (conv, norms, gate) while consumer warps write the
                                    current item's snapshots; the next state tile arrives by TMA
                                    meanwhile.  4 or 8 consumer warps, K <= 128 */
  KDA_VARIANT_ONE_ITEM_SMEM = 3, /* one item per CTA, the state kept in shared memory instead
                                    of registers (more CTAs per SM; 4 or 8 warps) */
  KDA_VARIANT_SPLIT = 4          /* two kernels: a prep kernel runs the conv / norm / gate work
                                    once per (sequence, q/k head) and rolls conv_state; the
                                    recurrence kernel, its programmatic dependent, issues its
                                    state-tile load first, then reads the item's staged q, k,
                                    alpha, v, beta and writes the snapshots (one item per CTA,
                                    2, 4 or 8 warps, K <= 128).  The stages travel through each
                                    item's own inter_ssm slice of the last token, which the
                                    recurrence overwrites: no workspace beyond the usual */
} kda_variant;

/* Problem shape.  Supported: T in [1, KDA_MAX_T] (N == 0 is a no-op),
 * H >= 1, HV a multiple of H, W == 4, K and V in {32, 64, 128, 256}.  The
 * pipelined variant is built for K <= 128 and V >= 64. */
typedef struct {
  int N, T, H, HV, K, V, W;
  kda_dtype act;
} kda_shape;

#define KDA_MAX_T 16

/* A launch plan (see kda_make_plan and kda_conv_verify_plan). */
typedef struct {
  int variant;
  int bv;
  int warps;
  int grid;
  int ctas_per_sm;
  long long items;
  /* L2 prefetch distance of the one-item variants: each CTA prefetches into
   * L2 the inputs and state tile of the item this many items ahead (default
   * about 3/8 of a wave of resident CTAs).  In a plan given to
   * kda_conv_verify_plan: < 0 off, 0 the default, > 0 explicit.  PIPELINED
   * requests every input one item ahead itself and ignores it (0). */
  int prefetch;
  /* When G * (V / bv) > 1 items read the same q/k channels: who rolls their
   * conv_state (0 for SPLIT, whose first kernel rolls every channel).
   * KDA_QK_ROLL_COUNTER: the last of those items to arrive on a counter in
   * the workspace, inside the verify kernel (one launch).
   * KDA_QK_ROLL_KERNEL: a second, small kernel launched after the verify
   * kernel on the same stream (no atomics in the verify kernel; faster on
   * large launches).  KDA_QK_ROLL_CLUSTER (ONE_ITEM with bv of 64 or 128
   * columns, 32 or 64 at K = 256, and G * (V / bv) <= KDA_MAX_QK_CLUSTER):
   * the items of a group run as one thread-block cluster whose first CTA
   * rolls after a cluster barrier (one launch, no atomics; the dispatcher's
   * pick below 2 waves of resident CTAs, where it is built).  In a plan
   * given to kda_conv_verify_plan, KDA_QK_ROLL_AUTO (0) lets the dispatcher
   * choose. */
  int qk_roll;
  /* Kernels one call with this plan launches (1 or 2). */
  int launches;
} kda_plan;

#define KDA_QK_ROLL_AUTO 0
#define KDA_QK_ROLL_COUNTER 1
#define KDA_QK_ROLL_KERNEL 2
#define KDA_QK_ROLL_CLUSTER 3
#define KDA_MAX_QK_CLUSTER 8  /* largest cluster of the cluster roll (portable size) */

/* Error codes (negative: rejected on the host, nothing launched). */
#define KDA_OK 0
#define KDA_ERR_NULL (-1)        /* a required pointer is NULL */
#define KDA_ERR_SHAPE (-2)       /* unsupported or inconsistent shape */
#define KDA_ERR_DTYPE (-3)       /* unknown activation type */
#define KDA_ERR_MISALIGNED (-4)  /* a pointer is not 16-byte aligned */
#define KDA_ERR_ALIAS (-5)       /* an output overlaps an input or another output */
#define KDA_ERR_WORKSPACE (-6)   /* workspace missing or smaller than kda_workspace_bytes */
#define KDA_ERR_GATE (-7)        /* unknown gate mode, or softplus without A_log/dt_bias */
#define KDA_ERR_VARIANT (-8)     /* unknown variant */
#define KDA_ERR_DEVICE (-9)      /* device query or driver entry point failed */
#define KDA_ERR_SCRATCH_LIMIT (-10) /* kda_conv_verify_noalloc: the shape needs more
                                       scratch than the built-in array holds */

/* Device status bits, written into the workspace by a kernel that gave up a
 * bounded wait (the kernel then returns without hanging the GPU). */
#define KDA_STATUS_OK 0
#define KDA_STATUS_TMA_TIMEOUT 1
#define KDA_STATUS_BAD_ACCEPT 2  /* kda_commit: an accepted count outside [1, T] */
#define KDA_STATUS_BAD_INDEX 4   /* a state-pool slot >= its pool size (sequence skipped) */

/* The fused verify decode.
 *   s              problem shape (host pointer, read during the call only)
 *   mixed_qkv      act  [N, T, dim]      packed pre-conv q|k|v, read
 *   conv_w         act  [dim, W]         read
 *   conv_state     act  [N, dim, W-1]    IN/OUT: rolled in place to the last
 *                                        W-1 raw inputs of each channel
 *   A_log          f32  [HV]             softplus gate only (NULL for safe)
 *   dt_bias        f32  [HV, K]          softplus gate only (NULL for safe)
 *   a              act  [N, T, HV, K]    gate input; safe gate: the log-decay
 *   b              act  [N, T, HV]       beta logit
 *   S0             f32  [N, HV, K, V]    persistent state, read only
 *   gate_mode      KDA_GATE_SOFTPLUS or KDA_GATE_SAFE
 *   o              act  [N, T, HV, V]    OUT
 *   inter_ssm      f32  [N, T, HV, K, V] OUT: S after token t
 *   conv_snapshots act  [N, T, dim, W-1] OUT: raw conv window after token t
 *                                        (the W-1 newest raw inputs)
 *   workspace      device scratch of >= kda_workspace_bytes(s) bytes, zeroed
 *                  once before its first use; every launch leaves it zeroed
 *                  again.  One workspace per stream: two launches that run
 *                  concurrently must not share one.
 *   workspace_bytes  size of `workspace`
 * All device pointers must be 16-byte aligned.  Outputs must not overlap
 * inputs or each other; conv_state is the only in-place buffer. */
int kda_conv_verify(const kda_shape* s, const void* mixed_qkv, const void* conv_w,
                    void* conv_state, const float* A_log, const float* dt_bias,
                    const void* a, const void* b, const float* S0, kda_gate_mode gate_mode,
                    void* o, float* inter_ssm, void* conv_snapshots, void* workspace,
                    size_t workspace_bytes, kda_stream_t stream);

/* Same as kda_conv_verify with an explicit variant (AUTO = the dispatcher's
 * choice).  Every variant produces bit-identical outputs. */
int kda_conv_verify_variant(const kda_shape* s, const void* mixed_qkv, const void* conv_w,
                            void* conv_state, const float* A_log, const float* dt_bias,
                            const void* a, const void* b, const float* S0,
                            kda_gate_mode gate_mode, void* o, float* inter_ssm,
                            void* conv_snapshots, void* workspace, size_t workspace_bytes,
                            kda_variant variant, kda_stream_t stream);

/* State-pool indirection ("[KDA] Fuse causal conv1d into MTP verify decode":
 * conv_state_indices, cache_indices and intermediate_state_indices are
 * normalised independently).  Each array is int32 [N] on the device, or NULL
 * for the identity (slot = n, pool of N slots):
 *   cache_indices               slot of sequence n's persistent state in the
 *                               S0 pool  f32 [state_pool, HV, K, V]
 *   conv_state_indices          slot of its conv window in the conv_state pool
 *                               act [conv_pool, dim, W-1]
 *   intermediate_state_indices  slot of its snapshots in the inter_ssm pool
 *                               f32 [inter_pool, T, HV, K, V] and the
 *                               conv_snapshots pool act [inter_pool, T, dim, W-1]
 * A negative slot in any array marks a padding sequence: nothing of it is read
 * or written (its o rows are left untouched).  A slot >= its pool size skips
 * the sequence the same way and sets KDA_STATUS_BAD_INDEX in the workspace
 * status word.  Two live sequences must not share a slot. */
typedef struct {
  const int32_t* cache_indices;
  const int32_t* conv_state_indices;
  const int32_t* intermediate_state_indices;
  int state_pool;  /* slots in the S0 pool (used when cache_indices != NULL) */
  int conv_pool;   /* slots in the conv_state pool */
  int inter_pool;  /* slots in the inter_ssm / conv_snapshots pools */
} kda_state_indices;

/* kda_conv_verify over state pools: conv_state, S0, inter_ssm and
 * conv_snapshots are the pools described by `idx` (NULL = dense, as
 * kda_conv_verify); mixed_qkv, a, b and o stay dense [N, ...].  `plan` may be
 * NULL (the dispatcher's choice) or an explicit plan as for
 * kda_conv_verify_plan.  Outputs of every plan are bit-identical to the dense
 * call on the gathered inputs. */
int kda_conv_verify_indexed(const kda_shape* s, const kda_state_indices* idx,
                            const void* mixed_qkv, const void* conv_w, void* conv_state,
                            const float* A_log, const float* dt_bias, const void* a,
                            const void* b, const float* S0, kda_gate_mode gate_mode, void* o,
                            float* inter_ssm, void* conv_snapshots, void* workspace,
                            size_t workspace_bytes, const kda_plan* plan, kda_stream_t stream);

/* Plain (non-speculative) decode: the same step without rollback snapshots.
 * Runs the T tokens of every sequence exactly as kda_conv_verify does, but
 * writes no inter_ssm and no conv_snapshots: the state after the last token
 * replaces the persistent state in place (S is read, then overwritten; it
 * equals the verify's inter_ssm[.., T-1] bit for bit), and conv_state is
 * rolled.  idx may be NULL (dense) or give cache_indices / conv_state_indices
 * pools (intermediate_state_indices is ignored); plan may be NULL or a
 * ONE_ITEM / ONE_ITEM_SMEM plan (PIPELINED: KDA_ERR_VARIANT).  Traffic per
 * sequence and head: the state read and written once.  Same error codes. */
int kda_conv_decode(const kda_shape* s, const kda_state_indices* idx, const void* mixed_qkv,
                    const void* conv_w, void* conv_state, const float* A_log,
                    const float* dt_bias, const void* a, const void* b, float* S,
                    kda_gate_mode gate_mode, void* o, void* workspace, size_t workspace_bytes,
                    const kda_plan* plan, kda_stream_t stream);

/* Commit / rollback after a verify: accept the first accepted[n] tokens of
 * every sequence ("[KDA] Fuse causal conv1d into MTP verify decode": the
 * verify writes per-token state and conv-window snapshots for rollback).
 * For each n with 1 <= accepted[n] <= T:
 *   S[n]          <- inter_ssm[n, accepted[n]-1]        f32 [HV, K, V]
 *   conv_state[n] <- conv_snapshots[n, accepted[n]-1]   act [dim, W-1]
 *   s               the shape of the verify call (T = tokens verified)
 *   accepted        int32 [N], device
 *   inter_ssm       f32 [N, T, HV, K, V], conv_snapshots act [N, T, dim, W-1]:
 *                   the verify's outputs (read)
 *   S               f32 [N, HV, K, V] OUT (e.g. the persistent state the
 *                   verify read as S0)
 *   conv_state      act [N, dim, W-1] OUT
 *   status          optional device int: KDA_STATUS_BAD_ACCEPT is OR-ed in
 *                   when a count is out of range; that sequence is left
 *                   untouched.  May be NULL.
 * A pure HBM copy, asynchronous on `stream`.  Outputs must not overlap the
 * inputs.  Returns 0, a negative KDA_ERR_* code, or a cudaError_t. */
int kda_commit(const kda_shape* s, const int32_t* accepted, const float* inter_ssm,
               const void* conv_snapshots, float* S, void* conv_state, int* status,
               kda_stream_t stream);

/* kda_commit over state pools: reads the snapshots of sequence n from slot
 * intermediate_state_indices[n] of the inter_ssm / conv_snapshots pools and
 * writes S slot cache_indices[n] and conv_state slot conv_state_indices[n]
 * (NULL arrays: identity).  Padding (negative) slots are skipped; slots beyond
 * a pool skip the sequence and set KDA_STATUS_BAD_INDEX in *status. */
int kda_commit_indexed(const kda_shape* s, const kda_state_indices* idx,
                       const int32_t* accepted, const float* inter_ssm,
                       const void* conv_snapshots, float* S, void* conv_state, int* status,
                       kda_stream_t stream);

/* Allocation-free variant of kda_conv_verify.  The verify-decode page has no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- a plugin given only its input and output buffers, a
 * serving loop whose memory pool is fixed after start-up, code that must not
 * call cudaMalloc (it synchronises the device and can fail under a memory
 * cap).  Arguments are those of kda_conv_verify without the workspace: the
 * scratch (the status word and, on launches whose q/k conv_state is rolled
 * by the counter, the arrival counters) lives in a static device array of
 * KDA_NOALLOC_MAX_SCRATCH_BYTES inside the library, held on every GPU that
 * loads the library until the process exits.  A shape whose
 * kda_workspace_bytes() exceeds that size is rejected with
 * KDA_ERR_SCRATCH_LIMIT (N*H up to 65532 fits).  The first call on a device,
 * with that device current, looks up the array's device address; make it
 * before any stream capture.  Each call clears the scratch it needs on
 * `stream`, then launches the same kernel as kda_conv_verify; it never
 * allocates or frees.  All calls share the one array: calls whose kernels
 * overlap on the GPU race and must be serialised by the caller. */
#define KDA_NOALLOC_MAX_SCRATCH_BYTES (256 * 1024)
/* An empty batch (N == 0) launches nothing and touches no scratch; its shape
 * and gate mode are checked as kda_conv_verify checks them.  The address is
 * kept per device together with the driver context it was looked up in; a
 * call under another context (after cudaDeviceReset, or a context the caller
 * made current) looks it up again. */
int kda_conv_verify_noalloc(const kda_shape* s, const void* mixed_qkv, const void* conv_w,
                            void* conv_state, const float* A_log, const float* dt_bias,
                            const void* a, const void* b, const float* S0,
                            kda_gate_mode gate_mode, void* o, float* inter_ssm,
                            void* conv_snapshots, kda_stream_t stream);

/* Synchronously read (and clear) the device status word of the built-in
 * scratch that kda_conv_verify_noalloc uses, on `stream`.  `s` is the shape
 * of the call whose status is wanted (the word sits after that shape's
 * arrival counters).  Read it before the next kda_conv_verify_noalloc call:
 * every call clears the scratch it uses first.  *status receives KDA_STATUS_*
 * bits (KDA_STATUS_TMA_TIMEOUT: a kernel gave up a bounded wait and its
 * outputs are incomplete).  Returns 0, KDA_ERR_NULL, KDA_ERR_SCRATCH_LIMIT,
 * KDA_ERR_DEVICE or a cudaError_t.  Allocates nothing. */
int kda_noalloc_read_status(const kda_shape* s, int* status, kda_stream_t stream);

/* Bytes of workspace a call with shape `s` needs (arrival counters for the
 * shared q/k conv_state write-back, N*H int32, used when the plan's qk_roll
 * is the counter, plus a status word), rounded up to 256.  Returns 0 for a
 * NULL shape. */
size_t kda_workspace_bytes(const kda_shape* s);

/* The launch plan the dispatcher picks; host-only, no CUDA call.
 *   num_sms   streaming multiprocessors of the device
 *   variant   requested variant (AUTO lets the dispatcher decide)
 * Out: chosen variant, v-tile width bv (columns of V per CTA), warps per
 * CTA, grid size, CTAs per SM, L2 prefetch distance, the q/k conv_state roll
 * when several items read one q/k head (the cluster below 2 waves of resident
 * CTAs where it is built, else the counter; the second kernel from 2 waves)
 * and the number of launches.  Returns 0 or a negative KDA_ERR_* code. */
int kda_make_plan(const kda_shape* s, int num_sms, kda_variant variant, kda_plan* out);

/* The plan kda_conv_decode picks for shape `s` (plain decode: ONE_ITEM or
 * ONE_ITEM_SMEM only; AUTO, ONE_ITEM or ONE_ITEM_SMEM may be requested).
 * Host-only, no CUDA call.  Returns 0 or a negative KDA_ERR_* code. */
int kda_make_decode_plan(const kda_shape* s, int num_sms, kda_variant variant, kda_plan* out);

/* Fill the derived fields of a hand-written plan (variant, bv and the
 * optional grid / prefetch / qk_roll requests set) exactly as
 * kda_conv_verify_plan would before launching it: warps, grid, ctas_per_sm,
 * items, prefetch, qk_roll, launches.  Host-only, no CUDA call.  `decode`
 * non-zero checks the plan against kda_conv_decode's variants.  Returns 0 or
 * KDA_ERR_SHAPE / KDA_ERR_VARIANT / KDA_ERR_NULL / KDA_ERR_DEVICE. */
int kda_resolve_plan(const kda_shape* s, int num_sms, int decode, kda_plan* plan);

/* Same as kda_conv_verify with an explicit launch plan, e.g. one returned by
 * kda_make_plan and then edited.  Read from `plan`: variant, bv (v-tile
 * width, at most V and dividing V: 1, 2, 4 or 8 warps of 16 columns for
 * ONE_ITEM, 4 or 8 for ONE_ITEM_SMEM -- at K = 256 warps of 8 columns, and 2,
 * 4 or 8 of them for ONE_ITEM; 64 or 128 for PIPELINED, whose shared memory
 * must also fit one CTA: at T = 16 with fp32 activations only 64; 32, 64 or
 * 128 for SPLIT, as long as the item's stage fits its K x bv slice, e.g. at
 * K = 128 and bv = 32 up to T = 7), for
 * PIPELINED grid (persistent CTAs; <= 0 picks one wave of resident CTAs),
 * prefetch and qk_roll (see kda_plan).  The other fields are recomputed.  An invalid plan
 * returns KDA_ERR_VARIANT.  Every plan produces bit-identical outputs. */
int kda_conv_verify_plan(const kda_shape* s, const void* mixed_qkv, const void* conv_w,
                         void* conv_state, const float* A_log, const float* dt_bias,
                         const void* a, const void* b, const float* S0, kda_gate_mode gate_mode,
                         void* o, float* inter_ssm, void* conv_snapshots, void* workspace,
                         size_t workspace_bytes, const kda_plan* plan, kda_stream_t stream);

/* Synchronously read (and clear) the device status word of `workspace` on
 * `stream`.  *status receives KDA_STATUS_* bits.  Returns 0 or an error. */
int kda_read_status(const kda_shape* s, void* workspace, int* status, kda_stream_t stream);

/* Diagnostic: run the kernels' bounded device waits against an mbarrier that
 * nothing arrives at, so that they give up on purpose, without a fault; the
 * context stays usable.  On `stream`:
 *   mode 0  one CTA: the one-item kernels' wait, limit_ns (0 .. 2e9) on the clock;
 *   mode 1  the same, then it raises the pipelined kernel's abort flag, which
 *           ends a second warp's pipelined-kernel wait early;
 *   mode 2  the pipelined kernel's wait alone, until its own 2 s limit;
 *   mode 3  a cluster of 4 CTAs: the one-item kernels' time-out path under the
 *           cluster q/k roll (arrive on the cluster barrier, the wait gives up
 *           at limit_ns, report, wait on the cluster barrier, return).
 * `status` is a device int[2], OR-ed into: status[0] gets KDA_STATUS_TMA_TIMEOUT
 * when a wait gave up, status[1] 1 (the one-item wait gave up), 2 (the
 * pipelined wait did), 4 (the cluster path's wait did).  Returns 0,
 * KDA_ERR_NULL, KDA_ERR_SHAPE (mode or limit out of range) or a cudaError_t. */
int kda_selftest_bounded_wait(int mode, long long limit_ns, int* status, kda_stream_t stream);

/* Human-readable text for a return code (negative KDA_ERR_* or positive
 * cudaError_t).  Never NULL. */
const char* kda_strerror(int code);

/* Library version, e.g. 0x000100 for 0.1.0. */
int kda_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_VERIFY_H */
