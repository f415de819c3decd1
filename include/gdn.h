/*
 * gdn.h — C ABI of the GB300 (sm_103a) Gated Delta Network chunked-prefill
 * forward pass (and its backward, gdn_chunk_bwd).
 *
 * The operation (FlashQLA talk "Qwen系列模型线性注意力高性能优化实践", the
 * recurrent-form and GDN paragraphs): for every sequence n and head h, with the
 * state S in R^{dv x dk},
 *
 *     S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = scale * S_t q_t,            alpha_t = exp(g_t),
 *
 * computed chunk by chunk (C = 64 tokens) in the WY form (same talk, WY and
 * four-step paragraphs): a gate kernel (chunk-local log-space cumsum, head
 * flags), a per-chunk kernel that inverts I + diag(beta) strictlower(K K^T)
 * without any exponentials (Gamma-extraction paragraph), optional intra-card
 * sequence parallelism (difference, compute-for-memory, auto-CP and
 * sliding-window paragraphs), and one fused kernel that forms U, runs the
 * chunk-to-chunk state recurrence and writes o.
 *
 * Layouts (all row-major, C order):
 *   q, k           [B, T, H, dk]   dtype (bf16 or fp32)
 *   v, o           [B, T, H, dv]   dtype
 *   g, beta        [B, T, H]       fp32 (g = log alpha <= 0, beta in [0, 1])
 *   initial_state,
 *   final_state    [N, H, dk, dv]  fp32; element [n][h][j][i] is S[i][j]
 *                                  (key index j outer, value index i inner)
 *   cu_seqlens     [N + 1]         int32, device memory; with it the batch is
 *                                  packed (B = 1, T = total tokens) and
 *                                  sequence n is tokens cu[n] .. cu[n+1]-1
 *
 * Ownership: the caller allocates every buffer (inputs, outputs, workspace)
 * and keeps them alive until the work on `stream` completes.  The library
 * allocates no device or host memory at run time, keeps no state between calls
 * besides per-device caches of device attributes, driver entry points and the
 * two copy streams of gdn_chunk_fwd_host (and the fixed scratch array of
 * gdn_chunk_fwd_static), and never synchronises the stream inside
 * gdn_chunk_fwd.
 *
 * Errors: every call returns a gdn_status and never aborts.  Argument errors
 * are found on the host before any launch.  Errors found on the device (a
 * malformed cu_seqlens, a bounded wait that ran out) are written to an error
 * word inside the workspace; gdn_chunk_fwd_check() reads it.
 *
 * Preconditions that are not checked: q and k rows are L2-normalised (the
 * sliding-window bound relies on it), g <= 0, 0 <= beta <= 1, all inputs
 * finite, and no two calls share a workspace concurrently.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer */
    GDN_ERR_UNSUPPORTED = 2,   /* shape/dtype/device the library does not handle */
    GDN_ERR_WORKSPACE = 3,     /* workspace smaller than gdn_chunk_fwd_workspace_size() */
    GDN_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    GDN_ERR_DEVICE_CHECK = 5,  /* the device found bad input (e.g. cu_seqlens) */
    GDN_ERR_TIMEOUT = 6        /* a bounded device-side wait ran out */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype;

/* Intra-card sequence parallelism (auto-CP paragraph): AUTO lets the planner
 * decide; OFF runs every (sequence, head) as one unit and is bitwise
 * deterministic; FORCE always splits sequences into segments. */
typedef enum { GDN_CP_AUTO = 0, GDN_CP_OFF = 1, GDN_CP_FORCE = 2 } gdn_cp_mode;

/* Which fused kernel runs: AUTO (and TC) pick the tcgen05 kernels for every
 * supported shape — kind::f16 for bf16 inputs, kind::tf32 for fp32 inputs
 * (fp32 operands read as tf32, fp32 accumulation), dk, dv in {32, 64, 128},
 * head sizes below 128 zero-padded to 128 inside the kernels, which is exact;
 * SIMT selects the CUDA-core kernel (fp32 arithmetic throughout; with fp32
 * inputs also the CUDA-core per-chunk inverse). */
typedef enum { GDN_KERNEL_AUTO = 0, GDN_KERNEL_TC = 1, GDN_KERNEL_SIMT = 2 } gdn_kernel;

typedef struct {
    int32_t cp_mode;            /* gdn_cp_mode */
    int32_t kernel;             /* gdn_kernel */
    int32_t chunks_per_segment; /* > 0 forces the segment length L (chunks) when CP is on */
    int32_t sliding;            /* 1 (default): heads with alpha != 1 restart from a
                                   look-back window; 0: every split head uses
                                   correction matrices */
    float sw_eps;               /* look-back tolerance: the window is long enough that
                                   prod(alpha) over it <= sw_eps (default 2^-24) */
    int32_t sm_count;           /* 0: query the device; > 0: plan for this many SMs */
    int32_t stages;             /* 0: the whole path; else a GDN_STAGE_* mask (stages not
                                   selected are skipped and their workspace outputs must
                                   already be there from an earlier call on the same
                                   problem and workspace) */
    int32_t debug_checks;       /* 0, or GDN_DEBUG_* bits (tests of the error paths) */
    void *prof_begin;           /* optional cudaEvent_t, recorded on `stream` right before
                                   the fused output pass is launched */
    void *prof_end;             /* optional cudaEvent_t, recorded right after it */
    int32_t qk_l2norm;          /* 1: the library scales every q and k row to unit L2 norm
                                   (gdn_qk_l2norm with eps 1e-6) into workspace copies
                                   before the pass; 0 (default): the caller's rows are
                                   used as they are (they should be unit-norm already) */
    int32_t inverse_overlap;    /* the tcgen05 path on equal sequences without a split, when
                                   the (sequence, head) units leave SMs idle: k > 0 lets the
                                   fused pass run the per-chunk inverse of the last k chunk
                                   columns (at most all) on those SMs while the other CTAs
                                   run the state recurrence (one cooperative launch; each
                                   such column is loaded only once all its units are in
                                   memory; the results are bitwise those of the separate
                                   inverse).  0 (default) and -1: off.  On a GB300 at
                                   B=4, T=8192, H=32 it moved the step by -6..+3 us (the
                                   24 idle SMs' inverse traffic slows the chain about as
                                   much as it hides), so it is not on by default */
    int32_t reserved[2];
} gdn_options;

/* GDN_DEBUG_TIMEOUT_PROBE: the tile producer of the tcgen05 fused pass signals
 * nothing, so every bounded wait of that pass runs out (about 2 s): the pass
 * records GDN_ERR_TIMEOUT, frees what it holds and returns, and the next call
 * on the same workspace runs normally.  It exists to test the timeout path
 * without faulting or hanging the GPU; the kind::tf32 and CUDA-core passes
 * ignore it. */
enum { GDN_DEBUG_TIMEOUT_PROBE = 1 };

enum {
    GDN_STAGE_PREP = 1,         /* sequence tables, gate kernel, device planner */
    GDN_STAGE_INVERSE = 2,      /* per-chunk inverse T' */
    GDN_STAGE_CORRECTION = 4,   /* correction pass and segment scan (when CP is on) */
    GDN_STAGE_FUSED = 8         /* fused output pass */
};

/* What the host planner decided for a problem (host-only, no GPU needed). */
typedef struct {
    int32_t kernel;             /* gdn_kernel actually used (TC or SIMT) */
    int32_t cp_enabled;         /* 1 when sequences may be split into segments */
    int32_t chunks_per_segment; /* segment length L in chunks */
    int32_t max_chunks;         /* upper bound on chunks over all sequences */
    int32_t max_items;          /* capacity of the fused-kernel work list */
    int32_t max_cp_slots;       /* capacity of the correction-matrix buffers */
    int32_t sm_count;           /* SMs the plan was made for */
    int32_t grid_fused;         /* CTAs of the persistent fused kernel */
    int32_t overlap_columns;    /* chunk columns whose inverse runs inside the fused pass
                                   (see gdn_options.inverse_overlap); 0: none */
    int32_t launches;           /* kernels one gdn_chunk_fwd call launches (the whole path:
                                   q/k normalisation, sequence prep, gate, planner, inverse,
                                   correction pass and scan, fused pass, as the plan needs) */
    size_t workspace_bytes;     /* bytes gdn_chunk_fwd needs */
} gdn_plan_info;

/* Byte offsets of the intermediate tensors inside the workspace, so tests and
 * tools can inspect them after a call (read them only after the stream syncs). */
typedef struct {
    size_t error_word;     /* int32: 0 or a gdn_status found on the device */
    size_t gate_cumsum;    /* fp32 [H, total_T]: chunk-local inclusive cumsum of g */
    size_t chunk_totals;   /* fp32 [H, max_chunks]: sum of g per chunk (chunks in sequence order) */
    size_t head_flags;     /* int32 [N, H]: 1 when some g != 0 (alpha not identically 1) */
    size_t tprime;         /* [H, total_T, 64] T' rows by token; bf16 for bf16 inputs, fp32 for fp32.
                              When the tcgen05 fused kernel runs (bf16) this holds
                              T' diag(c1) instead, c1_m = exp(G* - G_m) beta_m with G* the middle of
                              the chunk's gate cumsum range, or (Gamma ⊙ T') diag(beta) for a chunk
                              whose last cumsum is below -80 */
    size_t chunk_table;    /* int32x4 [max_chunks]: (seq, first token, length, chunk index in seq) */
    size_t num_chunks;     /* int32: chunks actually present */
    size_t items;          /* int32x8 [max_items]: fused-kernel work items (see gdn_work_item) */
    size_t num_items;      /* int32: [0] pass-2 items, [1] pass-1 items, [2] scan units */
    size_t total;
} gdn_workspace_layout;

/* One unit of fused-kernel work as the planner writes it. */
typedef struct {
    int32_t seq, head;
    int32_t c_begin, c_end;   /* chunks [c_begin, c_end) of the sequence produce output */
    int32_t c_start;          /* first chunk run (c_start <= c_begin); chunks before
                                 c_begin only advance the state (look-back) */
    int32_t flags;            /* GDN_ITEM_* bits */
    int32_t slot;             /* correction-buffer slot (CP) or -1 */
    int32_t pad;
} gdn_work_item;

enum {
    GDN_ITEM_OUTPUT = 1,        /* write o for chunks [c_begin, c_end) */
    GDN_ITEM_FROM_INITIAL = 2,  /* start from initial_state (or zero when it is NULL) */
    GDN_ITEM_FROM_ZERO = 4,     /* start from S = 0 */
    GDN_ITEM_FROM_IDENTITY = 8, /* start from S = I and use zero values (correction matrix) */
    GDN_ITEM_FROM_SLOT = 16,    /* start from the scanned segment start in `slot` */
    GDN_ITEM_WRITE_FINAL = 32,  /* write final_state */
    GDN_ITEM_WRITE_SLOT = 64,   /* write the end state to the S* buffer `slot` */
    GDN_ITEM_WRITE_M = 128      /* write the end state to the M buffer `slot` */
};

/* Fill *opts with the defaults (AUTO everywhere, sliding on, sw_eps 2^-24). */
void gdn_default_options(gdn_options *opts);

/*
 * Cost model of the auto-CP planner.  The intra-card sequence-parallel
 * paragraph of the FlashQLA talk "Qwen系列模型线性注意力高性能优化实践" models the
 * time of a split sequence as T = lambda1 L + lambda2 N / L (L chunks per
 * segment, N / L segments) with lambda measured on the hardware; the planner
 * here is the wave-aware form of that model and takes its lambdas from this
 * table, in microseconds on the target GPU with every SM busy:
 *   chunk_step_us  one chunk step of the fused output pass (lambda1, pass 2)
 *   state_step_us  one chunk step of a state-only correction item (lambda1, pass 1)
 *   scan_step_us   one segment step of the segment scan (lambda2)
 *   pass_us        the fixed cost of the correction pass and the scan launches
 * The library starts with values measured on a GB300; gdn_set_plan_costs()
 * replaces them for the whole process (NULL restores those defaults; a
 * non-finite, negative or zero step cost is GDN_ERR_INVALID_ARG) and
 * gdn_get_plan_costs() reads the current table.  The Python package's
 * `calibrate` module measures the table on the GPU at hand by timing this
 * library's own passes.  Plans made before a change keep the costs they were
 * made with; nothing else depends on the table (every plan is exact).
 */
typedef struct {
    float chunk_step_us;
    float state_step_us;
    float scan_step_us;
    float pass_us;
} gdn_plan_costs;

gdn_status gdn_set_plan_costs(const gdn_plan_costs *costs);
void gdn_get_plan_costs(gdn_plan_costs *costs);

/*
 * The enabling boundary of auto CP for batches of equal sequences: the least
 * sequence length, in chunks of 64 tokens, at which GDN_CP_AUTO splits
 * sequences when there are `units` = B x H (sequence, head) units on `sms`
 * SMs, under the current cost table; 0 when no length up to 2^20 chunks does
 * (always for units >= sms).  The talk's enabling-condition paragraph notes
 * that the boundary in the (B x H, length) plane is a curve rather than a
 * threshold on either axis: more units leave fewer idle SMs, so a longer
 * sequence is needed before splitting pays.  Host-only.
 */
int gdn_auto_cp_min_chunks(int units, int sms);

/* Host-only planning: which kernel, whether CP is on, the segment length and
 * the workspace size.  `total_T` is B*T for batched input or the packed token
 * count with cu_seqlens (then B must be 1 and n_seqs = N).  opts may be NULL. */
gdn_status gdn_plan_query(int B, int T, int H, int dk, int dv, int n_seqs, int varlen,
                          gdn_dtype dtype, const gdn_options *opts, gdn_plan_info *out);

/* Bytes of device workspace gdn_chunk_fwd needs for this problem (0 on bad
 * arguments).  `varlen` is 1 when cu_seqlens will be passed. */
size_t gdn_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int n_seqs, int varlen,
                                    gdn_dtype dtype, const gdn_options *opts);

/* Offsets of the intermediates inside the workspace for this problem. */
gdn_status gdn_workspace_query(int B, int T, int H, int dk, int dv, int n_seqs, int varlen,
                               gdn_dtype dtype, const gdn_options *opts, gdn_workspace_layout *out);

/*
 * The forward pass.  All pointers are device pointers (initial_state and
 * cu_seqlens may be NULL).  With cu_seqlens == NULL the batch is B sequences of
 * T tokens (n_seqs is ignored); otherwise B must be 1, T is the total token
 * count and n_seqs = N.  scale <= 0 selects dk^-0.5.  dk, dv in {32, 64, 128}.
 * q, k, v, o, g, beta, states and workspace must be 16-byte aligned.
 * The workspace must hold gdn_chunk_fwd_workspace_size() bytes; it needs no
 * initialisation.  Everything is enqueued on `stream`; nothing syncs.
 */
gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *g, const float *beta,
                         const float *initial_state,
                         const int32_t *cu_seqlens, int n_seqs,
                         float scale,
                         int B, int T, int H, int dk, int dv, gdn_dtype dtype,
                         void *o, float *final_state,
                         void *workspace, size_t workspace_bytes,
                         const gdn_options *opts, gdn_stream_t stream);

/* Synchronises `stream`, then reads the device error word of `workspace`:
 * GDN_OK, GDN_ERR_DEVICE_CHECK (bad cu_seqlens) or GDN_ERR_TIMEOUT. */
gdn_status gdn_chunk_fwd_check(const void *workspace, gdn_stream_t stream);

/* Device bytes gdn_chunk_fwd_host needs as its staging buffer (inputs, outputs
 * and workspace together). */
size_t gdn_chunk_fwd_host_buffer_size(int B, int T, int H, int dk, int dv, int n_seqs, int varlen,
                                      int has_initial_state, gdn_dtype dtype, const gdn_options *opts);

/*
 * The same forward pass for inputs and outputs in HOST memory (pinned memory
 * makes the copies asynchronous).  The call copies the inputs into
 * `device_buffer` (gdn_chunk_fwd_host_buffer_size() bytes, caller-owned), runs
 * gdn_chunk_fwd on `stream`, copies o and final_state back, waits for all of
 * it and returns the device error status as gdn_chunk_fwd_check does.
 * cu_seqlens is a host array here.
 *
 * Above 64 MB of input the problem goes through in up to eight parts: groups
 * of whole sequences with about equal token counts or, when there are fewer
 * sequences than parts and the plan runs every (sequence, head) as one unit,
 * 64-token-aligned pieces of each sequence, each starting from the state the
 * previous piece left in the device buffer.  Part p+1 is copied in on a
 * library copy stream while the pass runs part p on `stream` and part p-1 is
 * copied out on a second library copy stream (both created once per device,
 * non-blocking; they first wait for the work already on `stream`).  Every part
 * keeps the whole problem's plan (CP on or off, the segment length), so the
 * result is the one gdn_chunk_fwd gives on the whole problem, bit for bit.
 */
gdn_status gdn_chunk_fwd_host(const void *q, const void *k, const void *v,
                              const float *g, const float *beta,
                              const float *initial_state,
                              const int32_t *cu_seqlens, int n_seqs,
                              float scale,
                              int B, int T, int H, int dk, int dv, gdn_dtype dtype,
                              void *o, float *final_state,
                              void *device_buffer, size_t device_buffer_bytes,
                              const gdn_options *opts, gdn_stream_t stream);

/*
 * Inter-card sequence parallelism (the talk's difference and compute-for-memory
 * paragraphs, and its timeline paragraph's "inter-card sequence parallelism":
 * the three steps of intra-card CP with the segments on different GPUs).  A
 * batch of sequences is split along time into R slices, one per rank; every
 * rank holds the same (sequence, head) units.  Step one, on every rank:
 *
 *   gdn_chunk_transition: for each (sequence, head) of the local slice, the
 *   affine map the slice applies to the state, S_end = S_start M + S*:
 *   S* is the slice's end state from S_start = 0 with the slice's values, and
 *   M (dk x dk) the end state from S_start = I with zero values, i.e. the
 *   product of the slice's token transitions alpha_t (I - beta_t k_t k_t^T).
 *
 * q is not read (the map does not depend on the queries).  k, v, g, beta,
 * cu_seqlens, B, T, H, dk, dv, dtype as for gdn_chunk_fwd.  Outputs (device,
 * fp32, 16-byte aligned): s_star [N, H, dk, dv] in the state layout of
 * final_state, m [N, H, dk, dk] in the same transposed layout
 * (m[n][h][b][a] = M[a][b]).  An empty sequence maps to S* = 0, M = I.  The
 * workspace holds gdn_chunk_transition_workspace_size() bytes.  Nothing syncs;
 * device-side errors (bad cu_seqlens, timeout) land in the workspace's error
 * word: read them with gdn_chunk_fwd_check(workspace, stream).
 *
 * Step two is an all-gather of (S*, M) over the ranks (the caller's
 * collective), step three gdn_state_scan below, step four gdn_chunk_fwd on the
 * local slice from the rank's start state.
 */
size_t gdn_chunk_transition_workspace_size(int B, int T, int H, int dk, int dv, int n_seqs, int varlen,
                                           gdn_dtype dtype);
gdn_status gdn_chunk_transition(const void *k, const void *v, const float *g, const float *beta,
                                const int32_t *cu_seqlens, int n_seqs,
                                int B, int T, int H, int dk, int dv, gdn_dtype dtype,
                                float *s_star, float *m,
                                void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * Start states of R consecutive slices of the same sequences from their maps:
 * s_start[0] = s0 (NULL: zero) and s_start[r + 1] = s_start[r] M_r + S*_r.
 * s_star [R, N, H, dk, dv], m [R, N, H, dk, dk] as gdn_chunk_transition writes
 * them (rank-major, e.g. the result of an all-gather), s0 [N, H, dk, dv] or
 * NULL, s_start [R, N, H, dk, dv]; device fp32, 16-byte aligned; s_start must
 * not overlap the inputs.  The last map (r = R - 1) is not used.  fp32
 * arithmetic, one CUDA kernel, nothing syncs.
 */
gdn_status gdn_state_scan(const float *s0, const float *s_star, const float *m, int R, int N, int H, int dk,
                          int dv, float *s_start, gdn_stream_t stream);

/*
 * The same walk for the gradient of the state, from the last slice down
 * (sequence parallelism in the backward pass: the results paragraph of the
 * talk has the backward split with the same sliding-window / correction
 * scheme).  With S_end = S_start M + S* per slice, the gradient of the loss
 * with respect to a slice's start state is that of its end state times M^T
 * plus the slice's own term ds_star (its backward run with a zero end
 * gradient), so
 *
 *   ds_end[R - 1] = ds_last (NULL: zero),
 *   ds_end[r] = ds_end[r + 1] M_{r+1}^T + ds_star[r + 1].
 *
 * Layouts, alignment and errors as gdn_state_scan (ds_star in the state
 * layout, m as gdn_chunk_transition writes it); ds_star[0] and m[0] are not
 * used.
 */
gdn_status gdn_state_grad_scan(const float *ds_last, const float *ds_star, const float *m, int R, int N, int H,
                               int dk, int dv, float *ds_end, gdn_stream_t stream);

/*
 * The same forward pass for callers that cannot allocate device memory while
 * they run: a server that hands all of HBM to its own pool at start-up and
 * forbids allocation on the request path, or a plugin that receives tensors
 * from a host framework and has no allocator.  The paper has no counterpart;
 * this is an addition of this library.
 *
 * Arguments are those of gdn_chunk_fwd without the workspace: the scratch is a
 * static device array of 64 MiB inside the library, which every GPU that loads
 * the library holds until the process exits.  A problem whose
 * gdn_chunk_fwd_workspace_size() exceeds 64 MiB is rejected with
 * GDN_ERR_WORKSPACE before anything is enqueued (gdn_last_error_detail() then
 * says how many bytes it needed).  opts->stages must be 0 (the whole pass).
 *
 * The first call on a device looks up the array's device address and caches
 * it (cudaGetSymbolAddress, no allocation); make that first call before any
 * stream capture.  With lazy module loading (the CUDA default) that first
 * call is also when the runtime loads the library's device code and reserves
 * the 64 MiB array on the device, so a caller whose pool takes the rest of
 * HBM at start-up must make one call (any size, e.g. an empty batch) before
 * the pool reserves its memory.  The cached address belongs to the device's
 * current primary context: after cudaDeviceReset() in the same process this
 * entry point must not be called again.  Apart from that first load the call
 * allocates nothing, host or device.
 *
 * Every call on a device shares the one array, which keeps the previous call's
 * contents; the call clears what must start at zero (the error word and the
 * work counters) on `stream` itself.  Calls whose GPU work overlaps (other
 * streams, other host threads) race on the array and give wrong results: order
 * them, e.g. on one stream.
 *
 * device_status: NULL makes the call synchronise `stream` and return the
 * device-side status as gdn_chunk_fwd_check() does.  Otherwise it is a 4-byte
 * aligned device int32 into which the call enqueues a copy of the device
 * status word (0, or a gdn_status) after the pass, and the call returns
 * without synchronising.
 */
gdn_status gdn_chunk_fwd_static(const void *q, const void *k, const void *v,
                                const float *g, const float *beta,
                                const float *initial_state,
                                const int32_t *cu_seqlens, int n_seqs,
                                float scale,
                                int B, int T, int H, int dk, int dv, gdn_dtype dtype,
                                void *o, float *final_state,
                                int32_t *device_status,
                                const gdn_options *opts, gdn_stream_t stream);

/*
 * L2 normalisation of q and k rows over the head dimension, the step in front
 * of the recurrence (the sliding-window paragraph of the FlashQLA talk
 * "Qwen系列模型线性注意力高性能优化实践" takes every key to have unit L2 norm):
 *
 *     x_hat[d] = x[d] / sqrt(sum_d' x[d']^2 + eps)
 *
 * with the sum in fp32 and one rounding to the output type.  q, k: device
 * pointers to `rows` rows of dk contiguous elements (dk in {32, 64, 128};
 * rows = tokens x heads for a [.., H, dk] tensor); either may be NULL, and
 * then its output pointer must be NULL too.  q_out / k_out receive the
 * normalised rows in the same layout and dtype; they may equal q / k (in
 * place).  All pointers 16-byte aligned.  eps <= 0 selects 1e-6.  Enqueued on
 * `stream`; nothing syncs.  gdn_chunk_fwd runs this pass itself, into copies
 * in its workspace, when opts->qk_l2norm is 1.
 * Errors: GDN_ERR_INVALID_ARG (sizes, dtype, alignment, a NULL pairing),
 * GDN_ERR_CUDA (launch failure; see gdn_last_error_detail()).
 */
gdn_status gdn_qk_l2norm(const void *q, const void *k, void *q_out, void *k_out,
                         int64_t rows, int dk, gdn_dtype dtype, float eps,
                         gdn_stream_t stream);

/*
 * Backward of gdn_qk_l2norm for one tensor: with n = sqrt(sum_d x_d^2 + eps)
 * and dy the gradient of x_hat = x / n,
 *
 *     dx = dy / n - x (x . dy) / n^3        (the Jacobian of x / n)
 *
 * in fp32.  x: `rows` rows of dk elements in `dtype` (the tensor that was
 * normalised); dy, dx: fp32 rows in the same layout (dx may equal dy).  All
 * pointers 16-byte aligned, non-NULL when rows > 0; dk in {32, 64, 128};
 * eps <= 0 selects 1e-6 (the forward's default).  Enqueued on `stream`.
 * Errors: GDN_ERR_INVALID_ARG (sizes, dtype, alignment, NULL), GDN_ERR_CUDA.
 */
gdn_status gdn_qk_l2norm_bwd(const void *x, const float *dy, float *dx, int64_t rows, int dk,
                             gdn_dtype dtype, float eps, gdn_stream_t stream);

/*
 * The backward pass: gradients of L = sum <o, d_o> + <final_state,
 * d_final_state> with respect to q, k, v, g, beta and initial_state, for the
 * forward pass gdn_chunk_fwd computes (the backward paragraph of the FlashQLA
 * talk "Qwen系列模型线性注意力高性能优化实践": chunk by chunk in the WY form,
 * the dA and dA^T terms merged).  The library recomputes the chunk start
 * states itself (a forward sweep), so the forward's outputs are not inputs.
 *
 * Inputs as gdn_chunk_fwd (q, k, v in `dtype`; g, beta, initial_state fp32;
 * initial_state and cu_seqlens may be NULL), plus
 *   d_o             [B, T, H, dv]   dtype, the gradient of o
 *   d_final_state   [N, H, dk, dv]  fp32 or NULL (zero)
 * Outputs, all fp32 and written in full (no accumulation into them):
 *   dq, dk          [B, T, H, dk]
 *   dv              [B, T, H, dv]
 *   dg, dbeta       [B, T, H]
 *   d_initial_state [N, H, dk, dv]  (may be NULL: not written)
 * All pointers are device pointers, 16-byte aligned.  The workspace must hold
 * gdn_chunk_bwd_workspace_size() bytes (no initialisation needed; it keeps the
 * chunk start states and the per-chunk intermediates).  Enqueued on `stream`;
 * nothing syncs.  The result does not depend on the launch order of CTAs.
 *
 * Kernels (gdn_set_backward_kernel): by default the tensor-core backward, two
 * tcgen05 kernels with fp32 operands read as tf32 and fp32 accumulation — a
 * chain kernel per (sequence, head) for the state and state-gradient
 * recurrences, dv and d_initial_state, then one CTA per (chunk, head) for dq,
 * dk, dg and dbeta; GDN_KERNEL_SIMT selects the CUDA-core kernel (fp32
 * products, one CTA per 32 value columns, head and sequence).
 * Errors: GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED / GDN_ERR_WORKSPACE before
 * any launch; GDN_ERR_CUDA on a launch failure; a malformed cu_seqlens is
 * written to the workspace's error word, which gdn_chunk_bwd_check() reads.
 * Preconditions as gdn_chunk_fwd's; n_seqs (or B) at most 65535.
 */
size_t gdn_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dv, int n_seqs, int varlen,
                                    gdn_dtype dtype);

gdn_status gdn_chunk_bwd(const void *q, const void *k, const void *v,
                         const float *g, const float *beta,
                         const float *initial_state,
                         const int32_t *cu_seqlens, int n_seqs,
                         float scale,
                         int B, int T, int H, int dk, int dv, gdn_dtype dtype,
                         const void *d_o, const float *d_final_state,
                         float *dq, float *dk_out, float *dv_out, float *dg, float *dbeta,
                         float *d_initial_state,
                         void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * The gradient of the initial state alone: d_initial_state of the backward
 * pass above, from d_o and d_final_state (the state-gradient recurrence run
 * from the last chunk back to the first; it needs neither v nor the initial
 * state, and writes nothing else).  The same tensor-core chain kernel as
 * gdn_chunk_bwd's default, so the result equals its d_initial_state bit for
 * bit.  The sequence-parallel backward takes each segment's local map from it.
 * Arguments, workspace (gdn_chunk_bwd_workspace_size) and errors as
 * gdn_chunk_bwd's; d_initial_state [N, H, dk, dv] fp32 must not be NULL.
 */
gdn_status gdn_chunk_state_grad(const void *q, const void *k, const float *g, const float *beta,
                                const int32_t *cu_seqlens, int n_seqs, float scale,
                                int B, int T, int H, int dk, int dv, gdn_dtype dtype,
                                const void *d_o, const float *d_final_state, float *d_initial_state,
                                void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* Selects the kernels of later gdn_chunk_bwd calls in this process:
 * GDN_KERNEL_AUTO or GDN_KERNEL_TC (the tensor-core backward, the default) or
 * GDN_KERNEL_SIMT (the CUDA-core backward).  Both fit the same workspace size.
 * GDN_ERR_INVALID_ARG for another value. */
gdn_status gdn_set_backward_kernel(gdn_kernel kernel);
gdn_kernel gdn_get_backward_kernel(void);

/* Synchronises `stream` and reads the error word of a gdn_chunk_bwd
 * workspace: GDN_OK, GDN_ERR_DEVICE_CHECK (bad cu_seqlens) or GDN_ERR_TIMEOUT. */
gdn_status gdn_chunk_bwd_check(const void *workspace, gdn_stream_t stream);

/* The CUDA error (and, for tensor-map encoding, the driver result) behind the
 * most recent GDN_ERR_CUDA returned on the calling host thread, as text such
 * as "launch fused_tc: cudaErrorInvalidValue"; after gdn_chunk_fwd_static
 * returns GDN_ERR_WORKSPACE, the scratch it would have needed; "" when there
 * was none. */
const char *gdn_last_error_detail(void);

/* Human-readable name of a status. */
const char *gdn_status_string(gdn_status status);

/* Library version string. */
const char *gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
