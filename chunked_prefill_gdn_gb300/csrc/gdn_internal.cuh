// Internal declarations shared by the CUDA translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kChunk = 64;  // C, the chunk length (WY paragraph of the FlashQLA talk)

// Problem description as the kernels see it (device pointers).
struct Problem {
    const void *q, *k, *v;
    const float *g, *beta, *s0;
    const int32_t *cu;      // device cu_seqlens or nullptr (batched)
    void *o;
    float *sf;
    int B, T, H, dk, dv, N, total_T, varlen, dtype;
    float scale;
    int timeout_probe;      // GDN_DEBUG_TIMEOUT_PROBE: the fused tcgen05 pass's producer
                            // withholds every arrival (its consumers' bounded waits run out)
};

// Device pointers into the caller's workspace.
struct Workspace {
    int *err;               // error word (a gdn_status)
    int *counters;          // [8] work-queue counters, zeroed by the sequence-prep kernel
    int *num_chunks;        // [1]
    int *num_items;         // [4]: pass-2 items, pass-1 items, scan units, -
    int4 *seqinfo;          // [N]: (first token, length, first chunk, chunks)
    int4 *chunks;           // [max_chunks]: (seq, first token, length, chunk index in seq)
    int *flags;             // [N*H]
    float *G;               // [H, total_T]
    float *totals;          // [H, max_chunks]
    void *tprime;           // [H, total_T, C] bf16 (bf16 inputs) or fp32 (fp32 inputs): T', or
                            // T' diag(c1) when the tcgen05 fused kernel runs
    gdn_work_item *items2;  // [max_items]
    gdn_work_item *items_tmp;  // [max_items] or null (planned packed sequences): the planner's
                               // copy of the output list while it deals it out longest first
    gdn_work_item *items1;  // [max_items1]
    int4 *scan_units;       // [max_cp_slots]: (seq, head, segments, first slot)
    int *seq_order;         // [N]: sequences, longest first
    float *cp_s;            // [max_cp_slots, dk, dv]
    float *cp_m;            // [max_cp_slots, dk, dk]
    int max_chunks, max_items, max_items1, max_cp_slots;
};

struct PlanParams {
    int L;            // chunks per segment (huge when CP is off)
    int cp_enabled;
    int sliding;
    float ln_eps;
    int grid;         // CTAs of the persistent fused passes
    float state_ratio;  // measured: a state-only chunk step / an output chunk step
    float scan_ratio;   // measured: a scan step / an output chunk step
    int transition;     // 1: list, per (sequence, head), the two whole-sequence
                        // items of its affine map (S* from zero, M from the
                        // identity) for the correction pass, and nothing else
};

// Host-side layout of the workspace for one problem.
struct Layout {
    size_t err, counters, num_chunks, num_items, seqinfo, chunks, flags, G, totals, tprime,
        items2, items1, scan_units, seq_order, cp_s, cp_m, qn, kn, ready, items_tmp, total;
    int max_chunks, max_items, max_items1, max_cp_slots;
};

// Records the CUDA error behind a GDN_ERR_CUDA for gdn_last_error_detail().
void set_error_detail(const char *where, cudaError_t e, int driver_result = 0);
// Records a plain message for gdn_last_error_detail().
void set_error_text(const char *text);

// Launchers (each returns cudaGetLastError() of its launch).
// emit_items: also write the output pass's work list (equal sequences, no split), so
// that the planner need not run
cudaError_t launch_seqprep(const Problem &p, const Workspace &w, bool emit_items, cudaStream_t s);
cudaError_t launch_gate(const Problem &p, const Workspace &w, cudaStream_t s);
cudaError_t launch_plan(const Problem &p, const Workspace &w, const PlanParams &pp, cudaStream_t s);
// for_tc: a tcgen05 fused kernel consumes the result: for bf16 T' diag(c1)
// (the gate-scaled form that kernel multiplies by) instead of T' itself; for
// fp32 keys T' in fp32 from the tcgen05 inverse (kind::tf32 Gram) rather than
// from the CUDA-core one
// cols < nc (equal sequences of nc chunks, tcgen05 inverse only): chunk
// columns [0, cols) only, the fused kernel computing the others
cudaError_t launch_inverse(const Problem &p, const Workspace &w, bool for_tc, cudaStream_t s, int cols = 0, int nc = 0);
// T' itself (no gate factors) as fp32 rows [H, total_T, 64] into w.tprime (the
// backward pass's T = Gamma ⊙ T'); needs the chunk table (sequence prep).
// tc: the tcgen05 inverse for fp32 keys too (kind::tf32 Gram); else those take
// the CUDA-core inverse (fp32 throughout)
cudaError_t launch_inverse_f32(const Problem &p, const Workspace &w, cudaStream_t s, bool tc);
cudaError_t launch_scan(const Problem &p, const Workspace &w, cudaStream_t s);
// start states of R consecutive slices: out[0] = s0 (or 0), out[r+1] = out[r] M_r + S*_r;
// grad: end gradients, out[R-1] = s0 (or 0), out[r] = out[r+1] M_{r+1}^T + S*_{r+1}
cudaError_t launch_rank_scan(const float *s0, const float *s_star, const float *m, int R, int N, int H, int dk,
                             int dv, float *out, bool grad, cudaStream_t s);
// q and k rows ([rows][dk] each, either may be NULL) scaled to unit L2 norm
// into qo / ko (which may alias q / k)
constexpr float kQkNormEps = 1e-6f;
cudaError_t launch_qk_l2norm(const void *q, const void *k, void *qo, void *ko, long long rows, int dk, int dtype,
                             float eps, cudaStream_t s);
// pass 1 (state-only correction items) or pass 2 (output items) on the CUDA-core kernel
cudaError_t launch_fused_simt(const Problem &p, const Workspace &w, int pass, int grid, cudaStream_t s);
// the tcgen05 kernel; returns cudaErrorNotSupported when the compiled library or the device cannot run it
// The fused kernel can compute the T1 tiles of the last chunk columns itself:
// CTAs past the chain CTAs run the tcgen05 inverse on SMs the (sequence, head)
// units leave idle, column by column, in one cooperative launch.  Before
// loading the T1 tile of such a column the tile producer waits, bounded,
// until every unit of the column is in memory (an acquire of the column's
// count, then a proxy fence before the TMA read).
struct FusedOverlap {
    int chain_ctas;      // CTAs that run work items; the rest run the inverse
    int c0, nc;          // chunk columns [c0, nc) of nc-chunk equal sequences
    int expected;        // units per column (sequences x heads)
    int *ready;          // [nc] per-column counts, zero before the pass
    int gate_scaled;     // 1: T1 = T' diag(c1) as the tcgen05 fused kernel reads it
};

cudaError_t launch_fused_tc(const Problem &p, const Workspace &w, int pass, int grid, cudaStream_t s,
                            const FusedOverlap *ov = nullptr);
// bf16: the kernel above; fp32: the kind::tf32 kernel (launch_fused_tc dispatches)
bool fused_tc_supported(int dtype, int dk, int dv);
bool fused_tf32_supported(int dtype, int dk, int dv);
cudaError_t launch_fused_tf32(const Problem &p, const Workspace &w, int pass, int grid, cudaStream_t s);
int fused_simt_smem_bytes(int dk, int dv);

// The tensor-core backward (kind::tf32): a chain kernel per (sequence, head)
// runs the state recurrence forward and the state-gradient recurrence back,
// storing per-chunk intermediates, then a kernel per (chunk, head) forms the
// gradients of q, k, g and beta from them.
struct BwdTcArgs {
    const void *q, *k, *v, *dout;       // [total_T, H, d], input type
    const float *g, *beta, *s0, *dsf;   // s0, dsf: [N, H, dk, dv] or NULL
    const int32_t *cu;                  // device cu_seqlens or NULL
    const float *tp;                    // [H, total_T, 64]: T' of every chunk, fp32
    const int4 *chunks;                 // the chunk table (sequence prep)
    const int *num_chunks;
    float *s0t, *dst;                   // [slots, H, dk, dv]: chunk start states and end-state gradients
    float *ry, *rqs, *ru, *rdb, *rkds;  // [total_T, H, dv]: K S0^T, Q S0^T, U, dB, K dS^T rows
    float *gq, *gk, *gv, *gg, *gbeta, *gs0;
    int *err;
    int T, H, dk, dv, N, total_T, varlen, dtype;
    int state_grad_only;                // 1: the reverse recurrence alone, writing only gs0
    float scale;
};
cudaError_t launch_bwd_tc(const BwdTcArgs &a, int max_chunks, cudaStream_t s);

// Called once per CTA of a persistent pass after it found the queue empty: the
// last CTA to leave resets the item counter and the exit counter to zero.
__device__ __forceinline__ void finish_queue(int *item_counter, int *exit_counter) {
    __threadfence();
    const int done = atomicAdd(exit_counter, 1) + 1;
    if (done == (int)gridDim.x) {
        atomicExch(item_counter, 0);
        atomicExch(exit_counter, 0);
        __threadfence();
    }
}

// Programmatic dependent launch: every kernel of the path after the first is
// launched with programmatic stream serialisation, so its launch overlaps the
// end of the previous kernel; each kernel starts with grid_dependency_wait(),
// which returns once the previous grid has completed and its memory is
// visible (and at once when there is no such dependency).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Records `code` in the error word unless one is already recorded.
__device__ __forceinline__ void report_error(int *err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ float load_elem(const void *base, size_t idx, int dtype) {
    if (dtype == GDN_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
    return reinterpret_cast<const float *>(base)[idx];
}

__device__ __forceinline__ void store_elem(void *base, size_t idx, int dtype, float x) {
    if (dtype == GDN_BF16)
        reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float *>(base)[idx] = x;
}

}  // namespace gdn
