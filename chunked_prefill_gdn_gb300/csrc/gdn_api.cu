// C ABI of the library: argument checks, the host planner, the workspace
// layout and the launch sequence
//   sequence prep -> gate -> device planner -> per-chunk inverse
//   -> [correction pass -> segment scan] -> fused pass
// all on the caller's stream, with no host synchronisation.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "gdn_internal.cuh"

using namespace gdn;

namespace {

constexpr int kDefaultSMs = 152;        // GB300
constexpr int kMinSegmentChunks = 8;
// Priors of the host planner about the gates, which only the device sees (it
// refines the plan per pass once the head flags are known): the look-back a
// split segment of a decaying head re-runs, and the share of split heads that
// need correction matrices (alpha == 1).  They describe the workload, not the
// hardware; the hardware enters through the measured step costs below.
constexpr double kLookbackChunks = 4.0;
constexpr double kCorrectionShare = 0.5;

// Measured step costs of the auto-CP planner (the talk's one-wave model
// T = lambda1 L + lambda2 N / L, made wave-aware): gdn_plan_costs.  The
// defaults were measured on a GB300 (152 SMs, 2.07 GHz) with the package's
// calibrate module: an output chunk step 1.79 us, a state-only chunk step
// 1.51 us, a scan step 3.95 us, 38.3 us for the two extra launches.
// gdn_set_plan_costs() replaces them.
constexpr gdn_plan_costs kDefaultCosts = {1.79f, 1.51f, 3.95f, 38.3f};
std::mutex g_costs_mu;
gdn_plan_costs g_costs = kDefaultCosts;

gdn_plan_costs current_costs() {
    std::lock_guard<std::mutex> lock(g_costs_mu);
    return g_costs;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool valid_head_dim(int d) { return d == 32 || d == 64 || d == 128; }

int device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return kDefaultSMs;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = kDefaultSMs;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

struct HostPlan {
    int kernel;
    int cp;
    int L;
    int sms;
    int grid;
    int nc;             // chunks per sequence (equal sequences)
    int ov_cols;        // chunk columns whose inverse runs inside the fused pass
    int ov_ctas;        // CTAs of the fused launch that run it
    int units;          // (sequence, head) units
    int N;
    long long total_T;
    int launches;       // library kernels one call launches (whole path)
    Layout lay;
};

void default_options(gdn_options *o) {
    memset(o, 0, sizeof(*o));
    o->cp_mode = GDN_CP_AUTO;
    o->kernel = GDN_KERNEL_AUTO;
    o->chunks_per_segment = 0;
    o->sliding = 1;
    o->sw_eps = 5.9604645e-08f;  // 2^-24
    o->sm_count = 0;
}

// Modelled time (microseconds) of B equal sequences of nc chunks split into
// ns segments, on `sms` CTAs of the persistent passes: the output pass takes
// as many waves as its items need, each as long as a segment (plus the
// look-back a decaying head re-runs); the correction pass likewise for the
// expected share of heads that need correction matrices (2 ns - 3 items each),
// then the serial scan over segments and the fixed cost of the two launches.
double split_cost(int units, int nc, int ns, int sms, const gdn_plan_costs &c) {
    if (ns <= 1) return ceil((double)units / sms) * nc * c.chunk_step_us;
    const int L = (nc + ns - 1) / ns;
    const double w2 = ceil((double)units * ns / sms);
    double t = w2 * (L * (double)c.chunk_step_us + kLookbackChunks * c.state_step_us);
    const double w1 = ceil(kCorrectionShare * units * (2.0 * ns - 3.0) / sms);
    t += w1 * L * (double)c.state_step_us + (ns - 1) * (double)c.scan_step_us + c.pass_us;
    return t;
}

// Segments per unit for B equal sequences of nc chunks: the count with the
// least modelled time; one segment unless splitting wins by 10%.
int choose_segments(int units, int nc, int sms) {
    const gdn_plan_costs costs = current_costs();
    auto cost = [&](int ns) { return split_cost(units, nc, ns, sms, costs); };
    int best = 1;
    double best_cost = cost(1);
    const int max_ns = std::max(1, std::min(nc / kMinSegmentChunks, 4 * sms));
    for (int ns = 2; ns <= max_ns; ++ns) {
        const double c = cost(ns);
        if (c < best_cost) {
            best_cost = c;
            best = ns;
        }
    }
    return best_cost < 0.9 * cost(1) ? best : 1;
}

gdn_status make_plan(int B, int T, int H, int dk, int dv, int n_seqs, int varlen, int dtype,
                     const gdn_options *opts_in, int sms_query, HostPlan *hp) {
    gdn_options opts;
    if (opts_in) opts = *opts_in; else default_options(&opts);
    if (B < 1 || T < 0 || H < 1 || H > 4096) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return GDN_ERR_INVALID_ARG;
    if (!valid_head_dim(dk) || !valid_head_dim(dv)) return GDN_ERR_UNSUPPORTED;
    if (varlen && (B != 1 || n_seqs < 1)) return GDN_ERR_INVALID_ARG;
    if (opts.cp_mode < GDN_CP_AUTO || opts.cp_mode > GDN_CP_FORCE) return GDN_ERR_INVALID_ARG;
    if (opts.kernel < GDN_KERNEL_AUTO || opts.kernel > GDN_KERNEL_SIMT) return GDN_ERR_INVALID_ARG;
    if (opts.qk_l2norm != 0 && opts.qk_l2norm != 1) return GDN_ERR_INVALID_ARG;
    const int N = varlen ? n_seqs : B;
    const long long total_T = varlen ? (long long)T : (long long)B * T;
    const long long nc_seq = ((long long)T + kChunk - 1) / kChunk;
    const long long max_chunks_ll = varlen ? total_T / kChunk + N : (long long)B * nc_seq;
    if (total_T * H * kChunk >= (1LL << 40) || max_chunks_ll >= (1LL << 30) || (long long)N * H >= (1LL << 30))
        return GDN_ERR_UNSUPPORTED;
    const int max_chunks = (int)max_chunks_ll;
    const int sms = opts.sm_count > 0 ? opts.sm_count : sms_query;

    int kernel = GDN_KERNEL_SIMT;
    const bool tc_ok = fused_tc_supported(dtype, dk, dv);
    if (opts.kernel == GDN_KERNEL_TC && !tc_ok) return GDN_ERR_UNSUPPORTED;
    if (opts.kernel != GDN_KERNEL_SIMT && tc_ok) kernel = GDN_KERNEL_TC;

    int cp = 0;
    int L = std::max(1, max_chunks);
    const int units = N * H;
    if (opts.cp_mode == GDN_CP_FORCE) {
        cp = 1;
        L = opts.chunks_per_segment > 0
                ? opts.chunks_per_segment
                : std::max(1, (int)(((long long)max_chunks * H + sms - 1) / sms));
    } else if (opts.cp_mode == GDN_CP_AUTO) {
        if (opts.chunks_per_segment > 0) {
            cp = 1;
            L = opts.chunks_per_segment;
        } else if (!varlen) {
            const int ns = nc_seq > 0 ? choose_segments(units, (int)nc_seq, sms) : 1;
            if (ns > 1) {
                cp = 1;
                L = (int)((nc_seq + ns - 1) / ns);
            }
        } else {
            cp = 1;
            L = std::max(kMinSegmentChunks, (int)(((long long)max_chunks * H + sms - 1) / sms));
        }
    }
    // the inverse of the last chunk columns inside the fused pass (equal
    // sequences without a split, tcgen05 kernels, idle SMs)
    int ov_cols = 0, ov_ctas = 0;
    if (kernel == GDN_KERNEL_TC && dtype == GDN_BF16 && !cp && !varlen && opts.inverse_overlap > 0 && units < sms &&
        nc_seq > 0) {
        ov_cols = (int)std::min<long long>(opts.inverse_overlap, nc_seq);
        ov_ctas = sms - units;
    }
    const int segs_bound = cp ? (int)(((long long)max_chunks + L - 1) / L) : 0;
    Layout &lay = hp->lay;
    lay.max_chunks = max_chunks;
    lay.max_items = H * (N + segs_bound);
    lay.max_items1 = cp ? 2 * H * segs_bound : 0;
    lay.max_cp_slots = cp ? H * segs_bound : 0;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    lay.err = take(256);                      // error word, counters and counts share one block
    lay.counters = lay.err + 16;
    lay.num_chunks = lay.err + 48;
    lay.num_items = lay.err + 64;
    lay.seqinfo = take((size_t)N * 16);
    lay.chunks = take((size_t)max_chunks * 16);
    lay.flags = take((size_t)N * H * 4);
    lay.G = take((size_t)H * total_T * 4);
    lay.totals = take((size_t)H * max_chunks * 4);
    lay.tprime = take((size_t)H * total_T * kChunk * (dtype == GDN_BF16 ? 2 : 4));
    lay.items2 = take((size_t)lay.max_items * sizeof(gdn_work_item));
    lay.items1 = take((size_t)lay.max_items1 * sizeof(gdn_work_item));
    lay.scan_units = take((size_t)lay.max_cp_slots * 16);
    lay.seq_order = take((size_t)N * 4);
    lay.cp_s = take((size_t)lay.max_cp_slots * dk * dv * 4);
    lay.cp_m = take((size_t)lay.max_cp_slots * dk * dk * 4);
    // normalised copies of q and k when the library normalises them
    const size_t qk_bytes = opts.qk_l2norm ? (size_t)total_T * H * dk * (dtype == GDN_BF16 ? 2 : 4) : 0;
    lay.qn = take(qk_bytes);
    lay.kn = take(qk_bytes);
    lay.ready = take(ov_cols > 0 ? (size_t)nc_seq * 4 : 0);
    // the planner's copy of the output list while it deals it out (packed sequences)
    lay.items_tmp = take(varlen ? (size_t)lay.max_items * sizeof(gdn_work_item) : 0);
    lay.total = off;
    hp->kernel = kernel;
    hp->cp = cp;
    hp->L = L;
    hp->sms = sms;
    hp->grid = sms;
    hp->nc = (int)nc_seq;
    hp->ov_cols = ov_cols;
    hp->ov_ctas = ov_ctas;
    hp->units = units;
    hp->N = N;
    hp->total_T = total_T;
    // normalisation, sequence prep, gate, planner (not for equal sequences
    // without a split: the sequence-prep kernel lists their items), inverse,
    // correction pass and scan, fused pass
    const bool direct = !varlen && !cp;
    hp->launches = (opts.qk_l2norm && max_chunks > 0 ? 1 : 0) + 1 + (max_chunks > 0 ? 2 : 0) + (direct ? 0 : 1) +
                   (cp ? 2 : 0) + 1;
    return GDN_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

thread_local char g_error_detail[256] = "";

gdn_status cuda_fail(const char *where, cudaError_t e) {
    gdn::set_error_detail(where, e);
    return GDN_ERR_CUDA;
}

}  // namespace

namespace gdn {
void set_error_detail(const char *where, cudaError_t e, int driver_result) {
    if (driver_result)
        snprintf(g_error_detail, sizeof(g_error_detail), "%s: %s (driver result %d)", where, cudaGetErrorName(e),
                 driver_result);
    else
        snprintf(g_error_detail, sizeof(g_error_detail), "%s: %s", where, cudaGetErrorName(e));
}

void set_error_text(const char *text) { snprintf(g_error_detail, sizeof(g_error_detail), "%s", text); }
}  // namespace gdn

extern "C" {

void gdn_default_options(gdn_options *opts) {
    if (opts) default_options(opts);
}

gdn_status gdn_set_plan_costs(const gdn_plan_costs *costs) {
    gdn_plan_costs c = costs ? *costs : kDefaultCosts;
    auto ok = [](float x, float lo) { return x == x && x >= lo && x < 1e6f; };
    if (!ok(c.chunk_step_us, 1e-3f) || !ok(c.state_step_us, 1e-3f) || !ok(c.scan_step_us, 0.f) ||
        !ok(c.pass_us, 0.f))
        return GDN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_costs_mu);
    g_costs = c;
    return GDN_OK;
}

void gdn_get_plan_costs(gdn_plan_costs *costs) {
    if (costs) *costs = current_costs();
}

int gdn_auto_cp_min_chunks(int units, int sms) {
    if (units < 1 || sms < 1 || units >= sms) return 0;
    constexpr int kMax = 1 << 20;
    // the first length on a geometric grid where the planner splits, then the
    // exact boundary by bisection below it
    int lo = kMinSegmentChunks, hi = 0;
    for (int nc = kMinSegmentChunks; nc <= kMax; nc = std::max(nc + 1, nc + nc / 16)) {
        if (choose_segments(units, nc, sms) > 1) {
            hi = nc;
            break;
        }
        lo = nc;
    }
    if (hi == 0) return 0;
    while (hi - lo > 1) {
        const int mid = lo + (hi - lo) / 2;
        if (choose_segments(units, mid, sms) > 1) hi = mid; else lo = mid;
    }
    return hi;
}

gdn_status gdn_plan_query(int B, int T, int H, int dk, int dv, int n_seqs, int varlen, gdn_dtype dtype,
                          const gdn_options *opts, gdn_plan_info *out) {
    if (!out) return GDN_ERR_INVALID_ARG;
    HostPlan hp;
    const int sms = (opts && opts->sm_count > 0) ? opts->sm_count : device_sm_count();
    gdn_status st = make_plan(B, T, H, dk, dv, n_seqs, varlen, dtype, opts, sms, &hp);
    if (st != GDN_OK) return st;
    out->kernel = hp.kernel;
    out->cp_enabled = hp.cp;
    out->chunks_per_segment = hp.L;
    out->max_chunks = hp.lay.max_chunks;
    out->max_items = hp.lay.max_items;
    out->max_cp_slots = hp.lay.max_cp_slots;
    out->sm_count = hp.sms;
    out->grid_fused = hp.ov_cols > 0 ? hp.units + hp.ov_ctas : hp.grid;
    out->overlap_columns = hp.ov_cols;
    out->launches = hp.launches;
    out->workspace_bytes = hp.lay.total;
    return GDN_OK;
}

size_t gdn_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int n_seqs, int varlen, gdn_dtype dtype,
                                    const gdn_options *opts) {
    gdn_plan_info info;
    if (gdn_plan_query(B, T, H, dk, dv, n_seqs, varlen, dtype, opts, &info) != GDN_OK) return 0;
    return info.workspace_bytes;
}

gdn_status gdn_workspace_query(int B, int T, int H, int dk, int dv, int n_seqs, int varlen, gdn_dtype dtype,
                               const gdn_options *opts, gdn_workspace_layout *out) {
    if (!out) return GDN_ERR_INVALID_ARG;
    HostPlan hp;
    const int sms = (opts && opts->sm_count > 0) ? opts->sm_count : device_sm_count();
    gdn_status st = make_plan(B, T, H, dk, dv, n_seqs, varlen, dtype, opts, sms, &hp);
    if (st != GDN_OK) return st;
    out->error_word = hp.lay.err;
    out->gate_cumsum = hp.lay.G;
    out->chunk_totals = hp.lay.totals;
    out->head_flags = hp.lay.flags;
    out->tprime = hp.lay.tprime;
    out->chunk_table = hp.lay.chunks;
    out->num_chunks = hp.lay.num_chunks;
    out->items = hp.lay.items2;
    out->num_items = hp.lay.num_items;
    out->total = hp.lay.total;
    return GDN_OK;
}

gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                         const float *initial_state, const int32_t *cu_seqlens, int n_seqs, float scale,
                         int B, int T, int H, int dk, int dv, gdn_dtype dtype, void *o, float *final_state,
                         void *workspace, size_t workspace_bytes, const gdn_options *opts_in,
                         gdn_stream_t stream_in) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_in);
    gdn_options opts;
    if (opts_in) opts = *opts_in; else default_options(&opts);
    const int varlen = cu_seqlens != nullptr;
    HostPlan hp;
    const int sms = opts.sm_count > 0 ? opts.sm_count : device_sm_count();
    gdn_status st = make_plan(B, T, H, dk, dv, n_seqs, varlen, dtype, &opts, sms, &hp);
    if (st != GDN_OK) return st;
    if (!workspace || !final_state) return GDN_ERR_INVALID_ARG;
    if (hp.total_T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, g, beta, initial_state, o, final_state, workspace};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
    if (workspace_bytes < hp.lay.total) return GDN_ERR_WORKSPACE;
    if (!(opts.sw_eps > 0.f && opts.sw_eps < 1.f)) opts.sw_eps = 5.9604645e-08f;

    Problem p;
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.s0 = initial_state; p.cu = cu_seqlens;
    p.o = o; p.sf = final_state;
    p.B = B; p.T = T; p.H = H; p.dk = dk; p.dv = dv; p.N = hp.N; p.total_T = (int)hp.total_T;
    p.varlen = varlen; p.dtype = dtype;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)dk);
    p.timeout_probe = (opts.debug_checks & GDN_DEBUG_TIMEOUT_PROBE) ? 1 : 0;

    char *base = static_cast<char *>(workspace);
    const Layout &L = hp.lay;
    Workspace w;
    w.err = reinterpret_cast<int *>(base + L.err);
    w.counters = reinterpret_cast<int *>(base + L.counters);
    w.num_chunks = reinterpret_cast<int *>(base + L.num_chunks);
    w.num_items = reinterpret_cast<int *>(base + L.num_items);
    w.seqinfo = reinterpret_cast<int4 *>(base + L.seqinfo);
    w.chunks = reinterpret_cast<int4 *>(base + L.chunks);
    w.flags = reinterpret_cast<int *>(base + L.flags);
    w.G = reinterpret_cast<float *>(base + L.G);
    w.totals = reinterpret_cast<float *>(base + L.totals);
    w.tprime = base + L.tprime;
    w.items2 = reinterpret_cast<gdn_work_item *>(base + L.items2);
    w.items1 = reinterpret_cast<gdn_work_item *>(base + L.items1);
    w.scan_units = reinterpret_cast<int4 *>(base + L.scan_units);
    w.seq_order = reinterpret_cast<int *>(base + L.seq_order);
    w.cp_s = reinterpret_cast<float *>(base + L.cp_s);
    w.cp_m = reinterpret_cast<float *>(base + L.cp_m);
    w.items_tmp = varlen ? reinterpret_cast<gdn_work_item *>(base + L.items_tmp) : nullptr;
    w.max_chunks = L.max_chunks;
    w.max_items = L.max_items;
    w.max_items1 = L.max_items1;
    w.max_cp_slots = L.max_cp_slots;

    PlanParams pp;
    pp.L = hp.L;
    pp.cp_enabled = hp.cp;
    pp.sliding = opts.sliding ? 1 : 0;
    pp.ln_eps = logf(opts.sw_eps);
    pp.grid = hp.grid;
    {
        const gdn_plan_costs c = current_costs();
        pp.state_ratio = c.state_step_us / c.chunk_step_us;
        pp.scan_ratio = c.scan_step_us / c.chunk_step_us;
    }
    pp.transition = 0;

    const int stages = opts.stages ? opts.stages : (GDN_STAGE_PREP | GDN_STAGE_INVERSE | GDN_STAGE_CORRECTION |
                                                    GDN_STAGE_FUSED);
    cudaGetLastError();  // clear a stale error so it is not blamed on these launches
    if (opts.qk_l2norm) {
        // every later step reads the unit-norm copies in the workspace
        void *qn = base + L.qn, *kn = base + L.kn;
        if ((stages & GDN_STAGE_PREP) && hp.total_T > 0) {
            cudaError_t e = launch_qk_l2norm(q, k, qn, kn, hp.total_T * H, dk, dtype, kQkNormEps, stream);
            if (e != cudaSuccess) return cuda_fail("launch qk_l2norm", e);
        }
        p.q = qn;
        p.k = kn;
    }
    if (stages & GDN_STAGE_PREP) {
        // equal sequences without a split: every (sequence, head) is one whole
        // item, which the sequence-prep kernel lists itself
        const bool direct = !varlen && !hp.cp;
        cudaError_t e = launch_seqprep(p, w, direct, stream);
        if (e != cudaSuccess) return cuda_fail("launch seqprep", e);
        if (L.max_chunks > 0 && (e = launch_gate(p, w, stream)) != cudaSuccess) return cuda_fail("launch gate", e);
        if (!direct && (e = launch_plan(p, w, pp, stream)) != cudaSuccess) return cuda_fail("launch plan", e);
    }
    // with the overlap, the fused pass computes the inverse of chunk columns
    // [ov_c0, nc) and counts each column's finished units in `ready`
    const int ov_c0 = hp.nc - hp.ov_cols;
    FusedOverlap ov = {};
    if (hp.ov_cols > 0) {
        ov.chain_ctas = hp.units;
        ov.c0 = ov_c0;
        ov.nc = hp.nc;
        ov.expected = hp.units;
        ov.ready = reinterpret_cast<int *>(base + L.ready);
        ov.gate_scaled = 1;
        if (stages & GDN_STAGE_PREP) {
            cudaError_t e = cudaMemsetAsync(ov.ready, 0, (size_t)hp.nc * sizeof(int), stream);
            if (e != cudaSuccess) return cuda_fail("clear column counts", e);
        }
    }
    if ((stages & GDN_STAGE_INVERSE) && L.max_chunks > 0) {
        cudaError_t e = hp.ov_cols > 0 ? launch_inverse(p, w, true, stream, ov_c0, hp.nc)
                                       : launch_inverse(p, w, hp.kernel == GDN_KERNEL_TC, stream);
        if (e != cudaSuccess) return cuda_fail("launch inverse", e);
    }
    const bool tc = hp.kernel == GDN_KERNEL_TC;
    if (hp.cp && (stages & GDN_STAGE_CORRECTION)) {
        cudaError_t e = tc ? launch_fused_tc(p, w, 1, hp.grid, stream) : launch_fused_simt(p, w, 1, hp.grid, stream);
        if (e != cudaSuccess) return cuda_fail(tc ? "launch fused_tc pass 1" : "launch fused_simt pass 1", e);
        if ((e = launch_scan(p, w, stream)) != cudaSuccess) return cuda_fail("launch scan", e);
    }
    if (stages & GDN_STAGE_FUSED) {
        cudaError_t e;
        if (opts.prof_begin &&
            (e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(opts.prof_begin), stream)) != cudaSuccess)
            return cuda_fail("record prof_begin", e);
        if (!tc) {
            e = launch_fused_simt(p, w, 2, hp.grid, stream);
        } else if (hp.ov_cols > 0) {
            e = launch_fused_tc(p, w, 2, hp.units + hp.ov_ctas, stream, &ov);
            if (e == cudaErrorCooperativeLaunchTooLarge) {
                // the SMs are not all free: the whole inverse first, then the plain pass
                cudaGetLastError();
                if ((e = launch_inverse(p, w, true, stream)) == cudaSuccess)
                    e = launch_fused_tc(p, w, 2, hp.grid, stream);
            }
        } else {
            e = launch_fused_tc(p, w, 2, hp.grid, stream);
        }
        if (e != cudaSuccess) return cuda_fail(tc ? "launch fused_tc pass 2" : "launch fused_simt pass 2", e);
        if (opts.prof_end && (e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(opts.prof_end), stream)) != cudaSuccess)
            return cuda_fail("record prof_end", e);
    }
    return GDN_OK;
}

// ---------------------------------------------------------------------------
// Inter-card sequence parallelism: the affine map of a slice, and the scan of
// start states over the ranks' maps.

namespace {

// The forward pass's layout (no CP) plus a correction-item list of two items
// per (sequence, head); the maps go straight to the caller's outputs.
gdn_status transition_plan(int B, int T, int H, int dk, int dv, int n_seqs, int varlen, int dtype, HostPlan *hp) {
    gdn_options o;
    default_options(&o);
    o.cp_mode = GDN_CP_OFF;
    gdn_status st = make_plan(B, T, H, dk, dv, n_seqs, varlen, dtype, &o, device_sm_count(), hp);
    if (st != GDN_OK) return st;
    Layout &L = hp->lay;
    const long long pairs = 2LL * hp->N * H;
    if (pairs >= (1LL << 30)) return GDN_ERR_UNSUPPORTED;
    L.items1 = align_up(L.total, 256);
    L.max_items1 = (int)pairs;
    L.total = align_up(L.items1 + (size_t)pairs * sizeof(gdn_work_item), 256);
    return GDN_OK;
}

}  // namespace

size_t gdn_chunk_transition_workspace_size(int B, int T, int H, int dk, int dv, int n_seqs, int varlen,
                                           gdn_dtype dtype) {
    HostPlan hp;
    if (transition_plan(B, T, H, dk, dv, n_seqs, varlen, dtype, &hp) != GDN_OK) return 0;
    return hp.lay.total;
}

gdn_status gdn_chunk_transition(const void *k, const void *v, const float *g, const float *beta,
                                const int32_t *cu_seqlens, int n_seqs, int B, int T, int H, int dk, int dv,
                                gdn_dtype dtype, float *s_star, float *m, void *workspace, size_t workspace_bytes,
                                gdn_stream_t stream_in) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_in);
    const int varlen = cu_seqlens != nullptr;
    HostPlan hp;
    gdn_status st = transition_plan(B, T, H, dk, dv, n_seqs, varlen, dtype, &hp);
    if (st != GDN_OK) return st;
    if (!workspace || !s_star || !m) return GDN_ERR_INVALID_ARG;
    if (hp.total_T > 0 && (!k || !v || !g || !beta)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {k, v, g, beta, s_star, m, workspace};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
    if (workspace_bytes < hp.lay.total) return GDN_ERR_WORKSPACE;

    Problem p;
    memset(&p, 0, sizeof(p));
    p.q = k;   // the correction items read no queries; any tile of the right shape will do
    p.k = k; p.v = v; p.g = g; p.beta = beta; p.s0 = nullptr; p.cu = cu_seqlens;
    p.o = nullptr; p.sf = nullptr;
    p.B = B; p.T = T; p.H = H; p.dk = dk; p.dv = dv; p.N = hp.N; p.total_T = (int)hp.total_T;
    p.varlen = varlen; p.dtype = dtype;
    p.scale = 1.0f / sqrtf((float)dk);
    p.timeout_probe = 0;

    char *base = static_cast<char *>(workspace);
    const Layout &L = hp.lay;
    Workspace w;
    memset(&w, 0, sizeof(w));
    w.err = reinterpret_cast<int *>(base + L.err);
    w.counters = reinterpret_cast<int *>(base + L.counters);
    w.num_chunks = reinterpret_cast<int *>(base + L.num_chunks);
    w.num_items = reinterpret_cast<int *>(base + L.num_items);
    w.seqinfo = reinterpret_cast<int4 *>(base + L.seqinfo);
    w.chunks = reinterpret_cast<int4 *>(base + L.chunks);
    w.flags = reinterpret_cast<int *>(base + L.flags);
    w.G = reinterpret_cast<float *>(base + L.G);
    w.totals = reinterpret_cast<float *>(base + L.totals);
    w.tprime = base + L.tprime;
    w.items2 = reinterpret_cast<gdn_work_item *>(base + L.items2);
    w.items1 = reinterpret_cast<gdn_work_item *>(base + L.items1);
    w.scan_units = reinterpret_cast<int4 *>(base + L.scan_units);
    w.seq_order = reinterpret_cast<int *>(base + L.seq_order);
    w.cp_s = s_star;   // slot n H + h of the correction pass is unit (n, h) of the outputs
    w.cp_m = m;
    w.max_chunks = L.max_chunks;
    w.max_items = L.max_items;
    w.max_items1 = L.max_items1;
    w.max_cp_slots = hp.N * H;

    PlanParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.L = hp.L;
    pp.cp_enabled = 0;
    pp.sliding = 0;
    pp.ln_eps = logf(5.9604645e-08f);
    pp.grid = hp.grid;
    pp.state_ratio = 1.f;
    pp.scan_ratio = 1.f;
    pp.transition = 1;

    cudaGetLastError();
    cudaError_t e = launch_seqprep(p, w, false, stream);
    if (e != cudaSuccess) return cuda_fail("launch seqprep", e);
    if (L.max_chunks > 0 && (e = launch_gate(p, w, stream)) != cudaSuccess) return cuda_fail("launch gate", e);
    if ((e = launch_plan(p, w, pp, stream)) != cudaSuccess) return cuda_fail("launch plan", e);
    const bool tc = hp.kernel == GDN_KERNEL_TC;
    if (L.max_chunks > 0 && (e = launch_inverse(p, w, tc, stream)) != cudaSuccess)
        return cuda_fail("launch inverse", e);
    e = tc ? launch_fused_tc(p, w, 1, hp.grid, stream) : launch_fused_simt(p, w, 1, hp.grid, stream);
    if (e != cudaSuccess) return cuda_fail(tc ? "launch fused_tc (transition)" : "launch fused_simt (transition)", e);
    return GDN_OK;
}

namespace {

gdn_status state_scan_any(const float *s0, const float *s_star, const float *m, int R, int N, int H, int dk, int dv,
                          float *s_start, bool grad, gdn_stream_t stream) {
    if (R < 1 || N < 0 || H < 1 || (long long)N * H >= (1LL << 30)) return GDN_ERR_INVALID_ARG;
    if (!valid_head_dim(dk) || !valid_head_dim(dv)) return GDN_ERR_UNSUPPORTED;
    if (!s_start || (R > 1 && (!s_star || !m))) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {s0, s_star, m, s_start};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
    // the output must not overlap an input (the walk reads the maps while it writes)
    const size_t out_bytes = (size_t)R * N * H * dk * dv * 4;
    auto overlaps = [&](const void *a, size_t bytes) {
        if (!a) return false;
        const char *x = static_cast<const char *>(a), *y = reinterpret_cast<const char *>(s_start);
        return x < y + out_bytes && y < x + bytes;
    };
    if (overlaps(s0, (size_t)N * H * dk * dv * 4) || overlaps(s_star, out_bytes) ||
        overlaps(m, (size_t)R * N * H * dk * dk * 4))
        return GDN_ERR_INVALID_ARG;
    cudaGetLastError();
    cudaError_t e =
        launch_rank_scan(s0, s_star, m, R, N, H, dk, dv, s_start, grad, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("launch rank scan", e);
    return GDN_OK;
}

}  // namespace

gdn_status gdn_state_scan(const float *s0, const float *s_star, const float *m, int R, int N, int H, int dk, int dv,
                          float *s_start, gdn_stream_t stream) {
    return state_scan_any(s0, s_star, m, R, N, H, dk, dv, s_start, false, stream);
}

gdn_status gdn_state_grad_scan(const float *ds_last, const float *ds_star, const float *m, int R, int N, int H,
                               int dk, int dv, float *ds_end, gdn_stream_t stream) {
    return state_scan_any(ds_last, ds_star, m, R, N, H, dk, dv, ds_end, true, stream);
}

gdn_status gdn_chunk_fwd_check(const void *workspace, gdn_stream_t stream) {
    if (!workspace) return GDN_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("stream synchronize", e);
    int word = 0;
    if ((e = cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail("read error word", e);
    if (word == 0) return GDN_OK;
    if (word == GDN_ERR_TIMEOUT) return GDN_ERR_TIMEOUT;
    return GDN_ERR_DEVICE_CHECK;
}

namespace {
// The host-buffer entry point streams a large problem through in parts: the
// copies of part p+1 in, the pass on part p and the copies of part p-1 out
// overlap on three streams.  A part is a group of whole sequences, or, when
// there are fewer sequences than parts and the plan runs every (sequence,
// head) as one unit, a piece of one sequence (64-token aligned) that carries
// the state of the previous piece through a device buffer.
constexpr int kMaxHostParts = 8;
constexpr size_t kHostSplitBytes = size_t(64) << 20;   // below this, one part

struct HostLayout {
    size_t q, k, v, g, beta, s0, cu, o, sf, mid, status, ws, total;
};

bool host_layout(int B, int T, int H, int dk, int dv, int n_seqs, int varlen, int has_s0, int dtype,
                 const gdn_options *opts, HostLayout *hl, size_t *ws_bytes) {
    gdn_plan_info info;
    if (gdn_plan_query(B, T, H, dk, dv, n_seqs, varlen, (gdn_dtype)dtype, opts, &info) != GDN_OK) return false;
    const size_t e = dtype == GDN_BF16 ? 2 : 4;
    const size_t ntok = varlen ? (size_t)T : (size_t)B * T;
    const size_t N = varlen ? (size_t)n_seqs : (size_t)B;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    hl->q = take(ntok * H * dk * e);
    hl->k = take(ntok * H * dk * e);
    hl->v = take(ntok * H * dv * e);
    hl->g = take(ntok * H * 4);
    hl->beta = take(ntok * H * 4);
    hl->s0 = take(has_s0 ? N * H * dk * dv * 4 : 0);
    hl->cu = take(varlen ? (N + 1 + kMaxHostParts) * 4 : 0);   // each part's rebased cu_seqlens
    hl->o = take(ntok * H * dv * e);
    hl->sf = take(N * H * dk * dv * 4);
    hl->mid = take(varlen ? 0 : 2 * N * H * dk * dv * 4);       // states between pieces of a sequence
    hl->status = take(kMaxHostParts * 4);                       // each part's device status word
    hl->ws = take(info.workspace_bytes);
    hl->total = off;
    *ws_bytes = info.workspace_bytes;
    return true;
}
}  // namespace

size_t gdn_chunk_fwd_host_buffer_size(int B, int T, int H, int dk, int dv, int n_seqs, int varlen,
                                      int has_initial_state, gdn_dtype dtype, const gdn_options *opts) {
    HostLayout hl;
    size_t ws = 0;
    if (!host_layout(B, T, H, dk, dv, n_seqs, varlen, has_initial_state, dtype, opts, &hl, &ws)) return 0;
    return hl.total;
}

namespace {
// Copy streams of the host-buffer entry point, created once per device.
struct HostStreams {
    cudaStream_t in = nullptr, out = nullptr;
};
std::mutex g_host_streams_mu;
HostStreams g_host_streams[64];

gdn_status host_streams(HostStreams *hs) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("host entry: cudaGetDevice", e);
    if (dev < 0 || dev >= 64) return GDN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_host_streams_mu);
    HostStreams &h = g_host_streams[dev];
    if (!h.in && (e = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail("host entry: create copy-in stream", e);
    if (!h.out && (e = cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail("host entry: create copy-out stream", e);
    *hs = h;
    return GDN_OK;
}

struct HostPart {
    int s0, s1;           // sequences [s0, s1)
    size_t t0, ntok;      // tokens [t0, t0 + ntok) of the token axis
    int Tp;               // tokens per sequence (batched) or packed tokens (varlen)
    int src, dst;         // state in: -1 the caller's initial state, 0/1 a middle buffer;
                          // state out: -1 final_state, 0/1 a middle buffer
};
}  // namespace

gdn_status gdn_chunk_fwd_host(const void *q, const void *k, const void *v, const float *g, const float *beta,
                              const float *initial_state, const int32_t *cu_seqlens, int n_seqs, float scale,
                              int B, int T, int H, int dk, int dv, gdn_dtype dtype, void *o, float *final_state,
                              void *device_buffer, size_t device_buffer_bytes, const gdn_options *opts,
                              gdn_stream_t stream_in) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_in);
    const int varlen = cu_seqlens != nullptr;
    HostLayout hl;
    size_t ws_bytes = 0;
    if (!host_layout(B, T, H, dk, dv, n_seqs, varlen, initial_state != nullptr, dtype, opts, &hl, &ws_bytes))
        return GDN_ERR_INVALID_ARG;
    if (!device_buffer || !final_state) return GDN_ERR_INVALID_ARG;
    if (device_buffer_bytes < hl.total) return GDN_ERR_WORKSPACE;
    const size_t e = dtype == GDN_BF16 ? 2 : 4;
    const size_t ntok = varlen ? (size_t)T : (size_t)B * T;
    const int N = varlen ? n_seqs : B;
    if (ntok > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    const size_t tok_in = (size_t)H * ((2 * dk + dv) * e + 8);   // input bytes per token
    const size_t state = (size_t)H * dk * dv * 4;                // bytes per sequence state

    // Every part runs with the whole problem's plan decisions (CP on or off, the
    // same segment length), so each fits the workspace sized for the whole and
    // gives the whole problem's result.
    gdn_plan_info full;
    if (gdn_plan_query(B, T, H, dk, dv, n_seqs, varlen, dtype, opts, &full) != GDN_OK) return GDN_ERR_INVALID_ARG;
    gdn_options po;
    if (opts) po = *opts; else default_options(&po);
    po.cp_mode = full.cp_enabled ? GDN_CP_FORCE : GDN_CP_OFF;
    po.chunks_per_segment = full.cp_enabled ? full.chunks_per_segment : 0;
    po.sm_count = full.sm_count;

    // Parts.
    HostPart parts[kMaxHostParts];
    int P = 0;
    const bool big = ntok * tok_in >= kHostSplitBytes;
    int want = big ? std::min(N, kMaxHostParts) : 1;
    if (varlen && want > 1) {
        // splitting needs well-formed offsets; otherwise one part, and the
        // device check reports the bad cu_seqlens as it does for gdn_chunk_fwd
        for (int i = 0; i <= N && want > 1; ++i)
            if ((i == 0 && cu_seqlens[0] != 0) || (i > 0 && cu_seqlens[i] < cu_seqlens[i - 1]) ||
                (i == N && (size_t)cu_seqlens[N] != ntok))
                want = 1;
    }
    const int pieces = (!varlen && big && !full.cp_enabled && N < kMaxHostParts)
                           ? std::max(1, std::min(kMaxHostParts / N, T / 64))
                           : 1;
    if (varlen && want == 1) {
        parts[P++] = {0, N, 0, ntok, T, -1, -1};
    } else if (varlen) {
        int s = 0;
        for (int p = 0; p < want && s < N; ++p) {
            int s1 = N;
            if (p + 1 < want) {
                const size_t target = ntok * (size_t)(p + 1) / want;
                s1 = s + 1;
                while (s1 < N && (size_t)cu_seqlens[s1] < target) ++s1;
            }
            const size_t t0 = cu_seqlens[s], n = cu_seqlens[s1] - cu_seqlens[s];
            parts[P++] = {s, s1, t0, n, (int)n, -1, -1};
            s = s1;
        }
    } else if (pieces > 1) {
        // each sequence in `pieces` pieces of whole chunks, in order
        for (int b = 0; b < N; ++b) {
            int u0 = 0, j = 0;
            for (int q = 1; q <= pieces; ++q) {
                const int u1 = q == pieces ? T : (int)(((long long)T * q / pieces) / 64 * 64);
                if (u1 <= u0) continue;
                const bool last = u1 == T;
                parts[P++] = {b, b + 1, (size_t)b * T + u0, (size_t)(u1 - u0), u1 - u0, j == 0 ? -1 : (j - 1) & 1,
                              last ? -1 : j & 1};
                u0 = u1;
                ++j;
            }
        }
    } else {
        for (int p = 0; p < want; ++p) {
            const int s0 = (int)((long long)N * p / want), s1 = (int)((long long)N * (p + 1) / want);
            if (s1 > s0) parts[P++] = {s0, s1, (size_t)s0 * T, (size_t)(s1 - s0) * T, T, -1, -1};
        }
    }

    HostStreams hs;
    gdn_status st = host_streams(&hs);
    if (st != GDN_OK) return st;
    cudaGetLastError();
    char *d = static_cast<char *>(device_buffer);
    cudaEvent_t ev_start = nullptr, ev_in[kMaxHostParts] = {}, ev_done[kMaxHostParts] = {};
    auto make_event = [](cudaEvent_t *ev) { return cudaEventCreateWithFlags(ev, cudaEventDisableTiming); };
    cudaError_t ce = make_event(&ev_start);
    for (int p = 0; p < P && ce == cudaSuccess; ++p) {
        ce = make_event(&ev_in[p]);
        if (ce == cudaSuccess) ce = make_event(&ev_done[p]);
    }
    // each part's cu_seqlens, rebased to start at 0, one after another in the
    // device buffer (offsets in int32 elements)
    size_t cu_off[kMaxHostParts] = {};
    for (int p = 1; p < P; ++p) cu_off[p] = cu_off[p - 1] + (parts[p - 1].s1 - parts[p - 1].s0) + 1;

    // the device buffer may still be in use by work enqueued on `stream` before this call
    if (ce == cudaSuccess) ce = cudaEventRecord(ev_start, stream);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(hs.in, ev_start, 0);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(hs.out, ev_start, 0);
    // the parts' offsets first, through a small stack array (a copy from pageable
    // memory has read its source when cudaMemcpyAsync returns, and waits for the
    // stream, which is still empty of this call's large copies here)
    for (int p = 0; p < P && varlen && ce == cudaSuccess; ++p) {
        const size_t ns = parts[p].s1 - parts[p].s0;
        int32_t stage[256];
        for (size_t i = 0; i <= ns && ce == cudaSuccess; i += 256) {
            const size_t n = std::min<size_t>(256, ns + 1 - i);
            // (one part: the caller's values as they are, so that the device
            // check still sees a malformed array)
            const int32_t base = P > 1 ? cu_seqlens[parts[p].s0] : 0;
            for (size_t t = 0; t < n; ++t) stage[t] = cu_seqlens[parts[p].s0 + i + t] - base;
            ce = cudaMemcpyAsync(d + hl.cu + (cu_off[p] + i) * 4, stage, n * 4, cudaMemcpyHostToDevice, hs.in);
        }
    }
    // copies in, part by part
    for (int p = 0; p < P && ce == cudaSuccess; ++p) {
        const HostPart &pt = parts[p];
        const size_t ns = pt.s1 - pt.s0;
        struct Copy { size_t dst; const void *src; size_t off, n; };
        const Copy in[] = {
            {hl.q, q, pt.t0 * H * dk * e, pt.ntok * H * dk * e},
            {hl.k, k, pt.t0 * H * dk * e, pt.ntok * H * dk * e},
            {hl.v, v, pt.t0 * H * dv * e, pt.ntok * H * dv * e},
            {hl.g, g, pt.t0 * H * 4, pt.ntok * H * 4},
            {hl.beta, beta, pt.t0 * H * 4, pt.ntok * H * 4},
            {hl.s0, initial_state, (size_t)pt.s0 * state, (initial_state && pt.src < 0) ? ns * state : 0},
        };
        for (const Copy &c : in)
            if (ce == cudaSuccess && c.n)
                ce = cudaMemcpyAsync(d + c.dst + c.off, static_cast<const char *>(c.src) + c.off, c.n,
                                     cudaMemcpyHostToDevice, hs.in);
        if (ce == cudaSuccess) ce = cudaEventRecord(ev_in[p], hs.in);
    }
    // the pass on each part as soon as its inputs are in; its results out on the third stream
    for (int p = 0; p < P && ce == cudaSuccess && st == GDN_OK; ++p) {
        const HostPart &pt = parts[p];
        const int ns = pt.s1 - pt.s0;
        ce = cudaStreamWaitEvent(stream, ev_in[p], 0);
        if (ce != cudaSuccess) break;
        const int Bp = varlen ? 1 : ns;
        const float *s_in = pt.src >= 0 ? reinterpret_cast<float *>(d + hl.mid + ((size_t)pt.src * N + pt.s0) * state)
                            : initial_state ? reinterpret_cast<float *>(d + hl.s0 + (size_t)pt.s0 * state)
                                            : nullptr;
        float *s_out = pt.dst >= 0 ? reinterpret_cast<float *>(d + hl.mid + ((size_t)pt.dst * N + pt.s0) * state)
                                   : reinterpret_cast<float *>(d + hl.sf + (size_t)pt.s0 * state);
        st = gdn_chunk_fwd(d + hl.q + pt.t0 * H * dk * e, d + hl.k + pt.t0 * H * dk * e,
                           d + hl.v + pt.t0 * H * dv * e, reinterpret_cast<float *>(d + hl.g) + pt.t0 * H,
                           reinterpret_cast<float *>(d + hl.beta) + pt.t0 * H, s_in,
                           varlen ? reinterpret_cast<int32_t *>(d + hl.cu) + cu_off[p] : nullptr, ns, scale, Bp,
                           pt.Tp, H, dk, dv, dtype, d + hl.o + pt.t0 * H * dv * e, s_out, d + hl.ws, ws_bytes, &po,
                           stream_in);
        if (st != GDN_OK) break;
        // keep this part's device status: the next part's pass starts by clearing the word
        ce = cudaMemcpyAsync(d + hl.status + 4 * p, d + hl.ws, 4, cudaMemcpyDeviceToDevice, stream);
        if (ce == cudaSuccess) ce = cudaEventRecord(ev_done[p], stream);
        if (ce == cudaSuccess) ce = cudaStreamWaitEvent(hs.out, ev_done[p], 0);
        if (ce == cudaSuccess && pt.ntok)
            ce = cudaMemcpyAsync(static_cast<char *>(o) + pt.t0 * H * dv * e, d + hl.o + pt.t0 * H * dv * e,
                                 pt.ntok * H * dv * e, cudaMemcpyDeviceToHost, hs.out);
        if (ce == cudaSuccess && pt.dst < 0)
            ce = cudaMemcpyAsync(reinterpret_cast<char *>(final_state) + (size_t)pt.s0 * state,
                                 d + hl.sf + (size_t)pt.s0 * state, (size_t)ns * state, cudaMemcpyDeviceToHost,
                                 hs.out);
    }
    // everything this call enqueued has finished before it returns
    const cudaError_t e_in = cudaStreamSynchronize(hs.in);
    const cudaError_t e_run = cudaStreamSynchronize(stream);
    const cudaError_t e_out = cudaStreamSynchronize(hs.out);
    int status[kMaxHostParts] = {};
    cudaError_t e_st = cudaSuccess;
    if (ce == cudaSuccess && st == GDN_OK && e_in == cudaSuccess && e_run == cudaSuccess && e_out == cudaSuccess)
        e_st = cudaMemcpy(status, d + hl.status, 4 * P, cudaMemcpyDeviceToHost);
    if (ev_start) cudaEventDestroy(ev_start);
    for (int p = 0; p < P; ++p) {
        if (ev_in[p]) cudaEventDestroy(ev_in[p]);
        if (ev_done[p]) cudaEventDestroy(ev_done[p]);
    }
    if (st != GDN_OK) return st;
    if (ce != cudaSuccess) return cuda_fail("host entry: copy or event", ce);
    if (e_in != cudaSuccess) return cuda_fail("host entry: synchronize copy-in stream", e_in);
    if (e_run != cudaSuccess) return cuda_fail("host entry: synchronize stream", e_run);
    if (e_out != cudaSuccess) return cuda_fail("host entry: synchronize copy-out stream", e_out);
    if (e_st != cudaSuccess) return cuda_fail("host entry: read status", e_st);
    for (int p = 0; p < P; ++p) {
        if (status[p] == GDN_ERR_TIMEOUT) return GDN_ERR_TIMEOUT;
        if (status[p] != 0) return GDN_ERR_DEVICE_CHECK;
    }
    return GDN_OK;
}

const char *gdn_status_string(gdn_status s) {
    switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_DEVICE_CHECK: return "GDN_ERR_DEVICE_CHECK";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    }
    return "GDN_ERR_UNKNOWN";
}

const char *gdn_version(void) { return "gdn-gb300 0.1 (sm_103a)"; }

const char *gdn_last_error_detail(void) { return g_error_detail; }

}  // extern "C"
