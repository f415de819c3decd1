// Sequence preparation, the gate kernel and the device-side work planner.
//
// Gate kernel (FlashQLA talk "Qwen系列模型线性注意力高性能优化实践": the Gamma
// paragraph keeps the in-chunk gate product in log space, the SFU paragraph
// writes Gamma_{st} = exp(G_s - G_t); the sliding-window paragraph launches a
// light kernel that scans each head's gate to find the heads whose alpha is not
// identically 1): chunk-local inclusive cumsum G of g, per-chunk totals, and a
// per-(sequence, head) flag "some g != 0".
//
// Planner (compute-for-memory, auto-CP and sliding-window paragraphs): splits
// each (sequence, head) unit into segments of at most L chunks, orders the work
// longest sequence first, and gives each later segment either a look-back
// restart (flagged heads) or correction-matrix work plus a scan (alpha == 1
// heads).  It runs on the device so no cu_seqlens or gate data crosses to the
// host.
#include <limits.h>

#include "gdn_internal.cuh"

namespace gdn {

// ---------------------------------------------------------------------------
// Sequence preparation: validate cu_seqlens, build the per-sequence table and
// the chunk table, zero the counters and head flags.  One CTA.  With
// emit_items (equal sequences, no split) it also writes the output pass's work
// list, one whole-sequence item per (sequence, head), so that no planner
// launch is needed.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) seqprep_kernel(const __grid_constant__ Problem p, const __grid_constant__ Workspace w,
                                                       int emit_items) {
    grid_dependency_wait();
    __shared__ int s_bad;
    __shared__ int s_carry;
    __shared__ int s_warp[32];
    const int tid = threadIdx.x;
    const int N = p.N;
    if (tid == 0) {
        s_bad = 0;
        s_carry = 0;
        *w.err = 0;
        *w.num_chunks = 0;
    }
    if (tid < 8) w.counters[tid] = 0;
    if (tid < 4) w.num_items[tid] = 0;
    for (int i = tid; i < N * p.H; i += blockDim.x) w.flags[i] = 0;
    __syncthreads();
    if (p.varlen) {
        for (int n = tid; n <= N; n += blockDim.x) {
            int a = p.cu[n];
            bool bad = (n == 0 && a != 0) || (n == N && a != p.total_T) || a < 0 || a > p.total_T;
            if (n < N && p.cu[n + 1] < a) bad = true;
            if (bad) s_bad = 1;
        }
        __syncthreads();
        if (s_bad) {
            if (tid == 0) report_error(w.err, GDN_ERR_DEVICE_CHECK);
            return;
        }
    }
    // exclusive scan of chunk counts over sequences, 1024 at a time
    for (int base = 0; base < N; base += blockDim.x) {
        int n = base + tid;
        int t0 = 0, len = 0, nc = 0;
        if (n < N) {
            t0 = p.varlen ? p.cu[n] : n * p.T;
            len = p.varlen ? p.cu[n + 1] - t0 : p.T;
            nc = (len + kChunk - 1) / kChunk;
        }
        // block inclusive scan of nc
        int x = nc;
        const int lane = tid & 31, wid = tid >> 5;
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int y = s_warp[lane];
            for (int off = 1; off < 32; off <<= 1) {
                int z = __shfl_up_sync(0xffffffffu, y, off);
                if (lane >= off) y += z;
            }
            s_warp[lane] = y;
        }
        __syncthreads();
        int incl = x + (wid > 0 ? s_warp[wid - 1] : 0);
        int carry = s_carry;
        if (n < N) w.seqinfo[n] = make_int4(t0, len, carry + incl - nc, nc);
        __syncthreads();
        if (tid == blockDim.x - 1) s_carry = carry + incl;
        __syncthreads();
    }
    const int total = s_carry;
    if (total > w.max_chunks) {  // cannot happen for consistent sizes; never overrun the table
        if (tid == 0) report_error(w.err, GDN_ERR_DEVICE_CHECK);
        return;
    }
    __syncthreads();
    // chunk table: binary search the sequence of every chunk
    for (int c = tid; c < total; c += blockDim.x) {
        int lo = 0, hi = N - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (w.seqinfo[mid].z <= c) lo = mid; else hi = mid - 1;
        }
        // skip empty sequences that share the same first chunk
        while (lo + 1 < N && w.seqinfo[lo + 1].z <= c) ++lo;
        int4 si = w.seqinfo[lo];
        int ci = c - si.z;
        int t0 = si.x + ci * kChunk;
        int len = min(kChunk, si.x + si.y - t0);
        w.chunks[c] = make_int4(lo, t0, len, ci);
    }
    if (emit_items) {
        const int units = N * p.H;
        for (int u = tid; u < units && u < w.max_items; u += blockDim.x) {
            gdn_work_item it;
            it.seq = u / p.H;
            it.head = u % p.H;
            it.c_begin = it.c_start = 0;
            it.c_end = w.seqinfo[it.seq].w;
            it.flags = GDN_ITEM_OUTPUT | GDN_ITEM_FROM_INITIAL | GDN_ITEM_WRITE_FINAL;
            it.slot = -1;
            it.pad = 0;
            w.items2[u] = it;
        }
        if (tid == 0) {
            const bool fits = units <= w.max_items;
            if (!fits) report_error(w.err, GDN_ERR_DEVICE_CHECK);
            w.num_items[0] = fits ? units : 0;
            w.num_items[1] = 0;
            w.num_items[2] = 0;
        }
    }
    if (tid == 0) *w.num_chunks = total;
}

// ---------------------------------------------------------------------------
// Gate: one CTA per (chunk, group of 64 heads).
// ---------------------------------------------------------------------------
constexpr int kGateHeads = 64;

__global__ void __launch_bounds__(256) gate_kernel(const __grid_constant__ Problem p, const __grid_constant__ Workspace w) {
    __shared__ float tile[kChunk][kGateHeads + 1];
    __shared__ int s_nz[kGateHeads];
    const int cid = blockIdx.x;
    int4 ci;
    if (!p.varlen) {
        // equal sequences: the chunk's place follows from its index, so the
        // gate values are read while the sequence-prep kernel still runs
        // (programmatic dependent launch), and only the writes wait for it
        const int ncs = (p.T + kChunk - 1) / kChunk;
        const int seq = cid / ncs, c = cid - seq * ncs;
        ci = make_int4(seq, seq * p.T + c * kChunk, min(kChunk, p.T - c * kChunk), c);
    } else {
        grid_dependency_wait();
        if (cid >= *w.num_chunks) return;
        ci = w.chunks[cid];
    }
    const int t0 = ci.y, len = ci.z;
    const int h0 = blockIdx.y * kGateHeads;
    const int nh = min(kGateHeads, p.H - h0);
    for (int idx = threadIdx.x; idx < kChunk * nh; idx += blockDim.x) {
        int r = idx / nh, hh = idx % nh;
        tile[r][hh] = r < len ? p.g[(size_t)(t0 + r) * p.H + h0 + hh] : 0.f;
    }
    if (!p.varlen) grid_dependency_wait();   // the head flags are zeroed by the sequence-prep kernel
    __syncthreads();
    // one warp per head: lane l holds rows 2l and 2l+1; a shuffle scan of the
    // pair sums gives the inclusive cumsum (rows past the end are zero in the
    // tile, so they keep the last cumsum)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int hh = warp; hh < nh; hh += blockDim.x >> 5) {
        const float x0 = tile[2 * lane][hh], x1 = tile[2 * lane + 1][hh];
        float incl = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const float excl = incl - (x0 + x1);
        tile[2 * lane][hh] = excl + x0;
        tile[2 * lane + 1][hh] = incl;
        const bool nz = __any_sync(0xffffffffu, x0 != 0.f || x1 != 0.f);
        if (lane == 31) w.totals[(size_t)(h0 + hh) * w.max_chunks + cid] = incl;
        if (lane == 0) s_nz[hh] = nz;
    }
    __syncthreads();
    for (int hh = threadIdx.x; hh < nh; hh += blockDim.x)
        if (s_nz[hh]) w.flags[ci.x * p.H + h0 + hh] = 1;
    for (int idx = threadIdx.x; idx < kChunk * nh; idx += blockDim.x) {
        int hh = idx / kChunk, r = idx % kChunk;
        if (r < len) w.G[(size_t)(h0 + hh) * p.total_T + t0 + r] = tile[r][hh];
    }
}

// ---------------------------------------------------------------------------
// Planner: one CTA builds the work lists, in steps: (1) sequences ordered
// longest first; (2) the segment count of the units that take correction
// matrices (a cost search over the counts); (3) per (sequence, head) unit its
// segments, their look-back windows (walked by lane groups) or correction
// slots, and the items of the output pass, the correction pass and the scan;
// (4) for packed sequences, the output list dealt out longest first.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int block_exclusive_scan(int x, int *s_warp, int *s_total) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nw = (blockDim.x + 31) >> 5;
    int incl = x;
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int y = lane < nw ? s_warp[lane] : 0;
        for (int off = 1; off < 32; off <<= 1) {
            int z = __shfl_up_sync(0xffffffffu, y, off);
            if (lane >= off) y += z;
        }
        s_warp[lane] = y;
        if (lane == 31) *s_total = y;
    }
    __syncthreads();
    int excl = incl - x + (wid > 0 ? s_warp[wid - 1] : 0);
    __syncthreads();
    return excl;
}

// Look-back window for the segment starting at chunk c_begin of a unit: the
// least number of whole chunks whose summed gate is <= ln_eps, or the whole
// prefix.  Returns -1 when more than max_walk chunks would be needed (the unit
// then takes the exact correction-matrix path instead).  Walked by a group of
// W lanes (mask: the group's lanes): the group loads W chunk totals at once,
// then adds them one by one in the walk's order (every lane holds the same
// sum), so a window of n chunks costs ceil(n / W) memory round trips instead
// of n, with the sums rounded exactly as a one-thread walk rounds them.
template <int W>
__device__ int lookback_window(const Workspace &w, int h, int chunk0, int c_begin, float ln_eps, int max_walk,
                               unsigned mask) {
    const int sub = threadIdx.x & (W - 1);
    const float *tot = w.totals + (size_t)h * w.max_chunks + chunk0;   // chunk c_begin - 1 - i at i
    float acc = 0.f;
    for (int base = 0;; base += W) {
        const int i = base + sub;
        const float t = (i < c_begin && i < max_walk) ? tot[c_begin - 1 - i] : 0.f;
        for (int l = 0; l < W; ++l) {
            const int wnd = base + l;       // chunks summed so far
            if (wnd >= c_begin) return wnd;
            if (wnd >= max_walk) return -1;
            acc += __shfl_sync(mask, t, l, W);
            if (acc <= ln_eps) return wnd + 1;
        }
    }
}

constexpr int kMaxLookbackChunks = 256;
constexpr int kLptItems = 2048;     // longest-first dealing: at most this many output-pass items
constexpr int kLptCtas = 1024;      // and this many CTAs

// Ascending bitonic sort of n (a power of two) 64-bit keys in shared memory by
// the whole block; every thread calls it, after the keys are in place.
__device__ void bitonic_sort_u64(unsigned long long *k, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int l = i ^ stride;
                if (l > i) {
                    const unsigned long long a = k[i], b = k[l];
                    if ((a > b) == ((i & size) == 0)) {
                        k[i] = b;
                        k[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
}

constexpr int kPlanThreads = 1024;
constexpr int kWalkLanes = 8;       // lanes per look-back walk

// Segments per unit for the units that need correction matrices, when every
// unit has nc chunks and the planner's segment length gives NS0 segments.
// Per-pass cost model in output chunk steps of the persistent passes on `grid`
// CTAs (the talk's auto-CP paragraph: one-wave model T = lambda1 L +
// lambda2 N / L, refined per pass, with the measured step costs): pass 1 runs
// 2 NS - 3 state-only items per such unit (S* and M of every segment but the
// last, S* of the first), pass 2 one item per segment of every unit (n_s units
// keep NS0 segments and re-run a look-back of about four chunks), the scan one
// step per segment; a pass takes as many waves as its items need, each as long
// as its longest item.  Fewer, longer segments can save a whole wave of pass
// 1.  The planner keeps NS0 unless another count is at least 5% cheaper, and
// then takes the largest count of least cost; the block evaluates the counts
// side by side.
__device__ double correction_cost(int ns, int nc, int NS0, int n_m, int n_s, int grid, float state_ratio,
                                  float scan_ratio) {
    const int Ls = (nc + NS0 - 1) / NS0 + (n_s > 0 ? 4 : 0);
    const int Lm = (nc + ns - 1) / ns;
    const long long it1 = (long long)n_m * (2 * ns - 3);
    const long long it2 = (long long)n_m * ns + (long long)n_s * NS0;
    return (double)((it1 + grid - 1) / grid) * Lm * state_ratio +
           (double)((it2 + grid - 1) / grid) * max(Lm, n_s > 0 ? Ls : 0) + (double)scan_ratio * ns;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ Problem p, const __grid_constant__ Workspace w, const __grid_constant__ PlanParams pp) {
    grid_dependency_wait();
    __shared__ int s_warp[32];
    __shared__ int s_tot[4];
    __shared__ int s_base[4];
    const int tid = threadIdx.x;
    if (*w.err != 0) return;
    const int N = p.N, H = p.H;
    // 1. order sequences longest first (rank by counting; natural order when N is large)
    if (N <= 8192) {
        for (int n = tid; n < N; n += blockDim.x) {
            int mine = w.seqinfo[n].w;
            int rank = 0;
            for (int m = 0; m < N; ++m) {
                int o = w.seqinfo[m].w;
                rank += (o > mine) || (o == mine && m < n);
            }
            w.seq_order[rank] = n;
        }
    } else {
        for (int n = tid; n < N; n += blockDim.x) w.seq_order[n] = n;
    }
    if (tid < 4) s_base[tid] = 0;
    const int units = N * H;
    if (pp.transition) {
        // the affine map of every (sequence, head) over its whole sequence:
        // S* (values, from zero) and M (no values, from the identity), written
        // to slot n H + h of the caller's outputs; sequences longest first
        __syncthreads();
        for (int u = tid; u < units; u += blockDim.x) {
            const int seq = w.seq_order[u / H], h = u % H;
            gdn_work_item it;
            it.seq = seq;
            it.head = h;
            it.c_begin = it.c_start = 0;
            it.c_end = w.seqinfo[seq].w;
            it.slot = seq * H + h;
            it.pad = 0;
            it.flags = GDN_ITEM_FROM_ZERO | GDN_ITEM_WRITE_SLOT;
            w.items1[2 * u] = it;
            it.flags = GDN_ITEM_FROM_IDENTITY | GDN_ITEM_WRITE_M;
            w.items1[2 * u + 1] = it;
        }
        if (tid == 0) {
            w.num_items[0] = 0;
            w.num_items[1] = 2 * units;
            w.num_items[2] = 0;
        }
        return;
    }
    // 2. segment count of the units that need correction matrices (heads with
    //    alpha identically 1, or every split head without sliding); batched
    //    inputs only, where every sequence has the same chunk count
    __shared__ int s_nm, s_ns_m, s_best;
    __shared__ unsigned long long s_cmin;
    if (tid == 0) {
        s_nm = 0;
        s_ns_m = 0;
        s_best = 0;
        s_cmin = ~0ull;
    }
    __syncthreads();
    if (pp.cp_enabled && !p.varlen && units > 0) {
        const int nc = w.seqinfo[0].w;
        int NS0 = nc > pp.L ? (nc + pp.L - 1) / pp.L : 1;
        NS0 = nc > 0 ? (nc + max(1, (nc + NS0 - 1) / NS0) - 1) / max(1, (nc + NS0 - 1) / NS0) : 1;
        if (NS0 > 2) {
            int mine = 0;
            for (int u = tid; u < units; u += blockDim.x)
                if (!(w.flags[u] != 0 && pp.sliding)) ++mine;      // flags are [N, H]: unit u = (u / H, u % H)
            if (mine) atomicAdd(&s_nm, mine);
            __syncthreads();
            const int n_m = s_nm, n_s = units - n_m;
            if (n_m > 0 && pp.grid > 0) {
                // least cost over NS0 - 1 .. 2 (non-negative doubles order as their bits)
                for (int ns = NS0 - 1 - tid; ns >= 2; ns -= blockDim.x)
                    atomicMin(&s_cmin, (unsigned long long)__double_as_longlong(
                                           correction_cost(ns, nc, NS0, n_m, n_s, pp.grid, pp.state_ratio, pp.scan_ratio)));
                __syncthreads();
                const unsigned long long cmin = s_cmin;
                for (int ns = NS0 - 1 - tid; ns >= 2; ns -= blockDim.x)
                    if ((unsigned long long)__double_as_longlong(correction_cost(
                            ns, nc, NS0, n_m, n_s, pp.grid, pp.state_ratio, pp.scan_ratio)) == cmin)
                        atomicMax(&s_best, ns);
                __syncthreads();
                if (tid == 0) {
                    const double c0 = correction_cost(NS0, nc, NS0, n_m, n_s, pp.grid, pp.state_ratio, pp.scan_ratio);
                    s_ns_m = (s_best > 0 && __longlong_as_double((long long)cmin) < 0.95 * c0) ? s_best : 0;
                }
            }
            __syncthreads();
        }
    }
    const int ns_m = s_ns_m;
    const int max_walk = min(pp.L, kMaxLookbackChunks);
    // 3. the work items, kPlanThreads units per round, one thread per unit.
    //    The look-back windows of the sliding units' segments are walked by
    //    the whole block, one (unit, segment) pair per thread: each walk is a
    //    chain of dependent loads of chunk totals, so one thread walking all
    //    of its unit's segments would leave the round waiting on the longest
    //    chain of chains.
    __shared__ int4 s_unit[kPlanThreads];    // (seq, head, chunks, first chunk)
    __shared__ int4 s_seg[kPlanThreads];     // (segments, chunks per segment, first item, first walk)
    __shared__ __align__(16) int s_failed[kPlanThreads];   // some window needs more than max_walk chunks
    __shared__ int s_walks;
    for (int ubase = 0; ubase < units; ubase += blockDim.x) {
        const int u = ubase + tid;
        int seq = 0, h = 0, nc = 0, NS = 0, Lu = 1, chunk0 = 0;
        bool mpath = false;
        if (u < units) {
            seq = w.seq_order[u / H];
            h = u % H;
            nc = w.seqinfo[seq].w;
            chunk0 = w.seqinfo[seq].z;
            // an empty sequence still gets one (empty) item: it writes final = initial
            NS = (pp.cp_enabled && nc > pp.L) ? (nc + pp.L - 1) / pp.L : 1;
            Lu = max(1, (nc + NS - 1) / NS);
            NS = nc > 0 ? (nc + Lu - 1) / Lu : 1;
            const bool flagged = w.flags[seq * H + h] != 0;
            if (ns_m > 0 && NS > ns_m && !(flagged && pp.sliding)) {
                Lu = (nc + ns_m - 1) / ns_m;
                NS = (nc + Lu - 1) / Lu;
            }
            mpath = NS > 1 && !(flagged && pp.sliding);
        }
        // the output pass's items do not depend on the path: NS per unit
        const int c2 = NS, nwalk = (NS > 1 && !mpath) ? NS - 1 : 0;
        const int o2 = s_base[0] + block_exclusive_scan(c2, s_warp, &s_tot[0]);
        const int ow = block_exclusive_scan(nwalk, s_warp, &s_walks);
        s_unit[tid] = make_int4(seq, h, nc, chunk0);
        s_seg[tid] = make_int4(NS, Lu, o2, ow);
        s_failed[tid] = 0;
        __syncthreads();
        // segments 1.. of the sliding units: walk (a group of kWalkLanes lanes
        // per segment), and write the item when the window fits (a unit with
        // a failed walk is rewritten below)
        const int walks = s_walks;
        const int grp = tid / kWalkLanes, ngrp = blockDim.x / kWalkLanes;
        const unsigned gmask = ((1u << kWalkLanes) - 1u) << ((tid & 31) & ~(kWalkLanes - 1));
        for (int wi = grp; wi < walks; wi += ngrp) {
            int lo = 0, hi = blockDim.x - 1;   // the last unit whose first walk is <= wi
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_seg[mid].w <= wi) lo = mid; else hi = mid - 1;
            }
            const int4 un = s_unit[lo], sg = s_seg[lo];
            const int j = wi - sg.w + 1;
            gdn_work_item it;
            it.seq = un.x;
            it.head = un.y;
            it.c_begin = j * sg.y;
            it.c_end = min(un.z, (j + 1) * sg.y);
            const int wnd = lookback_window<kWalkLanes>(w, un.y, un.w, it.c_begin, pp.ln_eps, max_walk, gmask);
            if ((tid & (kWalkLanes - 1)) != 0) continue;
            if (wnd < 0) {
                s_failed[lo] = 1;
            } else if (sg.z + sg.x <= w.max_items) {
                it.c_start = it.c_begin - wnd;
                it.slot = -1;
                it.pad = 0;
                it.flags = GDN_ITEM_OUTPUT | (j == sg.x - 1 ? GDN_ITEM_WRITE_FINAL : 0) |
                           (it.c_start == 0 ? GDN_ITEM_FROM_INITIAL : GDN_ITEM_FROM_ZERO);
                w.items2[sg.z + j] = it;
            }
        }
        __syncthreads();
        if (u < units && s_failed[tid]) mpath = true;
        const int c1 = mpath ? 2 * NS - 3 : 0, cs = mpath ? NS - 1 : 0, cu = mpath ? 1 : 0;
        const int o1 = s_base[1] + block_exclusive_scan(c1, s_warp, &s_tot[1]);
        const int os = s_base[2] + block_exclusive_scan(cs, s_warp, &s_tot[2]);
        const int ou = s_base[3] + block_exclusive_scan(cu, s_warp, &s_tot[3]);
        const bool fits = o2 + c2 <= w.max_items && o1 + c1 <= w.max_items1 &&
                          os + cs <= w.max_cp_slots && ou + cu <= w.max_cp_slots;
        if (u < units && !fits) report_error(w.err, GDN_ERR_DEVICE_CHECK);
        if (u < units && fits) {
            // segment 0 always; the others on the correction path, over
            // whatever the walks above wrote (the barrier orders the writes)
            const int jend = mpath ? NS : 1;
            for (int j = 0; j < jend; ++j) {
                gdn_work_item it;
                it.seq = seq;
                it.head = h;
                it.c_begin = it.c_start = j * Lu;
                it.c_end = min(nc, (j + 1) * Lu);
                it.slot = j == 0 ? -1 : os + j - 1;
                it.pad = 0;
                it.flags = GDN_ITEM_OUTPUT | (j == NS - 1 ? GDN_ITEM_WRITE_FINAL : 0) |
                           (j == 0 ? GDN_ITEM_FROM_INITIAL : GDN_ITEM_FROM_SLOT);
                w.items2[o2 + j] = it;
            }
            if (mpath) {
                int k1 = o1;
                for (int j = 0; j < NS - 1; ++j) {
                    gdn_work_item it;
                    it.seq = seq;
                    it.head = h;
                    it.c_begin = it.c_start = j * Lu;
                    it.c_end = min(nc, (j + 1) * Lu);
                    it.slot = os + j;
                    it.pad = 0;
                    if (j == 0) {
                        it.flags = GDN_ITEM_FROM_INITIAL | GDN_ITEM_WRITE_SLOT;
                        w.items1[k1++] = it;
                    } else {
                        it.flags = GDN_ITEM_FROM_ZERO | GDN_ITEM_WRITE_SLOT;
                        w.items1[k1++] = it;
                        it.flags = GDN_ITEM_FROM_IDENTITY | GDN_ITEM_WRITE_M;
                        w.items1[k1++] = it;
                    }
                }
                w.scan_units[ou] = make_int4(seq, h, NS, os);
            }
        }
        __syncthreads();
        if (tid < 4) s_base[tid] += s_tot[tid];
        __syncthreads();
    }
    const bool ok = s_base[0] <= w.max_items && s_base[1] <= w.max_items1 && s_base[2] <= w.max_cp_slots;
    if (tid == 0) {
        w.num_items[0] = ok ? s_base[0] : 0;
        w.num_items[1] = ok ? s_base[1] : 0;
        w.num_items[2] = ok ? s_base[3] : 0;
    }
    // 4. packed sequences of unequal length: the output list reordered so that
    //    the fused pass's snake order (round r takes item r G + c, or
    //    r G + G - 1 - c in odd rounds) deals it out longest first.  Items
    //    sorted by length (chunks walked, look-back included; a bitonic sort)
    //    go out in rounds of G: the longest item of a round to the group with
    //    the least work so far, the next to the next, and so on
    //    (longest-processing-time dealing by rounds; the groups ranked by
    //    counting, one barrier a round); then each group is
    //    given the CTA whose snake positions hold its items (groups with an
    //    item in the last, partial round on its first positions).  Equal
    //    sequences keep the list as it is: the snake deals their nearly equal
    //    items as well.
    const int n2 = s_base[0], G = pp.grid;
    if (!(ok && p.varlen && w.items_tmp && G > 0 && G <= kLptCtas && n2 > G && n2 <= kLptItems)) return;
    __syncthreads();   // every item of the list is in memory
    unsigned long long *key = reinterpret_cast<unsigned long long *>(s_unit);   // [kLptItems]: (length, item)
    int *cta_at = reinterpret_cast<int *>(s_seg);    // [kLptCtas]: groups by load, then each group's CTA
    int *group = cta_at + kLptCtas;                  // [kLptItems]: group of the item of rank j
    int *load = s_failed;                            // [kLptCtas]: chunks dealt to each group (INT_MAX: padding)
    const int g4 = (G + 3) & ~3;
    int P = 1;
    while (P < n2) P <<= 1;
    for (int i = tid; i < P; i += blockDim.x) {
        unsigned long long k = ~0ull;
        if (i < n2) {
            const gdn_work_item it = w.items2[i];
            w.items_tmp[i] = it;
            const unsigned len = (unsigned)max(0, it.c_end - it.c_start);
            k = ((unsigned long long)(0xFFFFFFFFu - len) << 32) | (unsigned)i;   // longer first, then lower index
        }
        key[i] = k;
    }
    for (int c = tid; c < g4; c += blockDim.x) load[c] = c < G ? 0 : INT_MAX;
    __syncthreads();
    bitonic_sort_u64(key, P);
    const int rounds = (n2 + G - 1) / G;
    for (int r = 0; r < rounds; ++r) {
        for (int c = tid; c < G; c += blockDim.x) {  // less loaded first, then the lower index
            const int lc = load[c];
            int rank = 0;
#pragma unroll 4
            for (int m = 0; m < g4; m += 4) {
                const int4 l = *reinterpret_cast<const int4 *>(load + m);
                rank += (l.x < lc) || (l.x == lc && m < c);
                rank += (l.y < lc) || (l.y == lc && m + 1 < c);
                rank += (l.z < lc) || (l.z == lc && m + 2 < c);
                rank += (l.w < lc) || (l.w == lc && m + 3 < c);
            }
            cta_at[rank] = c;
        }
        __syncthreads();
        for (int k = tid; k < G; k += blockDim.x) {
            const int j = r * G + k;
            if (j < n2) {
                const int c = cta_at[k];
                group[j] = c;
                load[c] += (int)(0xFFFFFFFFu - (unsigned)(key[j] >> 32));
            }
        }
        __syncthreads();
    }
    // each group's CTA: those with an item in the last round first in that
    // round's snake order
    const int last = rounds - 1, rem = n2 - last * G;
    for (int c = tid; c < g4; c += blockDim.x) load[c] = 0;
    __syncthreads();
    for (int j = last * G + tid; j < n2; j += blockDim.x) load[group[j]] = 1;
    __syncthreads();
    for (int c = tid; c < G; c += blockDim.x) {
        const int has = load[c];
        int before = 0;   // groups below c in the same class
        for (int m = 0; m < c; ++m) before += load[m] == has;
        const int pos = has ? before : rem + before;
        cta_at[c] = (last & 1) ? G - 1 - pos : pos;
    }
    __syncthreads();
    for (int j = tid; j < n2; j += blockDim.x) {
        const int r = j / G, cp = cta_at[group[j]];
        w.items2[r * G + ((r & 1) ? G - 1 - cp : cp)] = w.items_tmp[(int)(key[j] & 0xFFFFFFFFu)];
    }
}

cudaError_t launch_seqprep(const Problem &p, const Workspace &w, bool emit_items, cudaStream_t s) {
    seqprep_kernel<<<1, 1024, 0, s>>>(p, w, emit_items ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_gate(const Problem &p, const Workspace &w, cudaStream_t s) {
    dim3 grid(w.max_chunks, (p.H + kGateHeads - 1) / kGateHeads);
    cudaError_t e = launch_dependent(gate_kernel, grid, dim3(256), 0, s, p, w);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_plan(const Problem &p, const Workspace &w, const PlanParams &pp, cudaStream_t s) {
    cudaError_t e = launch_dependent(plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, p, w, pp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn
