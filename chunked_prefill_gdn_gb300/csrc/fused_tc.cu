// tcgen05 fused chunk kernel for bf16 inputs with dk = dv = 128: steps two to
// four of the four-step paragraph of the FlashQLA talk
// "Qwen系列模型线性注意力高性能优化实践", with the state in tensor memory.
//
// Everything is written transposed so that the state's value index i (dv =
// 128) runs along the 128 TMEM lanes and every MMA has M = 128.  Per chunk,
// with S the state at chunk start (dv x dk, fp32 in TMEM), G the chunk-local
// gate cumsum, gamma = exp(G), G* the middle of the chunk's gate range and
//
//   Gamma_rm = exp(G_r - G_m) = a_r b_m,  a_r = exp(G_r - G*), b_m = exp(G* - G_m),
//
// the gated inverse T = Gamma ⊙ T' = D_a T' D_b (Gamma-extraction paragraph),
// so the MMAs take T1 = T' D_c1 with c1 = b beta, which the inverse kernel
// writes directly (it scales each column of T' before storing it):
//
//   P0     Q K^T                                 into the U' columns, masked
//                                                (times exp(-G*)) by the side warps
//   MMA1   P    = S [K;Q]^T                      A = bf16(S) (TMEM); P_K (N = 64) first,
//                                                then P_Q (N = 64) under E2
//   MMA2a  U'   = V^T T1^T                       A = the V tile (smem, MN-major)
//   E2     W2   = -gamma P_K                     (forward merge: "V - S first";
//   MMA2b  U'  += W2 T1^T                         c1 gamma = b beta gamma), U = D_a U'
//   E3     Ut   = e U',  W4 = U'                 e = exp(G_C - G*)
//   MMA3   S   += Ut K           (S pre-scaled by gamma_C in E1)
//   MMA4   P_Q += W4 (exp(-G*) tril(Q K^T))^T   since a_r / gamma_r = exp(-G*)
//   O      o    = scale gamma_r P_Q
//
// exp(-G*) U'_m = U_m / gamma_m, so a chunk whose gate cumsum falls below -80
// (where that could overflow) takes the exact form instead: a = b = 1,
// T = Gamma ⊙ T' element by element, and the output term goes to its own TMEM
// columns (o = scale (gamma P_Q + D4)).
//
// W, U and the per-chunk states never reach HBM.  Warp roles: warps 0-7 run
// only the epilogues on the state chain (E1, E2, E3; warps w and w+4 share TMEM
// lane quadrant w % 4 and split the columns), warps 8-11 run everything off the
// chain (the masked Q K^T and the output), warp 12 feeds q/k/v/T1 tiles by TMA
// into a three-stage ring and computes the per-row gate coefficients, warp 13
// allocates TMEM and issues the MMAs in an order that keeps the chain E1, MMA1,
// E2, MMA2b, E3, MMA3 free of work off it.  Every wait is bounded: on timeout
// the kernel records GDN_ERR_TIMEOUT, waits for its own copies in flight, frees
// TMEM and returns.
#include <limits.h>
#include <stddef.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "gdn_internal.cuh"
#include "inverse_tc.cuh"
#include "tc_ptx.cuh"

namespace gdn {

using namespace tc;

namespace {

constexpr int kD = 128;
constexpr int kThreads = 448;
constexpr int kChainThreads = 256;  // warps 0-7
constexpr int kSideThreads = 128;   // warps 8-11
constexpr int kEpiThreads = kChainThreads + kSideThreads;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint64_t kTimeoutNs = 2000000000ull;

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t kKQBytes = 32768;  // [dk half][K rows 0-63 | Q rows 64-127][128 B]
constexpr uint32_t kVBytes = 16384;   // [dv half][64 rows][128 B]
constexpr uint32_t kTPBytes = 8192;   // [64 rows][128 B]: T1 = T' D_c1
constexpr uint32_t kOffV = kKQBytes;
constexpr uint32_t kOffTP = kKQBytes + kVBytes;
constexpr uint32_t kOffT1 = kOffTP;
constexpr uint32_t kStageBytes = kOffTP + kTPBytes;
constexpr uint32_t kTxBytes = kKQBytes + kVBytes + kTPBytes;  // bytes TMA brings per stage
constexpr int kStages = 3;
// Gate coefficients live in a ring of their own: a data stage is read only by
// the MMAs and is refilled as soon as MMA3 of its chunk completes, while the
// coefficients of a chunk stay in use until its output is written, one chunk
// later.  (When the data waited for the output as well, the next tiles were
// requested only ~1.7 us before they were needed and every role of the CTA
// waited on them each chunk.)
constexpr int kCoefSlots = 6;
constexpr uint32_t kOffQM = kStages * kStageBytes;  // two tril(Q K^T) tiles (chunk parity), [64][128 B]
constexpr uint32_t kOffSmall = kOffQM + 16384;

// TMEM columns (512 allocated)
constexpr uint32_t kColS32 = 0;    // fp32 state
constexpr uint32_t kColS16 = 128;  // bf16 state (MMA1 A operand)
constexpr uint32_t kColP = 192;    // two P buffers of 128 columns (chunk parity):
                                   //   +0..63 P_K (W2, then W4, bf16 at +16..+47), +64..127 P_Q (+ output);
                                   //   in the exact form the other buffer's +0..63 takes D4
constexpr uint32_t kColU = 448;    // Q K^T (P0, lanes 64-127) until masked, then U' fp32 (Ut bf16 at +16..+47)

// Per-chunk gate coefficients (written by the producer warp with the tiles).
struct Coef {
    float G[64];     // chunk-local cumsum (rows past the end repeat the last)
    float gam[64];   // gamma_r
    float so[64];    // scale * gamma_r (output)
    float e[64];     // a_r gamma_C / gamma_r   (Ut = e U')
    float f[64];     // exp(-G*) (1 in the exact form), the same for every row
    float gC;        // gamma_C
    int exact;       // 1: Gamma is applied element by element
    int pad[2];
};

struct Small {
    Coef coef[kCoefSlots];
    uint64_t full[kStages], empty[kStages];  // empty: MMA3 of the stage's chunk is done
    uint64_t cempty[kCoefSlots];             // the chain and the side warps are done with the slot
    uint64_t e1, e2, e3, e4, qm;
    // by chunk parity (chunk n: [n & 1], phase n >> 1)
    uint64_t oepi[2];  // output of chunk n done
    uint64_t m4x[2];   // MMA4 of chunk n done
    uint64_t m1, m2, m3, p0, fin;
    uint32_t tmem_base;
    int abort;
};

constexpr uint32_t kSmemBytes = kOffSmall + sizeof(Small) + 1024;

struct TcMaps {
    CUtensorMap q, k, v, tp;
};

struct Ctx {
    const TcMaps *maps;
    uint8_t *smem;
    uint32_t sbase;  // shared-space address of smem
    Small *sm;
    const Problem *p;
    const Workspace *w;
    const gdn_work_item *items;
    int n_items;
    uint32_t tbase;
    int G;               // CTAs that run work items (the chain CTAs)
    int ov_c0;           // chunk columns from ov_c0 on are computed during this pass
    int ov_expected;     // units per column then
    int *ov_ready;       // [columns]: units of a column whose T1 rows are in memory
};


// Slow path of a wait, out of line so the per-chunk code stays small enough
// for the instruction cache: bounded spin, then GDN_ERR_TIMEOUT.
// (Scalars only: a reference to the context would force it into local memory.)
__device__ __noinline__ bool wait_slow(int *abort, int *err, uint64_t *bar, uint32_t parity) {
    if (mbar_wait(bar, parity, abort, kTimeoutNs)) return true;
    if (atomicExch(abort, 1) == 0) report_error(err, GDN_ERR_TIMEOUT);
    return false;
}

__device__ __forceinline__ bool wait_or_abort(const Ctx &cx, uint64_t *bar, uint32_t parity) {
    return mbar_try_wait(bar, parity) || wait_slow(&cx.sm->abort, cx.w->err, bar, parity);
}

// Epilogue waits: every lane waits, and the warp gives up together, so the
// warp-collective tcgen05.ld/st that follow are never reached by part of a warp.
__device__ __forceinline__ bool ewait(const Ctx &cx, uint64_t *bar, uint32_t parity) {
    const bool r = wait_or_abort(cx, bar, parity);
    return __all_sync(0xffffffffu, r);
}

// Shared-space address of coefficient array `field` of coefficient slot s.
#define COEF_ADDR(cx, s, field) ((cx).sbase + kOffSmall + (s) * sizeof(Coef) + offsetof(Coef, field))

// Items of this CTA: round r takes item r G + c in even rounds and
// r G + G - 1 - c in odd ones (c = blockIdx.x, G = gridDim.x).  The planner
// lists items longest first, so the rounds snake the long ones over the CTAs
// instead of stacking them on the first ones.  Every role of the CTA walks the
// same sequence; it ends at the first index past the list.
__device__ __forceinline__ int cta_item(int r, int G) {
    const int c = blockIdx.x;
    return r * G + ((r & 1) ? G - 1 - c : c);
}

// Stage ring: chunk n uses stage n % kStages; its use index is n / kStages.
__device__ __forceinline__ int stage_of(uint32_t n) { return static_cast<int>(n % kStages); }
__device__ __forceinline__ int coef_of(uint32_t n) { return static_cast<int>(n % kCoefSlots); }
__device__ __forceinline__ uint32_t use_parity(uint32_t n) { return (n / kStages) & 1u; }

// Bounded wait for every unit of chunk column `col` (see FusedOverlap).
__device__ __noinline__ bool wait_column(const Ctx cx, int col) {
    const int *cnt = cx.ov_ready + col;
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v < cx.ov_expected) {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t it = 1;; ++it) {
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
            if (v >= cx.ov_expected) break;
            if ((it & 63u) == 0u) {
                if (*(volatile int *)&cx.sm->abort) return false;
                if (global_timer_ns() - t0 > kTimeoutNs) {
                    if (atomicExch(&cx.sm->abort, 1) == 0) report_error(cx.w->err, GDN_ERR_TIMEOUT);
                    return false;
                }
            }
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// ---------------------------------------------------------------- producer
__device__ __forceinline__ void producer_role(const Ctx &cx, const TcMaps &maps, int lane) {
    const Problem &p = *cx.p;
    const Workspace &w = *cx.w;
    Small &sm = *cx.sm;
    // the timeout probe: no tile ever arrives, so every consumer's bounded wait
    // runs out and the CTA leaves through its error path (no copy was issued)
    if (p.timeout_probe) return;
    // cursor over this CTA's chunks, items in order, empty items skipped
    int r = 0, c = 0, cend = 0, chunk0 = 0, head = 0;
    bool started = false;
    auto advance = [&]() -> bool {
        if (started && c + 1 < cend) {
            ++c;
            return true;
        }
        if (started) ++r;
        started = true;
        for (; cta_item(r, cx.G) < cx.n_items; ++r) {
            const gdn_work_item it = cx.items[cta_item(r, cx.G)];
            if (it.c_start < it.c_end) {
                c = it.c_start;
                cend = it.c_end;
                chunk0 = w.seqinfo[it.seq].z;
                head = it.head;
                return true;
            }
        }
        return false;
    };
    // the gate values of the next chunk are fetched one step ahead, so their
    // latency overlaps the wait for a free stage
    float pg0 = 0.f, pg1 = 0.f;
    int ph = 0, pt0 = 0, plen = 1, pcol = 0;
    auto fetch = [&]() {
        const int4 ci = w.chunks[chunk0 + c];
        pt0 = ci.y;
        plen = ci.z;
        pcol = c;
        ph = head;
        const size_t gb = (size_t)ph * p.total_T + pt0;
        pg0 = w.G[gb + min(lane, plen - 1)];
        pg1 = w.G[gb + min(lane + 32, plen - 1)];
    };
    bool more = advance();
    if (more) fetch();
    uint32_t n = 0;
    while (more) {
        const float g0 = pg0, g1 = pg1;
        const int h = ph, t0 = pt0, col = pcol;
        more = advance();
        if (more) fetch();
        const int s = stage_of(n), cs = coef_of(n);
        if (n >= kStages && !wait_or_abort(cx, &sm.empty[s], ((n / kStages) - 1) & 1)) break;
        if (n >= kCoefSlots && !wait_or_abort(cx, &sm.cempty[cs], ((n / kCoefSlots) - 1) & 1)) break;
        {
            const float Gfirst = __shfl_sync(0xffffffffu, g0, 0);
            const float Glast = __shfl_sync(0xffffffffu, g1, 31);  // row 63 repeats row len-1
            // exp(-G*) U'_m equals U_m / gamma_m, so the factored form needs
            // gamma_m > e^-80 everywhere in the chunk; past that the exact form is
            // used (the inverse kernel takes the same decision from the same G)
            const bool exact = Glast < -80.f;
            const float Gs = 0.5f * (Gfirst + Glast);
            Coef &cf = sm.coef[cs];
            const float gg[2] = {g0, g1};
            const float fN = __expf(-Gs), eN = __expf(Glast - Gs);
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const int r = lane + 32 * q2;
                const float G = gg[q2];
                const float gam = __expf(G);
                cf.G[r] = G;
                cf.gam[r] = gam;
                cf.so[r] = p.scale * gam;
                cf.e[r] = exact ? __expf(Glast - G) : eN;
                cf.f[r] = exact ? 1.f : fN;
            }
            if (lane == 0) {
                cf.gC = __expf(Glast);
                cf.exact = exact;
            }
        }
        if (col >= cx.ov_c0) {
            bool ready = true;
            if (lane == 0) ready = wait_column(cx, col);
            if (!__shfl_sync(0xffffffffu, ready, 0)) break;
        }
        uint8_t *st = cx.smem + s * kStageBytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.full[s], kTxBytes);
            tma_load_3d(st + 0, &maps.k, &sm.full[s], 0, h, t0);
            tma_load_3d(st + 8192, &maps.q, &sm.full[s], 0, h, t0);
            tma_load_3d(st + 16384, &maps.k, &sm.full[s], 64, h, t0);
            tma_load_3d(st + 24576, &maps.q, &sm.full[s], 64, h, t0);
            tma_load_3d(st + kOffV, &maps.v, &sm.full[s], 0, h, t0);
            tma_load_3d(st + kOffV + 8192, &maps.v, &sm.full[s], 64, h, t0);
            tma_load_2d(st + kOffTP, &maps.tp, &sm.full[s], 0, h * p.total_T + t0);
        } else {
            mbar_arrive(&sm.full[s]);
        }
        ++n;
    }
    // never leave a copy in flight into shared memory that is about to be released
    if (lane == 0) {
        int dummy = 0;
        for (int s = 0; s < kStages; ++s) {
            const uint32_t arms = n > (uint32_t)s ? (n - 1 - s) / kStages + 1 : 0;
            if (arms) mbar_wait(&sm.full[s], (arms - 1) & 1, &dummy, kTimeoutNs);
        }
    }
}

// --------------------------------------------------------------------- MMA
// This CTA's chunks in order (its items cta_item(0), cta_item(1), ...; empty
// items skipped), for the MMA warp, which looks one chunk ahead.
struct MmaCursor {
    int r, c, cend, cbegin, flags;
    bool valid;
};

__device__ __forceinline__ void cursor_start(const Ctx &cx, MmaCursor &cu) {
    cu.valid = false;
    for (cu.r = 0; cta_item(cu.r, cx.G) < cx.n_items; ++cu.r) {
        const gdn_work_item it = cx.items[cta_item(cu.r, cx.G)];
        if (it.c_start < it.c_end) {
            cu.c = it.c_start;
            cu.cend = it.c_end;
            cu.cbegin = it.c_begin;
            cu.flags = it.flags;
            cu.valid = true;
            return;
        }
    }
}

__device__ __forceinline__ void cursor_next(const Ctx &cx, MmaCursor &cu) {
    if (++cu.c < cu.cend) return;
    cu.valid = false;
    for (++cu.r; cta_item(cu.r, cx.G) < cx.n_items; ++cu.r) {
        const gdn_work_item it = cx.items[cta_item(cu.r, cx.G)];
        if (it.c_start < it.c_end) {
            cu.c = it.c_start;
            cu.cend = it.c_end;
            cu.cbegin = it.c_begin;
            cu.flags = it.flags;
            cu.valid = true;
            return;
        }
    }
}

// Issue order per chunk n (the tensor pipe runs one thread's MMAs in order, so
// work off the chain is placed where the chain is in an epilogue):
//   (P0_n was issued after MMA3_{n-1}, into the U' columns, during E1_n)
//   E1_n -> MMA1_n -> m1 | MMA4_{n-1} (during E2_n) | V term (after the side warps
//   masked Q K^T) | E2_n -> MMA2b_n -> m2 | E3_n -> MMA3_n -> m3,
//   stage free | P0_{n+1}
// A chunk in the exact form issues its MMA4 right after MMA3 instead (its D4
// goes to the other P buffer, which MMA1_{n+1} then waits to see emptied).
__device__ __forceinline__ void mma_role(const Ctx &cx) {
    Small &sm = *cx.sm;
    const uint32_t t = cx.tbase;
    const uint32_t smem0 = smem_u32(cx.smem);
    constexpr uint32_t I1h = idesc_bf16_f32(128, 64, 0, 0);   // P_K = S16 K^T, then P_Q = S16 Q^T
    constexpr uint32_t I0 = idesc_bf16_f32(128, 64, 0, 0);    // [K;Q] K^T
    constexpr uint32_t I2a = idesc_bf16_f32(128, 64, 1, 0);   // U' = V^T (T' D_c1)^T, V^T MN-major
    constexpr uint32_t I2b = idesc_bf16_f32(128, 64, 0, 0);   // U' += W2 T1^T
    constexpr uint32_t I3 = idesc_bf16_f32(128, 128, 0, 1);   // S += Ut K   (K as MN-major B)
    constexpr uint32_t I4 = idesc_bf16_f32(128, 64, 0, 0);    // P_Q (or D4) += W4 Qm^T
    bool ok = true;
    // The whole warp runs this loop (so the warp-uniform descriptors can live in
    // uniform registers); one elected lane issues the MMAs and their commits.
    const bool leader = elect_one();
    // P0 of a chunk: [K;Q] K^T into the U' columns (Q K^T in lanes 64-127)
    auto issue_p0 = [&](uint32_t n, bool out) -> bool {
        const int s = stage_of(n);
        if (!wait_or_abort(cx, &sm.full[s], use_parity(n))) return false;
        tc_fence_after();
        const uint64_t dKQ = smem_desc_sw128(smem0 + s * kStageBytes, 16, 1024);
        if (leader) {
            if (out) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t a = dKQ + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    mma_ss(t + kColU, a, a, I0, kk > 0);
                }
            }
            tc_commit(&sm.p0);
        }
        __syncwarp();
        return true;
    };
    // MMA4 of chunk m: P_Q += W4 Qm^T (exact form: D4 = W4 Qm^T into the other buffer)
    auto issue_mma4 = [&](uint32_t m, bool out, bool exact) -> bool {
        if (!wait_or_abort(cx, &sm.e4, m & 1)) return false;
        tc_fence_after();
        const uint32_t pc = t + kColP + (m & 1) * 128, po = t + kColP + ((m + 1) & 1) * 128;
        const uint64_t dQM = smem_desc_sw128(smem0 + kOffQM + (m & 1) * 8192, 16, 1024);
        if (leader) {
            if (out) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t b = dQM + ((kk * 32) >> 4);
                    if (exact)
                        mma_ts(po, pc + 16 + 8 * kk, b, I4, kk > 0);
                    else
                        mma_ts(pc + 64, pc + 16 + 8 * kk, b, I4, 1);
                }
            }
            tc_commit(&sm.m4x[m & 1]);
        }
        __syncwarp();
        return true;
    };

    MmaCursor cu;
    cursor_start(cx, cu);
    uint32_t n = 0;
    bool prev_exact = false, pend4 = false, pend4_out = false;  // MMA4 of chunk n-1 still to issue
    if (cu.valid) ok = issue_p0(0, (cu.flags & GDN_ITEM_OUTPUT) && cu.c >= cu.cbegin);
    while (ok && cu.valid) {
        const int s = stage_of(n);
        const uint32_t par = n & 1;
        const bool out = (cu.flags & GDN_ITEM_OUTPUT) && cu.c >= cu.cbegin;
        const bool zero_v = cu.flags & GDN_ITEM_FROM_IDENTITY;  // correction items: no V term
        const uint32_t st = smem0 + s * kStageBytes;
        const uint32_t pc = t + kColP + (n & 1) * 128;        // this chunk's P buffer
        const bool exact = cx.sm->coef[coef_of(n)].exact;
        const uint64_t dKQ = smem_desc_sw128(st, 16, 1024);             // K|Q rows, K-major
        const uint64_t dV = smem_desc_sw128(st + kOffV, 8192, 1024);    // V^T, MN-major
        const uint64_t dT1 = smem_desc_sw128(st + kOffT1, 16, 1024);
        const uint64_t dK3 = smem_desc_sw128(st, 16384, 1024);          // K as MN-major B
        // this chunk's P buffer last held chunk n-2, whose output must be out;
        // in the exact form chunk n-1 keeps its D4 here too
        if (n >= 2 && !wait_or_abort(cx, &sm.oepi[n & 1], ((n - 2) >> 1) & 1)) break;
        if (prev_exact && !wait_or_abort(cx, &sm.oepi[(n - 1) & 1], ((n - 1) >> 1) & 1)) break;
        if (!wait_or_abort(cx, &sm.e1, par)) break;
        tc_fence_after();
        if (leader) {
            // P_K first (N = 64, the K rows of the tile): E2 needs only P_K, so
            // P_Q (the Q rows, 8 KB further) runs on the tensor pipe under E2
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ts(pc, t + kColS16 + 8 * kk, dKQ + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4), I1h, kk > 0);
            tc_commit(&sm.m1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ts(pc + 64, t + kColS16 + 8 * kk, dKQ + (((kk >> 2) * 16384 + (kk & 3) * 32 + 8192) >> 4), I1h,
                       kk > 0);
        }
        __syncwarp();
        if (pend4 && !issue_mma4(n - 1, pend4_out, false)) break;
        pend4 = false;
        // V term of U' once Q K^T has left the U' columns
        if (!wait_or_abort(cx, &sm.qm, par)) break;
        tc_fence_after();
        if (leader && !zero_v) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ss(t + kColU, dV + ((kk * 2048) >> 4), dT1 + ((kk * 32) >> 4), I2a, kk > 0);
        }
        __syncwarp();
        if (!wait_or_abort(cx, &sm.e2, par)) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ts(t + kColU, pc + 16 + 8 * kk, dT1 + ((kk * 32) >> 4), I2b, (kk > 0 || !zero_v) ? 1u : 0u);
            tc_commit(&sm.m2);
        }
        __syncwarp();
        if (!wait_or_abort(cx, &sm.e3, par)) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ts(t + kColS32, t + kColU + 16 + 8 * kk, dK3 + ((kk * 2048) >> 4), I3, 1);
            tc_commit(&sm.m3);
            tc_commit(&sm.empty[s]);
        }
        __syncwarp();
        if (out && exact) {
            if (!issue_mma4(n, true, true)) break;
        } else {
            pend4 = true;
            pend4_out = out;
        }
        prev_exact = out && exact;
        cursor_next(cx, cu);
        ++n;
        if (cu.valid && !issue_p0(n, (cu.flags & GDN_ITEM_OUTPUT) && cu.c >= cu.cbegin)) break;
    }
    if (pend4) issue_mma4(n - 1, pend4_out, false);
    // all issued MMAs must finish before TMEM is released
    if (leader) tc_commit(&sm.fin);
    __syncwarp();
    int dummy = 0;
    mbar_wait(&sm.fin, 0, &dummy, kTimeoutNs);
}

// ---------------------------------------------------------------- epilogue
struct EpiThread {
    int q, ch, i, et, lane;   // lane quadrant, column half, TMEM lane (= value row i), index in the role
    uint32_t lane_base;   // TMEM lane field of this warp's quadrant
};

__device__ __forceinline__ void load_tile32(const Ctx &cx, const EpiThread &e, uint32_t col, float *x) {
    uint32_t r[32];
    tmem_ld32(cx.tbase + e.lane_base + col, r);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
}

// Stores 32 state columns j0 .. j0+31 (key index) of this thread's value row.
// The destinations are formed once, before any store: a float store could
// alias the parameter blocks as far as the compiler can tell, and re-reading
// their fields after every store made the 64 KB flush of a CTA take ~9 us.
// With head sizes below 128 the tiles are zero-padded to 128 (the TMA fills
// features past dk / dv with zeros), which leaves the real rows and columns
// of the state exact; only those are stored: value rows i < dv (i < dk for a
// correction matrix, whose rows are key indices) and key columns j < dk.
__device__ __noinline__ void write_state32(const Ctx cx, const EpiThread e, const gdn_work_item it, int j0,
                                           const float *sv) {
    const Problem &p = *cx.p;
    const Workspace &w = *cx.w;
    const int dk = p.dk, dv = p.dv;
    if (j0 >= dk) return;
    const bool row_v = e.i < dv, row_k = e.i < dk;
    float *const df = (it.flags & GDN_ITEM_WRITE_FINAL) && row_v
                          ? p.sf + ((size_t)it.seq * p.H + it.head) * dk * dv + (size_t)j0 * dv + e.i : nullptr;
    float *const ds = (it.flags & GDN_ITEM_WRITE_SLOT) && row_v
                          ? w.cp_s + (size_t)it.slot * dk * dv + (size_t)j0 * dv + e.i : nullptr;
    float *const dm = (it.flags & GDN_ITEM_WRITE_M) && row_k
                          ? w.cp_m + (size_t)it.slot * dk * dk + (size_t)j0 * dk + e.i : nullptr;
    if (df) {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) df[jj * dv] = sv[jj];
    }
    if (ds) {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) ds[jj * dv] = sv[jj];
    }
    if (dm) {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) dm[jj * dk] = sv[jj];
    }
}

// Loads 32 start-state columns j0 .. j0+31 of this thread's value row.
__device__ __noinline__ void load_start_state32(const Ctx cx, const EpiThread e, const gdn_work_item it, int j0,
                                                float *sv) {
    const Problem &p = *cx.p;
    const Workspace &w = *cx.w;
    const int i = e.i, dk = p.dk, dv = p.dv;
    const size_t col = (size_t)j0 * dv + i;
    const float *src = nullptr;
    const bool real = i < dv && j0 < dk;   // padded rows and columns start at zero
    if (it.flags & GDN_ITEM_FROM_INITIAL)
        src = p.s0 && real ? p.s0 + ((size_t)it.seq * p.H + it.head) * dk * dv + col : nullptr;
    else if (!(it.flags & GDN_ITEM_FROM_IDENTITY) && (it.flags & GDN_ITEM_FROM_SLOT))
        src = real ? w.cp_s + (size_t)it.slot * dk * dv + col : nullptr;
    const bool ident = !(it.flags & GDN_ITEM_FROM_INITIAL) && (it.flags & GDN_ITEM_FROM_IDENTITY);
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) sv[jj] = src ? src[jj * dv] : (ident && i == j0 + jj) ? 1.f : 0.f;
}

// Writes the state held in TMEM (this thread's row, its 64 columns) for `it`.
__device__ __noinline__ void flush_state(const Ctx cx, const EpiThread e, const gdn_work_item it) {
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        float sv[32];
        load_tile32(cx, e, kColS32 + 64 * e.ch + 32 * hh, sv);
        write_state32(cx, e, it, 64 * e.ch + 32 * hh, sv);
    }
}

// E1 for 32 columns: S16 = bf16(S), S32 = gamma_C S.
__device__ __forceinline__ void store_state32(const Ctx &cx, const EpiThread &e, int hh, const float *sv, float gC) {
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(sv[2 * j], sv[2 * j + 1]);
    tmem_st16(cx.tbase + e.lane_base + kColS16 + 32 * e.ch + 16 * hh, pk);
    uint32_t sc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) sc[j] = __float_as_uint(gC * sv[j]);
    tmem_st32(cx.tbase + e.lane_base + kColS32 + 64 * e.ch + 32 * hh, sc);
}

// ---- the state chain: warps 0-7; warps w and w+4 share lane quadrant w % 4
__device__ __forceinline__ void chain_role(const Ctx &cx, int warp, int lane) {
    const Workspace &w = *cx.w;
    Small &sm = *cx.sm;
    EpiThread e;
    e.q = warp & 3;
    e.ch = warp >> 2;
    e.i = 32 * e.q + lane;
    e.et = threadIdx.x;
    e.lane = lane;
    e.lane_base = static_cast<uint32_t>(32 * e.q) << 16;
    const int ch = e.ch;
    uint32_t n = 0;
    // the item whose end state sits in TMEM and has not been written yet
    bool pending = false;
    gdn_work_item prev_item;
    prev_item.flags = 0;
    bool ok = true;

    for (int r = 0; cta_item(r, cx.G) < cx.n_items && ok; ++r) {
        const gdn_work_item it = cx.items[cta_item(r, cx.G)];
        const int4 si = w.seqinfo[it.seq];
        if (it.c_start >= it.c_end) {
            // an empty sequence: its end state is its start state
            if (pending) {
                if (!ewait(cx, &sm.m3, (n - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                flush_state(cx, e, prev_item);
                pending = false;
            }
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float sv[32];
                load_start_state32(cx, e, it, 64 * ch + 32 * hh, sv);
                write_state32(cx, e, it, 64 * ch + 32 * hh, sv);
            }
            continue;
        }
        for (int c = it.c_start; c < it.c_end; ++c, ++n) {
            const int s = stage_of(n), cs = coef_of(n);
            const uint32_t par = n & 1;
            const int len = w.chunks[si.z + c].z;
            const uint32_t pcol = kColP + (n & 1) * 128;
            const Coef &cf = sm.coef[cs];
            if (!ewait(cx, &sm.full[s], use_parity(n))) { ok = false; break; }

            // ---- E1: S16 = bf16(S), S32 = gamma_C S   (after MMA3 of the last chunk)
            const float gC = cf.gC;
            if (c == it.c_start) {
                if (pending) {
                    if (!ewait(cx, &sm.m3, (n - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    flush_state(cx, e, prev_item);
                    pending = false;
                }
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float sv[32];
                    load_start_state32(cx, e, it, 64 * ch + 32 * hh, sv);
                    store_state32(cx, e, hh, sv, gC);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sm.e1);
            } else {
                // MMA1 needs only bf16(S): arrive as soon as it is in TMEM, then
                // scale the fp32 state by gamma_C under MMA1 (MMA3, its next
                // writer, is issued only after this warp's e3 below)
                if (!ewait(cx, &sm.m3, (n - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                {
                    uint32_t sv[64], pk[32];
                    tmem_ld32(cx.tbase + e.lane_base + kColS32 + 64 * ch, sv);
                    tmem_ld32(cx.tbase + e.lane_base + kColS32 + 64 * ch + 32, sv + 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        pk[j] = pack_bf16x2(__uint_as_float(sv[2 * j]), __uint_as_float(sv[2 * j + 1]));
                    tmem_st32(cx.tbase + e.lane_base + kColS16 + 32 * ch, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&sm.e1);
#pragma unroll
                    for (int j = 0; j < 64; ++j) sv[j] = __float_as_uint(gC * __uint_as_float(sv[j]));
                    tmem_st32(cx.tbase + e.lane_base + kColS32 + 64 * ch, sv);
                    tmem_st32(cx.tbase + e.lane_base + kColS32 + 64 * ch + 32, sv + 32);
                }
            }

            // ---- E2: W2 = -gamma P_K   (after MMA1; it multiplies T1 = T' D_c1, and c2 = c1 gamma)
            if (!ewait(cx, &sm.m1, par)) { ok = false; break; }
            tc_fence_after();
            {
                float pk[32];
                load_tile32(cx, e, pcol + 32 * ch, pk);
                const uint32_t c2a = COEF_ADDR(cx, cs, gam) + 128 * ch;
                uint32_t w2[16];
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 c = lds_f4(c2a + 16 * q4);
                    w2[2 * q4] = pack_bf16x2(-c.x * pk[4 * q4], -c.y * pk[4 * q4 + 1]);
                    w2[2 * q4 + 1] = pack_bf16x2(-c.z * pk[4 * q4 + 2], -c.w * pk[4 * q4 + 3]);
                }
                tmem_st16(cx.tbase + e.lane_base + pcol + 16 + 16 * ch, w2);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&sm.e2);

            // ---- E3: Ut = e U' for the state (after MMA2); then W4 = U' for the output
            // (the uniform factor exp(-G*) of the factored form rides on the masked Q K^T)
            if (!ewait(cx, &sm.m2, par)) { ok = false; break; }
            tc_fence_after();
            {
                float u[32];
                load_tile32(cx, e, kColU + 32 * ch, u);
                if (len < 64) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (32 * ch + j >= len) u[j] = 0.f;
                }
                const uint32_t ea = COEF_ADDR(cx, cs, e) + 128 * ch;
                uint32_t ut[16];
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 ce = lds_f4(ea + 16 * q4);
                    ut[2 * q4] = pack_bf16x2(u[4 * q4] * ce.x, u[4 * q4 + 1] * ce.y);
                    ut[2 * q4 + 1] = pack_bf16x2(u[4 * q4 + 2] * ce.z, u[4 * q4 + 3] * ce.w);
                }
                tmem_st16(cx.tbase + e.lane_base + kColU + 16 + 16 * ch, ut);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sm.e3);
#pragma unroll
                for (int j = 0; j < 16; ++j) ut[j] = pack_bf16x2(u[2 * j], u[2 * j + 1]);
                tmem_st16(cx.tbase + e.lane_base + pcol + 16 + 16 * ch, ut);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&sm.e4);
            mbar_arrive(&sm.cempty[cs]);
        }
        if (!ok) break;
        prev_item = it;
        pending = true;
    }
    // tail: the last item's state
    if (ok && pending && n > 0 && ewait(cx, &sm.m3, (n - 1) & 1)) {
        tc_fence_after();
        flush_state(cx, e, prev_item);
    }
}

// Masked Q K^T -> the qm tile (side warps of lane quadrants 2-3: query row r =
// lane index - 64; key columns m <= r < len kept).
__device__ __forceinline__ void side_qmask(const Ctx &cx, const EpiThread &e, int len, uint32_t qm_tile, float f) {
    const int r = e.i - 64;
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        float qk[32];
        load_tile32(cx, e, kColU + 32 * hh, qk);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t wv[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const int mm = 8 * cc + 2 * e2;
                const int m0 = 32 * hh + mm;
                const float x0 = (r < len && m0 <= r) ? f * qk[mm] : 0.f;
                const float x1 = (r < len && m0 + 1 <= r) ? f * qk[mm + 1] : 0.f;
                wv[e2] = pack_bf16x2(x0, x1);
            }
            sts_u4(qm_tile + sw128_offset(r, 4 * hh + cc), make_uint4(wv[0], wv[1], wv[2], wv[3]));
        }
    }
}

// The same with Gamma applied element by element (exact form).
__device__ __noinline__ void side_qmask_exact(const Ctx cx, const EpiThread e, const Coef &cf, int len,
                                              uint8_t *qm_tile) {
    const int r = e.i - 64;
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        float qk[32];
        load_tile32(cx, e, kColU + 32 * hh, qk);
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t wv[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const int mm = 8 * cc + 2 * e2;
                const int m0 = 32 * hh + mm;
                const float x0 = (r < len && m0 <= r) ? qk[mm] * __expf(cf.G[r] - cf.G[m0]) : 0.f;
                const float x1 = (r < len && m0 + 1 <= r) ? qk[mm + 1] * __expf(cf.G[r] - cf.G[m0 + 1]) : 0.f;
                wv[e2] = pack_bf16x2(x0, x1);
            }
            *reinterpret_cast<uint4 *>(qm_tile + sw128_offset(r, 4 * hh + cc)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
    }
}

// Exact form: x += scale D4 (D4 read from TMEM).  Inline: an out-of-line call
// taking x by pointer would put x in local memory on every path.
__device__ __forceinline__ void add_d4(const Ctx &cx, const EpiThread &e, uint32_t col, float scale, float *x) {
    float d4[32];
    load_tile32(cx, e, col, d4);
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) x[rr] = fmaf(scale, d4[rr], x[rr]);
}

// Output of one finished chunk: usual form o = scale gamma_r P_Q (P_Q already
// holds the intra-chunk term); exact form o = scale (gamma_r P_Q + D4).  Side
// warps, lane = value row i, all 64 tokens; each store of a warp covers 64
// contiguous bytes of one token's row of o.
__device__ __forceinline__ void output_chunk(const Ctx &cx, const EpiThread &e, int s, bool exact, uint32_t pq_col,
                             uint32_t d4_col, int t0, int len, int h) {
    const Problem &p = *cx.p;
    const size_t rs = (size_t)p.H * p.dv;
    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.o) + ((size_t)t0 * p.H + h) * p.dv + e.i;
    const uint32_t soa = COEF_ADDR(cx, s, so);
    if (e.i >= p.dv) return;   // a padded value row
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        float x[32];
        load_tile32(cx, e, pq_col + 32 * hh, x);
        const int r0 = 32 * hh;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
            const float4 so = lds_f4(soa + 4 * r0 + 16 * q4);
            x[4 * q4 + 0] *= so.x;
            x[4 * q4 + 1] *= so.y;
            x[4 * q4 + 2] *= so.z;
            x[4 * q4 + 3] *= so.w;
        }
        if (exact) add_d4(cx, e, d4_col + 32 * hh, p.scale, x);
        __nv_bfloat16 *oh = o + (size_t)r0 * rs;
        if (len >= r0 + 32) {
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) oh[rr * rs] = __float2bfloat16_rn(x[rr]);
        } else {
#pragma unroll
            for (int rr = 0; rr < 32; ++rr)
                if (r0 + rr < len) oh[rr * rs] = __float2bfloat16_rn(x[rr]);
        }
    }
}

// ---- off the chain: warps 8-11 (lane quadrant w % 4)
__device__ __forceinline__ void side_role(const Ctx &cx, int warp, int lane) {
    const Workspace &w = *cx.w;
    Small &sm = *cx.sm;
    EpiThread e;
    e.q = warp & 3;
    e.ch = 0;
    e.i = 32 * e.q + lane;
    e.et = threadIdx.x - kChainThreads;
    e.lane = lane;
    e.lane_base = static_cast<uint32_t>(32 * e.q) << 16;

    uint32_t n = 0;
    // the previous chunk, whose output is written one step later
    int pv_out = 0, pv_t0 = 0, pv_len = 0, pv_h = 0, pv_s = 0, pv_exact = 0;
    uint32_t pv_pcol = 0, pv_ocol = 0;
    bool ok = true;

    for (int r = 0; cta_item(r, cx.G) < cx.n_items && ok; ++r) {
        const gdn_work_item it = cx.items[cta_item(r, cx.G)];
        const int4 si = w.seqinfo[it.seq];
        for (int c = it.c_start; c < it.c_end; ++c, ++n) {
            const int s = stage_of(n), cs = coef_of(n);
            const uint32_t par = n & 1;
            const int4 ci = w.chunks[si.z + c];
            const int t0 = ci.y, len = ci.z;
            const bool out = (it.flags & GDN_ITEM_OUTPUT) && c >= it.c_begin;
            const uint32_t pcol = kColP + (n & 1) * 128, ocol = kColP + ((n + 1) & 1) * 128;
            const Coef &cf = sm.coef[cs];
            if (!ewait(cx, &sm.full[s], use_parity(n))) { ok = false; break; }
            const bool exact = cf.exact;

            // ---- masked Q K^T (P0 put it in the U' columns; the qm tile is free once
            // MMA4 of the last chunk is done); the exact form also applies Gamma
            if (!ewait(cx, &sm.p0, par)) { ok = false; break; }
            // this parity's qm tile was last read by MMA4 of chunk n-2
            if (n >= 2 && !ewait(cx, &sm.m4x[n & 1], ((n - 2) >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            if (out && e.q >= 2) {
                if (exact)
                    side_qmask_exact(cx, e, cf, len, cx.smem + kOffQM + (n & 1) * 8192);
                else
                    side_qmask(cx, e, len, cx.sbase + kOffQM + (n & 1) * 8192, cf.f[0]);
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&sm.qm);

            // ---- output of the previous chunk (after its MMA4); then its stage is free
            if (n > 0) {
                if (!ewait(cx, &sm.m4x[(n - 1) & 1], ((n - 1) >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (pv_out) output_chunk(cx, e, pv_s, pv_exact, pv_pcol + 64, pv_ocol, pv_t0, pv_len, pv_h);
                tc_fence_before();
                mbar_arrive(&sm.oepi[(n - 1) & 1]);
                mbar_arrive(&sm.cempty[pv_s]);
            }

            pv_out = out;
            pv_t0 = t0;
            pv_len = len;
            pv_h = it.head;
            pv_s = cs;
            pv_exact = exact;
            pv_pcol = pcol;
            pv_ocol = ocol;
        }
    }
    // tail: output of the last chunk
    if (ok && n > 0 && ewait(cx, &sm.m4x[(n - 1) & 1], ((n - 1) >> 1) & 1)) {
        tc_fence_after();
        if (pv_out)
            output_chunk(cx, e, pv_s, pv_exact, pv_pcol + 64, pv_ocol, pv_t0, pv_len, pv_h);
    }
}

// ---------------------------------------------------------------- kernel
// 14 warps share the 4 SM sub-partitions 4/4/3/3, so a thread may hold at most
// 16384 / (4 * 32) = 128 registers.  OVL: the launch also has CTAs past the
// chain CTAs, which compute the T1 tiles of the last chunk columns (the
// inverse's 16 warps; the chain CTAs leave warps 14 and 15 idle).
template <bool OVL>
__global__ void __launch_bounds__(OVL ? kInvThreads : kThreads, 1)
    fused_tc_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ Problem p,
                    const __grid_constant__ Workspace w, const int pass, const __grid_constant__ FusedOverlap ov) {
    grid_dependency_wait();
    extern __shared__ uint8_t smem_raw[];
    if (OVL && (int)blockIdx.x >= ov.chain_ctas) {
        // (inline: the tensor map must be addressed in the kernel's parameter space)
        InvSel sel = {};
        sel.mode = 2;
        sel.nc = ov.nc;
        sel.c0 = ov.c0;
        sel.cta = (int)blockIdx.x - ov.chain_ctas;
        sel.ctas = (int)gridDim.x - ov.chain_ctas;
        sel.ready = ov.ready;
        inverse_tc_body(&maps.k, p, w, ov.gate_scaled, sel, smem_raw);
        return;
    }
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small &sm = *reinterpret_cast<Small *>(smem + kOffSmall);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 32);
            mbar_init(&sm.empty[s], 1);
        }
        for (int c = 0; c < kCoefSlots; ++c) mbar_init(&sm.cempty[c], kEpiThreads);
        mbar_init(&sm.e1, kChainThreads);
        mbar_init(&sm.e2, kChainThreads);
        mbar_init(&sm.e3, kChainThreads);
        mbar_init(&sm.e4, kChainThreads);
        mbar_init(&sm.m4x[0], 1);
        mbar_init(&sm.m4x[1], 1);
        mbar_init(&sm.oepi[0], kSideThreads);
        mbar_init(&sm.oepi[1], kSideThreads);
        mbar_init(&sm.qm, kSideThreads);
        mbar_init(&sm.m1, 1);
        mbar_init(&sm.m2, 1);
        mbar_init(&sm.m3, 1);
        mbar_init(&sm.p0, 1);
        mbar_init(&sm.fin, 1);
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&maps.q);
        tma_prefetch_map(&maps.k);
        tma_prefetch_map(&maps.v);
        tma_prefetch_map(&maps.tp);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    Ctx cx;
    cx.maps = &maps;
    cx.smem = smem;
    cx.sbase = smem_u32(smem);
    cx.sm = &sm;
    cx.p = &p;
    cx.w = &w;
    cx.items = pass == 2 ? w.items2 : w.items1;
    cx.n_items = *(volatile const int *)&w.num_items[pass == 2 ? 0 : 1];
    cx.tbase = sm.tmem_base;
    cx.G = OVL ? ov.chain_ctas : (int)gridDim.x;
    cx.ov_c0 = OVL ? ov.c0 : INT_MAX;
    cx.ov_expected = ov.expected;
    cx.ov_ready = ov.ready;

    if (warp == kProducerWarp) {
        producer_role(cx, maps, lane);
    } else if (warp == kMmaWarp) {
        mma_role(cx);
    } else if (warp < 8) {
        chain_role(cx, warp, lane);
    } else if (warp < 12) {
        side_role(cx, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(cx.tbase, 512);
    }
}

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
        cudaGetLastError();
    });
    return fn;
}

// [total_T, H, d] bf16 rows, boxes of 64 tokens x 64 features, 128-byte
// swizzle; with d < 128 the features past d read as zeros (the kernel always
// loads two 64-feature halves); returns the driver result (0 on success)
int encode_rows(EncodeTiledFn fn, CUtensorMap *m, const void *base, int H, int total_T, int d) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)total_T};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

bool fused_tc_supported(int dtype, int dk, int dv) {
    auto ok = [](int d) { return d == 32 || d == 64 || d == kD; };
    return (dtype == GDN_BF16 && ok(dk) && ok(dv)) || fused_tf32_supported(dtype, dk, dv);
}

cudaError_t launch_fused_tc(const Problem &p, const Workspace &w, int pass, int grid, cudaStream_t s,
                            const FusedOverlap *ov) {
    if (!fused_tc_supported(p.dtype, p.dk, p.dv)) return cudaErrorNotSupported;
    if (p.total_T == 0) return launch_fused_simt(p, w, pass, grid, s);  // only empty sequences: nothing to tile
    if (p.dtype == GDN_F32) return launch_fused_tf32(p, w, pass, grid, s);
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        set_error_detail("driver entry point cuTensorMapEncodeTiled", cudaErrorNotSupported);
        return cudaErrorNotSupported;
    }
    TcMaps maps;
    memset(&maps, 0, sizeof(maps));
    const int rows_tp = p.H * p.total_T;
    cuuint64_t dims[2] = {64, (cuuint64_t)rows_tp};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    int r;
    if ((r = encode_rows(fn, &maps.q, p.q, p.H, p.total_T, p.dk)) || (r = encode_rows(fn, &maps.k, p.k, p.H, p.total_T, p.dk)) ||
        (r = encode_rows(fn, &maps.v, p.v, p.H, p.total_T, p.dv)) ||
        (r = fn(&maps.tp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.tprime, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE))) {
        set_error_detail("encode tensor map", cudaErrorInvalidValue, r);
        return cudaErrorInvalidValue;
    }
    FusedOverlap none = {};
    const FusedOverlap *o = ov && ov->c0 < ov->nc ? ov : nullptr;
    if (!o) {
        cudaError_t e =
            cudaFuncSetAttribute(fused_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = launch_dependent(fused_tc_kernel<false>, dim3(grid), dim3(kThreads), (size_t)kSmemBytes, s, maps, p, w,
                             pass, none);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    // one cooperative launch, so that the chain CTAs, which wait on the
    // inverse CTAs, are guaranteed to run alongside them
    const size_t smem = std::max<size_t>(kSmemBytes, kInvSmem);
    cudaError_t e = cudaFuncSetAttribute(fused_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kInvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, fused_tc_kernel<true>, maps, p, w, pass, *o);
    if (e != cudaSuccess && e != cudaErrorCooperativeLaunchTooLarge) {
        // without the overlap with the previous kernel's tail
        cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, fused_tc_kernel<true>, maps, p, w, pass, *o);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn
