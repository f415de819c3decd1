// The tcgen05 per-chunk inverse as a device function, shared by the inverse
// kernel and by the fused kernel (whose otherwise idle CTAs compute the last
// chunk columns while the others run the state chain).  Step one of the
// four-step paragraph of the FlashQLA talk "Qwen系列模型线性注意力高性能优化实践",
// in the Gamma-free form of the Gamma-extraction paragraph.
#pragma once

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
// ---------------------------------------------------------------------------
// tcgen05 variant: a persistent, pipelined kernel, for bf16 keys (kind::f16
// Gram) or fp32 keys (F32K: kind::tf32 Gram, one key pair in flight), head
// sizes 32, 64 and 128 (features past dk arrive as zeros).
//
// Work unit: one chunk of one head; units travel in pairs (two heads of one
// chunk).  Per CTA (one per SM), in a software pipeline:
//   warp 15      TMA: both 64 x 128 key tiles of a pair (128-byte swizzle) into
//                a 3-stage ring; then one M = N = 128 MMA [K1;K2][K1;K2]^T into
//                one of two 128-column tensor-memory buffers (the two diagonal
//                64 x 64 blocks are the Gram matrices).
//   warps 0-3    converters: warp q reads TMEM lanes 32q..32q+31 (rows of one
//                unit's Gram) and writes beta_r (k_r . k_m), m < r, into the
//                unit's shared-memory slot as the 10 lower-triangular 16 x 16
//                fp32 blocks of A' (block (I, K), K <= I, at I(I+1)/2 + K,
//                column-major).  (An L2 tensor prefetch of the keys six pairs
//                ahead, issued by a converter, measured 6 us slower at the
//                layer shape: the issuing thread stalls on it.)
//   warps 4-14   solvers: one unit per warp; lane j forward-substitutes column
//                j of (I + A') X = I over rows 0..63 and then column 32 + j over
//                rows 32..63, 16 rows at a time (block rows of A' read as
//                broadcasts, solved blocks kept in tensor memory); each column
//                is scaled by the gate factor the fused kernel expects (T1 =
//                T' diag(c1), see below), and the finished bf16 tile is written
//                into the dead slot and leaves with one bulk copy (the rows of
//                a chunk are contiguous in the workspace).
// All waits are bounded; a timeout sets the error word and the CTA drains.
// ---------------------------------------------------------------------------
namespace {

constexpr int kInvConv = 4;                       // converter warps
constexpr int kInvSolvers = 11;                   // solver warps (= A' slots)
constexpr int kInvThreads = 32 * (kInvConv + kInvSolvers + 1);
constexpr int kInvKStages = 3;
constexpr uint32_t kInvPairBytes = 32768;         // two 64 x 128 bf16 key tiles
constexpr int kInvSlotFloats = 10 * 256 + 64;     // the 10 lower 16 x 16 blocks of A', then c1[64]

constexpr uint32_t kInvSlotBytes = kInvSlotFloats * 4;
constexpr uint64_t kInvTimeoutNs = 2000000000ull;

// Shared-memory plan for bf16 keys (F32K false: a 3-stage ring of 32 KB
// pairs) or fp32 keys (F32K true: the keys read as tf32 by the Gram, one
// 64 KB pair at a time — the eleven A' slots keep the rest).
template <bool F32K>
struct InvCfg {
    static constexpr int kStages = F32K ? 1 : kInvKStages;
    static constexpr uint32_t kPair = F32K ? 2 * kInvPairBytes : kInvPairBytes;
    static constexpr uint32_t kOffSlots = kStages * kPair;
    static constexpr uint32_t kOffBars = kOffSlots + kInvSolvers * kInvSlotBytes;
    static constexpr uint32_t kSmem = kOffBars + 512 + 1024;   // + barriers, + alignment slack
};
constexpr uint32_t kInvOffSlots = InvCfg<false>::kOffSlots;
constexpr uint32_t kInvOffBars = InvCfg<false>::kOffBars;
constexpr uint32_t kInvSmem = InvCfg<false>::kSmem;

static_assert(InvCfg<false>::kSmem <= 227 * 1024 && InvCfg<true>::kSmem <= 227 * 1024,
              "inverse kernel shared memory");

struct InvMaps {
    CUtensorMap k;
};

struct InvBars {
    uint64_t kfull[kInvKStages], kempty[kInvKStages];
    uint64_t tfull[2], tempty[2];
    uint64_t afull[kInvSolvers], aempty[kInvSolvers];
    int4 unit[kInvSolvers];     // per slot: first token, length, head, flags (1 store, 2 exact)
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(InvBars) <= 512, "barrier block");

__host__ __device__ constexpr int block_index(int I, int K) { return I * (I + 1) / 2 + K; }

// Pairs of fp32 values in one 64-bit register, for the two-wide FMA.
__device__ __forceinline__ void lds_2x2(uint32_t addr, uint64_t &a, uint64_t &b) {
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}
__device__ __forceinline__ uint64_t dup2(float x) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(x));
    return d;
}
__device__ __forceinline__ void fma2(uint64_t &acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// Column `col` of (I + A') X = I for rows 16*I0 .. 63 (I0 = 0 or 2), given
// x_r = 0 for r < 16*I0.  A' is stored as column-major 16 x 16 blocks, so one
// 16-byte load gives four consecutive rows of one column and the sums run on
// the two-wide FMA over row pairs.  Block row I: acc = sum_{K<I} A'[I, K] x_K,
// then the diagonal block is substituted right-looking (once x_i is known,
// every row below gets A'[k][i] x_i; A' is zero on and above the diagonal, so
// a pair that straddles row i is updated harmlessly).  Solved blocks go to
// tensor memory (this lane's row, columns xcol + 16 I), from where the rolled
// loop over K reads them back with one 16-column load: the code stays small
// enough for the instruction cache although eleven warps run it at once.
__device__ __forceinline__ void solve_blocked(uint32_t slot, uint32_t xcol, int col, int I0) {
#pragma unroll 1
    for (int I = I0; I < 4; ++I) {
        uint64_t acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0ull;
#pragma unroll 1
        for (int K = I0; K < I; ++K) {
            uint32_t xk[16];
            tc::tmem_ld16(xcol + 16 * K, xk);
            tc::tmem_wait_ld();
            const uint32_t blk = slot + block_index(I, K) * 1024;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const uint64_t xm = dup2(__uint_as_float(xk[m]));
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint64_t a01, a23;
                    lds_2x2(blk + 64 * m + 16 * q, a01, a23);
                    fma2(acc[2 * q], a01, xm);
                    fma2(acc[2 * q + 1], a23, xm);
                }
            }
        }
        const uint32_t dblk = slot + block_index(I, I) * 1024;
        uint32_t cur[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float s = (i & 1) ? hi2(acc[i >> 1]) : lo2(acc[i >> 1]);
            const int r = 16 * I + i;
            const float xi = r < col ? 0.f : (r == col ? 1.f : -s);
            cur[i] = __float_as_uint(xi);
            if (i < 15) {
                const uint64_t xd = dup2(xi);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (4 * q + 3 > i) {
                        uint64_t a01, a23;
                        lds_2x2(dblk + 64 * i + 16 * q, a01, a23);
                        if (4 * q + 1 > i) fma2(acc[2 * q], a01, xd);
                        fma2(acc[2 * q + 1], a23, xd);
                    }
                }
            }
        }
        tc::tmem_st16(xcol + 16 * I, cur);
        tc::tmem_wait_st();
    }
}

// Exact form: rows r0 .. r0+31 of one T' column (value index of column m):
// x_r *= exp(G_r - G_m) (rows past the chunk reuse its last cumsum; T' is zero
// above the diagonal, so only r >= m matters).
__device__ __forceinline__ void exact_gamma_rows(uint32_t *v, int r0, const float *Gh, float Gm, int len) {
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        const float Gr = Gh[min(r0 + t, len - 1)];
        v[t] = __float_as_uint(__uint_as_float(v[t]) * __expf(fminf(Gr - Gm, 0.f)));
    }
}

__device__ __forceinline__ void sts_u16(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(static_cast<unsigned short>(v & 0xFFFFu)) : "memory");
}

__device__ __forceinline__ bool inv_wait(InvBars &b, uint64_t *bar, uint32_t parity, int *err) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (tc::mbar_wait(bar, parity, &b.abort, kInvTimeoutNs)) return true;
    if (atomicExch(&b.abort, 1) == 0) report_error(err, GDN_ERR_TIMEOUT);
    return false;
}


// Which (chunk, head pair) units a CTA of the inverse runs.  Pairs are
// enumerated per mode and dealt round robin over `ctas` CTAs (this one is
// number `cta`):
//   mode 0  every chunk of the chunk table
//   mode 1  chunk columns [0, c0) of nseq equal sequences of nc chunks
//   mode 2  chunk columns [c0, nc) of the same, column by column; each stored
//           unit then adds one to ready[column] once its rows are in memory
struct InvSel {
    int mode, nc, c0, cta, ctas;
    int *ready;
    int f32_out;   // 1: store T' itself (no gate factors) as fp32 rows [H, total_T, 64]
};

struct PairInfo {
    int t0, len, h0, h1, col;
};

__device__ __forceinline__ int sel_pairs(const Problem &p, const Workspace &w, const InvSel &sel) {
    const int hp = (p.H + 1) >> 1;
    if (sel.mode == 1) return p.N * sel.c0 * hp;
    if (sel.mode == 2) return p.N * (sel.nc - sel.c0) * hp;
    return *w.num_chunks * hp;
}

__device__ __forceinline__ PairInfo sel_pair(const Problem &p, const Workspace &w, const InvSel &sel, int pair) {
    const int hp = (p.H + 1) >> 1;
    int cid, hh;
    if (sel.mode == 1) {
        const int per = sel.c0 * hp;
        const int seq = pair / per, rem = pair - seq * per, c = rem / hp;
        hh = rem - c * hp;
        cid = w.seqinfo[seq].z + c;
    } else if (sel.mode == 2) {
        const int per = p.N * hp;
        const int col = pair / per, rem = pair - col * per, seq = rem / hp;
        hh = rem - seq * hp;
        cid = w.seqinfo[seq].z + sel.c0 + col;
    } else {
        cid = pair / hp;
        hh = pair - cid * hp;
    }
    const int4 ci = w.chunks[cid];
    PairInfo pi;
    pi.t0 = ci.y;
    pi.len = ci.z;
    pi.col = ci.w;
    pi.h0 = 2 * hh;
    pi.h1 = min(2 * hh + 1, p.H - 1);
    return pi;
}

// The whole inverse for the pairs `sel` gives this CTA (kInvThreads threads,
// InvCfg<F32K>::kSmem bytes of dynamic shared memory at smem_raw; the caller
// has waited for the previous grid).  `kmap` is the key tensor map ([total_T,
// H, dk] rows, 128-byte swizzle; bf16 boxes of 64 features x 64 rows, or with
// F32K fp32 boxes of 32 features x 64 rows), features past dk read as zeros.
template <bool F32K = false>
__device__ __forceinline__ void inverse_tc_body(const CUtensorMap *kmap, const Problem &p, const Workspace &w,
                                                int gate_scaled, const InvSel &sel, uint8_t *smem_raw) {
    using Cfg = InvCfg<F32K>;
    constexpr int kStages = Cfg::kStages;
    constexpr uint32_t kPair = Cfg::kPair;
    constexpr uint32_t kOffSlots = Cfg::kOffSlots;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    InvBars &b = *reinterpret_cast<InvBars *>(smem + Cfg::kOffBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_pairs = sel_pairs(p, w, sel);
    // pairs of this CTA: sel.cta, sel.cta + sel.ctas, ...
    const int n_local = n_pairs > sel.cta ? (n_pairs - 1 - sel.cta) / sel.ctas + 1 : 0;
    if (n_local == 0) return;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&b.kfull[i], 1);
            tc::mbar_init(&b.kempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&b.tfull[i], 1);
            tc::mbar_init(&b.tempty[i], kInvConv * 32);
        }
        for (int i = 0; i < kInvSolvers; ++i) {
            tc::mbar_init(&b.afull[i], 64);
            tc::mbar_init(&b.aempty[i], 32);
        }
        b.abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) tc::tmem_alloc(&b.tmem_base, 512);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = b.tmem_base;

    if (warp == kInvConv + kInvSolvers) {
        // ---------------- TMA producer + MMA issuer: the whole warp runs the loop
        // (warp-uniform descriptors), one elected lane issues copies and MMAs
        const bool leader = tc::elect_one();
        constexpr uint32_t idesc = F32K ? tc::idesc_tf32_f32(128, 128) : tc::idesc_bf16_f32(128, 128, 0, 0);
        PairInfo pi_next = sel_pair(p, w, sel, sel.cta);   // info of the next pair to load
        auto load = [&](int i) -> bool {
            const int st = i % kStages;
            const uint32_t use = i / kStages;
            if (!inv_wait(b, &b.kempty[st], (use & 1) ^ 1, w.err)) return false;
            const PairInfo pi = pi_next;
            if (i + 1 < n_local) pi_next = sel_pair(p, w, sel, sel.cta + (i + 1) * sel.ctas);
            uint8_t *kt = smem + st * kPair;
            if (leader) {
                // [K1;K2] as 128 rows: each 128-byte feature block holds unit 0's
                // 64 rows, then unit 1's (bf16: 2 blocks of 64 features, fp32:
                // 4 blocks of 32)
                tc::mbar_arrive_expect_tx(&b.kfull[st], kPair);
                constexpr int kBlocks = F32K ? 4 : 2, kFeat = F32K ? 32 : 64;
#pragma unroll
                for (int fb = 0; fb < kBlocks; ++fb) {
                    tc::tma_load_3d(kt + fb * 16384, kmap, &b.kfull[st], fb * kFeat, pi.h0, pi.t0);
                    tc::tma_load_3d(kt + fb * 16384 + 8192, kmap, &b.kfull[st], fb * kFeat, pi.h1, pi.t0);
                }
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        int issued = 0, consumed = 0, mmas = 0;
        for (; issued < n_local && issued < kStages - 1 && ok; ++issued) ok = load(issued);
        if (!ok) --issued;
        for (int i = 0; i < n_local && ok; ++i) {
            if (issued < n_local) {
                if (!load(issued)) break;
                ++issued;
            }
            const int st = i % kStages, tb = i & 1;
            if (!inv_wait(b, &b.kfull[st], (i / kStages) & 1, w.err)) break;
            ++consumed;
            if (!inv_wait(b, &b.tempty[tb], ((i >> 1) & 1) ^ 1, w.err)) break;
            tc::tc_fence_after();
            const uint64_t d0 = tc::smem_desc_sw128(tc::smem_u32(smem + st * kPair), 16, 1024);
            if (leader) {
                // K-steps of 32 bytes: 16 bf16 features, or 8 fp32 ones (kind::tf32)
#pragma unroll
                for (int kk = 0; kk < (F32K ? 16 : 8); ++kk) {
                    const uint64_t d = d0 + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    if constexpr (F32K)
                        tc::mma_ss_tf32(tbase + tb * 128, d, d, idesc, kk > 0);
                    else
                        tc::mma_ss(tbase + tb * 128, d, d, idesc, kk > 0);
                }
                tc::tc_commit(&b.tfull[tb]);
                tc::tc_commit(&b.kempty[st]);
            }
            __syncwarp();
            ++mmas;
        }
        // After an abort: no copy may land and no MMA may run once the CTA is
        // gone.  Loads [consumed, issued) are each the latest use of their stage
        // and the last MMA the latest phase of its buffer, so their parities are
        // current.  (Waits are bounded; the abort flag is not consulted here.)
        int never = 0;
        for (int i = consumed; i < issued; ++i)
            tc::mbar_wait(&b.kfull[i % kStages], (i / kStages) & 1, &never, kInvTimeoutNs);
        if (mmas > 0) tc::mbar_wait(&b.tfull[(mmas - 1) & 1], ((mmas - 1) >> 1) & 1, &never, kInvTimeoutNs);
    } else if (warp < kInvConv) {
        // ---------------- converters: TMEM Gram rows -> packed A' rows
        const int half = warp >> 1;                 // unit 0 or 1 of the pair
        const int r = 32 * (warp & 1) + lane;       // row within the unit
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        // pair info two pairs ahead and beta one pair ahead, so that no global
        // load latency sits between two pairs
        auto beta_of = [&](const PairInfo &q) {
            const int hd = half ? q.h1 : q.h0;
            return r < q.len ? __ldg(&p.beta[(size_t)(q.t0 + r) * p.H + hd]) : 0.f;
        };
        // gate cumsum of this row, and the chunk's first and last (for c1)
        auto gate_of = [&](const PairInfo &q) {
            if (!gate_scaled) return make_float3(0.f, 0.f, 0.f);   // (no gate factors: G unread)
            const int hd = half ? q.h1 : q.h0;
            const float *Gh = w.G + (size_t)hd * p.total_T + q.t0;
            return make_float3(Gh[min(r, q.len - 1)], Gh[0], Gh[q.len - 1]);
        };
        PairInfo pi_next = sel_pair(p, w, sel, sel.cta);
        float br_next = beta_of(pi_next);
        float3 g_next = gate_of(pi_next);
        PairInfo pi_next2 = n_local > 1 ? sel_pair(p, w, sel, sel.cta + sel.ctas) : pi_next;
        for (int i = 0; i < n_local; ++i) {
            const PairInfo pi = pi_next;
            const float br = br_next;
            const float3 gr = g_next;
            pi_next = pi_next2;
            if (i + 1 < n_local) {
                br_next = beta_of(pi_next);
                g_next = gate_of(pi_next);
            }
            if (i + 2 < n_local) pi_next2 = sel_pair(p, w, sel, sel.cta + (i + 2) * sel.ctas);
            const int head = half ? pi.h1 : pi.h0;
            const int u = 2 * i + half, slot = u % kInvSolvers;
            const uint32_t use = u / kInvSolvers;
            const int tb = i & 1;
            bool ok = inv_wait(b, &b.tfull[tb], (i >> 1) & 1, w.err);
            ok = ok && inv_wait(b, &b.aempty[slot], (use & 1) ^ 1, w.err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::tc_fence_after();
            uint32_t g[64];
            tc::tmem_ld32(tbase + lane_base + tb * 128 + 64 * half, g);
            tc::tmem_ld32(tbase + lane_base + tb * 128 + 64 * half + 32, g + 32);
            tc::tmem_wait_ld();
            tc::tc_fence_before();
            tc::mbar_arrive(&b.tempty[tb]);
            float *sl = reinterpret_cast<float *>(smem + kOffSlots + slot * kInvSlotBytes);
            const int rb = r >> 4, ri = r & 15;
#pragma unroll
            for (int K = 0; K < 4; ++K) {
                if (K <= rb) {
                    float *dst = sl + block_index(rb, K) * 256 + ri;   // column-major block
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const int c = 16 * K + m;
                        dst[16 * m] = c < r ? br * __uint_as_float(g[c]) : 0.f;
                    }
                }
            }
            // c1_r of the gate-scaled T1 = T' diag(c1) (factored form; exact form: beta_r)
            const bool exact = gate_scaled && gr.z < -80.f;
            sl[kInvSlotFloats - 64 + r] =
                !gate_scaled ? 1.f : exact ? br : __expf(0.5f * (gr.y + gr.z) - gr.x) * br;
            if ((warp & 1) == 0 && lane == 0)
                b.unit[slot] = make_int4(pi.t0, pi.len, head,
                                         ((half && pi.h1 == pi.h0) ? 0 : 1) | (exact ? 2 : 0) | (pi.col << 8));
            tc::mbar_arrive(&b.afull[slot]);
        }
    } else {
        // ---------------- solvers: one unit per warp
        const int s = warp - kInvConv;
        const int j = lane;
        // this warp's 64 tensor-memory columns (its lane quadrant, above the Gram buffers)
        const uint32_t xcol = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 256 + 64 * (s >> 2);
        __nv_bfloat16 *tp = reinterpret_cast<__nv_bfloat16 *>(w.tprime);
        for (int u = s; u < 2 * n_local; u += kInvSolvers) {
            const uint32_t use = u / kInvSolvers;
            const bool ok = inv_wait(b, &b.afull[s], use & 1, w.err);
            if (!__all_sync(0xffffffffu, ok)) break;
            const int4 un = b.unit[s];
            const int len = un.y;
            const bool store = un.w & 1;
            uint8_t *slot_ptr = smem + kOffSlots + s * kInvSlotBytes;
            const uint32_t A = tc::smem_u32(slot_ptr);
            // The fused kernel consumes T1 = T' diag(c1) with the factored gate
            // c1_m = exp(G* - G_m) beta_m, G* the middle of the chunk's gate
            // range; a chunk whose last cumsum is below -80 takes the exact
            // form T1 = (Gamma ⊙ T') diag(beta) instead.  (The same rule, on
            // the same G values, picks the form in the fused kernel.)
            const bool exact = un.w & 2;
            const float *Gh = w.G + (size_t)un.z * p.total_T + un.x;
            const float *c1s = reinterpret_cast<const float *>(smem + kOffSlots + s * kInvSlotBytes) +
                               (kInvSlotFloats - 64);
            const float c1[2] = {c1s[j], c1s[32 + j]};
            float Gc[2] = {0.f, 0.f};
            if (exact) {
                Gc[0] = Gh[min(j, len - 1)];
                Gc[1] = Gh[min(32 + j, len - 1)];
            }
            if (sel.f32_out) {
                // T' as fp32 rows: column j over rows 0..63, then column 32 + j over
                // rows 32..63 (zero above); each store of a warp covers 128
                // contiguous bytes of one row
                float *rows = reinterpret_cast<float *>(w.tprime) + ((size_t)un.z * p.total_T + un.x) * kChunk;
                solve_blocked(A, xcol, j, 0);
                uint32_t v[64];
                tc::tmem_ld32(xcol, v);
                tc::tmem_ld32(xcol + 32, v + 32);
                tc::tmem_wait_ld();
                if (store) {
#pragma unroll
                    for (int r = 0; r < 64; ++r)
                        if (r < len) rows[(size_t)r * kChunk + j] = __uint_as_float(v[r]);
                }
                solve_blocked(A, xcol, 32 + j, 2);
                tc::tmem_ld32(xcol + 32, v + 32);
                tc::tmem_wait_ld();
                if (store) {
#pragma unroll
                    for (int r = 0; r < 64; ++r)
                        if (r < len) rows[(size_t)r * kChunk + 32 + j] = r < 32 ? 0.f : __uint_as_float(v[r]);
                }
                __syncwarp();
                tc::mbar_arrive(&b.aempty[s]);
                continue;
            }
            // pass A: column j over rows 0..63 -> x in columns xcol .. xcol+63;
            // then scaled and packed to bf16 pairs of rows in columns xcol .. xcol+31
            solve_blocked(A, xcol, j, 0);
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[32], pk[16];
                tc::tmem_ld32(xcol + 32 * hh, v);
                tc::tmem_wait_ld();
                if (exact) exact_gamma_rows(v, 32 * hh, Gh, Gc[0], len);
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    pk[t] = tc::pack_bf16x2(c1[0] * __uint_as_float(v[2 * t]), c1[0] * __uint_as_float(v[2 * t + 1]));
                tc::tmem_st16(xcol + 16 * hh, pk);
                tc::tmem_wait_st();
            }
            // pass B: column 32 + j over rows 32..63 -> columns xcol+32 .. xcol+63
            solve_blocked(A, xcol, 32 + j, 2);
            // A' is dead: the slot becomes the row-major bf16 T1 tile [64][64]
            __syncwarp();
            {
                uint32_t v[32];
                tc::tmem_ld32(xcol, v);   // 0..15: packed pass A; 16..31: unused
                tc::tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    sts_u16(A + (2 * t) * 128 + 2 * j, v[t]);
                    sts_u16(A + (2 * t + 1) * 128 + 2 * j, v[t] >> 16);
                }
                tc::tmem_ld16(xcol + 16, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    sts_u16(A + (32 + 2 * t) * 128 + 2 * j, v[t]);
                    sts_u16(A + (32 + 2 * t + 1) * 128 + 2 * j, v[t] >> 16);
                }
                tc::tmem_ld32(xcol + 32, v);
                tc::tmem_wait_ld();
                if (exact) exact_gamma_rows(v, 32, Gh, Gc[1], len);
#pragma unroll
                for (int r = 0; r < 32; ++r) sts_u16(A + r * 128 + 64 + 2 * j, 0u);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint32_t pv =
                        tc::pack_bf16x2(c1[1] * __uint_as_float(v[2 * t]), c1[1] * __uint_as_float(v[2 * t + 1]));
                    sts_u16(A + (32 + 2 * t) * 128 + 64 + 2 * j, pv);
                    sts_u16(A + (32 + 2 * t + 1) * 128 + 64 + 2 * j, pv >> 16);
                }
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && store && len > 0) {
                tc::bulk_store(tp + ((size_t)un.z * p.total_T + un.x) * kChunk, slot_ptr, (uint32_t)len * 128u);
                tc::bulk_commit_group();
                if (sel.mode == 2) {
                    // the rows are in memory before the column count says so
                    tc::bulk_wait_group_all();
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sel.ready + (un.w >> 8)) : "memory");
                } else {
                    tc::bulk_wait_group_read_all();
                }
            }
            __syncwarp();
            tc::mbar_arrive(&b.aempty[s]);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, 512);
    }
}

}  // namespace
}  // namespace gdn
