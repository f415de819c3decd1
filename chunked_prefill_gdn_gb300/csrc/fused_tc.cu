// tcgen05 fused chunk kernel for bf16 inputs with dk = dv = 128: steps two to
// four of the four-step paragraph of the FlashQLA talk
// "Qwen系列模型线性注意力高性能优化实践", with the state in tensor memory.
//
// Everything is written transposed so that the state's value index i (dv =
// 128) runs along the 128 TMEM lanes and every MMA has M = 128.  Per chunk,
// with S the state at chunk start (dv x dk, fp32 in TMEM), G the chunk-local
// gate cumsum, gamma = exp(G), Gamma_ri = exp(G_r - G_m):
//
//   MMA1  P^T   = S [K;Q]^T                      (A = bf16(S) from TMEM, N = 128)
//   E2    V'^T  = diag-beta (V^T - P_K^T D_gamma)   forward merge ("V - S first")
//   MMA2  U^T   = V'^T T^T,   T = Gamma ⊙ T'     (T' from the inverse kernel)
//   E3    Ut^T  = U^T diag(gamma_C / gamma)
//   MMA3  S    += Ut^T K      (S pre-scaled by gamma_C in E1)
//   P0    Q K^T                                   (for the output, off the chain)
//   MMA4  D4^T  = U^T (Gamma ⊙ tril(Q K^T))^T
//   O     o     = scale (D_gamma P_Q + D4)
//
// W, U and the per-chunk states never reach HBM.  Warp roles: warps 0-7 are
// the epilogue (warps w and w+4 share TMEM lane quadrant w % 4 and split the
// columns), warp 8 feeds q/k/v/T' tiles by TMA into a two-stage ring, warp 9
// allocates TMEM and issues the MMAs.  Every wait is bounded: on timeout the
// kernel records GDN_ERR_TIMEOUT, waits for its own copies in flight, frees
// TMEM and returns.
#include <string.h>

#include <mutex>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {

using namespace tc;

namespace {

constexpr int kD = 128;
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint64_t kTimeoutNs = 2000000000ull;

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t kKQBytes = 32768;  // [dk half][K rows 0-63 | Q rows 64-127][128 B]
constexpr uint32_t kVBytes = 16384;   // [dv half][64 rows][128 B]
constexpr uint32_t kTPBytes = 8192;   // [64 rows][128 B]: T', then T = Gamma ⊙ T'
constexpr uint32_t kStageBytes = kKQBytes + kVBytes + kTPBytes;
constexpr uint32_t kOffQM = 2 * kStageBytes;        // Gamma ⊙ tril(Q K^T), [64][128 B]
constexpr uint32_t kOffO = kOffQM + 8192;           // output tile [dv half][64][128 B]
constexpr uint32_t kOffSmall = kOffO + 16384;
constexpr uint32_t kTxBytes = kStageBytes;

// TMEM columns (512 allocated)
constexpr uint32_t kColS32 = 0;    // fp32 state, 128 cols
constexpr uint32_t kColS16 = 128;  // bf16 state (MMA1 A operand), 64 cols
constexpr uint32_t kColP = 192;    // MMA1 out: P_K^T cols 0-63 (V'^T bf16 at +16..+47), P_Q^T cols 64-127
constexpr uint32_t kColU = 320;    // MMA2 out: U^T fp32 64 cols (Ut^T bf16 at +16..+47)
constexpr uint32_t kColU16 = 384;  // U^T bf16 (MMA4 A operand), 32 cols
constexpr uint32_t kColD0 = 416;   // Q K^T (P0 out, lanes 64-127), then D4 (MMA4 out), 64 cols

struct Small {
    float G[2][64];
    float B[2][64];
    float coef[2][5][64];  // gamma, beta*gamma, gamma_C/gamma, Gamma row factor, Gamma column factor
    uint64_t full[2], empty[2];
    uint64_t e1, e2, e3, oepi, coefb, ofree, otile;
    uint64_t m1, m2, m3, m4, p0, fin;
    uint32_t tmem_base;
    int abort;
};

constexpr uint32_t kSmemBytes = kOffSmall + sizeof(Small) + 1024;

struct TcMaps {
    CUtensorMap q, k, v, o, tp;
};

struct Ctx {
    const TcMaps *maps;
    uint8_t *smem;
    Small *sm;
    const Problem *p;
    const Workspace *w;
    const gdn_work_item *items;
    int n_items;
    uint32_t tbase;
};

__device__ __forceinline__ bool wait_or_abort(const Ctx &cx, uint64_t *bar, uint32_t parity) {
    if (mbar_wait(bar, parity, &cx.sm->abort, kTimeoutNs)) return true;
    if (atomicExch(&cx.sm->abort, 1) == 0) report_error(cx.w->err, GDN_ERR_TIMEOUT);
    return false;
}

// Epilogue waits: every lane waits, and the warp gives up together, so the
// warp-collective tcgen05.ld/st that follow are never reached by part of a warp.
__device__ __forceinline__ bool ewait(const Ctx &cx, uint64_t *bar, uint32_t parity) {
    const bool r = wait_or_abort(cx, bar, parity);
    return __all_sync(0xffffffffu, r);
}

// ---------------------------------------------------------------- producer
__device__ void producer_role(const Ctx &cx, const TcMaps &maps, int lane) {
    const Problem &p = *cx.p;
    const Workspace &w = *cx.w;
    Small &sm = *cx.sm;
    uint32_t n = 0;
    uint32_t arms0 = 0, arms1 = 0;
    bool ok = true;
    for (int k = blockIdx.x; k < cx.n_items && ok; k += gridDim.x) {
        const gdn_work_item it = cx.items[k];
        const int4 si = w.seqinfo[it.seq];
        const int h = it.head;
        for (int c = it.c_start; c < it.c_end; ++c, ++n) {
            const int s = n & 1;
            if (n >= 2 && !wait_or_abort(cx, &sm.empty[s], ((n >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            const int4 ci = w.chunks[si.z + c];
            const int t0 = ci.y, len = ci.z;
            for (int rr = lane; rr < 64; rr += 32) {
                const int rc = rr < len ? rr : len - 1;
                sm.G[s][rr] = w.G[(size_t)h * p.total_T + t0 + rc];
                sm.B[s][rr] = rr < len ? p.beta[(size_t)(t0 + rr) * p.H + h] : 0.f;
            }
            uint8_t *st = cx.smem + s * kStageBytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&sm.full[s], kTxBytes);
                tma_load_3d(st + 0, &maps.k, &sm.full[s], 0, h, t0);
                tma_load_3d(st + 8192, &maps.q, &sm.full[s], 0, h, t0);
                tma_load_3d(st + 16384, &maps.k, &sm.full[s], 64, h, t0);
                tma_load_3d(st + 24576, &maps.q, &sm.full[s], 64, h, t0);
                tma_load_3d(st + kKQBytes, &maps.v, &sm.full[s], 0, h, t0);
                tma_load_3d(st + kKQBytes + 8192, &maps.v, &sm.full[s], 64, h, t0);
                tma_load_2d(st + kKQBytes + kVBytes, &maps.tp, &sm.full[s], 0, h * p.total_T + t0);
            } else {
                mbar_arrive(&sm.full[s]);
            }
            if (s) ++arms1; else ++arms0;
        }
    }
    // never leave a copy in flight into shared memory that is about to be released
    if (lane == 0) {
        int dummy = 0;
        if (arms0) mbar_wait(&sm.full[0], (arms0 - 1) & 1, &dummy, kTimeoutNs);
        if (arms1) mbar_wait(&sm.full[1], (arms1 - 1) & 1, &dummy, kTimeoutNs);
    }
}

// --------------------------------------------------------------------- MMA
__device__ void mma_role(const Ctx &cx) {
    const Workspace &w = *cx.w;
    Small &sm = *cx.sm;
    const uint32_t t = cx.tbase;
    const uint32_t smem0 = smem_u32(cx.smem);
    constexpr uint32_t I1 = idesc_bf16_f32(128, 128, 0, 0);  // P^T = S16 x [K;Q]^T
    constexpr uint32_t I0 = idesc_bf16_f32(128, 64, 0, 0);   // [K;Q] K^T
    constexpr uint32_t I2 = idesc_bf16_f32(128, 64, 0, 0);   // U^T = V'^T T^T
    constexpr uint32_t I3 = idesc_bf16_f32(128, 128, 0, 1);  // S += Ut^T K   (K as MN-major B)
    constexpr uint32_t I4 = idesc_bf16_f32(128, 64, 0, 0);   // D4^T = U^T Qm^T
    uint32_t n = 0;
    bool ok = true;
    for (int k = blockIdx.x; k < cx.n_items && ok; k += gridDim.x) {
        const gdn_work_item it = cx.items[k];
        for (int c = it.c_start; c < it.c_end; ++c, ++n) {
            const int s = n & 1;
            const uint32_t par = n & 1;
            const bool out = (it.flags & GDN_ITEM_OUTPUT) && c >= it.c_begin;
            const uint32_t kq = smem0 + s * kStageBytes;
            const uint32_t tp = kq + kKQBytes + kVBytes;
            if (!wait_or_abort(cx, &sm.full[s], (n >> 1) & 1) || !wait_or_abort(cx, &sm.e1, par)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t b = smem_desc_sw128(kq + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                mma_ts(t + kColP, t + kColS16 + 8 * kk, b, I1, kk > 0);
            }
            tc_commit(&sm.m1);
            if (n > 0 && !wait_or_abort(cx, &sm.oepi, (n - 1) & 1)) {
                ok = false;
                break;
            }
            if (out) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t a = smem_desc_sw128(kq + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    mma_ss(t + kColD0, a, a, I0, kk > 0);
                }
            }
            tc_commit(&sm.p0);
            if (!wait_or_abort(cx, &sm.e2, par)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t b = smem_desc_sw128(tp + kk * 32, 16, 1024);
                mma_ts(t + kColU, t + kColP + 16 + 8 * kk, b, I2, kk > 0);
            }
            tc_commit(&sm.m2);
            if (!wait_or_abort(cx, &sm.e3, par)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t b = smem_desc_sw128(kq + kk * 2048, 16384, 1024);
                mma_ts(t + kColS32, t + kColU + 16 + 8 * kk, b, I3, 1);
            }
            tc_commit(&sm.m3);
            if (out) {
                const uint32_t qm = smem0 + kOffQM;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t b = smem_desc_sw128(qm + kk * 32, 16, 1024);
                    mma_ts(t + kColD0, t + kColU16 + 8 * kk, b, I4, kk > 0);
                }
            }
            tc_commit(&sm.m4);
            tc_commit(&sm.empty[s]);
        }
    }
    (void)w;
    // all issued MMAs must finish before TMEM is released
    tc_commit(&sm.fin);
    int dummy = 0;
    mbar_wait(&sm.fin, 0, &dummy, kTimeoutNs);
}

// ---------------------------------------------------------------- epilogue
struct EpiThread {
    int q, ch, i, et, lane;
    uint32_t lane_base;  // TMEM lane field of this warp's quadrant
};

__device__ __forceinline__ float gamma_rm(const float *G, const float *ga, const float *gb, bool exact, int r,
                                          int m) {
    return exact ? __expf(G[r] - G[m]) : ga[r] * gb[m];
}

__device__ __forceinline__ void load_tile32(const Ctx &cx, const EpiThread &e, uint32_t col, float *x) {
    uint32_t r[32];
    tmem_ld32(cx.tbase + e.lane_base + col, r);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
}

// Stores 32 state columns j0 .. j0+31 (key index) of this thread's value row.
__device__ void write_state32(const Ctx &cx, const EpiThread &e, const gdn_work_item &it, int j0, const float *sv) {
    const Problem &p = *cx.p;
    const Workspace &w = *cx.w;
    const int i = e.i;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        if (it.flags & GDN_ITEM_WRITE_FINAL)
            p.sf[(((size_t)it.seq * p.H + it.head) * kD + j) * kD + i] = sv[jj];
        if (it.flags & GDN_ITEM_WRITE_SLOT) w.cp_s[((size_t)it.slot * kD + j) * kD + i] = sv[jj];
        if (it.flags & GDN_ITEM_WRITE_M) w.cp_m[((size_t)it.slot * kD + j) * kD + i] = sv[jj];
    }
}

// Loads 32 start-state columns j0 .. j0+31 of this thread's value row.
__device__ void load_start_state32(const Ctx &cx, const EpiThread &e, const gdn_work_item &it, int j0, float *sv) {
    const Problem &p = *cx.p;
    const Workspace &w = *cx.w;
    const int i = e.i;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        float x = 0.f;
        if (it.flags & GDN_ITEM_FROM_INITIAL) {
            if (p.s0) x = p.s0[(((size_t)it.seq * p.H + it.head) * kD + j) * kD + i];
        } else if (it.flags & GDN_ITEM_FROM_IDENTITY) {
            x = (i == j) ? 1.f : 0.f;
        } else if (it.flags & GDN_ITEM_FROM_SLOT) {
            x = w.cp_s[((size_t)it.slot * kD + j) * kD + i];
        }
        sv[jj] = x;
    }
}

// Writes the state held in TMEM (this thread's row, its 64 columns) for `it`.
__device__ void flush_state(const Ctx &cx, const EpiThread &e, const gdn_work_item &it) {
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

__device__ void epilogue_role(const Ctx &cx, int warp, int lane) {
    const Problem &p = *cx.p;
    const Workspace &w = *cx.w;
    Small &sm = *cx.sm;
    EpiThread e;
    e.q = warp & 3;
    e.ch = warp >> 2;
    e.i = 32 * e.q + lane;
    e.et = threadIdx.x;
    e.lane = lane;
    e.lane_base = static_cast<uint32_t>(32 * e.q) << 16;
    const int ch = e.ch, i = e.i;
    uint8_t *qm_tile = cx.smem + kOffQM;
    uint8_t *o_tile = cx.smem + kOffO;

    uint32_t n = 0, ocount = 0;
    int pv_out = 0, pv_t0 = 0, pv_len = 0, pv_h = 0;
    // the item whose end state sits in TMEM and has not been written yet
    bool pending = false;
    gdn_work_item prev_item;
    prev_item.flags = 0;
    float pq[32];
    bool ok = true;

    for (int k = blockIdx.x; k < cx.n_items && ok; k += gridDim.x) {
        const gdn_work_item it = cx.items[k];
        const int4 si = w.seqinfo[it.seq];
        const bool ident = it.flags & GDN_ITEM_FROM_IDENTITY;
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
            const int s = n & 1;
            const uint32_t par = n & 1;
            const int4 ci = w.chunks[si.z + c];
            const int t0 = ci.y, len = ci.z;
            const bool out = (it.flags & GDN_ITEM_OUTPUT) && c >= it.c_begin;
            uint8_t *st = cx.smem + s * kStageBytes;
            const uint8_t *vt = st + kKQBytes;
            uint8_t *tpt = st + kKQBytes + kVBytes;
            if (!ewait(cx, &sm.full[s], (n >> 1) & 1)) { ok = false; break; }

            // ---- per-chunk coefficients
            const float *G = sm.G[s];
            if (e.et < 64) {
                const int r = e.et;
                const float Gr = G[r], Gc = G[63];
                const float Gref = 0.5f * (G[0] + Gc);
                const float gam = __expf(Gr);
                sm.coef[s][0][r] = gam;
                sm.coef[s][1][r] = sm.B[s][r] * gam;
                sm.coef[s][2][r] = __expf(Gc - Gr);
                sm.coef[s][3][r] = __expf(Gr - Gref);
                sm.coef[s][4][r] = __expf(Gref - Gr);
                mbar_arrive(&sm.coefb);
            }
            if (!ewait(cx, &sm.coefb, par)) { ok = false; break; }
            const float *gam = sm.coef[s][0], *bg = sm.coef[s][1], *dec = sm.coef[s][2];
            const float *ga = sm.coef[s][3], *gb = sm.coef[s][4];
            const bool exact = (G[0] - G[63]) > 160.f;

            // ---- T = Gamma ⊙ T' in place (rows 0-63 by quadrants 0 and 1)
            if (e.q < 2) {
                const int r = i;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c16 = 4 * ch + cc;
                    uint4 *ptr = reinterpret_cast<uint4 *>(tpt + sw128_offset(r, c16));
                    uint4 v = *ptr;
                    uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const int m0 = 8 * c16 + 2 * e2;
                        float x0 = bf16_lo(wv[e2]), x1 = bf16_hi(wv[e2]);
                        x0 = (r < len && m0 <= r) ? x0 * gamma_rm(G, ga, gb, exact, r, m0) : 0.f;
                        x1 = (r < len && m0 + 1 <= r) ? x1 * gamma_rm(G, ga, gb, exact, r, m0 + 1) : 0.f;
                        wv[e2] = pack_bf16x2(x0, x1);
                    }
                    *ptr = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                fence_proxy_async_smem();
            }
            // ---- beta_r V[r][i] for this thread's 32 rows
            float vb[32];
            {
                const int half = i >> 6, col = i & 63;
#pragma unroll
                for (int rr = 0; rr < 32; ++rr) {
                    const int r = 32 * ch + rr;
                    const uint16_t raw = *reinterpret_cast<const uint16_t *>(
                        vt + half * 8192 + sw128_offset(r, col >> 3) + (col & 7) * 2);
                    vb[rr] = ident ? 0.f : sm.B[s][r] * __uint_as_float(static_cast<uint32_t>(raw) << 16);
                }
            }

            // ---- E1: S16 = bf16(S), S32 = gamma_C S
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
                    store_state32(cx, e, hh, sv, gam[63]);
                }
            } else {
                if (!ewait(cx, &sm.m3, (n - 1) & 1)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float sv[32];
                    load_tile32(cx, e, kColS32 + 64 * ch + 32 * hh, sv);
                    store_state32(cx, e, hh, sv, gam[63]);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.e1);

            // ---- output of the previous chunk
            if (n > 0) {
                if (!ewait(cx, &sm.m4, (n - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (pv_out) {
                    float d4[32];
                    load_tile32(cx, e, kColD0 + 32 * ch, d4);
                    if (pv_len == 64) {
                        if (e.et == 0) {
                            bulk_wait_group_read_all();
                            mbar_arrive(&sm.ofree);
                        }
                        if (!ewait(cx, &sm.ofree, ocount & 1)) { ok = false; break; }
                        const int half = i >> 6, col = i & 63;
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr) {
                            const int r = 32 * ch + rr;
                            const __nv_bfloat16 b = __float2bfloat16_rn(p.scale * (pq[rr] + d4[rr]));
                            *reinterpret_cast<__nv_bfloat16 *>(o_tile + half * 8192 + sw128_offset(r, col >> 3) +
                                                               (col & 7) * 2) = b;
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(&sm.otile);
                        if (e.et == 0) {
                            if (!wait_or_abort(cx, &sm.otile, ocount & 1)) { ok = false; break; }
                            tma_store_3d(&cx.maps->o, o_tile, 0, pv_h, pv_t0);
                            tma_store_3d(&cx.maps->o, o_tile + 8192, 64, pv_h, pv_t0);
                            bulk_commit_group();
                        }
                        ++ocount;
                    } else {
                        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.o);
                        for (int rr = 0; rr < 32; ++rr) {
                            const int r = 32 * ch + rr;
                            if (r < pv_len)
                                o[((size_t)(pv_t0 + r) * p.H + pv_h) * kD + i] =
                                    __float2bfloat16_rn(p.scale * (pq[rr] + d4[rr]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&sm.oepi);
            }

            // ---- E2: V'^T = beta (V^T - gamma P_K^T)
            if (!ewait(cx, &sm.m1, par)) { ok = false; break; }
            tc_fence_after();
            {
                float pk[32];
                load_tile32(cx, e, kColP + 32 * ch, pk);
                uint32_t vp[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r0 = 32 * ch + 2 * j;
                    vp[j] = pack_bf16x2(vb[2 * j] - bg[r0] * pk[2 * j], vb[2 * j + 1] - bg[r0 + 1] * pk[2 * j + 1]);
                }
                tmem_st16(cx.tbase + e.lane_base + kColP + 16 + 16 * ch, vp);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&sm.e2);

            // ---- P_Q and the masked Q K^T
            if (!ewait(cx, &sm.p0, par)) { ok = false; break; }
            tc_fence_after();
            if (out) {
                load_tile32(cx, e, kColP + 64 + 32 * ch, pq);
#pragma unroll
                for (int rr = 0; rr < 32; ++rr) pq[rr] *= gam[32 * ch + rr];
                if (e.q >= 2) {
                    const int r = i - 64;
                    float qk[32];
                    load_tile32(cx, e, kColD0 + 32 * ch, qk);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t wv[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const int mm = 8 * cc + 2 * e2;
                            const int m0 = 32 * ch + mm;
                            const float x0 =
                                (r < len && m0 <= r) ? qk[mm] * gamma_rm(G, ga, gb, exact, r, m0) : 0.f;
                            const float x1 =
                                (r < len && m0 + 1 <= r) ? qk[mm + 1] * gamma_rm(G, ga, gb, exact, r, m0 + 1) : 0.f;
                            wv[e2] = pack_bf16x2(x0, x1);
                        }
                        *reinterpret_cast<uint4 *>(qm_tile + sw128_offset(r, 4 * ch + cc)) =
                            make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                    fence_proxy_async_smem();
                }
            }

            // ---- E3: Ut^T = U^T diag(gamma_C / gamma), U^T in bf16 for the output MMA
            if (!ewait(cx, &sm.m2, par)) { ok = false; break; }
            tc_fence_after();
            {
                float u[32];
                load_tile32(cx, e, kColU + 32 * ch, u);
                uint32_t ut[16], ub[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r0 = 32 * ch + 2 * j;
                    ut[j] = pack_bf16x2(u[2 * j] * dec[r0], u[2 * j + 1] * dec[r0 + 1]);
                    ub[j] = pack_bf16x2(u[2 * j], u[2 * j + 1]);
                }
                tmem_st16(cx.tbase + e.lane_base + kColU + 16 + 16 * ch, ut);
                tmem_st16(cx.tbase + e.lane_base + kColU16 + 16 * ch, ub);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&sm.e3);
            mbar_arrive(&sm.empty[s]);

            pv_out = out;
            pv_t0 = t0;
            pv_len = len;
            pv_h = it.head;
        }
        if (!ok) break;
        prev_item = it;
        pending = true;
    }
    // tail: output of the last chunk and the last item's state
    if (ok && n > 0) {
        if (ewait(cx, &sm.m4, (n - 1) & 1)) {
            tc_fence_after();
            if (pv_out) {
                float d4[32];
                load_tile32(cx, e, kColD0 + 32 * ch, d4);
                __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.o);
                for (int rr = 0; rr < 32; ++rr) {
                    const int r = 32 * ch + rr;
                    if (r < pv_len)
                        o[((size_t)(pv_t0 + r) * p.H + pv_h) * kD + i] = __float2bfloat16_rn(p.scale * (pq[rr] + d4[rr]));
                }
            }
        }
        if (pending && ewait(cx, &sm.m3, (n - 1) & 1)) {
            tc_fence_after();
            flush_state(cx, e, prev_item);
        }
    }
    if (e.et == 0) bulk_wait_group_all();
}

// ---------------------------------------------------------------- kernel
// 10 warps share the 4 SM sub-partitions 3/3/2/2, so a thread may hold at most
// 16384 / (3 * 32) registers: 168 after rounding.
__global__ void __launch_bounds__(kThreads, 1)
    fused_tc_kernel(const __grid_constant__ TcMaps maps, const Problem p, const Workspace w, const int pass) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small &sm = *reinterpret_cast<Small *>(smem + kOffSmall);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.full[s], 32);
            mbar_init(&sm.empty[s], 1 + kEpiThreads);
        }
        mbar_init(&sm.e1, kEpiThreads);
        mbar_init(&sm.e2, kEpiThreads);
        mbar_init(&sm.e3, kEpiThreads);
        mbar_init(&sm.oepi, kEpiThreads);
        mbar_init(&sm.coefb, 64);
        mbar_init(&sm.ofree, 1);
        mbar_init(&sm.otile, kEpiThreads);
        mbar_init(&sm.m1, 1);
        mbar_init(&sm.m2, 1);
        mbar_init(&sm.m3, 1);
        mbar_init(&sm.m4, 1);
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
        tma_prefetch_map(&maps.o);
        tma_prefetch_map(&maps.tp);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    Ctx cx;
    cx.maps = &maps;
    cx.smem = smem;
    cx.sm = &sm;
    cx.p = &p;
    cx.w = &w;
    cx.items = pass == 2 ? w.items2 : w.items1;
    cx.n_items = *(volatile const int *)&w.num_items[pass == 2 ? 0 : 1];
    cx.tbase = sm.tmem_base;

    if (warp == kProducerWarp) {
        producer_role(cx, maps, lane);
    } else if (warp == kMmaWarp) {
        if (lane == 0) mma_role(cx);
        __syncwarp();
    } else {
        epilogue_role(cx, warp, lane);
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

// [total_T, H, 128] bf16 rows, boxes of 64 tokens x 64 features, 128-byte swizzle;
// returns the driver result (0 on success)
int encode_rows(EncodeTiledFn fn, CUtensorMap *m, const void *base, int H, int total_T) {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)total_T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

bool fused_tc_supported(int dtype, int dk, int dv) { return dtype == GDN_BF16 && dk == kD && dv == kD; }

cudaError_t launch_fused_tc(const Problem &p, const Workspace &w, int pass, int grid, cudaStream_t s) {
    if (!fused_tc_supported(p.dtype, p.dk, p.dv)) return cudaErrorNotSupported;
    if (p.total_T == 0) return launch_fused_simt(p, w, pass, grid, s);  // only empty sequences: nothing to tile
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
    if ((r = encode_rows(fn, &maps.q, p.q, p.H, p.total_T)) || (r = encode_rows(fn, &maps.k, p.k, p.H, p.total_T)) ||
        (r = encode_rows(fn, &maps.v, p.v, p.H, p.total_T)) || (r = encode_rows(fn, &maps.o, p.o, p.H, p.total_T)) ||
        (r = fn(&maps.tp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.tprime, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE))) {
        set_error_detail("encode tensor map", cudaErrorInvalidValue, r);
        return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(fused_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    fused_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(maps, p, w, pass);
    return cudaGetLastError();
}

}  // namespace gdn
