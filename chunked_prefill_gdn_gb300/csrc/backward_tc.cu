// Tensor-core backward of the chunked GDN forward (tcgen05, kind::tf32): the
// gradients of q, k, v, g, beta and the initial state from those of o and of
// the final state.  The algebra is the chain rule through one chunk of the WY
// form (the backward paragraph of the talk "Qwen系列模型线性注意力高性能优化实践";
// math orientation, S dv x dk, start state S0, end-state gradient dS, chunk-local
// G = cumsum g, gamma = exp(G), Gamma_rm = exp(G_r - G_m), e = gamma_C / gamma):
//
//   forward   Y = K S0^T, X = D_gamma Y, B = diag(beta)(V - X), U = T B,
//             M = Gamma ⊙ tril(Q K^T), S_C = gamma_C S0 + U^T D_e K
//   backward  dU = scale M^T dO + D_e K dS^T,  dB = T^T dU,  dv = diag(beta) dB,
//             dS0 = gamma_C dS + scale dO^T D_gamma Q - dB^T D_gamma diag(beta) K,
//             dM = scale dO U^T (lower),  dA = -dB U^T (strictly lower),
//             P = dA ⊙ Gamma ⊙ beta_r,  R = dM ⊙ Gamma,
//             dK = (P + P^T) K + R^T Q + D_gamma dX S0 + D_e U dS   (dX = -diag(beta) dB)
//             dQ = R K + scale D_gamma dO S0,
//             dbeta and dG from every place beta and G enter (dg: the reverse
//             cumsum of dG inside the chunk)
//
// Two kernels.  The chain kernel (one CTA per (head, sequence)) carries the
// state forward over the chunks (storing each chunk's start state transposed,
// and the rows of K S0^T, Q S0^T and U), then the state gradient back (storing
// each chunk's end-state gradient transposed and the rows of dB and K dS^T,
// and writing dv and the initial state's gradient).  The chunk kernel (one CTA
// per (chunk, head), all independent) reads those and forms dq, dk, dg, dbeta.
// Every product is a tcgen05 MMA of M = 128 with fp32 operands read as tf32 and
// fp32 accumulation; the 128-wide dimension (value rows in the chain kernel, key
// columns in the chunk kernel) runs along the TMEM lanes, padded with zeros
// for head sizes 32 and 64.  Operands are staged by the CTA's threads as
// 128-byte-swizzled K-major fp32 tiles; T = Gamma ⊙ T' comes from the T' of the
// per-chunk inverse (Gamma-extraction identity).  Every wait on an MMA is
// bounded: on timeout the kernels record GDN_ERR_TIMEOUT and return.
#include <math.h>

#include <type_traits>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {

using namespace tc;

namespace {

constexpr int kBT = 512;                      // threads: warps w, w + 4, w + 8, w + 12 share TMEM lane quadrant w
constexpr int kParts = kBT / 128;             // warps per lane quadrant: each takes 16 of 64 columns (32 of 128)
constexpr uint64_t kBtTimeoutNs = 2000000000ull;
constexpr uint32_t kBlk128 = 16384;           // block stride of a 128-row fp32 tile
constexpr uint32_t kBlk64 = 8192;             // block stride of a 64-row fp32 tile

struct BtCoef {
    float G[64], beta[64], gam[64], e[64];    // rows past the chunk: g = beta = 0 (G repeats the last)
};

template <typename TI>
__device__ __forceinline__ float4 ld4(const TI *p);
template <>
__device__ __forceinline__ float4 ld4<float>(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}
template <typename TI>
__device__ __forceinline__ float ld1(const TI *p) {
    if constexpr (std::is_same<TI, float>::value) return __ldg(p);
    else return __bfloat162float(*p);
}

__device__ __forceinline__ void sts_f4(uint32_t a, float x, float y, float z, float w) {
    sts_u4_stage(a, make_uint4(__float_as_uint(x), __float_as_uint(y), __float_as_uint(z), __float_as_uint(w)));
}
__device__ __forceinline__ void sts_f32(uint32_t a, float x) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(x));
}

__device__ __forceinline__ float warp_sum(float x) {
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Gate and beta coefficients of a chunk (warp 0): inclusive scans of g over
// both halves, rows past len with g = 0.
__device__ __forceinline__ void chunk_coef(BtCoef *cf, const float *g, const float *b, int t0, int len, int H,
                                           int h) {
    const int lane = threadIdx.x & 31;
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
    if (lane < len) {
        g0 = g[(size_t)(t0 + lane) * H + h];
        b0 = b[(size_t)(t0 + lane) * H + h];
    }
    if (32 + lane < len) {
        g1 = g[(size_t)(t0 + 32 + lane) * H + h];
        b1 = b[(size_t)(t0 + 32 + lane) * H + h];
    }
    for (int off = 1; off < 32; off <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, g0, off);
        const float y1 = __shfl_up_sync(0xffffffffu, g1, off);
        if (lane >= off) { g0 += y0; g1 += y1; }
    }
    g1 += __shfl_sync(0xffffffffu, g0, 31);
    const float glast = __shfl_sync(0xffffffffu, g1, 31);
    cf->G[lane] = g0;
    cf->G[32 + lane] = g1;
    cf->gam[lane] = expf(g0);
    cf->gam[32 + lane] = expf(g1);
    cf->e[lane] = expf(glast - g0);
    cf->e[32 + lane] = expf(glast - g1);
    cf->beta[lane] = b0;
    cf->beta[32 + lane] = b1;
}

// The loaders below issue their global loads in batches of kLB per thread
// (all in flight) before the shared-memory stores: a store is an asm
// statement the compiler does not move loads across, so a load-store loop
// would wait one memory round trip per element.
constexpr int kLB = 4;

__device__ __forceinline__ int log2i(int x) { return 31 - __clz(x); }

// Tile rows row0 + r (r < 64) = f(r) x[t0 + r][0, d); zero past len.
template <typename TI, typename F>
__device__ __forceinline__ void tile_rows(uint32_t tile, uint32_t block, int row0, const TI *x, int t0, int len,
                                          int H, int h, int d, F f) {
    const int sh = log2i(d >> 2), total = 64 << sh;
    const TI *x0 = x + ((size_t)t0 * H + h) * d;     // row r at x0 + r * H * d
    const int stride = H * d;
    for (int base = threadIdx.x; base < total; base += kLB * kBT) {
        float4 v[kLB];
#pragma unroll
        for (int b = 0; b < kLB; ++b) {
            const int idx = base + b * kBT;
            const int r = idx >> sh, c4 = idx & ((1 << sh) - 1);
            v[b] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < total && r < len) {
                v[b] = ld4<TI>(x0 + r * stride + 4 * c4);
                const float s = f(r);
                v[b].x *= s; v[b].y *= s; v[b].z *= s; v[b].w *= s;
            }
        }
#pragma unroll
        for (int b = 0; b < kLB; ++b) {
            const int idx = base + b * kBT;
            if (idx < total) {
                const int r = idx >> sh, c4 = idx & ((1 << sh) - 1);
                sts_f4(tile + f32_tile_off(row0 + r, 4 * c4, block), v[b].x, v[b].y, v[b].z, v[b].w);
            }
        }
    }
}

// Tile row j < rows, columns r < 64: f(r) x[t0 + r][j] (zero for j >= d or
// r >= len).  Lanes take consecutive j, so the reads of a token row coalesce.
// rows is 32, 64 or 128.
template <typename TI, typename F>
__device__ __forceinline__ void tile_cols(uint32_t tile, uint32_t block, int rows, const TI *x, int t0, int len,
                                          int H, int h, int d, F f) {
    const int sh = log2i(rows), total = rows * 16;
    const TI *x0 = x + ((size_t)t0 * H + h) * d;
    const int stride = H * d;
    for (int base = threadIdx.x; base < total; base += kLB * kBT) {
        float e[kLB][4];
#pragma unroll
        for (int b = 0; b < kLB; ++b) {
            const int idx = base + b * kBT;
            const int r4 = idx >> sh, j = idx & (rows - 1);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = 4 * r4 + u;
                e[b][u] = (idx < total && j < d && r < len) ? f(r) * ld1<TI>(x0 + r * stride + j) : 0.f;
            }
        }
#pragma unroll
        for (int b = 0; b < kLB; ++b) {
            const int idx = base + b * kBT;
            if (idx < total) {
                const int r4 = idx >> sh, j = idx & (rows - 1);
                sts_f4(tile + f32_tile_off(j, 4 * r4, block), e[b][0], e[b][1], e[b][2], e[b][3]);
            }
        }
    }
}

// Tile row j < 128 = src[j][0, dv) for j < dk (zero past dk), src rows dv
// apart; with `dot`, also the sum over the tile of this times `dot_tile` at
// the same place (same block stride).
__device__ __forceinline__ float tile_state(uint32_t tile, const float *src, int dk, int dv, uint32_t dot_tile) {
    const int sh = log2i(dv >> 2), total = 128 << sh;
    float part = 0.f;
    for (int base = threadIdx.x; base < total; base += kLB * kBT) {
        float4 v[kLB];
#pragma unroll
        for (int b = 0; b < kLB; ++b) {
            const int idx = base + b * kBT;
            const int j = idx >> sh, c4 = idx & ((1 << sh) - 1);
            v[b] = (idx < total && j < dk) ? __ldg(reinterpret_cast<const float4 *>(src + (size_t)j * dv + 4 * c4))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < kLB; ++b) {
            const int idx = base + b * kBT;
            if (idx < total) {
                const int j = idx >> sh, c4 = idx & ((1 << sh) - 1);
                const uint32_t off = f32_tile_off(j, 4 * c4, kBlk128);
                if (dot_tile) {
                    const float4 o = lds_f4(dot_tile + off);
                    part += v[b].x * o.x + v[b].y * o.y + v[b].z * o.z + v[b].w * o.w;
                }
                sts_f4(tile + off, v[b].x, v[b].y, v[b].z, v[b].w);
            }
        }
    }
    return part;
}

// T = Gamma ⊙ T' rows [n][m] (fwd) or transposed [r][n] = T[n][r] (rev), from
// T' rows (row n at tp + 64 n, entries past the chunk not read).  1024 items:
// four per thread, loaded together.
__device__ __forceinline__ void tile_t(uint32_t tile, const float *tp, int len, const float *G) {
    constexpr int kN = 1024 / kBT;
    float4 t[kN];
#pragma unroll
    for (int b = 0; b < kN; ++b) {
        const int idx = threadIdx.x + b * kBT;
        const int n = idx >> 4, m4 = (idx & 15) * 4;
        t[b] = (n < len && m4 <= n) ? __ldg(reinterpret_cast<const float4 *>(tp + (size_t)n * 64 + m4))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int b = 0; b < kN; ++b) {
        const int idx = threadIdx.x + b * kBT;
        const int n = idx >> 4, m4 = (idx & 15) * 4;
        const float tv[4] = {t[b].x, t[b].y, t[b].z, t[b].w};
        float x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = (n < len && m4 + u <= n) ? tv[u] * expf(G[n] - G[m4 + u]) : 0.f;
        sts_f4(tile + f32_tile_off(n, m4, kBlk64), x[0], x[1], x[2], x[3]);
    }
}
__device__ __forceinline__ void tile_t_transposed(uint32_t tile, const float *tp, int len, const float *G) {
    constexpr int kN = 1024 / kBT;
    float x[kN][4];
#pragma unroll
    for (int b = 0; b < kN; ++b) {
        const int idx = threadIdx.x + b * kBT;
        const int n4 = idx >> 6, r = idx & 63;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int n = 4 * n4 + u;
            x[b][u] = (n < len && r <= n) ? __ldg(tp + (size_t)n * 64 + r) : 0.f;
        }
    }
#pragma unroll
    for (int b = 0; b < kN; ++b) {
        const int idx = threadIdx.x + b * kBT;
        const int n4 = idx >> 6, r = idx & 63;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int n = 4 * n4 + u;
            if (n < len && r <= n) x[b][u] *= expf(G[n] - G[r]);
        }
        sts_f4(tile + f32_tile_off(r, 4 * n4, kBlk64), x[b][0], x[b][1], x[b][2], x[b][3]);
    }
}

// L2 prefetch of the lines of `bytes` bytes at p (this thread's share).
__device__ __forceinline__ void prefetch_lines(const void *p, uint32_t bytes) {
    for (uint32_t o = 0; o < bytes; o += 128) l2_prefetch_line(static_cast<const char *>(p) + o);
}

// L2 prefetch of row r (r < len) of a [total_T][H][d] tensor (head h) by
// thread thr0 + r: one or two lines each.
template <typename T>
__device__ __forceinline__ void prefetch_rows(const T *x, int t0, int len, int H, int h, int d, int thr0) {
    const int r = (int)threadIdx.x - thr0;
    if (r >= 0 && r < len && r < 64) prefetch_lines(x + ((size_t)(t0 + r) * H + h) * d, (uint32_t)(d * sizeof(T)));
}

// The chain kernel's inputs of one chunk — K, Q and V or dO rows, the T'
// rows, the g and beta rows of all heads — a row or two lines per thread.
template <typename TI>
__device__ __forceinline__ void prefetch_chain_chunk(const BwdTcArgs &a, int t0, int len, int h, bool rev) {
    const TI *kg = static_cast<const TI *>(a.k), *qg = static_cast<const TI *>(a.q);
    const TI *xg = static_cast<const TI *>(rev ? a.dout : a.v);
    prefetch_rows(kg, t0, len, a.H, h, a.dk, 0);
    prefetch_rows(qg, t0, len, a.H, h, a.dk, 64);
    prefetch_rows(xg, t0, len, a.H, h, a.dv, 128);
    prefetch_rows(a.tp + (size_t)h * a.total_T * kChunk, t0, len, 1, 0, kChunk, 192);
    const int r = (int)threadIdx.x - 256;
    if (r >= 0 && r < 2 * len) {   // g and beta rows of the chunk (all heads)
        const float *x = (r < len ? a.g : a.beta) + (size_t)(t0 + (r < len ? r : r - len)) * a.H;
        prefetch_lines(x, (uint32_t)a.H * 4u);
    }
}

// Transposed copies out of a [K;Q] row tile in shared memory (K rows 0-63,
// Q rows 64-127, 128-byte-swizzled fp32, block stride kBlk128):
//   dst0[j][r] = f0(r) src[q0 + r][j],  dst1[j][r] = f1(r) src[q1 + r][j]
// for key rows j < rows (zero for j >= dk) and chunk rows r < 64 (n_dst = 1:
// dst0 only).  With
// `in_place` the destinations overlap the source, so every value is read
// into registers before a barrier and written after it.
template <typename F0, typename F1>
__device__ __forceinline__ void tile_transpose_kq(uint32_t src, uint32_t dst0, int q0, F0 f0, uint32_t dst1, int q1,
                                                  F1 f1, int rows, int dk, bool in_place, int n_dst = 2) {
    const int sh = log2i(rows), per = rows * 16;        // float4 items per destination
    const int items = n_dst * per;
    constexpr int kN = 2 * 128 * 16 / kBT;              // items per thread at rows = 128
    float e[kN][4];
#pragma unroll
    for (int b = 0; b < kN; ++b) {
        const int idx = threadIdx.x + b * kBT;
        const int which = idx >= per, k = idx - which * per;
        const int r4 = k >> sh, j = k & (rows - 1);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = 4 * r4 + u;
            float x = 0.f;
            if (idx < items && j < dk) {
                uint32_t a = src + f32_tile_off((which ? q1 : q0) + r, j, kBlk128);
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(x) : "r"(a));
                x *= which ? f1(r) : f0(r);
            }
            e[b][u] = x;
        }
    }
    if (in_place) __syncthreads();
#pragma unroll
    for (int b = 0; b < kN; ++b) {
        const int idx = threadIdx.x + b * kBT;
        if (idx < items) {
            const int which = idx >= per, k = idx - which * per;
            const int r4 = k >> sh, j = k & (rows - 1);
            sts_f4((which ? dst1 : dst0) + f32_tile_off(j, 4 * r4, kBlk128), e[b][0], e[b][1], e[b][2], e[b][3]);
        }
    }
}

struct One {
    __device__ float operator()(int) const { return 1.f; }
};

__device__ __forceinline__ bool bt_wait(uint64_t *bar, uint32_t parity, int *abort) {
    const bool ok = mbar_wait(bar, parity, abort, kBtTimeoutNs);
    return !__syncthreads_or(!ok);
}

// Sequence bounds of sequence n; false (and the error recorded) for bad cu_seqlens.
__device__ __forceinline__ bool seq_bounds(const BwdTcArgs &a, int n, int &t_begin, int &len_seq) {
    if (a.varlen) {
        const int c0 = a.cu[n], c1 = a.cu[n + 1];
        if (c0 < 0 || c1 < c0 || c1 > a.total_T || (n == 0 && c0 != 0) || (n == a.N - 1 && c1 != a.total_T)) {
            if (threadIdx.x == 0) report_error(a.err, GDN_ERR_DEVICE_CHECK);
            return false;
        }
        t_begin = c0;
        len_seq = c1 - c0;
    } else {
        t_begin = n * a.T;
        len_seq = a.T;
    }
    return true;
}

// ------------------------------------------------------------------ chain kernel
// shared memory (1024-byte aligned offsets)
constexpr uint32_t kA_KQ = 0;         // [K;Q] rows (64 KB); reverse: scale gamma Q^T, then -gamma beta K^T (32 KB each)
constexpr uint32_t kA_AV = 65536;     // A tile [128 value rows][64]: B^T, U^T / dU^T, dB^T
constexpr uint32_t kA_TT = 98304;     // T [n][m] (forward), T^T [r][n] (reverse)
constexpr uint32_t kA_MT = 114688;    // M^T [n][r] (reverse)
constexpr uint32_t kA_X = 131072;     // decay-scaled K^T [j][r] (forward), dO^T [i][r] (reverse)
constexpr uint32_t kA_Small = 163840;

struct ChainSmall {
    BtCoef cf[2];   // chunk c's coefficients in cf[c & 1]; warp 15 forms the next chunk's during this one
    uint64_t bar[4];
    uint32_t tmem_base;
    int abort;
};
constexpr uint32_t kChainSmem = kA_Small + sizeof(ChainSmall) + 1024;

// TMEM columns
constexpr uint32_t tS = 0;     // state (forward), state gradient (reverse): [value row][key column]
constexpr uint32_t tP = 128;   // [S K^T | S Q^T]
constexpr uint32_t tU = 256;   // U^T (forward), dS K^T (reverse)
constexpr uint32_t tQK = 320;  // [K K^T; Q K^T]
constexpr uint32_t tDU = 384;  // dO^T M
constexpr uint32_t tDB = 448;  // dB^T

template <typename TI>
__global__ void __launch_bounds__(kBT, 1) bwd_tc_chain_kernel(const __grid_constant__ BwdTcArgs a) {
    const int h = blockIdx.x, n = blockIdx.y;
    int t_begin, len_seq;
    if (!seq_bounds(a, n, t_begin, len_seq)) return;   // uniform over the CTA
    extern __shared__ uint8_t bt_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(bt_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    ChainSmall *sm = reinterpret_cast<ChainSmall *>(smem + kA_Small);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int li = quad * 32 + lane;
    if (warp == 0) {
        tmem_alloc(&sm->tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int b = 0; b < 4; ++b) mbar_init(&sm->bar[b], 1);
        sm->abort = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = sm->tmem_base;
    const uint32_t tl = tb + ((uint32_t)(quad * 32) << 16);
    const int H = a.H, dk = a.dk, dv = a.dv;
    const TI *qg = static_cast<const TI *>(a.q);
    const TI *kg = static_cast<const TI *>(a.k);
    const TI *vg = static_cast<const TI *>(a.v);
    const TI *og = static_cast<const TI *>(a.dout);
    const uint64_t dKQ = smem_desc_sw128(sb + kA_KQ, 16, 1024);
    const uint64_t dKT2 = smem_desc_sw128(sb + kA_KQ + 32768, 16, 1024);
    const uint64_t dAV = smem_desc_sw128(sb + kA_AV, 16, 1024);
    const uint64_t dTT = smem_desc_sw128(sb + kA_TT, 16, 1024);
    const uint64_t dMT = smem_desc_sw128(sb + kA_MT, 16, 1024);
    const uint64_t dX = smem_desc_sw128(sb + kA_X, 16, 1024);
    const uint32_t I64 = idesc_tf32_f32(128, 64), I128 = idesc_tf32_f32(128, 128), IDK = idesc_tf32_f32(128, dk);
    uint32_t ph[4] = {0u, 0u, 0u, 0u};
    bool failed = false;
    const int nc = (len_seq + kChunk - 1) / kChunk;
    const float scale = a.scale;

    // ---------------- forward sweep: the start state of every chunk ----------------
    // (not run for the state gradient alone: the reverse recurrence needs no state)
    const int nc_fwd = a.state_grad_only ? 0 : nc;
    const bool full = !a.state_grad_only;
    for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
        uint32_t r[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int j = c0 + u;
            const float x = (a.s0 && li < dv && j < dk) ? a.s0[(((size_t)n * H + h) * dk + j) * dv + li] : 0.f;
            r[u] = __float_as_uint(x);
        }
        tmem_st32(tl + tS + c0, r);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (nc_fwd > 0) prefetch_chain_chunk<TI>(a, t_begin, min(kChunk, len_seq), h, false);
    if (nc_fwd > 0 && warp == 15) chunk_coef(&sm->cf[0], a.g, a.beta, t_begin, min(kChunk, len_seq), H, h);
    for (int c = 0; c < nc_fwd; ++c) {
        const int t0 = t_begin + c * kChunk, len = min(kChunk, t_begin + len_seq - t0);
        const size_t slot = (size_t)(t0 / kChunk + n);
        BtCoef *cf = &sm->cf[c & 1];
        if (c + 1 < nc_fwd)
            prefetch_chain_chunk<TI>(a, t0 + kChunk, min(kChunk, t_begin + len_seq - t0 - kChunk), h, false);
        tile_rows<TI>(sb + kA_KQ, kBlk128, 0, kg, t0, len, H, h, dk, One());
        tile_rows<TI>(sb + kA_KQ, kBlk128, 64, qg, t0, len, H, h, dk, One());
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();  // the [K;Q] tile and the coefficients
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < dk / 8; ++kk)
                    mma_ts_tf32(tb + tP, tb + tS + 8 * kk, f32_desc_kstep(dKQ, kk, kBlk128), I128, kk > 0);
                tc_commit(&sm->bar[0]);
            }
            __syncwarp();
        }
        // while the MMA runs (it only reads S and the [K;Q] tile): the next
        // chunk's coefficients; this chunk's start state, transposed
        // ([key][value]), to the workspace; the T and decay-scaled K^T tiles;
        // the values
        tc_fence_after();
        if (warp == 15 && c + 1 < nc_fwd)
            chunk_coef(&sm->cf[(c + 1) & 1], a.g, a.beta, t0 + kChunk, min(kChunk, t_begin + len_seq - t0 - kChunk),
                       H, h);
        {
            float *dst = a.s0t + (slot * H + h) * (size_t)dk * dv;
            for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tl + tS + c0, r);
                tmem_wait_ld();
                if (li < dv) {
#pragma unroll
                    for (int u = 0; u < 32; ++u)
                        if (c0 + u < dk) dst[(size_t)(c0 + u) * dv + li] = __uint_as_float(r[u]);
                }
            }
        }
        tile_t(sb + kA_TT, a.tp + ((size_t)h * a.total_T + t0) * kChunk, len, cf->G);
        tile_transpose_kq(sb + kA_KQ, sb + kA_X, 0, [cf](int r) { return cf->e[r]; }, sb + kA_X, 0,
                          [cf](int r) { return cf->e[r]; }, dk, dk, false, 1);   // decay-scaled K^T
        float vv[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int r = 16 * part + u;
            vv[u] = (li < dv && r < len) ? ld1<TI>(vg + ((size_t)(t0 + r) * H + h) * dv + li) : 0.f;
        }
        if (!bt_wait(&sm->bar[0], ph[0] & 1u, &sm->abort)) { failed = true; break; }
        ++ph[0];
        tc_fence_after();
        {
            uint32_t pk[16], pq[16];
            tmem_ld16(tl + tP + 16 * part, pk);
            tmem_ld16(tl + tP + 64 + 16 * part, pq);
            tmem_wait_ld();
            if (li < dv) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = 16 * part + u;
                    if (r < len) {
                        const size_t o = ((size_t)(t0 + r) * H + h) * dv + li;
                        a.ry[o] = __uint_as_float(pk[u]);
                        a.rqs[o] = __uint_as_float(pq[u]);
                    }
                }
            }
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                float x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int r = 16 * part + 4 * c4 + u;
                    x[u] = cf->beta[r] * (vv[4 * c4 + u] - cf->gam[r] * __uint_as_float(pk[4 * c4 + u]));
                }
                sts_f4(sb + kA_AV + f32_tile_off(li, 16 * part + 4 * c4, kBlk128), x[0], x[1], x[2], x[3]);
            }
        }
        {   // S <- gamma_C S (the MMA that read S is complete)
            const float gC = cf->gam[len - 1];
            for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tl + tS + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(gC * __uint_as_float(r[u]));
                tmem_st32(tl + tS + c0, r);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss_tf32(tb + tU, f32_desc_kstep(dAV, kk, kBlk128), f32_desc_kstep(dTT, kk, kBlk64), I64,
                                kk > 0);
                tc_commit(&sm->bar[1]);
            }
            __syncwarp();
        }
        if (!bt_wait(&sm->bar[1], ph[1] & 1u, &sm->abort)) { failed = true; break; }
        ++ph[1];
        tc_fence_after();
        {
            uint32_t u32[16];
            tmem_ld16(tl + tU + 16 * part, u32);
            tmem_wait_ld();
            if (li < dv) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = 16 * part + u;
                    if (r < len) a.ru[((size_t)(t0 + r) * H + h) * dv + li] = __uint_as_float(u32[u]);
                }
            }
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
                sts_u4_stage(sb + kA_AV + f32_tile_off(li, 16 * part + 4 * c4, kBlk128),
                       make_uint4(u32[4 * c4], u32[4 * c4 + 1], u32[4 * c4 + 2], u32[4 * c4 + 3]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss_tf32(tb + tS, f32_desc_kstep(dAV, kk, kBlk128), f32_desc_kstep(dX, kk, kBlk128), IDK, 1);
                tc_commit(&sm->bar[2]);
            }
            __syncwarp();
        }
        if (!bt_wait(&sm->bar[2], ph[2] & 1u, &sm->abort)) { failed = true; break; }
        ++ph[2];
        tc_fence_after();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    // ---------------- reverse sweep: the state gradient back to the start ----------------
    if (!failed) {
        for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int j = c0 + u;
                const float x = (a.dsf && li < dv && j < dk) ? a.dsf[(((size_t)n * H + h) * dk + j) * dv + li] : 0.f;
                r[u] = __float_as_uint(x);
            }
            tmem_st32(tl + tS + c0, r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (nc > 0 && !failed) {
        prefetch_chain_chunk<TI>(a, t_begin + (nc - 1) * kChunk, len_seq - (nc - 1) * kChunk, h, true);
        if (warp == 15)
            chunk_coef(&sm->cf[(nc - 1) & 1], a.g, a.beta, t_begin + (nc - 1) * kChunk, len_seq - (nc - 1) * kChunk,
                       H, h);
    }
    for (int c = nc - 1; c >= 0 && !failed; --c) {
        const int t0 = t_begin + c * kChunk, len = min(kChunk, t_begin + len_seq - t0);
        const size_t slot = (size_t)(t0 / kChunk + n);
        BtCoef *cf = &sm->cf[c & 1];
        if (c > 0) prefetch_chain_chunk<TI>(a, t0 - kChunk, kChunk, h, true);
        tile_rows<TI>(sb + kA_KQ, kBlk128, 0, kg, t0, len, H, h, dk, One());
        tile_rows<TI>(sb + kA_KQ, kBlk128, 64, qg, t0, len, H, h, dk, One());
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();  // the [K;Q] tile and the coefficients
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < dk / 8; ++kk)      // dS K^T
                    mma_ts_tf32(tb + tU, tb + tS + 8 * kk, f32_desc_kstep(dKQ, kk, kBlk128), I64, kk > 0);
                for (int kk = 0; kk < dk / 8; ++kk)      // [K;Q] K^T
                    mma_ss_tf32(tb + tQK, f32_desc_kstep(dKQ, kk, kBlk128), f32_desc_kstep(dKQ, kk, kBlk128), I64,
                                kk > 0);
                tc_commit(&sm->bar[0]);
            }
            __syncwarp();
        }
        // while the MMAs run (they read dS and the [K;Q] tile): the previous
        // chunk's coefficients; this chunk's end-state gradient, transposed, to
        // the workspace; the dO^T and T^T tiles
        tc_fence_after();
        if (warp == 15 && c > 0) chunk_coef(&sm->cf[(c - 1) & 1], a.g, a.beta, t0 - kChunk, kChunk, H, h);
        if (full) {
            float *dst = a.dst + (slot * H + h) * (size_t)dk * dv;
            for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tl + tS + c0, r);
                tmem_wait_ld();
                if (li < dv) {
#pragma unroll
                    for (int u = 0; u < 32; ++u)
                        if (c0 + u < dk) dst[(size_t)(c0 + u) * dv + li] = __uint_as_float(r[u]);
                }
            }
        }
        tile_cols<TI>(sb + kA_X, kBlk128, 128, og, t0, len, H, h, dv, One());   // dO^T, rows past dv zero
        tile_t_transposed(sb + kA_TT, a.tp + ((size_t)h * a.total_T + t0) * kChunk, len, cf->G);
        if (!bt_wait(&sm->bar[0], ph[0] & 1u, &sm->abort)) { failed = true; break; }
        ++ph[0];
        tc_fence_after();
        {
            uint32_t x[16];
            tmem_ld16(tl + tU + 16 * part, x);
            tmem_wait_ld();
            if (full && li < dv) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = 16 * part + u;
                    if (r < len) a.rkds[((size_t)(t0 + r) * H + h) * dv + li] = __uint_as_float(x[u]);
                }
            }
        }
        if (quad >= 2) {   // M^T [m][r] = Gamma ⊙ tril(Q K^T) [r][m], row r = lane - 64 of Q K^T
            uint32_t qk[16];
            tmem_ld16(tl + tQK + 16 * part, qk);
            tmem_wait_ld();
            const int r = li - 64;
            const float Gr = cf->G[r];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int m = 16 * part + u;
                const float x = (r < len && m <= r) ? __uint_as_float(qk[u]) * expf(Gr - cf->G[m]) : 0.f;
                sts_f32(sb + kA_MT + f32_tile_off(m, r, kBlk64), x);
            }
        }
        {   // dS <- gamma_C dS (the MMA that read it is complete)
            const float gC = cf->gam[len - 1];
            for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tl + tS + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(gC * __uint_as_float(r[u]));
                tmem_st32(tl + tS + c0, r);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < 8; ++kk)           // dO^T M = (M^T dO)^T
                    mma_ss_tf32(tb + tDU, f32_desc_kstep(dX, kk, kBlk128), f32_desc_kstep(dMT, kk, kBlk64), I64,
                                kk > 0);
                tc_commit(&sm->bar[1]);
            }
            __syncwarp();
        }
        if (!bt_wait(&sm->bar[1], ph[1] & 1u, &sm->abort)) { failed = true; break; }
        ++ph[1];
        tc_fence_after();
        {   // dU^T = scale dO^T M + (dS K^T) D_e into the A tile
            uint32_t du[16], x[16];
            tmem_ld16(tl + tDU + 16 * part, du);
            tmem_ld16(tl + tU + 16 * part, x);
            tmem_wait_ld();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                float y[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int m = 16 * part + 4 * c4 + u;
                    y[u] = scale * __uint_as_float(du[4 * c4 + u]) + cf->e[m] * __uint_as_float(x[4 * c4 + u]);
                }
                sts_f4(sb + kA_AV + f32_tile_off(li, 16 * part + 4 * c4, kBlk128), y[0], y[1], y[2], y[3]);
            }
        }
        // B operands of the state-gradient update, over the [K;Q] tile (its MMAs are done)
        tile_transpose_kq(sb + kA_KQ, sb + kA_KQ, 64, [cf, scale](int r) { return scale * cf->gam[r]; },
                          sb + kA_KQ + 32768, 0, [cf](int r) { return -cf->gam[r] * cf->beta[r]; }, dk, dk, true);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < 8; ++kk)           // dB^T = dU^T T
                    mma_ss_tf32(tb + tDB, f32_desc_kstep(dAV, kk, kBlk128), f32_desc_kstep(dTT, kk, kBlk64), I64,
                                kk > 0);
                tc_commit(&sm->bar[2]);
            }
            __syncwarp();
        }
        if (!bt_wait(&sm->bar[2], ph[2] & 1u, &sm->abort)) { failed = true; break; }
        ++ph[2];
        tc_fence_after();
        {
            uint32_t db[16];
            tmem_ld16(tl + tDB + 16 * part, db);
            tmem_wait_ld();
            if (full && li < dv) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = 16 * part + u;
                    if (r < len) {
                        const size_t o = ((size_t)(t0 + r) * H + h) * dv + li;
                        a.gv[o] = cf->beta[r] * __uint_as_float(db[u]);
                        a.rdb[o] = __uint_as_float(db[u]);
                    }
                }
            }
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
                sts_u4_stage(sb + kA_AV + f32_tile_off(li, 16 * part + 4 * c4, kBlk128),
                       make_uint4(db[4 * c4], db[4 * c4 + 1], db[4 * c4 + 2], db[4 * c4 + 3]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < 8; ++kk)           // dS += dO^T (scale D_gamma Q)
                    mma_ss_tf32(tb + tS, f32_desc_kstep(dX, kk, kBlk128), f32_desc_kstep(dKQ, kk, kBlk128), IDK, 1);
                for (int kk = 0; kk < 8; ++kk)           // dS += dB^T (-D_gamma diag(beta) K)
                    mma_ss_tf32(tb + tS, f32_desc_kstep(dAV, kk, kBlk128), f32_desc_kstep(dKT2, kk, kBlk128), IDK, 1);
                tc_commit(&sm->bar[3]);
            }
            __syncwarp();
        }
        if (!bt_wait(&sm->bar[3], ph[3] & 1u, &sm->abort)) { failed = true; break; }
        ++ph[3];
        tc_fence_after();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (!failed && a.gs0) {
        for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tl + tS + c0, r);
            tmem_wait_ld();
            if (li < dv) {
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    if (c0 + u < dk) a.gs0[(((size_t)n * H + h) * dk + c0 + u) * dv + li] = __uint_as_float(r[u]);
            }
        }
    }
    if (failed && tid == 0) {
        report_error(a.err, GDN_ERR_TIMEOUT);
        sm->abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// ------------------------------------------------------------------ chunk kernel
constexpr uint32_t kB_R0 = 0;          // [K;Q] rows; then K^T | Q^T; then dS^T
constexpr uint32_t kB_R1 = 65536;      // [dO;dB] rows; then the C x C work arrays (into R2); then S0^T
constexpr uint32_t kB_R2 = 131072;     // U rows; then -gamma beta dB rows; then e U rows
constexpr uint32_t kB_R3 = 163840;     // P + P^T | R | R^T (16 KB each); then scale gamma dO rows
constexpr uint32_t kB_Small = 212992;

struct ChunkSmall {
    BtCoef cf;
    float dG[64], db[64], de[64];
    float s_vdb[64], s_ydb[64], s_oqs[64];   // value-row dot products of each chunk row
    float red[kBT / 32];
    uint64_t bar;
    uint32_t tmem_base;
    int abort;
};
constexpr uint32_t kChunkSmem = kB_Small + sizeof(ChunkSmall) + 1024;
constexpr int kCP = 65;  // row stride of the C x C work arrays

// TMEM columns
constexpr uint32_t tG = 0;     // [K K^T; Q K^T]
constexpr uint32_t tH = 64;    // [dO U^T; dB U^T]
constexpr uint32_t tDK = 128;  // dK^T [key][row]
constexpr uint32_t tDQ = 192;  // dQ^T

template <typename TI>
__global__ void __launch_bounds__(kBT, 1) bwd_tc_chunk_kernel(const __grid_constant__ BwdTcArgs a) {
    const int ci = blockIdx.x, h = blockIdx.y;
    if (ci >= *a.num_chunks) return;
    extern __shared__ uint8_t bt_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(bt_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    ChunkSmall *sm = reinterpret_cast<ChunkSmall *>(smem + kB_Small);
    BtCoef *cf = &sm->cf;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int li = quad * 32 + lane;
    if (warp == 0) {
        tmem_alloc(&sm->tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(&sm->bar, 1);
        sm->abort = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = sm->tmem_base;
    const uint32_t tl = tb + ((uint32_t)(quad * 32) << 16);
    const int H = a.H, dk = a.dk, dv = a.dv;
    const TI *qg = static_cast<const TI *>(a.q);
    const TI *kg = static_cast<const TI *>(a.k);
    const TI *vg = static_cast<const TI *>(a.v);
    const TI *og = static_cast<const TI *>(a.dout);
    const int4 ch = a.chunks[ci];
    const int seq = ch.x, t0 = ch.y, len = ch.z;
    const size_t slot = (size_t)(t0 / kChunk + seq);
    const float scale = a.scale;
    const uint64_t dR0 = smem_desc_sw128(sb + kB_R0, 16, 1024);
    const uint64_t dR0q = smem_desc_sw128(sb + kB_R0 + 32768, 16, 1024);
    const uint64_t dR1 = smem_desc_sw128(sb + kB_R1, 16, 1024);
    const uint64_t dR2 = smem_desc_sw128(sb + kB_R2, 16, 1024);
    const uint64_t dR3 = smem_desc_sw128(sb + kB_R3, 16, 1024);
    const uint64_t dRR = smem_desc_sw128(sb + kB_R3 + 16384, 16, 1024);
    const uint64_t dRT = smem_desc_sw128(sb + kB_R3 + 32768, 16, 1024);
    const uint32_t I64 = idesc_tf32_f32(128, 64);
    uint32_t ph = 0;
    bool failed = false;

    if (warp == 0) chunk_coef(cf, a.g, a.beta, t0, len, H, h);
    // phase 1: the Gram [K;Q] K^T and [dO;dB] U^T
    tile_rows<TI>(sb + kB_R0, kBlk128, 0, kg, t0, len, H, h, dk, One());
    tile_rows<TI>(sb + kB_R0, kBlk128, 64, qg, t0, len, H, h, dk, One());
    tile_rows<TI>(sb + kB_R1, kBlk128, 0, og, t0, len, H, h, dv, One());
    tile_rows<float>(sb + kB_R1, kBlk128, 64, a.rdb, t0, len, H, h, dv, One());
    tile_rows<float>(sb + kB_R2, kBlk64, 0, a.ru, t0, len, H, h, dv, One());
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        if (elect_one()) {
            tc_fence_after();
            for (int kk = 0; kk < dk / 8; ++kk)
                mma_ss_tf32(tb + tG, f32_desc_kstep(dR0, kk, kBlk128), f32_desc_kstep(dR0, kk, kBlk128), I64, kk > 0);
            for (int kk = 0; kk < dv / 8; ++kk)
                mma_ss_tf32(tb + tH, f32_desc_kstep(dR1, kk, kBlk128), f32_desc_kstep(dR2, kk, kBlk64), I64, kk > 0);
            tc_commit(&sm->bar);
        }
        __syncwarp();
    }
    // while the MMAs run: the value-row dot products of each chunk row (dO and
    // dB from the [dO;dB] tile, U from its tile, the rest from memory)
    for (int r = warp; r < 64; r += kBT / 32) {
        float s_vdb = 0.f, s_ydb = 0.f, s_oqs = 0.f, s_ukds = 0.f;
        if (r < len && 4 * lane < dv) {   // four value columns per lane (dv <= 128)
            const size_t base = ((size_t)(t0 + r) * H + h) * dv + 4 * lane;
            const float4 y = __ldg(reinterpret_cast<const float4 *>(a.ry + base));
            const float4 qs = __ldg(reinterpret_cast<const float4 *>(a.rqs + base));
            const float4 kd = __ldg(reinterpret_cast<const float4 *>(a.rkds + base));
            const float4 vv = ld4<TI>(vg + base);
            const float4 oo = lds_f4(sb + kB_R1 + f32_tile_off(r, 4 * lane, kBlk128));
            const float4 db = lds_f4(sb + kB_R1 + f32_tile_off(64 + r, 4 * lane, kBlk128));
            const float4 uu = lds_f4(sb + kB_R2 + f32_tile_off(r, 4 * lane, kBlk64));
            s_vdb = vv.x * db.x + vv.y * db.y + vv.z * db.z + vv.w * db.w;
            s_ydb = y.x * db.x + y.y * db.y + y.z * db.z + y.w * db.w;
            s_oqs = oo.x * qs.x + oo.y * qs.y + oo.z * qs.z + oo.w * qs.w;
            s_ukds = uu.x * kd.x + uu.y * kd.y + uu.z * kd.z + uu.w * kd.w;
        }
        s_vdb = warp_sum(s_vdb);
        s_ydb = warp_sum(s_ydb);
        s_oqs = warp_sum(s_oqs);
        s_ukds = warp_sum(s_ukds);
        if (lane == 0) {
            sm->s_vdb[r] = s_vdb;
            sm->s_ydb[r] = s_ydb;
            sm->s_oqs[r] = s_oqs;
            sm->de[r] = s_ukds;
        }
    }
    do {
        if (!bt_wait(&sm->bar, ph & 1u, &sm->abort)) { failed = true; break; }
        ++ph;
        tc_fence_after();
        // phase 2: the C x C algebra on CUDA cores, in plain fp32 arrays over R1 / R2
        float *KK = reinterpret_cast<float *>(smem + kB_R1);
        float *QK = KK + 64 * kCP, *DM = QK + 64 * kCP, *DA = DM + 64 * kCP;
        {
            uint32_t x[16], y[16];
            tmem_ld16(tl + tG + 16 * part, x);
            tmem_ld16(tl + tH + 16 * part, y);
            tmem_wait_ld();
            const int r = li & 63;
            float *fa = li < 64 ? KK : QK;
            float *fb = li < 64 ? DM : DA;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                fa[r * kCP + 16 * part + u] = __uint_as_float(x[u]);
                fb[r * kCP + 16 * part + u] = __uint_as_float(y[u]);
            }
        }
        __syncthreads();
        for (int idx = tid; idx < 64 * 64; idx += kBT) {
            const int r = idx >> 6, m = idx & 63;
            float P = 0.f, R = 0.f, E = 0.f, dagk = 0.f;
            if (m <= r) {
                const float gm = expf(cf->G[r] - cf->G[m]);
                const float kk = KK[r * kCP + m], qk = QK[r * kCP + m];
                R = scale * DM[r * kCP + m] * gm;                   // dM ⊙ Gamma
                if (m < r) {
                    const float da = -DA[r * kCP + m];
                    dagk = da * gm * kk;
                    P = da * gm * cf->beta[r];
                }
                E = P * kk + R * qk;
            }
            DA[r * kCP + m] = P;
            DM[r * kCP + m] = R;
            KK[r * kCP + m] = E;
            QK[r * kCP + m] = dagk;
        }
        __syncthreads();
        // per-row sums: E by rows and columns, dA Gamma KK
        for (int r = warp; r < 64; r += kBT / 32) {
            const float rowE = warp_sum(KK[r * kCP + lane] + KK[r * kCP + 32 + lane]);
            const float colE = warp_sum(KK[lane * kCP + r] + KK[(32 + lane) * kCP + r]);
            const float dagk = warp_sum(QK[r * kCP + lane] + QK[r * kCP + 32 + lane]);
            if (lane == 0) {
                const float gam = cf->gam[r], beta = cf->beta[r];
                const float dgam = scale * sm->s_oqs[r] - beta * sm->s_ydb[r];   // D_gamma in O and X
                sm->db[r] = sm->s_vdb[r] - gam * sm->s_ydb[r] + dagk;
                sm->dG[r] = rowE - colE + dgam * gam - sm->de[r] * cf->e[r];
            }
        }
        // B operands of dK and dQ: P + P^T, R, R^T ([row][m], 64 x 64)
        for (int idx = tid; idx < 64 * 16; idx += kBT) {
            const int r = idx >> 4, m4 = (idx & 15) * 4;
            float pp[4], rr[4], rt[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int m = m4 + u;
                pp[u] = DA[r * kCP + m] + DA[m * kCP + r];
                rr[u] = DM[r * kCP + m];
                rt[u] = DM[m * kCP + r];
            }
            const uint32_t off = f32_tile_off(r, m4, kBlk64);
            sts_f4(sb + kB_R3 + off, pp[0], pp[1], pp[2], pp[3]);
            sts_f4(sb + kB_R3 + 16384 + off, rr[0], rr[1], rr[2], rr[3]);
            sts_f4(sb + kB_R3 + 32768 + off, rt[0], rt[1], rt[2], rt[3]);
        }
        // A operands K^T, Q^T ([key][m], rows past dk zero) over the [K;Q] tile
        tile_transpose_kq(sb + kB_R0, sb + kB_R0, 0, One(), sb + kB_R0 + 32768, 64, One(), 128, dk, true);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // phase 3a: dK^T = K^T (P + P^T)^T + Q^T R, dQ^T = K^T R^T
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss_tf32(tb + tDK, f32_desc_kstep(dR0, kk, kBlk128), f32_desc_kstep(dR3, kk, kBlk64), I64, kk > 0);
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss_tf32(tb + tDK, f32_desc_kstep(dR0q, kk, kBlk128), f32_desc_kstep(dRT, kk, kBlk64), I64, 1);
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss_tf32(tb + tDQ, f32_desc_kstep(dR0, kk, kBlk128), f32_desc_kstep(dRR, kk, kBlk64), I64, kk > 0);
                tc_commit(&sm->bar);
            }
            __syncwarp();
        }
        // meanwhile: S0^T ([key][value], rows past dk zero) over R1, -gamma beta dB rows over R2
        tile_state(sb + kB_R1, a.s0t + (slot * H + h) * (size_t)dk * dv, dk, dv, 0u);
        tile_rows<float>(sb + kB_R2, kBlk64, 0, a.rdb, t0, len, H, h, dv,
                         [cf](int r) { return -cf->gam[r] * cf->beta[r]; });
        if (!bt_wait(&sm->bar, ph & 1u, &sm->abort)) { failed = true; break; }
        ++ph;
        tc_fence_after();
        tile_rows<TI>(sb + kB_R3, kBlk64, 0, og, t0, len, H, h, dv, [cf, scale](int r) { return scale * cf->gam[r]; });
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // phase 3b: dK^T += S0^T (D_gamma dX)^T, dQ^T += S0^T (scale D_gamma dO)^T
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < dv / 8; ++kk)
                    mma_ss_tf32(tb + tDK, f32_desc_kstep(dR1, kk, kBlk128), f32_desc_kstep(dR2, kk, kBlk64), I64, 1);
                for (int kk = 0; kk < dv / 8; ++kk)
                    mma_ss_tf32(tb + tDQ, f32_desc_kstep(dR1, kk, kBlk128), f32_desc_kstep(dR3, kk, kBlk64), I64, 1);
                tc_commit(&sm->bar);
            }
            __syncwarp();
        }
        if (!bt_wait(&sm->bar, ph & 1u, &sm->abort)) { failed = true; break; }
        ++ph;
        tc_fence_after();
        // phase 3c: dS^T over R0 (with <dS, S0> on the way, S0^T still in R1), e U rows over R2
        {
            float part = tile_state(sb + kB_R0, a.dst + (slot * H + h) * (size_t)dk * dv, dk, dv, sb + kB_R1);
            part = warp_sum(part);
            if (lane == 0) sm->red[warp] = part;
        }
        tile_rows<float>(sb + kB_R2, kBlk64, 0, a.ru, t0, len, H, h, dv, [cf](int r) { return cf->e[r]; });
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                for (int kk = 0; kk < dv / 8; ++kk)   // dK^T += dS^T (D_e U)^T
                    mma_ss_tf32(tb + tDK, f32_desc_kstep(dR0, kk, kBlk128), f32_desc_kstep(dR2, kk, kBlk64), I64, 1);
                tc_commit(&sm->bar);
            }
            __syncwarp();
            // dg (reverse cumsum of dG, with the terms of gamma_C and of e's
            // numerator at row len - 1) and dbeta
            float t = sm->de[lane] * cf->e[lane] + sm->de[32 + lane] * cf->e[32 + lane];
            t = warp_sum(t);
            float ss = 0.f;
            for (int w = 0; w < kBT / 32; ++w) ss += sm->red[w];
            const float extra = t + cf->gam[len - 1] * ss;
            float x0 = sm->dG[lane], x1 = sm->dG[32 + lane];
            if (lane == len - 1) x0 += extra;
            if (32 + lane == len - 1) x1 += extra;
            for (int off = 1; off < 32; off <<= 1) {
                const float y0 = __shfl_down_sync(0xffffffffu, x0, off);
                const float y1 = __shfl_down_sync(0xffffffffu, x1, off);
                if (lane + off < 32) { x0 += y0; x1 += y1; }
            }
            x0 += __shfl_sync(0xffffffffu, x1, 0);
            if (lane < len) {
                a.gg[(size_t)(t0 + lane) * H + h] = x0;
                a.gbeta[(size_t)(t0 + lane) * H + h] = sm->db[lane];
            }
            if (32 + lane < len) {
                a.gg[(size_t)(t0 + 32 + lane) * H + h] = x1;
                a.gbeta[(size_t)(t0 + 32 + lane) * H + h] = sm->db[32 + lane];
            }
        }
        if (!bt_wait(&sm->bar, ph & 1u, &sm->abort)) { failed = true; break; }
        ++ph;
        tc_fence_after();
        {   // dK^T, dQ^T: lane = key index, columns = chunk rows
            uint32_t xk[16], xq[16];
            tmem_ld16(tl + tDK + 16 * part, xk);
            tmem_ld16(tl + tDQ + 16 * part, xq);
            tmem_wait_ld();
            if (li < dk) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = 16 * part + u;
                    if (r < len) {
                        const size_t o = ((size_t)(t0 + r) * H + h) * dk + li;
                        a.gk[o] = __uint_as_float(xk[u]);
                        a.gq[o] = __uint_as_float(xq[u]);
                    }
                }
            }
        }
    } while (false);
    if (failed && tid == 0) {
        report_error(a.err, GDN_ERR_TIMEOUT);
        sm->abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 256);
    }
}

template <typename TI>
cudaError_t launch_bwd_tc_t(const BwdTcArgs &a, int max_chunks, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(bwd_tc_chain_kernel<TI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kChainSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_tc_chunk_kernel<TI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kChunkSmem);
    if (e != cudaSuccess) return e;
    bwd_tc_chain_kernel<TI><<<dim3(a.H, a.N), kBT, kChainSmem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (max_chunks > 0 && !a.state_grad_only) {
        bwd_tc_chunk_kernel<TI><<<dim3(max_chunks, a.H), kBT, kChunkSmem, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdTcArgs &a, int max_chunks, cudaStream_t s) {
    if (a.dtype == GDN_BF16) return launch_bwd_tc_t<__nv_bfloat16>(a, max_chunks, s);
    return launch_bwd_tc_t<float>(a, max_chunks, s);
}

}  // namespace gdn
