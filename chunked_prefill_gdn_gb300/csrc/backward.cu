// Backward pass of the chunked GDN forward: gradients of q, k, v, g, beta and
// the initial state from the gradients of o and of the final state.
//
// The talk "Qwen系列模型线性注意力高性能优化实践" (backward paragraph) runs the
// backward chunk by chunk in the WY form with the dA and dA^T terms merged; it
// prints no formulas.  The algebra here is the chain rule through one chunk of
// the forward (math orientation, S dv x dk, C = 64 tokens, start state S0,
// chunk-local G = cumsum g, gamma = exp(G), Gamma_ri = exp(G_r - G_i),
// e_i = exp(G_C - G_i)):
//
//   forward   A = strictlower(diag(beta)(Gamma . K K^T)),  T = (I + A)^-1
//             X = D_gamma K S0^T,  B = diag(beta)(V - X),  U = T B
//             M = Gamma . tril(Q K^T),  O = scale (D_gamma Q S0^T + M U)
//             S_C = gamma_C S0 + U^T D_e K
//   backward  dU = scale M^T dO + D_e K dS_C^T,   dB = T^T dU
//             dM = scale dO U^T (lower),  dA = -dB U^T (strictly lower)
//             dV = diag(beta) dB,   dX = -diag(beta) dB
//             P = dA . Gamma . beta_r,  R = dM . Gamma
//             dK = (P + P^T) K + R^T Q + D_gamma dX S0 + D_e U dS_C
//             dQ = R K + scale D_gamma dO S0
//             dS0 = scale dO^T D_gamma Q + dX^T D_gamma K + gamma_C dS_C
//             dbeta, dg from every place beta, G enter (then dg is the reverse
//             cumsum of dG inside the chunk)
//
// This file holds the C entry points (gdn_chunk_bwd and its workspace) and
// the CUDA-core kernels, selected with gdn_set_backward_kernel; the default
// kernels, with every product on the tensor cores, are in backward_tc.cu.
//
// Design of the CUDA-core kernels: one CTA per (value-column slice of 32, head, sequence).  The state's
// rows along dv evolve independently, so a slice runs the whole recurrence on
// its own columns: a forward sweep stores every chunk's start state (slice)
// in the workspace, then a reverse sweep carries dS from the last chunk to the
// first.  dv, dS0 come out complete per slice; dq, dk, dg, dbeta are sums over
// the dv columns, so each slice writes its partial and a second kernel adds the
// slices in a fixed order (deterministic, no atomics).
//
// With bf16 inputs and dk = 128 the two Gram products K K^T and Q K^T (exact
// bf16 operands, fp32 accumulation) run on the tensor cores: one tcgen05 MMA
// chain per chunk, [K;Q] (128 x 128, bf16, 128-byte swizzle, written by the
// chunk loader into shared memory that is dead at that point) times K^T into 64
// tensor-memory columns, read back by the lane-quadrant warps.  All other
// products are fp32 on CUDA cores with operands in shared memory (padded
// strides, conflict-free), the work of each phase spread over the 16 warps.
// T is not solved here: before the kernel, the sequence-prep kernel builds the
// chunk table and the library's per-chunk inverse writes T' = (I + A')^-1
// (A' = diag(beta) strictlower(K K^T), fp32) for every chunk once, and the
// kernel takes T = Gamma ⊙ T' (the Gamma-extraction identity, exact) — the
// substitution on two warps, repeated per chunk, value slice and sweep, was
// ~45% of the kernel's time.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kBwdCols = 32;      // value columns per CTA
constexpr int kBwdThreads = 512;  // 16 warps
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int C = kChunk;
constexpr int CP = C + 1;         // padded row stride of C x C tiles
constexpr int WP = kBwdCols + 1;  // padded row stride of C x 32 and dk x 32 tiles

// Shared-memory layout (in floats) for head dimension DK.  K and Q rows are
// padded to an odd length (conflict-free column walks of the CUDA-core Gram),
// or with W (the tensor-core Gram, no column walks) to a multiple of four
// floats, so that a row's elements load four at a time.
template <int DK, bool W = false>
struct BwdSmem {
    static constexpr int KP = W ? DK + 4 : DK + 1;
    static constexpr int kK = 0;                 // K      [C][KP]
    static constexpr int kQ = kK + C * KP;       // Q      [C][KP]
    static constexpr int kS0 = kQ + C * KP;      // S0     [DK][WP]  chunk start state (slice)
    static constexpr int kdS = kS0 + DK * WP;    // dS     [DK][WP]  gradient of the chunk's end state
    static constexpr int kV = kdS + DK * WP;     // V      [C][WP]
    static constexpr int kdO = kV + C * WP;      // dO     [C][WP]
    static constexpr int kY = kdO + C * WP;      // K S0   [C][WP]
    static constexpr int kKdS = kY + C * WP;     // K dS   [C][WP]
    static constexpr int kU = kKdS + C * WP;     // U      [C][WP]
    static constexpr int kTmp = kU + C * WP;     // B, then dU
    static constexpr int kdB = kTmp + C * WP;    // dB     [C][WP]
    static constexpr int kKK = kdB + C * WP;     // K K^T (strictly lower), then E
    static constexpr int kGam = kKK + C * CP;    // Gamma (lower), then R
    static constexpr int kA = kGam + C * CP;     // A, then Q K^T (lower)
    static constexpr int kT = kA + C * CP;       // T, then P' = dA . Gamma
    static constexpr int kG = kT + C * CP;       // vectors of C
    static constexpr int kGamma = kG + C;
    static constexpr int kE = kGamma + C;
    static constexpr int kBeta = kE + C;
    static constexpr int kDgam = kBeta + C;      // scale dO . (Q S0) per row
    static constexpr int kDe = kDgam + C;
    static constexpr int kDb = kDe + C;
    static constexpr int kDG = kDb + C;
    static constexpr int kRed = kDG + C;         // [kBwdWarps]
    static constexpr int kBar = (kRed + kBwdWarps + 1) & ~1;   // mbarrier (8-byte aligned)
    static constexpr int kTslot = kBar + 2;      // tensor-memory base address, then a zero word
                                                 // (the bounded wait's abort flag: never set)
    static constexpr int kFloats = kTslot + 2;
    static constexpr size_t kBytes = (size_t)kFloats * sizeof(float);
};
static_assert(BwdSmem<128>::kBytes <= 232448 && BwdSmem<128, true>::kBytes <= 232448,
              "backward tile set exceeds the shared memory of a CTA");
// the [K;Q] operand tile of the tensor-core Gram (32 KB, 1024-byte aligned)
// lives in the Y .. dB tiles, dead while the Gram runs
static_assert((BwdSmem<128, true>::kdB + C * WP - BwdSmem<128, true>::kY) * 4 >= 32768 + 1008,
              "operand tile does not fit");
static_assert(kChunk % kBwdWarps == 0 && 32 % kBwdWarps == 0, "rows per warp must divide evenly");

struct BwdArgs {
    const void *q, *k, *v, *dout;
    const float *g, *beta, *s0, *dsf;
    const int32_t *cu;
    float *gq, *gk, *gv, *gg, *gbeta, *gs0;   // gradients; gq, gk, gg, gbeta: per-slice partials
                                              // when slices > 1
    float *states;                            // [slots][H][DK][dv] chunk start states
    const float *tp;                          // [H, total_T, C] T' (no gate factors), fp32
    int *err;
    long long part_stride_k;                  // total_T * H * DK: slice stride of the dq / dk partials
    long long part_stride_t;                  // total_T * H: slice stride of the dg / dbeta partials
    int T, H, dv, N, total_T, varlen;
    float scale;
};

template <typename TI>
__device__ __forceinline__ float ld_in(const void *base, size_t i) {
    return static_cast<float>(reinterpret_cast<const TI *>(base)[i]);
}
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const void *base, size_t i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[i]);
}

// Four consecutive floats: one 16-byte load when the row layout keeps them
// 16-byte aligned (V), else four loads.
template <bool V>
__device__ __forceinline__ float4 ld4f(const float *p) {
    if constexpr (V) return *reinterpret_cast<const float4 *>(p);
    else return make_float4(p[0], p[1], p[2], p[3]);
}

__device__ __forceinline__ float warp_sum(float x) {
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// The tensor-core Gram runs for bf16 inputs with dk = 128.
template <int DK, typename TI>
constexpr bool kTcGram = DK == 128 && std::is_same<TI, __nv_bfloat16>::value;

template <int DK, bool W>
__device__ __forceinline__ uint32_t operand_tile(float *sm) {
    return (smem_u32(sm + BwdSmem<DK, W>::kY) + 1023u) & ~1023u;
}

// Loads one chunk (rows >= len zero, g = 0 and beta = 0 there, which leaves the
// algebra of a short chunk unchanged) and forms G, gamma, e in warp 0.
template <int DK, typename TI>
__device__ void load_chunk(const BwdArgs &a, float *sm, int t0, int len, int h, int col0, bool with_q) {
    using L = BwdSmem<DK, kTcGram<DK, TI>>;
    constexpr int KP = L::KP;
    const int tid = threadIdx.x;
    const int H = a.H;
    if constexpr (kTcGram<DK, TI>) {
        // 16-byte loads; fp32 copies plus the bf16 [K;Q] operand tile (two
        // 16 KB halves of 64 features; row r at r * 128 B, 16-byte chunk c
        // at (c ^ (r & 7)) * 16), then the proxy fence for the MMA's reads
        const uint32_t opnd = operand_tile<DK, true>(sm);
        for (int idx = tid; idx < C * 16; idx += kBwdThreads) {
            const int r = idx >> 4, c16 = idx & 15;
            uint4 kv = make_uint4(0u, 0u, 0u, 0u), qv = kv;
            if (r < len) {
                const size_t off = ((size_t)(t0 + r) * H + h) * DK + c16 * 8;
                kv = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.k) + off);
                if (with_q) qv = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.q) + off);
            }
            const uint32_t hoff = (uint32_t)(c16 >> 3) * 16384u;
            sts_u4(opnd + hoff + sw128_offset((uint32_t)r, (uint32_t)(c16 & 7)), kv);
            if (with_q) sts_u4(opnd + hoff + sw128_offset((uint32_t)(64 + r), (uint32_t)(c16 & 7)), qv);
            float4 *dk4 = reinterpret_cast<float4 *>(sm + L::kK + r * KP + c16 * 8);   // KP % 4 == 0
            dk4[0] = make_float4(bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y));
            dk4[1] = make_float4(bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w));
            if (with_q) {
                float4 *dq4 = reinterpret_cast<float4 *>(sm + L::kQ + r * KP + c16 * 8);
                dq4[0] = make_float4(bf16_lo(qv.x), bf16_hi(qv.x), bf16_lo(qv.y), bf16_hi(qv.y));
                dq4[1] = make_float4(bf16_lo(qv.z), bf16_hi(qv.z), bf16_lo(qv.w), bf16_hi(qv.w));
            }
        }
        fence_proxy_async_smem();
    } else {
        for (int idx = tid; idx < C * DK; idx += kBwdThreads) {
            const int r = idx / DK, d = idx % DK;
            float kv = 0.f, qv = 0.f;
            if (r < len) {
                const size_t off = ((size_t)(t0 + r) * H + h) * DK + d;
                kv = ld_in<TI>(a.k, off);
                if (with_q) qv = ld_in<TI>(a.q, off);
            }
            sm[L::kK + r * KP + d] = kv;
            if (with_q) sm[L::kQ + r * KP + d] = qv;
        }
    }
    for (int idx = tid; idx < C * kBwdCols; idx += kBwdThreads) {
        const int r = idx / kBwdCols, w = idx % kBwdCols;
        float vv = 0.f, ov = 0.f;
        if (r < len) {
            const size_t off = ((size_t)(t0 + r) * H + h) * a.dv + col0 + w;
            vv = ld_in<TI>(a.v, off);
            if (with_q) ov = ld_in<TI>(a.dout, off);
        }
        sm[L::kV + r * WP + w] = vv;
        if (with_q) sm[L::kdO + r * WP + w] = ov;
    }
    if (tid < 32) {
        const int lane = tid;
        float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
        if (lane < len) {
            g0 = a.g[(size_t)(t0 + lane) * H + h];
            b0 = a.beta[(size_t)(t0 + lane) * H + h];
        }
        if (32 + lane < len) {
            g1 = a.g[(size_t)(t0 + 32 + lane) * H + h];
            b1 = a.beta[(size_t)(t0 + 32 + lane) * H + h];
        }
        for (int off = 1; off < 32; off <<= 1) {      // inclusive scans of both halves
            const float y0 = __shfl_up_sync(0xffffffffu, g0, off);
            const float y1 = __shfl_up_sync(0xffffffffu, g1, off);
            if (lane >= off) { g0 += y0; g1 += y1; }
        }
        g1 += __shfl_sync(0xffffffffu, g0, 31);
        const float glast = __shfl_sync(0xffffffffu, g1, 31);   // = G at row len-1 (zero-padded g)
        sm[L::kG + lane] = g0;
        sm[L::kG + 32 + lane] = g1;
        sm[L::kGamma + lane] = expf(g0);
        sm[L::kGamma + 32 + lane] = expf(g1);
        sm[L::kE + lane] = expf(glast - g0);
        sm[L::kE + 32 + lane] = expf(glast - g1);
        sm[L::kBeta + lane] = b0;
        sm[L::kBeta + 32 + lane] = b1;
    }
}

// K K^T (strictly lower), Gamma (lower) and A.  Ends synchronised.
template <int DK, bool W>
__device__ void chunk_gram(float *sm) {
    using L = BwdSmem<DK, W>;
    constexpr int KP = L::KP;
    const int tid = threadIdx.x;
    const float *sK = sm + L::kK;
    for (int idx = tid; idx < C * C; idx += kBwdThreads) {
        const int r = idx / C, i = idx % C;            // a warp holds one r and 32 consecutive i
        float kk = 0.f, gm = 0.f;
        if (i <= r) {
            gm = expf(sm[L::kG + r] - sm[L::kG + i]);
            if (i < r) {
#pragma unroll 8
                for (int d = 0; d < DK; ++d) kk += sK[r * KP + d] * sK[i * KP + d];
            }
        }
        sm[L::kKK + r * CP + i] = kk;
        sm[L::kGam + r * CP + i] = gm;
        sm[L::kA + r * CP + i] = (i < r) ? sm[L::kBeta + r] * gm * kk : 0.f;
    }
    __syncthreads();
}

// The Gram on the tensor cores: [K;Q] K^T into tensor memory (lanes 0-63
// K K^T, lanes 64-127 Q K^T; column i), then K K^T, Gamma and A as
// chunk_gram writes them, from the quadrant-0/1 warps.  Q K^T stays in tensor
// memory until tc_read_qk.  Ends synchronised.
template <int DK, bool W>
__device__ void tc_gram(float *sm, uint32_t tbase, uint32_t &phase, int *err) {
    using L = BwdSmem<DK, W>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kBar);
    if (warp == 0) {
        tc_fence_after();
        if (elect_one()) {
            constexpr uint32_t I0 = idesc_bf16_f32(128, 64, 0, 0);
            const uint64_t d = smem_desc_sw128(operand_tile<DK, W>(sm), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t o = d + ((uint64_t)((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                mma_ss(tbase, o, o, I0, kk > 0);
            }
            tc_commit(bar);
        }
        __syncwarp();
    }
    // bounded (2 s): a wait that runs out records GDN_ERR_TIMEOUT
    if (!mbar_wait(bar, phase & 1u, reinterpret_cast<volatile int *>(sm + L::kTslot + 1), 2000000000ull) &&
        threadIdx.x == 0)
        report_error(err, GDN_ERR_TIMEOUT);
    ++phase;
    tc_fence_after();
    const int q = warp & 3, cb = warp >> 2;
    if (q < 2) {
        uint32_t v[16];
        tmem_ld16(tbase + ((uint32_t)(32 * q) << 16) + 16 * cb, v);
        tmem_wait_ld();
        const int r = 32 * q + lane;
        const float gr = sm[L::kG + r], br = sm[L::kBeta + r];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = 16 * cb + u;
            float kk = 0.f, gm = 0.f;
            if (i <= r) {
                gm = expf(gr - sm[L::kG + i]);
                if (i < r) kk = __uint_as_float(v[u]);
            }
            sm[L::kKK + r * CP + i] = kk;
            sm[L::kGam + r * CP + i] = gm;
            sm[L::kA + r * CP + i] = (i < r) ? br * gm * kk : 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
}

// Q K^T (lower) from tensor memory into the A tile (quadrant-2/3 warps).
template <int DK, bool W>
__device__ void tc_read_qk(float *sm, uint32_t tbase) {
    using L = BwdSmem<DK, W>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, cb = warp >> 2;
    if (q >= 2) {
        tc_fence_after();
        uint32_t v[16];
        tmem_ld16(tbase + ((uint32_t)(32 * q) << 16) + 16 * cb, v);
        tmem_wait_ld();
        const int r = 32 * (q - 2) + lane;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = 16 * cb + u;
            sm[L::kA + r * CP + i] = (i <= r) ? __uint_as_float(v[u]) : 0.f;
        }
        tc_fence_before();
    }
}

// T = Gamma ⊙ T' (the Gamma-extraction identity: T_rm = exp(G_r - G_m) T'_rm,
// exact) from the T' rows formed before the kernel; rows past the chunk's
// length are identity rows (their A rows are zero).  Called by warps 0-1 only,
// after the Gamma tile is formed; one column per thread, each load of a warp
// 128 contiguous bytes.
template <int DK, bool W>
__device__ void chunk_load_t(float *sm, const float *tp_rows, int len) {
    using L = BwdSmem<DK, W>;
    const int j = threadIdx.x;
    float *sT = sm + L::kT;
    const float *sGam = sm + L::kGam;
#pragma unroll 4
    for (int r = 0; r < C; ++r) {
        float t = (r == j) ? 1.f : 0.f;
        if (r < len && j <= r) t = sGam[r * CP + j] * __ldg(tp_rows + (size_t)r * C + j);
        sT[r * CP + j] = t;
    }
}

// B = diag(beta)(V - gamma Y) into the scratch tile, then U = T B.  Expects Y
// in place and ends synchronised.
template <int DK, bool W>
__device__ void chunk_u(float *sm) {
    using L = BwdSmem<DK, W>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int idx = tid; idx < C * kBwdCols; idx += kBwdThreads) {
        const int r = idx / kBwdCols, w = idx % kBwdCols;
        sm[L::kTmp + r * WP + w] =
            sm[L::kBeta + r] * (sm[L::kV + r * WP + w] - sm[L::kGamma + r] * sm[L::kY + r * WP + w]);
    }
    __syncthreads();
    for (int r = warp; r < C; r += kBwdWarps) {
        float u = 0.f;
        for (int i = 0; i <= r; ++i) u += sm[L::kT + r * CP + i] * sm[L::kTmp + i * WP + lane];
        sm[L::kU + r * WP + lane] = u;
    }
    __syncthreads();
}

template <int DK, typename TI>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(const __grid_constant__ BwdArgs a) {
    constexpr bool TC = kTcGram<DK, TI>;
    using L = BwdSmem<DK, TC>;
    constexpr int KP = L::KP;
    constexpr int DPL = DK / 32;          // head-dimension elements per lane
    constexpr int DPW = DK / kBwdWarps;   // state rows per warp (a contiguous block)
    constexpr int RPW = C / kBwdWarps;    // chunk rows per warp
    extern __shared__ __align__(16) float sm[];
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, dv = a.dv, col0 = slice * kBwdCols;
    const float scale = a.scale;

    int t_begin, len_seq;
    if (a.varlen) {
        const int c0 = a.cu[n], c1 = a.cu[n + 1];
        const bool bad = c0 < 0 || c1 < c0 || c1 > a.total_T || (n == 0 && c0 != 0) ||
                         (n == a.N - 1 && c1 != a.total_T);
        if (bad) {                                   // uniform over the CTA
            if (tid == 0) report_error(a.err, GDN_ERR_DEVICE_CHECK);
            return;
        }
        t_begin = c0;
        len_seq = c1 - c0;
    } else {
        t_begin = n * a.T;
        len_seq = a.T;
    }
    const int nc = (len_seq + C - 1) / C;
    uint32_t tbase = 0, phase = 0;
    if constexpr (TC) {
        if (tid == 0) {
            mbar_init(reinterpret_cast<uint64_t *>(sm + L::kBar), 1);
            reinterpret_cast<int *>(sm + L::kTslot)[1] = 0;
            fence_barrier_init();
        }
        if (warp == 0) {
            tmem_alloc(reinterpret_cast<uint32_t *>(sm + L::kTslot), 64);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tbase = *reinterpret_cast<volatile uint32_t *>(sm + L::kTslot);
    }
    // chunk c of this sequence stores its start state in slot (first token)/C + n:
    // distinct for distinct chunks and below total_T/C + N
    auto state_ptr = [&](int t0) {
        return a.states + ((size_t)(t0 / C + n) * H + h) * DK * dv + col0;
    };

    float *sS0 = sm + L::kS0;
    float *sdS = sm + L::kdS;
    const float *sK = sm + L::kK;
    const float *sQ = sm + L::kQ;

    // ---------------- forward sweep: the start state of every chunk ----------------
    for (int idx = tid; idx < DK * kBwdCols; idx += kBwdThreads) {
        const int d = idx / kBwdCols, w = idx % kBwdCols;
        sS0[d * WP + w] = a.s0 ? a.s0[(((size_t)n * H + h) * DK + d) * dv + col0 + w] : 0.f;
    }
    for (int c = 0; c < nc; ++c) {
        const int t0 = t_begin + c * C;
        const int len = min(C, t_begin + len_seq - t0);
        __syncthreads();
        load_chunk<DK, TI>(a, sm, t0, len, h, col0, false);
        float *st = state_ptr(t0);
        for (int idx = tid; idx < DK * kBwdCols; idx += kBwdThreads) {
            const int d = idx / kBwdCols, w = idx % kBwdCols;
            st[(size_t)d * dv + w] = sS0[d * WP + w];
        }
        __syncthreads();
        if constexpr (TC) tc_gram<DK, TC>(sm, tbase, phase, a.err); else chunk_gram<DK, TC>(sm);
        if (warp < 2) {
            chunk_load_t<DK, TC>(sm, a.tp + ((size_t)h * a.total_T + t0) * C, len);
        } else {
            for (int r = warp - 2; r < C; r += kBwdWarps - 2) {     // Y = K S0
                float y = 0.f;
#pragma unroll 2
                for (int d = 0; d < DK; d += 4) {
                    const float4 k4 = ld4f<TC>(sK + r * KP + d);
                    y += k4.x * sS0[d * WP + lane] + k4.y * sS0[(d + 1) * WP + lane] +
                         k4.z * sS0[(d + 2) * WP + lane] + k4.w * sS0[(d + 3) * WP + lane];
                }
                sm[L::kY + r * WP + lane] = y;
            }
        }
        __syncthreads();
        chunk_u<DK, TC>(sm);
        {                                               // S_C = gamma_C S0 + K^T D_e U
            const float gC = sm[L::kGamma + C - 1];
            float acc[DPW];
#pragma unroll
            for (int m = 0; m < DPW; ++m) acc[m] = 0.f;
            const int d0 = warp * DPW;                  // this warp's state rows d0 .. d0 + DPW - 1
            for (int r = 0; r < C; ++r) {
                const float eu = sm[L::kE + r] * sm[L::kU + r * WP + lane];
                if constexpr (DPW % 4 == 0) {
#pragma unroll
                    for (int m = 0; m < DPW; m += 4) {
                        const float4 k4 = ld4f<TC>(sK + r * KP + d0 + m);
                        acc[m] += k4.x * eu; acc[m + 1] += k4.y * eu; acc[m + 2] += k4.z * eu; acc[m + 3] += k4.w * eu;
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < DPW; ++m) acc[m] += sK[r * KP + d0 + m] * eu;
                }
            }
#pragma unroll
            for (int m = 0; m < DPW; ++m) {
                const int d = d0 + m;
                sS0[d * WP + lane] = gC * sS0[d * WP + lane] + acc[m];
            }
        }
    }

    // ---------------- reverse sweep ----------------
    __syncthreads();
    for (int idx = tid; idx < DK * kBwdCols; idx += kBwdThreads) {
        const int d = idx / kBwdCols, w = idx % kBwdCols;
        sdS[d * WP + w] = a.dsf ? a.dsf[(((size_t)n * H + h) * DK + d) * dv + col0 + w] : 0.f;
    }
    float *pdq = a.gq + (size_t)slice * a.part_stride_k;
    float *pdk = a.gk + (size_t)slice * a.part_stride_k;
    float *pdg = a.gg + (size_t)slice * a.part_stride_t;
    float *pdb = a.gbeta + (size_t)slice * a.part_stride_t;
    for (int c = nc - 1; c >= 0; --c) {
        const int t0 = t_begin + c * C;
        const int len = min(C, t_begin + len_seq - t0);
        __syncthreads();
        load_chunk<DK, TI>(a, sm, t0, len, h, col0, true);
        const float *st = state_ptr(t0);
        for (int idx = tid; idx < DK * kBwdCols; idx += kBwdThreads) {
            const int d = idx / kBwdCols, w = idx % kBwdCols;
            sS0[d * WP + w] = st[(size_t)d * dv + w];
        }
        __syncthreads();
        if constexpr (TC) tc_gram<DK, TC>(sm, tbase, phase, a.err); else chunk_gram<DK, TC>(sm);
        if (warp < 2) {
            chunk_load_t<DK, TC>(sm, a.tp + ((size_t)h * a.total_T + t0) * C, len);
        } else {
            // while T is solved: Y = K S0; K dS; scale dO . (Q S0) per row
            for (int r = warp - 2; r < C; r += kBwdWarps - 2) {
                float y = 0.f, qs = 0.f, kd = 0.f;
#pragma unroll 2
                for (int d = 0; d < DK; d += 4) {
                    const float4 k4 = ld4f<TC>(sK + r * KP + d);
                    const float4 q4 = ld4f<TC>(sQ + r * KP + d);
                    const float s0a = sS0[d * WP + lane], s0b = sS0[(d + 1) * WP + lane];
                    const float s0c = sS0[(d + 2) * WP + lane], s0d = sS0[(d + 3) * WP + lane];
                    y += k4.x * s0a + k4.y * s0b + k4.z * s0c + k4.w * s0d;
                    qs += q4.x * s0a + q4.y * s0b + q4.z * s0c + q4.w * s0d;
                    kd += k4.x * sdS[d * WP + lane] + k4.y * sdS[(d + 1) * WP + lane] +
                          k4.z * sdS[(d + 2) * WP + lane] + k4.w * sdS[(d + 3) * WP + lane];
                }
                sm[L::kY + r * WP + lane] = y;
                sm[L::kKdS + r * WP + lane] = kd;
                const float t = warp_sum(sm[L::kdO + r * WP + lane] * qs);
                if (lane == 0) sm[L::kDgam + r] = scale * t;
            }
        }
        __syncthreads();
        // Q K^T (lower) over A (the solve is done with it)
        if constexpr (TC) {
            tc_read_qk<DK, TC>(sm, tbase);
        } else {
            for (int idx = tid; idx < C * C; idx += kBwdThreads) {
                const int r = idx / C, i = idx % C;
                float qk = 0.f;
                if (i <= r) {
#pragma unroll 8
                    for (int d = 0; d < DK; ++d) qk += sQ[r * KP + d] * sK[i * KP + d];
                }
                sm[L::kA + r * CP + i] = qk;
            }
        }
        chunk_u<DK, TC>(sm);

        // dU = scale M^T dO + D_e K dS  (into the scratch tile; B is dead)
        for (int i = warp; i < C; i += kBwdWarps) {
            float acc = 0.f;
            for (int r = i; r < C; ++r)
                acc += sm[L::kGam + r * CP + i] * sm[L::kA + r * CP + i] * sm[L::kdO + r * WP + lane];
            sm[L::kTmp + i * WP + lane] = scale * acc + sm[L::kE + i] * sm[L::kKdS + i * WP + lane];
        }
        __syncthreads();
        // dB = T^T dU; dv = beta dB (complete for this slice's columns)
        for (int r = warp; r < C; r += kBwdWarps) {
            float acc = 0.f;
            for (int i = r; i < C; ++i) acc += sm[L::kT + i * CP + r] * sm[L::kTmp + i * WP + lane];
            sm[L::kdB + r * WP + lane] = acc;
            if (r < len) a.gv[((size_t)(t0 + r) * H + h) * dv + col0 + lane] = sm[L::kBeta + r] * acc;
        }
        __syncthreads();
        // P' = dA . Gamma over T (dead), R = dM . Gamma over Gamma (same element, same thread)
        for (int idx = tid; idx < C * C; idx += kBwdThreads) {
            const int r = idx / C, i = idx % C;
            float pa = 0.f, rm = 0.f;
            if (i <= r) {
                float dbu = 0.f, dou = 0.f;
#pragma unroll 8
                for (int w = 0; w < kBwdCols; ++w) {
                    const float u = sm[L::kU + i * WP + w];
                    dbu += sm[L::kdB + r * WP + w] * u;
                    dou += sm[L::kdO + r * WP + w] * u;
                }
                const float gm = sm[L::kGam + r * CP + i];
                if (i < r) pa = -gm * dbu;
                rm = gm * scale * dou;
            }
            sm[L::kT + r * CP + i] = pa;
            sm[L::kGam + r * CP + i] = rm;
        }
        __syncthreads();
        // per-row sums: dbeta, dG's gamma and e terms; and <dS, S0> for gamma_C
        for (int r = warp; r < C; r += kBwdWarps) {
            const float db = sm[L::kdB + r * WP + lane], y = sm[L::kY + r * WP + lane];
            const float a1 = warp_sum((sm[L::kV + r * WP + lane] - sm[L::kGamma + r] * y) * db);
            const float a2 = warp_sum(db * y);
            const float a3 = warp_sum(sm[L::kU + r * WP + lane] * sm[L::kKdS + r * WP + lane]);
            const float a4 = warp_sum(sm[L::kT + r * CP + lane] * sm[L::kKK + r * CP + lane] +
                                      sm[L::kT + r * CP + 32 + lane] * sm[L::kKK + r * CP + 32 + lane]);
            if (lane == 0) {
                sm[L::kDb + r] = a1 + a4;
                const float dgam = sm[L::kDgam + r] - sm[L::kBeta + r] * a2;
                sm[L::kDG + r] = dgam * sm[L::kGamma + r] - a3 * sm[L::kE + r];
                sm[L::kDe + r] = a3;
            }
        }
        {
            float part = 0.f;
            for (int idx = tid; idx < DK * kBwdCols; idx += kBwdThreads) {
                const int d = idx / kBwdCols, w = idx % kBwdCols;
                part += sdS[d * WP + w] * sS0[d * WP + w];
            }
            part = warp_sum(part);
            if (lane == 0) sm[L::kRed + warp] = part;
        }
        __syncthreads();
        // E = beta_r P' . KK + R . QK (where Gamma enters A and M), over K K^T;
        // the scaled tiles of the products below over tiles that are dead now:
        // GX = gamma dX = -gamma beta dB (over dU), GO = scale gamma dO (over Y),
        // EU = e U (over K dS)
        for (int idx = tid; idx < C * C; idx += kBwdThreads) {
            const int r = idx / C, i = idx % C;
            sm[L::kKK + r * CP + i] = sm[L::kBeta + r] * sm[L::kT + r * CP + i] * sm[L::kKK + r * CP + i] +
                                      sm[L::kGam + r * CP + i] * sm[L::kA + r * CP + i];
        }
        for (int idx = tid; idx < C * kBwdCols; idx += kBwdThreads) {
            const int r = idx / kBwdCols, w = idx % kBwdCols;
            const float gr = sm[L::kGamma + r];
            sm[L::kTmp + r * WP + w] = -gr * sm[L::kBeta + r] * sm[L::kdB + r * WP + w];
            sm[L::kY + r * WP + w] = scale * gr * sm[L::kdO + r * WP + w];
            sm[L::kKdS + r * WP + w] = sm[L::kE + r] * sm[L::kU + r * WP + w];
        }
        __syncthreads();
        if (tid < C) {
            const int r = tid;
            float rs = 0.f, cs = 0.f;
            for (int i = 0; i < C; ++i) {
                rs += sm[L::kKK + r * CP + i];
                cs += sm[L::kKK + i * CP + r];
            }
            sm[L::kDG + r] += rs - cs;
        }
        __syncthreads();
        if (warp == 0) {
            // gamma_C = exp(G_{len-1}) and the numerators of e enter at row len-1
            float t = sm[L::kDe + lane] * sm[L::kE + lane] + sm[L::kDe + 32 + lane] * sm[L::kE + 32 + lane];
            t = warp_sum(t);
            float ss = 0.f;
            for (int w = 0; w < kBwdWarps; ++w) ss += sm[L::kRed + w];
            const float extra = t + sm[L::kGamma + C - 1] * ss;
            float x0 = sm[L::kDG + lane], x1 = sm[L::kDG + 32 + lane];
            if (lane == len - 1) x0 += extra;
            if (32 + lane == len - 1) x1 += extra;
            for (int off = 1; off < 32; off <<= 1) {    // suffix sums (reverse cumsum)
                const float y0 = __shfl_down_sync(0xffffffffu, x0, off);
                const float y1 = __shfl_down_sync(0xffffffffu, x1, off);
                if (lane + off < 32) { x0 += y0; x1 += y1; }
            }
            x0 += __shfl_sync(0xffffffffu, x1, 0);
            if (lane < len) {
                pdg[(size_t)(t0 + lane) * H + h] = x0;
                pdb[(size_t)(t0 + lane) * H + h] = sm[L::kDb + lane];
            }
            if (32 + lane < len) {
                pdg[(size_t)(t0 + 32 + lane) * H + h] = x1;
                pdb[(size_t)(t0 + 32 + lane) * H + h] = sm[L::kDb + 32 + lane];
            }
        }
        // dK = (P + P^T) K + R^T Q + D_gamma dX S0 + D_e U dS;  dQ = R K + scale D_gamma dO S0.
        // Each warp takes rows warp + 16 m (m < RPW) together, so every K, Q and
        // S0 / dS element it loads serves RPW rows.
        {
            float ak[RPW][DPL], aq[RPW][DPL];
#pragma unroll
            for (int m = 0; m < RPW; ++m)
#pragma unroll
                for (int j = 0; j < DPL; ++j) ak[m][j] = aq[m][j] = 0.f;
            for (int i = 0; i < C; ++i) {
                const float bi = sm[L::kBeta + i];
                float c1[RPW], rir[RPW], rri[RPW];
#pragma unroll
                for (int m = 0; m < RPW; ++m) {
                    const int r = warp + kBwdWarps * m;
                    c1[m] = sm[L::kBeta + r] * sm[L::kT + r * CP + i] + bi * sm[L::kT + i * CP + r];
                    rir[m] = sm[L::kGam + i * CP + r];
                    rri[m] = sm[L::kGam + r * CP + i];
                }
#pragma unroll
                for (int j = 0; j < DPL; ++j) {
                    const float kv = sK[i * KP + lane + 32 * j];
                    const float qv = sQ[i * KP + lane + 32 * j];
#pragma unroll
                    for (int m = 0; m < RPW; ++m) {
                        ak[m][j] += c1[m] * kv + rir[m] * qv;
                        aq[m][j] += rri[m] * kv;
                    }
                }
            }
            for (int w = 0; w < kBwdCols; ++w) {
                float gx[RPW], eu[RPW], go[RPW];
#pragma unroll
                for (int m = 0; m < RPW; ++m) {
                    const int r = warp + kBwdWarps * m;
                    gx[m] = sm[L::kTmp + r * WP + w];
                    go[m] = sm[L::kY + r * WP + w];
                    eu[m] = sm[L::kKdS + r * WP + w];
                }
#pragma unroll
                for (int j = 0; j < DPL; ++j) {
                    const int d = lane + 32 * j;
                    const float s0 = sS0[d * WP + w];
                    const float ds = sdS[d * WP + w];
#pragma unroll
                    for (int m = 0; m < RPW; ++m) {
                        ak[m][j] += gx[m] * s0 + eu[m] * ds;
                        aq[m][j] += go[m] * s0;
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < RPW; ++m) {
                const int r = warp + kBwdWarps * m;
                if (r < len) {
                    const size_t base = ((size_t)(t0 + r) * H + h) * DK;
#pragma unroll
                    for (int j = 0; j < DPL; ++j) {
                        pdk[base + lane + 32 * j] = ak[m][j];
                        pdq[base + lane + 32 * j] = aq[m][j];
                    }
                }
            }
        }
        __syncthreads();
        // dS for the chunk before: scale Q^T D_gamma dO + K^T D_gamma dX + gamma_C dS
        // (GO and GX hold scale gamma dO and gamma dX); each warp takes DPW
        // consecutive state rows together
        {
            const float gC = sm[L::kGamma + C - 1];
            float acc[DPW];
#pragma unroll
            for (int m = 0; m < DPW; ++m) acc[m] = 0.f;
            const int d0 = warp * DPW;                  // this warp's state rows d0 .. d0 + DPW - 1
            for (int r = 0; r < C; ++r) {
                const float go = sm[L::kY + r * WP + lane];
                const float gx = sm[L::kTmp + r * WP + lane];
                if constexpr (DPW % 4 == 0) {
#pragma unroll
                    for (int m = 0; m < DPW; m += 4) {
                        const float4 q4 = ld4f<TC>(sQ + r * KP + d0 + m);
                        const float4 k4 = ld4f<TC>(sK + r * KP + d0 + m);
                        acc[m] += q4.x * go + k4.x * gx;
                        acc[m + 1] += q4.y * go + k4.y * gx;
                        acc[m + 2] += q4.z * go + k4.z * gx;
                        acc[m + 3] += q4.w * go + k4.w * gx;
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < DPW; ++m) acc[m] += sQ[r * KP + d0 + m] * go + sK[r * KP + d0 + m] * gx;
                }
            }
#pragma unroll
            for (int m = 0; m < DPW; ++m) {
                const int d = d0 + m;
                sdS[d * WP + lane] = gC * sdS[d * WP + lane] + acc[m];
            }
        }
    }
    if constexpr (TC) tc_fence_before();
    __syncthreads();
    if (a.gs0) {
        for (int idx = tid; idx < DK * kBwdCols; idx += kBwdThreads) {
            const int d = idx / kBwdCols, w = idx % kBwdCols;
            a.gs0[(((size_t)n * H + h) * DK + d) * dv + col0 + w] = sdS[d * WP + w];
        }
    }
    if constexpr (TC) {
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tbase, 64);
        }
    }
}

// out[i] = sum over slices s of part[s * stride + i], the slices added in order
// (V = float4 for the dq / dk partials, float for dg / dbeta).
template <typename V>
__device__ __forceinline__ V add_v(V a, V b);
template <>
__device__ __forceinline__ float add_v<float>(float a, float b) { return a + b; }
template <>
__device__ __forceinline__ float4 add_v<float4>(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

template <typename V>
__global__ void __launch_bounds__(256) bwd_reduce_kernel(const V *part, V *out, long long n, long long stride,
                                                         int slices) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        V s = part[i];
        for (int sl = 1; sl < slices; ++sl) s = add_v(s, part[(size_t)sl * stride + i]);
        out[i] = s;
    }
}

template <int DK, typename TI>
cudaError_t launch_bwd_t(const BwdArgs &a, int slices, cudaStream_t s) {
    const size_t smem = BwdSmem<DK, kTcGram<DK, TI>>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel<DK, TI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_kernel<DK, TI><<<dim3(slices, a.H, a.N), kBwdThreads, smem, s>>>(a);
    return cudaGetLastError();
}

// n elements per slice, slices `stride` elements apart
cudaError_t launch_reduce(const float *part, float *out, long long n, long long stride, int slices, int sms,
                          cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const bool vec = (n % 4 == 0) && (stride % 4 == 0);
    const long long m = vec ? n / 4 : n;
    const long long blocks = std::min<long long>((m + 255) / 256, (long long)sms * 8);
    if (vec)
        bwd_reduce_kernel<float4><<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const float4 *>(part),
                                                                   reinterpret_cast<float4 *>(out), m, stride / 4,
                                                                   slices);
    else
        bwd_reduce_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(part, out, m, stride, slices);
    return cudaGetLastError();
}

std::atomic<int> g_bwd_kernel{GDN_KERNEL_AUTO};

bool head_dim_ok(int d) { return d == 32 || d == 64 || d == 128; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

struct BwdLayout {
    size_t err, states, pdq, pdk, pdg, pdb, prep, seqinfo, chunks, flags, tp, total;
    size_t dst, ry, rqs, ru, rdb, rkds;   // the tensor-core backward's intermediates (over the partials)
    int slices, max_chunks;
    long long total_T;
    int N;
};

bool bwd_layout(int B, int T, int H, int dk, int dv, int n_seqs, int varlen, int dtype, BwdLayout *L) {
    if (B < 1 || T < 0 || H < 1 || H > 4096) return false;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return false;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return false;
    if (varlen && (B != 1 || n_seqs < 1)) return false;
    const int N = varlen ? n_seqs : B;
    if (N > 65535) return false;
    const long long total_T = varlen ? (long long)T : (long long)B * T;
    if (total_T * H * 128 >= (1LL << 40) || total_T >= (1LL << 31)) return false;
    const long long slots = total_T / C + N;
    L->slices = dv / kBwdCols;
    L->total_T = total_T;
    L->N = N;
    size_t off = 0;
    L->err = off;
    off = round_up(off + sizeof(int));
    L->states = off;
    off = round_up(off + (size_t)slots * H * dk * dv * sizeof(float));
    // the CUDA-core kernel's per-slice partials and the tensor-core kernels'
    // intermediates share one region (a call uses one of them)
    const size_t shared0 = off;
    L->pdq = L->pdk = L->pdg = L->pdb = 0;
    if (L->slices > 1) {
        const size_t nk = (size_t)L->slices * total_T * H * dk * sizeof(float);
        const size_t nt = (size_t)L->slices * total_T * H * sizeof(float);
        L->pdq = off; off = round_up(off + nk);
        L->pdk = off; off = round_up(off + nk);
        L->pdg = off; off = round_up(off + nt);
        L->pdb = off; off = round_up(off + nt);
    }
    const size_t end_partials = off;
    off = shared0;
    L->dst = off; off = round_up(off + (size_t)slots * H * dk * dv * sizeof(float));
    const size_t rows = (size_t)total_T * H * dv * sizeof(float);
    L->ry = off; off = round_up(off + rows);
    L->rqs = off; off = round_up(off + rows);
    L->ru = off; off = round_up(off + rows);
    L->rdb = off; off = round_up(off + rows);
    L->rkds = off; off = round_up(off + rows);
    off = std::max(off, end_partials);
    // the chunk table (sequence prep) and T' of every chunk in fp32, formed
    // once before the backward kernel instead of a substitution per chunk,
    // value slice and sweep
    const long long nc_seq = ((long long)T + C - 1) / C;
    L->max_chunks = (int)(varlen ? total_T / C + N : (long long)B * nc_seq);
    L->prep = off;                                   // counters [8], num_chunks, num_items [4]
    off = round_up(off + 64);
    L->seqinfo = off;
    off = round_up(off + (size_t)N * 16);
    L->chunks = off;
    off = round_up(off + (size_t)L->max_chunks * 16);
    L->flags = off;
    off = round_up(off + (size_t)N * H * 4);
    L->tp = off;
    off = round_up(off + (size_t)total_T * H * C * sizeof(float));
    L->total = off;
    return true;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dv, int n_seqs, int varlen, gdn_dtype dtype) {
    BwdLayout L;
    if (!bwd_layout(B, T, H, dk, dv, n_seqs, varlen, dtype, &L)) return 0;
    return L.total;
}

}  // extern "C"

namespace {

// gdn_chunk_bwd, or with state_grad_only the reverse recurrence alone
// (gdn_chunk_state_grad: v and the per-token gradients unused).
gdn_status chunk_bwd_impl(const void *q, const void *k, const void *v, const float *g, const float *beta,
                          const float *initial_state, const int32_t *cu_seqlens, int n_seqs, float scale,
                          int B, int T, int H, int dk, int dv, gdn_dtype dtype,
                          const void *d_o, const float *d_final_state,
                          float *dq, float *dk_out, float *dv_out, float *dg, float *dbeta,
                          float *d_initial_state, void *workspace, size_t workspace_bytes, gdn_stream_t stream_in,
                          int state_grad_only) {
    const int varlen = cu_seqlens != nullptr;
    // the tensor-core kernels (the default) or the CUDA-core ones, fixed for the call
    const bool use_tc = state_grad_only || g_bwd_kernel.load() != GDN_KERNEL_SIMT;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return GDN_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDN_ERR_UNSUPPORTED;
    BwdLayout L;
    if (!bwd_layout(B, T, H, dk, dv, n_seqs, varlen, dtype, &L)) return GDN_ERR_INVALID_ARG;
    if (!workspace) return GDN_ERR_INVALID_ARG;
    if (state_grad_only) {
        if (!d_initial_state || (L.total_T > 0 && (!q || !k || !g || !beta || !d_o))) return GDN_ERR_INVALID_ARG;
    } else if (L.total_T > 0 &&
               (!q || !k || !v || !g || !beta || !d_o || !dq || !dk_out || !dv_out || !dg || !dbeta)) {
        return GDN_ERR_INVALID_ARG;
    }
    const void *ptrs[] = {q, k, v, g, beta, initial_state, d_o, d_final_state, dq, dk_out, dv_out, dg, dbeta,
                          d_initial_state, workspace};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
    if (workspace_bytes < L.total) return GDN_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_in);

    char *base = static_cast<char *>(workspace);
    BwdArgs a = {};
    a.q = q; a.k = k; a.v = v; a.dout = d_o;
    a.g = g; a.beta = beta; a.s0 = initial_state; a.dsf = d_final_state; a.cu = cu_seqlens;
    a.gv = dv_out; a.gs0 = d_initial_state;
    a.states = reinterpret_cast<float *>(base + L.states);
    a.err = reinterpret_cast<int *>(base + L.err);
    if (L.slices > 1) {
        a.gq = reinterpret_cast<float *>(base + L.pdq);
        a.gk = reinterpret_cast<float *>(base + L.pdk);
        a.gg = reinterpret_cast<float *>(base + L.pdg);
        a.gbeta = reinterpret_cast<float *>(base + L.pdb);
    } else {
        a.gq = dq; a.gk = dk_out; a.gg = dg; a.gbeta = dbeta;
    }
    a.part_stride_k = L.total_T * H * dk;
    a.part_stride_t = L.total_T * H;
    a.T = T; a.H = H; a.dv = dv; a.N = L.N; a.total_T = (int)L.total_T; a.varlen = varlen;
    a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)dk);

    cudaError_t e = cudaMemsetAsync(a.err, 0, sizeof(int), s);
    if (e != cudaSuccess) { set_error_detail("clear error word", e); return GDN_ERR_CUDA; }
    // the chunk table, then T' of every chunk (the kernel multiplies it by Gamma)
    a.tp = reinterpret_cast<float *>(base + L.tp);
    if (L.total_T > 0) {
        Problem p = {};
        p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.cu = cu_seqlens;
        p.B = B; p.T = T; p.H = H; p.dk = dk; p.dv = dv; p.N = L.N; p.total_T = (int)L.total_T;
        p.varlen = varlen; p.dtype = dtype; p.scale = a.scale;
        Workspace w = {};
        w.err = a.err;
        w.counters = reinterpret_cast<int *>(base + L.prep);
        w.num_chunks = reinterpret_cast<int *>(base + L.prep + 32);
        w.num_items = reinterpret_cast<int *>(base + L.prep + 48);
        w.seqinfo = reinterpret_cast<int4 *>(base + L.seqinfo);
        w.chunks = reinterpret_cast<int4 *>(base + L.chunks);
        w.flags = reinterpret_cast<int *>(base + L.flags);
        w.G = reinterpret_cast<float *>(base + L.tp);   // (not read: no gate factors)
        w.tprime = base + L.tp;
        w.max_chunks = L.max_chunks;
        if ((e = launch_seqprep(p, w, false, s)) != cudaSuccess) {
            set_error_detail("launch backward sequence prep", e);
            return GDN_ERR_CUDA;
        }
        if ((e = launch_inverse_f32(p, w, s, use_tc)) != cudaSuccess) {
            set_error_detail("launch backward inverse", e);
            return GDN_ERR_CUDA;
        }
    }
    const bool bf = dtype == GDN_BF16;
    if (use_tc) {
        if (L.total_T == 0 && !d_initial_state) return GDN_OK;
        BwdTcArgs t = {};
        t.q = q; t.k = k; t.v = v; t.dout = d_o;
        t.g = g; t.beta = beta; t.s0 = initial_state; t.dsf = d_final_state; t.cu = cu_seqlens;
        t.tp = a.tp;
        t.chunks = reinterpret_cast<const int4 *>(base + L.chunks);
        t.num_chunks = reinterpret_cast<const int *>(base + L.prep + 32);
        t.s0t = a.states;
        t.dst = reinterpret_cast<float *>(base + L.dst);
        t.ry = reinterpret_cast<float *>(base + L.ry);
        t.rqs = reinterpret_cast<float *>(base + L.rqs);
        t.ru = reinterpret_cast<float *>(base + L.ru);
        t.rdb = reinterpret_cast<float *>(base + L.rdb);
        t.rkds = reinterpret_cast<float *>(base + L.rkds);
        t.gq = dq; t.gk = dk_out; t.gv = dv_out; t.gg = dg; t.gbeta = dbeta; t.gs0 = d_initial_state;
        t.err = a.err;
        t.T = T; t.H = H; t.dk = dk; t.dv = dv; t.N = L.N; t.total_T = (int)L.total_T; t.varlen = varlen;
        t.dtype = dtype;
        t.state_grad_only = state_grad_only;
        t.scale = a.scale;
        if ((e = launch_bwd_tc(t, L.total_T > 0 ? L.max_chunks : 0, s)) != cudaSuccess) {
            set_error_detail("launch tensor-core backward", e);
            return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    if (dk == 32) e = bf ? launch_bwd_t<32, __nv_bfloat16>(a, L.slices, s) : launch_bwd_t<32, float>(a, L.slices, s);
    else if (dk == 64) e = bf ? launch_bwd_t<64, __nv_bfloat16>(a, L.slices, s) : launch_bwd_t<64, float>(a, L.slices, s);
    else e = bf ? launch_bwd_t<128, __nv_bfloat16>(a, L.slices, s) : launch_bwd_t<128, float>(a, L.slices, s);
    if (e != cudaSuccess) { set_error_detail("launch backward", e); return GDN_ERR_CUDA; }
    if (L.slices > 1) {
        int dev = 0, sms = 152;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            sms = 152;
        }
        const long long nk = L.total_T * H * dk, nt = L.total_T * H;
        if ((e = launch_reduce(a.gq, dq, nk, nk, L.slices, sms, s)) != cudaSuccess ||
            (e = launch_reduce(a.gk, dk_out, nk, nk, L.slices, sms, s)) != cudaSuccess ||
            (e = launch_reduce(a.gg, dg, nt, nt, L.slices, sms, s)) != cudaSuccess ||
            (e = launch_reduce(a.gbeta, dbeta, nt, nt, L.slices, sms, s)) != cudaSuccess) {
            set_error_detail("launch backward reduce", e);
            return GDN_ERR_CUDA;
        }
    }
    return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_bwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                         const float *initial_state, const int32_t *cu_seqlens, int n_seqs, float scale,
                         int B, int T, int H, int dk, int dv, gdn_dtype dtype,
                         const void *d_o, const float *d_final_state,
                         float *dq, float *dk_out, float *dv_out, float *dg, float *dbeta,
                         float *d_initial_state, void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
    return chunk_bwd_impl(q, k, v, g, beta, initial_state, cu_seqlens, n_seqs, scale, B, T, H, dk, dv, dtype, d_o,
                          d_final_state, dq, dk_out, dv_out, dg, dbeta, d_initial_state, workspace, workspace_bytes,
                          stream, 0);
}

gdn_status gdn_chunk_state_grad(const void *q, const void *k, const float *g, const float *beta,
                                const int32_t *cu_seqlens, int n_seqs, float scale, int B, int T, int H, int dk,
                                int dv, gdn_dtype dtype, const void *d_o, const float *d_final_state,
                                float *d_initial_state, void *workspace, size_t workspace_bytes,
                                gdn_stream_t stream) {
    return chunk_bwd_impl(q, k, nullptr, g, beta, nullptr, cu_seqlens, n_seqs, scale, B, T, H, dk, dv, dtype, d_o,
                          d_final_state, nullptr, nullptr, nullptr, nullptr, nullptr, d_initial_state, workspace,
                          workspace_bytes, stream, 1);
}

gdn_status gdn_set_backward_kernel(gdn_kernel kernel) {
    if (kernel != GDN_KERNEL_AUTO && kernel != GDN_KERNEL_TC && kernel != GDN_KERNEL_SIMT) return GDN_ERR_INVALID_ARG;
    g_bwd_kernel.store(kernel);
    return GDN_OK;
}

gdn_kernel gdn_get_backward_kernel(void) { return static_cast<gdn_kernel>(g_bwd_kernel.load()); }

gdn_status gdn_chunk_bwd_check(const void *workspace, gdn_stream_t stream) {
    return gdn_chunk_fwd_check(workspace, stream);
}

}  // extern "C"
