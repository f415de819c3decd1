// Per-chunk inverse (step one of the four-step paragraph of the FlashQLA talk
// "Qwen系列模型线性注意力高性能优化实践"), in the Gamma-free form of the
// Gamma-extraction paragraph:
//
//     A' = diag(beta) strictlower(K K^T),   T' = (I + A')^{-1}
//
// T' is unit lower-triangular; the gate enters later as T = Gamma ⊙ T' (the
// fused kernel builds Gamma anyway), so this kernel issues no exponentials.
// Output: T' rows by token, [H, total_T, 64], bf16 for bf16 inputs and fp32 for
// fp32 inputs; entries past the chunk's length are zero and rows past the end
// of a sequence are not written.
#include <string.h>

#include <mutex>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {

// One CTA per (chunk, head).  K K^T on CUDA cores, then each of 64 threads
// solves one column of (I + A') X = I by forward substitution; the columns are
// independent, so the substitution needs no barrier.
__global__ void __launch_bounds__(128) inverse_simt_kernel(Problem p, Workspace w) {
    extern __shared__ float smem[];
    __shared__ float sb[kChunk];
    const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    if (cid >= *w.num_chunks) return;
    const int4 ci = w.chunks[cid];
    const int t0 = ci.y, len = ci.z;
    const int dk = p.dk, ks = dk + 1;
    float *Ks = smem;                 // [64][dk+1]
    float *A = Ks + kChunk * ks;      // [64][65]
    float *X = A + kChunk * 65;       // [64][65]
    for (int idx = tid; idx < kChunk * dk; idx += blockDim.x) {
        const int r = idx / dk, j = idx % dk;
        Ks[r * ks + j] = r < len ? load_elem(p.k, ((size_t)(t0 + r) * p.H + h) * dk + j, p.dtype) : 0.f;
    }
    if (tid < kChunk) sb[tid] = tid < len ? p.beta[(size_t)(t0 + tid) * p.H + h] : 0.f;
    __syncthreads();
    for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
        const int r = idx / kChunk, m = idx % kChunk;
        float a = 0.f;
        if (m < r) {
            for (int j = 0; j < dk; ++j) a = fmaf(Ks[r * ks + j], Ks[m * ks + j], a);
            a *= sb[r];
        }
        A[r * 65 + m] = a;
    }
    __syncthreads();
    if (tid < kChunk) {
        const int j = tid;
        for (int m = 0; m < kChunk; ++m) X[m * 65 + j] = (m == j) ? 1.f : 0.f;
        for (int r = j + 1; r < kChunk; ++r) {
            float acc = 0.f;
            for (int m = j; m < r; ++m) acc = fmaf(A[r * 65 + m], X[m * 65 + j], acc);
            X[r * 65 + j] = -acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < len * kChunk; idx += blockDim.x) {
        const int r = idx / kChunk, m = idx % kChunk;
        store_elem(w.tprime, ((size_t)h * p.total_T + t0 + r) * kChunk + m, p.dtype, X[r * 65 + m]);
    }
}

// ---------------------------------------------------------------------------
// tcgen05 variant for bf16 keys with dk = 128.  One CTA takes one chunk of two
// heads: TMA brings both 64 x 128 key tiles (128-byte swizzle), one M = N = 128
// MMA forms [K1; K2] [K1; K2]^T in tensor memory (the two diagonal 64 x 64
// blocks are the Gram matrices), each thread turns its row into A' in shared
// memory, and each of the four warps solves 32 columns of one head's
// (I + A') X = I by forward substitution with the column held in registers.
// ---------------------------------------------------------------------------
namespace {

constexpr int kInvThreads = 128;
constexpr int kAStride = 68;  // floats per row of A' (16-byte aligned rows)
constexpr uint32_t kInvKBytes = 32768;
constexpr uint32_t kInvABytes = 2 * kChunk * kAStride * 4;  // 34816
constexpr uint32_t kInvSmem = kInvKBytes + kInvABytes + 1024 + 1024;  // T' staging reuses the key tile
constexpr uint64_t kInvTimeoutNs = 2000000000ull;

struct InvMaps {
    CUtensorMap k;
};

// x_r for r in [R0, 64): x_r = -sum_{m in [R0, r)} A'[r][m] x_m, with x_j = 1 and
// x_r = 0 for r < j.  All indices are compile-time after unrolling.
// Four independent partial sums keep the FMA pipe busy instead of one chain.
template <int R0>
__device__ __forceinline__ void solve_column(const float *A, int j, float *x) {
#pragma unroll
    for (int r = R0; r < kChunk; ++r) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int m = R0; m + 3 < r; m += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(A + r * kAStride + m);
            a0 = fmaf(a.x, x[m], a0);
            a1 = fmaf(a.y, x[m + 1], a1);
            a2 = fmaf(a.z, x[m + 2], a2);
            a3 = fmaf(a.w, x[m + 3], a3);
        }
#pragma unroll
        for (int m = R0 + ((r - R0) & ~3); m < r; ++m) a0 = fmaf(A[r * kAStride + m], x[m], a0);
        const float acc = (a0 + a1) + (a2 + a3);
        x[r] = (r < j) ? 0.f : ((r == j) ? 1.f : -acc);
    }
}

__global__ void __launch_bounds__(kInvThreads) inverse_tc_kernel(const __grid_constant__ InvMaps maps, Problem p,
                                                                  Workspace w) {
    extern __shared__ uint8_t inv_smem_raw[];
    uint8_t *smem =
        reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(inv_smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ktile = smem;
    float *A = reinterpret_cast<float *>(smem + kInvKBytes);
    __nv_bfloat16 *X = reinterpret_cast<__nv_bfloat16 *>(smem);  // the key tile is dead after the MMA
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kInvKBytes + kInvABytes);
    float *sbeta = reinterpret_cast<float *>(bars + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbeta + 128);
    __shared__ int s_abort;

    const int cid = blockIdx.x;
    if (cid >= *w.num_chunks) return;
    const int4 ci = w.chunks[cid];
    const int t0 = ci.y, len = ci.z;
    const int h0 = 2 * blockIdx.y;
    const int h1 = min(h0 + 1, p.H - 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        tc::mbar_init(&bars[0], 1);
        tc::mbar_init(&bars[1], 1);
        s_abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, 128);
    {
        const int r = threadIdx.x, rl = r & 63;
        const int head = r < 64 ? h0 : h1;
        sbeta[r] = rl < len ? p.beta[(size_t)(t0 + rl) * p.H + head] : 0.f;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    if (threadIdx.x == 0) {
        tc::mbar_arrive_expect_tx(&bars[0], kInvKBytes);
        tc::tma_load_3d(ktile + 0, &maps.k, &bars[0], 0, h0, t0);
        tc::tma_load_3d(ktile + 8192, &maps.k, &bars[0], 0, h1, t0);
        tc::tma_load_3d(ktile + 16384, &maps.k, &bars[0], 64, h0, t0);
        tc::tma_load_3d(ktile + 24576, &maps.k, &bars[0], 64, h1, t0);
    }
    bool ok = tc::mbar_wait(&bars[0], 0, &s_abort, kInvTimeoutNs);
    if (threadIdx.x == 0 && ok) {
        tc::tc_fence_after();
        const uint32_t kb = tc::smem_u32(ktile);
        constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint64_t d = tc::smem_desc_sw128(kb + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
            tc::mma_ss(tbase, d, d, idesc, kk > 0);
        }
        tc::tc_commit(&bars[1]);
    }
    ok = ok && tc::mbar_wait(&bars[1], 0, &s_abort, kInvTimeoutNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        if (atomicExch(&s_abort, 1) == 0) report_error(w.err, GDN_ERR_TIMEOUT);
    } else {
        // row r of [K1;K2][K1;K2]^T -> A' row of its head: beta_r * (k_r . k_m) for m < r
        tc::tc_fence_after();
        const int r = threadIdx.x, c = r >> 6, rl = r & 63;
        float *Arow = A + (c * kChunk + rl) * kAStride;
        const float br = sbeta[r];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
            tc::tmem_ld32(tbase + (static_cast<uint32_t>(32 * warp) << 16) + 64 * c + 32 * hh, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int m = 32 * hh + jj;
                Arow[m] = m < rl ? br * __uint_as_float(v[jj]) : 0.f;
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, 128);
    }
    if (s_abort) return;
    // forward substitution: warp q solves columns 32 (q & 1) + lane of head (q >> 1)
    {
        const int c = warp >> 1, j = 32 * (warp & 1) + lane;
        const float *Ac = A + c * kChunk * kAStride;
        float x[kChunk];
        if ((warp & 1) == 0) {
            solve_column<0>(Ac, j, x);
        } else {
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = 0.f;
            solve_column<32>(Ac, j, x);
        }
        __nv_bfloat16 *Xc = X + c * kChunk * kChunk;
#pragma unroll
        for (int r = 0; r < kChunk; ++r) Xc[r * kChunk + j] = __float2bfloat16_rn(x[r]);
    }
    __syncthreads();
    // coalesced 16-byte stores of the valid rows of both heads
    for (int idx = threadIdx.x; idx < 2 * kChunk * 8; idx += kInvThreads) {
        const int c = idx >> 9, r = (idx >> 3) & 63, q = idx & 7;
        const int head = c ? h1 : h0;
        if (r >= len || (c == 1 && h1 == h0)) continue;
        const uint4 v = *reinterpret_cast<const uint4 *>(X + (c * kChunk + r) * kChunk + 8 * q);
        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(w.tprime) +
                                   ((size_t)head * p.total_T + t0 + r) * kChunk + 8 * q) = v;
    }
}

typedef CUresult (*EncodeTiledFnInv)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);

EncodeTiledFnInv inv_encode_fn() {
    static std::once_flag once;
    static EncodeTiledFnInv fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnInv>(ptr);
        cudaGetLastError();
    });
    return fn;
}

cudaError_t launch_inverse_tc(const Problem &p, const Workspace &w, cudaStream_t s) {
    EncodeTiledFnInv fn = inv_encode_fn();
    if (!fn) {
        set_error_detail("driver entry point cuTensorMapEncodeTiled", cudaErrorNotSupported);
        return cudaErrorNotSupported;
    }
    InvMaps maps;
    memset(&maps, 0, sizeof(maps));
    cuuint64_t dims[3] = {(cuuint64_t)p.dk, (cuuint64_t)p.H, (cuuint64_t)p.total_T};
    cuuint64_t strides[2] = {(cuuint64_t)p.dk * 2, (cuuint64_t)p.H * p.dk * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    const int r = fn(&maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.k), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != 0) {
        set_error_detail("encode tensor map (inverse)", cudaErrorInvalidValue, r);
        return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(inverse_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kInvSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(w.max_chunks, (p.H + 1) / 2);
    inverse_tc_kernel<<<grid, kInvThreads, kInvSmem, s>>>(maps, p, w);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_inverse(const Problem &p, const Workspace &w, cudaStream_t s) {
    if (p.dtype == GDN_BF16 && p.dk == 128 && p.total_T > 0) return launch_inverse_tc(p, w, s);
    const int smem = (kChunk * (p.dk + 1) + 2 * kChunk * 65) * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(inverse_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(w.max_chunks, p.H);
    inverse_simt_kernel<<<grid, 128, smem, s>>>(p, w);
    return cudaGetLastError();
}

}  // namespace gdn
