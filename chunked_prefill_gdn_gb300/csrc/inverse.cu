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

#include <algorithm>
#include <mutex>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {

// One CTA per (chunk, head).  K K^T on CUDA cores, then each of 64 threads
// solves one column of (I + A') X = I by forward substitution; the columns are
// independent, so the substitution needs no barrier.
__global__ void __launch_bounds__(128) inverse_simt_kernel(const __grid_constant__ Problem p, const __grid_constant__ Workspace w) {
    grid_dependency_wait();
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

}  // namespace gdn

#include "inverse_tc.cuh"

namespace gdn {
namespace {

template <bool F32K>
__global__ void __launch_bounds__(kInvThreads, 1) inverse_tc_kernel(const __grid_constant__ InvMaps maps, const __grid_constant__ Problem p,
                                                                     const __grid_constant__ Workspace w, int gate_scaled,
                                                                     const InvSel sel) {
    grid_dependency_wait();
    extern __shared__ uint8_t inv_smem_raw[];
    InvSel s = sel;
    s.cta = blockIdx.x;
    s.ctas = gridDim.x;
    inverse_tc_body<F32K>(&maps.k, p, w, gate_scaled, s, inv_smem_raw);
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

cudaError_t launch_inverse_tc(const Problem &p, const Workspace &w, int gate_scaled, int cols, int nc, int f32_out,
                              cudaStream_t s) {
    EncodeTiledFnInv fn = inv_encode_fn();
    if (!fn) {
        set_error_detail("driver entry point cuTensorMapEncodeTiled", cudaErrorNotSupported);
        return cudaErrorNotSupported;
    }
    InvMaps maps;
    memset(&maps, 0, sizeof(maps));
    // bf16 keys: boxes of 64 features; fp32 keys (read as tf32): 32 features,
    // both 128 bytes wide, 64 token rows
    const bool f32k = p.dtype == GDN_F32;
    const cuuint64_t es_bytes = f32k ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)p.dk, (cuuint64_t)p.H, (cuuint64_t)p.total_T};
    cuuint64_t strides[2] = {(cuuint64_t)p.dk * es_bytes, (cuuint64_t)p.H * p.dk * es_bytes};
    cuuint32_t box[3] = {f32k ? 32u : 64u, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    const int r = fn(&maps.k, f32k ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void *>(p.k), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != 0) {
        set_error_detail("encode tensor map (inverse)", cudaErrorInvalidValue, r);
        return cudaErrorInvalidValue;
    }
    auto kernel = f32k ? inverse_tc_kernel<true> : inverse_tc_kernel<false>;
    const uint32_t smem = f32k ? InvCfg<true>::kSmem : InvCfg<false>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // all chunks, or only chunk columns [0, cols) of equal sequences when the
    // fused kernel computes the others
    InvSel sel = {};
    sel.mode = cols < nc ? 1 : 0;
    sel.nc = nc;
    sel.c0 = cols;
    sel.f32_out = f32_out;
    const long long pairs = (sel.mode ? (long long)p.N * cols : (long long)w.max_chunks) * ((p.H + 1) / 2);
    if (pairs == 0) return cudaSuccess;
    const int grid = (int)std::max(1LL, std::min<long long>(sms, pairs));
    e = launch_dependent(kernel, dim3(grid), dim3(kInvThreads), smem, s, maps, p, w, gate_scaled, sel);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_inverse(const Problem &p, const Workspace &w, bool for_tc, cudaStream_t s, int cols, int nc) {
    // (the tcgen05 inverse pads head sizes 32 and 64 to 128 with zero features)
    const bool dk_ok = p.dk == 32 || p.dk == 64 || p.dk == 128;
    if (p.dtype == GDN_BF16 && dk_ok && p.total_T > 0) return launch_inverse_tc(p, w, for_tc ? 1 : 0, cols, nc, 0, s);
    // fp32 keys for the tcgen05 fused kernel: the Gram on kind::tf32, T'
    // itself stored in fp32 (the CUDA-core kernel keeps fp32 throughout below)
    if (p.dtype == GDN_F32 && for_tc && dk_ok && p.total_T > 0) return launch_inverse_tc(p, w, 0, 0, 0, 1, s);
    const int smem = (kChunk * (p.dk + 1) + 2 * kChunk * 65) * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(inverse_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(w.max_chunks, p.H);
    e = launch_dependent(inverse_simt_kernel, grid, dim3(128), (size_t)smem, s, p, w);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// T' itself (no gate factors) as fp32 rows [H, total_T, 64], for the
// backward pass: the tcgen05 inverse for bf16 keys and, with tc, for fp32 keys
// (Gram on kind::tf32); else the CUDA-core one (fp32 throughout).
cudaError_t launch_inverse_f32(const Problem &p, const Workspace &w, cudaStream_t s, bool tc) {
    if (p.total_T == 0) return cudaSuccess;
    if ((p.dtype == GDN_BF16 || tc) && (p.dk == 32 || p.dk == 64 || p.dk == 128))
        return launch_inverse_tc(p, w, 0, 0, 0, 1, s);
    if (p.dtype != GDN_F32) return cudaErrorNotSupported;
    return launch_inverse(p, w, false, s);
}

}  // namespace gdn
