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
#include "gdn_internal.cuh"

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

cudaError_t launch_inverse(const Problem &p, const Workspace &w, cudaStream_t s) {
    const int smem = (kChunk * (p.dk + 1) + 2 * kChunk * 65) * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(inverse_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(w.max_chunks, p.H);
    inverse_simt_kernel<<<grid, 128, smem, s>>>(p, w);
    return cudaGetLastError();
}

}  // namespace gdn
