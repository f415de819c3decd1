// Segment scan of intra-card sequence parallelism (FlashQLA talk
// "Qwen系列模型线性注意力高性能优化实践", difference and compute-for-memory
// paragraphs): each segment j of a unit was run once from a wrong start, giving
// its end state S*_j and its correction matrix M_j (the difference between
// right and wrong states is carried by M: S_end = S_start M_j + S*_j).  This
// kernel walks the segments in order to turn those pairs into exact start
// states.
//
// Stored (k-major) layout: X[j][i] = S[i][j].  The correction pass stores its
// end state the same way, X_M = M^T, so one step reads
//     X_start(j+1) = X_M(j) X_start(j) + X*(j)
// Slot b of a unit first holds the exact end of segment 0 (= start of
// segment 1); slot b+j (j >= 1) holds X*(j) and M(j) and is overwritten with
// X_start(j+1).  Columns (value rows of S) are independent, so the grid splits
// them into blocks of 16.
#include "gdn_internal.cuh"

namespace gdn {

constexpr int kScanCols = 16;

__global__ void __launch_bounds__(256) scan_kernel(const __grid_constant__ Problem p, const __grid_constant__ Workspace w) {
    grid_dependency_wait();
    __shared__ float X[128][kScanCols + 1];
    const int u = blockIdx.x;
    if (u >= w.num_items[2]) return;
    const int4 su = w.scan_units[u];
    const int NS = su.z, b = su.w;
    const int dk = p.dk, dv = p.dv;
    const int i0 = blockIdx.y * kScanCols;
    if (i0 >= dv) return;
    const int ni = min(kScanCols, dv - i0);
    const int tid = threadIdx.x;
    for (int idx = tid; idx < dk * kScanCols; idx += blockDim.x) {
        const int jr = idx / kScanCols, ii = idx % kScanCols;
        X[jr][ii] = ii < ni ? w.cp_s[((size_t)b * dk + jr) * dv + i0 + ii] : 0.f;
    }
    __syncthreads();
    constexpr int kPer = 128 * kScanCols / 256;
    for (int j = 1; j <= NS - 2; ++j) {
        const float *XM = w.cp_m + (size_t)(b + j) * dk * dk;
        float *XS = w.cp_s + (size_t)(b + j) * dk * dv;
        float acc[kPer];
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int idx = tid + q * 256;
            const int jr = idx / kScanCols, ii = idx % kScanCols;
            float a = 0.f;
            if (jr < dk && ii < ni) {
                a = XS[(size_t)jr * dv + i0 + ii];
                for (int m = 0; m < dk; ++m) a = fmaf(XM[(size_t)jr * dk + m], X[m][ii], a);
            }
            acc[q] = a;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int idx = tid + q * 256;
            const int jr = idx / kScanCols, ii = idx % kScanCols;
            if (jr < dk) {
                X[jr][ii] = acc[q];
                if (ii < ni) XS[(size_t)jr * dv + i0 + ii] = acc[q];
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_scan(const Problem &p, const Workspace &w, cudaStream_t s) {
    if (w.max_cp_slots <= 0) return cudaSuccess;
    dim3 grid(w.max_cp_slots, (p.dv + kScanCols - 1) / kScanCols);
    cudaError_t e = launch_dependent(scan_kernel, grid, dim3(256), 0, s, p, w);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn
