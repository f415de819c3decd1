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
// X_start(j+1).
//
// The walk is sequential in j, so each step must be short.  Columns (value
// rows of S) are independent: a CTA owns kScanCols of them for one unit and
// keeps its X_start columns in shared memory; X_M(j) (dk x dk fp32, contiguous)
// arrives by one bulk copy into a double buffer, the next one in flight while
// this one is used, and the product runs from shared memory with the reads of
// a warp spread over all banks.  CTAs loop over units (unit u, u + gridDim.x,
// ...), so the grid stays one wave.
#include <algorithm>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {

namespace {

constexpr int kScanCols = 8;       // value rows of S per CTA
constexpr int kScanThreads = 256;
constexpr uint64_t kScanTimeoutNs = 2000000000ull;

template <int DK>
constexpr size_t scan_smem_bytes() {
    // X_M double buffer | X_start [DK][kScanCols] | two mbarriers | abort flag
    return 2 * (size_t)DK * DK * 4 + (size_t)DK * kScanCols * 4 + 16 + 16;
}

template <int DK>
__global__ void __launch_bounds__(kScanThreads, 1) scan_kernel(const __grid_constant__ Problem p,
                                                                const __grid_constant__ Workspace w) {
    grid_dependency_wait();
    extern __shared__ __align__(128) float scan_smem[];
    float *X = scan_smem + 2 * DK * DK;                                   // [DK][kScanCols]
    uint64_t *bar = reinterpret_cast<uint64_t *>(X + DK * kScanCols);     // [2]
    int *abort_flag = reinterpret_cast<int *>(bar + 2);
    constexpr int kRows = DK * kScanCols / kScanThreads;                  // outputs per thread (same column)
    constexpr uint32_t kXmBytes = DK * DK * 4;
    static_assert(kRows >= 1 && (DK * kScanCols) % kScanThreads == 0, "scan tiling");

    const int dv = p.dv;
    const int i0 = blockIdx.y * kScanCols;
    if (i0 >= dv) return;
    const int n_units = w.num_items[2];
    const int tid = threadIdx.x, lane = tid & 31;
    const int ii = tid % kScanCols;                  // this thread's column
    const int jr0 = tid / kScanCols;                 // its first row; rows jr0 + q * (256 / kScanCols)
    const int grp = lane / kScanCols;                // rotation of the m loop (bank spread)
    if (tid == 0) {
        tc::mbar_init(&bar[0], 1);
        tc::mbar_init(&bar[1], 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    // per buffer: phases waited for (every thread; gives the parity) and copies
    // issued (thread 0 only); scalars, so that nothing is indexed at run time
    uint32_t uses0 = 0, uses1 = 0, issued0 = 0, issued1 = 0;

    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int4 su = w.scan_units[u];
        const int NS = su.z, b = su.w;
        for (int idx = tid; idx < DK * kScanCols; idx += kScanThreads) {
            const int jr = idx / kScanCols, c = idx % kScanCols;
            X[idx] = w.cp_s[((size_t)b * DK + jr) * dv + i0 + c];
        }
        if (tid == 0 && NS - 2 >= 1) {
            tc::mbar_arrive_expect_tx(&bar[0], kXmBytes);
            tc::bulk_load(scan_smem, w.cp_m + (size_t)(b + 1) * DK * DK, kXmBytes, &bar[0]);
            ++issued0;
        }
        __syncthreads();
        bool ok = true;
        for (int j = 1; j <= NS - 2; ++j) {
            const int cur = (j - 1) & 1, nxt = j & 1;
            if (tid == 0 && j + 1 <= NS - 2) {
                // buffer nxt was last read in step j - 1, which every thread has left
                tc::mbar_arrive_expect_tx(&bar[nxt], kXmBytes);
                tc::bulk_load(scan_smem + nxt * DK * DK, w.cp_m + (size_t)(b + j + 1) * DK * DK, kXmBytes,
                              &bar[nxt]);
                if (nxt) ++issued1; else ++issued0;
            }
            float *XS = w.cp_s + (size_t)(b + j) * DK * dv;
            float acc[kRows];
#pragma unroll
            for (int q = 0; q < kRows; ++q) acc[q] = XS[(size_t)(jr0 + q * (kScanThreads / kScanCols)) * dv + i0 + ii];
            const bool got = tc::mbar_wait(&bar[cur], (cur ? uses1 : uses0) & 1u, abort_flag, kScanTimeoutNs);
            if (cur) ++uses1; else ++uses0;
            if (!__syncthreads_and(got)) {
                if (tid == 0 && atomicExch(abort_flag, 1) == 0) report_error(w.err, GDN_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const float *XM = scan_smem + cur * DK * DK;
#pragma unroll 4
            for (int mm = 0; mm < DK; ++mm) {
                const int m = (mm + grp) & (DK - 1);
                const float xv = X[m * kScanCols + ii];
#pragma unroll
                for (int q = 0; q < kRows; ++q)
                    acc[q] = fmaf(XM[(jr0 + q * (kScanThreads / kScanCols)) * DK + m], xv, acc[q]);
            }
            __syncthreads();                         // every read of X and of this X_M buffer is done
#pragma unroll
            for (int q = 0; q < kRows; ++q) {
                const int jr = jr0 + q * (kScanThreads / kScanCols);
                X[jr * kScanCols + ii] = acc[q];
                XS[(size_t)jr * dv + i0 + ii] = acc[q];
            }
            __syncthreads();
        }
        if (!ok) break;
    }
    // no bulk copy may still be landing when the CTA leaves: a buffer never has
    // more than one copy in flight, so waiting for its latest one covers it
    if (tid == 0) {
        int never = 0;
        if (issued0 > 0) tc::mbar_wait(&bar[0], (issued0 - 1) & 1u, &never, kScanTimeoutNs);
        if (issued1 > 0) tc::mbar_wait(&bar[1], (issued1 - 1) & 1u, &never, kScanTimeoutNs);
    }
}

template <int DK>
cudaError_t launch_scan_dk(const Problem &p, const Workspace &w, cudaStream_t s) {
    constexpr size_t smem = scan_smem_bytes<DK>();
    cudaError_t e = cudaFuncSetAttribute(scan_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        sms = 152;
    }
    const int col_blocks = (p.dv + kScanCols - 1) / kScanCols;
    const int gx = std::max(1, std::min(w.max_cp_slots, sms / col_blocks));   // one wave at one CTA per SM
    e = launch_dependent(scan_kernel<DK>, dim3(gx, col_blocks), dim3(kScanThreads), smem, s, p, w);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Start states of R consecutive slices (inter-card sequence parallelism): the
// same step as above, X_start(r+1) = X_M(r) X_start(r) + X*(r), over maps laid
// out rank-major ([R][N][H][...]), as an all-gather delivers them.  One CTA
// per (unit, kScanCols value rows) walks the ranks in order; X_M(r) is staged
// in shared memory by plain 16-byte loads (R is the rank count: a handful of
// steps, so no copy pipeline).
//
// GRAD: the gradient of the state walks the other way, dS_end(r) =
// dS_end(r+1) M(r+1)^T + dS*(r+1) (S_end = S_start M + S* gives
// dL/dS_start = dL/dS_end M^T plus the slice's own term), which in the stored
// layout reads Y(r) = X_M(r+1)^T Y(r+1) + Y*(r+1): the same walk from the last
// slice down, with X_M read transposed.
template <int DK, bool GRAD>
__global__ void __launch_bounds__(kScanThreads) rank_scan_kernel(const float *__restrict__ s0,
                                                                 const float *__restrict__ s_star,
                                                                 const float *__restrict__ m, int R, int units,
                                                                 int dv, float *__restrict__ out) {
    extern __shared__ __align__(16) float rs_smem[];
    float *XM = rs_smem;                   // [DK][DK]
    float *X = rs_smem + DK * DK;          // [DK][kScanCols]
    constexpr int kRows = DK * kScanCols / kScanThreads;
    const int u = blockIdx.x, i0 = blockIdx.y * kScanCols;
    if (u >= units || i0 >= dv) return;
    const int tid = threadIdx.x;
    const int ii = tid % kScanCols, jr0 = tid / kScanCols;
    const size_t sstride = (size_t)units * DK * dv, mstride = (size_t)units * DK * DK;
    const size_t ubase = (size_t)u * DK * dv;
    const int first = GRAD ? R - 1 : 0;
    for (int idx = tid; idx < DK * kScanCols; idx += kScanThreads) {
        const int jr = idx / kScanCols, c = idx % kScanCols;
        const float x = (s0 && i0 + c < dv) ? s0[ubase + (size_t)jr * dv + i0 + c] : 0.f;
        X[idx] = x;
        if (i0 + c < dv) out[first * sstride + ubase + (size_t)jr * dv + i0 + c] = x;
    }
    for (int step = 0; step + 1 < R; ++step) {
        const int r = GRAD ? R - 1 - step : step;     // the map applied in this step
        const int dst = GRAD ? r - 1 : r + 1;         // the slice whose value it gives
        const float4 *src = reinterpret_cast<const float4 *>(m + r * mstride + (size_t)u * DK * DK);
        for (int idx = tid; idx < DK * DK / 4; idx += kScanThreads) reinterpret_cast<float4 *>(XM)[idx] = src[idx];
        __syncthreads();
        float acc[kRows];
        const float *xs = s_star + r * sstride + ubase;
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int jr = jr0 + q * (kScanThreads / kScanCols);
            acc[q] = i0 + ii < dv ? xs[(size_t)jr * dv + i0 + ii] : 0.f;
        }
#pragma unroll 4
        for (int mm = 0; mm < DK; ++mm) {
            const float xv = X[mm * kScanCols + ii];
#pragma unroll
            for (int q = 0; q < kRows; ++q) {
                const int jr = jr0 + q * (kScanThreads / kScanCols);
                acc[q] = fmaf(GRAD ? XM[mm * DK + jr] : XM[jr * DK + mm], xv, acc[q]);
            }
        }
        __syncthreads();                   // every read of X and XM is done
        float *o = out + dst * sstride + ubase;
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int jr = jr0 + q * (kScanThreads / kScanCols);
            X[jr * kScanCols + ii] = acc[q];
            if (i0 + ii < dv) o[(size_t)jr * dv + i0 + ii] = acc[q];
        }
        __syncthreads();
    }
}

template <int DK, bool GRAD>
cudaError_t launch_rank_scan_dk(const float *s0, const float *s_star, const float *m, int R, int units, int dv,
                                float *out, cudaStream_t s) {
    const size_t smem = ((size_t)DK * DK + (size_t)DK * kScanCols) * 4;
    cudaError_t e =
        cudaFuncSetAttribute(rank_scan_kernel<DK, GRAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(units, (dv + kScanCols - 1) / kScanCols);
    rank_scan_kernel<DK, GRAD><<<grid, kScanThreads, smem, s>>>(s0, s_star, m, R, units, dv, out);
    return cudaGetLastError();
}

template <bool GRAD>
cudaError_t launch_rank_scan_any(const float *s0, const float *s_star, const float *m, int R, int units, int dk,
                                 int dv, float *out, cudaStream_t s) {
    if (dk == 32) return launch_rank_scan_dk<32, GRAD>(s0, s_star, m, R, units, dv, out, s);
    if (dk == 64) return launch_rank_scan_dk<64, GRAD>(s0, s_star, m, R, units, dv, out, s);
    return launch_rank_scan_dk<128, GRAD>(s0, s_star, m, R, units, dv, out, s);
}

}  // namespace

cudaError_t launch_rank_scan(const float *s0, const float *s_star, const float *m, int R, int N, int H, int dk,
                             int dv, float *out, bool grad, cudaStream_t s) {
    const int units = N * H;
    if (units == 0 || R == 0) return cudaSuccess;
    return grad ? launch_rank_scan_any<true>(s0, s_star, m, R, units, dk, dv, out, s)
                : launch_rank_scan_any<false>(s0, s_star, m, R, units, dk, dv, out, s);
}

cudaError_t launch_scan(const Problem &p, const Workspace &w, cudaStream_t s) {
    if (w.max_cp_slots <= 0) return cudaSuccess;
    if (p.dk == 32) return launch_scan_dk<32>(p, w, s);
    if (p.dk == 64) return launch_scan_dk<64>(p, w, s);
    return launch_scan_dk<128>(p, w, s);
}

}  // namespace gdn
