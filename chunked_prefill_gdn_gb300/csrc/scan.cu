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
// keeps its X_start columns in shared memory, and CTAs loop over units (unit
// u, u + gridDim.x, ...), so the grid stays one wave.  X_M(j) (dk x dk fp32,
// contiguous) arrives by 16-byte asynchronous copies into a double buffer
// whose rows are padded by four floats, the next one in flight while this one
// is used.  Each thread forms a 4 x 2 block of the product (rows r + dk/4 q,
// q = 0..3, of one pair of columns) over one quarter of k from 16-byte loads:
// with the padding the eight rows a warp reads at one k fall in distinct
// banks, and the columns are broadcast; the quarters' sums meet in shared
// memory (four warps per sub-partition instead of one, to hide latency).  X_start is kept with consecutive k paired, [k/2][column][k%2],
// so that one load gives two (k, k+1) pairs and the sums run on the two-wide
// FMA over even and odd k, added at the end.
#include <algorithm>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {

namespace {

constexpr int kScanCols = 8;       // value rows of S per CTA
constexpr int kScanThreads = 256;  // the rank scan below

template <int DK>
struct ScanCfg {
    static constexpr int kRowGroups = DK / 4;                          // rows r = g + kRowGroups q
    static constexpr int kTile = 4 * kRowGroups;                       // threads per k quarter: four column pairs
    static constexpr int kSplit = 4;                                   // k quarters, summed in shared memory
    static constexpr int kThreads = kSplit * kTile;
    static constexpr int kPitch = DK + 4;                              // floats per X_M row in shared memory
    static constexpr int kBufFloats = DK * kPitch;
    static constexpr int kRedFloats = (kSplit - 1) * kTile * 8;        // partial sums of quarters 1..3
    static constexpr size_t kSmem = (2 * (size_t)kBufFloats + (size_t)DK * kScanCols + kRedFloats) * 4;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// (lo, hi) pairs of fp32 in one 64-bit register, for the two-wide FMA
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void fma2(uint64_t &acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// X_M(slot) into a padded buffer (all threads; one commit group)
template <int DK>
__device__ __forceinline__ void load_xm(float *buf, const float *src, int tid) {
    constexpr int kPerRow = DK / 4;
    for (int idx = tid; idx < DK * kPerRow; idx += ScanCfg<DK>::kThreads) {
        const int r = idx / kPerRow, k = idx - r * kPerRow;
        cp_async16(tc::smem_u32(buf + r * ScanCfg<DK>::kPitch + 4 * k), src + (size_t)r * DK + 4 * k);
    }
    cp_async_commit();
}

template <int DK>
__global__ void __launch_bounds__(ScanCfg<DK>::kThreads, 1) scan_kernel(const __grid_constant__ Problem p,
                                                                         const __grid_constant__ Workspace w) {
    using Cfg = ScanCfg<DK>;
    grid_dependency_wait();
    extern __shared__ __align__(128) float scan_smem[];
    float *X2 = scan_smem + 2 * Cfg::kBufFloats;    // [DK/2][kScanCols][2]: X_start, k pairs
    float *red = X2 + DK * kScanCols;               // [kSplit - 1][kTile][8]
    const int dv = p.dv;
    const int i0 = blockIdx.y * kScanCols;
    if (i0 >= dv) return;
    const int n_units = w.num_items[2];
    const int tid = threadIdx.x;
    const int kz = tid / Cfg::kTile, tt = tid - kz * Cfg::kTile;   // k quarter (whole warps); place in it
    const int cg = tt & 3, g = tt >> 2;             // columns i0 + 2 cg, + 1; rows g + kRowGroups q
    constexpr int kQ = DK / Cfg::kSplit;            // k per quarter

    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int4 su = w.scan_units[u];
        const int NS = su.z, b = su.w;
        if (NS > 2) {
            // the unit's correction matrices into L2, shared out over the CTAs
            // of its columns, and this CTA's columns of the end states
            const char *m0 = reinterpret_cast<const char *>(w.cp_m + (size_t)(b + 1) * DK * DK);
            const int lines = (NS - 2) * (DK * DK * 4 / 128);
            for (int l = blockIdx.y * Cfg::kThreads + tid; l < lines; l += gridDim.y * Cfg::kThreads)
                tc::l2_prefetch_line(m0 + (size_t)l * 128);
            for (int idx = tid; idx < (NS - 2) * DK; idx += Cfg::kThreads)
                tc::l2_prefetch_line(w.cp_s + ((size_t)(b + 1) * DK + idx) * dv + i0);
        }
        for (int idx = tid; idx < DK * kScanCols; idx += Cfg::kThreads) {
            const int k = idx / kScanCols, c = idx - k * kScanCols;
            X2[((k >> 1) * kScanCols + c) * 2 + (k & 1)] = w.cp_s[((size_t)b * DK + k) * dv + i0 + c];
        }
        // X*(j) at this thread's outputs, read one step ahead
        auto load_xs = [&](int j, float2 *xs) {
            const float *src = w.cp_s + (size_t)(b + j) * DK * dv + i0 + 2 * cg;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                xs[q] = *reinterpret_cast<const float2 *>(src + (size_t)(g + Cfg::kRowGroups * q) * dv);
        };
        float2 xs[4], xs_next[4];
        if (NS - 2 >= 1) {
            load_xm<DK>(scan_smem, w.cp_m + (size_t)(b + 1) * DK * DK, tid);
            if (kz == 0) load_xs(1, xs);
        }
        for (int j = 1; j <= NS - 2; ++j) {
            const float *XM = scan_smem + ((j - 1) & 1) * Cfg::kBufFloats;
            float *XS = w.cp_s + (size_t)(b + j) * DK * dv;
            if (kz == 0 && j + 1 <= NS - 2) load_xs(j + 1, xs_next);
            // the other buffer was last read in step j - 1, which every thread has left
            if (j + 1 <= NS - 2) {
                load_xm<DK>(scan_smem + (j & 1) * Cfg::kBufFloats, w.cp_m + (size_t)(b + j + 1) * DK * DK, tid);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();                         // X_M(j) and X_start(j) are in shared memory
            uint64_t acc[4][2];                      // [row q][column c]: (sum over even k, sum over odd k)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = 0ull;
#pragma unroll
            for (int k = kz * kQ; k < (kz + 1) * kQ; k += 4) {
                ulonglong2 a[4];                     // (X_M[r][k], X_M[r][k+1]), (X_M[r][k+2], X_M[r][k+3])
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    a[q] = *reinterpret_cast<const ulonglong2 *>(XM + (g + Cfg::kRowGroups * q) * Cfg::kPitch + k);
                ulonglong2 x[2];                     // [k pair]: (X[k][c], X[k+1][c]), (X[k][c+1], X[k+1][c+1])
#pragma unroll
                for (int kp = 0; kp < 2; ++kp)
                    x[kp] = *reinterpret_cast<const ulonglong2 *>(X2 + (((k >> 1) + kp) * kScanCols + 2 * cg) * 2);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    fma2(acc[q][0], a[q].x, x[0].x);
                    fma2(acc[q][1], a[q].x, x[0].y);
                    fma2(acc[q][0], a[q].y, x[1].x);
                    fma2(acc[q][1], a[q].y, x[1].y);
                }
            }
            float v[8];                              // this quarter's sums, [q][c]
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float e0, o0, e1, o1;
                unpack2(acc[q][0], e0, o0);
                unpack2(acc[q][1], e1, o1);
                v[2 * q] = e0 + o0;
                v[2 * q + 1] = e1 + o1;
            }
            if (kz > 0) {
                float4 *dst = reinterpret_cast<float4 *>(red + ((kz - 1) * Cfg::kTile + tt) * 8);
                dst[0] = make_float4(v[0], v[1], v[2], v[3]);
                dst[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
            __syncthreads();                         // every read of X_start(j); the partial sums are stored
            if (kz == 0) {
#pragma unroll
                for (int z = 0; z < Cfg::kSplit - 1; ++z) {
                    const float4 *src = reinterpret_cast<const float4 *>(red + (z * Cfg::kTile + tt) * 8);
                    const float4 p0 = src[0], p1 = src[1];
                    v[0] += p0.x; v[1] += p0.y; v[2] += p0.z; v[3] += p0.w;
                    v[4] += p1.x; v[5] += p1.y; v[6] += p1.z; v[7] += p1.w;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = g + Cfg::kRowGroups * q;
                    const float2 o = make_float2(v[2 * q] + xs[q].x, v[2 * q + 1] + xs[q].y);
                    float *x2 = X2 + ((r >> 1) * kScanCols + 2 * cg) * 2 + (r & 1);
                    x2[0] = o.x;
                    x2[2] = o.y;
                    *reinterpret_cast<float2 *>(XS + (size_t)r * dv + i0 + 2 * cg) = o;
                    xs[q] = xs_next[q];
                }
            }
            __syncthreads();                         // X_start(j + 1) is in place; the partial sums are read
        }
        __syncthreads();                             // the next unit rewrites X_start and buffer 0
    }
    cp_async_wait<0>();                              // no copy may still be landing when the CTA leaves
}

template <int DK>
cudaError_t launch_scan_dk(const Problem &p, const Workspace &w, cudaStream_t s) {
    constexpr size_t smem = ScanCfg<DK>::kSmem;
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
    e = launch_dependent(scan_kernel<DK>, dim3(gx, col_blocks), dim3(ScanCfg<DK>::kThreads), smem, s, p, w);
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
