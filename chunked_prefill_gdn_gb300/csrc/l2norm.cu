// L2 normalisation of q and k rows over the head dimension, the step in front
// of the recurrence: the sliding-window paragraph of the FlashQLA talk
// "Qwen系列模型线性注意力高性能优化实践" relies on every key having unit L2 norm
// (that is what bounds I - beta k k^T), and models of this family apply the same
// normalisation to the queries.
//
//     x_hat = x * rsqrt(sum_d x_d^2 + eps)          (fp32 sum, one rounding to the
//                                                     output type)
//
// and its backward, for an upstream gradient dy of x_hat,
//
//     dx = dy * inv - x * (x . dy) * inv^3,      inv = rsqrt(sum_d x_d^2 + eps)
//
// (the Jacobian of x / n is I / n - x x^T / n^3), in fp32 with dy and dx fp32.
//
// Both passes are pure streams (one read, one write of each row), so they are
// written for HBM: one warp per row, four rows in flight per warp, vector
// loads of the lane's dk / 32 consecutive elements, the sum by shuffles, and a
// grid of eight 256-thread blocks per SM striding over the rows.
#include <cuda_bf16.h>

#include <algorithm>

#include "gdn_internal.cuh"

namespace gdn {

namespace {

constexpr int kNormWarps = 8;   // warps per block
constexpr int kNormRows = 4;    // rows in flight per warp

template <int E>
struct BfVec;
template <>
struct BfVec<1> {
    using T = unsigned short;
};
template <>
struct BfVec<2> {
    using T = uint32_t;
};
template <>
struct BfVec<4> {
    using T = uint2;
};
template <int E>
struct F32Vec;
template <>
struct F32Vec<1> {
    using T = float;
};
template <>
struct F32Vec<2> {
    using T = float2;
};
template <>
struct F32Vec<4> {
    using T = float4;
};

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf_pack(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// E consecutive elements of one row into fp32 registers, and back.
template <int E>
__device__ __forceinline__ void load_e(const __nv_bfloat16 *src, float *x) {
    const typename BfVec<E>::T v = *reinterpret_cast<const typename BfVec<E>::T *>(src);
    if constexpr (E == 1) {
        x[0] = __uint_as_float(static_cast<uint32_t>(v) << 16);
    } else if constexpr (E == 2) {
        x[0] = bf_lo(v);
        x[1] = bf_hi(v);
    } else {
        x[0] = bf_lo(v.x);
        x[1] = bf_hi(v.x);
        x[2] = bf_lo(v.y);
        x[3] = bf_hi(v.y);
    }
}
template <int E>
__device__ __forceinline__ void store_e(__nv_bfloat16 *dst, const float *x) {
    if constexpr (E == 1) {
        *reinterpret_cast<__nv_bfloat16 *>(dst) = __float2bfloat16_rn(x[0]);
    } else if constexpr (E == 2) {
        *reinterpret_cast<uint32_t *>(dst) = bf_pack(x[0], x[1]);
    } else {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(bf_pack(x[0], x[1]), bf_pack(x[2], x[3]));
    }
}
template <int E>
__device__ __forceinline__ void load_e(const float *src, float *x) {
    const typename F32Vec<E>::T v = *reinterpret_cast<const typename F32Vec<E>::T *>(src);
    if constexpr (E == 1) {
        x[0] = v;
    } else if constexpr (E == 2) {
        x[0] = v.x;
        x[1] = v.y;
    } else {
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
    }
}
template <int E>
__device__ __forceinline__ void store_e(float *dst, const float *x) {
    if constexpr (E == 1) {
        *dst = x[0];
    } else if constexpr (E == 2) {
        *reinterpret_cast<float2 *>(dst) = make_float2(x[0], x[1]);
    } else {
        *reinterpret_cast<float4 *>(dst) = make_float4(x[0], x[1], x[2], x[3]);
    }
}

// Rows [0, rows) are q, rows [rows, 2 rows) are k (a NULL tensor contributes
// no rows: its half of the index range is skipped).
template <typename T, int DK>
__global__ void __launch_bounds__(32 * kNormWarps, 8) qk_l2norm_kernel(const T *q, const T *k, T *qo, T *ko,
                                                                    long long rows, float eps) {
    constexpr int E = DK / 32;
    const int lane = threadIdx.x & 31;
    const long long warp0 = (long long)blockIdx.x * kNormWarps + (threadIdx.x >> 5);
    const long long stride = (long long)gridDim.x * kNormWarps * kNormRows;
    const long long total = 2 * rows;
    for (long long base = warp0 * kNormRows; base < total; base += stride) {
        float x[kNormRows][E];
        bool live[kNormRows];
#pragma unroll
        for (int u = 0; u < kNormRows; ++u) {
            const long long r = base + u;
            const bool is_k = r >= rows;
            const T *src = is_k ? k : q;
            live[u] = r < total && src != nullptr;
            if (live[u]) {
                load_e<E>(src + (is_k ? r - rows : r) * DK + lane * E, x[u]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) x[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kNormRows; ++u) {
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss = fmaf(x[u][e], x[u][e], ss);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrtf(ss + eps);
#pragma unroll
            for (int e = 0; e < E; ++e) x[u][e] *= inv;
        }
#pragma unroll
        for (int u = 0; u < kNormRows; ++u) {
            if (!live[u]) continue;
            const long long r = base + u;
            const bool is_k = r >= rows;
            store_e<E>((is_k ? ko : qo) + (is_k ? r - rows : r) * DK + lane * E, x[u]);
        }
    }
}

// dx rows from x (T) and dy (fp32); dx may alias dy.  Two rows of inputs per
// row in flight, so four blocks per SM (64 registers) instead of eight.
template <typename T, int DK>
__global__ void __launch_bounds__(32 * kNormWarps, 4) qk_l2norm_bwd_kernel(const T *x, const float *dy, float *dx,
                                                                        long long rows, float eps) {
    constexpr int E = DK / 32;
    const int lane = threadIdx.x & 31;
    const long long warp0 = (long long)blockIdx.x * kNormWarps + (threadIdx.x >> 5);
    const long long stride = (long long)gridDim.x * kNormWarps * kNormRows;
    for (long long base = warp0 * kNormRows; base < rows; base += stride) {
        float xv[kNormRows][E], gv[kNormRows][E];
#pragma unroll
        for (int u = 0; u < kNormRows; ++u) {
            const long long r = base + u;
            if (r < rows) {
                load_e<E>(x + r * DK + lane * E, xv[u]);
                load_e<E>(dy + r * DK + lane * E, gv[u]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) xv[u][e] = gv[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kNormRows; ++u) {
            float ss = 0.f, xd = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ss = fmaf(xv[u][e], xv[u][e], ss);
                xd = fmaf(xv[u][e], gv[u][e], xd);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                ss += __shfl_xor_sync(0xffffffffu, ss, off);
                xd += __shfl_xor_sync(0xffffffffu, xd, off);
            }
            const float inv = rsqrtf(ss + eps);
            const float c = xd * inv * inv * inv;
#pragma unroll
            for (int e = 0; e < E; ++e) gv[u][e] = gv[u][e] * inv - xv[u][e] * c;
        }
#pragma unroll
        for (int u = 0; u < kNormRows; ++u) {
            const long long r = base + u;
            if (r < rows) store_e<E>(dx + r * DK + lane * E, gv[u]);
        }
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

template <typename T>
cudaError_t launch_typed(const void *q, const void *k, void *qo, void *ko, long long rows, int dk, float eps,
                         cudaStream_t s) {
    const int sms = sm_count();
    const long long warps_needed = (2 * rows + kNormRows - 1) / kNormRows;
    const long long blocks_needed = (warps_needed + kNormWarps - 1) / kNormWarps;
    const int grid = (int)std::min<long long>(blocks_needed, (long long)sms * 8);
    const T *qt = static_cast<const T *>(q);
    const T *kt = static_cast<const T *>(k);
    T *qot = static_cast<T *>(qo);
    T *kot = static_cast<T *>(ko);
    if (dk == 32) qk_l2norm_kernel<T, 32><<<grid, 32 * kNormWarps, 0, s>>>(qt, kt, qot, kot, rows, eps);
    else if (dk == 64) qk_l2norm_kernel<T, 64><<<grid, 32 * kNormWarps, 0, s>>>(qt, kt, qot, kot, rows, eps);
    else qk_l2norm_kernel<T, 128><<<grid, 32 * kNormWarps, 0, s>>>(qt, kt, qot, kot, rows, eps);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_typed(const void *x, const float *dy, float *dx, long long rows, int dk, float eps,
                             cudaStream_t s) {
    const int sms = sm_count();
    const long long warps_needed = (rows + kNormRows - 1) / kNormRows;
    const long long blocks_needed = (warps_needed + kNormWarps - 1) / kNormWarps;
    const int grid = (int)std::min<long long>(blocks_needed, (long long)sms * 4);
    const T *xt = static_cast<const T *>(x);
    if (dk == 32) qk_l2norm_bwd_kernel<T, 32><<<grid, 32 * kNormWarps, 0, s>>>(xt, dy, dx, rows, eps);
    else if (dk == 64) qk_l2norm_bwd_kernel<T, 64><<<grid, 32 * kNormWarps, 0, s>>>(xt, dy, dx, rows, eps);
    else qk_l2norm_bwd_kernel<T, 128><<<grid, 32 * kNormWarps, 0, s>>>(xt, dy, dx, rows, eps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_l2norm(const void *q, const void *k, void *qo, void *ko, long long rows, int dk, int dtype,
                             float eps, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    return dtype == GDN_BF16 ? launch_typed<__nv_bfloat16>(q, k, qo, ko, rows, dk, eps, s)
                             : launch_typed<float>(q, k, qo, ko, rows, dk, eps, s);
}

}  // namespace gdn

extern "C" gdn_status gdn_qk_l2norm(const void *q, const void *k, void *q_out, void *k_out, int64_t rows, int dk,
                                    gdn_dtype dtype, float eps, gdn_stream_t stream) {
    if (rows < 0 || (dk != 32 && dk != 64 && dk != 128)) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return GDN_ERR_INVALID_ARG;
    if ((q == nullptr) != (q_out == nullptr) || (k == nullptr) != (k_out == nullptr)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, q_out, k_out};
    for (const void *ptr : ptrs)
        if (ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u)) return GDN_ERR_INVALID_ARG;
    if (!(eps > 0.f)) eps = gdn::kQkNormEps;
    const cudaError_t e = gdn::launch_qk_l2norm(q, k, q_out, k_out, rows, dk, dtype, eps,
                                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        gdn::set_error_detail("launch qk_l2norm", e);
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

extern "C" gdn_status gdn_qk_l2norm_bwd(const void *x, const float *dy, float *dx, int64_t rows, int dk,
                                        gdn_dtype dtype, float eps, gdn_stream_t stream) {
    if (rows < 0 || (dk != 32 && dk != 64 && dk != 128)) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return GDN_ERR_INVALID_ARG;
    if (rows > 0 && (!x || !dy || !dx)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {x, dy, dx};
    for (const void *ptr : ptrs)
        if (ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u)) return GDN_ERR_INVALID_ARG;
    if (rows == 0) return GDN_OK;
    if (!(eps > 0.f)) eps = gdn::kQkNormEps;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == GDN_BF16 ? gdn::launch_bwd_typed<__nv_bfloat16>(x, dy, dx, rows, dk, eps, s)
                                            : gdn::launch_bwd_typed<float>(x, dy, dx, rows, dk, eps, s);
    if (e != cudaSuccess) {
        gdn::set_error_detail("launch qk_l2norm_bwd", e);
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}
