// tcgen05 fused chunk kernel for fp32 inputs (kind::tf32): steps two to four of
// the four-step paragraph of the FlashQLA talk "Qwen系列模型线性注意力高性能优化实践"
// with the state in tensor memory, for head sizes dk, dv in {32, 64, 128}.
//
// The orientation is the transposed one of the bf16 kernel: the state's value
// index i runs along the 128 TMEM lanes (rows past dv, or past dk for a
// correction matrix, stay zero), so every MMA has M = 128.  Per chunk, with S
// the state at chunk start (dv x dk, fp32 in TMEM), G the chunk-local gate
// cumsum, gamma = exp(G), Gamma_rm = exp(G_r - G_m) (every exponent <= 0) and
// T = Gamma ⊙ T' (Gamma-extraction paragraph), element by element:
//
//   MMA P   [P_K | P_Q] = S [K;Q]^T        A = S itself (fp32 in TMEM, read as tf32)
//   MMA QK  Q K^T                          A = [K;Q] tile, lanes 64-127 kept
//   E1      V'^T = (V - D_gamma P_K)^T diag(beta)      (forward merge: V - S first)
//           S <- gamma_C S;  Mq = Gamma ⊙ tril(Q K^T)
//   MMA U   U^T  = V'^T T^T
//   E2      U^T into the A tile
//   MMA O   O2   = U^T Mq^T
//   MMA S   S   += U^T (D_dec K),  dec_r = gamma_C / gamma_r
//   E3      o    = scale (gamma_r P_Q + O2)
//
// Operands are staged by the CTA's threads as 128-byte-swizzled K-major tiles
// (fp32, 32 elements per 128-byte row segment), one MMA K-step being eight
// elements.  Chunk rows past the chunk's length are zero in K, Q and V and
// have beta = 0, so ragged chunks need no other masking.  Persistent CTAs pull
// work items (a unit or a segment of one, with look-back, correction or scan
// starts) from a counter, as the CUDA-core kernel does.  Every wait on an MMA
// is bounded: on timeout the kernel records GDN_ERR_TIMEOUT, frees its tensor
// memory and returns.
#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {

using namespace tc;

namespace {

constexpr int kT32Threads = 512;  // warps w, w + 4, w + 8, w + 12 share TMEM lane quadrant w, a quarter of the columns each
constexpr uint64_t kT32TimeoutNs = 2000000000ull;

// shared memory (offsets from a 1024-byte aligned base): [K/32 blocks][rows][128 B]
constexpr uint32_t kOffKQ = 0;          // [4][128: K rows 0-63 | Q rows 64-127]   64 KB
constexpr uint32_t kBlk128 = 16384;     // block stride of a 128-row tile
constexpr uint32_t kOffKT = 65536;      // [2][dk rows j][r]: dec_r K[r][j]       32 KB
constexpr uint32_t kOffTT = 98304;      // [2][64 rows n][m]: T                    16 KB
constexpr uint32_t kOffMQ = 114688;     // [2][64 rows r][m]: Gamma ⊙ tril(Q K^T)  16 KB
constexpr uint32_t kBlk64 = 8192;       // block stride of a 64-row tile
constexpr uint32_t kOffAV = 131072;     // [2][128 rows i][r]: V'^T, then U^T      32 KB
constexpr uint32_t kOffSmallT = 163840;

// TMEM columns (512 allocated)
constexpr uint32_t kCS = 0;     // state, dk columns
constexpr uint32_t kCP = 128;   // P_K (64), then P_Q (64)
constexpr uint32_t kCQK = 256;  // [K K^T; Q K^T], lanes 64-127 used
constexpr uint32_t kCU = 320;   // U^T
constexpr uint32_t kCO = 384;   // U^T Mq^T

struct T32Small {
    float G[64], beta[64], gam[64], dec[64];
    uint64_t bar_p, bar_u, bar_s;
    uint32_t tmem_base;
    int item;
    int abort;
};

constexpr uint32_t kT32Smem = kOffSmallT + sizeof(T32Small) + 1024;

__device__ __forceinline__ uint32_t tile_off(uint32_t row, uint32_t k, uint32_t block) {
    return f32_tile_off(row, k, block);
}

__device__ __forceinline__ uint64_t kstep(uint64_t desc, int kk, uint32_t block) {
    return f32_desc_kstep(desc, kk, block);
}

__device__ __forceinline__ float4 ldg_f4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }

__global__ void __launch_bounds__(kT32Threads, 1)
    fused_tf32_kernel(const __grid_constant__ Problem p, const __grid_constant__ Workspace w, int pass) {
    grid_dependency_wait();
    extern __shared__ uint8_t t32_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(t32_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    T32Small *sm = reinterpret_cast<T32Small *>(smem + kOffSmallT);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int li = quad * 32 + lane;  // TMEM lane = state row i
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;

    if (warp == 0) {
        tmem_alloc(&sm->tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(&sm->bar_p, 1);
        mbar_init(&sm->bar_u, 1);
        mbar_init(&sm->bar_s, 1);
        sm->abort = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = sm->tmem_base;
    const uint32_t tl = tb + lane_addr;

    const int dk = p.dk, dv = p.dv, H = p.H;
    const float *qg = static_cast<const float *>(p.q);
    const float *kg = static_cast<const float *>(p.k);
    const float *vg = static_cast<const float *>(p.v);
    float *og = static_cast<float *>(p.o);
    const float *tpg = static_cast<const float *>(w.tprime);
    const int n_items = w.num_items[pass == 2 ? 0 : 1];
    const gdn_work_item *items = pass == 2 ? w.items2 : w.items1;
    int *counter = &w.counters[pass == 2 ? 0 : 1];
    const uint64_t dKQ = smem_desc_sw128(sb + kOffKQ, 16, 1024);
    const uint64_t dKT = smem_desc_sw128(sb + kOffKT, 16, 1024);
    const uint64_t dTT = smem_desc_sw128(sb + kOffTT, 16, 1024);
    const uint64_t dMQ = smem_desc_sw128(sb + kOffMQ, 16, 1024);
    const uint64_t dAV = smem_desc_sw128(sb + kOffAV, 16, 1024);
    const int dk4 = dk >> 2;
    uint32_t ph = 0;  // chunks run by this CTA: the parity of every barrier's next phase
    bool failed = false;

    for (;;) {
        if (tid == 0) sm->item = atomicAdd(counter, 1);
        __syncthreads();
        const int it_idx = sm->item;
        __syncthreads();
        if (it_idx >= n_items) {
            // the last CTA out re-arms the queue, so the pass can be relaunched alone
            if (tid == 0) finish_queue(counter, &w.counters[pass == 2 ? 4 : 5]);
            break;
        }
        const gdn_work_item it = items[it_idx];
        const int seq = it.seq, h = it.head, fl = it.flags;
        const bool ident = fl & GDN_ITEM_FROM_IDENTITY;
        const int R = ident ? dk : dv;  // state rows of this item
        const int4 si = w.seqinfo[seq];

        // start state: lane li, columns [32 part, 32 part + 32)
        for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int j = c0 + u;
                float x = 0.f;
                if (li < R && j < dk) {
                    if (fl & GDN_ITEM_FROM_INITIAL) {
                        if (p.s0) x = p.s0[(((size_t)seq * H + h) * dk + j) * dv + li];
                    } else if (ident) {
                        x = li == j ? 1.f : 0.f;
                    } else if (fl & GDN_ITEM_FROM_SLOT) {
                        x = w.cp_s[((size_t)it.slot * dk + j) * dv + li];
                    }
                }
                r[u] = __float_as_uint(x);
            }
            tmem_st32(tl + kCS + c0, r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        for (int c = it.c_start; c < it.c_end; ++c) {
            const int4 ci = w.chunks[si.z + c];
            const int t0 = ci.y, len = ci.z;
            const bool out = (fl & GDN_ITEM_OUTPUT) && c >= it.c_begin;
            if (tid < kChunk) {
                const int r = tid < len ? tid : len - 1;
                sm->G[tid] = w.G[(size_t)h * p.total_T + t0 + r];
                sm->beta[tid] = tid < len ? p.beta[(size_t)(t0 + tid) * H + h] : 0.f;
            }
            // K rows 0-63 and (output chunks) Q rows 64-127
            for (int idx = tid; idx < (out ? 2 : 1) * kChunk * dk4; idx += kT32Threads) {
                const int row = idx / dk4, c4 = idx - row * dk4, r = row & 63;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < len) x = ldg_f4((row < 64 ? kg : qg) + ((size_t)(t0 + r) * H + h) * dk + 4 * c4);
                sts_u4_stage(sb + kOffKQ + tile_off(row, 4 * c4, kBlk128), *reinterpret_cast<uint4 *>(&x));
            }
            __syncthreads();
            if (tid < kChunk) {
                sm->gam[tid] = expf(sm->G[tid]);
                sm->dec[tid] = expf(sm->G[len - 1] - sm->G[tid]);
            }
            __syncthreads();
            // decay-scaled K^T: row j, four chunk rows r per store (lanes take consecutive j)
            for (int idx = tid; idx < dk * (kChunk / 4); idx += kT32Threads) {
                const int r4 = idx / dk, j = idx - r4 * dk;
                float x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int r = 4 * r4 + u;
                    x[u] = r < len ? sm->dec[r] * __ldg(kg + ((size_t)(t0 + r) * H + h) * dk + j) : 0.f;
                }
                sts_u4_stage(sb + kOffKT + tile_off(j, 4 * r4, kBlk128),
                       make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                                  __float_as_uint(x[3])));
            }
            // T = Gamma ⊙ T' (rows past the chunk's length are not stored: zero)
            for (int idx = tid; idx < kChunk * 16; idx += kT32Threads) {
                const int n = idx >> 4, m4 = (idx & 15) * 4;
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                if (n < len && m4 <= n) {
                    const float4 t = ldg_f4(tpg + ((size_t)h * p.total_T + t0 + n) * kChunk + m4);
                    const float tv[4] = {t.x, t.y, t.z, t.w};
                    const float Gn = sm->G[n];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (m4 + u <= n) x[u] = tv[u] * expf(Gn - sm->G[m4 + u]);
                }
                sts_u4_stage(sb + kOffTT + tile_off(n, m4, kBlk64),
                       make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                                  __float_as_uint(x[3])));
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (warp == 0) {
                if (elect_one()) {
                    tc_fence_after();
                    const uint32_t IP = out ? idesc_tf32_f32(128, 128) : idesc_tf32_f32(128, 64);
                    for (int kk = 0; kk < dk / 8; ++kk)
                        mma_ts_tf32(tb + kCP, tb + kCS + 8 * kk, kstep(dKQ, kk, kBlk128), IP, kk > 0);
                    if (out) {
                        constexpr uint32_t IQ = idesc_tf32_f32(128, 64);
                        for (int kk = 0; kk < dk / 8; ++kk)
                            mma_ss_tf32(tb + kCQK, kstep(dKQ, kk, kBlk128), kstep(dKQ, kk, kBlk128), IQ, kk > 0);
                    }
                    tc_commit(&sm->bar_p);
                }
                __syncwarp();
            }
            // the values this thread combines with P_K, fetched while the MMAs run
            float vv[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int r = 16 * part + u;
                vv[u] = (!ident && li < dv && r < len) ? vg[((size_t)(t0 + r) * H + h) * dv + li] : 0.f;
            }
            bool ok = mbar_wait(&sm->bar_p, ph & 1u, &sm->abort, kT32TimeoutNs);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
            {
                // V'^T row li, chunk rows [16 part, 16 part + 16)
                uint32_t pk[16];
                tmem_ld16(tl + kCP + 16 * part, pk);
                tmem_wait_ld();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t x[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int r = 16 * part + 4 * c4 + u;
                        x[u] = __float_as_uint(sm->beta[r] * (vv[4 * c4 + u] - sm->gam[r] * __uint_as_float(pk[4 * c4 + u])));
                    }
                    sts_u4_stage(sb + kOffAV + tile_off(li, 16 * part + 4 * c4, kBlk128), make_uint4(x[0], x[1], x[2], x[3]));
                }
            }
            {
                // S <- gamma_C S (the MMAs that read S are complete)
                const float gC = sm->gam[len - 1];
                for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
                    uint32_t s[32];
                    tmem_ld32(tl + kCS + c0, s);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 32; ++u) s[u] = __float_as_uint(gC * __uint_as_float(s[u]));
                    tmem_st32(tl + kCS + c0, s);
                }
                tmem_wait_st();
            }
            if (out && quad >= 2) {
                // Mq row r = li - 64: Gamma ⊙ tril(Q K^T), columns [16 part, 16 part + 16)
                uint32_t qk[16];
                tmem_ld16(tl + kCQK + 16 * part, qk);
                tmem_wait_ld();
                const int r = li - 64;
                const float Gr = sm->G[r];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t x[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int m = 16 * part + 4 * c4 + u;
                        x[u] = __float_as_uint((r < len && m <= r) ? __uint_as_float(qk[4 * c4 + u]) * expf(Gr - sm->G[m])
                                                                   : 0.f);
                    }
                    sts_u4_stage(sb + kOffMQ + tile_off(r, 16 * part + 4 * c4, kBlk64), make_uint4(x[0], x[1], x[2], x[3]));
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (warp == 0) {
                if (elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t IU = idesc_tf32_f32(128, 64);
                    for (int kk = 0; kk < kChunk / 8; ++kk)
                        mma_ss_tf32(tb + kCU, kstep(dAV, kk, kBlk128), kstep(dTT, kk, kBlk64), IU, kk > 0);
                    tc_commit(&sm->bar_u);
                }
                __syncwarp();
            }
            ok = mbar_wait(&sm->bar_u, ph & 1u, &sm->abort, kT32TimeoutNs);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
            {
                // U^T row li into the A tile (the MMA that read V'^T is complete)
                uint32_t u32[16];
                tmem_ld16(tl + kCU + 16 * part, u32);
                tmem_wait_ld();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    sts_u4_stage(sb + kOffAV + tile_off(li, 16 * part + 4 * c4, kBlk128),
                           make_uint4(u32[4 * c4], u32[4 * c4 + 1], u32[4 * c4 + 2], u32[4 * c4 + 3]));
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (warp == 0) {
                if (elect_one()) {
                    tc_fence_after();
                    if (out) {
                        constexpr uint32_t IO = idesc_tf32_f32(128, 64);
                        for (int kk = 0; kk < kChunk / 8; ++kk)
                            mma_ss_tf32(tb + kCO, kstep(dAV, kk, kBlk128), kstep(dMQ, kk, kBlk64), IO, kk > 0);
                    }
                    const uint32_t IS = idesc_tf32_f32(128, dk);
                    for (int kk = 0; kk < kChunk / 8; ++kk)
                        mma_ss_tf32(tb + kCS, kstep(dAV, kk, kBlk128), kstep(dKT, kk, kBlk128), IS, 1);
                    tc_commit(&sm->bar_s);
                }
                __syncwarp();
            }
            ok = mbar_wait(&sm->bar_s, ph & 1u, &sm->abort, kT32TimeoutNs);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
            ++ph;
            if (out) {
                uint32_t pq[16], o2[16];
                tmem_ld16(tl + kCP + 64 + 16 * part, pq);
                tmem_ld16(tl + kCO + 16 * part, o2);
                tmem_wait_ld();
                if (li < dv) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int r = 16 * part + u;
                        if (r < len)
                            og[((size_t)(t0 + r) * H + h) * dv + li] =
                                p.scale * fmaf(sm->gam[r], __uint_as_float(pq[u]), __uint_as_float(o2[u]));
                    }
                }
            }
            tc_fence_before();
            __syncthreads();  // tiles and coefficients are rewritten by the next chunk
            tc_fence_after();
        }
        if (failed) break;
        // end state
        for (int c0 = 32 * part; c0 < 32 * part + 32 && c0 < dk; c0 += 32) {
            uint32_t s[32];
            tmem_ld32(tl + kCS + c0, s);
            tmem_wait_ld();
            if (li < R) {
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int j = c0 + u;
                    if (j >= dk) break;
                    const float x = __uint_as_float(s[u]);
                    if (fl & GDN_ITEM_WRITE_FINAL) p.sf[(((size_t)seq * H + h) * dk + j) * dv + li] = x;
                    if (fl & GDN_ITEM_WRITE_SLOT) w.cp_s[((size_t)it.slot * dk + j) * dv + li] = x;
                    if (fl & GDN_ITEM_WRITE_M) w.cp_m[((size_t)it.slot * dk + j) * dk + li] = x;
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (failed && tid == 0) {
        report_error(w.err, GDN_ERR_TIMEOUT);
        sm->abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

}  // namespace

bool fused_tf32_supported(int dtype, int dk, int dv) {
    auto ok = [](int d) { return d == 32 || d == 64 || d == 128; };
    return dtype == GDN_F32 && ok(dk) && ok(dv);
}

cudaError_t launch_fused_tf32(const Problem &p, const Workspace &w, int pass, int grid, cudaStream_t s) {
    if (!fused_tf32_supported(p.dtype, p.dk, p.dv)) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(fused_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kT32Smem);
    if (e != cudaSuccess) return e;
    e = launch_dependent(fused_tf32_kernel, dim3(grid), dim3(kT32Threads), (size_t)kT32Smem, s, p, w, pass);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn
