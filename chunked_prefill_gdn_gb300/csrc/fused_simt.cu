// CUDA-core fused chunk kernel: steps two to four of the four-step paragraph of
// the FlashQLA talk "Qwen系列模型线性注意力高性能优化实践" for any supported head
// size and input type.  It is the path for fp32 inputs and for head sizes the
// tcgen05 kernel does not take, and the GPU-side cross-check of that kernel.
//
// Per chunk (rows r of the chunk, S the state at chunk start, dv x dk):
//   T   = Gamma ⊙ T'                       (Gamma-extraction paragraph)
//   V'  = diag(beta) (V - D_gamma K S^T)    (forward-merge paragraph: V - S first)
//   U   = T V'
//   O   = scale (D_gamma Q S^T + (Gamma ⊙ tril(Q K^T)) U)
//   S  <- gamma_C S + U^T diag(gamma_C / gamma) K
// with Gamma_ri = exp(G_r - G_i) (every exponent <= 0).  W, U and the per-chunk
// states stay in shared memory.  Persistent CTAs pull work items (a unit or a
// segment of one, with look-back, correction or scan starts) from a counter.
#include "gdn_internal.cuh"

namespace gdn {

int fused_simt_smem_bytes(int dk, int dv) {
    const int R = dk > dv ? dk : dv;
    const int floats = R * (dk + 1) + 2 * kChunk * (dk + 1) + 2 * kChunk * (R + 1) + kChunk * 65 + 4 * kChunk;
    return floats * (int)sizeof(float);
}

__global__ void __launch_bounds__(256, 1) fused_simt_kernel(const __grid_constant__ Problem p, const __grid_constant__ Workspace w, int pass) {
    grid_dependency_wait();
    extern __shared__ float smem[];
    __shared__ int s_item;
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int dk = p.dk, dv = p.dv, H = p.H;
    const int Rmax = dk > dv ? dk : dv;
    const int ks = dk + 1, rs = Rmax + 1;
    float *S = smem;                      // [Rmax][dk+1]  math orientation S[i][j]
    float *Ks = S + Rmax * ks;            // [64][dk+1]
    float *Qs = Ks + kChunk * ks;         // [64][dk+1]
    float *Vs = Qs + kChunk * ks;         // [64][Rmax+1]  V, then V'
    float *Us = Vs + kChunk * rs;         // [64][Rmax+1]
    float *Tm = Us + kChunk * rs;         // [64][65]      T, then Gamma ⊙ tril(Q K^T)
    float *Gs = Tm + kChunk * 65;         // [64]
    float *bs = Gs + kChunk;              // [64]
    float *gam = bs + kChunk;             // [64]
    float *dec = gam + kChunk;            // [64]
    const int n_items = w.num_items[pass == 2 ? 0 : 1];
    const gdn_work_item *items = pass == 2 ? w.items2 : w.items1;
    int *counter = &w.counters[pass == 2 ? 0 : 1];

    for (;;) {
        if (tid == 0) s_item = atomicAdd(counter, 1);
        __syncthreads();
        const int it_idx = s_item;
        __syncthreads();
        if (it_idx >= n_items) {
            // the last CTA out re-arms the queue, so the pass can be relaunched alone
            if (tid == 0) finish_queue(counter, &w.counters[pass == 2 ? 4 : 5]);
            break;
        }
        const gdn_work_item it = items[it_idx];
        const int seq = it.seq, h = it.head, fl = it.flags;
        const bool ident = fl & GDN_ITEM_FROM_IDENTITY;
        const int R = ident ? dk : dv;          // state rows of this item
        const int4 si = w.seqinfo[seq];
        // start state
        for (int idx = tid; idx < R * dk; idx += nthr) {
            const int i = idx / dk, j = idx % dk;
            float x = 0.f;
            if (fl & GDN_ITEM_FROM_INITIAL) {
                if (p.s0) x = p.s0[(((size_t)seq * H + h) * dk + j) * dv + i];
            } else if (ident) {
                x = (i == j) ? 1.f : 0.f;
            } else if (fl & GDN_ITEM_FROM_SLOT) {
                x = w.cp_s[((size_t)it.slot * dk + j) * dv + i];
            }
            S[i * ks + j] = x;
        }
        __syncthreads();
        for (int c = it.c_start; c < it.c_end; ++c) {
            const int4 ci = w.chunks[si.z + c];
            const int t0 = ci.y, len = ci.z;
            const bool out = (fl & GDN_ITEM_OUTPUT) && c >= it.c_begin;
            for (int idx = tid; idx < kChunk * dk; idx += nthr) {
                const int r = idx / dk, j = idx % dk;
                const size_t g_idx = ((size_t)(t0 + r) * H + h) * dk + j;
                Ks[r * ks + j] = r < len ? load_elem(p.k, g_idx, p.dtype) : 0.f;
                if (out) Qs[r * ks + j] = r < len ? load_elem(p.q, g_idx, p.dtype) : 0.f;
            }
            for (int idx = tid; idx < kChunk * R; idx += nthr) {
                const int r = idx / R, i = idx % R;
                Vs[r * rs + i] = (r < len && !ident) ? load_elem(p.v, ((size_t)(t0 + r) * H + h) * dv + i, p.dtype) : 0.f;
            }
            if (tid < kChunk) {
                const int r = tid < len ? tid : len - 1;
                Gs[tid] = w.G[(size_t)h * p.total_T + t0 + r];
                bs[tid] = tid < len ? p.beta[(size_t)(t0 + tid) * H + h] : 0.f;
            }
            __syncthreads();
            if (tid < kChunk) {
                gam[tid] = expf(Gs[tid]);
                dec[tid] = expf(Gs[len - 1] - Gs[tid]);
            }
            for (int idx = tid; idx < kChunk * kChunk; idx += nthr) {
                const int r = idx / kChunk, m = idx % kChunk;
                float x = 0.f;
                if (r < len && m <= r) {
                    const size_t tp = ((size_t)h * p.total_T + t0 + r) * kChunk + m;
                    x = load_elem(w.tprime, tp, p.dtype) * expf(Gs[r] - Gs[m]);
                }
                Tm[r * 65 + m] = x;
            }
            __syncthreads();
            // V' = diag(beta) (V - D_gamma K S^T)
            for (int idx = tid; idx < kChunk * R; idx += nthr) {
                const int r = idx / R, i = idx % R;
                float a = 0.f;
                for (int j = 0; j < dk; ++j) a = fmaf(Ks[r * ks + j], S[i * ks + j], a);
                Vs[r * rs + i] = bs[r] * (Vs[r * rs + i] - gam[r] * a);
            }
            __syncthreads();
            // U = T V'
            for (int idx = tid; idx < kChunk * R; idx += nthr) {
                const int r = idx / R, i = idx % R;
                float a = 0.f;
                for (int m = 0; m <= r; ++m) a = fmaf(Tm[r * 65 + m], Vs[m * rs + i], a);
                Us[r * rs + i] = a;
            }
            __syncthreads();
            if (out) {
                for (int idx = tid; idx < kChunk * kChunk; idx += nthr) {
                    const int r = idx / kChunk, m = idx % kChunk;
                    float a = 0.f;
                    if (r < len && m <= r) {
                        for (int j = 0; j < dk; ++j) a = fmaf(Qs[r * ks + j], Ks[m * ks + j], a);
                        a *= expf(Gs[r] - Gs[m]);
                    }
                    Tm[r * 65 + m] = a;
                }
                __syncthreads();
                for (int idx = tid; idx < len * dv; idx += nthr) {
                    const int r = idx / dv, i = idx % dv;
                    float a = 0.f;
                    for (int j = 0; j < dk; ++j) a = fmaf(Qs[r * ks + j], S[i * ks + j], a);
                    float b = 0.f;
                    for (int m = 0; m <= r; ++m) b = fmaf(Tm[r * 65 + m], Us[m * rs + i], b);
                    store_elem(p.o, ((size_t)(t0 + r) * H + h) * dv + i, p.dtype, p.scale * (gam[r] * a + b));
                }
                __syncthreads();
            }
            // S <- gamma_C S + U^T diag(gamma_C / gamma) K
            const float gC = gam[len - 1];
            for (int idx = tid; idx < R * dk; idx += nthr) {
                const int i = idx / dk, j = idx % dk;
                float a = 0.f;
                for (int r = 0; r < len; ++r) a = fmaf(Us[r * rs + i] * dec[r], Ks[r * ks + j], a);
                S[i * ks + j] = fmaf(gC, S[i * ks + j], a);
            }
            __syncthreads();
        }
        // end state
        for (int idx = tid; idx < R * dk; idx += nthr) {
            const int i = idx / dk, j = idx % dk;
            const float x = S[i * ks + j];
            if (fl & GDN_ITEM_WRITE_FINAL) p.sf[(((size_t)seq * H + h) * dk + j) * dv + i] = x;
            if (fl & GDN_ITEM_WRITE_SLOT) w.cp_s[((size_t)it.slot * dk + j) * dv + i] = x;
            if (fl & GDN_ITEM_WRITE_M) w.cp_m[((size_t)it.slot * dk + j) * dk + i] = x;
        }
        __syncthreads();
    }
}

cudaError_t launch_fused_simt(const Problem &p, const Workspace &w, int pass, int grid, cudaStream_t s) {
    const int smem = fused_simt_smem_bytes(p.dk, p.dv);
    cudaError_t e = cudaFuncSetAttribute(fused_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_dependent(fused_simt_kernel, dim3(grid), dim3(256), (size_t)smem, s, p, w, pass);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn
