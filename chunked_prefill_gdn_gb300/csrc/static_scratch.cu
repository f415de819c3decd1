// gdn_chunk_fwd_static: the forward pass with its workspace in a fixed,
// file-scope device array instead of caller memory.
//
// Who needs it: a caller that must not allocate device memory while it runs —
// an inference server that reserves all of HBM for its own pool at start-up
// and forbids allocation on the request path (cudaMalloc synchronises the
// device and can fail once the pool holds the memory), or a plugin that is
// handed tensors by a host framework and has no allocator of its own.  Such a
// caller still owns the inputs and outputs; only the scratch (sequence tables,
// gate cumsum, T', work lists, segment buffers) comes from here.
//
// The array is a plain static __device__ allocation: every GPU that loads the
// library holds kStaticScratchBytes of it until the process exits, and every
// call on that GPU reuses the same bytes.
#include <mutex>
#include <stdio.h>

#include "gdn_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device.  In host code the array's
// name is only a host-side stand-in; the real address comes from the runtime.
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

gdn_status scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        gdn::set_error_detail("static scratch: cudaGetDevice", e);
        return GDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || !ptr) {
            gdn::set_error_detail("static scratch: cudaGetSymbolAddress", e);
            return GDN_ERR_CUDA;
        }
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_static(const void *q, const void *k, const void *v, const float *g,
                                           const float *beta, const float *initial_state,
                                           const int32_t *cu_seqlens, int n_seqs, float scale, int B, int T,
                                           int H, int dk, int dv, gdn_dtype dtype, void *o, float *final_state,
                                           int32_t *device_status, const gdn_options *opts,
                                           gdn_stream_t stream_in) {
    if (opts && opts->stages != 0) return GDN_ERR_INVALID_ARG;  // only the whole pass
    const int varlen = cu_seqlens != nullptr;
    gdn_workspace_layout lay;
    gdn_status st = gdn_workspace_query(B, T, H, dk, dv, n_seqs, varlen, dtype, opts, &lay);
    if (st != GDN_OK) return st;
    if (lay.total > kStaticScratchBytes) {
        char msg[160];
        snprintf(msg, sizeof(msg), "problem needs %zu bytes of scratch; the static scratch holds %zu", lay.total,
                 kStaticScratchBytes);
        gdn::set_error_text(msg);
        return GDN_ERR_WORKSPACE;
    }
    if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)) return GDN_ERR_INVALID_ARG;

    // First call on a device: look up the array's device address (no allocation).
    void *scratch = nullptr;
    if ((st = scratch_address(&scratch)) != GDN_OK) return st;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_in);
    char *base = static_cast<char *>(scratch);
    // The error word and the work-queue counters share the first 256-byte
    // block and must start at zero; the previous call left its values there.
    // (The sequence-prep kernel zeroes them too; clearing here keeps the
    // status copy below meaningful even when a launch is refused.)
    cudaGetLastError();
    cudaError_t e = cudaMemsetAsync(base + lay.error_word, 0, 256, stream);
    if (e != cudaSuccess) {
        gdn::set_error_detail("static scratch: clear header", e);
        return GDN_ERR_CUDA;
    }
    st = gdn_chunk_fwd(q, k, v, g, beta, initial_state, cu_seqlens, n_seqs, scale, B, T, H, dk, dv, dtype, o,
                       final_state, scratch, kStaticScratchBytes, opts, stream_in);
    if (st != GDN_OK) return st;
    if (device_status) {
        e = cudaMemcpyAsync(device_status, base + lay.error_word, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream);
        if (e != cudaSuccess) {
            gdn::set_error_detail("static scratch: copy status", e);
            return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    return gdn_chunk_fwd_check(base + lay.error_word, stream_in);
}
