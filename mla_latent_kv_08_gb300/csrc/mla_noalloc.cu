// Decode without caller-provided scratch: mla_decode_noalloc.
//
// Some callers cannot allocate device memory when they call decode. An
// inference-engine plugin whose enqueue step is forbidden to allocate is one;
// a serving process whose memory pool has already claimed the device's memory
// is another. cudaMalloc can block, can synchronise the device, and fails once
// the pool holds everything, so these callers need a decode that brings its
// own scratch. This file keeps that scratch in a fixed, file-scope device
// array that lives as long as the library is loaded, on every GPU that loads
// it, and routes the call through the ordinary decode path with that array as
// its workspace.
#include "mla_internal.cuh"

#include <mutex>

namespace mla {

// Fixed scratch of MLA_NOALLOC_SCRATCH_BYTES (32 MiB) per device.
constexpr size_t kNoallocScratchBytes = (size_t)32 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device. In host code the
// array's name is only a stand-in, so the address is looked up with the device
// current. The lookup is repeated on every call made outside stream capture
// (cheap once the module is loaded, and it follows a module reload after
// cudaDeviceReset); a call made while `stream` is capturing uses the address
// cached by the last call outside capture, so the first call on a device must
// come before any capture.
static mla_status noalloc_scratch(cudaStream_t stream, void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return MLA_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    } else if (!g_noalloc_ptr[dev]) {
        return MLA_ERR_CUDA;           // no address looked up on this device before capture
    }
    *out = g_noalloc_ptr[dev];
    return MLA_OK;
}

}  // namespace mla

extern "C" mla_status mla_decode_noalloc(const mla_shape *shape, const mla_cache *cache,
                                         const int32_t *block_table, int32_t max_blocks_per_seq,
                                         const int32_t *seq_lens, int32_t B, const void *q, const void *W_UV,
                                         const float *R, float scale, void *out, float *lse, int32_t *status,
                                         void *stream) {
    using namespace mla;
    if (!shape || B < 1) return MLA_ERR_INVALID;
    // The same shape and implementation checks as mla_decode, with its codes.
    const int32_t impl = mla_resolve_impl(shape, 1);
    if (impl < 0) return (mla_status)impl;
    // Pick the largest split target the fixed scratch can hold; the planner's
    // own choice (hint 0: one target per SM) is used when it fits.
    mla_shape s = *shape;
    if (mla_workspace_bytes(&s, B, 1) > kNoallocScratchBytes) {
        int lo = 1, hi = s.num_splits_hint > 0 ? s.num_splits_hint : 4096;
        s.num_splits_hint = 1;
        if (mla_workspace_bytes(&s, B, 1) > kNoallocScratchBytes) return MLA_ERR_WORKSPACE;
        while (lo < hi) {            // largest hint whose workspace fits
            const int mid = (lo + hi + 1) / 2;
            s.num_splits_hint = mid;
            if (mla_workspace_bytes(&s, B, 1) <= kNoallocScratchBytes) lo = mid; else hi = mid - 1;
        }
        s.num_splits_hint = lo;
    }
    void *scratch = nullptr;
    mla_status st = noalloc_scratch((cudaStream_t)stream, &scratch);
    if (st != MLA_OK) return st;
    st = mla_decode(&s, cache, block_table, max_blocks_per_seq, seq_lens, B, q, W_UV, R, scale, out, lse,
                    scratch, kNoallocScratchBytes, stream);
    if (st != MLA_OK) return st;
    // The flags word sits at offset 0 of the workspace; hand it to the caller.
    if (status && cudaMemcpyAsync(status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                  (cudaStream_t)stream) != cudaSuccess)
        return MLA_ERR_CUDA;
    return MLA_OK;
}
