// decode_no_alloc.cu -- nvfp4_sparse_mla_decode_no_alloc: the sparse MLA decode for callers
// that cannot provide device scratch memory.
//
// nvfp4_sparse_mla_decode needs a caller-owned workspace whenever it splits each top-k list
// into several parts (the fp32 partial outputs and log-sum-exps of the parts). Some callers
// cannot hand one over: code that runs with a device-memory budget fixed at start-up and may
// not call cudaMalloc afterwards, code that must not call cudaFree/cudaMalloc because those
// can synchronize the whole device, or a host program that only lends the library its
// input and output buffers. This entry point takes the same inputs and outputs but keeps its
// scratch in one fixed-size array of device memory that belongs to the library itself.
//
// Limits and sharing (also stated in include/nvfp4_mla.h):
//  * The array holds NVFP4_MLA_NO_ALLOC_SCRATCH_BYTES = 32 MiB. Every GPU that loads the library keeps it
//    reserved until the process exits. A problem whose split count needs more returns
//    NVFP4_MLA_ERR_WORKSPACE and launches nothing.
//  * All calls share the array and it keeps what the last call wrote. Nothing in it has to
//    start at zero: each call writes every partial value it later reads. Two calls whose
//    kernels overlap on the GPU (different streams, no ordering) race on it.
//  * The host cannot use the array's name as a device address. A call outside stream capture
//    asks the runtime for it (cudaGetSymbolAddress, with the device current) and keeps it for
//    the device; a call under capture uses the one kept, so make one call before any capture,
//    and again after a device or primary-context reset (cudaDeviceReset), which may move the array.
//  * Every host-side check of the workspace entry point runs first, so a call with a bad
//    argument returns the same status as that entry point and asks the runtime for nothing.
//  * No cudaMalloc, cudaFree or allocating library routine is called.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/nvfp4_mla.h"
#include "launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = NVFP4_MLA_NO_ALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device: looked up again on every call outside
// stream capture, the kept one under capture. A failed runtime call leaves no error pending.
int scratch_address(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return NVFP4_MLA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return NVFP4_MLA_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) {
        (void)cudaGetLastError();
        return NVFP4_MLA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (capture == cudaStreamCaptureStatusNone || g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return NVFP4_MLA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return NVFP4_MLA_OK;
}

}  // namespace

extern "C" NVFP4_MLA_API int nvfp4_sparse_mla_decode_no_alloc(
    const void* q, const uint8_t* cache, int64_t num_slots, int32_t record_bytes, const int32_t* indices,
    int32_t batch, int32_t s_q, int32_t h_q, int32_t topk, float sm_scale, const float* attn_sink, void* out,
    float* lse, int32_t num_splits, uint32_t* dev_status, void* stream) {
    int64_t rows = 0;
    int sms = 0;
    const int chk = nvfp4mla::check_decode_call(q, cache, num_slots, record_bytes, indices, batch, s_q, h_q, topk,
                                                attn_sink, out, lse, num_splits, &rows, &sms);
    if (chk != NVFP4_MLA_OK || rows == 0) return chk;
    size_t need = 0;
    const int st = nvfp4_sparse_mla_decode_workspace_size(batch, s_q, h_q, topk, record_bytes, num_splits, &need);
    if (st != NVFP4_MLA_OK) return st;
    if (need > kNoAllocScratchBytes) return NVFP4_MLA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        const int s = scratch_address(static_cast<cudaStream_t>(stream), &scratch);
        if (s != NVFP4_MLA_OK) return s;
    }
    return nvfp4_sparse_mla_decode(q, cache, num_slots, record_bytes, indices, batch, s_q, h_q, topk, sm_scale,
                                   attn_sink, out, lse, num_splits, scratch, need ? kNoAllocScratchBytes : 0,
                                   dev_status, stream);
}
