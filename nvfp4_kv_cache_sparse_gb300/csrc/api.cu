// api.cu -- the C ABI (include/nvfp4_mla.h): host-side argument checks, the platform gate,
// the split choice, and the kernel launches. Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/nvfp4_mla.h"
#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 64;
constexpr int kDecodeTile = 64;

// Per-device cache of (arch ok, SM count); 0 = unknown.
std::atomic<int> g_dev_state[kMaxDevices];   // -1 unsupported, >0 SM count

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Platform gate: the kernels are built for sm_103a only. Returns the SM count (> 0) or a
// negative status.
int device_sm_count(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        *status = NVFP4_MLA_ERR_CUDA;
        return -1;
    }
    if (dev >= 0 && dev < kMaxDevices) {
        const int cached = g_dev_state[dev].load(std::memory_order_relaxed);
        if (cached > 0) return cached;
        if (cached < 0) {
            *status = NVFP4_MLA_ERR_UNSUPPORTED;
            return -1;
        }
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        *status = NVFP4_MLA_ERR_CUDA;
        return -1;
    }
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < kMaxDevices) g_dev_state[dev].store(ok ? sms : -1, std::memory_order_relaxed);
    if (!ok) {
        *status = NVFP4_MLA_ERR_UNSUPPORTED;
        return -1;
    }
    return sms;
}

// 352, 432, 656 (fp8), or 352 with its scales in block order (NVFP4_MLA_SCALES_BLOCK_ORDER)
bool record_ok(int32_t r) {
    return r == 352 || r == 432 || r == 656 || r == (352 | NVFP4_MLA_SCALES_BLOCK_ORDER);
}
int record_width(int32_t r) { return r & 0xFFFF; }
bool block_scales(int32_t r) { return (r & NVFP4_MLA_SCALES_BLOCK_ORDER) != 0; }

// One CTA per SM: aim for one full wave. The 64-head decode of NVFP4 records runs one CTA per
// (row, split), the other decodes two; the NVFP4 decodes take keys in tiles of 128, the fp8 one 64.
int auto_splits(int64_t rows, int32_t topk, int sm_count, int32_t h_q, int32_t record_bytes) {
    const int r = record_width(record_bytes);
    const bool nvfp4 = r == 352 || r == 432;
    const int64_t ctas_per_split = rows * (nvfp4 && h_q == 64 ? 1 : 2);
    const int tile = nvfp4 ? 2 * kDecodeTile : kDecodeTile;
    int64_t s = ctas_per_split >= sm_count ? 1 : sm_count / ctas_per_split;
    const int64_t max_by_keys = (topk + tile - 1) / tile;
    if (s > max_by_keys) s = max_by_keys;
    if (s > kMaxSplits) s = kMaxSplits;
    if (s < 1) s = 1;
    return static_cast<int>(s);
}

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Workspace (splits > 1): f16 partial outputs [rows, splits, h_q, 512], then the fp32 partial
// log2-sum-exps [rows, splits, h_q].
size_t workspace_for(int64_t rows, int32_t h_q, int splits) {
    if (splits <= 1) return 0;
    const size_t n = static_cast<size_t>(rows) * splits * h_q;
    return n * 512 * sizeof(uint16_t) + round256(n * sizeof(float));
}

int check_decode_shape(int32_t batch, int32_t s_q, int32_t h_q, int32_t topk, int32_t record_bytes,
                       int32_t num_splits) {
    if (batch < 0 || s_q < 0 || topk < 1 || num_splits < 0 || num_splits > kMaxSplits) return NVFP4_MLA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(batch) * s_q > (int64_t(1) << 31) / (2 * kMaxSplits)) return NVFP4_MLA_ERR_INVALID_ARG;
    if (!record_ok(record_bytes) || (h_q != 64 && h_q != 128)) return NVFP4_MLA_ERR_UNSUPPORTED;
    return NVFP4_MLA_OK;
}

}  // namespace

namespace nvfp4mla {

int check_decode_call(const void* q, const uint8_t* cache, int64_t num_slots, int32_t record_bytes,
                      const int32_t* indices, int32_t batch, int32_t s_q, int32_t h_q, int32_t topk,
                      const float* attn_sink, const void* out, const float* lse, int32_t num_splits, int64_t* rows,
                      int* sms) {
    *rows = 0;
    *sms = 0;
    const int st = check_decode_shape(batch, s_q, h_q, topk, record_bytes, num_splits);
    if (st != NVFP4_MLA_OK) return st;
    if (num_slots < 0) return NVFP4_MLA_ERR_INVALID_ARG;
    *rows = static_cast<int64_t>(batch) * s_q;
    if (*rows == 0) return NVFP4_MLA_OK;
    if (!q || !cache || !indices || !out || !lse) return NVFP4_MLA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(cache, 16) || !aligned(out, 16) || !aligned(indices, 4) || !aligned(lse, 4))
        return NVFP4_MLA_ERR_INVALID_ARG;
    if (attn_sink && !aligned(attn_sink, 4)) return NVFP4_MLA_ERR_INVALID_ARG;
    int status = NVFP4_MLA_OK;
    *sms = device_sm_count(&status);
    return *sms > 0 ? NVFP4_MLA_OK : status;
}

}  // namespace nvfp4mla

extern "C" {

NVFP4_MLA_API int nvfp4_mla_quantize_append(const void* kv_latent, int64_t latent_row_stride, const void* k_rope,
                                            int64_t rope_row_stride, const int64_t* slot_mapping,
                                            int64_t num_tokens, uint8_t* cache, int64_t num_slots,
                                            int32_t record_bytes, uint32_t* dev_status, void* stream) {
    if (!record_ok(record_bytes)) return NVFP4_MLA_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_slots < 0) return NVFP4_MLA_ERR_INVALID_ARG;
    if (num_tokens == 0) return NVFP4_MLA_OK;
    if (!kv_latent || !k_rope || !slot_mapping || !cache) return NVFP4_MLA_ERR_INVALID_ARG;
    if (!aligned(kv_latent, 16) || !aligned(k_rope, 16) || !aligned(cache, 16) || !aligned(slot_mapping, 8))
        return NVFP4_MLA_ERR_INVALID_ARG;
    if (latent_row_stride < 512 || latent_row_stride % 8 != 0) return NVFP4_MLA_ERR_INVALID_ARG;
    if (rope_row_stride < 64 || rope_row_stride % 8 != 0) return NVFP4_MLA_ERR_INVALID_ARG;
    int status = NVFP4_MLA_OK;
    const int sms = device_sm_count(&status);
    if (sms <= 0) return status;
    const cudaError_t e = nvfp4mla::launch_quantize_append(kv_latent, latent_row_stride, k_rope, rope_row_stride,
                                                           slot_mapping, num_tokens, cache, num_slots,
                                                           record_width(record_bytes), block_scales(record_bytes),
                                                           dev_status, sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_MLA_OK : NVFP4_MLA_ERR_CUDA;
}

NVFP4_MLA_API int nvfp4_mla_norm_rope_quantize_append(const void* kv_latent, int64_t latent_row_stride,
                                                      const void* norm_weight, float eps, const void* k_pe,
                                                      int64_t rope_row_stride, const int64_t* positions,
                                                      const float* cos_table, const float* sin_table,
                                                      int64_t num_positions, int32_t rotate_half,
                                                      const int64_t* slot_mapping, int64_t num_tokens,
                                                      uint8_t* cache, int64_t num_slots, int32_t record_bytes,
                                                      uint32_t* dev_status, void* stream) {
    if (!record_ok(record_bytes)) return NVFP4_MLA_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_slots < 0 || num_positions < 0 || !(eps >= 0.0f) || (rotate_half != 0 && rotate_half != 1))
        return NVFP4_MLA_ERR_INVALID_ARG;
    if (num_tokens == 0) return NVFP4_MLA_OK;
    if (!kv_latent || !k_pe || !slot_mapping || !cache || !norm_weight || !positions || !cos_table || !sin_table)
        return NVFP4_MLA_ERR_INVALID_ARG;
    if (!aligned(kv_latent, 16) || !aligned(k_pe, 16) || !aligned(cache, 16) || !aligned(slot_mapping, 8) ||
        !aligned(norm_weight, 16) || !aligned(positions, 8) || !aligned(cos_table, 8) || !aligned(sin_table, 8))
        return NVFP4_MLA_ERR_INVALID_ARG;
    if (latent_row_stride < 512 || latent_row_stride % 8 != 0) return NVFP4_MLA_ERR_INVALID_ARG;
    if (rope_row_stride < 64 || rope_row_stride % 8 != 0) return NVFP4_MLA_ERR_INVALID_ARG;
    int status = NVFP4_MLA_OK;
    const int sms = device_sm_count(&status);
    if (sms <= 0) return status;
    nvfp4mla::ProducerArgs pr;
    pr.norm_weight = static_cast<const uint16_t*>(norm_weight);
    pr.eps = eps;
    pr.positions = positions;
    pr.cos_table = cos_table;
    pr.sin_table = sin_table;
    pr.num_positions = num_positions;
    pr.rotate_half = rotate_half;
    const cudaError_t e = nvfp4mla::launch_quantize_append(kv_latent, latent_row_stride, k_pe, rope_row_stride,
                                                           slot_mapping, num_tokens, cache, num_slots,
                                                           record_width(record_bytes), block_scales(record_bytes),
                                                           dev_status, sms, static_cast<cudaStream_t>(stream), &pr);
    return e == cudaSuccess ? NVFP4_MLA_OK : NVFP4_MLA_ERR_CUDA;
}

NVFP4_MLA_API int nvfp4_sparse_mla_decode_workspace_size(int32_t batch, int32_t s_q, int32_t h_q, int32_t topk,
                                                         int32_t record_bytes, int32_t num_splits, size_t* bytes) {
    if (!bytes) return NVFP4_MLA_ERR_INVALID_ARG;
    const int st = check_decode_shape(batch, s_q, h_q, topk, record_bytes, num_splits);
    if (st != NVFP4_MLA_OK) return st;
    const int64_t rows = static_cast<int64_t>(batch) * s_q;
    int splits = num_splits;
    if (splits == 0) {
        int status = NVFP4_MLA_OK;
        const int sms = device_sm_count(&status);
        if (sms <= 0) return status;
        splits = auto_splits(rows, topk, sms, h_q, record_bytes);
    }
    *bytes = workspace_for(rows, h_q, splits);
    return NVFP4_MLA_OK;
}

NVFP4_MLA_API int nvfp4_sparse_mla_decode_plan(int32_t batch, int32_t s_q, int32_t h_q, int32_t topk,
                                               int32_t record_bytes, int32_t num_splits, int32_t* splits,
                                               int32_t* kernels) {
    if (!splits || !kernels) return NVFP4_MLA_ERR_INVALID_ARG;
    const int st = check_decode_shape(batch, s_q, h_q, topk, record_bytes, num_splits);
    if (st != NVFP4_MLA_OK) return st;
    const int64_t rows = static_cast<int64_t>(batch) * s_q;
    int status = NVFP4_MLA_OK;
    const int sms = device_sm_count(&status);
    if (sms <= 0) return status;
    const int sp = num_splits > 0 ? num_splits : auto_splits(rows, topk, sms, h_q, record_bytes);
    nvfp4mla::DecodeArgs d;
    d.record_bytes = record_width(record_bytes);
    d.block_scales = block_scales(record_bytes);
    d.rows = static_cast<int>(rows);
    d.h_q = h_q;
    d.topk = topk;
    d.splits = sp;
    *splits = sp;
    *kernels = rows == 0 ? 0 : (sp == 1 || nvfp4mla::decode_pair_merges(d)) ? 1 : 2;
    return NVFP4_MLA_OK;
}

NVFP4_MLA_API int nvfp4_sparse_mla_decode(const void* q, const uint8_t* cache, int64_t num_slots, int32_t record_bytes,
                                          const int32_t* indices, int32_t batch, int32_t s_q, int32_t h_q,
                                          int32_t topk, float sm_scale, const float* attn_sink, void* out, float* lse,
                                          int32_t num_splits, void* workspace, size_t workspace_bytes,
                                          uint32_t* dev_status, void* stream) {
    int64_t rows = 0;
    int sms = 0;
    const int st = nvfp4mla::check_decode_call(q, cache, num_slots, record_bytes, indices, batch, s_q, h_q, topk,
                                               attn_sink, out, lse, num_splits, &rows, &sms);
    if (st != NVFP4_MLA_OK || rows == 0) return st;
    const int splits = num_splits > 0 ? num_splits : auto_splits(rows, topk, sms, h_q, record_bytes);
    const size_t need = workspace_for(rows, h_q, splits);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256))) return NVFP4_MLA_ERR_WORKSPACE;

    nvfp4mla::DecodeArgs d;
    d.q = q;
    d.cache = cache;
    d.num_slots = num_slots;
    d.record_bytes = record_width(record_bytes);
    d.block_scales = block_scales(record_bytes);
    d.indices = indices;
    d.rows = static_cast<int>(rows);
    d.h_q = h_q;
    d.topk = topk;
    d.sm_scale = sm_scale;
    d.attn_sink = attn_sink;
    d.out = out;
    d.lse = lse;
    d.splits = splits;
    const size_t n_part = static_cast<size_t>(rows) * splits * h_q;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    d.part_out = need ? reinterpret_cast<uint16_t*>(ws) : nullptr;
    d.part_lse = need ? reinterpret_cast<float*>(ws + n_part * 512 * sizeof(uint16_t)) : nullptr;
    d.dev_status = dev_status;
    const cudaError_t e = nvfp4mla::launch_sparse_decode(d, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_MLA_OK : NVFP4_MLA_ERR_CUDA;
}

NVFP4_MLA_API int nvfp4_mla_selftest_wait_timeout(uint32_t* dev_status, uint64_t* elapsed_ns, void* stream) {
    if (!dev_status || !elapsed_ns || !aligned(elapsed_ns, 8)) return NVFP4_MLA_ERR_INVALID_ARG;
    int status = NVFP4_MLA_OK;
    if (device_sm_count(&status) <= 0) return status;
    const cudaError_t e =
        nvfp4mla::launch_wait_timeout_probe(dev_status, elapsed_ns, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_MLA_OK : NVFP4_MLA_ERR_CUDA;
}

NVFP4_MLA_API const char* nvfp4_mla_status_string(int status) {
    switch (status) {
        case NVFP4_MLA_OK: return "ok";
        case NVFP4_MLA_ERR_INVALID_ARG: return "invalid argument (null pointer, size, stride or alignment)";
        case NVFP4_MLA_ERR_UNSUPPORTED: return "unsupported (record width, head count, or device is not sm_103)";
        case NVFP4_MLA_ERR_CUDA: return "CUDA runtime error";
        case NVFP4_MLA_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        default: return "unknown status";
    }
}

NVFP4_MLA_API int nvfp4_mla_version(void) { return 100; }

}  // extern "C"
