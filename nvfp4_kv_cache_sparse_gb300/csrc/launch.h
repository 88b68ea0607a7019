// launch.h -- host-side launchers shared between the kernel translation units and the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace nvfp4mla {

// The fused producer stage ahead of the quantizer (nvfp4_mla_norm_rope_quantize_append).
struct ProducerArgs {
    const uint16_t* norm_weight;   // bf16 [512]
    float eps;
    const int64_t* positions;      // [num_tokens]
    const float* cos_table;        // fp32 [num_positions, 32]
    const float* sin_table;
    int64_t num_positions;
    int rotate_half;               // 1: pairs (f, f + 32); 0: pairs (2f, 2f + 1)
};

cudaError_t launch_quantize_append(const void* kv_latent, int64_t latent_row_stride, const void* k_rope,
                                   int64_t rope_row_stride, const int64_t* slot_mapping, int64_t num_tokens,
                                   uint8_t* cache, int64_t num_slots, int record_bytes, bool block_scales,
                                   uint32_t* dev_status, int sm_count, cudaStream_t stream,
                                   const ProducerArgs* producer = nullptr);

struct DecodeArgs {
    const void* q;             // bf16 [rows, h_q, 576]
    const uint8_t* cache;      // [num_slots, record_bytes]
    int64_t num_slots;
    int record_bytes;          // 352 or 432
    bool block_scales;         // 352 only: scales in block order instead of the permuted placement
    const int32_t* indices;    // [rows, topk]
    int rows;                  // batch * s_q
    int h_q;
    int topk;
    float sm_scale;
    const float* attn_sink;    // nullable [h_q]
    void* out;                 // bf16 [rows, h_q, 512]
    float* lse;                // [rows, h_q]
    int splits;
    uint16_t* part_out;        // f16 [rows, splits, h_q, 512] when splits > 1 (O / l of each split)
    float* part_lse;           // fp32 [rows, splits, h_q], log2 domain
    uint32_t* dev_status;
};

// The host-side checks of a decode call, in the order the entry points apply them: shape and
// record width, pointers and alignment (skipped when there are no rows), then a usable sm_103
// device. Sets rows (batch x s_q) and sms (0 unless every check passed).
int check_decode_call(const void* q, const uint8_t* cache, int64_t num_slots, int32_t record_bytes,
                      const int32_t* indices, int32_t batch, int32_t s_q, int32_t h_q, int32_t topk,
                      const float* attn_sink, const void* out, const float* lse, int32_t num_splits, int64_t* rows,
                      int* sms);

// Keys of one split, rounded to whole tiles.
int decode_keys_per_split(int topk, int splits);
cudaError_t launch_sparse_decode(const DecodeArgs& a, cudaStream_t stream);

// The CTA-pair decode with shared MMAs (sparse_decode_pair.cu): 128 heads, 352- or 432-byte records.
bool decode_pair_supported(const DecodeArgs& a);
int decode_pair_keys_per_split(int topk, int splits);
// Whether a decode of these arguments merges its splits inside the decode grid (2-4 splits per
// row in one cluster, the whole grid resident at once).
bool decode_pair_merges(const DecodeArgs& a);
// merged: set when the grid merges the splits itself (2-4 splits per row in one cluster).
cudaError_t launch_decode_pair(const DecodeArgs& a, cudaStream_t stream, bool* merged);
// The transposed-score decode for 64 heads on one SM (sparse_decode_h64.cu): 352- or 432-byte
// records.
bool decode_h64_supported(const DecodeArgs& a);
int decode_h64_keys_per_split(int topk, int splits);
cudaError_t launch_decode_h64(const DecodeArgs& a, cudaStream_t stream);
// The split merge (out, lse from the f16 partials), launched as a programmatic dependent.
cudaError_t launch_split_merge(const DecodeArgs& a, cudaStream_t stream);
// One time-bounded mbarrier wait that runs out (see nvfp4_mla_selftest_wait_timeout).
cudaError_t launch_wait_timeout_probe(uint32_t* status, uint64_t* elapsed_ns, cudaStream_t stream);

}  // namespace nvfp4mla
