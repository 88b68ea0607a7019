/*
 * nvfp4_mla.h -- C ABI of the NVFP4 MLA KV-cache library for GB300 (sm_103a).
 *
 * Two operations, as the pages state the problem:
 *
 *  1. nvfp4_mla_quantize_append: quantize each token's 512-dim MLA latent (NoPE) and 64-dim
 *     RoPE key into one self-describing record and scatter it to its cache slot.
 *     - 352-byte "nvfp4.fp8rope" record: FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for
 *       SM100 sparse decode", format block "nvfp4.fp8rope (352 B/token)": bytes [0,256) hold
 *       512 e2m1 values two per byte, [256,320) 64 unscaled e4m3 RoPE values, [320,352) 32
 *       e4m3 scales, one per 16 values, the scale of block s at byte 320 + 8*(s&3) + (s>>2).
 *     - 432-byte "nvfp4_ds_mla" record: vLLM PR 82 "kv: nvfp4_ds_mla - 4-bit NVFP4 KV cache for
 *       B12X sparse MLA (SM120)", Problem and Fix / Write side: 256 B e2m1 NoPE, 32 B e4m3
 *       scales in block order, 16 zero bytes, 128 B bf16 RoPE copied verbatim.
 *     - Scale rule (vLLM PR 82, Tests): scale = E4M3(group_amax / 6); values are rounded to
 *       the nearest e2m1 grid point after division by the decoded scale.
 *     - 656-byte fp8 record, the one the NVFP4 records are measured against (vLLM PR 82,
 *       Problem: "512 B fp8 NoPE + 16 B fp32 tile scales + 128 B BF16 RoPE"): bytes [0,512)
 *       e4m3 NoPE codes, [512,528) four little-endian fp32 scales (scale t covers NoPE values
 *       [128t, 128t+128)), [528,656) bf16 RoPE copied verbatim. The page gives no fp8 scale
 *       rule; this library uses scale = amax / 448 and code = e4m3(x / scale) (fp32 quotients;
 *       a zero tile stores scale 0), and the decode's keys are bf16(e4m3 * scale). The decode
 *       takes V in f16, so NoPE magnitudes must stay below 65536 (the append flags larger
 *       ones with NVFP4_MLA_DEV_FP8_RANGE and stores them anyway).
 *
 *  2. nvfp4_sparse_mla_decode: DeepSeek-style sparse MLA decode over one shared latent KV
 *     head: for each query row (b, i) and head h, the keys are the records its top-k index
 *     list selects (FlashMLA PR 18, "Kernel:" paragraph: keys dequantized to bf16, QK^T over
 *     576 = 512 NoPE + 64 RoPE dims, PV over the 512 NoPE dims, bf16 MMAs with fp32
 *     accumulation, attention sink and invalid indices per its validation list).
 *
 * Conventions shared by every call
 *  - All data pointers are DEVICE pointers unless stated; the caller owns every buffer.
 *    No call allocates device memory. The only device memory the library owns is the
 *    fixed scratch array of nvfp4_sparse_mla_decode_no_alloc (see there).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is enqueued on it
 *    and the call returns without synchronizing. Stream order is kept as usual: every kernel
 *    of the library is launched as a programmatic dependent of the preceding work on the
 *    stream, so its prologue (for the decode: barrier setup, tensor-memory allocation) may
 *    overlap the preceding kernel's tail, but it reads and writes no memory before that kernel
 *    has completed and its writes are visible. The append and decode kernels let the next
 *    kernel on the stream start its prologue early in the same way; the decode's split merge
 *    does not (a waiting successor would hold the SMs the merge runs on).
 *  - Every argument check runs on the host before any launch; a failed check returns a
 *    status below and launches nothing. Kernels never trap: problems found on the device
 *    are OR-ed into *dev_status (if non-NULL) as NVFP4_MLA_DEV_* bits, readable after the
 *    stream has been synchronized.
 *  - The library is built for sm_103a only; calls on any other device return
 *    NVFP4_MLA_ERR_UNSUPPORTED.
 */
#ifndef NVFP4_MLA_H_
#define NVFP4_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_MLA_API __attribute__((visibility("default")))

/* Return codes of every call. */
typedef enum {
    NVFP4_MLA_OK = 0,
    NVFP4_MLA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, stride or alignment      */
    NVFP4_MLA_ERR_UNSUPPORTED = 2,   /* record width, head count or device not supported */
    NVFP4_MLA_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute)   */
    NVFP4_MLA_ERR_WORKSPACE = 4      /* workspace missing, too small or misaligned        */
} nvfp4_mla_status;

/*
 * Record layout. Every call's `record_bytes` is 352, 432 or 656, or
 * (352 | NVFP4_MLA_SCALES_BLOCK_ORDER): a 352-byte record equal to "nvfp4.fp8rope" except that its
 * 32 scales are stored in block order, block s at byte 320 + s. No page defines that record; it
 * is the unpermuted side of the scale-layout comparison (FlashMLA PR 18, format block, credits
 * the permuted placement with 10-12% of decode latency). A cache is read with the value it was
 * written with; its rows are (record_bytes & 0xFFFF) bytes wide. Any other value returns
 * NVFP4_MLA_ERR_UNSUPPORTED.
 */
#define NVFP4_MLA_SCALES_BLOCK_ORDER 0x10000

/* Bits the kernels OR into *dev_status. */
#define NVFP4_MLA_DEV_SLOT_OUT_OF_RANGE 0x1u  /* quantize_append: slot >= num_slots (skipped) */
#define NVFP4_MLA_DEV_INDEX_OUT_OF_RANGE 0x2u /* decode: index >= num_slots (masked)          */
#define NVFP4_MLA_DEV_TIMEOUT 0x4u            /* decode: a pipeline wait gave up; out invalid */
#define NVFP4_MLA_DEV_FP8_RANGE 0x8u          /* quantize_append, 656 B: a NoPE |x| >= 65536  */
#define NVFP4_MLA_DEV_POSITION_OUT_OF_RANGE 0x10u /* norm_rope_quantize_append: position outside
                                                     [0, num_positions) (token skipped)         */

/*
 * Quantize-and-append (write side).
 *   kv_latent          bf16 [num_tokens, 512], row stride latent_row_stride ELEMENTS, inner
 *                      stride 1; base 16-byte aligned, latent_row_stride % 8 == 0.
 *   k_rope             bf16 [num_tokens, 64], its own row stride rope_row_stride ELEMENTS
 *                      (may differ from the latent's); base 16-byte aligned, stride % 8 == 0.
 *   slot_mapping       int64 [num_tokens]: record slot of each token. A negative slot skips
 *                      the token (padding); a slot >= num_slots is skipped and sets
 *                      NVFP4_MLA_DEV_SLOT_OUT_OF_RANGE. Slots should be distinct; if two tokens
 *                      share a slot, which record lands there is unspecified.
 *   cache              uint8 [num_slots, record_bytes & 0xFFFF], 16-byte aligned. Only the
 *                      slots named by slot_mapping are written; every other byte is untouched.
 *   record_bytes       352, 432 or 656, or 352 | NVFP4_MLA_SCALES_BLOCK_ORDER (see above).
 *   dev_status         nullable device uint32 (see NVFP4_MLA_DEV_*).
 * num_tokens == 0 is valid and launches nothing.
 */
NVFP4_MLA_API int nvfp4_mla_quantize_append(const void* kv_latent, int64_t latent_row_stride,
                                            const void* k_rope, int64_t rope_row_stride,
                                            const int64_t* slot_mapping, int64_t num_tokens,
                                            uint8_t* cache, int64_t num_slots, int32_t record_bytes,
                                            uint32_t* dev_status, void* stream);

/*
 * Fused producer: RMSNorm of the latent, rotary embedding of k_pe, quantize and append, in one
 * kernel. SGLang PR 38646 "[SM120] Add opt-in NVFP4 sparse-MLA KV cache format for
 * DeepSeek-V4", "Limitations": the NVFP4 path lacks the fused norm+rope+quantize+store kernel and
 * pays a bf16 intermediate plus a separate quantize kernel per layer; "Stores": the existing
 * fused store kernels emit only the fp8 layout. The pages fix none of the stages' parameters, so
 * they are arguments here:
 *   kv_latent          bf16 [num_tokens, 512] BEFORE the norm (layout as in quantize_append).
 *   norm_weight        bf16 [512], 16-byte aligned: y_i = norm_weight[i] * x_i /
 *                      sqrt(mean_j x_j^2 + eps).
 *   eps                the norm's epsilon (>= 0).
 *   k_pe               bf16 [num_tokens, 64] BEFORE the rotary embedding (layout as k_rope).
 *   positions          int64 [num_tokens], 8-byte aligned: each token's position p. A position
 *                      outside [0, num_positions) skips the token and sets
 *                      NVFP4_MLA_DEV_POSITION_OUT_OF_RANGE.
 *   cos_table,         fp32 [num_positions, 32] each, 8-byte aligned: cos and sin of frequency f
 *   sin_table          at position p. The pair (a, b) of frequency f becomes (a c - b s, b c + a s).
 *   rotate_half        1: the pair of frequency f is (k_pe[f], k_pe[f + 32]); 0: (k_pe[2f],
 *                      k_pe[2f + 1]) ("interleaved").
 *   slot_mapping, cache, num_slots, record_bytes, dev_status: as in quantize_append.
 * Both stages compute in fp32 and round each result once to bf16, the value an unfused path
 * stores in its bf16 intermediate; the records are then those quantize_append writes for these
 * bf16 values. A result within about 2^-19 (relative to its terms) of a bf16 rounding midpoint may
 * round to either neighbour. num_tokens == 0 is valid and launches nothing.
 */
NVFP4_MLA_API int nvfp4_mla_norm_rope_quantize_append(const void* kv_latent, int64_t latent_row_stride,
                                                      const void* norm_weight, float eps, const void* k_pe,
                                                      int64_t rope_row_stride, const int64_t* positions,
                                                      const float* cos_table, const float* sin_table,
                                                      int64_t num_positions, int32_t rotate_half,
                                                      const int64_t* slot_mapping, int64_t num_tokens,
                                                      uint8_t* cache, int64_t num_slots, int32_t record_bytes,
                                                      uint32_t* dev_status, void* stream);

/*
 * Scratch size of nvfp4_sparse_mla_decode for a problem (host-only, no CUDA call).
 *   num_splits: the top-k list of each query row is cut into num_splits consecutive parts
 *   computed in parallel and merged by a second kernel (launched as a programmatic dependent
 *   of the first on the same stream); 0 lets the library choose from the problem size and the
 *   SM count of the current device (then this call reads the device attribute). The workspace
 *   holds each part's normalized partial output (f16, [rows, parts, h_q, 512]) and fp32
 *   log-sum-exp; it is 0 bytes when a single part is used.
 * Returns NVFP4_MLA_OK and sets *bytes, or an error code for an invalid problem.
 */
NVFP4_MLA_API int nvfp4_sparse_mla_decode_workspace_size(int32_t batch, int32_t s_q, int32_t h_q,
                                                         int32_t topk, int32_t record_bytes,
                                                         int32_t num_splits, size_t* bytes);

/*
 * How a decode of this shape runs on the current device (no launch, no device memory): the split
 * count it uses (num_splits, or the library's choice when 0) and how many kernels one call
 * launches (1: the decode grid alone, which also merges its 2-4 splits per row when they share a
 * cluster; 2: decode grid + merge grid; 0: nothing to do). Errors as ..._workspace_size, plus
 * NVFP4_MLA_ERR_UNSUPPORTED without a usable sm_103 device. (A service of this library; the pages
 * have no counterpart.)
 */
NVFP4_MLA_API int nvfp4_sparse_mla_decode_plan(int32_t batch, int32_t s_q, int32_t h_q, int32_t topk,
                                               int32_t record_bytes, int32_t num_splits, int32_t* splits,
                                               int32_t* kernels);

/*
 * Sparse MLA decode (read side).
 *   q            bf16 [batch, s_q, h_q, 576], contiguous, 16-byte aligned. Dims [0,512) are
 *                the NoPE (latent) part, [512,576) the RoPE part.
 *   cache        uint8 [num_slots, record_bytes & 0xFFFF], 16-byte aligned, as written by
 *                nvfp4_mla_quantize_append with the same record_bytes.
 *   indices      int32 [batch, s_q, topk], contiguous: the cache slots each query row attends.
 *                An entry < 0 is masked (padding); an entry >= num_slots is masked and sets
 *                NVFP4_MLA_DEV_INDEX_OUT_OF_RANGE. Repeated entries count once per occurrence.
 *   h_q          64 or 128. topk >= 1 (any value; the tail tile is masked).
 *   sm_scale     softmax scale applied to q.k (e.g. 1/sqrt(576)).
 *   attn_sink    nullable fp32 [h_q]: per-head extra logit that enters the softmax
 *                denominator of `out` only (no value vector) and not `lse`.
 *   out          bf16 [batch, s_q, h_q, 512], contiguous, 16-byte aligned:
 *                out = sum_j e^{z_j} V_j / (sum_j e^{z_j} + e^{sink_h}), z_j = sm_scale q.K_j
 *   lse          fp32 [batch, s_q, h_q]: natural-log log-sum-exp of the z_j of the used
 *                entries (sink excluded). A row with no used entry gets out = 0, lse = -inf.
 *   num_splits   0 = library choice, else 1..64 (see ..._workspace_size).
 *   workspace    device scratch of at least the size ..._workspace_size reports for the same
 *                arguments, 256-byte aligned; may be NULL when that size is 0. Its contents
 *                need no initialization.
 *   dev_status   nullable device uint32 (see NVFP4_MLA_DEV_*).
 * Precision: dequantized NVFP4 keys are exact in f16 and enter both contractions as f16, with q
 * as f16 times a per-head power of two (the same products as bf16 q for every element within
 * 2^28 of its head's largest |q|; the bf16 RoPE of 432-byte records and its q part stay bf16);
 * fp8 keys are e4m3 * scale rounded in fp32 and then to bf16 (QK^T) or f16 (PV); the
 * contractions run on tcgen05 16-bit MMAs with fp32 accumulation (P enters PV as f16); softmax
 * in fp32; `out` is rounded to bf16 once, after the parts' f16 partial outputs (relative error
 * <= 2^-11 each) are merged in fp32 when the top-k list is split.
 */
NVFP4_MLA_API int nvfp4_sparse_mla_decode(const void* q, const uint8_t* cache, int64_t num_slots,
                                          int32_t record_bytes, const int32_t* indices,
                                          int32_t batch, int32_t s_q, int32_t h_q, int32_t topk,
                                          float sm_scale, const float* attn_sink, void* out,
                                          float* lse, int32_t num_splits, void* workspace,
                                          size_t workspace_bytes, uint32_t* dev_status,
                                          void* stream);

/*
 * Sparse MLA decode for callers that cannot allocate device memory. (The pages have no
 * counterpart to this call; it is a service of this library.)
 *
 * nvfp4_sparse_mla_decode needs a caller-provided workspace when it splits the top-k lists.
 * Some callers cannot provide one: code that works within a device-memory budget fixed at
 * start-up and may not call cudaMalloc afterwards, code that must avoid cudaMalloc/cudaFree
 * because they can synchronize the device, or a host that lends the library only its input
 * and output buffers. This call takes the same arguments as nvfp4_sparse_mla_decode without
 * the workspace, and keeps its scratch in a library-owned, fixed-size device array of
 * NVFP4_MLA_NO_ALLOC_SCRATCH_BYTES bytes (reserved on every GPU that loads the library until
 * the process exits). It calls no cudaMalloc, cudaFree or allocating routine.
 *  - A problem whose split count (num_splits, or the library's choice when 0) needs more
 *    scratch than that returns NVFP4_MLA_ERR_WORKSPACE and launches nothing; pass a smaller
 *    num_splits (1 needs no scratch).
 *  - A call outside stream capture looks up the array's device address with the device
 *    current and keeps it; a call under capture uses the kept address. So make one call
 *    before any capture, and make one again after cudaDeviceReset or any other reset of the
 *    device's primary context: the reset may move the array, and an address kept from before
 *    it is invalid until an uncaptured call looks the array up again.
 *  - Argument checks come first and match nvfp4_sparse_mla_decode's (same status for the same
 *    bad argument); a failed runtime query leaves no pending CUDA error behind.
 *  - All calls share the array and it keeps the last call's contents (nothing in it needs to
 *    start at zero: each call writes every value it reads). Calls whose kernels may overlap on
 *    the GPU, e.g. on unordered streams, race on it and must be serialized by the caller.
 * Results equal those of nvfp4_sparse_mla_decode with the same num_splits.
 */
#define NVFP4_MLA_NO_ALLOC_SCRATCH_BYTES (((size_t)32) << 20)

NVFP4_MLA_API int nvfp4_sparse_mla_decode_no_alloc(const void* q, const uint8_t* cache, int64_t num_slots,
                                                   int32_t record_bytes, const int32_t* indices, int32_t batch,
                                                   int32_t s_q, int32_t h_q, int32_t topk, float sm_scale,
                                                   const float* attn_sink, void* out, float* lse,
                                                   int32_t num_splits, uint32_t* dev_status, void* stream);

/*
 * Self-test of the decode's wait bound (no counterpart on the pages). Every pipeline wait in
 * the decode kernel gives up after about one second (then the kernel sets
 * NVFP4_MLA_DEV_TIMEOUT, drains its own work and returns; the context stays usable). This call
 * runs one such wait on an mbarrier that nothing arrives on, on `stream`:
 *   dev_status   device uint32: NVFP4_MLA_DEV_TIMEOUT is OR-ed in when the wait gives up.
 *   elapsed_ns   device uint64: how long the wait lasted, in nanoseconds.
 * Returns NVFP4_MLA_ERR_INVALID_ARG for NULL pointers, NVFP4_MLA_ERR_UNSUPPORTED off sm_103.
 */
NVFP4_MLA_API int nvfp4_mla_selftest_wait_timeout(uint32_t* dev_status, uint64_t* elapsed_ns, void* stream);

/* Static text for a status code (never NULL). */
NVFP4_MLA_API const char* nvfp4_mla_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
NVFP4_MLA_API int nvfp4_mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_MLA_H_ */
