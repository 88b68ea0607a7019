// quantize_append.cu -- write side: quantize each token's 512 bf16 NoPE values and 64 bf16
// RoPE values into one NVFP4 record and scatter it to its cache slot.
//
// Record formats:
//  * 352 B, FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode",
//    format block "nvfp4.fp8rope (352 B/token)": [0,256) e2m1 pairs, [256,320) unscaled e4m3
//    RoPE, [320,352) e4m3 scales with block s at byte 320 + 8*(s&3) + (s>>2). With kBlk the
//    scales of a 352-byte record are stored in block order instead (block s at 320 + s), the
//    unpermuted record of the scale-layout comparison in the same format block.
//  * 432 B, vLLM PR 82 "kv: nvfp4_ds_mla - 4-bit NVFP4 KV cache for B12X sparse MLA (SM120)",
//    Problem / Fix (Write side): [0,256) e2m1 pairs, [256,288) scales in block order,
//    [288,304) zeros, [304,432) bf16 RoPE copied verbatim.
//  * 656 B, the fp8 record the same vLLM page (Problem) measures against: [0,512) e4m3 NoPE,
//    [512,528) four fp32 scales (one per 128 values), [528,656) bf16 RoPE copied verbatim.
//    The page states no fp8 scale rule; this kernel uses scale = amax / 448 per 128-value tile
//    and code = e4m3(x / scale), both IEEE fp32 divisions (a zero tile stores scale 0 and
//    signed zero codes).
// Scale rule (vLLM PR 82, Tests): scale = E4M3(group_amax / 6), round-to-nearest-even and
// saturating; each value is rounded to the nearest e2m1 grid point (ties to even, saturating)
// after division by the decoded scale; the sign of the input is always kept.
//
// Design: one warp per token, lane g owns the 16-value group g. The group maximum is taken on
// the |bf16| bit patterns (non-negative floats order like integers) with packed 16-bit maxima,
// so no shuffles are needed. An NVFP4 record is written in place, each store instruction of
// the warp covering one contiguous field of it; an fp8 record is assembled in a per-warp
// shared-memory stage and written with 16-byte stores (41 chunks over 32 lanes).
//
// Exactness of x / s without a division per value: s is an e4m3 value (<= 4 significant bits)
// and x a bf16 value (<= 8), so the exact quotient x/s is either exactly one of the e2m1 tie
// points {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5} or at least 1/300 (relative) away from all of
// them. q = |x| * rn(1/s) is within 2^-23 (relative) of x/s; rounding q to 12 significant bits
// therefore lands exactly on the tie point in the first case and cannot cross one in the
// second, so the hardware e2m1 rounding of that value equals the rounding of the IEEE
// quotient. The same holds for q keeping the sign of x (the rounding acts on the magnitude
// bits), and the hardware conversions keep the sign, so a negative value that rounds to zero
// gives the negative-zero code.
//
// amax / 6 as amax * rn(1/6): amax has at most 8 significant bits. If amax / 6 is an e4m3 tie
// point T (at most 5 significant bits), the product is T (1 + d) with |d| <= 2^-24, which rounds
// to T in fp32; otherwise amax / 6 lies at least 2^-10.6 (relative) from every tie point, far
// beyond the product's error. Either way the e4m3 rounding equals that of amax / 6. Per block,
// rn(1/s) of every e4m3 scale is kept in a shared table.
//
// Fused producer (kFused): SGLang PR 38646 "[SM120] Add opt-in NVFP4 sparse-MLA KV cache format
// for DeepSeek-V4", "Limitations" (no fused norm+rope+quantize+store kernel for NVFP4, so the
// path pays a bf16 intermediate and a separate quantize kernel) and "Stores". Ahead of the
// quantizer, the kernel takes the pre-norm latent and the pre-rotation k_pe and computes, in
// fp32, the RMSNorm y_i = w_i x_i / sqrt(mean_j x_j^2 + eps) (sum of squares by a warp butterfly,
// so every lane holds the same sum) and the rotation of each k_pe pair (a, b) by the token's
// position, (a c - b s, b c + a s), pairs (f, f + 32) or (2f, 2f + 1); each result is rounded
// once to bf16, the value the unfused path would store in its intermediate, and then quantized
// exactly as in the plain append. The fp32 results lie within about 2^-19 (relative to the
// terms) of the exact ones, so the bf16 rounding can differ from the exact one only for values
// that close to a rounding midpoint.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"

namespace nvfp4mla {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kTokensPerRound = 2;
constexpr int kBlocksPerSm = 4;
constexpr int kFusedBlocksPerSm = 2;   // the producer stage holds the norm weights and more per token

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// e4m3 codes of two non-negative floats, round-to-nearest-even, saturating:
// bits [15:8] = code(hi), [7:0] = code(lo).
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// e2m1 codes of two non-negative floats, round-to-nearest-even, saturating:
// bits [7:4] = code(hi), [3:0] = code(lo).
__device__ __forceinline__ uint32_t e2m1x2_rn_sat(float hi, float lo) {
    uint32_t r;
    asm("{\n"
        "  .reg .b8 t;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n"
        "  cvt.u32.u8 %0, t;\n"
        "}\n"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Value of a non-negative finite e4m3 code (0x00..0x7E), built from its bit fields.
__device__ __forceinline__ float e4m3_code_value(uint32_t c) {
    const uint32_t e = c >> 3, m = c & 7u;
    return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;
}

// Round a float's magnitude to 12 significant bits, half away from zero (see the file comment).
__device__ __forceinline__ float round_to_12_bits(float v) {
    return __uint_as_float((__float_as_uint(v) + 0x800u) & ~0xFFFu);
}

// Per-halfword unsigned maximum of two packed pairs.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// e4m3 codes of two floats (signs kept), round-to-nearest-even, saturating:
// bits [15:8] = code(hi), [7:0] = code(lo).
__device__ __forceinline__ uint32_t e4m3x2_signed(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int R, bool kBlk, bool kFused>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, kFused ? kFusedBlocksPerSm : kBlocksPerSm)
quantize_append_kernel(const uint16_t* __restrict__ latent, int64_t latent_stride, const uint16_t* __restrict__ rope,
                       int64_t rope_stride, const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                       uint8_t* __restrict__ cache, int64_t num_slots, uint32_t* __restrict__ dev_status,
                       const ProducerArgs pr) {
    __shared__ __align__(16) uint8_t stage[kWarpsPerBlock][R];
    __shared__ float inv_scale[128];   // rn(1 / value) of each e4m3 scale code; 0 for code 0
    // A decode launched next on the stream may start its prologue now; it waits for this grid
    // before it reads anything. This grid is itself a programmatic dependent of the preceding
    // kernel and waits for it to complete before reading or writing memory (the table needs
    // neither).
    asm volatile("griddepcontrol.launch_dependents;");
    if (R != 656 && threadIdx.x < 128)
        inv_scale[threadIdx.x] = threadIdx.x ? __frcp_rn(e4m3_code_value(threadIdx.x)) : 0.0f;
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* rec = stage[warp];
    // fused producer: the lane's 16 norm weights (group `lane`), and its rotation frequencies
    uint32_t nw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    int freq = 0;
    if constexpr (kFused) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(pr.norm_weight) + 2 * lane);
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(pr.norm_weight) + 2 * lane + 1);
        nw[0] = a.x; nw[1] = a.y; nw[2] = a.z; nw[3] = a.w;
        nw[4] = b.x; nw[5] = b.y; nw[6] = b.z; nw[7] = b.w;
        // rotate half: elements 2 lane, 2 lane + 1 have frequencies (2 lane) % 32 and the next;
        // interleaved: the lane's two elements are the pair of frequency `lane`
        freq = pr.rotate_half ? (2 * lane) & 31 : lane;
    }

    // kTokensPerRound tokens per warp per round. The loads of a round (slot, 32 latent bytes and
    // 4 RoPE bytes per lane per token) are issued before the previous round is converted, so a
    // warp always has a round in flight while it converts.
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
    struct Round {
        int64_t slot[kTokensPerRound];
        uint4 va[kTokensPerRound], vb[kTokensPerRound];
        uint32_t rw[kTokensPerRound];
        int64_t pos[kTokensPerRound];   // fused producer only
    };
    auto load_round = [&](int64_t t0, Round& r) {
#pragma unroll
        for (int u = 0; u < kTokensPerRound; ++u) {
            const int64_t t = t0 + u * stride;
            r.slot[u] = -1;
            if (t < num_tokens) {
                r.slot[u] = __ldg(slot_mapping + t);
                const uint4* src = reinterpret_cast<const uint4*>(latent + t * latent_stride) + 2 * lane;
                r.va[u] = __ldg(src);
                r.vb[u] = __ldg(src + 1);
                r.rw[u] = __ldg(reinterpret_cast<const uint32_t*>(rope + t * rope_stride) + lane);
                if constexpr (kFused) r.pos[u] = __ldg(pr.positions + t);
            }
        }
    };
    Round cur;
    load_round(static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp, cur);
    for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp; t0 < num_tokens;
         t0 += stride * kTokensPerRound) {
        Round nxt;
        load_round(t0 + stride * kTokensPerRound, nxt);
        const int64_t* slot = cur.slot;
        const uint4* va = cur.va;
        const uint4* vb = cur.vb;
        const uint32_t* rw = cur.rw;
#pragma unroll
        for (int u = 0; u < kTokensPerRound; ++u) {
            if (slot[u] < 0) continue;                       // padding token (or past the end)
            if (slot[u] >= num_slots) {
                if (lane == 0 && dev_status != nullptr) atomicOr(dev_status, 0x1u);
                continue;
            }
            uint8_t* const dst = cache + slot[u] * R;   // NVFP4 records are written in place (below)
            // ---- NoPE group `lane`: 16 bf16 values
            uint32_t w[8] = {va[u].x, va[u].y, va[u].z, va[u].w, vb[u].x, vb[u].y, vb[u].z, vb[u].w};
            uint32_t rwv = rw[u];
            if constexpr (kFused) {
                const int64_t p = cur.pos[u];
                if (p < 0 || p >= pr.num_positions) {
                    if (lane == 0 && dev_status != nullptr) atomicOr(dev_status, 0x10u);
                    continue;
                }
                // the rotation's cos / sin first: their loads overlap the norm
                float c0, c1, s0, s1;
                if (pr.rotate_half) {
                    const float2 c = __ldg(reinterpret_cast<const float2*>(pr.cos_table + p * 32 + freq));
                    const float2 sn = __ldg(reinterpret_cast<const float2*>(pr.sin_table + p * 32 + freq));
                    c0 = c.x; c1 = c.y; s0 = sn.x; s1 = sn.y;
                } else {
                    c0 = c1 = __ldg(pr.cos_table + p * 32 + freq);
                    s0 = s1 = __ldg(pr.sin_table + p * 32 + freq);
                }
                // RMSNorm of the token's 512 values
                float ss = 0.0f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    ss = fmaf(bf16_lo(w[k]), bf16_lo(w[k]), ss);
                    ss = fmaf(bf16_hi(w[k]), bf16_hi(w[k]), ss);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);   // same sum in every lane
                const float inv = __fdiv_rn(1.0f, __fsqrt_rn(fmaf(ss, 1.0f / 512.0f, pr.eps)));
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    w[k] = bf16x2_rn(bf16_lo(w[k]) * bf16_lo(nw[k]) * inv, bf16_hi(w[k]) * bf16_hi(nw[k]) * inv);
                // rotation of the lane's two k_pe values
                const float e0 = bf16_lo(rwv), e1 = bf16_hi(rwv);
                if (pr.rotate_half) {
                    // partner elements +-32 live in lane ^ 16; the first half subtracts b s
                    const uint32_t pw = __shfl_xor_sync(0xffffffffu, rwv, 16);
                    const float sg = lane < 16 ? -1.0f : 1.0f;
                    rwv = bf16x2_rn(fmaf(e0, c0, sg * (bf16_lo(pw) * s0)), fmaf(e1, c1, sg * (bf16_hi(pw) * s1)));
                } else {
                    rwv = bf16x2_rn(fmaf(e0, c0, -(e1 * s0)), fmaf(e1, c0, e0 * s0));
                }
            }
            // group maximum on |bf16| bit patterns (non-negative floats order like integers), two
            // per 32-bit word
            uint32_t m2 = max_u16x2(max_u16x2(max_u16x2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                              max_u16x2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu)),
                                    max_u16x2(max_u16x2(w[4] & 0x7FFF7FFFu, w[5] & 0x7FFF7FFFu),
                                              max_u16x2(w[6] & 0x7FFF7FFFu, w[7] & 0x7FFF7FFFu)));
            uint32_t amax_bits = max(m2 & 0xFFFFu, m2 >> 16);
            if constexpr (R == 656) {
                // ---- fp8 record: the 8 lanes of a 128-value tile share its maximum
                amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, 1));
                amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, 2));
                amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, 4));
                const float scale = __fdiv_rn(__uint_as_float(amax_bits << 16), 448.0f);
                // |x| >= 65536 is stored, but lies beyond the f16 value operand of the decode
                if ((lane & 7) == 0 && amax_bits >= 0x4780u && dev_status != nullptr) atomicOr(dev_status, 0x8u);
                uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float q0 = scale != 0.0f ? __fdiv_rn(fabsf(bf16_lo(w[k])), scale) : 0.0f;
                    const float q1 = scale != 0.0f ? __fdiv_rn(fabsf(bf16_hi(w[k])), scale) : 0.0f;
                    uint32_t c = e4m3x2_rn_sat(q1, q0);                       // byte 2k: element 2k
                    c |= ((w[k] >> 8) & 0x80u) | ((w[k] >> 16) & 0x8000u);   // signs of both elements
                    packed[k >> 1] |= c << (16 * (k & 1));
                }
                *reinterpret_cast<uint4*>(rec + 16 * lane) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                if ((lane & 7) == 0) *reinterpret_cast<float*>(rec + 512 + 4 * (lane >> 3)) = scale;
                *reinterpret_cast<uint32_t*>(rec + 528 + 4 * lane) = rwv;
            } else {
            const float amax = __uint_as_float(amax_bits << 16);
            const uint32_t sbyte = e4m3x2_rn_sat(0.0f, amax * (1.0f / 6.0f)) & 0xFFu;
            const float inv_s = inv_scale[sbyte];

            uint32_t packed[2] = {0u, 0u};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                // both products with one f32x2 FMA (addend -0, so that -0 stays -0)
                float q0, q1;
                asm("{\n .reg .b64 x, s, z, r;\n mov.b64 x, {%2, %3};\n mov.b64 s, {%4, %4};\n mov.b64 z, {%5, %5};\n"
                    " fma.rn.f32x2 r, x, s, z;\n mov.b64 {%0, %1}, r;\n}\n"
                    : "=f"(q0), "=f"(q1)
                    : "f"(bf16_lo(w[k])), "f"(bf16_hi(w[k])), "f"(inv_s), "f"(-0.0f));
                q0 = round_to_12_bits(q0);
                q1 = round_to_12_bits(q1);
                const uint32_t byte = e2m1x2_rn_sat(q1, q0);              // even element -> low nibble
                packed[k >> 2] = (k & 3) ? __byte_perm(packed[k >> 2], byte, (k & 3) == 1 ? 0x3240u
                                                                            : (k & 3) == 2 ? 0x3410u
                                                                                           : 0x4210u)
                                         : byte;
            }
            // each store instruction of the warp covers one contiguous run of the record (codes 256 B,
            // scales 32 B, RoPE 64 or 128 B, pad 16 B), so the record reaches L2 as whole lines
            *reinterpret_cast<uint2*>(dst + 8 * lane) = make_uint2(packed[0], packed[1]);

            // ---- RoPE: lane owns elements 2*lane and 2*lane+1
            if constexpr (R == 352) {
                dst[kBlk ? 320 + lane : 320 + 8 * (lane & 3) + (lane >> 2)] = static_cast<uint8_t>(sbyte);
                const uint32_t c = e4m3x2_signed(bf16_hi(rwv), bf16_lo(rwv));
                *reinterpret_cast<uint16_t*>(dst + 256 + 2 * lane) = static_cast<uint16_t>(c);
            } else {
                dst[256 + lane] = static_cast<uint8_t>(sbyte);
                *reinterpret_cast<uint32_t*>(dst + 304 + 4 * lane) = rwv;
                if (lane < 4) *reinterpret_cast<uint32_t*>(dst + 288 + 4 * lane) = 0u;
            }
            }
            if constexpr (R == 656) {   // the fp8 record goes out from its stage as 16-byte stores
                __syncwarp();
                for (int c = lane; c < R / 16; c += 32) {
                    const uint4 v = reinterpret_cast<const uint4*>(rec)[c];
                    reinterpret_cast<uint4*>(dst)[c] = v;
                }
                __syncwarp();
            }
        }
        cur = nxt;
    }
}

}  // namespace

cudaError_t launch_quantize_append(const void* kv_latent, int64_t latent_row_stride, const void* k_rope,
                                   int64_t rope_row_stride, const int64_t* slot_mapping, int64_t num_tokens,
                                   uint8_t* cache, int64_t num_slots, int record_bytes, bool block_scales,
                                   uint32_t* dev_status, int sm_count, cudaStream_t stream,
                                   const ProducerArgs* producer) {
    const int64_t want = (num_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t cap = static_cast<int64_t>(sm_count) * (producer ? kFusedBlocksPerSm : kBlocksPerSm);   // one wave
    const int grid = static_cast<int>(want < cap ? want : cap);
    const dim3 block(kWarpsPerBlock * 32);
    const auto* lat = static_cast<const uint16_t*>(kv_latent);
    const auto* rope = static_cast<const uint16_t*>(k_rope);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddepcontrol.wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool f = producer != nullptr;
    const auto kernel = record_bytes == 656 ? (f ? quantize_append_kernel<656, false, true> : quantize_append_kernel<656, false, false>)
                        : record_bytes == 432 ? (f ? quantize_append_kernel<432, false, true> : quantize_append_kernel<432, false, false>)
                        : block_scales ? (f ? quantize_append_kernel<352, true, true> : quantize_append_kernel<352, true, false>)
                                       : (f ? quantize_append_kernel<352, false, true> : quantize_append_kernel<352, false, false>);
    const ProducerArgs pr = f ? *producer : ProducerArgs{};
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, lat, latent_row_stride, rope, rope_row_stride,
                                               slot_mapping, num_tokens, cache, num_slots, dev_status, pr);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace nvfp4mla
