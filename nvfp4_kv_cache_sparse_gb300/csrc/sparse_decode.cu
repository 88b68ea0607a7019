// sparse_decode.cu -- read side: sparse MLA decode over NVFP4 records (and the split merge).
//
// What is computed (FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode",
// "Kernel:" paragraph and validation list): for query row t and head h, with J the used
// entries of t's index list,
//     z_j = sm_scale * q[t,h,:] . K_j          (K_j: 576 dequantized values of record j)
//     out = sum_j e^{z_j} V_j / (sum_j e^{z_j} + e^{sink_h}),   V_j = K_j[0:512]
//     lse = ln sum_j e^{z_j}
// Keys are dequantized to bf16 in shared memory (exact: e2m1 x e4m3 has <= 5 significant
// bits), both contractions run as tcgen05 bf16 MMAs with fp32 accumulation in tensor memory.
//
// Kernel organisation (one CTA per (query row, top-k split, half of the 512 value dims)):
//   warps 0-3  softmax: thread r owns head r = TMEM lane r. Reads S = Q K^T from TMEM, keeps
//              the running max/sum, writes P (bf16) back into TMEM over S, rescales O when
//              the reference max moves, and writes the result.
//   warps 4-7  gather/dequant: 4 threads per key, 32 keys per tile; each thread loads its
//              part of the record with 8/16-byte loads and writes bf16 rows into a
//              128-byte-swizzled K-major tile (the same bytes serve as the MN-major V tile).
//   warp 8     TMEM allocation and MMA issue (one elected lane):
//              QK: S[128 x 32]  = Q[128 x 576] (smem) * K_tile^T, 36 MMAs of K=16
//              PV: O[128 x 256] += P[128 x 32] (TMEM) * V_tile[32 x 256] (smem), 2 MMAs
// Heads are the MMA M dimension (h_q = 64 pads rows 64..127 with zeros). A full fp32 O of
// 128 heads x 512 dims would fill all 512 TMEM columns, so each CTA owns 256 value dims and
// both CTAs of a pair compute the same S (this duplicates QK; a later revision removes it).
// TMEM columns: O [0,256), S/P double buffer [256,288) and [288,320).
//
// Every wait is bounded: on timeout the CTA sets NVFP4_MLA_DEV_TIMEOUT, stops issuing work,
// waits (bounded) for its MMAs to drain and frees its tensor memory before returning.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace nvfp4mla {
namespace {

constexpr int kTile = 32;                         // keys per tile
constexpr int kHeadsM = 128;                      // MMA M (heads, zero padded)
constexpr int kDqk = 576;
constexpr int kDBlocks = kDqk / 64;               // 9 swizzle blocks of 64 bf16 along d
constexpr int kQBytes = kHeadsM * kDqk * 2;       // 147456
constexpr int kQBlockBytes = kHeadsM * 128;       // 16384: one 64-wide d block of Q
constexpr int kKTileBytes = kTile * kDqk * 2;     // 36864
constexpr int kKBlockBytes = kTile * 128;         // 4096: one 64-wide d block of a K tile
constexpr int kOCols = 256;
constexpr int kSCol = 256;                        // S/P buffers at columns 256 and 288
constexpr int kTmemCols = 512;
constexpr int kThreads = 288;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;         // log2 units: rescale O only when max grows by > 2^8

struct __align__(8) SmemCtl {
    uint64_t kfull[2];
    uint64_t kempty[2];
    uint64_t sfull[2];
    uint64_t pfull[2];
    uint64_t odone[2];
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort;
};

constexpr int kSmemBytes = 1024 + kQBytes + 2 * kKTileBytes + 256;

struct KernelArgs {
    const uint16_t* q;
    const uint8_t* cache;
    int64_t num_slots;
    const int32_t* indices;
    int h_q;
    int topk;
    int splits;
    int keys_per_split;
    float scale_log2;            // sm_scale * log2(e)
    const float* sink;
    __nv_bfloat16* out;
    float* lse;
    float* part_out;
    float* part_lse;
    uint32_t* status;
};

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside one 128B-swizzled block.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}

// Two e2m1 codes (one byte: low nibble = even element) times a scale -> bf16x2 (exact).
__device__ __forceinline__ uint32_t dq_e2m1x2(uint32_t byte, __half2 scale2) {
    uint32_t h;
    asm("{\n"
        "  .reg .b8 t;\n"
        "  cvt.u8.u32 t, %1;\n"
        "  cvt.rn.f16x2.e2m1x2 %0, t;\n"
        "}\n"
        : "=r"(h)
        : "r"(byte));
    __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h), scale2);
    const float2 f = __half22float2(v);
    return pack_bf16x2(f.x, f.y);
}

// Two e4m3 codes (low byte = even element) -> bf16x2 (exact).
__device__ __forceinline__ uint32_t dq_e4m3x2(uint32_t two_bytes) {
    uint32_t h;
    const uint16_t in = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    return pack_bf16x2(f.x, f.y);
}

// e4m3 scale byte -> (s, s) as half2 (exact: e4m3 values are f16 values).
__device__ __forceinline__ __half2 scale_half2(uint32_t sbyte) {
    uint32_t h;
    const uint16_t in = static_cast<uint16_t>(sbyte | (sbyte << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    return *reinterpret_cast<__half2*>(&h);
}

// 16 e2m1 values (8 bytes) of one 16-wide block times its scale -> 2 x 16 bytes of bf16.
__device__ __forceinline__ void dq_block(uint2 codes, uint32_t sbyte, uint4& lo, uint4& hi) {
    const __half2 s2 = scale_half2(sbyte);
    lo.x = dq_e2m1x2(codes.x & 0xFFu, s2);
    lo.y = dq_e2m1x2((codes.x >> 8) & 0xFFu, s2);
    lo.z = dq_e2m1x2((codes.x >> 16) & 0xFFu, s2);
    lo.w = dq_e2m1x2(codes.x >> 24, s2);
    hi.x = dq_e2m1x2(codes.y & 0xFFu, s2);
    hi.y = dq_e2m1x2((codes.y >> 8) & 0xFFu, s2);
    hi.z = dq_e2m1x2((codes.y >> 16) & 0xFFu, s2);
    hi.w = dq_e2m1x2(codes.y >> 24, s2);
}

__device__ __forceinline__ void set_abort(SmemCtl* ctl, uint32_t* status) {
    if (atomicExch(&ctl->abort, 1u) == 0u && status != nullptr) atomicOr(status, 0x4u);
}

__device__ __forceinline__ bool wait_or_abort(SmemCtl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    if (*reinterpret_cast<volatile uint32_t*>(&ctl->abort)) return false;
    if (mbar_wait(bar, parity)) return true;
    set_abort(ctl, status);
    return false;
}

// Same, with one answer for the whole warp (warps that go on to warp-collective tcgen05
// instructions must take the same branch).
__device__ __forceinline__ bool wait_warp(SmemCtl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    const bool ok = wait_or_abort(ctl, bar, parity, status);
    return __all_sync(0xffffffffu, ok);
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1) sparse_decode_kernel(const KernelArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = smem + kQBytes;
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + kQBytes + 2 * kKTileBytes);

    const int half = blockIdx.x & 1;                       // which 256 value dims
    const int split = (blockIdx.x >> 1) % a.splits;
    const int row = (blockIdx.x >> 1) / a.splits;
    const int warp = threadIdx.x >> 5;
    const int key_begin = split * a.keys_per_split;
    const int key_end = min(a.topk, key_begin + a.keys_per_split);
    const int n_tiles = key_end > key_begin ? (key_end - key_begin + kTile - 1) / kTile : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->kfull[i], 128);
            mbar_init(&ctl->kempty[i], 1);
            mbar_init(&ctl->sfull[i], 1);
            mbar_init(&ctl->pfull[i], 128);
            mbar_init(&ctl->odone[i], 1);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0u;
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }

    // ---- Q rows -> 128B-swizzled K-major tile (rows >= h_q are zero)
    {
        const uint4* qsrc = reinterpret_cast<const uint4*>(a.q + static_cast<int64_t>(row) * a.h_q * kDqk);
        for (int c = threadIdx.x; c < kHeadsM * (kDqk / 8); c += kThreads) {
            const int h = c / (kDqk / 8);
            const int ch = c % (kDqk / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (h < a.h_q) v = __ldg(qsrc + h * (kDqk / 8) + ch);
            *reinterpret_cast<uint4*>(sQ + (ch >> 3) * kQBlockBytes + swz(h, ch & 7)) = v;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 8) {
        // ================= MMA issuer =================
        const uint32_t idesc_qk = idesc_bf16_f32(kHeadsM, kTile, false, false);
        const uint32_t idesc_pv = idesc_bf16_f32(kHeadsM, kOCols, false, true);
        const uint32_t q_base = smem_addr(sQ);
        const uint32_t k_base = smem_addr(sK);
        const bool leader = elect_one_in_warp();
        bool ok = true;
        auto issue_pv = [&](int j) {
            const int buf = j & 1;
            if (!wait_warp(ctl, &ctl->pfull[buf], (j >> 1) & 1, a.status)) return false;
            tc_fence_after_sync();
            if (leader) {
                const uint32_t v_base = k_base + buf * kKTileBytes + (4 * half) * kKBlockBytes;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint64_t bdesc = sdesc_sw128(v_base + kk * 2048, kKBlockBytes, 1024);
                    mma_ts(tmem, tmem + kSCol + 32 * buf + 8 * kk, bdesc, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&ctl->kempty[buf]);
                mma_commit(&ctl->odone[buf]);
            }
            __syncwarp();
            return true;
        };
        for (int i = 0; i < n_tiles && ok; ++i) {
            const int buf = i & 1;
            ok = wait_warp(ctl, &ctl->kfull[buf], (i >> 1) & 1, a.status);
            if (!ok) break;
            tc_fence_after_sync();
            if (leader) {
                const uint32_t kb = k_base + buf * kKTileBytes;
#pragma unroll 4
                for (int kk = 0; kk < kDqk / 16; ++kk) {
                    const uint64_t adesc = sdesc_sw128(q_base + (kk >> 2) * kQBlockBytes + (kk & 3) * 32, 16, 1024);
                    const uint64_t bdesc = sdesc_sw128(kb + (kk >> 2) * kKBlockBytes + (kk & 3) * 32, 16, 1024);
                    mma_ss(tmem + kSCol + 32 * buf, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(&ctl->sfull[buf]);
            }
            __syncwarp();
            if (i >= 1) ok = issue_pv(i - 1);
        }
        if (ok && n_tiles > 0) issue_pv(n_tiles - 1);
        // drain: every MMA issued by this thread has completed once `drain` flips
        if (leader) mma_commit(&ctl->drain);
        __syncwarp();
        if (!mbar_wait(&ctl->drain, 0)) set_abort(ctl, a.status);
    } else if (warp >= 4) {
        // ================= gather / dequant =================
        const int t = threadIdx.x - 128;
        const int key = t >> 2;        // 0..31 within the tile
        const int qd = t & 3;          // owns 16-wide blocks 4c + qd, c = 0..7
        const int32_t* idx_row = a.indices + static_cast<int64_t>(row) * a.topk;
        for (int i = 0; i < n_tiles; ++i) {
            const int buf = i & 1;
            if (i >= 2 && !wait_or_abort(ctl, &ctl->kempty[buf], ((i - 2) >> 1) & 1, a.status)) break;
            const int pos = key_begin + i * kTile + key;
            int64_t slot = pos < key_end ? static_cast<int64_t>(__ldg(idx_row + pos)) : -1;
            if (slot >= a.num_slots) {
                if (qd == 0 && a.status != nullptr) atomicOr(a.status, 0x2u);
                slot = -1;
            }
            uint8_t* tile = sK + buf * kKTileBytes;
            if (slot >= 0) {
                const uint8_t* rec = a.cache + slot * R;
                uint32_t sb[8];
                if constexpr (R == 352) {
                    const uint2 s8 = __ldg(reinterpret_cast<const uint2*>(rec + 320 + 8 * qd));
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        sb[c] = (s8.x >> (8 * c)) & 0xFFu;
                        sb[c + 4] = (s8.y >> (8 * c)) & 0xFFu;
                    }
                } else {
                    const uint4 s0 = __ldg(reinterpret_cast<const uint4*>(rec + 256));
                    const uint4 s1 = __ldg(reinterpret_cast<const uint4*>(rec + 272));
                    const uint32_t words[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) sb[c] = (words[c] >> (8 * qd)) & 0xFFu;   // byte 4c + qd
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint2 codes = __ldg(reinterpret_cast<const uint2*>(rec + 32 * c + 8 * qd));
                    uint4 lo, hi;
                    dq_block(codes, sb[c], lo, hi);
                    uint8_t* blk = tile + c * kKBlockBytes;
                    *reinterpret_cast<uint4*>(blk + swz(key, 2 * qd)) = lo;
                    *reinterpret_cast<uint4*>(blk + swz(key, 2 * qd + 1)) = hi;
                }
                uint4 r0, r1;
                if constexpr (R == 352) {
                    const uint4 e = __ldg(reinterpret_cast<const uint4*>(rec + 256 + 16 * qd));
                    r0 = make_uint4(dq_e4m3x2(e.x), dq_e4m3x2(e.x >> 16), dq_e4m3x2(e.y), dq_e4m3x2(e.y >> 16));
                    r1 = make_uint4(dq_e4m3x2(e.z), dq_e4m3x2(e.z >> 16), dq_e4m3x2(e.w), dq_e4m3x2(e.w >> 16));
                } else {
                    r0 = __ldg(reinterpret_cast<const uint4*>(rec + 304 + 32 * qd));
                    r1 = __ldg(reinterpret_cast<const uint4*>(rec + 304 + 32 * qd + 16));
                }
                uint8_t* blk = tile + 8 * kKBlockBytes;
                *reinterpret_cast<uint4*>(blk + swz(key, 2 * qd)) = r0;
                *reinterpret_cast<uint4*>(blk + swz(key, 2 * qd + 1)) = r1;
            } else {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int c = 0; c < kDBlocks; ++c) {
                    uint8_t* blk = tile + c * kKBlockBytes;
                    *reinterpret_cast<uint4*>(blk + swz(key, 2 * qd)) = z;
                    *reinterpret_cast<uint4*>(blk + swz(key, 2 * qd + 1)) = z;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&ctl->kfull[buf]);
        }
    } else {
        // ================= softmax / epilogue (thread = head row) =================
        const int h = threadIdx.x;                              // TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const int32_t* idx_row = a.indices + static_cast<int64_t>(row) * a.topk;
        float m_ref = -INFINITY;   // reference max, log2 units of scaled logits
        float l = 0.0f;            // sum of 2^(s - m_ref) over used keys
        bool ok = true;
        int done_tiles = 0;
        for (int i = 0; i < n_tiles; ++i) {
            const int buf = i & 1;
            // used-key mask of this tile
            uint32_t used = 0u;
            const int pos0 = key_begin + i * kTile;
#pragma unroll 4
            for (int j = 0; j < kTile; ++j) {
                if (pos0 + j < key_end) {
                    const int32_t s = __ldg(idx_row + pos0 + j);
                    if (s >= 0 && s < a.num_slots) used |= 1u << j;
                }
            }
            ok = wait_warp(ctl, &ctl->sfull[buf], (i >> 1) & 1, a.status);
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t sr[32];
            tmem_ld32(lane_base + kSCol + 32 * buf, sr);
            tmem_wait_ld();
            float s[32];
            float tile_max = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                s[j] = ((used >> j) & 1u) ? __uint_as_float(sr[j]) * a.scale_log2 : -INFINITY;
                tile_max = fmaxf(tile_max, s[j]);
            }
            bool rescale = false;
            float alpha = 1.0f;
            if (tile_max > m_ref + kRescaleThreshold) {
                if (m_ref != -INFINITY) {
                    alpha = exp2f(m_ref - tile_max);
                    rescale = true;
                }
                m_ref = tile_max;
            }
            l *= alpha;
            uint32_t p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float p0 = (m_ref == -INFINITY) ? 0.0f : exp2f(s[2 * j] - m_ref);
                const float p1 = (m_ref == -INFINITY) ? 0.0f : exp2f(s[2 * j + 1] - m_ref);
                l += p0 + p1;
                p[j] = pack_bf16x2(p0, p1);
            }
            if (__any_sync(0xffffffffu, rescale) && i > 0) {
                ok = wait_warp(ctl, &ctl->odone[(i - 1) & 1], ((i - 1) >> 1) & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
#pragma unroll 1
                for (int c = 0; c < kOCols / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(lane_base + 32 * c, o);
                }
            }
            tmem_st16(lane_base + kSCol + 32 * buf, p);
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(&ctl->pfull[buf]);
            done_tiles = i + 1;
        }
        // ---- epilogue
        bool have_o = false;
        if (ok && done_tiles == n_tiles && n_tiles > 0) {
            have_o = wait_warp(ctl, &ctl->odone[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, a.status);
            if (have_o) tc_fence_after_sync();
        }
        const bool empty = !(l > 0.0f);
        const bool write = h < a.h_q;
        float inv = 0.0f;
        float lse_nat = -INFINITY;
        if (!empty) {
            lse_nat = (m_ref + log2f(l)) * kLn2;
            float denom = l;
            if (a.splits == 1 && a.sink != nullptr) denom += exp2f(__ldg(a.sink + (h < a.h_q ? h : 0)) * kLog2e - m_ref);
            inv = 1.0f / denom;
        }
        const int64_t rh = static_cast<int64_t>(row) * a.h_q + h;
        if (a.splits == 1) {
            __nv_bfloat16* dst = a.out + rh * 512 + 256 * half;
#pragma unroll 1
            for (int c = 0; c < kOCols / 32; ++c) {
                uint32_t o[32];
                if (have_o) {
                    tmem_ld32(lane_base + 32 * c, o);
                    tmem_wait_ld();
                }
                if (write) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = (have_o && !empty) ? __uint_as_float(o[8 * v + 2 * e]) * inv : 0.0f;
                            const float x1 = (have_o && !empty) ? __uint_as_float(o[8 * v + 2 * e + 1]) * inv : 0.0f;
                            wp[e] = pack_bf16x2(x0, x1);
                        }
                        *reinterpret_cast<uint4*>(dst + 32 * c + 8 * v) = w;
                    }
                }
            }
            if (write && half == 0) a.lse[rh] = lse_nat;
        } else {
            const int64_t ph = (static_cast<int64_t>(row) * a.splits + split) * a.h_q + h;
            float* dst = a.part_out + ph * 512 + 256 * half;
#pragma unroll 1
            for (int c = 0; c < kOCols / 32; ++c) {
                uint32_t o[32];
                if (have_o) {
                    tmem_ld32(lane_base + 32 * c, o);
                    tmem_wait_ld();
                }
                if (write) {
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        float4 w;
                        w.x = (have_o && !empty) ? __uint_as_float(o[4 * v + 0]) * inv : 0.0f;
                        w.y = (have_o && !empty) ? __uint_as_float(o[4 * v + 1]) * inv : 0.0f;
                        w.z = (have_o && !empty) ? __uint_as_float(o[4 * v + 2]) * inv : 0.0f;
                        w.w = (have_o && !empty) ? __uint_as_float(o[4 * v + 3]) * inv : 0.0f;
                        *reinterpret_cast<float4*>(dst + 32 * c + 4 * v) = w;
                    }
                }
            }
            if (write && half == 0) a.part_lse[ph] = lse_nat;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// out = sum_p e^{lse_p - lse} out_p / (1 + e^{sink - lse}),  lse = ln sum_p e^{lse_p}
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ part_out,
                                                      const float* __restrict__ part_lse, int splits, int h_q,
                                                      const float* __restrict__ sink, __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse) {
    const int rh = blockIdx.x;             // row * h_q + h
    const int row = rh / h_q;
    const int h = rh % h_q;
    float m = -INFINITY;
    for (int p = 0; p < splits; ++p) m = fmaxf(m, __ldg(part_lse + (static_cast<int64_t>(row) * splits + p) * h_q + h));
    const int d0 = threadIdx.x * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float total = -INFINITY;
    if (m != -INFINITY) {
        float sum = 0.0f;
        for (int p = 0; p < splits; ++p)
            sum += expf(__ldg(part_lse + (static_cast<int64_t>(row) * splits + p) * h_q + h) - m);
        total = m + logf(sum);
        const float scale = 1.0f + (sink != nullptr ? expf(__ldg(sink + h) - total) : 0.0f);
        for (int p = 0; p < splits; ++p) {
            const int64_t ph = (static_cast<int64_t>(row) * splits + p) * h_q + h;
            const float w = expf(__ldg(part_lse + ph) - total) / scale;
            const float4 v = __ldg(reinterpret_cast<const float4*>(part_out + ph * 512 + d0));
            acc[0] += w * v.x;
            acc[1] += w * v.y;
            acc[2] += w * v.z;
            acc[3] += w * v.w;
        }
    }
    uint2 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    *reinterpret_cast<uint2*>(out + static_cast<int64_t>(rh) * 512 + d0) = o;
    if (threadIdx.x == 0) lse[rh] = total;
}

}  // namespace

int decode_keys_per_split(int topk, int splits) {
    const int per = (topk + splits - 1) / splits;
    return (per + kTile - 1) / kTile * kTile;
}

cudaError_t launch_sparse_decode(const DecodeArgs& d, cudaStream_t stream) {
    static bool attr_done[2] = {false, false};
    KernelArgs a;
    a.q = static_cast<const uint16_t*>(d.q);
    a.cache = d.cache;
    a.num_slots = d.num_slots;
    a.indices = d.indices;
    a.h_q = d.h_q;
    a.topk = d.topk;
    a.splits = d.splits;
    a.keys_per_split = decode_keys_per_split(d.topk, d.splits);
    a.scale_log2 = d.sm_scale * kLog2e;
    a.sink = d.attn_sink;
    a.out = static_cast<__nv_bfloat16*>(d.out);
    a.lse = d.lse;
    a.part_out = d.part_out;
    a.part_lse = d.part_lse;
    a.status = d.dev_status;
    const dim3 grid(static_cast<unsigned>(d.rows) * static_cast<unsigned>(d.splits) * 2u);
    const dim3 block(kThreads);
    cudaError_t err;
    if (d.record_bytes == 352) {
        if (!attr_done[0]) {
            err = cudaFuncSetAttribute(sparse_decode_kernel<352>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (err != cudaSuccess) return err;
            attr_done[0] = true;
        }
        sparse_decode_kernel<352><<<grid, block, kSmemBytes, stream>>>(a);
    } else {
        if (!attr_done[1]) {
            err = cudaFuncSetAttribute(sparse_decode_kernel<432>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (err != cudaSuccess) return err;
            attr_done[1] = true;
        }
        sparse_decode_kernel<432><<<grid, block, kSmemBytes, stream>>>(a);
    }
    err = cudaGetLastError();
    if (err != cudaSuccess || d.splits == 1) return err;
    combine_kernel<<<d.rows * d.h_q, 128, 0, stream>>>(d.part_out, d.part_lse, d.splits, d.h_q, d.attn_sink,
                                                       static_cast<__nv_bfloat16*>(d.out), d.lse);
    return cudaGetLastError();
}

}  // namespace nvfp4mla
