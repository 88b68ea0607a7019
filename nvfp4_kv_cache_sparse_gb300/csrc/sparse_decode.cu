// sparse_decode.cu -- read side: sparse MLA decode over NVFP4 records (and the split merge).
//
// What is computed (FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode",
// "Kernel:" paragraph and validation list): for query row t and head h, with J the used
// entries of t's index list,
//     z_j = sm_scale * q[t,h,:] . K_j          (K_j: 576 dequantized values of record j)
//     out = sum_j e^{z_j} V_j / (sum_j e^{z_j} + e^{sink_h}),   V_j = K_j[0:512]
//     lse = ln sum_j e^{z_j}
// Keys are dequantized to bf16 in shared memory (exact: e2m1 x e4m3 has <= 5 significant
// bits); both contractions run as tcgen05 bf16 MMAs with fp32 accumulation in tensor memory.
//
// Work split: a cluster of two CTAs per (query row, top-k split), with different roles.
// With 128 heads, the fp32 accumulator O [128 x 512] fills all 512 TMEM columns of an SM, so
// QK^T and PV run on different SMs and only the bf16 P tile travels between them:
//   CTA 0 (QK): gathers whole records, dequantizes K tiles (576 dims), keeps Q [128 x 576]
//     in TMEM as the MMA A operand, computes S = Q K^T, runs the online softmax, and sends
//     each row's P (bf16) and rescale factor to CTA 1 with st.async (DSMEM, one way:
//     132 B per head per 64 keys).
//   CTA 1 (PV): gathers the NoPE half of the same records, dequantizes V tiles (512 dims),
//     keeps O in TMEM and computes O += P V with P read from shared memory; its MMA commit
//     multicasts back to CTA 0 to release the P slot. At the end CTA 0 sends each row's
//     running max and sum, and CTA 1 normalizes and writes `out` (CTA 0 writes `lse`).
// Warp roles (448 threads):
//   CTA 0: warps 0-3 softmax (thread r = head r = TMEM lane r), 4-11 gather/dequant,
//          12-13 QK issuers (even / odd tiles; one elected lane each).
//   CTA 1: warps 0-3 rescale/epilogue (thread r = TMEM lane r), 4-11 gather/dequant, 12 PV issuer.
// Tiles are 64 keys; every K/V tile is written in a 128B-swizzled layout that is the K-major
// B operand of QK (CTA 0) or the MN-major B operand of PV (CTA 1).
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

constexpr int kTile = 64;                          // keys per tile
constexpr int kHeadsM = 128;                       // MMA M (heads, zero padded)
constexpr int kDqk = 576;
constexpr int kBlkBytes = kTile * 128;             // one 64-wide d block of a tile: 8 KB
constexpr int kKStages = 2;                        // CTA 0: K tiles of 9 blocks (8 NoPE + RoPE)
constexpr int kKTileBytes = 9 * kBlkBytes;         // 72 KB
constexpr int kVStages = 2;                        // CTA 1: V tiles of 8 blocks
constexpr int kVTileBytes = 8 * kBlkBytes;         // 64 KB
constexpr int kPStages = 2;                        // CTA 1: P tiles [128 heads x 64 keys] bf16
constexpr int kPBytes = kHeadsM * 128;             // 16 KB
constexpr int kMaskSlots = 8;
constexpr int kRawStages = 3;                      // raw records in flight (cp.async), in tiles
// Raw record slot of one key: CTA 0 copies the whole record; CTA 1 the 256 NoPE bytes and the
// 32 scale bytes (16-byte chunks 0..15 and 16..17 of the slot).
template <int R, bool kWhole>
struct RawSlot {
    static constexpr int kChunks = kWhole ? R / 16 : 18;
    static constexpr int kKeyBytes = kChunks * 16;
    static constexpr int kTileBytes = kTile * kKeyBytes;
    // record byte offset of slot chunk j
    static __device__ __forceinline__ int src_offset(int j) {
        return (kWhole || j < 16) ? 16 * j : (R == 352 ? 320 : 256) + 16 * (j - 16);
    }
    static constexpr int kScaleOffset = kWhole ? (R == 352 ? 320 : 256) : 256;
};
constexpr int kRaw0Bytes = kRawStages * kTile * 432;     // CTA 0 raw ring (largest record)
constexpr int kRaw1Bytes = kRawStages * kTile * 288;     // CTA 1 raw ring
constexpr uint32_t kColS = 0;                      // CTA 0: S buffers [0,64), [64,128)
constexpr uint32_t kColQ = 128;                    // CTA 0: Q, 576 bf16 = 288 columns
constexpr uint32_t kColO = 0;                      // CTA 1: O, 512 columns
constexpr int kTmemCols = 512;
constexpr int kThreads = 448;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;          // log2 units: rescale O only when max grows by > 2^8

// Control block at the same offset in both CTAs (CTA 1's commits multicast into CTA 0's
// pempty, and CTA 0's st.async completions land on CTA 1's pfull / fin).
struct __align__(8) SmemCtl {
    // CTA 0
    uint64_t kfull[kKStages];     // dequant -> QK issuer
    uint64_t kempty[kKStages];    // QK commit -> dequant
    uint64_t sfull[2];            // QK commit -> softmax
    uint64_t sfree[2];            // softmax has read S -> QK issuer
    uint64_t mfull[kMaskSlots];   // used-key mask of a tile written
    uint64_t pempty[kPStages];    // CTA 1's PV has read the P slot (multicast commit)
    uint64_t qready;              // Q in TMEM
    // CTA 1
    uint64_t vfull[kVStages];     // dequant -> PV issuer
    uint64_t vempty[kVStages];    // PV commit -> dequant
    uint64_t pfull[kPStages];     // P + alpha of a tile landed (tx-counted)
    uint64_t ready[kPStages];     // epilogue warps checked alpha (and rescaled O) -> PV issuer
    uint64_t odone[2];            // PV commit -> epilogue warps
    uint64_t fin;                 // final (max, sum) of every row landed (tx-counted)
    // both
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort;
    uint8_t mask[kMaskSlots][8];
};

constexpr int kCtlBytes = 1024;
static_assert(sizeof(SmemCtl) <= kCtlBytes, "control block");
// CTA 0 data
constexpr int kOffK = kCtlBytes;
constexpr int kOffRaw0 = kOffK + kKStages * kKTileBytes;
// CTA 1 data
constexpr int kOffV = kCtlBytes;
constexpr int kOffP = kOffV + kVStages * kVTileBytes;
constexpr int kOffAlpha = kOffP + kPStages * kPBytes;          // [kPStages][128] fp32
constexpr int kOffFin = kOffAlpha + kPStages * kHeadsM * 4;    // [128] (max, sum) pairs
constexpr int kOffRaw1 = kOffFin + kHeadsM * 8;
constexpr int kSmem0 = kOffRaw0 + kRaw0Bytes;
constexpr int kSmem1 = kOffRaw1 + kRaw1Bytes;
constexpr int kSmemBytes = 1024 + (kSmem0 > kSmem1 ? kSmem0 : kSmem1);

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

__device__ __forceinline__ bool aborted(SmemCtl* ctl) {
    return *reinterpret_cast<volatile uint32_t*>(&ctl->abort) != 0u;
}

__device__ __forceinline__ bool wait_or_abort(SmemCtl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    if (aborted(ctl)) return false;
    if (mbar_wait(bar, parity)) return true;
    set_abort(ctl, status);
    return false;
}

// One answer for the whole warp (warps that go on to warp-collective instructions must take
// the same branch).
__device__ __forceinline__ bool wait_warp(SmemCtl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    const bool ok = wait_or_abort(ctl, bar, parity, status);
    return __all_sync(0xffffffffu, ok);
}

// Index of this thread's key (or -1 past the end of the split).
__device__ __forceinline__ int32_t load_index(const int32_t* idx_row, int pos, int key_end) {
    return pos < key_end ? __ldg(idx_row + pos) : -1;
}

// Start the asynchronous copy of this thread's 16-byte chunks (j = q, q+4, ...) of one key's
// raw record into its slot, or nothing for a masked key. Always commits a group, so the group
// count stays one per tile.
template <int R, bool kWhole>
__device__ __forceinline__ void issue_raw(const KernelArgs& a, int32_t index, uint32_t slot_saddr, int q) {
    using S = RawSlot<R, kWhole>;
    if (index >= 0 && index < a.num_slots) {
        const uint8_t* rec = a.cache + static_cast<int64_t>(index) * R;
#pragma unroll
        for (int j = q; j < S::kChunks; j += 4) cp_async16(slot_saddr + 16 * j, rec + S::src_offset(j));
    }
    cp_async_commit();
}

// Convert this thread's part of one key from its raw slot into the bf16 tile: the 16-wide NoPE
// blocks 4c+q (c = 0..7) and, with kRope, RoPE dims [16q, 16q+16). A masked key writes zeros.
template <int R, bool kRope>
__device__ __forceinline__ void convert_part(const uint8_t* slot, bool valid, uint8_t* tile, int key, int q) {
    using S = RawSlot<R, kRope>;
    if (valid) {
        uint32_t sw[8];
        if constexpr (R == 352) {
            // blocks 4c+q have their scales at bytes 8q + c of the scale field (permuted layout):
            // one 8-byte load
            const uint2 s8 = *reinterpret_cast<const uint2*>(slot + S::kScaleOffset + 8 * q);
#pragma unroll
            for (int c = 0; c < 8; ++c) sw[c] = ((c < 4 ? s8.x : s8.y) >> (8 * (c & 3))) & 0xFFu;
        } else {
            const uint4 s0 = *reinterpret_cast<const uint4*>(slot + S::kScaleOffset);
            const uint4 s1 = *reinterpret_cast<const uint4*>(slot + S::kScaleOffset + 16);
            const uint32_t w[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int c = 0; c < 8; ++c) sw[c] = (w[c] >> (8 * q)) & 0xFFu;   // byte 4c + q
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint2 codes = *reinterpret_cast<const uint2*>(slot + 32 * c + 8 * q);
            uint4 lo, hi;
            dq_block(codes, sw[c], lo, hi);
            *reinterpret_cast<uint4*>(tile + c * kBlkBytes + swz(key, 2 * q)) = lo;
            *reinterpret_cast<uint4*>(tile + c * kBlkBytes + swz(key, 2 * q + 1)) = hi;
        }
        if constexpr (kRope) {
            uint4 r0, r1;
            if constexpr (R == 352) {
                const uint4 e = *reinterpret_cast<const uint4*>(slot + 256 + 16 * q);
                r0 = make_uint4(dq_e4m3x2(e.x), dq_e4m3x2(e.x >> 16), dq_e4m3x2(e.y), dq_e4m3x2(e.y >> 16));
                r1 = make_uint4(dq_e4m3x2(e.z), dq_e4m3x2(e.z >> 16), dq_e4m3x2(e.w), dq_e4m3x2(e.w >> 16));
            } else {
                r0 = *reinterpret_cast<const uint4*>(slot + 304 + 32 * q);
                r1 = *reinterpret_cast<const uint4*>(slot + 304 + 32 * q + 16);
            }
            *reinterpret_cast<uint4*>(tile + 8 * kBlkBytes + swz(key, 2 * q)) = r0;
            *reinterpret_cast<uint4*>(tile + 8 * kBlkBytes + swz(key, 2 * q + 1)) = r1;
        }
    } else {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < (kRope ? 9 : 8); ++c) {
            *reinterpret_cast<uint4*>(tile + c * kBlkBytes + swz(key, 2 * q)) = z;
            *reinterpret_cast<uint4*>(tile + c * kBlkBytes + swz(key, 2 * q + 1)) = z;
        }
    }
}

// Gather/dequant warps (256 threads, t = 0..255): 4 threads per key, one 64-key tile per
// iteration. Raw records are copied with cp.async kRawStages tiles ahead into a ring of raw
// slots; each iteration waits for its own tile's copies, then converts into stage
// i % kStages of `ring` once the consumer released it (`empty`), and arrives on `full`.
// With kRope (CTA 0: whole records, RoPE included) the used-key mask of each tile is also
// published (mask ring + mfull) and K stages are only written once Q has left them (qready).
template <int R, bool kRope, int kStages, int kStageBytes>
__device__ __forceinline__ void gather_dequant(const KernelArgs& a, SmemCtl* ctl, uint8_t* ring, uint8_t* raw,
                                               uint64_t* full, uint64_t* empty, const int32_t* idx_row,
                                               int key_begin, int key_end, int n_tiles, int t) {
    using S = RawSlot<R, kRope>;
    const int key = t >> 2;
    const int q = t & 3;
    const int wq = t >> 5;
    const int lane = t & 31;
    auto pos_of = [&](int i) { return key_begin + kTile * i + key; };
    const uint32_t raw_key = smem_addr(raw) + key * S::kKeyBytes;
    int32_t ix[kRawStages + 1];
#pragma unroll
    for (int k = 0; k < kRawStages; ++k) {
        ix[k] = load_index(idx_row, pos_of(k), key_end);
        issue_raw<R, kRope>(a, k < n_tiles ? ix[k] : -1, raw_key + k * S::kTileBytes, q);
    }
    ix[kRawStages] = load_index(idx_row, pos_of(kRawStages), key_end);
    for (int i = 0; i < n_tiles; ++i) {
        const int ks = i % kStages;
        const int rs = i % kRawStages;
        const int32_t index = ix[0];
        if (kRope && q == 0 && index >= a.num_slots && a.status != nullptr) atomicOr(a.status, 0x2u);
        const bool valid = index >= 0 && index < a.num_slots;
        cp_async_wait<kRawStages - 1>();      // this thread's copies of tile i have landed
        __syncwarp();                          // ... and those of the 3 other threads of its key
        if (i >= kStages && !wait_warp(ctl, &empty[ks], ((i - kStages) / kStages) & 1, a.status)) break;
        if (kRope && i == 0 && !wait_warp(ctl, &ctl->qready, 0, a.status)) break;   // K stages held Q
        convert_part<R, kRope>(raw + rs * S::kTileBytes + key * S::kKeyBytes, valid, ring + ks * kStageBytes, key, q);
        if constexpr (kRope) {
            const uint32_t used = __ballot_sync(0xffffffffu, valid);
            if (lane == 0) {
                uint32_t m = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) m |= ((used >> (4 * k)) & 1u) << k;
                ctl->mask[i % kMaskSlots][wq] = static_cast<uint8_t>(m);
                mbar_arrive(&ctl->mfull[i % kMaskSlots]);
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&full[ks]);
        // the raw slot of tile i is free: start tile i + kRawStages there
        __syncwarp();
        const int nx = i + kRawStages;
        issue_raw<R, kRope>(a, nx < n_tiles ? ix[kRawStages] : -1, raw_key + rs * S::kTileBytes, q);
#pragma unroll
        for (int k = 0; k < kRawStages; ++k) ix[k] = ix[k + 1];
        ix[kRawStages] = load_index(idx_row, pos_of(nx + 1), key_end);
    }
    cp_async_wait<0>();
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// CTA 1, warps 0-3 (thread h = TMEM lane h): O * factor for the row's 128 x 512 block, written
// out (bf16 `out` when there is one split, fp32 partial otherwise) through shared memory so
// that every warp store covers whole 128-byte lines. Four quarters of 128 columns, staged in
// the two V stages alternately (row h at h * 512, 16-byte chunk k at slot k ^ (h & 7)).
__device__ __forceinline__ void write_rows(const KernelArgs& a, uint8_t* smem, uint32_t lane_base, bool use_o,
                                           float factor, int row, int split, int warp, int lane, int h) {
#pragma unroll 1
    for (int qt = 0; qt < 4; ++qt) {
        uint8_t* buf = smem + kOffV + (qt & 1) * kVTileBytes;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            if (use_o) {
                tmem_ld32(lane_base + kColO + 128 * qt + 32 * c, o);
                tmem_wait_ld();
            }
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                float4 w;
                w.x = use_o ? __uint_as_float(o[4 * v + 0]) * factor : 0.0f;
                w.y = use_o ? __uint_as_float(o[4 * v + 1]) * factor : 0.0f;
                w.z = use_o ? __uint_as_float(o[4 * v + 2]) * factor : 0.0f;
                w.w = use_o ? __uint_as_float(o[4 * v + 3]) * factor : 0.0f;
                *reinterpret_cast<float4*>(buf + h * 512 + (((8 * c + v) ^ (h & 7)) << 4)) = w;
            }
        }
        named_bar_sync(1, 128);
        const int nrows = min(32, a.h_q - 32 * warp);
        if (a.splits == 1) {
            __nv_bfloat16* dst = a.out + (static_cast<int64_t>(row) * a.h_q + 32 * warp) * 512 + 128 * qt + 4 * lane;
#pragma unroll 4
            for (int r = 0; r < nrows; ++r) {
                const int hh = 32 * warp + r;
                const float4 x = *reinterpret_cast<const float4*>(buf + hh * 512 + ((lane ^ (hh & 7)) << 4));
                *reinterpret_cast<uint2*>(dst + static_cast<int64_t>(r) * 512) =
                    make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
            }
        } else {
            float* dst = a.part_out + ((static_cast<int64_t>(row) * a.splits + split) * a.h_q + 32 * warp) * 512 +
                         128 * qt + 4 * lane;
#pragma unroll 4
            for (int r = 0; r < nrows; ++r) {
                const int hh = 32 * warp + r;
                *reinterpret_cast<float4*>(dst + static_cast<int64_t>(r) * 512) =
                    *reinterpret_cast<const float4*>(buf + hh * 512 + ((lane ^ (hh & 7)) << 4));
            }
        }
    }
}

template <int R>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) sparse_decode_kernel(const KernelArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem);

    const int crank = static_cast<int>(cluster_ctarank());   // 0: QK + softmax, 1: PV
    const int pair = blockIdx.x >> 1;
    const int split = pair % a.splits;
    const int row = pair / a.splits;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int key_begin = split * a.keys_per_split;
    const int key_end = min(a.topk, key_begin + a.keys_per_split);
    const int n_tiles = key_end > key_begin ? (key_end - key_begin + kTile - 1) / kTile : 0;
    const int32_t* idx_row = a.indices + static_cast<int64_t>(row) * a.topk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&ctl->kfull[i], 256);
            mbar_init(&ctl->kempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->sfull[i], 1);
            mbar_init(&ctl->sfree[i], 128);
            mbar_init(&ctl->vfull[i], 256);
            mbar_init(&ctl->vempty[i], 1);
            mbar_init(&ctl->odone[i], 1);
        }
        for (int i = 0; i < kMaskSlots; ++i) mbar_init(&ctl->mfull[i], 8);
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(&ctl->pempty[i], 1);
            mbar_init(&ctl->pfull[i], 4);
            mbar_init(&ctl->ready[i], 128);
        }
        mbar_init(&ctl->qready, 128);
        mbar_init(&ctl->fin, 4);
        mbar_init(&ctl->drain, crank == 0 ? 2 : 1);
        ctl->abort = 0u;
        fence_barrier_init();
    }
    if (warp == 12) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;
    asm volatile("griddepcontrol.launch_dependents;");   // the split merge may be scheduled now
    // Every thread arrives on the cluster barrier now (barriers of both CTAs initialized); only
    // the threads that touch the peer CTA wait on it before their first remote access, the
    // others at exit.
    cluster_arrive();

    if (crank == 0) {
        // Q [128 x 576] bf16 is staged through the two K stages (exactly 144 KB) with coalesced
        // loads by every thread; row h's 16-byte chunk c sits at h*1152 + (c ^ (h & 7))*16 so the
        // row reads below are conflict-free. The K stages are written only after qready.
        uint8_t* sQ = smem + kOffK;
        {
            const uint4* src = reinterpret_cast<const uint4*>(a.q + static_cast<int64_t>(row) * a.h_q * kDqk);
            for (int g = threadIdx.x; g < kHeadsM * (kDqk / 8); g += kThreads) {
                const int hh = g / (kDqk / 8), c = g % (kDqk / 8);
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                if (hh < a.h_q) x = __ldg(src + g);
                *reinterpret_cast<uint4*>(sQ + hh * (kDqk * 2) + ((c ^ (hh & 7)) << 4)) = x;
            }
        }
        __syncthreads();
        if (warp < 4) {
            // ============ CTA 0, warps 0-3: Q into TMEM, then the softmax ============
            const int h = threadIdx.x;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
            {
                const uint8_t* qrow = sQ + h * (kDqk * 2);
#pragma unroll 1
                for (int c = 0; c < 9; ++c) {          // 9 x 64 dims = 9 x 32 columns
                    uint32_t v[32];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 x = *reinterpret_cast<const uint4*>(qrow + (((8 * c + j) ^ (h & 7)) << 4));
                        v[4 * j] = x.x;
                        v[4 * j + 1] = x.y;
                        v[4 * j + 2] = x.z;
                        v[4 * j + 3] = x.w;
                    }
                    tmem_st32(lane_base + kColQ + 32 * c, v);
                }
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(&ctl->qready);
            }
            cluster_wait();
            // row h of CTA 1's P slot 0 (128B-swizzled K-major rows; chunk c at (c ^ (h & 7)) * 16)
            const uint32_t peer_p = mapa_shared(smem_addr(smem + kOffP) + (h >> 3) * 1024 + (h & 7) * 128, 1);
            const uint32_t peer_alpha = mapa_shared(smem_addr(smem + kOffAlpha) + 4 * h, 1);
            const uint32_t peer_fin = mapa_shared(smem_addr(smem + kOffFin) + 8 * h, 1);
            const uint32_t peer_pfull0 = mapa_shared(smem_addr(&ctl->pfull[0]), 1);
            const uint32_t peer_finbar = mapa_shared(smem_addr(&ctl->fin), 1);
            float m_ref = -INFINITY;   // reference max, log2 units of scaled logits
            float l = 0.0f;            // sum of 2^(s - m_ref) over used keys
            bool ok = true;
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int b = i & 1;
                ok = wait_warp(ctl, &ctl->sfull[b], (i >> 1) & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                uint32_t s[64];
                tmem_ld32(lane_base + kColS + 64 * b, *reinterpret_cast<uint32_t(*)[32]>(s));
                tmem_ld32(lane_base + kColS + 64 * b + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
                tmem_wait_ld();
                tc_fence_before_sync();
                mbar_arrive(&ctl->sfree[b]);
                ok = wait_warp(ctl, &ctl->mfull[i % kMaskSlots], (i / kMaskSlots) & 1, a.status);
                if (!ok) break;
                const uint64_t used = *reinterpret_cast<const volatile uint64_t*>(ctl->mask[i % kMaskSlots]);
                // ---- online softmax (log2 domain, lazy reference max): z = s * scale_log2.
                // Common case (every key used, scale > 0): the max is taken on the raw scores and
                // each z - m is one fused multiply-add; otherwise masked keys become -inf first.
                float zs = a.scale_log2;      // multiplier applied to s[] below
                float tile_max;
                if (used == ~0ull && zs > 0.0f) {
                    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
                        m0 = fmax3(m0, __uint_as_float(s[j]), __uint_as_float(s[j + 1]));
                        m1 = fmax3(m1, __uint_as_float(s[j + 2]), __uint_as_float(s[j + 3]));
                    }
                    tile_max = fmaxf(m0, m1) * zs;
                } else {
                    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 64; j += 2) {
                        const float v0 = ((used >> j) & 1ull) ? __uint_as_float(s[j]) * zs : -INFINITY;
                        const float v1 = ((used >> (j + 1)) & 1ull) ? __uint_as_float(s[j + 1]) * zs : -INFINITY;
                        s[j] = __float_as_uint(v0);
                        s[j + 1] = __float_as_uint(v1);
                        m0 = fmaxf(m0, v0);
                        m1 = fmaxf(m1, v1);
                    }
                    tile_max = fmaxf(m0, m1);
                    zs = 1.0f;
                }
                float alpha = 1.0f;
                if (tile_max > m_ref + kRescaleThreshold) {
                    if (m_ref != -INFINITY) alpha = ex2_approx(m_ref - tile_max);
                    m_ref = tile_max;
                }
                uint32_t p[32];
                if (m_ref != -INFINITY) {
                    const uint64_t mul2 = f32x2_pack(zs, zs);
                    const uint64_t neg_m2 = f32x2_pack(-m_ref, -m_ref);
                    uint64_t la = f32x2_pack(0.0f, 0.0f), lb = la;
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
                        const float2 z0 = f32x2_unpack(
                            f32x2_fma(f32x2_pack(__uint_as_float(s[j]), __uint_as_float(s[j + 1])), mul2, neg_m2));
                        const float2 z1 = f32x2_unpack(
                            f32x2_fma(f32x2_pack(__uint_as_float(s[j + 2]), __uint_as_float(s[j + 3])), mul2, neg_m2));
                        const float p0 = ex2_approx(z0.x), p1 = ex2_approx(z0.y);
                        const float p2 = ex2_approx(z1.x), p3 = ex2_approx(z1.y);
                        la = f32x2_add(la, f32x2_pack(p0, p1));
                        lb = f32x2_add(lb, f32x2_pack(p2, p3));
                        p[j / 2] = pack_bf16x2(p0, p1);
                        p[j / 2 + 1] = pack_bf16x2(p2, p3);
                    }
                    const float2 sa = f32x2_unpack(la), sb = f32x2_unpack(lb);
                    l = l * alpha + ((sa.x + sa.y) + (sb.x + sb.y));
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) p[j] = 0u;
                }
                // ---- P row h and alpha -> CTA 1's slot (i % kPStages), once its PV released it
                const int ps = i % kPStages;
                if (i >= kPStages) {
                    ok = wait_warp(ctl, &ctl->pempty[ps], ((i / kPStages) - 1) & 1, a.status);
                    if (!ok) break;
                }
                const uint32_t dst = peer_p + ps * kPBytes;
                const uint32_t bar = peer_pfull0 + 8 * ps;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_async_u4(dst + ((c ^ (h & 7)) << 4),
                                make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]), bar);
                st_async_f32(peer_alpha + ps * kHeadsM * 4, alpha, bar);
            }
            // ---- running max and sum to CTA 1, which writes out and lse
            if (ok) st_async_v2(peer_fin, m_ref, l, peer_finbar);
        } else if (warp < 12) {
            // ============ CTA 0, warps 4-11: gather/dequant of whole records ============
            gather_dequant<R, true, kKStages, kKTileBytes>(a, ctl, smem + kOffK, smem + kOffRaw0, ctl->kfull,
                                                           ctl->kempty, idx_row, key_begin, key_end, n_tiles,
                                                           threadIdx.x - 128);
        } else {
            // ============ CTA 0, warps 12-13: QK issuers (warp 12 even tiles, warp 13 odd tiles) ============
            const uint32_t idesc_qk = idesc_bf16_f32(kHeadsM, kTile, false, false);
            const uint64_t kdesc0 = sdesc_sw128(smem_addr(smem + kOffK), 16, 1024);
            const bool leader = elect_one_in_warp();
            bool ok = wait_warp(ctl, &ctl->qready, 0, a.status);
            for (int i = warp - 12; i < n_tiles && ok; i += 2) {
                const int ks = i % kKStages;
                const int b = i & 1;
                ok = wait_warp(ctl, &ctl->kfull[ks], (i / kKStages) & 1, a.status);
                if (ok && i >= 2) ok = wait_warp(ctl, &ctl->sfree[b], ((i - 2) >> 1) & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                if (leader) {
                    const uint64_t kd = kdesc0 + static_cast<uint64_t>((ks * kKTileBytes) >> 4);
                    const uint32_t d = tmem + kColS + 64 * b;
#pragma unroll
                    for (int kk = 0; kk < 36; ++kk)
                        mma_ts(d, tmem + kColQ + 8 * kk, kd + (((kk >> 2) * kBlkBytes + (kk & 3) * 32) >> 4), idesc_qk,
                               kk > 0 ? 1u : 0u);
                    mma_commit(&ctl->kempty[ks]);
                    mma_commit(&ctl->sfull[b]);
                }
                __syncwarp();
            }
            if (leader) mma_commit(&ctl->drain);
            __syncwarp();
            if (!mbar_wait(&ctl->drain, 0)) set_abort(ctl, a.status);
        }
    } else {
        if (warp < 4) {
            // ============ CTA 1, warps 0-3: per-tile alpha check / O rescale, then the output ============
            const int h = threadIdx.x;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
            const float* s_alpha = reinterpret_cast<const float*>(smem + kOffAlpha);
            bool ok = true;
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int ps = i % kPStages;
                if (lane == 0) mbar_arrive_expect_tx(&ctl->pfull[ps], 32 * (128 + 4));
                ok = wait_warp(ctl, &ctl->pfull[ps], (i / kPStages) & 1, a.status);
                if (!ok) break;
                const float alpha = s_alpha[ps * kHeadsM + h];
                if (__any_sync(0xffffffffu, alpha != 1.0f) && i > 0) {
                    ok = wait_warp(ctl, &ctl->odone[(i - 1) & 1], ((i - 1) >> 1) & 1, a.status);
                    if (!ok) break;
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < 16; ++c) {
                        uint32_t o[32];
                        tmem_ld32(lane_base + kColO + 32 * c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        tmem_st32(lane_base + kColO + 32 * c, o);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();     // P written by the peer's st.async, read by the MMA
                tc_fence_before_sync();
                mbar_arrive(&ctl->ready[ps]);
            }
            // ---- output
            if (lane == 0) mbar_arrive_expect_tx(&ctl->fin, 32 * 8);
            const bool have_fin = ok && wait_warp(ctl, &ctl->fin, 0, a.status);
            bool have_o = false;
            if (have_fin && n_tiles > 0) {
                have_o = wait_warp(ctl, &ctl->odone[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, a.status);
                if (have_o) tc_fence_after_sync();
            }
            float m_ref = -INFINITY, l = 0.0f;
            if (have_fin) {
                const float2 f = *reinterpret_cast<const float2*>(smem + kOffFin + 8 * h);
                m_ref = f.x;
                l = f.y;
            }
            const bool empty = !(l > 0.0f);
            const float lse2 = empty ? -INFINITY : m_ref + log2f(l);   // log2 units
            float factor = 0.0f;
            if (!empty) {
                float denom = l;
                if (a.splits == 1 && a.sink != nullptr)
                    denom += exp2f(__ldg(a.sink + (h < a.h_q ? h : 0)) * kLog2e - m_ref);
                factor = 1.0f / denom;
            }
            if (h < a.h_q) {
                if (a.splits == 1)
                    a.lse[static_cast<int64_t>(row) * a.h_q + h] = lse2 * kLn2;
                else
                    a.part_lse[(static_cast<int64_t>(row) * a.splits + split) * a.h_q + h] = lse2;
            }
            write_rows(a, smem, lane_base, have_o && !empty, factor, row, split, warp, lane, h);
        } else if (warp < 12) {
            // ============ CTA 1, warps 4-11: gather/dequant of the NoPE halves (V) ============
            gather_dequant<R, false, kVStages, kVTileBytes>(a, ctl, smem + kOffV, smem + kOffRaw1, ctl->vfull,
                                                            ctl->vempty, idx_row, key_begin, key_end, n_tiles,
                                                            threadIdx.x - 128);
        } else if (warp == 12) {
            // ============ CTA 1, warp 12: PV issuer (warp 13 idle) ============
            cluster_wait();          // CTA 0's pempty barriers exist before the first multicast commit
            const uint32_t idesc_pv = idesc_bf16_f32(kHeadsM, 256, false, true);
            const uint64_t pdesc0 = sdesc_sw128(smem_addr(smem + kOffP), 16, 1024);
            const uint64_t vdesc0 = sdesc_sw128(smem_addr(smem + kOffV), kBlkBytes, 1024);
            const bool leader = elect_one_in_warp();
            bool ok = true;
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int vs = i % kVStages;
                const int ps = i % kPStages;
                ok = wait_warp(ctl, &ctl->vfull[vs], (i / kVStages) & 1, a.status);
                if (ok) ok = wait_warp(ctl, &ctl->ready[ps], (i / kPStages) & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                if (leader) {
                    const uint64_t pd = pdesc0 + static_cast<uint64_t>((ps * kPBytes) >> 4);
                    const uint64_t vd = vdesc0 + static_cast<uint64_t>((vs * kVTileBytes) >> 4);
#pragma unroll
                    for (int half = 0; half < 2; ++half)
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ss(tmem + kColO + 256 * half, pd + ((kk * 32) >> 4),
                                   vd + ((half * 4 * kBlkBytes + kk * 2048) >> 4), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&ctl->vempty[vs]);
                    mma_commit(&ctl->odone[i & 1]);
                    mma_commit_multicast(&ctl->pempty[ps], 0x1);
                }
                __syncwarp();
            }
            if (leader) mma_commit(&ctl->drain);
            __syncwarp();
            if (!mbar_wait(&ctl->drain, 0)) set_abort(ctl, a.status);
        }
    }

    // threads that have not waited on the prologue's cluster phase do so now
    const bool waited = (crank == 0 && warp < 4) || (crank == 1 && warp == 12);
    if (!waited) cluster_wait();
    tc_fence_before_sync();
    cluster_sync();          // no CTA leaves while its peer may still touch its shared memory
    if (warp == 12) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Split merge, one CTA per (query row, head), launched as a programmatic dependent of the
// decode kernel: out = sum_s w_s part_s with w_s = 2^{lse2_s} / (sum_s 2^{lse2_s} + e^{sink}),
// lse = ln sum_s e^{lse_s} (the sink is not part of lse). lse2 = log2-domain partial lse.
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ part_out,
                                                      const float* __restrict__ part_lse, int splits, int h_q,
                                                      const float* __restrict__ sink, __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the decode grid's partials are visible
    const int rh = blockIdx.x;             // row * h_q + h
    const int row = rh / h_q;
    const int h = rh % h_q;
    const int64_t base = static_cast<int64_t>(row) * splits;
    float m = -INFINITY;
    for (int p = 0; p < splits; ++p) m = fmaxf(m, part_lse[(base + p) * h_q + h]);
    const int d0 = threadIdx.x * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float total = -INFINITY;
    if (m != -INFINITY) {
        float sum = 0.0f;
        for (int p = 0; p < splits; ++p) sum += exp2f(part_lse[(base + p) * h_q + h] - m);
        total = (m + log2f(sum)) * kLn2;
        const float inv = 1.0f / (sum + (sink != nullptr ? exp2f(__ldg(sink + h) * kLog2e - m) : 0.0f));
        for (int p = 0; p < splits; ++p) {
            const int64_t ph = (base + p) * h_q + h;
            const float w = exp2f(part_lse[ph] - m) * inv;
            const float4 v = *reinterpret_cast<const float4*>(part_out + ph * 512 + d0);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
    }
    *reinterpret_cast<uint2*>(out + static_cast<int64_t>(rh) * 512 + d0) =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
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
    // the merge launches while the decode grid runs and waits for it on the device
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(d.rows) * static_cast<unsigned>(d.h_q));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, static_cast<const float*>(d.part_out),
                              static_cast<const float*>(d.part_lse), d.splits, d.h_q, d.attn_sink,
                              static_cast<__nv_bfloat16*>(d.out), d.lse);
}

}  // namespace nvfp4mla
