// sparse_decode.cu -- read side: sparse MLA decode over NVFP4 records (and the split merge).
//
// What is computed (FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode",
// "Kernel:" paragraph and validation list): for query row t and head h, with J the used
// entries of t's index list,
//     z_j = sm_scale * q[t,h,:] . K_j          (K_j: 576 dequantized values of record j)
//     out = sum_j e^{z_j} V_j / (sum_j e^{z_j} + e^{sink_h}),   V_j = K_j[0:512]
//     lse = ln sum_j e^{z_j}
// Keys are dequantized in shared memory, exactly (e2m1 x e4m3 has <= 5 significant bits): to
// bf16 for QK^T (q is bf16) and to f16 for PV (P in f16 keeps 11 significant bits); both
// contractions run as tcgen05 16-bit MMAs with fp32 accumulation in tensor memory.
//
// Work split: a cluster of two CTAs per (query row, top-k split), with different roles.
// With 128 heads, the fp32 accumulator O [128 x 512] fills all 512 TMEM columns of an SM, so
// QK^T and PV run on different SMs and only the 16-bit P tile travels between them:
//   CTA 0 (QK): keeps Q [128 x 576] in TMEM as the MMA A operand (loaded by nine TMA boxes),
//     dequantizes K tiles (576 dims), computes S = Q K^T, runs the online softmax, and sends
//     each row's P (f16) and rescale factor to CTA 1 with st.async (DSMEM, one way:
//     132 B per head per 64 keys; each store instruction covers 8 rows x 64 B).
//   CTA 1 (PV): dequantizes V tiles (the 512 NoPE dims of the same records), keeps O in
//     TMEM and computes O += P V with P read from shared memory; its MMA commit multicasts
//     back to CTA 0 to release the P slot. At the end CTA 0 sends each row's running max and
//     sum, and CTA 1 normalizes, writes `out` (or the split's partial) and `lse`.
// Warp roles (kThreads = 896 threads, 28 warps):
//   both:  warps 8-23 convert (8 threads per key of a 64-key tile), warps 26-27 gather
//          records with TMA tile::gather4 into a ring of raw tiles (CTA 0: three for 352-B
//          records, two for 432-B, one for 656-B; CTA 1: two, one for 656-B) and publish the
//          used-key bits of each
//          tile; warp 24 owns tensor memory.
//   CTA 0: warps 0-7 softmax (warp w: TMEM lanes 32 (w & 3).., score columns 32 (w >> 2)..+32;
//          the two column halves exchange tile maxima), warps 24-25 QK issuers (even / odd
//          tiles; one elected lane each).
//   CTA 1: warps 0-3 rescale O (thread r = TMEM lane r), warps 0-7 stage the output, warp 24
//          PV issuer; the converter warps copy the staged output out.
// Tiles are 64 keys; every K/V tile is written in a 128B-swizzled layout that is the K-major
// B operand of QK (CTA 0) or the MN-major B operand of PV (CTA 1).
//
// Every wait is bounded: on timeout the CTA sets NVFP4_MLA_DEV_TIMEOUT, stops issuing work,
// waits (bounded) for its MMAs to drain and frees its tensor memory before returning.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
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
constexpr int kPStages = 2;                        // CTA 1: P tiles [128 heads x 64 keys] f16
constexpr int kPBytes = kHeadsM * 128;             // 16 KB
// Raw-record ring, filled by TMA tile::gather4 (four whole records per instruction, each group of
// four starting on a 128-byte boundary): CTA 0 keeps 3 tiles in flight for 352-byte records and
// 2 for 432-byte records, CTA 1 keeps 2. A 64-key tile of 656-byte fp8 records takes 42 KB, so
// each CTA holds one; its converters hand the slot back as soon as the bytes are in registers.
template <int R>
struct RawRing {
    static constexpr int kGroupBytes = (4 * R + 127) / 128 * 128;   // 1408 | 1792 | 2688
    static constexpr int kTileBytes = 16 * kGroupBytes;             // 64 keys
    static constexpr int kStages0 = R == 352 ? 3 : R == 432 ? 2 : 1;
    static constexpr int kStages1 = R == 656 ? 1 : 2;
    static __device__ __forceinline__ int key_offset(int key) { return (key >> 2) * kGroupBytes + (key & 3) * R; }
};
constexpr int kProducerWarps = 2;
constexpr int kMaxRawStages = 3;
constexpr uint32_t kColS = 0;                      // CTA 0: S buffers [0,64), [64,128)
constexpr uint32_t kColQ = 128;                    // CTA 0: Q, 576 bf16 = 288 columns
constexpr uint32_t kColO = 0;                      // CTA 1: O, 512 columns
constexpr int kTmemCols = 512;
constexpr int kThreads = 896;                      // 28 warps, roles below
constexpr int kConvWarps = 16;                     // converter warps: 8 threads per key of a 64-key tile
constexpr int kWarpConv0 = 8;                      // first converter warp
constexpr int kWarpMma = 24;                       // QK issuers 24-25 (CTA 0), PV issuer 24 (CTA 1); TMEM owner
constexpr int kWarpProd = 26;                      // producer warps 26-27
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
    uint64_t pempty[kPStages];    // CTA 1's PV has read the P slot (multicast commit)
    uint64_t qload;               // CTA 0: Q's nine 64-column boxes landed in shared memory (TMA)
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
    uint64_t rawfull[kMaxRawStages];    // producer warps: expect_tx + gather4 bytes -> converters
    uint64_t rawempty[kMaxRawStages];   // converter warps (one arrival each) -> producers
    uint32_t rawvalid[kMaxRawStages][2];   // used-key bits of the tile in each raw slot
    uint64_t xbar[2];             // CTA 0: both softmax halves posted their tile max (tile parity)
    uint64_t lbar;                // CTA 0: softmax half 1 posted its final row sum
    uint32_t tmem_base;
    uint32_t abort;
};

constexpr int kCtlBytes = 1024;
static_assert(sizeof(SmemCtl) <= kCtlBytes, "control block");
// CTA 0 data
constexpr int kOffK = kCtlBytes;
// CTA 1 data
constexpr int kOffV = kCtlBytes;
constexpr int kOffP = kOffV + kVStages * kVTileBytes;
constexpr int kOffAlpha = kOffP + kPStages * kPBytes;          // [kPStages][128] fp32
constexpr int kOffFin = kOffAlpha + kPStages * kHeadsM * 4;    // [128] (max, sum) pairs
constexpr int kOffRaw0 = kOffK + kKStages * kKTileBytes;        // CTA 0 raw ring
constexpr int kOffRaw1 = kOffFin + kHeadsM * 8;                 // CTA 1 raw ring
constexpr int kXchgBytes = (2 * 2 + 1) * kHeadsM * 4;          // CTA 0: [parity][half][128] maxima, [128] sums
template <int R>
struct SmemSize {
    static constexpr int xchg0 = kOffRaw0 + RawRing<R>::kStages0 * RawRing<R>::kTileBytes;   // CTA 0 exchange
    static constexpr int c0 = xchg0 + kXchgBytes;
    static constexpr int c1 = kOffRaw1 + RawRing<R>::kStages1 * RawRing<R>::kTileBytes;
    static constexpr int value = 1024 + (c0 > c1 ? c0 : c1);
};
static_assert(SmemSize<352>::value <= 232448 && SmemSize<432>::value <= 232448 && SmemSize<656>::value <= 232448,
              "shared memory");
static_assert(kOffRaw0 % 128 == 0 && kOffRaw1 % 128 == 0, "gather4 destinations are 128-byte aligned");

struct KernelArgs {
    CUtensorMap tmap;            // the cache as u32 [num_slots, R / 4], box one record
    CUtensorMap qmap;            // q as bf16 [rows * h_q, 576], box 64 columns x 128 heads, 128B swizzle
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
    uint16_t* part_out;          // f16 partial outputs [rows, splits, h_q, 512]
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

// P entries lie in [0, 2^8] (lazy reference max), so f16 holds them with 11 significant bits.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
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

// Two e2m1 codes times a scale -> f16x2 (exact: the products need at most 5 significant bits and
// lie in [2^-10, 2688], inside the f16 normal range).
__device__ __forceinline__ uint32_t dq_e2m1x2_f16(uint32_t byte, __half2 scale2) {
    uint32_t h;
    asm("{\n"
        "  .reg .b8 t;\n"
        "  cvt.u8.u32 t, %1;\n"
        "  cvt.rn.f16x2.e2m1x2 %0, t;\n"
        "}\n"
        : "=r"(h)
        : "r"(byte));
    const __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h), scale2);
    return *reinterpret_cast<const uint32_t*>(&v);
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
// kF16: f16 output (the PV operand), else bf16 (the QK operand).
template <bool kF16>
__device__ __forceinline__ uint32_t dq_pair(uint32_t byte, __half2 scale2) {
    if constexpr (kF16)
        return dq_e2m1x2_f16(byte, scale2);
    else
        return dq_e2m1x2(byte, scale2);
}

template <bool kF16>
__device__ __forceinline__ void dq_block(uint2 codes, uint32_t sbyte, uint4& lo, uint4& hi) {
    const __half2 s2 = scale_half2(sbyte);
    lo.x = dq_pair<kF16>(codes.x & 0xFFu, s2);
    lo.y = dq_pair<kF16>((codes.x >> 8) & 0xFFu, s2);
    lo.z = dq_pair<kF16>((codes.x >> 16) & 0xFFu, s2);
    lo.w = dq_pair<kF16>(codes.x >> 24, s2);
    hi.x = dq_pair<kF16>(codes.y & 0xFFu, s2);
    hi.y = dq_pair<kF16>((codes.y >> 8) & 0xFFu, s2);
    hi.z = dq_pair<kF16>((codes.y >> 16) & 0xFFu, s2);
    hi.w = dq_pair<kF16>(codes.y >> 24, s2);
}

// Two e4m3 codes (low byte = even element) of a 656-byte fp8 record times its fp32 tile scale:
// each product is formed in fp32 (round to nearest) and rounded once more to bf16 (kF16 false,
// the QK operand) or f16 (kF16 true, the PV operand; NoPE magnitudes up to 65504).
template <bool kF16>
__device__ __forceinline__ uint32_t dq_e4m3x2_scaled(uint32_t two_bytes, float scale) {
    uint32_t h;
    const uint16_t in = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    const float a = __fmul_rn(f.x, scale), b = __fmul_rn(f.y, scale);
    return kF16 ? pack_f16x2(a, b) : pack_bf16x2(a, b);
}

// 16 e4m3 values (16 bytes) of one 16-wide block -> 2 x 16 bytes of bf16 (or f16).
template <bool kF16>
__device__ __forceinline__ void dq_block_fp8(uint4 codes, float scale, uint4& lo, uint4& hi) {
    lo.x = dq_e4m3x2_scaled<kF16>(codes.x, scale);
    lo.y = dq_e4m3x2_scaled<kF16>(codes.x >> 16, scale);
    lo.z = dq_e4m3x2_scaled<kF16>(codes.y, scale);
    lo.w = dq_e4m3x2_scaled<kF16>(codes.y >> 16, scale);
    hi.x = dq_e4m3x2_scaled<kF16>(codes.z, scale);
    hi.y = dq_e4m3x2_scaled<kF16>(codes.z >> 16, scale);
    hi.z = dq_e4m3x2_scaled<kF16>(codes.w, scale);
    hi.w = dq_e4m3x2_scaled<kF16>(codes.w >> 16, scale);
}

__device__ __forceinline__ void set_abort(SmemCtl* ctl, uint32_t* status) {
    if (atomicExch(&ctl->abort, 1u) == 0u && status != nullptr) atomicOr(status, 0x4u);
}

__device__ __forceinline__ bool aborted(SmemCtl* ctl) {
    return *reinterpret_cast<volatile uint32_t*>(&ctl->abort) != 0u;
}

__device__ __forceinline__ bool wait_or_abort(SmemCtl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;   // the common case: already complete
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

// Convert this thread's part of one key from its raw record in shared memory into the bf16
// tile. Eight threads share a key: thread (q, hi) = (sub & 3, sub >> 2) converts the 16-wide NoPE
// blocks 4c+q for c = 4hi..4hi+3 (their four scales are bytes 8q+4hi.. of the permuted scale field
// of a 352-byte record: one 4-byte load; with the scales in block order, as in the 432-byte record
// and the 352-byte record with kBlk, one 16-byte load of blocks 16hi..16hi+15 and a byte
// selection) and RoPE dims [8 sub, 8 sub + 8). A masked key writes zeros in a V tile and quiet
// NaNs in a K tile.
template <int R, bool kRope, bool kBlk>
__device__ __forceinline__ void convert_part(uint32_t rec, bool valid, uint32_t tile, int key, int sub) {
    const int q = sub & 3;
    const int hi = sub >> 2;
    if (valid) {
        // all shared-memory reads first (they are issued back to back), then convert and store
        uint2 codes[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) codes[j] = lds_u64(rec + 32 * (4 * hi + j) + 8 * q);
        uint32_t sw;   // four scale bytes, block 4(4hi + j) + q in byte j
        if constexpr (R == 352 && !kBlk) {
            sw = lds_u32(rec + 320 + 8 * q + 4 * hi);
        } else {
            // block order: block b at byte 320 + b (352 B) or 256 + b (432 B)
            const uint4 s4 = lds_u128(rec + (R == 352 ? 320 : 256) + 16 * hi);
            const uint32_t w[4] = {s4.x, s4.y, s4.z, s4.w};
            sw = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) sw |= ((w[j] >> (8 * q)) & 0xFFu) << (8 * j);
        }
        uint4 rope = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (kRope) {
            if constexpr (R == 352) {
                const uint2 e = lds_u64(rec + 256 + 8 * sub);
                rope.x = e.x;
                rope.y = e.y;
            } else {
                rope = lds_u128(rec + 304 + 16 * sub);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = 4 * hi + j;
            uint4 lo, hv;
            dq_block<!kRope>(codes[j], (sw >> (8 * j)) & 0xFFu, lo, hv);
            sts_u128(tile + c * kBlkBytes + swz(key, 2 * q), lo);
            sts_u128(tile + c * kBlkBytes + swz(key, 2 * q + 1), hv);
        }
        if constexpr (kRope) {
            uint4 r = rope;
            if constexpr (R == 352)
                r = make_uint4(dq_e4m3x2(rope.x), dq_e4m3x2(rope.x >> 16), dq_e4m3x2(rope.y), dq_e4m3x2(rope.y >> 16));
            sts_u128(tile + 8 * kBlkBytes + swz(key, sub), r);
        }
    } else {
        // A masked key: zeros in a V tile; quiet NaNs in a K tile, so that every score of the
        // key comes out NaN and the softmax drops it without reading a mask.
        const uint32_t f = kRope ? 0x7FC07FC0u : 0u;
        const uint4 z = make_uint4(f, f, f, f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = 4 * hi + j;
            sts_u128(tile + c * kBlkBytes + swz(key, 2 * q), z);
            sts_u128(tile + c * kBlkBytes + swz(key, 2 * q + 1), z);
        }
        if constexpr (kRope) sts_u128(tile + 8 * kBlkBytes + swz(key, sub), z);
    }
}

// Producer warps (kProducerWarps of them, pw = 0, 1): lane l < 8 of warp pw owns group
// g = 8 pw + l, keys 4g..4g+3 of every tile. For tile j the warp publishes its 32 used-key bits,
// registers the bytes it will gather on rawfull[j % kRaw] and issues one TMA gather4 per group
// with a used key (a masked row re-fetches a used row of its group, so every coordinate lies
// inside the cache; its bytes are never read), once the converters released the raw slot.
// Indices are read one tile ahead. Out-of-range indices are masked (CTA 0 reports them). Before
// returning, the warp waits for every gather it started.
template <int R, bool kRope, int kRaw>
__device__ __forceinline__ void produce_raw(const KernelArgs& a, SmemCtl* ctl, uint8_t* raw, const int32_t* idx_row,
                                            int key_begin, int key_end, int n_tiles, int pw, int lane) {
    using RR = RawRing<R>;
    const int g = 8 * pw + (lane & 7);
    auto load4 = [&](int j, int32_t (&r)[4]) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int pos = key_begin + kTile * j + 4 * g + m;
            r[m] = (lane < 8 && pos < key_end) ? __ldg(idx_row + pos) : -1;
        }
    };
    int32_t nxt[4];
    load4(0, nxt);
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
        const int rs = j % kRaw;
        int32_t r[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
        if (j + 1 < n_tiles) load4(j + 1, nxt);
        if (j >= kRaw && !wait_warp(ctl, &ctl->rawempty[rs], ((j / kRaw) - 1) & 1, a.status)) break;
        uint32_t bits = 0;
        int32_t first = -1;
#pragma unroll
        for (int m = 3; m >= 0; --m) {
            const bool ok = r[m] >= 0 && r[m] < a.num_slots;
            if (kRope && a.status != nullptr && r[m] >= a.num_slots) atomicOr(a.status, 0x2u);
            bits |= (ok ? 1u : 0u) << m;
            if (ok) first = r[m];
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (!((bits >> m) & 1u)) r[m] = first;
        const uint32_t word = __reduce_or_sync(0xffffffffu, lane < 8 ? bits << (4 * lane) : 0u);
        const uint32_t groups = __popc(__ballot_sync(0xffffffffu, lane < 8 && bits != 0u));
        if (lane == 0) {
            ctl->rawvalid[rs][pw] = word;
            mbar_arrive_expect_tx(&ctl->rawfull[rs], groups * 4u * R);
        }
        __syncwarp();
        if (lane < 8 && bits != 0u)
            tma_gather4(smem_addr(raw + rs * RR::kTileBytes + g * RR::kGroupBytes), &a.tmap, 0, r[0], r[1], r[2], r[3],
                        &ctl->rawfull[rs]);
        issued = j + 1;
    }
    // only after a timeout can gathers still be in flight here; they must land before the CTA exits
    for (int j = issued - 1; j >= 0 && j >= issued - kRaw; --j) mbar_wait(&ctl->rawfull[j % kRaw], (j / kRaw) & 1);
}

// Converter warps (kConvWarps of them, t = 0..511): eight threads per key, one 64-key tile per
// iteration. Waits for tile i's records in raw slot i % kRaw, converts them into stage
// i % kStages of `ring` once the consumer released it (`empty`), arrives on `full` and hands the
// raw slot back. With kRope (CTA 0) the K stages are written only after Q has left them (qready).
template <int R, bool kRope, bool kBlk, int kStages, int kStageBytes, int kRaw>
__device__ __forceinline__ void convert_tiles(const KernelArgs& a, SmemCtl* ctl, uint8_t* ring, uint8_t* raw,
                                              uint64_t* full, uint64_t* empty, int n_tiles, int t) {
    using RR = RawRing<R>;
    const int key = t >> 3;
    const int sub = t & 7;
    const int lane = t & 31;
    const uint32_t raw_s = smem_addr(raw);
    const uint32_t ring_s = smem_addr(ring);
    for (int i = 0; i < n_tiles; ++i) {
        const int ks = i % kStages;
        const int rs = i % kRaw;
        if (!wait_warp(ctl, &ctl->rawfull[rs], (i / kRaw) & 1, a.status)) break;
        if (i >= kStages && !wait_warp(ctl, &empty[ks], ((i - kStages) / kStages) & 1, a.status)) break;
        if (kRope && i == 0 && !wait_warp(ctl, &ctl->qready, 0, a.status)) break;   // K stages held Q
        const bool valid = ((ctl->rawvalid[rs][key >> 5] >> (key & 31)) & 1u) != 0u;
        convert_part<R, kRope, kBlk>(raw_s + rs * RR::kTileBytes + RR::key_offset(key), valid, ring_s + ks * kStageBytes,
                               key, sub);
        fence_proxy_async_smem();
        mbar_arrive(&full[ks]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->rawempty[rs]);
    }
}

// Converter warps for 656-byte fp8 records (one raw slot per CTA). Thread (q, hi) = (sub & 3,
// sub >> 2) of key `key` converts NoPE dims 64c + 16q .. +15 for c = 4hi..4hi+3 (codes at byte
// 64c + 16q, fp32 scales of tiles 2hi and 2hi + 1 at byte 512 + 8hi) and, in a K tile, RoPE dims
// [8 sub, 8 sub + 8) (bf16 at byte 528 + 16 sub). All of a tile's record bytes are loaded into
// registers first; then the warp hands the raw slot back (so the next gather overlaps the
// conversion), waits for the ring stage, converts and stores. Masked keys as in convert_part.
template <bool kRope, int kStages, int kStageBytes>
__device__ __forceinline__ void convert_tiles_fp8(const KernelArgs& a, SmemCtl* ctl, uint8_t* ring, uint8_t* raw,
                                                  uint64_t* full, uint64_t* empty, int n_tiles, int t) {
    using RR = RawRing<656>;
    const int key = t >> 3;
    const int sub = t & 7;
    const int lane = t & 31;
    const int q = sub & 3;
    const int hi = sub >> 2;
    const uint32_t rec = smem_addr(raw) + RR::key_offset(key);
    const uint32_t ring_s = smem_addr(ring);
    for (int i = 0; i < n_tiles; ++i) {
        const int ks = i % kStages;
        if (!wait_warp(ctl, &ctl->rawfull[0], i & 1, a.status)) break;
        const bool valid = ((ctl->rawvalid[0][key >> 5] >> (key & 31)) & 1u) != 0u;
        uint4 codes[4];
        uint2 sc = make_uint2(0u, 0u);
        uint4 rope = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) codes[j] = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
#pragma unroll
            for (int j = 0; j < 4; ++j) codes[j] = lds_u128(rec + 64 * (4 * hi + j) + 16 * q);
            sc = lds_u64(rec + 512 + 8 * hi);
            if constexpr (kRope) rope = lds_u128(rec + 528 + 16 * sub);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->rawempty[0]);
        if (i >= kStages && !wait_warp(ctl, &empty[ks], ((i - kStages) / kStages) & 1, a.status)) break;
        if (kRope && i == 0 && !wait_warp(ctl, &ctl->qready, 0, a.status)) break;   // K stages held Q
        const uint32_t tile = ring_s + ks * kStageBytes;
        if (valid) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 4 * hi + j;
                uint4 lo, hv;
                dq_block_fp8<!kRope>(codes[j], __uint_as_float(j < 2 ? sc.x : sc.y), lo, hv);
                sts_u128(tile + c * kBlkBytes + swz(key, 2 * q), lo);
                sts_u128(tile + c * kBlkBytes + swz(key, 2 * q + 1), hv);
            }
            if constexpr (kRope) sts_u128(tile + 8 * kBlkBytes + swz(key, sub), rope);
        } else {
            const uint32_t f = kRope ? 0x7FC07FC0u : 0u;
            const uint4 z = make_uint4(f, f, f, f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 4 * hi + j;
                sts_u128(tile + c * kBlkBytes + swz(key, 2 * q), z);
                sts_u128(tile + c * kBlkBytes + swz(key, 2 * q + 1), z);
            }
            if constexpr (kRope) sts_u128(tile + 8 * kBlkBytes + swz(key, sub), z);
        }
        fence_proxy_async_smem();
        mbar_arrive(&full[ks]);
    }
}

// One word of a chunk swap with lane ^ xor_mask: the lane gives `a` and takes the partner's
// word into `a` when give_a, else gives and takes `b`.
__device__ __forceinline__ void swap_word(uint32_t& a, uint32_t& b, bool give_a, int xor_mask) {
    const uint32_t r = __shfl_xor_sync(0xffffffffu, give_a ? a : b, xor_mask);
    a = give_a ? r : a;
    b = give_a ? b : r;
}

// In each group of four lanes (k = lane & 3) holding chunks c[0..3] of their own rows, leaves
// chunk k of lane (4a + j)'s row in c[j]: two butterfly exchanges of half the chunks each.
__device__ __forceinline__ void transpose4_chunks(uint4 (&c)[4], int lane) {
    const bool up = (lane & 2) != 0;   // lanes k, k ^ 2 swap the chunks whose bit 1 differs from k's
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        swap_word(c[m].x, c[m + 2].x, up, 2);
        swap_word(c[m].y, c[m + 2].y, up, 2);
        swap_word(c[m].z, c[m + 2].z, up, 2);
        swap_word(c[m].w, c[m + 2].w, up, 2);
    }
    const bool odd = (lane & 1) != 0;  // lanes k, k ^ 1 swap the chunks whose bit 0 differs from k's
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        swap_word(c[2 * m].x, c[2 * m + 1].x, odd, 1);
        swap_word(c[2 * m].y, c[2 * m + 1].y, odd, 1);
        swap_word(c[2 * m].z, c[2 * m + 1].z, odd, 1);
        swap_word(c[2 * m].w, c[2 * m + 1].w, odd, 1);
    }
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Output of CTA 1: O * factor for the row's 128 x 512 block goes out (bf16 `out` when there is
// one split, the split's f16 partial otherwise) through shared memory, so every warp store
// covers whole 128-byte lines. Four quarters of 128 columns are staged in the two V stages
// alternately (row h at h * 512, 16-byte chunk k at slot k ^ (h & 7)) by warps 0-7 (warps w and
// w + 4 serve TMEM lanes 32w.., each half of the columns) and copied out by the converter warps
// (one row per warp instruction), so staging of a quarter overlaps the copy of the previous
// one. Named barriers: kBarFull + b (staged -> copy) and kBarEmpty + b (copied -> restage),
// b = quarter & 1, each counting all kOutThreads threads.
constexpr int kOutThreads = 256 + 32 * kConvWarps;
constexpr uint32_t kBarFull = 2;
constexpr uint32_t kBarEmpty = 4;

__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void copy_quarter(const KernelArgs& a, const uint8_t* buf, int qt, int row, int split,
                                             int wi, int lane) {
    const uint32_t b = smem_addr(buf);
    if (a.splits == 1) {
#pragma unroll 2
        for (int hh = wi; hh < a.h_q; hh += kConvWarps) {
            const uint4 x = lds_u128(b + hh * 512 + ((lane ^ (hh & 7)) << 4));
            *reinterpret_cast<uint2*>(a.out + (static_cast<int64_t>(row) * a.h_q + hh) * 512 + 128 * qt + 4 * lane) =
                make_uint2(pack_bf16x2(__uint_as_float(x.x), __uint_as_float(x.y)),
                           pack_bf16x2(__uint_as_float(x.z), __uint_as_float(x.w)));
        }
    } else {
        uint16_t* base = a.part_out + (static_cast<int64_t>(row) * a.splits + split) * a.h_q * 512 + 128 * qt + 4 * lane;
#pragma unroll 2
        for (int hh = wi; hh < a.h_q; hh += kConvWarps) {
            const uint4 x = lds_u128(b + hh * 512 + ((lane ^ (hh & 7)) << 4));
            *reinterpret_cast<uint2*>(base + static_cast<int64_t>(hh) * 512) =
                make_uint2(pack_f16x2(__uint_as_float(x.x), __uint_as_float(x.y)),
                           pack_f16x2(__uint_as_float(x.z), __uint_as_float(x.w)));
        }
    }
}

// Warps 0-7 (TMEM lane quadrant w & 3): stage 64 of each quarter's 128 columns (from c0 * 32)
// once the copy of the quarter before last has left its buffer. use_o must be warp-uniform.
__device__ __forceinline__ void write_rows(uint8_t* smem, uint32_t lane_base, bool use_o, float factor, int h,
                                           int c0) {
#pragma unroll 1
    for (int qt = 0; qt < 4; ++qt) {
        const uint32_t buf = smem_addr(smem + kOffV + (qt & 1) * kVTileBytes);
        if (qt >= 2) named_bar_sync(kBarEmpty + (qt & 1), kOutThreads);
#pragma unroll 1
        for (int c = c0; c < c0 + 2; ++c) {
            uint32_t o[32];
            if (use_o) {
                tmem_ld32(lane_base + kColO + 128 * qt + 32 * c, o);
                tmem_wait_ld();
            }
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                uint4 w;
                w.x = __float_as_uint(use_o ? __uint_as_float(o[4 * v + 0]) * factor : 0.0f);
                w.y = __float_as_uint(use_o ? __uint_as_float(o[4 * v + 1]) * factor : 0.0f);
                w.z = __float_as_uint(use_o ? __uint_as_float(o[4 * v + 2]) * factor : 0.0f);
                w.w = __float_as_uint(use_o ? __uint_as_float(o[4 * v + 3]) * factor : 0.0f);
                sts_u128(buf + h * 512 + (((8 * c + v) ^ (h & 7)) << 4), w);
            }
        }
        named_bar_arrive(kBarFull + (qt & 1), kOutThreads);
    }
}

// Converter warps of CTA 1, once their tiles are done: copy each quarter out as it is staged.
__device__ __forceinline__ void help_write_rows(const KernelArgs& a, const uint8_t* smem, int row, int split, int wi,
                                                int lane) {
#pragma unroll 1
    for (int qt = 0; qt < 4; ++qt) {
        named_bar_sync(kBarFull + (qt & 1), kOutThreads);
        copy_quarter(a, smem + kOffV + (qt & 1) * kVTileBytes, qt, row, split, wi, lane);
        if (qt < 2) named_bar_arrive(kBarEmpty + (qt & 1), kOutThreads);
    }
}

template <int R, bool kBlk>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) sparse_decode_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, computed as an offset into the shared array so that every access
    // through `smem` stays a shared-memory access
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
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
            mbar_init(&ctl->kfull[i], 32 * kConvWarps);
            mbar_init(&ctl->kempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->sfull[i], 1);
            mbar_init(&ctl->sfree[i], 256);
            mbar_init(&ctl->vfull[i], 32 * kConvWarps);
            mbar_init(&ctl->vempty[i], 1);
            mbar_init(&ctl->odone[i], 1);
            mbar_init(&ctl->xbar[i], 256);
        }
        for (int i = 0; i < kMaxRawStages; ++i) {
            mbar_init(&ctl->rawfull[i], kProducerWarps);
            mbar_init(&ctl->rawempty[i], kConvWarps);
        }
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(&ctl->pempty[i], 1);
            mbar_init(&ctl->pfull[i], 4);
            mbar_init(&ctl->ready[i], 128);
        }
        mbar_init(&ctl->qload, 1);
        mbar_init(&ctl->qready, 256);
        mbar_init(&ctl->lbar, 128);
        mbar_init(&ctl->fin, 4);
        mbar_init(&ctl->drain, crank == 0 ? 2 : 1);
        ctl->abort = 0u;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;
    // Launched as a programmatic dependent of the preceding kernel (typically the append that
    // wrote the newest records): the prologue above overlaps its tail; nothing is read before
    // that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");   // the split merge may be scheduled now
    // Every thread arrives on the cluster barrier now (barriers of both CTAs initialized); only
    // the threads that touch the peer CTA wait on it before their first remote access, the
    // others at exit.
    cluster_arrive();

    const bool converter = warp >= kWarpConv0 && warp < kWarpConv0 + kConvWarps;
    const int conv_t = threadIdx.x - 32 * kWarpConv0;
    if (crank == 0) {
        // Q [128 x 576] bf16 is staged through the two K stages (exactly 144 KB) by nine TMA box
        // loads (64 columns x 128 heads each, 128B-swizzled: head h's 16-byte chunk c of box b at
        // b*16384 + (h >> 3)*1024 + (h & 7)*128 + (c ^ (h & 7))*16, so the row reads below are
        // conflict-free). Heads past the last query row read zeros. The K stages are written only
        // after qready.
        uint8_t* sQ = smem + kOffK;
        if (threadIdx.x == 32 * kWarpMma) {
            mbar_arrive_expect_tx(&ctl->qload, 9u * 16384u);
            for (int bx = 0; bx < 9; ++bx)
                tma_load_2d(smem_addr(sQ + bx * 16384), &a.qmap, 64 * bx, row * a.h_q, &ctl->qload);
        }
        if (warp < 8) {
            // ============ CTA 0, warps 0-7: Q into TMEM, then the softmax ============
            // Warp w serves TMEM lanes 32 (w & 3) .. +31 (thread = head h) and score columns
            // [32 half, 32 half + 32) of each tile, half = w >> 2. The halves exchange their tile
            // maxima (xbar) so both rescale identically, and merge their row sums at the end.
            const int quad = warp & 3;
            const int half = warp >> 2;
            const int h = quad * 32 + lane;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
            {
                const bool have_q = wait_warp(ctl, &ctl->qload, 0, a.status);
                const uint32_t q_s = smem_addr(sQ) + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll 1
                for (int c = half ? 5 : 0; c < (half ? 9 : 5); ++c) {   // 9 x 64 dims = 9 x 32 columns
                    uint32_t v[32];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 x = have_q ? lds_u128(q_s + c * 16384 + ((j ^ (h & 7)) << 4)) : make_uint4(0u, 0u, 0u, 0u);
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
            // 8-row atom of row h in CTA 1's P slot 0 (128B-swizzled K-major rows; chunk c of row r
            // of the atom at r * 128 + (c ^ r) * 16)
            const uint32_t peer_p_atom = mapa_shared(smem_addr(smem + kOffP) + (h >> 3) * 1024, 1);
            const uint32_t peer_alpha = mapa_shared(smem_addr(smem + kOffAlpha) + 4 * h, 1);
            const uint32_t peer_pfull0 = mapa_shared(smem_addr(&ctl->pfull[0]), 1);
            float* xmax = reinterpret_cast<float*>(smem + SmemSize<R>::xchg0);   // [parity][half][128]
            float* xsum = xmax + 4 * kHeadsM;                                      // [128]
            float m_ref = -INFINITY;   // reference max, log2 units of scaled logits (same in both halves)
            float l = 0.0f;            // this half's sum of 2^(z - m_ref) over used keys
            bool ok = true;
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int b = i & 1;
                ok = wait_warp(ctl, &ctl->sfull[b], (i >> 1) & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                uint32_t s[32];
                tmem_ld32(lane_base + kColS + 64 * b + 32 * half, s);
                tmem_wait_ld();
                tc_fence_before_sync();
                mbar_arrive(&ctl->sfree[b]);
                // ---- online softmax (log2 domain, lazy reference max): z = s * scale_log2.
                // A masked key's scores are NaN (its K row is NaN): max ignores them, and
                // max(z, -inf) turns their z into -inf, whose exponential is 0.
                float zs = a.scale_log2;      // multiplier applied to s[] below
                float part_max;
                {
                    float m0 = -INFINITY, m1 = -INFINITY;
                    if (zs > 0.0f) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            m0 = fmax3(m0, __uint_as_float(s[j]), __uint_as_float(s[j + 1]));
                            m1 = fmax3(m1, __uint_as_float(s[j + 2]), __uint_as_float(s[j + 3]));
                        }
                        part_max = fmaxf(m0, m1) * zs;
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float v = __uint_as_float(s[j]) * zs;
                            s[j] = __float_as_uint(v);
                            m0 = fmaxf(m0, v);
                        }
                        part_max = m0;
                        zs = 1.0f;
                    }
                }
                // ---- tile max over both halves
                xmax[(b * 2 + half) * kHeadsM + h] = part_max;
                mbar_arrive(&ctl->xbar[b]);
                ok = wait_warp(ctl, &ctl->xbar[b], (i >> 1) & 1, a.status);
                if (!ok) break;
                const float tile_max = fmaxf(part_max, xmax[(b * 2 + (half ^ 1)) * kHeadsM + h]);
                float alpha = 1.0f;
                if (tile_max > m_ref + kRescaleThreshold) {
                    if (m_ref != -INFINITY) alpha = ex2_approx(m_ref - tile_max);
                    m_ref = tile_max;
                }
                uint4 pc[4];   // this half of P row h: chunk j = keys 32 half + 8j .. +7 (f16)
                if (m_ref != -INFINITY) {
                    const uint64_t mul2 = f32x2_pack(zs, zs);
                    const uint64_t neg_m2 = f32x2_pack(-m_ref, -m_ref);
                    uint64_t la = f32x2_pack(0.0f, 0.0f), lb = la;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t p[4];
#pragma unroll
                        for (int j = 8 * c; j < 8 * c + 8; j += 4) {
                            const float2 z0 = f32x2_unpack(
                                f32x2_fma(f32x2_pack(__uint_as_float(s[j]), __uint_as_float(s[j + 1])), mul2, neg_m2));
                            const float2 z1 = f32x2_unpack(
                                f32x2_fma(f32x2_pack(__uint_as_float(s[j + 2]), __uint_as_float(s[j + 3])), mul2, neg_m2));
                            const float p0 = ex2_approx(fmaxf(z0.x, -INFINITY)), p1 = ex2_approx(fmaxf(z0.y, -INFINITY));
                            const float p2 = ex2_approx(fmaxf(z1.x, -INFINITY)), p3 = ex2_approx(fmaxf(z1.y, -INFINITY));
                            la = f32x2_add(la, f32x2_pack(p0, p1));
                            lb = f32x2_add(lb, f32x2_pack(p2, p3));
                            p[(j & 7) / 2] = pack_f16x2(p0, p1);
                            p[(j & 7) / 2 + 1] = pack_f16x2(p2, p3);
                        }
                        pc[c] = make_uint4(p[0], p[1], p[2], p[3]);
                    }
                    const float2 sa = f32x2_unpack(la), sb = f32x2_unpack(lb);
                    l = l * alpha + ((sa.x + sa.y) + (sb.x + sb.y));
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) pc[c] = make_uint4(0u, 0u, 0u, 0u);
                }
                // ---- 4 x 4 transpose of 16-byte chunks inside each group of four lanes: lane 4a + k
                // ends up with chunk k of the rows of lanes 4a .. 4a + 3, so that every store below
                // writes 8 rows x 64 contiguous bytes (DSMEM moves 64-byte pieces at twice the rate
                // of 16-byte ones)
                transpose4_chunks(pc, lane);
                // ---- -> CTA 1's slot (i % kPStages), once its PV released it
                const int ps = i % kPStages;
                if (i >= kPStages) {
                    ok = wait_warp(ctl, &ctl->pempty[ps], ((i / kPStages) - 1) & 1, a.status);
                    if (!ok) break;
                }
                const uint32_t bar = peer_pfull0 + 8 * ps;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int r = (h & 4) + c;    // row (h & ~3) + c, within its 8-row atom
                    st_async_u4(peer_p_atom + ps * kPBytes + r * 128 + (((4 * half + (lane & 3)) ^ r) << 4), pc[c], bar);
                }
                if (half == 0) st_async_f32(peer_alpha + ps * kHeadsM * 4, alpha, bar);
            }
            // ---- running max and the merged row sum to CTA 1, which writes out and lse
            if (half == 1) {
                xsum[h] = l;
                mbar_arrive(&ctl->lbar);
            } else if (ok && wait_warp(ctl, &ctl->lbar, 0, a.status)) {
                st_async_v2(mapa_shared(smem_addr(smem + kOffFin) + 8 * h, 1), m_ref, l + xsum[h],
                            mapa_shared(smem_addr(&ctl->fin), 1));
            }
        } else if (converter) {
            // ============ CTA 0, warps 8-23: dequant of whole records (K tiles) ============
            if constexpr (R == 656)
                convert_tiles_fp8<true, kKStages, kKTileBytes>(a, ctl, smem + kOffK, smem + kOffRaw0, ctl->kfull,
                                                               ctl->kempty, n_tiles, conv_t);
            else
                convert_tiles<R, true, kBlk, kKStages, kKTileBytes, RawRing<R>::kStages0>(
                    a, ctl, smem + kOffK, smem + kOffRaw0, ctl->kfull, ctl->kempty, n_tiles, conv_t);
        } else if (warp >= kWarpProd) {
            // ============ CTA 0, warps 26-27: record gathers (TMA gather4) ============
            produce_raw<R, true, RawRing<R>::kStages0>(a, ctl, smem + kOffRaw0, idx_row, key_begin, key_end, n_tiles,
                                                       warp - kWarpProd, lane);
        } else {
            // ============ CTA 0, warps 24-25: QK issuers (warp 24 even tiles, warp 25 odd tiles) ============
            const uint32_t idesc_qk = idesc_bf16_f32(kHeadsM, kTile, false, false);
            const uint64_t kdesc0 = sdesc_sw128(smem_addr(smem + kOffK), 16, 1024);
            const bool leader = elect_one_in_warp();
            bool ok = wait_warp(ctl, &ctl->qready, 0, a.status);
            for (int i = warp - kWarpMma; i < n_tiles && ok; i += 2) {
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
        if (warp < 8) {
            // ============ CTA 1, warps 0-3: per-tile alpha check / O rescale; warps 0-7: the output ============
            const int quad = warp & 3;
            const bool second = warp >= 4;   // warps 4-7 only help stage the output
            const int h = quad * 32 + lane;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
            const float* s_alpha = reinterpret_cast<const float*>(smem + kOffAlpha);
            bool ok = true;
            for (int i = 0; i < n_tiles && ok && !second; ++i) {
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
            if (!second && lane == 0) mbar_arrive_expect_tx(&ctl->fin, 32 * 8);
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
            if (h < a.h_q && !second) {
                if (a.splits == 1)
                    a.lse[static_cast<int64_t>(row) * a.h_q + h] = lse2 * kLn2;
                else
                    a.part_lse[(static_cast<int64_t>(row) * a.splits + split) * a.h_q + h] = lse2;
            }
            // have_o is the same in every lane of the warp (tcgen05.ld in write_rows is
            // warp-collective); an empty row has factor 0 and an all-zero O row
            write_rows(smem, lane_base, have_o, factor, h, second ? 2 : 0);
        } else if (converter) {
            // ============ CTA 1, warps 8-23: dequant of the NoPE halves (V tiles) ============
            if constexpr (R == 656)
                convert_tiles_fp8<false, kVStages, kVTileBytes>(a, ctl, smem + kOffV, smem + kOffRaw1, ctl->vfull,
                                                                ctl->vempty, n_tiles, conv_t);
            else
                convert_tiles<R, false, kBlk, kVStages, kVTileBytes, RawRing<R>::kStages1>(
                    a, ctl, smem + kOffV, smem + kOffRaw1, ctl->vfull, ctl->vempty, n_tiles, conv_t);
            help_write_rows(a, smem, row, split, warp - kWarpConv0, lane);
        } else if (warp >= kWarpProd) {
            // ============ CTA 1, warps 26-27: record gathers (TMA gather4) ============
            produce_raw<R, false, RawRing<R>::kStages1>(a, ctl, smem + kOffRaw1, idx_row, key_begin, key_end, n_tiles,
                                                        warp - kWarpProd, lane);
        } else if (warp == kWarpMma) {
            // ============ CTA 1, warp 24: PV issuer (warp 25 idle) ============
            cluster_wait();          // CTA 0's pempty barriers exist before the first multicast commit
            const uint32_t idesc_pv = idesc_f16_f32(kHeadsM, 256, false, true);
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
                    for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ss(tmem + kColO + 256 * nh, pd + ((kk * 32) >> 4),
                                   vd + ((nh * 4 * kBlkBytes + kk * 2048) >> 4), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
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
    const bool waited = (crank == 0 && warp < 8) || (crank == 1 && warp == kWarpMma);
    if (!waited) cluster_wait();
    tc_fence_before_sync();
    cluster_sync();          // no CTA leaves while its peer may still touch its shared memory
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Split merge, one warp per (query row, head), 8 per CTA, launched as a programmatic dependent of
// the decode kernel: out = sum_s w_s part_s with w_s = 2^{lse2_s} / (sum_s 2^{lse2_s} + e^{sink}),
// lse = ln sum_s e^{lse_s} (the sink is not part of lse); lse2 = log2-domain partial lse. Lane s
// holds splits s and s + 32; lane l accumulates columns 4l + 128k (k = 0..3).
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ part_out,
                                                      const float* __restrict__ part_lse, int splits, int h_q,
                                                      int rows_heads, const float* __restrict__ sink,
                                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    // No early trigger here: a decode launched next would park its CTAs on the SMs this grid
    // needs while it waits for it.
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the decode grid's partials are visible
    const int lane = threadIdx.x & 31;
    const int rh = blockIdx.x * 8 + (threadIdx.x >> 5);   // row * h_q + h
    if (rh >= rows_heads) return;
    const int row = rh / h_q;
    const int h = rh % h_q;
    const int64_t base = static_cast<int64_t>(row) * splits;
    // every load of the first four splits goes out before any result is used: one memory round trip
    const float sk = sink != nullptr ? __ldg(sink + h) : 0.0f;
    const float v0 = lane < splits ? part_lse[(base + lane) * h_q + h] : -INFINITY;
    const float v1 = lane + 32 < splits ? part_lse[(base + lane + 32) * h_q + h] : -INFINITY;
    constexpr int kEarly = 4;
    uint2 early[kEarly][4];
#pragma unroll
    for (int sp = 0; sp < kEarly; ++sp) {
        const uint16_t* src = part_out + ((base + sp) * h_q + h) * 512 + 4 * lane;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            early[sp][k] = sp < splits ? __ldg(reinterpret_cast<const uint2*>(src + 128 * k)) : make_uint2(0u, 0u);
    }
    float m = fmaxf(v0, v1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float total = -INFINITY;
    if (m != -INFINITY) {
        const float e0 = exp2f(v0 - m), e1 = exp2f(v1 - m);
        float sum = e0 + e1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        total = (m + log2f(sum)) * kLn2;
        const float inv = 1.0f / (sum + (sink != nullptr ? exp2f(sk * kLog2e - m) : 0.0f));
        const float w0 = e0 * inv, w1 = e1 * inv;
        auto accumulate = [&](float w, const uint2 (&u)[4]) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&u[k].x));
                const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&u[k].y));
                acc[k].x += w * lo.x;
                acc[k].y += w * lo.y;
                acc[k].z += w * hi.x;
                acc[k].w += w * hi.y;
            }
        };
#pragma unroll
        for (int sp = 0; sp < kEarly; ++sp) {
            const float w = __shfl_sync(0xffffffffu, w0, sp);
            if (sp < splits) accumulate(w, early[sp]);
        }
        for (int sp = kEarly; sp < splits; ++sp) {
            const float w = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
            const uint16_t* src = part_out + ((base + sp) * h_q + h) * 512 + 4 * lane;
            uint2 u[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) u[k] = __ldg(reinterpret_cast<const uint2*>(src + 128 * k));
            accumulate(w, u);
        }
    }
    __nv_bfloat16* dst = out + static_cast<int64_t>(rh) * 512 + 4 * lane;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint2*>(dst + 128 * k) =
            make_uint2(pack_bf16x2(acc[k].x, acc[k].y), pack_bf16x2(acc[k].z, acc[k].w));
    if (lane == 0) lse[rh] = total;
}

// One thread waits on an mbarrier that nothing arrives on, with the same time-bounded wait the
// decode uses: the wait gives up, the kernel records NVFP4_MLA_DEV_TIMEOUT and the time it
// waited, and returns normally.
__global__ void wait_timeout_probe_kernel(uint32_t* status, uint64_t* elapsed_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint64_t t0 = global_ns();
    const bool done = mbar_wait(&bar, 0);
    const uint64_t t1 = global_ns();
    if (!done) atomicOr(status, 0x4u);   // NVFP4_MLA_DEV_TIMEOUT
    *elapsed_ns = t1 - t0;
}

}  // namespace

int decode_keys_per_split(int topk, int splits) {
    const int per = (topk + splits - 1) / splits;
    return (per + kTile - 1) / kTile * kTile;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The cache as a 2-D tensor of u32 [rows, R / 4] whose box is one record, for tile::gather4.
// Rows are capped at 2^31 - 1 (indices are int32); an empty cache maps one row that is never
// fetched (no index is in range).
bool encode_cache_map(CUtensorMap* map, const uint8_t* cache, int64_t num_slots, int record_bytes) {
    const EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return false;
    const int64_t rows = num_slots < 1 ? 1 : (num_slots > 0x7FFFFFFF ? 0x7FFFFFFF : num_slots);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(record_bytes / 4), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(record_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(record_bytes / 4), 1u};
    const cuuint32_t elem_strides[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(cache), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q as a 2-D tensor of bf16 [rows * h_q, 576], box 64 columns x 128 heads with the 128B swizzle;
// heads past the end read zeros.
bool encode_q_map(CUtensorMap* map, const void* q, int64_t heads) {
    const EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr || heads < 1 || heads > 0x7FFFFFFF) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(heads)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk) * 2u};
    const cuuint32_t box[2] = {64u, 128u};
    const cuuint32_t elem_strides[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raises the kernel's dynamic shared memory limit once per device.
template <int R, bool kBlk>
cudaError_t prepare_kernel() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    err = cudaFuncSetAttribute(sparse_decode_kernel<R, kBlk>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SmemSize<R>::value);
    if (err == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_relaxed);
    return err;
}

}  // namespace

cudaError_t launch_wait_timeout_probe(uint32_t* status, uint64_t* elapsed_ns, cudaStream_t stream) {
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status, elapsed_ns);
    return cudaGetLastError();
}

cudaError_t launch_sparse_decode(const DecodeArgs& d, cudaStream_t stream) {
    cudaError_t err;
    bool merged = false;   // the decode grid merged the splits itself
    if (decode_pair_supported(d)) {
        err = launch_decode_pair(d, stream, &merged);
    } else if (decode_h64_supported(d)) {
        err = launch_decode_h64(d, stream);
    } else {
        KernelArgs a;
        if (!encode_cache_map(&a.tmap, d.cache, d.num_slots, d.record_bytes)) return cudaErrorInvalidValue;
        if (!encode_q_map(&a.qmap, d.q, static_cast<int64_t>(d.rows) * d.h_q)) return cudaErrorInvalidValue;
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
        err = d.record_bytes == 656 ? prepare_kernel<656, false>()
              : d.record_bytes == 432 ? prepare_kernel<432, false>()
              : d.block_scales      ? prepare_kernel<352, true>()
                                    : prepare_kernel<352, false>();
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = d.record_bytes == 656   ? SmemSize<656>::value
                               : d.record_bytes == 432 ? SmemSize<432>::value
                                                       : SmemSize<352>::value;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddepcontrol.wait
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const auto kernel = d.record_bytes == 656 ? sparse_decode_kernel<656, false>
                            : d.record_bytes == 432 ? sparse_decode_kernel<432, false>
                            : d.block_scales      ? sparse_decode_kernel<352, true>
                                                  : sparse_decode_kernel<352, false>;
        err = cudaLaunchKernelEx(&cfg, kernel, a);
        if (err == cudaSuccess) err = cudaGetLastError();
    }
    if (err != cudaSuccess || d.splits == 1 || merged) return err;
    return launch_split_merge(d, stream);
}

// The merge launches while the decode grid runs and waits for it on the device. It asks for the
// same shared-memory carveout as the decode kernels, so that the SMs need not repartition their
// L1 and shared memory between the two grids.
cudaError_t launch_split_merge(const DecodeArgs& d, cudaStream_t stream) {
    static const cudaError_t carveout =
        cudaFuncSetAttribute(combine_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (carveout != cudaSuccess) return carveout;
    cudaLaunchConfig_t cfg = {};
    const int rows_heads = d.rows * d.h_q;
    cfg.gridDim = dim3(static_cast<unsigned>((rows_heads + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, static_cast<const uint16_t*>(d.part_out),
                              static_cast<const float*>(d.part_lse), d.splits, d.h_q, rows_heads, d.attn_sink,
                              static_cast<__nv_bfloat16*>(d.out), d.lse);
}

}  // namespace nvfp4mla
