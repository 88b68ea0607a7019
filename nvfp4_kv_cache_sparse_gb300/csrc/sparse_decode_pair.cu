// sparse_decode_pair.cu -- sparse MLA decode for 128 query heads on a CTA pair whose tensor cores
// share every MMA (tcgen05 cta_group::2), for 352-byte and 432-byte NVFP4 records.
//
// What is computed (FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode",
// "Kernel:" paragraph and validation list): for query row t and head h, with J the used entries
// of t's index list,
//     z_j = sm_scale * q[t,h,:] . K_j          (K_j: 576 dequantized values of record j)
//     out = sum_j e^{z_j} V_j / (sum_j e^{z_j} + e^{sink_h}),   V_j = K_j[0:512]
//     lse = ln sum_j e^{z_j}
// Both contractions are 16-bit tcgen05 MMAs with fp32 accumulation in tensor memory.
//
// Work split. A cluster of two CTAs per (query row, top-k split); CTA c owns heads 64c..64c+63.
// Keys go in tiles of 128: CTA c loads the records of keys 64c..64c+63 of each tile ("own" keys).
//   QK^T: one M = 128 (heads) x N = 128 (keys) x K = 576 pair MMA per tile: each CTA supplies its
//     64 heads of q and its 64 own keys' K rows; S of its heads for all 128 keys lands in its own
//     tensor memory (lanes 0-63: keys 0-63, lanes 64-127: keys 64-127).
//   P V: M = 128 (heads) x N = 256 x K = 128 (keys) pair MMAs; CTA 0 supplies V dims 0-255 and
//     CTA 1 dims 256-511, each for all 128 keys, so O of a CTA's 64 heads spans all 512 dims
//     (lanes 0-63: dims 0-255, lanes 64-127: dims 256-511) in 256 tensor-memory columns.
//   Every record is loaded once per pair. A CTA dequantizes its own keys' K rows (576 dims) and
//   the V rows of its own half of the dims for all 128 keys; the raw e2m1 codes and scales of the
//   other CTA's half of the dims cross to it over DSMEM (36 bytes per key and thread quarter).
// Numbers. e2m1 x e4m3 products are exact in f16 (<= 5 significant bits in [2^-10, 2688]), so K
// and V tiles are f16 (the bf16 RoPE of 432-byte records stays bf16). q enters as f16 scaled by a
// per-head power of two (2^pre with max|q| 2^pre in [2^14, 2^15)): the products q_d K_d are the
// same numbers as with bf16 q, and S comes out as 2^pre times the exact score, which the softmax
// folds into its scale. P is f16 (entries in [0, 2^8]).
// Softmax. A lazy reference maximum m per head (log2 domain): P = 2^(z - m) and O, l accumulate
// against m. A tile only needs the reference to move when some score exceeds m + 8; the softmax
// warps vote on that once per tile (one barrier reduction) and only then exchange maxima and
// rescale O in tensor memory, so the common tile has no cross-thread exchange at all. Masked keys
// have quiet-NaN K rows: their scores are NaN, max() ignores them and max(2^NaN, 0) = 0.
// Warp roles (kThreads = 832, 26 warps):
//   0-7   softmax (warp w: lane quadrant w & 3, score columns 32 (w >> 2)..+32); q staging in the
//         prologue; output in the epilogue
//   8-15  K converters: load own records (registers, one tile ahead, L2 prefetch two ahead), write
//         K rows, the own-half raw codes (local) and the other half's raw codes (to the peer)
//   16-23 V converters: V rows of this CTA's dims for all 128 keys, from the two raw buffers
//   24    QK issuer (CTA 0) and tensor-memory owner (both)
//   25    PV issuer (CTA 0)
// Every wait is bounded by time; on timeout a CTA sets NVFP4_MLA_DEV_TIMEOUT, stops issuing work,
// drains what it issued and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace nvfp4mla {
namespace pairdec {
namespace {

constexpr int kTile = 128;                 // keys per tile (QK N over the pair)
constexpr int kOwn = 64;                   // keys per tile whose records one CTA loads
constexpr int kHeads = 64;                 // heads per CTA
constexpr int kThreads = 832;
constexpr int kWarpK = 8;
constexpr int kWarpV = 16;
constexpr int kWarpQK = 24;
constexpr int kWarpPV = 25;
constexpr uint32_t kColO = 0;              // O: 256 columns
constexpr uint32_t kColS = 256;            // S: 64 columns (128 keys folded over the lane halves)
constexpr uint32_t kColQ = 320;            // q dims [0, 384): 192 columns, both lane halves
constexpr int kQTmemSteps = 24;            // K-steps of 16 dims taken from tensor memory
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// Shared memory (offsets from a 1024-byte aligned base)
constexpr int kBlk = 8192;                 // 64 rows x 128 B (one 64-wide 16-bit block)
constexpr int kVBlk = 16384;               // 128 rows x 128 B
constexpr int kOffXmax = 1024;             // float [4][64] tile maxima (slow path) / row sums
constexpr int kOffXl = 2048;               // float [4][64]
constexpr int kOffK = 4096;                // 9 blocks: K rows of the 64 own keys (K-major)
constexpr int kOffV = kOffK + 9 * kBlk;    // 4 blocks of 128 keys: this CTA's 256 V dims (MN-major)
constexpr int kOffP = kOffV + 4 * kVBlk;   // 2 blocks: P [64 heads x 128 keys] (K-major)
constexpr int kOffQs = kOffP + 2 * kBlk;   // 3 blocks: q dims [384, 576)
constexpr int kRawCodes = kOwn * 4 * 32;   // [key][quarter] 32 B of e2m1 codes
constexpr int kRawBytes = kRawCodes + kOwn * 4 * 4;   // + [key][quarter] 4 scale bytes
constexpr int kOffOwnRaw = kOffQs + 3 * kBlk;         // [2] own keys, this CTA's dims
constexpr int kOffPeerRaw = kOffOwnRaw + 2 * kRawBytes;   // [2] the peer's keys, this CTA's dims
constexpr int kSmemBytes = kOffPeerRaw + 2 * kRawBytes;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0 && kOffQs % 1024 == 0, "operand alignment");
static_assert(9 * kBlk <= 4 * kVBlk + 2 * kBlk, "q staging fits in the V and P buffers");
static_assert(kHeads * 1024 <= 9 * kBlk, "output staging fits in the K buffer");

struct __align__(8) Ctl {
    uint64_t qkdone;          // QK commit (multicast): S ready, K buffer free
    uint64_t pvdone;          // PV commit (multicast): V and P buffers free, O updated
    uint64_t kfull;           // CTA 0: 16 warps (8 per CTA) wrote K rows
    uint64_t vfull;           // CTA 0: 16 warps wrote V rows
    uint64_t sfree;           // CTA 0: 16 softmax warps read S
    uint64_t pfull;           // CTA 0: 16 softmax warps wrote P (and rescaled O)
    uint64_t qready;          // CTA 0: 16 softmax warps put q into tensor and shared memory
    uint64_t qstaged;         // 8 local softmax warps finished reading the q staging area
    uint64_t qload;           // q boxes landed (TMA, tx-counted)
    uint64_t own_full[2];     // K converters wrote own raw codes
    uint64_t own_empty[2];    // V converters read them
    uint64_t peer_full[2];    // the peer's raw codes landed (st.async, tx-counted)
    uint64_t peer_empty[2];   // the peer's V converters read what this CTA sent (remote arrivals)
    uint64_t drain;           // CTA 0: both issuers' MMAs completed
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(Ctl) <= kOffXmax, "control block");

struct KernelArgs {
    CUtensorMap qmap;         // q as bf16 [rows * 128, 576], box 64 dims x 64 heads, 128B swizzle
    const uint8_t* cache;
    int64_t num_slots;
    const int32_t* indices;
    int topk;
    int splits;
    int keys_per_split;
    float sm_scale;
    const float* sink;
    __nv_bfloat16* out;
    float* lse;
    uint16_t* part_out;       // f16 partial outputs [rows, splits, 128, 512]
    float* part_lse;          // log2 domain
    uint32_t* status;
};

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void set_abort(Ctl* ctl, uint32_t* status) {
    if (atomicExch(&ctl->abort, 1u) == 0u && status != nullptr) atomicOr(status, 0x4u);
}
__device__ __forceinline__ bool aborted(Ctl* ctl) { return *reinterpret_cast<volatile uint32_t*>(&ctl->abort) != 0u; }

// Bounded wait, cluster-scope acquire (several barriers here receive arrivals or bytes from the
// peer CTA). One answer per warp.
__device__ __forceinline__ bool wait_warp(Ctl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    bool ok = mbar_try_wait_cluster(bar, parity);
    if (!ok && !aborted(ctl)) {
        ok = mbar_wait_cluster(bar, parity);
        if (!ok) set_abort(ctl, status);
    }
    return __all_sync(0xffffffffu, ok);
}

// Arrival on a barrier that lives in CTA 0 (the pair's MMA issuer), from either CTA.
__device__ __forceinline__ void arrive_leader(uint64_t* bar, int crank) {
    if (crank == 0)
        mbar_arrive(bar);
    else
        mbar_arrive_cluster(mapa_shared(smem_addr(bar), 0));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// e4m3 scale byte -> (s, s) as f16x2 (exact).
__device__ __forceinline__ __half2 scale_half2(uint32_t sbyte) {
    uint32_t h;
    const uint16_t in = static_cast<uint16_t>(sbyte | (sbyte << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    return *reinterpret_cast<__half2*>(&h);
}

// Eight e2m1 codes (one word, low nibble first) times a scale -> four f16x2 words (exact).
__device__ __forceinline__ uint4 dq8(uint32_t w, __half2 s2) {
    uint32_t h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t v;
        asm("{\n"
            "  .reg .b8 t;\n"
            "  cvt.u8.u32 t, %1;\n"
            "  cvt.rn.f16x2.e2m1x2 %0, t;\n"
            "}\n"
            : "=r"(v)
            : "r"(w >> (8 * k)));
        const __half2 p = __hmul2(*reinterpret_cast<__half2*>(&v), s2);
        h[k] = *reinterpret_cast<const uint32_t*>(&p);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

// Four e4m3 codes -> two f16x2 words (exact).
__device__ __forceinline__ uint2 e4m3x4_to_f16(uint32_t w) {
    uint32_t a, b;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(a) : "h"(static_cast<uint16_t>(w)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(b) : "h"(static_cast<uint16_t>(w >> 16)));
    return make_uint2(a, b);
}

// The bytes of one own key that one converter thread (quarter q) needs: e2m1 codes of the 16-wide
// blocks 4c + q (c = 0..7; block s holds dims 16s..16s+15 at bytes 8s..8s+7), their eight scale
// bytes (byte c = block 4c + q) and 16 RoPE dims 16q..16q+15 (e4m3 in one word-quad for 352-byte
// records, bf16 in two for 432-byte records).
struct Raw {
    uint2 codes[8];
    uint2 sc;
    uint4 rope[2];
};

// kBlkOrder: the 32 scale bytes are in block order (432-byte records, and the 352-byte record of
// the scale-layout comparison) instead of the permuted placement 8 (s & 3) + (s >> 2).
template <int R, bool kBlkOrder>
__device__ __forceinline__ void load_raw(const uint8_t* rec, int q, Raw& r) {
#pragma unroll
    for (int c = 0; c < 8; ++c) r.codes[c] = __ldg(reinterpret_cast<const uint2*>(rec + 32 * c + 8 * q));
    if constexpr (R == 352 && !kBlkOrder) {
        // permuted placement: blocks {4c + q, c = 0..7} are the eight bytes at 320 + 8q
        r.sc = __ldg(reinterpret_cast<const uint2*>(rec + 320 + 8 * q));
    } else {
        const int sb = R == 352 ? 320 : 256;   // block s at byte sb + s
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(rec + sb));
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(rec + sb + 16));
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};   // w[c] holds blocks 4c..4c+3
        uint32_t lo = 0u, hi = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            lo |= ((w[c] >> (8 * q)) & 0xFFu) << (8 * c);
            hi |= ((w[c + 4] >> (8 * q)) & 0xFFu) << (8 * c);
        }
        r.sc = make_uint2(lo, hi);
    }
    if constexpr (R == 352) {
        r.rope[0] = __ldg(reinterpret_cast<const uint4*>(rec + 256 + 16 * q));
        r.rope[1] = make_uint4(0u, 0u, 0u, 0u);
    } else {
        r.rope[0] = __ldg(reinterpret_cast<const uint4*>(rec + 304 + 32 * q));
        r.rope[1] = __ldg(reinterpret_cast<const uint4*>(rec + 304 + 32 * q + 16));
    }
}

__device__ __forceinline__ void zero_raw(Raw& r) {
#pragma unroll
    for (int c = 0; c < 8; ++c) r.codes[c] = make_uint2(0u, 0u);
    r.sc = make_uint2(0u, 0u);
    r.rope[0] = r.rope[1] = make_uint4(0u, 0u, 0u, 0u);
}

// One thread's share of a raw buffer entry (key j, quarter q): the codes of blocks 4c + q for the
// receiving CTA's four c (32 B) and their scale bytes (4 B).
__device__ __forceinline__ uint32_t raw_codes_at(uint32_t buf, int j, int q) { return buf + (j * 4 + q) * 32; }
__device__ __forceinline__ uint32_t raw_scale_at(uint32_t buf, int j, int q) { return buf + kRawCodes + (j * 4 + q) * 4; }

// V rows: the four blocks 4c + q (c = 4 half + cl) of one key into V block cl, chunks 2q, 2q + 1.
__device__ __forceinline__ void write_v(uint32_t v_s, int row, int q, const uint4& c01, const uint4& c23,
                                        uint32_t sbytes) {
    const uint32_t cw[8] = {c01.x, c01.y, c01.z, c01.w, c23.x, c23.y, c23.z, c23.w};
#pragma unroll
    for (int cl = 0; cl < 4; ++cl) {
        const __half2 s2 = scale_half2((sbytes >> (8 * cl)) & 0xFFu);
        sts_u128(v_s + cl * kVBlk + swz(row, 2 * q), dq8(cw[2 * cl], s2));
        sts_u128(v_s + cl * kVBlk + swz(row, 2 * q + 1), dq8(cw[2 * cl + 1], s2));
    }
}

template <int R, bool kBlkOrder>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_pair_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    Ctl* ctl = reinterpret_cast<Ctl*>(smem);
    const uint32_t sbase = smem_addr(smem);

    const int crank = static_cast<int>(cluster_ctarank());
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
        mbar_init(&ctl->qkdone, 1);
        mbar_init(&ctl->pvdone, 1);
        mbar_init(&ctl->kfull, 16);
        mbar_init(&ctl->vfull, 16);
        mbar_init(&ctl->sfree, 16);
        mbar_init(&ctl->pfull, 16);
        mbar_init(&ctl->qready, 16);
        mbar_init(&ctl->qstaged, 8);
        mbar_init(&ctl->qload, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->own_full[b], 8);
            mbar_init(&ctl->own_empty[b], 8);
            mbar_init(&ctl->peer_full[b], 1);
            mbar_init(&ctl->peer_empty[b], 8);
        }
        mbar_init(&ctl->drain, 2);
        ctl->abort = 0u;
        fence_barrier_init();
        // the first two tiles' bytes from the peer may arrive as soon as the cluster barrier opens
        if (n_tiles > 0) mbar_arrive_expect_tx(&ctl->peer_full[0], kRawBytes);
        if (n_tiles > 1) mbar_arrive_expect_tx(&ctl->peer_full[1], kRawBytes);
    }
    if (warp == kWarpQK) {
        tmem_alloc_cg2(&ctl->tmem_base, kTmemCols);
        tmem_relinquish_cg2();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;
    // Launched as a programmatic dependent of the preceding kernel: nothing is read before that grid
    // has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    cluster_arrive();
    cluster_wait();   // both CTAs' barriers exist before any remote access

    if (warp < 8) {
        // ======================= softmax warps =======================
        const int qd = warp & 3;               // TMEM lane quadrant
        const int h2 = warp >> 2;              // score column half
        const int L = 32 * qd + lane;          // TMEM lane
        const int hl = L & 63;                 // head within the CTA
        const int qi = ((qd >> 1) << 1) | h2;  // this thread's slot among the head's four
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        float* xmax = reinterpret_cast<float*>(smem + kOffXmax);
        float* xl = reinterpret_cast<float*>(smem + kOffXl);
        // ---- q: largest magnitude of the head, the power-of-two prescale, f16 (or bf16 RoPE) copies
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&ctl->qload, 9u * kBlk);
            for (int bx = 0; bx < 9; ++bx)
                tma_load_2d(sbase + kOffV + bx * kBlk, &a.qmap, 64 * bx, row * 128 + 64 * crank, &ctl->qload);
        }
        bool ok = wait_warp(ctl, &ctl->qload, 0, a.status);
        const uint32_t stage = sbase + kOffV;   // box b (dims 64b..): head hl chunk c at b*8192 + swz(hl, c)
        float qmax = 0.0f;
        if (ok) {
#pragma unroll 1
            for (int k = 18 * qi; k < 18 * qi + 18; ++k) {   // 72 chunks of 8 dims per head, 18 per thread
                const uint4 x = lds_u128(stage + (k >> 3) * kBlk + swz(hl, k & 7));
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    qmax = fmaxf(qmax, fabsf(__uint_as_float(w[m] << 16)));
                    qmax = fmaxf(qmax, fabsf(__uint_as_float(w[m] & 0xFFFF0000u)));
                }
            }
        }
        xmax[qi * 64 + hl] = qmax;
        named_bar_sync(1, 256);
        qmax = fmaxf(fmaxf(xmax[hl], xmax[64 + hl]), fmaxf(xmax[128 + hl], xmax[192 + hl]));
        int pre = 0;
        if (qmax > 0.0f) {
            int e;
            frexpf(qmax, &e);   // qmax < 2^e <= 2 qmax
            pre = min(100, max(-100, 15 - e));
        }
        const int p1 = pre / 2, p2 = pre - p1;
        const float f1 = __int_as_float((127 + p1) << 23), f2 = __int_as_float((127 + p2) << 23);
        // c = sm_scale log2(e) 2^-pre: S' = 2^pre S, so z = c S' (log2 domain)
        const float ch = a.sm_scale * kLog2e * __int_as_float((127 - p1) << 23) * __int_as_float((127 - p2) << 23);
        auto cvt_pair = [&](uint32_t w, bool bf) -> uint32_t {
            const float lo = __uint_as_float(w << 16) * f1 * f2, hi = __uint_as_float(w & 0xFFFF0000u) * f1 * f2;
            return bf ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
        };
        if (ok) {
            // dims [0, 384): TMEM columns kColQ.. in this lane (both lane halves hold a copy);
            // this thread takes dims [192 h2, 192 h2 + 192) = 24 chunks
#pragma unroll 1
            for (int g = 0; g < 3; ++g) {
                uint32_t v[32];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const int k = 24 * h2 + 8 * g + cc;   // dim chunk
                    const uint4 x = lds_u128(stage + (k >> 3) * kBlk + swz(hl, k & 7));
                    v[4 * cc + 0] = cvt_pair(x.x, false);
                    v[4 * cc + 1] = cvt_pair(x.y, false);
                    v[4 * cc + 2] = cvt_pair(x.z, false);
                    v[4 * cc + 3] = cvt_pair(x.w, false);
                }
                tmem_st32(lane_base + kColQ + 96 * h2 + 32 * g, v);
            }
            // dims [384, 576) into shared memory (one copy: lanes 0-63), K-major blocks of 64 dims
            if (qd < 2) {
#pragma unroll 1
                for (int cc = 0; cc < 12; ++cc) {
                    const int k = 48 + 12 * h2 + cc;      // dim chunk 48..71
                    const bool bf = R == 432 && k >= 64;  // bf16 RoPE of 432-byte records
                    const uint4 x = lds_u128(stage + (k >> 3) * kBlk + swz(hl, k & 7));
                    const uint4 y = make_uint4(cvt_pair(x.x, bf), cvt_pair(x.y, bf), cvt_pair(x.z, bf), cvt_pair(x.w, bf));
                    sts_u128(sbase + kOffQs + ((k - 48) >> 3) * kBlk + swz(hl, k & 7), y);
                }
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&ctl->qstaged);
            arrive_leader(&ctl->qready, crank);
        }
        // ---- tiles
        float m_ref = -INFINITY;   // reference max (log2 units), the same in the head's four threads
        float l = 0.0f;            // this thread's sum of 2^(z - m_ref)
        const bool pos_scale = a.sm_scale > 0.0f;
        const uint32_t p_row = sbase + kOffP + (qd >> 1) * kBlk;
        // Every softmax warp takes part in every named barrier below, also after a wait ran out
        // (then it only passes the barriers), so no warp can be left waiting on a missing one.
        for (int i = 0; i < n_tiles; ++i) {
            uint32_t s[32];
            float mx = -INFINITY;
            float mul = ch;
            if (ok) ok = wait_warp(ctl, &ctl->qkdone, i & 1, a.status);
            if (ok) {
                tc_fence_after_sync();
                tmem_ld32(lane_base + kColS + 32 * h2, s);
                tmem_wait_ld();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) arrive_leader(&ctl->sfree, crank);
                float m0 = -INFINITY, m1 = -INFINITY;
                if (pos_scale) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        m0 = fmax3(m0, __uint_as_float(s[j]), __uint_as_float(s[j + 1]));
                        m1 = fmax3(m1, __uint_as_float(s[j + 2]), __uint_as_float(s[j + 3]));
                    }
                    mx = fmaxf(m0, m1) * ch;
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float z = __uint_as_float(s[j]) * ch;
                        s[j] = __float_as_uint(z);
                        m0 = fmaxf(m0, z);
                    }
                    mx = m0;
                    mul = 1.0f;
                }
            }
            // ---- does any head of this CTA need a new reference? (one barrier reduction)
            if (bar_red_or(1, 256, mx > m_ref + kRescaleThreshold)) {
                xmax[qi * 64 + hl] = mx;
                named_bar_sync(1, 256);
                const float tmax = fmaxf(fmaxf(xmax[hl], xmax[64 + hl]), fmaxf(xmax[128 + hl], xmax[192 + hl]));
                float alpha = 1.0f;
                if (tmax > m_ref + kRescaleThreshold) {
                    alpha = m_ref == -INFINITY ? 0.0f : ex2_approx(m_ref - tmax);
                    m_ref = tmax;
                }
                l *= alpha;
                if (ok && i > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                    // O (this lane, columns 128 h2 ..) *= alpha once PV of the previous tile is done
                    ok = wait_warp(ctl, &ctl->pvdone, (i - 1) & 1, a.status);
                    if (ok) {
                        tc_fence_after_sync();
#pragma unroll 1
                        for (int c = 0; c < 8; ++c) {   // 16 columns at a time: the scores stay in registers
                            uint32_t o[16];
                            tmem_ld16(lane_base + kColO + 128 * h2 + 16 * c, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                            tmem_st16(lane_base + kColO + 128 * h2 + 16 * c, o);
                        }
                        tmem_wait_st();
                    }
                }
            }
            if (!ok) continue;
            // ---- P = 2^(z - m_ref) in f16; masked keys (NaN scores) give 0
            uint32_t pw[16];
            if (m_ref != -INFINITY) {
                const uint64_t mul2 = f32x2_pack(mul, mul);
                const uint64_t neg_m2 = f32x2_pack(-m_ref, -m_ref);
                uint64_t la = f32x2_pack(0.0f, 0.0f), lb = la;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float2 z0 =
                        f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(s[j]), __uint_as_float(s[j + 1])), mul2, neg_m2));
                    const float2 z1 = f32x2_unpack(
                        f32x2_fma(f32x2_pack(__uint_as_float(s[j + 2]), __uint_as_float(s[j + 3])), mul2, neg_m2));
                    const float p0 = fmaxf(ex2_approx(z0.x), 0.0f), p1v = fmaxf(ex2_approx(z0.y), 0.0f);
                    const float p2v = fmaxf(ex2_approx(z1.x), 0.0f), p3 = fmaxf(ex2_approx(z1.y), 0.0f);
                    la = f32x2_add(la, f32x2_pack(p0, p1v));
                    lb = f32x2_add(lb, f32x2_pack(p2v, p3));
                    pw[j / 2] = pack_f16x2(p0, p1v);
                    pw[j / 2 + 1] = pack_f16x2(p2v, p3);
                }
                const float2 sa = f32x2_unpack(la), sb = f32x2_unpack(lb);
                l += (sa.x + sa.y) + (sb.x + sb.y);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) pw[j] = 0u;
            }
            // ---- P into shared memory once PV of the previous tile released it
            if (i > 0) ok = wait_warp(ctl, &ctl->pvdone, (i - 1) & 1, a.status);
            if (!ok) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                sts_u128(p_row + swz(hl, 4 * h2 + c), make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]));
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) arrive_leader(&ctl->pfull, crank);
        }
        // ---- epilogue: row sums, O / l, out (or the split's partial) and lse
        xl[qi * 64 + hl] = l;
        named_bar_sync(1, 256);
        const float lt = (xl[hl] + xl[64 + hl]) + (xl[128 + hl] + xl[192 + hl]);
        bool have_o = false;
        if (ok && n_tiles > 0) {
            have_o = wait_warp(ctl, &ctl->pvdone, (n_tiles - 1) & 1, a.status);
            if (have_o) tc_fence_after_sync();
        }
        const int head = 64 * crank + hl;
        const bool empty = !(lt > 0.0f);
        const float lse2 = empty ? -INFINITY : m_ref + log2f(lt);
        float factor = 0.0f;
        if (!empty) {
            float denom = lt;
            if (a.splits == 1 && a.sink != nullptr) denom += exp2f(__ldg(a.sink + head) * kLog2e - m_ref);
            factor = 1.0f / denom;
        }
        if (qi == 0) {
            if (a.splits == 1)
                a.lse[static_cast<int64_t>(row) * 128 + head] = lse2 * kLn2;
            else
                a.part_lse[(static_cast<int64_t>(row) * a.splits + split) * 128 + head] = lse2;
        }
        // stage O * factor as 16-bit rows of 1024 B in the K buffer (the last QK finished with it)
        const int dbase = (L >= 64 ? 256 : 0) + 128 * h2;
        const uint32_t orow = sbase + kOffK + hl * 1024;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            if (have_o) {
                tmem_ld32(lane_base + kColO + 128 * h2 + 32 * c, o);
                tmem_wait_ld();
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = have_o ? __uint_as_float(o[8 * m + 2 * e]) * factor : 0.0f;
                    const float hi = have_o ? __uint_as_float(o[8 * m + 2 * e + 1]) * factor : 0.0f;
                    w4[e] = a.splits == 1 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
                }
                const int k = (dbase + 32 * c + 8 * m) >> 3;   // 16-byte chunk of the row
                sts_u128(orow + ((((k & ~7) | ((k ^ hl) & 7))) << 4), make_uint4(w4[0], w4[1], w4[2], w4[3]));
            }
        }
        named_bar_sync(1, 256);
        // copy out: warp w takes rows w, w + 8, ...; 64 chunks per row, two per lane
        uint16_t* dst0 = a.splits == 1
                             ? reinterpret_cast<uint16_t*>(a.out) + (static_cast<int64_t>(row) * 128 + 64 * crank) * 512
                             : a.part_out + ((static_cast<int64_t>(row) * a.splits + split) * 128 + 64 * crank) * 512;
#pragma unroll 2
        for (int r = warp; r < kHeads; r += 8) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int k = lane + 32 * hh;
                const uint4 x = lds_u128(sbase + kOffK + r * 1024 + ((((k & ~7) | ((k ^ r) & 7))) << 4));
                *reinterpret_cast<uint4*>(dst0 + static_cast<int64_t>(r) * 512 + 8 * k) = x;
            }
        }
    } else if (warp < kWarpV) {
        // ======================= K converters =======================
        const int t = threadIdx.x - 32 * kWarpK;
        const int j = t >> 2;    // own key of the tile
        const int q = t & 3;     // quarter: blocks 4c + q, RoPE dims 16q..
        const uint32_t k_s = sbase + kOffK;
        auto index_of = [&](int i) -> int32_t {
            if (i >= n_tiles) return -1;
            const int pos = key_begin + kTile * i + kOwn * crank + j;
            return pos < key_end ? __ldg(idx_row + pos) : -1;
        };
        auto in_range = [&](int32_t v) { return v >= 0 && static_cast<int64_t>(v) < a.num_slots; };
        int32_t idx0 = index_of(0), idx1 = index_of(1), idx2 = index_of(2);
        Raw r;
        if (in_range(idx0))
            load_raw<R, kBlkOrder>(a.cache + static_cast<int64_t>(idx0) * R, q, r);
        else
            zero_raw(r);
        if (in_range(idx1)) prefetch_l2(a.cache + static_cast<int64_t>(idx1) * R + (q == 3 ? R - 1 : 128 * q));
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
            const int b = i & 1;
            const bool valid = in_range(idx0);
            if (q == 0 && idx0 >= 0 && !valid && a.status != nullptr) atomicOr(a.status, 0x2u);
            if (i >= 1) ok = wait_warp(ctl, &ctl->qkdone, (i - 1) & 1, a.status);   // K buffer free
            if (ok && i >= 2) ok = wait_warp(ctl, &ctl->own_empty[b], ((i >> 1) - 1) & 1, a.status);
            if (ok && i >= 2) ok = wait_warp(ctl, &ctl->peer_empty[b], ((i >> 1) - 1) & 1, a.status);
            if (!ok) break;
            // ---- K rows: NoPE blocks (f16) and RoPE (f16 from e4m3, or bf16 verbatim)
            if (valid) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const __half2 s2 = scale_half2((c < 4 ? r.sc.x >> (8 * c) : r.sc.y >> (8 * (c - 4))) & 0xFFu);
                    sts_u128(k_s + c * kBlk + swz(j, 2 * q), dq8(r.codes[c].x, s2));
                    sts_u128(k_s + c * kBlk + swz(j, 2 * q + 1), dq8(r.codes[c].y, s2));
                }
                if constexpr (R == 352) {
                    const uint2 e0 = e4m3x4_to_f16(r.rope[0].x), e1 = e4m3x4_to_f16(r.rope[0].y);
                    const uint2 e2 = e4m3x4_to_f16(r.rope[0].z), e3 = e4m3x4_to_f16(r.rope[0].w);
                    sts_u128(k_s + 8 * kBlk + swz(j, 2 * q), make_uint4(e0.x, e0.y, e1.x, e1.y));
                    sts_u128(k_s + 8 * kBlk + swz(j, 2 * q + 1), make_uint4(e2.x, e2.y, e3.x, e3.y));
                } else {
                    sts_u128(k_s + 8 * kBlk + swz(j, 2 * q), r.rope[0]);
                    sts_u128(k_s + 8 * kBlk + swz(j, 2 * q + 1), r.rope[1]);
                }
            } else {
                // a masked key: quiet-NaN K row, so every score of it is NaN
                const uint32_t f = 0x7E007E00u;                      // f16 quiet NaN pairs
                const uint32_t fr = R == 352 ? 0x7E007E00u : 0x7FC07FC0u;   // RoPE block: f16 / bf16
                const uint4 z = make_uint4(f, f, f, f), zr = make_uint4(fr, fr, fr, fr);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    sts_u128(k_s + c * kBlk + swz(j, 2 * q), z);
                    sts_u128(k_s + c * kBlk + swz(j, 2 * q + 1), z);
                }
                sts_u128(k_s + 8 * kBlk + swz(j, 2 * q), zr);
                sts_u128(k_s + 8 * kBlk + swz(j, 2 * q + 1), zr);
            }
            // ---- raw codes of this CTA's dims (local) and of the peer's dims (DSMEM); zeros for a masked key
            {
                // codes of blocks 4c + q: c = 0..3 (dims 0-255, CTA 0's half) and c = 4..7 (CTA 1's half)
                const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
                const uint4 lo01 = valid ? make_uint4(r.codes[0].x, r.codes[0].y, r.codes[1].x, r.codes[1].y) : z4;
                const uint4 lo23 = valid ? make_uint4(r.codes[2].x, r.codes[2].y, r.codes[3].x, r.codes[3].y) : z4;
                const uint4 hi01 = valid ? make_uint4(r.codes[4].x, r.codes[4].y, r.codes[5].x, r.codes[5].y) : z4;
                const uint4 hi23 = valid ? make_uint4(r.codes[6].x, r.codes[6].y, r.codes[7].x, r.codes[7].y) : z4;
                const uint32_t slo = valid ? r.sc.x : 0u, shi = valid ? r.sc.y : 0u;
                const uint32_t own_buf = sbase + kOffOwnRaw + b * kRawBytes;
                sts_u128(raw_codes_at(own_buf, j, q), crank == 0 ? lo01 : hi01);
                sts_u128(raw_codes_at(own_buf, j, q) + 16, crank == 0 ? lo23 : hi23);
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(raw_scale_at(own_buf, j, q)), "r"(crank == 0 ? slo : shi)
                             : "memory");
                const uint32_t peer_buf = mapa_shared(sbase + kOffPeerRaw + b * kRawBytes, 1 - crank);
                const uint32_t peer_bar = mapa_shared(smem_addr(&ctl->peer_full[b]), 1 - crank);
                st_async_u4(raw_codes_at(peer_buf, j, q), crank == 0 ? hi01 : lo01, peer_bar);
                st_async_u4(raw_codes_at(peer_buf, j, q) + 16, crank == 0 ? hi23 : lo23, peer_bar);
                st_async_b32(raw_scale_at(peer_buf, j, q), crank == 0 ? shi : slo, peer_bar);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                arrive_leader(&ctl->kfull, crank);
                mbar_arrive(&ctl->own_full[b]);
            }
            // ---- next tile's record into registers (L2-prefetched a tile ago), prefetch the one after
            idx0 = idx1;
            idx1 = idx2;
            idx2 = index_of(i + 3);
            if (in_range(idx0))
                load_raw<R, kBlkOrder>(a.cache + static_cast<int64_t>(idx0) * R, q, r);
            else
                zero_raw(r);
            if (in_range(idx1)) prefetch_l2(a.cache + static_cast<int64_t>(idx1) * R + (q == 3 ? R - 1 : 128 * q));
        }
    } else if (warp < kWarpQK) {
        // ======================= V converters =======================
        const int t = threadIdx.x - 32 * kWarpV;
        const int j = t >> 2;
        const int q = t & 3;
        const uint32_t v_s = sbase + kOffV;
        const int row_own = kOwn * crank + j;
        const int row_peer = kOwn * (1 - crank) + j;
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
            const int b = i & 1;
            if (i == 0) ok = wait_warp(ctl, &ctl->qstaged, 0, a.status);   // the V buffer held q
            if (ok && i >= 1) ok = wait_warp(ctl, &ctl->pvdone, (i - 1) & 1, a.status);
            if (ok) ok = wait_warp(ctl, &ctl->own_full[b], (i >> 1) & 1, a.status);
            if (ok) ok = wait_warp(ctl, &ctl->peer_full[b], (i >> 1) & 1, a.status);
            if (!ok) break;
            const uint32_t own_buf = sbase + kOffOwnRaw + b * kRawBytes;
            const uint32_t peer_buf = sbase + kOffPeerRaw + b * kRawBytes;
            write_v(v_s, row_own, q, lds_u128(raw_codes_at(own_buf, j, q)), lds_u128(raw_codes_at(own_buf, j, q) + 16),
                    lds_u32(raw_scale_at(own_buf, j, q)));
            write_v(v_s, row_peer, q, lds_u128(raw_codes_at(peer_buf, j, q)),
                    lds_u128(raw_codes_at(peer_buf, j, q) + 16), lds_u32(raw_scale_at(peer_buf, j, q)));
            fence_proxy_async_smem();
            // the peer may send tile i + 2 into this buffer once it is armed again and released
            if (t == 0 && i + 2 < n_tiles) mbar_arrive_expect_tx(&ctl->peer_full[b], kRawBytes);
            __syncwarp();
            if (lane == 0) {
                arrive_leader(&ctl->vfull, crank);
                mbar_arrive(&ctl->own_empty[b]);
                mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->peer_empty[b]), 1 - crank));
            }
        }
    } else if (warp == kWarpQK) {
        // ======================= QK issuer (CTA 0) =======================
        if (crank == 0) {
            const uint32_t idesc_f16 = idesc_f16_f32(128, kTile, false, false);
            const uint32_t idesc_rope = R == 432 ? idesc_bf16_f32(128, kTile, false, false) : idesc_f16;
            const uint64_t kdesc0 = sdesc_sw128(sbase + kOffK, 16, 1024);
            const uint64_t qdesc0 = sdesc_sw128(sbase + kOffQs, 16, 1024);
            const bool leader = elect_one_in_warp();
            bool ok = wait_warp(ctl, &ctl->qready, 0, a.status);
            for (int i = 0; i < n_tiles && ok; ++i) {
                ok = wait_warp(ctl, &ctl->kfull, i & 1, a.status);
                if (ok && i >= 1) ok = wait_warp(ctl, &ctl->sfree, (i - 1) & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                if (leader) {
                    const uint32_t d = tmem + kColS;
#pragma unroll
                    for (int kk = 0; kk < 36; ++kk) {
                        const uint64_t kd = kdesc0 + static_cast<uint64_t>(((kk >> 2) * kBlk + (kk & 3) * 32) >> 4);
                        if (kk < kQTmemSteps)
                            mma_ts_cg2(d, tmem + kColQ + 8 * kk, kd, idesc_f16, kk > 0 ? 1u : 0u);
                        else
                            mma_ss_cg2(d, qdesc0 + static_cast<uint64_t>((((kk - 24) >> 2) * kBlk + (kk & 3) * 32) >> 4),
                                       kd, kk >= 32 ? idesc_rope : idesc_f16, 1u);
                    }
                    mma_commit_cg2(&ctl->qkdone, 0x3);
                }
                __syncwarp();
            }
            if (leader) mma_commit_cg2(&ctl->drain, 0x1);
            __syncwarp();
        }
    } else {
        // ======================= PV issuer (CTA 0) =======================
        if (crank == 0) {
            const uint32_t idesc_pv = idesc_f16_f32(128, 256, false, true);
            const uint64_t pdesc0 = sdesc_sw128(sbase + kOffP, 16, 1024);
            const uint64_t vdesc0 = sdesc_sw128(sbase + kOffV, kVBlk, 1024);
            const bool leader = elect_one_in_warp();
            bool ok = true;
            for (int i = 0; i < n_tiles && ok; ++i) {
                ok = wait_warp(ctl, &ctl->vfull, i & 1, a.status);
                if (ok) ok = wait_warp(ctl, &ctl->pfull, i & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks) {
                        const uint64_t pd = pdesc0 + static_cast<uint64_t>(((ks >> 2) * kBlk + (ks & 3) * 32) >> 4);
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj)
                            mma_ss_cg2(tmem + kColO + 128 * jj, pd,
                                       vdesc0 + static_cast<uint64_t>((2 * jj * kVBlk + ks * 2048) >> 4), idesc_pv,
                                       (i > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit_cg2(&ctl->pvdone, 0x3);
                }
                __syncwarp();
            }
            if (leader) mma_commit_cg2(&ctl->drain, 0x1);
            __syncwarp();
        }
    }

    // CTA 0 waits (bounded) until every MMA it issued has completed before anyone leaves
    if (crank == 0 && (warp == kWarpQK || warp == kWarpPV)) {
        if (!mbar_wait(&ctl->drain, 0)) set_abort(ctl, a.status);
    }
    tc_fence_before_sync();
    cluster_sync();   // no CTA leaves while its peer may still write its shared or tensor memory
    if (warp == kWarpQK) {
        tc_fence_after_sync();
        tmem_dealloc_cg2(tmem, kTmemCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

// q as bf16 [rows * 128, 576], box 64 dims x 64 heads, 128B swizzle.
bool encode_q_map(CUtensorMap* map, const void* q, int64_t heads) {
    const EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr || heads < 1 || heads > 0x7FFFFFFF) return false;
    const cuuint64_t dims[2] = {576u, static_cast<cuuint64_t>(heads)};
    const cuuint64_t strides[1] = {576u * 2u};
    const cuuint32_t box[2] = {64u, 64u};
    const cuuint32_t elem_strides[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int R, bool kBlkOrder>
cudaError_t prepare_kernel() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    err = cudaFuncSetAttribute(decode_pair_kernel<R, kBlkOrder>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (err == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_relaxed);
    return err;
}

}  // namespace
}  // namespace pairdec

bool decode_pair_supported(const DecodeArgs& d) { return d.h_q == 128 && (d.record_bytes == 352 || d.record_bytes == 432); }

int decode_pair_keys_per_split(int topk, int splits) {
    const int per = (topk + splits - 1) / splits;
    return (per + pairdec::kTile - 1) / pairdec::kTile * pairdec::kTile;
}

cudaError_t launch_decode_pair(const DecodeArgs& d, cudaStream_t stream) {
    using namespace pairdec;
    KernelArgs a;
    if (!encode_q_map(&a.qmap, d.q, static_cast<int64_t>(d.rows) * 128)) return cudaErrorInvalidValue;
    a.cache = d.cache;
    a.num_slots = d.num_slots;
    a.indices = d.indices;
    a.topk = d.topk;
    a.splits = d.splits;
    a.keys_per_split = decode_pair_keys_per_split(d.topk, d.splits);
    a.sm_scale = d.sm_scale;
    a.sink = d.attn_sink;
    a.out = static_cast<__nv_bfloat16*>(d.out);
    a.lse = d.lse;
    a.part_out = d.part_out;
    a.part_lse = d.part_lse;
    a.status = d.dev_status;
    const auto kernel = d.record_bytes == 432 ? decode_pair_kernel<432, false>
                        : d.block_scales      ? decode_pair_kernel<352, true>
                                              : decode_pair_kernel<352, false>;
    cudaError_t err = d.record_bytes == 432 ? prepare_kernel<432, false>()
                      : d.block_scales      ? prepare_kernel<352, true>()
                                            : prepare_kernel<352, false>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(d.rows) * static_cast<unsigned>(d.splits) * 2u);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddepcontrol.wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kernel, a);
    if (err == cudaSuccess) err = cudaGetLastError();
    return err;
}

}  // namespace nvfp4mla
