// sparse_decode_h64.cu -- sparse MLA decode for 64 query heads on one SM, with the scores computed
// transposed so that every MMA row is real work, for 352-byte and 432-byte NVFP4 records.
//
// What is computed (FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode",
// "Kernel:" paragraph and validation list): for query row t and head h, with J the used entries
// of t's index list,
//     z_j = sm_scale * q[t,h,:] . K_j          (K_j: 576 dequantized values of record j)
//     out = sum_j e^{z_j} V_j / (sum_j e^{z_j} + e^{sink_h}),   V_j = K_j[0:512]
//     lse = ln sum_j e^{z_j}
//
// Work split. One CTA per (query row, top-k split); keys in tiles of 128. With 64 heads an MMA
// with the heads on its M side (M = 128) would be half padding, so both contractions put keys or
// value dims on M instead:
//   S^T [128 keys x 64 heads] = K [128 x 576] . Q^T: M = 128 keys, N = 64 heads, 36 K-steps. K dims
//     0-511 come from shared memory, the 64 RoPE dims from tensor memory (A operand there); Q stays
//     in shared memory for the whole CTA (B operand, K-major).
//   O^T [512 dims x 64 heads] += V^T . P^T: four M = 128 (dims) x N = 64 x K = 128 (keys) MMAs.
//     V^T is the same shared-memory tile as K (dims 0-511), read MN-major: each record is
//     dequantized once, into one buffer, and serves both contractions.
// Tensor memory: O^T 256 columns (block b: lanes = dims 128b.., columns = heads), S^T 64 columns
// (lanes = keys), the RoPE rows of K 32 columns (lanes = keys), and each key lane's share of every
// head's row sum l, two buffers of 64 columns (kept there rather than in the softmax threads'
// registers; a tile reads one and writes the other).
// Shared memory: Q 72 KB, the K tile 128 KB (eight 64-dim blocks of 128 keys, 128B-swizzled), P^T
// 16 KB (128 keys x 64 heads, heads contiguous: the MN-major B operand of the PV MMAs).
// Pipeline. One buffer per operand. The converters refill K dims block b (128 dims) of tile k + 1
// as soon as the PV MMAs of tile k have read it; the QK MMAs of tile k + 1 follow the converters
// block by block; the softmax of tile k + 1 then writes P^T, and the PV MMAs of tile k + 1 start.
// The softmax warps load and convert the RoPE rows of tile k + 1 while they score tile k.
// Numbers. K is f16 (exact: e2m1 x e4m3 has <= 5 significant bits in [2^-10, 2688]; the bf16 RoPE
// of 432-byte records stays bf16 and those four K-steps run as bf16 MMAs). q enters as f16 scaled
// by a per-head power of two (2^pre with max|q| 2^pre in [2^14, 2^15)), so that the products
// q_d K_d are the same numbers as with bf16 q; S^T column h comes out as 2^pre_h times the exact
// score, which the softmax folds into its per-head scale. P is f16 (entries in [0, 2^8]).
// Softmax. A lazy reference maximum m_h per head (log2 domain): P = 2^(z - m) and O, l accumulate
// against m. A tile needs the reference to move only when some score exceeds m + 8. One pass over a
// key's scores writes P and the row sums against the current references and finds the largest
// z - m; the softmax warps then vote once per tile (one barrier reduction), and only when a
// reference has to move do they reduce the tile's maxima across keys (lanes), rescale O^T and redo
// the pass. Masked keys (index -1 or out of range) get zero K rows and P = 0: the thread that
// scores a key also loads its index.
// Warp roles (kThreads = 544, 17 warps):
//   0-7   softmax: warp w scores keys 32 (w & 3).. of a tile (its TMEM lane quadrant) for heads
//         32 (w >> 2)..+31, and writes the RoPE rows of those keys for the next tile; q staging in
//         the prologue; row sums, O^T / l and the output in the epilogue
//   8-15  converters: four threads per key (keys j and j + 64); thread q converts record bytes
//         64c + 16q .. + 15 (c = 0..3: 16-dim blocks 8c + 2q, 8c + 2q + 1). The next tile's bytes
//         are loaded into registers as soon as this tile no longer needs them (the scale bytes at
//         the start of a tile, the codes of block c right after block c is converted), and the
//         records two tiles ahead are prefetched into L2
//   16    MMA issuer (one elected thread) and tensor-memory owner
// Every wait is bounded by time; on timeout the CTA sets NVFP4_MLA_DEV_TIMEOUT, stops issuing work,
// drains what it issued and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "dequant.cuh"
#include "launch.h"
#include "sm103_ptx.cuh"

namespace nvfp4mla {
namespace h64dec {
namespace {

constexpr int kTile = 128;                 // keys per tile (M of the QK MMAs)
constexpr int kHeads = 64;
constexpr int kThreads = 544;
constexpr int kWarpConv = 8;
constexpr int kWarpMma = 16;
constexpr uint32_t kColO = 0;              // O^T: 4 blocks of 64 columns
constexpr uint32_t kColS = 256;            // S^T: 64 columns
constexpr uint32_t kColR = 320;            // RoPE rows of K: 32 columns (64 16-bit values a lane)
constexpr uint32_t kColL = 352;            // row-sum partials: two buffers of 64 columns (lane = key lane, column = head)
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// Shared memory (offsets from a 1024-byte aligned base)
constexpr int kQBlk = 8192;                // 64 heads x 128 B: one 64-dim block of Q
constexpr int kKBlk = 16384;               // 128 keys x 128 B: one 64-dim block of the K tile
constexpr int kOffCM = 256;                // float [32][4]: per head pair {ch_a, ch_b, -m_a, -m_b}: the score
                                           // scale sm_scale log2(e) 2^-pre and the negated reference maximum
constexpr int kOffAlpha = 768;             // float [64]: rescale factors (slow path), then 1 / l
constexpr int kOffXmax = 1024;             // float [64][4]: per-head maxima of the 4 key quadrants
constexpr int kOffQ = 2048;                // 9 blocks
constexpr int kOffK = kOffQ + 9 * kQBlk;   // 8 blocks
constexpr int kOffP = kOffK + 8 * kKBlk;   // P^T [128 keys x 128 B]
constexpr int kSmemBytes = kOffP + kTile * 128;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory");
static_assert(kOffQ % 1024 == 0 && kOffK % 1024 == 0 && kOffP % 1024 == 0, "operand alignment");
static_assert(kHeads * 129 * 4 <= 8 * kKBlk, "row-sum exchange fits in the K tile");

struct __align__(8) Ctl {
    uint64_t qload;           // q boxes landed (TMA, tx-counted)
    uint64_t qready;          // 8 softmax warps: q converted in shared memory
    uint64_t kfull[4];        // 8 converter warps: K dims block b (dims 128b..) of the tile written
    uint64_t ropefull;        // 8 softmax warps: RoPE rows of the tile in tensor memory
    uint64_t sfull;           // QK commit: S^T ready (every earlier MMA completed too)
    uint64_t pfull;           // 8 softmax warps: P^T written (and O^T rescaled)
    uint64_t pvblk[4];        // PV commit after dims block b: K block b free; block 3: O^T and P^T done
    uint64_t drain;           // every MMA issued completed
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(Ctl) <= kOffCM, "control block");

struct KernelArgs {
    CUtensorMap qmap;         // q as bf16 [rows * 64, 576], box 64 dims x 64 heads, 128B swizzle
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
    uint16_t* part_out;       // f16 partial outputs [rows, splits, 64, 512]
    float* part_lse;          // log2 domain
    uint32_t* status;
};

__device__ __forceinline__ void set_abort(Ctl* ctl, uint32_t* status) {
    if (atomicExch(&ctl->abort, 1u) == 0u && status != nullptr) atomicOr(status, 0x4u);
}
__device__ __forceinline__ bool aborted(Ctl* ctl) { return *reinterpret_cast<volatile uint32_t*>(&ctl->abort) != 0u; }

// Bounded wait, one answer per warp.
__device__ __forceinline__ bool wait_warp(Ctl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    bool ok = mbar_try_wait(bar, parity);
    if (!ok && !aborted(ctl)) {
        ok = mbar_wait(bar, parity);
        if (!ok) set_abort(ctl, status);
    }
    return __all_sync(0xffffffffu, ok);
}

// Read-only global loads that do not allocate in L1 (every record byte is used once per CTA).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) { asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory"); }

__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// One key's share of a converter thread q (0..3): record bytes 64c + 16q .. + 15 (c = 0..3), the codes
// of 16-dim blocks 8c + 2q and 8c + 2q + 1, and the scale bytes of those blocks.
template <int R, bool kBlkOrder>
struct KeyRaw {
    // 352-byte records with the permuted placement (block s at 320 + 8 (s & 3) + (s >> 2)): the eight
    // scale bytes of the thread's blocks lie in one 16-byte half of the field; otherwise all 32 bytes
    static constexpr bool kPermuted = R == 352 && !kBlkOrder;
    uint4 codes[4];
    uint4 sc[kPermuted ? 1 : 2];

    __device__ __forceinline__ void load_codes(const uint8_t* rec, int q, int c) { codes[c] = ldg_stream16(rec + 64 * c + 16 * q); }
    __device__ __forceinline__ void load_scales(const uint8_t* rec, int q) {
        if constexpr (kPermuted) {
            sc[0] = ldg_stream16(rec + 320 + 16 * (q & 1));
        } else {
            constexpr int sb = R == 352 ? 320 : 256;
            sc[0] = ldg_stream16(rec + sb);
            sc[1] = ldg_stream16(rec + sb + 16);
        }
    }
    __device__ __forceinline__ void load(const uint8_t* rec, int q) {
#pragma unroll
        for (int c = 0; c < 4; ++c) load_codes(rec, q, c);
        load_scales(rec, q);
    }
    // the scale pairs of blocks c = 0..3, two per word (c even: low half)
    __device__ __forceinline__ void scale_pairs(int q, uint32_t (&sp)[2]) const {
        sp[0] = (scale_pair(0, q) & 0xFFFFu) | (scale_pair(1, q) << 16);
        sp[1] = (scale_pair(2, q) & 0xFFFFu) | (scale_pair(3, q) << 16);
    }
    // byte 0: the scale of block 8c + 2q, byte 1: of block 8c + 2q + 1
    __device__ __forceinline__ uint32_t scale_pair(int c, int q) const {
        if constexpr (kPermuted) {
            // block 8c + 2q at byte 16 (q & 1) + 2c + (q >> 1), the next block eight bytes further
            const uint32_t wa = c < 2 ? sc[0].x : sc[0].y, wb = c < 2 ? sc[0].z : sc[0].w;
            const uint32_t bi = static_cast<uint32_t>(2 * c + (q >> 1)) & 3u;
            return __byte_perm(wa, wb, bi | ((bi + 4u) << 4));
        } else {
            // block s at byte s: bytes 2q, 2q + 1 of word 2c + (q >> 1)
            const uint32_t w[8] = {sc[0].x, sc[0].y, sc[0].z, sc[0].w, sc[1].x, sc[1].y, sc[1].z, sc[1].w};
            const uint32_t wv = (q >> 1) != 0 ? w[2 * c + 1] : w[2 * c];
            const uint32_t lo = 2u * static_cast<uint32_t>(q & 1);
            return __byte_perm(wv, 0u, lo | ((lo + 1u) << 4));
        }
    }
};

template <int R, bool kBlkOrder>
__global__ void __launch_bounds__(kThreads, 1) decode_h64_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    Ctl* ctl = reinterpret_cast<Ctl*>(smem);
    const uint32_t sbase = smem_addr(smem);

    const int split = blockIdx.x % a.splits;
    const int row = blockIdx.x / a.splits;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int key_begin = split * a.keys_per_split;
    const int key_end = min(a.topk, key_begin + a.keys_per_split);
    const int n_tiles = key_end > key_begin ? (key_end - key_begin + kTile - 1) / kTile : 0;
    const int32_t* idx_row = a.indices + static_cast<int64_t>(row) * a.topk;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->qload, 1);
        mbar_init(&ctl->qready, 8);
        for (int b = 0; b < 4; ++b) {
            mbar_init(&ctl->kfull[b], 8);
            mbar_init(&ctl->pvblk[b], 1);
        }
        mbar_init(&ctl->ropefull, 8);
        mbar_init(&ctl->sfull, 1);
        mbar_init(&ctl->pfull, 8);
        mbar_init(&ctl->drain, 1);
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
    // Launched as a programmatic dependent of the preceding kernel: nothing is read before that grid
    // has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    auto index_at = [&](int i, int key) -> int32_t {   // key 0..127 of tile i
        if (i >= n_tiles) return -1;
        const int pos = key_begin + kTile * i + key;
        return pos < key_end ? __ldg(idx_row + pos) : -1;
    };
    auto in_range = [&](int32_t v) { return v >= 0 && static_cast<int64_t>(v) < a.num_slots; };

    if (warp < 8) {
        // ======================= softmax warps =======================
        const int qd = warp & 3;              // TMEM lane quadrant: keys 32 qd.. of a tile
        const int h2 = warp >> 2;             // heads 32 h2 ..
        const int key = 32 * qd + lane;
        const int hb = 32 * h2;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        const uint32_t cm_s = sbase + kOffCM;         // head pair u at cm_s + 16 u
        const uint32_t alpha_s = sbase + kOffAlpha;   // head h at alpha_s + 4 h
        const uint32_t xmax_s = sbase + kOffXmax;     // head h, quadrant r at xmax_s + 16 h + 4 r
        auto ch_addr = [&](int h) { return cm_s + 16 * (h >> 1) + 4 * (h & 1); };
        auto negm_addr = [&](int h) { return cm_s + 16 * (h >> 1) + 8 + 4 * (h & 1); };
        // RoPE bytes of this key for heads-half h2's 32 dims: 32 e4m3 (352) or 32 bf16 (432)
        constexpr int kRopeVec = R == 352 ? 2 : 4;
        uint4 rope[kRopeVec];
        auto load_rope = [&](int32_t v) {
            if (in_range(v)) {
                const uint8_t* src = a.cache + static_cast<int64_t>(v) * R + (R == 352 ? 256 + 32 * h2 : 304 + 64 * h2);
#pragma unroll
                for (int e = 0; e < kRopeVec; ++e) rope[e] = ldg_stream16(src + 16 * e);
            }
        };
        // RoPE rows (dims 32 h2 ..) of this key into tensor memory; zero for a masked key
        auto store_rope = [&](bool valid) {
            uint32_t v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0u;
            if (valid) {
                if constexpr (R == 352) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t w[4] = {rope[e].x, rope[e].y, rope[e].z, rope[e].w};
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const uint2 f = e4m3x4_to_f16(w[m]);
                            v[8 * e + 2 * m] = f.x;
                            v[8 * e + 2 * m + 1] = f.y;
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[4 * e] = rope[e].x;
                        v[4 * e + 1] = rope[e].y;
                        v[4 * e + 2] = rope[e].z;
                        v[4 * e + 3] = rope[e].w;
                    }
                }
            }
            tmem_st16(lane_base + kColR + 16 * h2, v);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->ropefull);
        };

        // ---- prologue: q into shared memory (TMA), per-head prescale, f16 (bf16 RoPE for 432) in place
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&ctl->qload, 9u * kQBlk);
            for (int bx = 0; bx < 9; ++bx)
                tma_load_2d(sbase + kOffQ + bx * kQBlk, &a.qmap, 64 * bx, row * kHeads, &ctl->qload);
        }
        int32_t cur_idx = index_at(0, key);
        load_rope(cur_idx);
        int32_t next_idx = index_at(1, key);   // the index of the next tile's key, a tile ahead of its RoPE loads
        bool ok = wait_warp(ctl, &ctl->qload, 0, a.status);
        {
            const int hq = threadIdx.x >> 2;   // head 0..63
            const int part = threadIdx.x & 3;  // 18 of the head's 72 chunks of 8 dims
            float qmax = 0.0f;
            if (ok) {
#pragma unroll 6
                for (int k = 18 * part; k < 18 * part + 18; ++k) {
                    const uint4 x = lds_u128(sbase + kOffQ + (k >> 3) * kQBlk + swz(hq, k & 7));
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        qmax = fmax3(qmax, fabsf(__uint_as_float(w[m] << 16)), fabsf(__uint_as_float(w[m] & 0xFFFF0000u)));
                }
            }
            qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
            qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
            int pre = 0;
            if (qmax > 0.0f) {
                int e;
                frexpf(qmax, &e);   // qmax < 2^e <= 2 qmax
                pre = min(100, max(-100, 15 - e));
            }
            const float fpre = __int_as_float((127 + pre) << 23);
            if (part == 0) {
                sts_f32(ch_addr(hq), a.sm_scale * kLog2e * __int_as_float((127 - pre) << 23));   // S' = 2^pre S, z = ch S'
                sts_f32(negm_addr(hq), INFINITY);   // reference maximum -inf
            }
            if (ok) {
#pragma unroll 6
                for (int k = 18 * part; k < 18 * part + 18; ++k) {
                    const bool bf = R == 432 && k >= 64;   // bf16 RoPE of 432-byte records
                    const uint32_t addr = sbase + kOffQ + (k >> 3) * kQBlk + swz(hq, k & 7);
                    const uint4 x = lds_u128(addr);
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
                    uint32_t y[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float lo = __uint_as_float(w[m] << 16) * fpre, hi = __uint_as_float(w[m] & 0xFFFF0000u) * fpre;
                        y[m] = bf ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
                    }
                    sts_u128(addr, make_uint4(y[0], y[1], y[2], y[3]));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->qready);
        }
        bool valid = in_range(cur_idx);
        store_rope(ok && valid);
        named_bar_sync(1, 256);   // per-head scales and maxima are written

        {   // this key lane's share of each head's sum of 2^(z - m), in tensor memory
            uint32_t zero[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) zero[j] = 0u;
            tmem_st32(lane_base + kColL + hb, zero);
            tmem_wait_st();
        }
        const uint32_t p_row = sbase + kOffP + (key >> 3) * 1024 + (key & 7) * 128;   // this key's row of P^T
        // Every softmax warp takes part in every named barrier below, also after a wait ran out
        // (then it only passes the barriers), so no warp can be left waiting on a missing one.
        // One pass over this key's scores: P^T row = 2^(z - m) in f16 (0 for a masked key) against the
        // current references, the row sums l_new = alpha l_old + P (alpha = 1 unless `rescale`), and
        // the largest z - m. P^T of the previous tile was read by its PV, which completed before this
        // tile's QK did. The sums go to the other of two TMEM buffers, so that a tile whose vote
        // moves a reference can redo the pass from the previous sums.
        auto score = [&](uint32_t l_old, uint32_t l_new, bool rescale) -> float {
            float tmax = -INFINITY;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t sv[16], lv[16];
                tmem_ld16(lane_base + kColS + hb + 16 * half, sv);
                tmem_ld16(lane_base + l_old + hb + 16 * half, lv);
                tmem_wait_ld();
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t pw[4];
#pragma unroll
                    for (int g2 = 0; g2 < 4; ++g2) {
                        const int e = 8 * c2 + 2 * g2;     // column in sv / lv
                        const int h = hb + 16 * half + e;  // heads h, h + 1
                        const uint4 c = lds_u128(cm_s + 16 * (h >> 1));
                        const float2 z = f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                                f32x2_pack(__uint_as_float(c.x), __uint_as_float(c.y)),
                                                                f32x2_pack(__uint_as_float(c.z), __uint_as_float(c.w))));
                        tmax = fmax3(tmax, z.x, z.y);
                        const float p0 = valid ? ex2_approx(z.x) : 0.0f, p1 = valid ? ex2_approx(z.y) : 0.0f;
                        uint64_t l2 = f32x2_pack(__uint_as_float(lv[e]), __uint_as_float(lv[e + 1]));
                        if (rescale) {
                            const uint2 al = lds_u64(alpha_s + 4 * h);
                            l2 = f32x2_fma(l2, f32x2_pack(__uint_as_float(al.x), __uint_as_float(al.y)), f32x2_pack(p0, p1));
                        } else {
                            l2 = f32x2_add(l2, f32x2_pack(p0, p1));
                        }
                        const float2 ls = f32x2_unpack(l2);
                        lv[e] = __float_as_uint(ls.x);
                        lv[e + 1] = __float_as_uint(ls.y);
                        pw[g2] = pack_f16x2(p0, p1);
                    }
                    sts_u128(p_row + (((4 * h2 + 2 * half + c2) ^ (key & 7)) << 4), make_uint4(pw[0], pw[1], pw[2], pw[3]));
                }
                tmem_st16(lane_base + l_new + hb + 16 * half, lv);
            }
            return valid ? tmax : -INFINITY;
        };
        for (int i = 0; i < n_tiles; ++i) {
            if (i + 1 < n_tiles) load_rope(next_idx);   // in flight while this tile is scored
            const int32_t next2_idx = index_at(i + 2, key);
            const uint32_t l_old = kColL + 64 * (i & 1), l_new = kColL + 64 * ((i + 1) & 1);
            float tmax = -INFINITY;
            if (ok) ok = wait_warp(ctl, &ctl->sfull, i & 1, a.status);
            if (ok) {
                // (tensor-memory loads and stores are warp-collective: every lane takes part, and a
                // masked key only changes the values)
                tc_fence_after_sync();
                tmax = score(l_old, l_new, false);
            }
            // ---- does any head need a new reference? (one barrier reduction)
            if (bar_red_or(1, 256, tmax > kRescaleThreshold)) {
                // per head: the tile's largest z over the 128 keys (warp maximum, then the 4 quadrants)
                float mine = -INFINITY;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t sv[16];
                    if (ok) {
                        tmem_ld16(lane_base + kColS + hb + 16 * half, sv);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float z = (ok && valid) ? __uint_as_float(sv[e]) * lds_f32(ch_addr(hb + 16 * half + e)) : -INFINITY;
                        const float wm = warp_max(z);
                        if (lane == 16 * half + e) mine = wm;
                    }
                }
                sts_f32(xmax_s + 16 * (hb + lane) + 4 * qd, mine);
                named_bar_sync(1, 256);
                if (qd == 0) {   // one thread per head: the new reference and the rescale factor
                    const uint4 x = lds_u128(xmax_s + 16 * (hb + lane));
                    const float zt = fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)),
                                           fmaxf(__uint_as_float(x.z), __uint_as_float(x.w)));
                    const float mo = -lds_f32(negm_addr(hb + lane));
                    float al = 1.0f;
                    if (zt > mo + kRescaleThreshold) {
                        al = mo == -INFINITY ? 0.0f : ex2_approx(mo - zt);
                        sts_f32(negm_addr(hb + lane), -zt);
                    }
                    sts_f32(alpha_s + 4 * (hb + lane), al);
                }
                named_bar_sync(1, 256);
                if (ok && i > 0) {
                    // O^T (dims 128b + key lane, this warp's heads) *= alpha; PV of the previous tile
                    // has completed (it was issued before the QK whose commit was just waited for)
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {   // 16 columns at a time
                        const uint32_t col = kColO + 64 * (c >> 1) + hb + 16 * (c & 1);
                        uint32_t o[16];
                        tmem_ld16(lane_base + col, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * lds_f32(alpha_s + 4 * (hb + 16 * (c & 1) + e)));
                        tmem_st16(lane_base + col, o);
                    }
                }
                // P and the sums again against the moved references
                if (ok) (void)score(l_old, l_new, true);
            }
            if (!ok) continue;
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->pfull);
            // ---- RoPE rows of the next tile (this tile's QK, which read the current ones, is done)
            valid = in_range(next_idx);
            if (i + 1 < n_tiles) store_rope(valid);
            next_idx = next2_idx;
        }

        // ---- epilogue: row sums, O^T / l, out (or the split's partial) and lse
        bool have_o = false;
        if (ok && n_tiles > 0) {
            have_o = wait_warp(ctl, &ctl->pvblk[3], (n_tiles - 1) & 1, a.status);
            if (have_o) tc_fence_after_sync();
        }
        named_bar_sync(1, 256);   // every MMA has read the K tile (or timed out): it holds the sums now
        float* xl = reinterpret_cast<float*>(smem + kOffK);   // [64 heads][129]
        {
            uint32_t lv[32];
            tmem_ld32(lane_base + kColL + 64 * (n_tiles & 1) + hb, lv);   // the buffer the last tile wrote
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) xl[(hb + j) * 129 + key] = __uint_as_float(lv[j]);
        }
        named_bar_sync(1, 256);
        {
            const int hh = threadIdx.x >> 2, part = threadIdx.x & 3;
            float sum = 0.0f;
#pragma unroll 8
            for (int e = 0; e < 32; ++e) sum += xl[hh * 129 + 32 * part + e];
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (part == 0) {
                const float mref = -lds_f32(negm_addr(hh));
                const bool empty = !(sum > 0.0f);
                const float lse2 = empty ? -INFINITY : mref + log2f(sum);
                float factor = 0.0f;
                if (!empty) {
                    float denom = sum;
                    if (a.splits == 1 && a.sink != nullptr) denom += exp2f(__ldg(a.sink + hh) * kLog2e - mref);
                    factor = 1.0f / denom;
                }
                sts_f32(alpha_s + 4 * hh, factor);
                if (a.splits == 1)
                    a.lse[static_cast<int64_t>(row) * kHeads + hh] = lse2 * kLn2;
                else
                    a.part_lse[(static_cast<int64_t>(row) * a.splits + split) * kHeads + hh] = lse2;
            }
        }
        named_bar_sync(1, 256);
        // O^T block b: this thread's lane is dim 128b + 32qd + lane; each warp store covers 32
        // consecutive dims of one head (64 bytes)
        uint16_t* dst = a.splits == 1 ? reinterpret_cast<uint16_t*>(a.out) + static_cast<int64_t>(row) * kHeads * 512
                                      : a.part_out + (static_cast<int64_t>(row) * a.splits + split) * kHeads * 512;
        const bool bf16_out = a.splits == 1;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {   // O^T block c >> 1, 16 of this warp's heads
            const int b = c >> 1, h0 = hb + 16 * (c & 1);
            uint32_t o[16];
            if (have_o) {
                tmem_ld16(lane_base + kColO + 64 * b + h0, o);
                tmem_wait_ld();
            }
            uint16_t* p = dst + static_cast<int64_t>(h0) * 512 + 128 * b + 32 * qd + lane;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float v = have_o ? __uint_as_float(o[e]) * lds_f32(alpha_s + 4 * (h0 + e)) : 0.0f;
                p[e * 512] = bf16_out ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
            }
        }
    } else if (warp < kWarpMma) {
        // ============ converters: K dims 0-511 of keys j and j + 64, 16-dim blocks 8c + 2q, 8c + 2q + 1 ============
        const int t = threadIdx.x - 32 * kWarpConv;
        // lane l of converter warp w: key 8w + (l & 7) (and 64 more), quarter q = l >> 3, so that the
        // eight lanes of a quarter-warp store to eight different 16-byte bank slots (eight keys, one
        // q), while the four quarters of a key still load one contiguous 64-byte run per instruction
        const int q = (t >> 3) & 3;
        const int j = (t & 7) + 8 * (t >> 5);
        const uint32_t k_s = sbase + kOffK;
        bool ok = !aborted(ctl);
        KeyRaw<R, kBlkOrder> r0, r1;
        int32_t i0 = index_at(0, j), i1 = index_at(0, j + 64);
        if (in_range(i0)) r0.load(a.cache + static_cast<int64_t>(i0) * R, q);
        if (in_range(i1)) r1.load(a.cache + static_cast<int64_t>(i1) * R, q);
        int32_t n0 = index_at(1, j), n1 = index_at(1, j + 64);
        int32_t m0 = index_at(2, j), m1 = index_at(2, j + 64);
        // The records two tiles ahead go into L2 (the four threads of a key touch every 128-byte line
        // of its record: points 64 apart), so that the register loads of the next tile find them there.
        auto prefetch_record = [&](int32_t v) {
            if (in_range(v)) {
                const uint8_t* rec = a.cache + static_cast<int64_t>(v) * R;
                prefetch_l2(rec + min(128 * q, R - 1));
                prefetch_l2(rec + min(128 * q + 64, R - 1));
            }
        };
        for (int k = 0; k < n_tiles; ++k) {
            const bool v0 = in_range(i0), v1 = in_range(i1);
            if (q == 0 && ((i0 >= 0 && !v0) || (i1 >= 0 && !v1)) && a.status != nullptr) atomicOr(a.status, 0x2u);
            // The next tile's record bytes go out as soon as this tile no longer needs the registers
            // they land in: the scale bytes now (this tile's scale pairs are taken first), the codes of
            // block b right after block b is converted.
            uint32_t sp0[2], sp1[2];
            r0.scale_pairs(q, sp0);
            r1.scale_pairs(q, sp1);
            const bool ld0 = in_range(n0), ld1 = in_range(n1);
            const uint8_t* rec0 = a.cache + static_cast<int64_t>(ld0 ? n0 : 0) * R;
            const uint8_t* rec1 = a.cache + static_cast<int64_t>(ld1 ? n1 : 0) * R;
            if (ld0) r0.load_scales(rec0, q);
            if (ld1) r1.load_scales(rec1, q);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                // dims 128b .. 128b + 127 once the previous tile's PV has read them: 64-dim block
                // 2b + (q >> 1), chunks 4 (q & 1) .. + 3 of each of the thread's two keys
                if (k >= 1) ok = wait_warp(ctl, &ctl->pvblk[b], (k - 1) & 1, a.status);
                if (!ok) break;
                const uint32_t blk = k_s + (2 * b + (q >> 1)) * kKBlk;
                const int ch0 = 4 * (q & 1);
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                {
                    const uint32_t sp = sp0[b >> 1] >> (16 * (b & 1));
                    const __half2 sa = scale_half2(sp & 0xFFu), sb = scale_half2((sp >> 8) & 0xFFu);
                    sts_u128(blk + swz(j, ch0), v0 ? dq8(r0.codes[b].x, sa) : z);
                    sts_u128(blk + swz(j, ch0 + 1), v0 ? dq8(r0.codes[b].y, sa) : z);
                    sts_u128(blk + swz(j, ch0 + 2), v0 ? dq8(r0.codes[b].z, sb) : z);
                    sts_u128(blk + swz(j, ch0 + 3), v0 ? dq8(r0.codes[b].w, sb) : z);
                }
                {
                    const uint32_t sp = sp1[b >> 1] >> (16 * (b & 1));
                    const __half2 sa = scale_half2(sp & 0xFFu), sb = scale_half2((sp >> 8) & 0xFFu);
                    sts_u128(blk + swz(j + 64, ch0), v1 ? dq8(r1.codes[b].x, sa) : z);
                    sts_u128(blk + swz(j + 64, ch0 + 1), v1 ? dq8(r1.codes[b].y, sa) : z);
                    sts_u128(blk + swz(j + 64, ch0 + 2), v1 ? dq8(r1.codes[b].z, sb) : z);
                    sts_u128(blk + swz(j + 64, ch0 + 3), v1 ? dq8(r1.codes[b].w, sb) : z);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->kfull[b]);
                if (ld0) r0.load_codes(rec0, q, b);
                if (ld1) r1.load_codes(rec1, q, b);
            }
            if (!ok) break;
            prefetch_record(m0);
            prefetch_record(m1);
            i0 = n0;
            i1 = n1;
            n0 = m0;
            n1 = m1;
            m0 = index_at(k + 3, j);
            m1 = index_at(k + 3, j + 64);
        }
    } else {
        // ======================= MMA issuer =======================
        const uint32_t idesc_qk = idesc_f16_f32(128, 64, false, false);
        const uint32_t idesc_rope = R == 432 ? idesc_bf16_f32(128, 64, false, false) : idesc_qk;
        const uint32_t idesc_pv = idesc_f16_f32(128, 64, true, true);
        const uint64_t kdesc0 = sdesc_sw128(sbase + kOffK, 16, 1024);       // K-major: keys x dims
        const uint64_t qdesc0 = sdesc_sw128(sbase + kOffQ, 16, 1024);       // K-major: heads x dims
        const uint64_t vdesc0 = sdesc_sw128(sbase + kOffK, kKBlk, 1024);    // MN-major: dims x keys
        const uint64_t pdesc0 = sdesc_sw128(sbase + kOffP, kTile * 128, 1024);   // MN-major: heads x keys
        const bool leader = elect_one_in_warp();
        bool ok = wait_warp(ctl, &ctl->qready, 0, a.status);
        for (int i = 0; i < n_tiles && ok; ++i) {
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {   // dims 128b .. 128b + 127 as soon as they are converted
                ok = wait_warp(ctl, &ctl->kfull[b], i & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                if (leader) {
#pragma unroll
                    for (int kk = 8 * b; kk < 8 * b + 8; ++kk)
                        mma_ss(tmem + kColS, kdesc0 + static_cast<uint64_t>(((kk >> 2) * kKBlk + (kk & 3) * 32) >> 4),
                               qdesc0 + static_cast<uint64_t>(((kk >> 2) * kQBlk + (kk & 3) * 32) >> 4), idesc_qk,
                               kk > 0 ? 1u : 0u);
                }
                __syncwarp();
            }
            if (ok) ok = wait_warp(ctl, &ctl->ropefull, i & 1, a.status);
            if (!ok) break;
            tc_fence_after_sync();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)   // dims 512-575: K rows from tensor memory
                    mma_ts(tmem + kColS, tmem + kColR + 8 * kk, qdesc0 + static_cast<uint64_t>((8 * kQBlk + kk * 32) >> 4),
                           idesc_rope, 1u);
                mma_commit(&ctl->sfull);
            }
            __syncwarp();
            ok = wait_warp(ctl, &ctl->pfull, i & 1, a.status);
            if (!ok) break;
            tc_fence_after_sync();
            if (leader) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
#pragma unroll
                    for (int s = 0; s < 8; ++s)   // keys 16s .. 16s + 15
                        mma_ss(tmem + kColO + 64 * b, vdesc0 + static_cast<uint64_t>((2 * b * kKBlk + s * 2048) >> 4),
                               pdesc0 + static_cast<uint64_t>((s * 2048) >> 4), idesc_pv, (i > 0 || s > 0) ? 1u : 0u);
                    mma_commit(&ctl->pvblk[b]);
                }
            }
            __syncwarp();
        }
        if (leader) mma_commit(&ctl->drain);
        __syncwarp();
        if (!mbar_wait(&ctl->drain, 0)) set_abort(ctl, a.status);
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
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

// q as bf16 [rows * 64, 576], box 64 dims x 64 heads, 128B swizzle.
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
    err = cudaFuncSetAttribute(decode_h64_kernel<R, kBlkOrder>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (err == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_relaxed);
    return err;
}

}  // namespace
}  // namespace h64dec

bool decode_h64_supported(const DecodeArgs& d) { return d.h_q == 64 && (d.record_bytes == 352 || d.record_bytes == 432); }

int decode_h64_keys_per_split(int topk, int splits) {
    const int per = (topk + splits - 1) / splits;
    return (per + h64dec::kTile - 1) / h64dec::kTile * h64dec::kTile;
}

cudaError_t launch_decode_h64(const DecodeArgs& d, cudaStream_t stream) {
    using namespace h64dec;
    KernelArgs a;
    if (!encode_q_map(&a.qmap, d.q, static_cast<int64_t>(d.rows) * kHeads)) return cudaErrorInvalidValue;
    a.cache = d.cache;
    a.num_slots = d.num_slots;
    a.indices = d.indices;
    a.topk = d.topk;
    a.splits = d.splits;
    a.keys_per_split = decode_h64_keys_per_split(d.topk, d.splits);
    a.sm_scale = d.sm_scale;
    a.sink = d.attn_sink;
    a.out = static_cast<__nv_bfloat16*>(d.out);
    a.lse = d.lse;
    a.part_out = d.part_out;
    a.part_lse = d.part_lse;
    a.status = d.dev_status;
    const auto kernel = d.record_bytes == 432 ? decode_h64_kernel<432, false>
                        : d.block_scales      ? decode_h64_kernel<352, true>
                                              : decode_h64_kernel<352, false>;
    cudaError_t err = d.record_bytes == 432 ? prepare_kernel<432, false>()
                      : d.block_scales      ? prepare_kernel<352, true>()
                                            : prepare_kernel<352, false>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(d.rows) * static_cast<unsigned>(d.splits));
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
