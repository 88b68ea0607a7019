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
//   A CTA dequantizes its own keys' K rows (576 dims) from their whole records, and the V rows of
//   its own half of the dims for all 128 keys from that half's codes and scales. Both CTAs read
//   the V half of a record around the time its owner reads the whole, so DRAM delivers each
//   record once per pair and the second read comes from L2.
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
//   8-15  K converters: K rows of the own keys, blocks 0-3 as soon as the previous QK has read
//         its first half, blocks 4-8 once it has finished
//   16-23 V converters: V rows of keys 0-63 once the previous PV has read them, then of keys
//         64-127; they also help to stage q
//         Converter threads stage the record bytes they convert with cp.async one tile ahead, so
//         no load sits between a thread's conversion and its arrive
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

#include "dequant.cuh"
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
constexpr int kOffXmax = 512;              // float [8][64]: maxima of q, tile maxima (slow path)
constexpr int kOffXl = 2560;               // float [4][64]: row sums
constexpr int kOffK = 4096;                // 9 blocks: K rows of the 64 own keys (K-major)
constexpr int kOffV = kOffK + 9 * kBlk;    // 4 blocks of 128 keys: this CTA's 256 V dims (MN-major)
constexpr int kOffP = kOffV + 4 * kVBlk;   // 2 blocks: P [64 heads x 128 keys] (K-major)
constexpr int kOffQs = kOffP + 2 * kBlk;   // 3 blocks: q dims [384, 576)
// Staging (cp.async, one tile ahead; entry strides are 8 words modulo 32 banks, so the 64-bit reads
// of a quarter-warp's 4 keys x 4 quarters meet 32 different banks, except 144-byte V entries):
//   a: [64 own keys] record bytes 0-127 (codes of blocks 0-15), then the 32 scale bytes
//   b: [64 own keys] record bytes 128-255 (codes of blocks 16-31), then the RoPE bytes
//   v: [2 halves][64 keys] this CTA's 128 code bytes (record bytes 128 crank ..), then the 16 scale
//      bytes of its 32 blocks
constexpr int kStrA = 160;
template <int R> constexpr int kStrB = R == 352 ? 224 : 288;
template <int R> constexpr int kStrV = R == 352 ? 160 : 144;
constexpr int kOffStA = kOffQs + 3 * kBlk;
constexpr int kOffStB = kOffStA + kOwn * kStrA;
template <int R> constexpr int kOffStV = kOffStB + kOwn * kStrB<R>;
template <int R> constexpr int kSmemBytes = kOffStV<R> + 2 * kOwn * kStrV<R>;
template <int R> constexpr int kSmemAlloc = kSmemBytes<R> + 1024;
static_assert(kSmemAlloc<352> <= 232448 && kSmemAlloc<432> <= 232448, "shared memory");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0 && kOffQs % 1024 == 0, "operand alignment");
static_assert(9 * kBlk <= 4 * kVBlk + 2 * kBlk, "q staging fits in the V and P buffers");
static_assert(kHeads * 1024 <= 9 * kBlk, "output staging fits in the K buffer");

// Buffers are handed back in halves so that converters refill one half while the MMAs still
// read the other: K blocks 0-3 (dims 0-255) and 4-8, V rows / P columns of keys 0-63 and 64-127.
struct __align__(8) Ctl {
    uint64_t khalf;           // QK commit after dims 0-255 (multicast): K blocks 0-3 free
    uint64_t qkdone;          // QK commit (multicast): S ready, K buffer free
    uint64_t pvhalf;          // PV commit after keys 0-63 (multicast): V rows / P columns 0-63 free
    uint64_t pvdone;          // PV commit (multicast): V and P buffers free, O updated
    uint64_t kfull_a;         // CTA 0: 16 warps (8 per CTA) wrote K blocks 0-3
    uint64_t kfull_b;         // CTA 0: 16 warps wrote K blocks 4-8
    uint64_t vfull_a;         // CTA 0: 16 warps wrote V rows 0-63
    uint64_t vfull_b;         // CTA 0: 16 warps wrote V rows 64-127
    uint64_t sfree;           // CTA 0: 16 softmax warps read S
    uint64_t pfull_a;         // CTA 0: 16 softmax warps: P columns 0-63 written, O rescaled
    uint64_t pfull_b;         // CTA 0: 8 softmax warps (lanes 64-127) wrote P columns 64-127
    uint64_t qready;          // CTA 0: 32 warps (16 per CTA) put q into tensor and shared memory
    uint64_t qstaged;         // 16 local warps finished reading the q staging area
    uint64_t qload;           // q boxes landed (TMA, tx-counted)
    uint64_t drain;           // CTA 0: both issuers' MMAs completed
    uint32_t tmem_base;
    uint32_t abort;
    uint32_t sig_sink;        // target of the 4-byte st.async signals (the value is never read)
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
    int merge;                // 1: the row's splits share a cluster (pair p = ranks 2p, 2p + 1) and pair 0
                              // merges their partials into out and lse after the whole cluster is done
};

__device__ __forceinline__ void set_abort(Ctl* ctl, uint32_t* status) {
    if (atomicExch(&ctl->abort, 1u) == 0u && status != nullptr) atomicOr(status, 0x4u);
}
__device__ __forceinline__ bool aborted(Ctl* ctl) { return *reinterpret_cast<volatile uint32_t*>(&ctl->abort) != 0u; }

// Bounded wait, one answer per warp. CTA-scope acquire for barriers that this CTA's threads or the
// pair's MMA commits complete; cluster-scope acquire (wait_peer) for those that the peer CTA's
// st.async data or signals complete.
__device__ __forceinline__ bool wait_warp(Ctl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    bool ok = mbar_try_wait(bar, parity);
    if (!ok && !aborted(ctl)) {
        ok = mbar_wait(bar, parity);
        if (!ok) set_abort(ctl, status);
    }
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool wait_peer(Ctl* ctl, uint64_t* bar, uint32_t parity, uint32_t* status) {
    bool ok = mbar_try_wait_cluster(bar, parity);
    if (!ok && !aborted(ctl)) {
        ok = mbar_wait_cluster(bar, parity);
        if (!ok) set_abort(ctl, status);
    }
    return __all_sync(0xffffffffu, ok);
}

// A warp's signal (lane 0) on a barrier that lives in CTA 0, the pair's MMA issuer. CTA 0's warps
// arrive (one of them, `arm` true, also registers the 4 bytes that each of CTA 1's `n_peer` warps
// sends); CTA 1's warps send 4 bytes with complete_tx. The send is asynchronous: the warp does not
// wait until its earlier writes are visible across the cluster, as a remote release arrive would
// (the complete_tx carries release semantics at cluster scope).
__device__ __forceinline__ void signal_leader(Ctl* ctl, uint64_t* bar, int crank, bool arm, uint32_t n_peer) {
    const uint32_t leader = cluster_ctarank() & ~1u;   // the pair's first CTA
    if (crank == 0) {
        if (arm)
            mbar_arrive_expect_tx(bar, 4u * n_peer);
        else
            mbar_arrive(bar);
    } else {
        st_async_b32(mapa_shared(smem_addr(&ctl->sig_sink), leader), 0u, mapa_shared(smem_addr(bar), leader));
    }
}

// V row of one key: the four blocks 4c + q (c = 4 half + cl) into V block cl, chunks 2q, 2q + 1.
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

// kBlkOrder: the 32 scale bytes are in block order (432-byte records, and the 352-byte record of
// the scale-layout comparison) instead of the permuted placement 8 (s & 3) + (s >> 2).
// The row's split merge, by every CTA of its cluster once every split's partial is written: the
// cluster's 2S CTAs x 26 warps take the 128 heads in turn (warp-sized work items), lane l dims
// 16l .. 16l + 15.
//   out = sum_s w_s part_s,  w_s = 2^{lse2_s} / (sum_s 2^{lse2_s} + e^{sink}),  lse = ln sum_s e^{lse_s}
// (lse2 = log2-domain partial lse; the sink is not part of lse). Every load of a head goes out before
// any is used.
constexpr int kMaxClusterSplits = 4;   // a cluster holds at most 8 CTAs

__device__ __forceinline__ void merge_splits(const KernelArgs& a, int row) {
    const int lane = threadIdx.x & 31;
    const int64_t rbase = static_cast<int64_t>(row) * a.splits;
    const int workers = 2 * a.splits * (kThreads / 32);
    const int me = static_cast<int>(cluster_ctarank()) * (kThreads / 32) + (threadIdx.x >> 5);
#pragma unroll 1
    for (int head = me; head < 128; head += workers) {
        float v[kMaxClusterSplits];
        uint4 d0[kMaxClusterSplits], d1[kMaxClusterSplits];
        const float sk = a.sink != nullptr ? __ldg(a.sink + head) : 0.0f;
#pragma unroll
        for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
            v[sp] = -INFINITY;
            d0[sp] = d1[sp] = make_uint4(0u, 0u, 0u, 0u);
            if (sp < a.splits) {
                v[sp] = __ldcg(a.part_lse + (rbase + sp) * 128 + head);
                const uint4* src = reinterpret_cast<const uint4*>(a.part_out + ((rbase + sp) * 128 + head) * 512 + 16 * lane);
                d0[sp] = __ldcg(src);
                d1[sp] = __ldcg(src + 1);
            }
        }
        float m = v[0];
#pragma unroll
        for (int sp = 1; sp < kMaxClusterSplits; ++sp) m = fmaxf(m, v[sp]);
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
        float total = -INFINITY;
        if (m != -INFINITY) {
            float ex[kMaxClusterSplits];
            float sum = 0.0f;
#pragma unroll
            for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
                ex[sp] = exp2f(v[sp] - m);
                sum += ex[sp];
            }
            total = (m + log2f(sum)) * kLn2;
            const float inv = 1.0f / (sum + (a.sink != nullptr ? exp2f(sk * kLog2e - m) : 0.0f));
#pragma unroll
            for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
                const float w = ex[sp] * inv;
                const uint32_t hw[8] = {d0[sp].x, d0[sp].y, d0[sp].z, d0[sp].w, d1[sp].x, d1[sp].y, d1[sp].z, d1[sp].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[e]));
                    acc[2 * e] += w * f.x;
                    acc[2 * e + 1] += w * f.y;
                }
            }
        }
        uint4* dst = reinterpret_cast<uint4*>(a.out + (static_cast<int64_t>(row) * 128 + head) * 512 + 16 * lane);
        dst[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                            pack_bf16x2(acc[6], acc[7]));
        dst[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]), pack_bf16x2(acc[12], acc[13]),
                            pack_bf16x2(acc[14], acc[15]));
        if (lane == 0) a.lse[static_cast<int64_t>(row) * 128 + head] = total;
    }
}

// Launched in clusters of two CTAs per split pair (one pair, or all splits of a row when they merge
// in the kernel).
template <int R, bool kBlkOrder>
__global__ void __launch_bounds__(kThreads, 1)
    decode_pair_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    Ctl* ctl = reinterpret_cast<Ctl*>(smem);
    const uint32_t sbase = smem_addr(smem);

    const int crank = static_cast<int>(cluster_ctarank() & 1u);   // CTA within the pair
    const int pb = static_cast<int>(cluster_ctarank() & ~1u);     // the pair's first rank in the cluster
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
        mbar_init(&ctl->khalf, 1);
        mbar_init(&ctl->qkdone, 1);
        mbar_init(&ctl->pvhalf, 1);
        mbar_init(&ctl->pvdone, 1);
        // CTA 0's own warps arrive on these; CTA 1's warps send 4 bytes each (complete_tx), which
        // one arriving warp of CTA 0 registers with expect_tx
        mbar_init(&ctl->kfull_a, 8);
        mbar_init(&ctl->kfull_b, 8);
        mbar_init(&ctl->vfull_a, 8);
        mbar_init(&ctl->vfull_b, 8);
        mbar_init(&ctl->sfree, 8);
        mbar_init(&ctl->pfull_a, 8);
        mbar_init(&ctl->pfull_b, 4);
        mbar_init(&ctl->qready, 16);
        mbar_init(&ctl->qstaged, 16);
        mbar_init(&ctl->qload, 1);
        mbar_init(&ctl->drain, 2);
        ctl->abort = 0u;
        fence_barrier_init();
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

    // ---- q: the softmax warps (0-7) and the V converters (16-23), idle until the first V tile,
    // stage q: largest magnitude per head, the power-of-two prescale, f16 (or bf16 RoPE) copies in
    // tensor memory (dims 0-383, both lane halves) and shared memory (dims 384-575).
    const bool qwarp = warp < 8 || (warp >= kWarpV && warp < kWarpQK);
    float ch = 0.0f;   // sm_scale log2(e) 2^-pre of this thread's head (softmax warps)
    if (qwarp) {
        const int qd = warp & 3;                                      // TMEM lane quadrant
        const int g = (warp >= kWarpV ? 2 : 0) + ((warp >> 2) & 1);   // 0..3: warp of the quadrant
        const int L = 32 * qd + lane;
        const int hl = L & 63;
        const int slot = ((qd >> 1) << 2) | g;                        // 0..7 among the head's threads
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        float* xmax = reinterpret_cast<float*>(smem + kOffXmax);
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&ctl->qload, 9u * kBlk);
            for (int bx = 0; bx < 9; ++bx)
                tma_load_2d(sbase + kOffV + bx * kBlk, &a.qmap, 64 * bx, row * 128 + 64 * crank, &ctl->qload);
        }
        const bool okq = wait_warp(ctl, &ctl->qload, 0, a.status);
        const uint32_t stage = sbase + kOffV;   // box b (dims 64b..): head hl chunk c at b*8192 + swz(hl, c)
        float qmax = 0.0f;
        if (okq) {
#pragma unroll 3
            for (int k = 9 * slot; k < 9 * slot + 9; ++k) {   // 72 chunks of 8 dims per head, 9 per thread
                const uint4 x = lds_u128(stage + (k >> 3) * kBlk + swz(hl, k & 7));
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    qmax = fmax3(qmax, fabsf(__uint_as_float(w[m] << 16)), fabsf(__uint_as_float(w[m] & 0xFFFF0000u)));
            }
        }
        xmax[slot * 64 + hl] = qmax;
        named_bar_sync(2, 512);
#pragma unroll
        for (int k = 0; k < 8; ++k) qmax = fmaxf(qmax, xmax[k * 64 + hl]);
        int pre = 0;
        if (qmax > 0.0f) {
            int e;
            frexpf(qmax, &e);   // qmax < 2^e <= 2 qmax
            pre = min(100, max(-100, 15 - e));
        }
        const float fpre = __int_as_float((127 + pre) << 23);
        ch = a.sm_scale * kLog2e * __int_as_float((127 - pre) << 23);   // S' = 2^pre S, z = ch S'
        auto cvt_pair = [&](uint32_t w, bool bf) -> uint32_t {
            const float lo = __uint_as_float(w << 16) * fpre, hi = __uint_as_float(w & 0xFFFF0000u) * fpre;
            return bf ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
        };
        if (okq) {
            // dims [0, 384) = 48 chunks into TMEM columns kColQ + 4 chunk: 12 chunks per warp of the quadrant
            uint32_t v[16];
#pragma unroll
            for (int half = 0; half < 3; ++half) {   // 3 x 4 chunks = 12 chunks = 48 columns
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int k = 12 * g + 4 * half + cc;
                    const uint4 x = lds_u128(stage + (k >> 3) * kBlk + swz(hl, k & 7));
                    v[4 * cc + 0] = cvt_pair(x.x, false);
                    v[4 * cc + 1] = cvt_pair(x.y, false);
                    v[4 * cc + 2] = cvt_pair(x.z, false);
                    v[4 * cc + 3] = cvt_pair(x.w, false);
                }
                tmem_st16(lane_base + kColQ + 48 * g + 16 * half, v);
            }
            // dims [384, 576) = chunks 48..71 into shared memory (one copy, lanes 0-63): 6 chunks per warp
            if (qd < 2) {
#pragma unroll 2
                for (int cc = 0; cc < 6; ++cc) {
                    const int k = 48 + 6 * g + cc;
                    const bool bf = R == 432 && k >= 64;   // bf16 RoPE of 432-byte records
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
            signal_leader(ctl, &ctl->qready, crank, warp == 0, 16);
        }
    }

    if (warp < 8) {
        // ======================= softmax warps =======================
        const int qd = warp & 3;               // TMEM lane quadrant
        const int h2 = warp >> 2;              // score column half
        const int L = 32 * qd + lane;          // TMEM lane
        const int hl = L & 63;                 // head within the CTA
        const int qi = ((qd >> 1) << 1) | h2;  // this thread's slot among the head's four
        const bool upper = qd >= 2;            // lanes 64-127: keys 64-127 of a tile, dims 256-511 of O
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        float* xmax = reinterpret_cast<float*>(smem + kOffXmax);
        float* xl = reinterpret_cast<float*>(smem + kOffXl);
        bool ok = !aborted(ctl);
        float m_ref = -INFINITY;   // reference max (log2 units), the same in the head's four threads
        float l = 0.0f;            // this thread's sum of 2^(z - m_ref)
        const bool pos_scale = a.sm_scale > 0.0f;
        const uint32_t p_row = sbase + kOffP + (upper ? kBlk : 0);
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
                if (lane == 0) signal_leader(ctl, &ctl->sfree, crank, warp == 0, 8);
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
                // the tile maxima are read before anyone writes the next ones
                named_bar_sync(1, 256);
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
            // ---- P columns of this warp's keys once PV of the previous tile released them. Lanes
            // 64-127 report their O rescale done on pfull_a first (the first PV half writes O too).
            if (upper) {
                // (after the first half of the previous PV, so that this arrival cannot reach CTA 0's
                // barrier while it still counts the previous tile)
                if (i > 0) ok = wait_warp(ctl, &ctl->pvhalf, (i - 1) & 1, a.status);
                if (!ok) continue;
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) signal_leader(ctl, &ctl->pfull_a, crank, false, 8);
            }
            if (i > 0) ok = wait_warp(ctl, upper ? &ctl->pvdone : &ctl->pvhalf, (i - 1) & 1, a.status);
            if (!ok) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                sts_u128(p_row + swz(hl, 4 * h2 + c), make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]));
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) signal_leader(ctl, upper ? &ctl->pfull_b : &ctl->pfull_a, crank, warp == 0 || warp == 2, upper ? 4 : 8);
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
        const int dbase = (upper ? 256 : 0) + 128 * h2;
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
    } else if (warp < kWarpQK) {
        // ============ converters: warps 8-15 K rows of the own keys, warps 16-23 V rows of all keys ============
        // Each thread stages the bytes it converts itself with cp.async one tile ahead (commit groups in
        // issue order: part a of tile k, part b of tile k, part a of tile k + 1, ...), so a wait for the
        // older part leaves the newer one in flight and no arrive of the thread waits for a load.
        const bool vrole = warp >= kWarpV;
        const int t = threadIdx.x - 32 * (vrole ? kWarpV : kWarpK);
        const int j = t >> 2;    // key of the half tile (K: own key j; V: key 64 hv + j)
        const int q = t & 3;     // quarter: blocks 4c + q, RoPE dims 16q..
        const uint32_t fnan = 0x7E007E00u;   // f16 quiet-NaN pairs: a masked key's K row
        constexpr int sb = R == 352 ? 320 : 256;                 // scale bytes of a record
        auto index_at = [&](int i, int key) -> int32_t {        // key 0..127 of tile i
            if (i >= n_tiles) return -1;
            const int pos = key_begin + kTile * i + key;
            return pos < key_end ? __ldg(idx_row + pos) : -1;
        };
        auto in_range = [&](int32_t v) { return v >= 0 && static_cast<int64_t>(v) < a.num_slots; };
        bool ok = !aborted(ctl);
        if (!vrole) {
            const uint32_t st_a = sbase + kOffStA + j * kStrA;
            const uint32_t st_b = sbase + kOffStB + j * kStrB<R>;
            const uint32_t k_s = sbase + kOffK;
            auto stage_a = [&](int32_t v) {   // codes of blocks 0-15 (bytes 0-127) and the 32 scale bytes
                if (in_range(v)) {
                    const uint8_t* rec = a.cache + static_cast<int64_t>(v) * R;
                    cp_async16(st_a + 16 * q, rec + 16 * q);
                    cp_async16(st_a + 16 * (q + 4), rec + 16 * (q + 4));
                    if (q < 2) cp_async16(st_a + 128 + 16 * q, rec + sb + 16 * q);
                }
                cp_async_commit();
            };
            auto stage_b = [&](int32_t v) {   // codes of blocks 16-31 (bytes 128-255) and the RoPE bytes
                if (in_range(v)) {
                    const uint8_t* rec = a.cache + static_cast<int64_t>(v) * R;
                    cp_async16(st_b + 16 * q, rec + 128 + 16 * q);
                    cp_async16(st_b + 16 * (q + 4), rec + 128 + 16 * (q + 4));
                    cp_async16(st_b + 128 + 16 * q, rec + (R == 352 ? 256 : 304) + 16 * q);
                    if constexpr (R == 432) cp_async16(st_b + 192 + 16 * q, rec + 304 + 64 + 16 * q);
                }
                cp_async_commit();
            };
            // the split's index list into L2 (32 indices a line), so that the index loads two tiles
            // ahead hit L2
            if (32 * t < key_end - key_begin) prefetch_l2(idx_row + key_begin + 32 * t);
            const int own = kOwn * crank + j;
            int32_t idx0 = index_at(0, own), idx1 = index_at(1, own);
            stage_a(idx0);
            stage_b(idx0);
            int32_t idx2 = index_at(2, own);
            for (int k = 0; k < n_tiles; ++k) {
                const bool valid = in_range(idx0);
                if (q == 0 && idx0 >= 0 && !valid && a.status != nullptr) atomicOr(a.status, 0x2u);
                // ---- blocks 0-3 (dims 0-255) once the previous QK's first half has read them
                cp_async_wait<1>();
                __syncwarp();
                if (k >= 1) ok = wait_warp(ctl, &ctl->khalf, (k - 1) & 1, a.status);
                if (!ok) break;
                uint32_t sc_lo, sc_hi;   // byte c: scale of block 4c + q (c = 0..3, 4..7)
                if constexpr (R == 352 && !kBlkOrder) {
                    const uint2 s8 = lds_u64(st_a + 128 + 8 * q);   // permuted placement
                    sc_lo = s8.x;
                    sc_hi = s8.y;
                } else {
                    const uint4 w0 = lds_u128(st_a + 128), w1 = lds_u128(st_a + 144);   // block order
                    sc_lo = gather_byte4(w0, q);
                    sc_hi = gather_byte4(w1, q);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint2 cw = lds_u64(st_a + 32 * c + 8 * q);
                    const __half2 s2 = scale_half2((sc_lo >> (8 * c)) & 0xFFu);
                    const uint4 lo = valid ? dq8(cw.x, s2) : make_uint4(fnan, fnan, fnan, fnan);
                    const uint4 hi = valid ? dq8(cw.y, s2) : make_uint4(fnan, fnan, fnan, fnan);
                    sts_u128(k_s + c * kBlk + swz(j, 2 * q), lo);
                    sts_u128(k_s + c * kBlk + swz(j, 2 * q + 1), hi);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) signal_leader(ctl, &ctl->kfull_a, crank, t == 0, 8);
                stage_a(idx1);   // the key's four threads have read part a of tile k (the warp synced)
                // ---- blocks 4-8 (dims 256-575) once the previous QK has finished
                cp_async_wait<1>();
                __syncwarp();
                if (k >= 1) ok = wait_warp(ctl, &ctl->qkdone, (k - 1) & 1, a.status);
                if (!ok) break;
#pragma unroll
                for (int c = 4; c < 8; ++c) {
                    const uint2 cw = lds_u64(st_b + 32 * (c - 4) + 8 * q);
                    const __half2 s2 = scale_half2((sc_hi >> (8 * (c - 4))) & 0xFFu);
                    const uint4 lo = valid ? dq8(cw.x, s2) : make_uint4(fnan, fnan, fnan, fnan);
                    const uint4 hi = valid ? dq8(cw.y, s2) : make_uint4(fnan, fnan, fnan, fnan);
                    sts_u128(k_s + c * kBlk + swz(j, 2 * q), lo);
                    sts_u128(k_s + c * kBlk + swz(j, 2 * q + 1), hi);
                }
                if (valid) {
                    if constexpr (R == 352) {
                        const uint4 e = lds_u128(st_b + 128 + 16 * q);
                        const uint2 e0 = e4m3x4_to_f16(e.x), e1 = e4m3x4_to_f16(e.y);
                        const uint2 e2 = e4m3x4_to_f16(e.z), e3 = e4m3x4_to_f16(e.w);
                        sts_u128(k_s + 8 * kBlk + swz(j, 2 * q), make_uint4(e0.x, e0.y, e1.x, e1.y));
                        sts_u128(k_s + 8 * kBlk + swz(j, 2 * q + 1), make_uint4(e2.x, e2.y, e3.x, e3.y));
                    } else {
                        sts_u128(k_s + 8 * kBlk + swz(j, 2 * q), lds_u128(st_b + 128 + 32 * q));
                        sts_u128(k_s + 8 * kBlk + swz(j, 2 * q + 1), lds_u128(st_b + 128 + 32 * q + 16));
                    }
                } else {
                    const uint32_t fr = R == 352 ? fnan : 0x7FC07FC0u;   // RoPE block: f16 / bf16 quiet NaN
                    sts_u128(k_s + 8 * kBlk + swz(j, 2 * q), make_uint4(fr, fr, fr, fr));
                    sts_u128(k_s + 8 * kBlk + swz(j, 2 * q + 1), make_uint4(fr, fr, fr, fr));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) signal_leader(ctl, &ctl->kfull_b, crank, t == 0, 8);
                stage_b(idx1);
                idx0 = idx1;
                idx1 = idx2;
                idx2 = index_at(k + 3, own);   // in flight until the next tile's first arrive
            }
        } else {
            const uint32_t v_s = sbase + kOffV;
            auto stage_v = [&](int hv, int32_t v) {   // this CTA's half of the codes and its 16 scale bytes
                const uint32_t st = sbase + kOffStV<R> + (hv * kOwn + j) * kStrV<R>;
                if (in_range(v)) {
                    const uint8_t* rec = a.cache + static_cast<int64_t>(v) * R;
                    cp_async16(st + 16 * q, rec + 128 * crank + 16 * q);
                    cp_async16(st + 16 * (q + 4), rec + 128 * crank + 16 * (q + 4));
                    if constexpr (R == 352 && !kBlkOrder)
                        cp_async4(st + 128 + 4 * q, rec + 320 + 8 * q + 4 * crank);   // blocks 4c + q, c in half
                    else if (q == 0)
                        cp_async16(st + 128, rec + sb + 16 * crank);   // blocks 16 crank ..
                }
                cp_async_commit();
            };
            int32_t ia0 = index_at(0, j), ib0 = index_at(0, kOwn + j);
            int32_t ia1 = index_at(1, j), ib1 = index_at(1, kOwn + j);
            stage_v(0, ia0);
            stage_v(1, ib0);
            int32_t ia2 = index_at(2, j), ib2 = index_at(2, kOwn + j);
            for (int k = 0; k < n_tiles; ++k) {
#pragma unroll
                for (int hv = 0; hv < 2; ++hv) {   // V rows 64 hv + j: CTA hv's keys
                    cp_async_wait<1>();
                    __syncwarp();
                    if (k == 0 && hv == 0) ok = wait_warp(ctl, &ctl->qstaged, 0, a.status);   // the V buffer held q
                    if (ok && k >= 1) ok = wait_warp(ctl, hv == 0 ? &ctl->pvhalf : &ctl->pvdone, (k - 1) & 1, a.status);
                    if (!ok) break;
                    const uint32_t st = sbase + kOffStV<R> + (hv * kOwn + j) * kStrV<R>;
                    const bool valid = in_range(hv == 0 ? ia0 : ib0);
                    uint32_t sbytes;   // byte cl: scale of block 4 (4 crank + cl) + q
                    if constexpr (R == 352 && !kBlkOrder)
                        sbytes = lds_u32(st + 128 + 4 * q);
                    else
                        sbytes = gather_byte4(lds_u128(st + 128), q);
                    const uint2 c0 = lds_u64(st + 8 * q), c1 = lds_u64(st + 32 + 8 * q);
                    const uint2 c2 = lds_u64(st + 64 + 8 * q), c3 = lds_u64(st + 96 + 8 * q);
                    // a masked key's V row is zero (its probability is zero, and 0 x 0 stays 0)
                    write_v(v_s, 64 * hv + j, q,
                            valid ? make_uint4(c0.x, c0.y, c1.x, c1.y) : make_uint4(0u, 0u, 0u, 0u),
                            valid ? make_uint4(c2.x, c2.y, c3.x, c3.y) : make_uint4(0u, 0u, 0u, 0u),
                            valid ? sbytes : 0u);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) signal_leader(ctl, hv == 0 ? &ctl->vfull_a : &ctl->vfull_b, crank, t == 0, 8);
                    stage_v(hv, hv == 0 ? ia1 : ib1);
                }
                if (!ok) break;
                ia0 = ia1;
                ib0 = ib1;
                ia1 = ia2;
                ib1 = ib2;
                ia2 = index_at(k + 3, j);
                ib2 = index_at(k + 3, kOwn + j);
            }
        }
        cp_async_wait<0>();   // no copy into shared memory outlives the loop
    } else if (warp == kWarpQK) {
        // ======================= QK issuer (CTA 0) =======================
        if (crank == 0) {
            const uint32_t idesc_f16 = idesc_f16_f32(128, kTile, false, false);
            const uint32_t idesc_rope = R == 432 ? idesc_bf16_f32(128, kTile, false, false) : idesc_f16;
            const uint64_t kdesc0 = sdesc_sw128(sbase + kOffK, 16, 1024);
            const uint64_t qdesc0 = sdesc_sw128(sbase + kOffQs, 16, 1024);
            const bool leader = elect_one_in_warp();
            bool ok = wait_peer(ctl, &ctl->qready, 0, a.status);
            for (int i = 0; i < n_tiles && ok; ++i) {
                ok = wait_peer(ctl, &ctl->kfull_a, i & 1, a.status);
                if (ok && i >= 1) ok = wait_peer(ctl, &ctl->sfree, (i - 1) & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t d = tmem + kColS;
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)   // dims 0-255: q from tensor memory
                        mma_ts_cg2(d, tmem + kColQ + 8 * kk,
                                   kdesc0 + static_cast<uint64_t>(((kk >> 2) * kBlk + (kk & 3) * 32) >> 4), idesc_f16,
                                   kk > 0 ? 1u : 0u);
                    mma_commit_cg2(&ctl->khalf, 0x3u << pb);
                }
                __syncwarp();
                ok = wait_peer(ctl, &ctl->kfull_b, i & 1, a.status);
                if (!ok) break;
                tc_fence_after_sync();
                if (leader) {
#pragma unroll
                    for (int kk = 16; kk < 36; ++kk) {
                        const uint64_t kd = kdesc0 + static_cast<uint64_t>(((kk >> 2) * kBlk + (kk & 3) * 32) >> 4);
                        if (kk < kQTmemSteps)
                            mma_ts_cg2(d, tmem + kColQ + 8 * kk, kd, idesc_f16, 1u);
                        else
                            mma_ss_cg2(d, qdesc0 + static_cast<uint64_t>((((kk - 24) >> 2) * kBlk + (kk & 3) * 32) >> 4),
                                       kd, kk >= 32 ? idesc_rope : idesc_f16, 1u);
                    }
                    mma_commit_cg2(&ctl->qkdone, 0x3u << pb);
                }
                __syncwarp();
            }
            if (leader) mma_commit_cg2(&ctl->drain, 0x1u << pb);
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
#pragma unroll
                for (int hv = 0; hv < 2; ++hv) {   // keys 0-63, then keys 64-127
                    ok = wait_peer(ctl, hv == 0 ? &ctl->vfull_a : &ctl->vfull_b, i & 1, a.status);
                    if (ok) ok = wait_peer(ctl, hv == 0 ? &ctl->pfull_a : &ctl->pfull_b, i & 1, a.status);
                    if (!ok) break;
                    tc_fence_after_sync();
                    if (leader) {
#pragma unroll
                        for (int ks = 4 * hv; ks < 4 * hv + 4; ++ks) {
                            const uint64_t pd = pdesc0 + static_cast<uint64_t>(((ks >> 2) * kBlk + (ks & 3) * 32) >> 4);
#pragma unroll
                            for (int jj = 0; jj < 2; ++jj)
                                mma_ss_cg2(tmem + kColO + 128 * jj, pd,
                                           vdesc0 + static_cast<uint64_t>((2 * jj * kVBlk + ks * 2048) >> 4), idesc_pv,
                                           (i > 0 || ks > 0) ? 1u : 0u);
                        }
                        mma_commit_cg2(hv == 0 ? &ctl->pvhalf : &ctl->pvdone, 0x3u << pb);
                    }
                    __syncwarp();
                }
            }
            if (leader) mma_commit_cg2(&ctl->drain, 0x1u << pb);
            __syncwarp();
        }
    }

    // CTA 0 waits (bounded) until every MMA it issued has completed before anyone leaves
    if (crank == 0 && (warp == kWarpQK || warp == kWarpPV)) {
        if (!mbar_wait(&ctl->drain, 0)) set_abort(ctl, a.status);
    }
    tc_fence_before_sync();
    // No CTA leaves while its peer may still write its shared or tensor memory; with a merge, every
    // split's partial is also written (release / acquire at cluster scope) once this returns.
    cluster_sync();
    if (warp == kWarpQK) {
        tc_fence_after_sync();
        tmem_dealloc_cg2(tmem, kTmemCols);
    }
    if (a.merge) merge_splits(a, row);
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
    err = cudaFuncSetAttribute(decode_pair_kernel<R, kBlkOrder>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc<R>);
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

// How many clusters of 2 * splits CTAs of this kernel variant fit on the current device at once
// (0: none), asked once per variant, split count and device.
int pair_clusters_fit(int record_bytes, bool block_scales, int splits) {
    using namespace pairdec;
    if (splits < 1 || splits > kMaxClusterSplits) return 0;
    static std::atomic<int> fits[3][kMaxClusterSplits + 1][8];   // 0 unknown, else 1 + clusters
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const int variant = record_bytes == 432 ? 2 : block_scales ? 1 : 0;
    std::atomic<int>& known = fits[variant][splits][dev & 7];
    int state = known.load(std::memory_order_relaxed);
    if (state == 0) {
        const auto kernel = record_bytes == 432 ? decode_pair_kernel<432, false>
                            : block_scales      ? decode_pair_kernel<352, true>
                                                : decode_pair_kernel<352, false>;
        const cudaError_t err = record_bytes == 432 ? prepare_kernel<432, false>()
                                : block_scales      ? prepare_kernel<352, true>()
                                                    : prepare_kernel<352, false>();
        int clusters = 0;
        if (err == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2u * static_cast<unsigned>(splits));
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = record_bytes == 432 ? kSmemAlloc<432> : kSmemAlloc<352>;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2u * static_cast<unsigned>(splits);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) clusters = 0;
        }
        (void)cudaGetLastError();
        state = 1 + (clusters > 0 ? clusters : 0);
        known.store(state, std::memory_order_relaxed);
    }
    return state - 1;
}

// All splits of a row in one cluster when there are 2-4 of them and such clusters fit on this
// GPU all at once (a second wave of large clusters would leave SMs idle): the kernel then merges
// them itself and no merge grid follows.
bool decode_pair_merges(const DecodeArgs& d) {
    if (!decode_pair_supported(d) || d.splits < 2 || d.splits > pairdec::kMaxClusterSplits) return false;
    return static_cast<int64_t>(pair_clusters_fit(d.record_bytes, d.block_scales, d.splits)) >= d.rows;
}

cudaError_t launch_decode_pair(const DecodeArgs& d, cudaStream_t stream, bool* merged) {
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
    cfg.dynamicSmemBytes = d.record_bytes == 432 ? kSmemAlloc<432> : kSmemAlloc<352>;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddepcontrol.wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // All splits of a row in one cluster when there are 2-4 of them and such clusters fit on this
    // GPU: the kernel then merges them itself and no merge grid follows.
    a.merge = decode_pair_merges(d) ? 1 : 0;
    attr[1].val.clusterDim.x = a.merge ? 2u * static_cast<unsigned>(d.splits) : 2u;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    *merged = a.merge != 0;
    err = cudaLaunchKernelEx(&cfg, kernel, a);
    if (err == cudaSuccess) err = cudaGetLastError();
    return err;
}

}  // namespace nvfp4mla
