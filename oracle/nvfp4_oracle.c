/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the NVFP4 MLA KV-cache codec and the sparse
 * MLA decode that reads it.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, the smoke check in __graft_entry__.py and the CPU
 * baseline leg of bench.py load this file's library. It shares no code, header, table or
 * constant with the CUDA library, and the CUDA library never calls it.
 *
 * Every floating-point step runs in fp64, except where the pages fix a narrower precision
 * (the fp32 quotients that feed the e4m3/e2m1 rounding, and the bf16 inputs themselves).
 *
 * Sources (web pages; cited by title and section):
 *  [FlashMLA-18] "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode" (FlashMLA pull
 *                request 18): the "nvfp4.fp8rope (352 B/token)" layout and its scale
 *                permutation, the "RoPE part carries no block scale" paragraph, and the
 *                "Kernel:" paragraph (dequantize e2m1/e4m3 -> bf16; bf16 MMAs, fp32 accumulate).
 *  [vLLM-82]     "kv: nvfp4_ds_mla - 4-bit NVFP4 KV cache for B12X sparse MLA (SM120)"
 *                (vLLM fork pull request 82): "Problem" (the 432-B record field list),
 *                "Fix / Write side" (E2M1 data + per-16-group E4M3 scales, implicit global
 *                scale 1.0, zeroed pad, verbatim 16-bit RoPE) and "Tests" (scale =
 *                E4M3(group_amax/6), the E2M1 nibble table); the same "Problem" section
 *                gives the 656-B fp8_ds_mla record (512 B fp8 NoPE + 16 B fp32 tile scales +
 *                128 B bf16 RoPE) that the NVFP4 records are measured against.
 *
 * Readings of points the pages leave open:
 *  - e4m3 is the "fn" variant: no infinities, 0x7F/0xFF are NaN, largest finite 448.
 *  - Rounding is round-to-nearest, ties to the code whose least significant bit is 0,
 *    saturating to the largest finite magnitude; the sign of the input is kept, so a
 *    negative input that rounds to zero gives the negative-zero code.
 *  - amax/6 and x/s are IEEE fp32 divisions; s is the decoded stored scale.
 *  - A group whose stored scale decodes to 0 stores magnitude-0 nibbles carrying the sign
 *    of each input.
 *  - The even element of a pair sits in the low nibble of its byte.
 *  - 432-B record: NoPE at 0, scales in group order at 256, 16 zero bytes at 288, bf16 RoPE
 *    (little-endian) at 304.
 *  - 656-B record: the fields in the order the page lists them: 512 e4m3 NoPE codes at 0, four
 *    little-endian fp32 scales at 512 (scale t covers NoPE values [128t, 128t+128)), 64 bf16
 *    RoPE values (little-endian) at 528. No page states the fp8 scale rule; the one used is
 *    the plain analogue of the NVFP4 rule: scale = amax / 448 (IEEE fp32 division, 448 = the
 *    largest e4m3 magnitude) and code = e4m3(x / scale) (fp32 quotient); a tile whose amax is 0
 *    stores scale 0 and zero codes carrying the input signs. Its dequantized key is rounded to
 *    bf16 ("the kernel dequantizes to bf16", [FlashMLA-18]): K = bf16(e4m3(code) * scale),
 *    one round-to-nearest-even of the exact product.
 *  - Decode: an index i is used iff 0 <= i < num_slots; repeated indices count as often as
 *    they appear. The log-sum-exp is natural-log, over the scaled logits of the used
 *    tokens only; an attention sink adds exp(sink - m) to the softmax denominator of `out`
 *    and nothing to `lse`. A row with no used index gives out = 0 and lse = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The e2m1 grid ("E2M1 nibble table", [vLLM-82] Tests): magnitudes of codes 0..7. */
static const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static float bf16_bits_to_float(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

double oracle_bf16_to_double(uint16_t bits) { return (double)bf16_bits_to_float(bits); }

/* Round a finite double to the nearest bf16 value (8 significant bits, the fp32 exponent
 * range, subnormals in steps of 2^-133), ties to even; beyond the largest bf16 value it
 * overflows to infinity. Used for the fp8 record's keys. */
double oracle_round_to_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    (void)frexp(x, &e);                         /* |x| = m * 2^e, m in [0.5, 1) */
    int lsb = e - 8;                            /* weight of the last kept bit */
    if (lsb < -133) lsb = -133;                 /* bf16 subnormal spacing */
    double q = ldexp(x, -lsb);                  /* exact: a power-of-two scaling */
    double r = ldexp(nearbyint(q), lsb);        /* default rounding mode: ties to even */
    /* past the largest bf16 value (just below 2^128) the nearest is infinity */
    return fabs(r) >= ldexp(1.0, 128) ? copysign(INFINITY, x) : r;
}

/* e4m3 (fn) decode by its bit fields: sign, 4 exponent bits (bias 7), 3 mantissa bits. */
double oracle_e4m3_decode(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9)          /* subnormal: m/8 * 2^-6 */
                          : ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7)   */
    return sign ? -mag : mag;
}

double oracle_e2m1_decode(uint8_t nibble) {
    double mag = kE2M1Magnitude[nibble & 7];
    return (nibble & 8) ? -mag : mag;
}

/* Nearest finite e4m3 code to a finite float, found by trying all 127 non-negative finite
 * codes; ties go to the even code; anything above 448 becomes 448; the sign is copied. */
uint8_t oracle_e4m3_encode(float f) {
    double a = fabs((double)f);
    /* at or above the largest finite magnitude the nearest finite code is that magnitude
     * (checked first: for huge inputs every distance rounds to the same double) */
    if (a >= 448.0) return (uint8_t)((signbit(f) ? 0x80 : 0x00) | 0x7E);
    int best = 0;
    double best_dist = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double dist = fabs(oracle_e4m3_decode((uint8_t)c) - a);
        if (dist < best_dist || (dist == best_dist && (c & 1) == 0)) {
            best = c;
            best_dist = dist;
        }
    }
    return (uint8_t)((signbit(f) ? 0x80 : 0x00) | best);
}

/* Nearest e2m1 code to a finite float, by trying the 8 magnitudes; same tie, saturation
 * and sign rules as oracle_e4m3_encode. */
uint8_t oracle_e2m1_encode(float f) {
    double a = fabs((double)f);
    if (a >= 6.0) return (uint8_t)((signbit(f) ? 0x8 : 0x0) | 7);
    int best = 0;
    double best_dist = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double dist = fabs(kE2M1Magnitude[c] - a);
        if (dist < best_dist || (dist == best_dist && (c & 1) == 0)) {
            best = c;
            best_dist = dist;
        }
    }
    return (uint8_t)((signbit(f) ? 0x8 : 0x0) | best);
}

/* Byte offset of the e4m3 scale of 16-element block g inside a record.
 * 352 B ([FlashMLA-18] layout): block s is stored at 320 + 8*(s & 3) + (s >> 2).
 * 352 B with block_order != 0: the same 32-byte field holds the scales in block order (block s
 *   at 320 + s). No page defines this record; it is the unpermuted side of the scale-layout
 *   comparison that [FlashMLA-18] (layout) credits with 10-12% of decode latency.
 * 432 B ([vLLM-82] Problem): 32 scale bytes in block order after the 256 NoPE bytes
 *   (block_order is ignored). */
int oracle_scale_offset(int record_bytes, int block_order, int g) {
    if (record_bytes == 352) return block_order ? 320 + g : 320 + 8 * (g & 3) + (g >> 2);
    return 256 + g;
}

/* Quantize one token: 512 bf16 NoPE values and 64 bf16 RoPE values -> one record. */
/* The 656-B fp8 record: per 128-value tile t, scale = amax / 448 and code = e4m3(x / scale). */
static void quantize_record_fp8(const uint16_t* latent, const uint16_t* rope, uint8_t* rec) {
    for (int t = 0; t < 4; ++t) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float a = fabsf(bf16_bits_to_float(latent[128 * t + i]));
            if (a > amax) amax = a;
        }
        volatile float scale = amax / 448.0f;
        float s = scale;
        memcpy(rec + 512 + 4 * t, &s, 4);       /* little-endian fp32 on every host this runs on */
        for (int i = 0; i < 128; ++i) {
            float x = bf16_bits_to_float(latent[128 * t + i]);
            if (s == 0.0f) {
                rec[128 * t + i] = signbit(x) ? 0x80 : 0x00;
            } else {
                volatile float v = x / s;
                rec[128 * t + i] = oracle_e4m3_encode(v);
            }
        }
    }
    for (int j = 0; j < 64; ++j) {
        rec[528 + 2 * j] = (uint8_t)(rope[j] & 0xFF);
        rec[529 + 2 * j] = (uint8_t)(rope[j] >> 8);
    }
}

void oracle_quantize_record(const uint16_t* latent, const uint16_t* rope, int record_bytes,
                            int block_order, uint8_t* rec) {
    if (record_bytes == 656) {
        quantize_record_fp8(latent, rope, rec);
        return;
    }
    uint8_t nib[512];
    for (int g = 0; g < 32; ++g) {
        /* scale = E4M3(group_amax / 6)  ([vLLM-82] Tests) */
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(bf16_bits_to_float(latent[16 * g + i]));
            if (a > amax) amax = a;
        }
        volatile float quotient = amax / 6.0f;
        uint8_t sbyte = oracle_e4m3_encode(quotient);
        float s = (float)oracle_e4m3_decode(sbyte);
        rec[oracle_scale_offset(record_bytes, block_order, g)] = sbyte;
        /* values round-to-nearest-even onto the e2m1 grid after division by the scale */
        for (int i = 0; i < 16; ++i) {
            float x = bf16_bits_to_float(latent[16 * g + i]);
            if (s == 0.0f) {
                nib[16 * g + i] = signbit(x) ? 0x8 : 0x0;
            } else {
                volatile float v = x / s;
                nib[16 * g + i] = oracle_e2m1_encode(v);
            }
        }
    }
    /* [0,256): 512 e2m1 values, two per byte, even element in the low nibble */
    for (int i = 0; i < 256; ++i) rec[i] = (uint8_t)(nib[2 * i] | (nib[2 * i + 1] << 4));
    if (record_bytes == 352) {
        /* [256,320): 64 RoPE values as unscaled e4m3 ([FlashMLA-18] layout) */
        for (int j = 0; j < 64; ++j) rec[256 + j] = oracle_e4m3_encode(bf16_bits_to_float(rope[j]));
    } else {
        /* [288,304) zero pad, [304,432) RoPE copied verbatim as 16-bit ([vLLM-82] Write side) */
        for (int i = 288; i < 304; ++i) rec[i] = 0;
        for (int j = 0; j < 64; ++j) {
            rec[304 + 2 * j] = (uint8_t)(rope[j] & 0xFF);
            rec[305 + 2 * j] = (uint8_t)(rope[j] >> 8);
        }
    }
}

/* Write T records into cache[slot * record_bytes]; a negative slot skips its token.
 * Returns the number of tokens whose slot was >= num_slots (those are skipped too). */
int64_t oracle_quantize_append(const uint16_t* latent, int64_t latent_row_stride,
                               const uint16_t* rope, int64_t rope_row_stride,
                               const int64_t* slot_mapping, int64_t T, uint8_t* cache,
                               int64_t num_slots, int record_bytes, int block_order) {
    int64_t out_of_range = 0;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            ++out_of_range;
            continue;
        }
        oracle_quantize_record(latent + t * latent_row_stride, rope + t * rope_row_stride,
                               record_bytes, block_order, cache + slot * (int64_t)record_bytes);
    }
    return out_of_range;
}

/* Dequantize a record into the 576-dim key: K[0:512] = e2m1(code) * scale of its block,
 * K[512:576] = RoPE (e4m3 for 352 B, bf16 for 432 B). V is K[0:512]. */
void oracle_dequant_record(const uint8_t* rec, int record_bytes, int block_order, double* k) {
    if (record_bytes == 656) {
        /* K[0:512] = bf16(e4m3(code) * scale of its tile), K[512:576] = bf16 RoPE */
        for (int d = 0; d < 512; ++d) {
            float s;
            memcpy(&s, rec + 512 + 4 * (d / 128), 4);
            k[d] = oracle_round_to_bf16(oracle_e4m3_decode(rec[d]) * (double)s);
        }
        for (int j = 0; j < 64; ++j) {
            uint16_t bits = (uint16_t)(rec[528 + 2 * j] | (rec[529 + 2 * j] << 8));
            k[512 + j] = oracle_bf16_to_double(bits);
        }
        return;
    }
    for (int d = 0; d < 512; ++d) {
        uint8_t byte = rec[d / 2];
        uint8_t nibble = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
        double s = oracle_e4m3_decode(rec[oracle_scale_offset(record_bytes, block_order, d / 16)]);
        k[d] = oracle_e2m1_decode(nibble) * s;
    }
    for (int j = 0; j < 64; ++j) {
        if (record_bytes == 352) {
            k[512 + j] = oracle_e4m3_decode(rec[256 + j]);
        } else {
            uint16_t bits = (uint16_t)(rec[304 + 2 * j] | (rec[305 + 2 * j] << 8));
            k[512 + j] = oracle_bf16_to_double(bits);
        }
    }
}

void oracle_dequant_records(const uint8_t* recs, int64_t n, int record_bytes, int block_order, double* k) {
    for (int64_t i = 0; i < n; ++i)
        oracle_dequant_record(recs + i * record_bytes, record_bytes, block_order, k + i * 576);
}

/*
 * Sparse MLA decode, straight from its definition, for query rows tok_list[0..n_list)
 * (all n_tok rows when tok_list is NULL).
 *   q        bf16 bits [n_tok, h_q, 576]
 *   indices  int32 [n_tok, *] with row stride idx_row_stride; topk entries used per row
 *   sink     NULL or fp32 [h_q]
 *   out      fp64 [n_list, h_q, 512], lse fp64 [n_list, h_q]
 * For one row t and head h, with J the used indices of row t:
 *   z_j = sm_scale * sum_d q[t,h,d] * K_j[d]
 *   m = max z_j, Z = sum_j exp(z_j - m), lse = m + ln Z
 *   out = sum_j exp(z_j - m) * V_j / (Z + [sink] exp(sink_h - m))
 * The keys of a row are dequantized once and reused by all of its heads.
 */
void oracle_sparse_mla_decode(const uint16_t* q, const uint8_t* cache, int64_t num_slots,
                              int record_bytes, int block_order, const int32_t* indices, int64_t idx_row_stride,
                              int64_t n_tok, int h_q, int topk, double sm_scale,
                              const float* sink, const int64_t* tok_list, int64_t n_list,
                              double* out, double* lse, int threads) {
    if (tok_list == NULL) n_list = n_tok;
    /* threads > 0: that many OpenMP threads for this call only; 0: every host core */
#ifdef _OPENMP
    const int n_threads = threads > 0 ? threads : omp_get_num_procs();
#else
    (void)threads;
#endif
    double* keys = (double*)malloc(sizeof(double) * 576 * (size_t)(topk > 0 ? topk : 1));
    for (int64_t r = 0; r < n_list; ++r) {
        int64_t t = tok_list ? tok_list[r] : r;
        const int32_t* row = indices + t * idx_row_stride;
        int n_used = 0;
        for (int j = 0; j < topk; ++j) {
            int64_t slot = row[j];
            if (slot < 0 || slot >= num_slots) continue;
            oracle_dequant_record(cache + slot * (int64_t)record_bytes, record_bytes, block_order,
                                  keys + 576 * (size_t)n_used);
            ++n_used;
        }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic) num_threads(n_threads)
#endif
        for (int h = 0; h < h_q; ++h) {
            double* o = out + ((size_t)r * h_q + h) * 512;
            double* l = lse + (size_t)r * h_q + h;
            for (int d = 0; d < 512; ++d) o[d] = 0.0;
            if (n_used == 0) {
                *l = -INFINITY;
                continue;
            }
            const uint16_t* qrow = q + ((size_t)t * h_q + h) * 576;
            double qd[576];
            for (int d = 0; d < 576; ++d) qd[d] = oracle_bf16_to_double(qrow[d]);
            double* z = (double*)malloc(sizeof(double) * (size_t)n_used);
            double m = -INFINITY;
            for (int j = 0; j < n_used; ++j) {
                const double* k = keys + 576 * (size_t)j;
                double acc = 0.0;
                for (int d = 0; d < 576; ++d) acc += qd[d] * k[d];
                z[j] = sm_scale * acc;
                if (z[j] > m) m = z[j];
            }
            double Z = 0.0;
            for (int j = 0; j < n_used; ++j) {
                double p = exp(z[j] - m);
                Z += p;
                const double* v = keys + 576 * (size_t)j;
                for (int d = 0; d < 512; ++d) o[d] += p * v[d];
            }
            double denom = Z + (sink ? exp((double)sink[h] - m) : 0.0);
            for (int d = 0; d < 512; ++d) o[d] /= denom;
            *l = m + log(Z);
            free(z);
        }
    }
    free(keys);
}

/*
 * Merge of P partial results of one (row, head), each over a disjoint part of the used
 * indices and without the sink: partial p has out_p (normalised over its own part) and
 * lse_p (-inf when its part is empty). The merged result is
 *   lse = ln sum_p exp(lse_p),  out = sum_p exp(lse_p - lse) out_p / (1 + [sink] exp(sink - lse))
 * which is the same softmax over the union of the parts.
 */
void oracle_merge_partials(int P, const double* lse_p, const double* out_p, const double* sink,
                           double* out, double* lse) {
    double m = -INFINITY;
    for (int p = 0; p < P; ++p)
        if (lse_p[p] > m) m = lse_p[p];
    for (int d = 0; d < 512; ++d) out[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int p = 0; p < P; ++p) sum += exp(lse_p[p] - m);
    double total = m + log(sum);
    double scale = 1.0 + (sink ? exp(*sink - total) : 0.0);
    for (int p = 0; p < P; ++p) {
        double w = exp(lse_p[p] - total);
        for (int d = 0; d < 512; ++d) out[d] += w * out_p[(size_t)p * 512 + d];
    }
    for (int d = 0; d < 512; ++d) out[d] /= scale;
    *lse = total;
}

/* Vector helpers so the Python side can check single-value conversions in bulk. */
/* ---- the producer ahead of the append: RMSNorm + rotary embedding ------------------------
 *
 * [SGLang-38646] "[SM120] Add opt-in NVFP4 sparse-MLA KV cache format for DeepSeek-V4"
 * (SGLang pull request 38646), "Limitations" (the NVFP4 path has no fused
 * norm+rope+quantize+store kernel and pays a bf16 intermediate plus a separate quantize kernel)
 * and "Stores" (the fused store kernels emit only the fp8 layout). The pages name the stages but
 * fix none of their parameters; the readings used here:
 *  - RMSNorm of the 512 latent values of a token: y_i = w_i * x_i / sqrt(mean_j x_j^2 + eps),
 *    with a weight vector w (bf16) and eps given by the caller;
 *  - rotary embedding of the 64 k_pe values at the token's position p, frequency f in 0..31
 *    with c = cos_table[p][f], s = sin_table[p][f] (fp32 tables given by the caller), the pair
 *    (a, b) of frequency f rotated to (a c - b s, b c + a s); pairs are (f, f + 32) ("rotate
 *    half") or (2f, 2f + 1) ("interleaved"), a flag of the call;
 *  - both in fp64 from the bf16 inputs, each result rounded once to bf16 (round to nearest,
 *    ties to even): the same numbers the unfused path stores in its bf16 intermediate, which
 *    the append then quantizes;
 *  - a token whose position is outside [0, num_positions) is not written.
 * A kernel computing in fp32 may round a value the other way when the exact value lies within
 * its own error of a bf16 rounding midpoint. So every value whose exact result lies within
 * 2^-16 times the size of its terms (|y_i| for the norm, |a c| + |b s| for the rotation) of a
 * midpoint is flagged, with the other admissible bf16 value, and a test accepts either. */
static const double kMidpointBand = 1.0 / 65536.0;

/* bf16 bits of a double that is exactly a bf16 value */
static uint16_t bf16_bits_of(double r) {
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Rounds v to bf16 (bits into *near); when v lies within `band` of the midpoint between the two
 * bf16 values around it, *flag = 1 and *other = the bits of the other one; else *other = *near. */
static void round_with_flag(double v, double band, uint16_t* near, uint16_t* other, uint8_t* flag) {
    const double r = oracle_round_to_bf16(v);
    *near = bf16_bits_of(r);
    *other = *near;
    *flag = 0;
    if (v == r || !isfinite(r)) return;
    /* the neighbour of r on v's side, one bf16 step away */
    uint16_t nb = *near;
    const int up = (v > r);            /* v lies above r */
    const int neg = (nb & 0x8000) != 0;
    if (r == 0.0) nb = (uint16_t)(up ? 0x0001 : 0x8001);
    else nb = (uint16_t)((up != neg) ? nb + 1 : nb - 1);
    const double n2 = oracle_bf16_to_double(nb);
    const double mid = 0.5 * (r + n2);
    if (fabs(v - mid) <= band) {
        *flag = 1;
        *other = nb;
    }
}

/* latent [T, 512] and k_pe [T, 64] bf16 bits (row strides in elements), positions [T],
 * weight [512] bf16 bits, cos/sin [num_positions, 32]. Outputs, per token: the normalized
 * latent and rotated k_pe as bf16 bits (lat_out [T, 512], rope_out [T, 64]), the exact values
 * (exact [T, 576], may be NULL), the flags and other admissible roundings (flag, other
 * [T, 576], the latent first), and valid[T] (0: position out of range, nothing else set). */
void oracle_norm_rope(const uint16_t* latent, int64_t latent_row_stride, const uint16_t* k_pe,
                      int64_t rope_row_stride, const int64_t* positions, int64_t T,
                      const uint16_t* weight, double eps, const float* cos_table, const float* sin_table,
                      int64_t num_positions, int rotate_half, uint16_t* lat_out, uint16_t* rope_out,
                      double* exact, uint8_t* flag, uint16_t* other, uint8_t* valid) {
    for (int64_t t = 0; t < T; ++t) {
        const int64_t p = positions[t];
        valid[t] = (uint8_t)(p >= 0 && p < num_positions);
        if (!valid[t]) continue;
        const uint16_t* x = latent + t * latent_row_stride;
        const uint16_t* k = k_pe + t * rope_row_stride;
        /* RMSNorm */
        double ss = 0.0;
        for (int i = 0; i < 512; ++i) {
            const double v = oracle_bf16_to_double(x[i]);
            ss += v * v;
        }
        const double inv = 1.0 / sqrt(ss / 512.0 + eps);
        for (int i = 0; i < 512; ++i) {
            const double y = oracle_bf16_to_double(weight[i]) * oracle_bf16_to_double(x[i]) * inv;
            if (exact) exact[t * 576 + i] = y;
            round_with_flag(y, kMidpointBand * fabs(y), &lat_out[t * 512 + i], &other[t * 576 + i],
                            &flag[t * 576 + i]);
        }
        /* rotary embedding */
        for (int f = 0; f < 32; ++f) {
            const int ia = rotate_half ? f : 2 * f;
            const int ib = rotate_half ? f + 32 : 2 * f + 1;
            const double a = oracle_bf16_to_double(k[ia]), b = oracle_bf16_to_double(k[ib]);
            const double c = (double)cos_table[p * 32 + f], s = (double)sin_table[p * 32 + f];
            const double oa = a * c - b * s, ob = b * c + a * s;
            const double band = kMidpointBand * (fabs(a * c) + fabs(b * s));
            const double bandb = kMidpointBand * (fabs(b * c) + fabs(a * s));
            if (exact) {
                exact[t * 576 + 512 + ia] = oa;
                exact[t * 576 + 512 + ib] = ob;
            }
            round_with_flag(oa, band, &rope_out[t * 64 + ia], &other[t * 576 + 512 + ia], &flag[t * 576 + 512 + ia]);
            round_with_flag(ob, bandb, &rope_out[t * 64 + ib], &other[t * 576 + 512 + ib], &flag[t * 576 + 512 + ib]);
        }
    }
}

void oracle_e4m3_encode_many(const float* f, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(f[i]);
}
void oracle_e2m1_encode_many(const float* f, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(f[i]);
}
void oracle_e4m3_decode_many(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}
int oracle_threads_available(void) {
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}
