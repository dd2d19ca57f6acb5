/*
 * CPU oracle for MoE expert-parallel dispatch / combine.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or
 * calls this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Plain, single-threaded, slow on purpose: every step is the definition
 * written out as loops, in the order the method states it. Compiled with
 * -O2 -ffp-contract=off and without fast-math so that float arithmetic is
 * IEEE binary32 with round-to-nearest-even and no contraction; where a fused
 * multiply-add is meant, fmaf() is called explicitly.
 *
 * Source pages (cited by title and section):
 *   [Guide]  "MORI-EP User Guide" -- sections 2 (EpDispatchCombineConfig),
 *            3 (Operator API: dispatch(), combine(), reset(),
 *            get_dispatch_src_token_pos()), 4 (Standard MoE Compatibility),
 *            7 (Complete Example).
 *   [Back]   "Choosing an EP API and backend" -- EP paths table (the
 *            combine is a gather, in bf16 or f32; dispatch may quantise),
 *            restrictions (OCP E4M3).
 *   [Issue]  MORI issue 57 -- a token travels to each owning rank once.
 *   [OCP]    OCP 8-bit Floating Point Specification (OFP8), E4M3 encoding.
 *   [IEEE]   IEEE 754 round-to-nearest-even; bfloat16 = binary32 with the
 *            low 16 significand bits removed.
 *
 * Readings of points the pages leave open (one line each):
 *   R1 recv row order: per destination rank, rows sorted by (src rank asc, token asc).
 *   R2 src_token_pos = src_rank * (world_size * max_tokens) + token, taken literally.
 *   R3 dispatched indices: the full top-k row of global expert ids, -1 kept.
 *   R4 FP8: per 128-element block, scale = amax / 448 (f32 divide), q = E4M3_RNE_sat(x / scale);
 *      amax == 0 gives scale 0 and q = enc(x) (signed zero).
 *   R5 combine: fp32 accumulator starting at +0.0f, ranks in ascending order, plain adds
 *      (unweighted) or fmaf(w_r, y, acc) (weighted, w_r = sum of the rank's slot weights
 *      in ascending slot order starting at +0.0f), one final rounding.
 *   R6 combine_weights: the weight row carried by the copy on the lowest destination rank.
 *   R7 standard-MoE: per destination rank, one contiguous segment per local expert in
 *      ascending expert order, each padded to a multiple of 128 rows; rows inside a
 *      segment in (src rank, token) order; layout_range[r][e][s] = (begin << 32) | count
 *      with begin = rows from source ranks below s; padding rows have src_info = -1.
 *   R8 standard-MoE combine: ranks ascending, then slots ascending, fmaf(w_j, y, acc).
 *   R9 convert_combine_input: per (token, rank) the unweighted fp32 sum of that token's
 *      expert rows on the rank, slots ascending, rounded once to the output dtype.
 *   R10 FP4: OCP E2M1 codes (bias 1, 1 mantissa bit, max 6, no Inf/NaN), one f32 scale per
 *      32-element block, scale = amax / 6, code = E2M1_RNE_sat(x / scale) (amax == 0: enc(x));
 *      two codes per byte, the even element in the low nibble.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_CAPACITY (-3)
#define ORC_ERR_INDEX (-4)
#define ORC_MAX_RANKS 64

#define DT_BF16 0
#define DT_F32 1

/* ---------------------------------------------------------------- codecs */

/* [IEEE] binary32 -> bfloat16, round to nearest, ties to even. */
uint16_t oracle_bf16_from_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, sign kept */
    uint32_t hi = u >> 16;           /* truncated bfloat16 */
    uint32_t lo = u & 0xFFFFu;       /* discarded bits */
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u; /* carry may reach Inf: correct */
    return (uint16_t)hi;
}

float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* [OCP] E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * NaN = S.1111.111; largest finite 448 = 0.1111.110; subnormals M * 2^-9.
 * Round to nearest with ties to the even code, then saturate to +-448. */
uint8_t oracle_e4m3_from_f32(float v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);             /* a = m * 2^e2, m in [0.5, 1) */
    int ue = e2 - 1;                 /* a in [2^ue, 2^(ue+1)) */
    if (ue < -6) ue = -6;            /* subnormals share the smallest normal's spacing */
    double quantum = ldexp(1.0, ue - 3);     /* distance between neighbouring codes */
    double n = rint(a / quantum);            /* exact scaling; rint = ties-to-even */
    double q = n * quantum;                  /* the chosen representable magnitude */
    if (q > 448.0) return (uint8_t)(sign | 0x7E);
    if (q == 0.0) return sign;
    if (q < ldexp(1.0, -6)) {                /* subnormal: q = M * 2^-9 */
        int M = (int)(q / ldexp(1.0, -9));
        return (uint8_t)(sign | M);
    }
    (void)frexp(q, &e2);
    int E = (e2 - 1) + 7;
    int M = (int)(q / ldexp(1.0, e2 - 1) * 8.0) - 8;
    return (uint8_t)(sign | (E << 3) | M);
}

float oracle_e4m3_to_f32(uint8_t c) {
    int s = c >> 7, E = (c >> 3) & 15, M = c & 7;
    if (E == 15 && M == 7) return NAN;
    double v = (E == 0) ? M * ldexp(1.0, -9) : (1.0 + M / 8.0) * ldexp(1.0, E - 7);
    return (float)(s ? -v : v);
}

void oracle_e4m3_from_f32_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_f32(v[i]);
}

void oracle_bf16_from_f32_array(const float* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_f32(v[i]);
}

/* [OCP] E2M1 (FP4): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; no
 * infinities or NaN; magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6.
 * Round to nearest with ties to the even code, then saturate to +-6. */
uint8_t oracle_e2m1_from_f32(float v) {
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    if (isnan(v)) return 0x7;                /* no NaN code: saturate (never generated) */
    double a = fabs((double)v);
    if (a >= 6.0) return (uint8_t)(sign | 0x7);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);
    int ue = e2 - 1;                         /* a in [2^ue, 2^(ue+1)) */
    if (ue < 0) ue = 0;                      /* subnormal 0.5 shares the spacing of [1, 2) */
    double quantum = ldexp(1.0, ue - 1);     /* one mantissa bit */
    double q = rint(a / quantum) * quantum;  /* ties to even */
    if (q > 6.0) return (uint8_t)(sign | 0x7);
    if (q == 0.0) return sign;
    if (q < 1.0) return (uint8_t)(sign | 0x1); /* 0.5 */
    (void)frexp(q, &e2);
    int E = (e2 - 1) + 1;
    int M = (int)(q / ldexp(1.0, e2 - 1) * 2.0) - 2;
    return (uint8_t)(sign | (E << 1) | M);
}

float oracle_e2m1_to_f32(uint8_t c) {
    int s = (c >> 3) & 1, E = (c >> 1) & 3, M = c & 1;
    double v = (E == 0) ? M * 0.5 : (1.0 + M / 2.0) * ldexp(1.0, E - 1);
    return (float)(s ? -v : v);
}

void oracle_e2m1_from_f32_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_from_f32(v[i]);
}

static float load_elem(int dtype, const void* base, int64_t i) {
    if (dtype == DT_BF16) return oracle_bf16_to_f32(((const uint16_t*)base)[i]);
    return ((const float*)base)[i];
}

static void store_elem(int dtype, void* base, int64_t i, float v) {
    if (dtype == DT_BF16) ((uint16_t*)base)[i] = oracle_bf16_from_f32(v);
    else ((float*)base)[i] = v;
}

/* ------------------------------------------------------- FP8 quantisation */

/* [Back] restrictions (OCP E4M3) + reading R4: one token row of H bf16 values
 * -> H E4M3 codes and H/128 f32 scales. */
void oracle_quant_row(int H, const uint16_t* x, uint8_t* q, float* scales) {
    for (int b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float a = fabsf(oracle_bf16_to_f32(x[b * 128 + i]));
            if (a > amax) amax = a;
        }
        float scale = amax / 448.0f;
        scales[b] = scale;
        for (int i = 0; i < 128; ++i) {
            float v = oracle_bf16_to_f32(x[b * 128 + i]);
            q[b * 128 + i] = (amax == 0.0f) ? oracle_e4m3_from_f32(v)
                                            : oracle_e4m3_from_f32(v / scale);
        }
    }
}

void oracle_quant_tokens(int64_t n, int H, const uint16_t* x, uint8_t* q, float* scales) {
    for (int64_t i = 0; i < n; ++i)
        oracle_quant_row(H, x + i * H, q + i * H, scales + i * (H / 128));
}

/* Reading R10: one token row of H bf16 values -> H/2 bytes of packed E2M1
 * codes and H/32 f32 scales. */
void oracle_quant_row_fp4(int H, const uint16_t* x, uint8_t* q, float* scales) {
    for (int b = 0; b < H / 32; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(oracle_bf16_to_f32(x[b * 32 + i]));
            if (a > amax) amax = a;
        }
        float scale = amax / 6.0f;
        scales[b] = scale;
        for (int i = 0; i < 32; i += 2) {
            float v0 = oracle_bf16_to_f32(x[b * 32 + i]);
            float v1 = oracle_bf16_to_f32(x[b * 32 + i + 1]);
            uint8_t c0 = (amax == 0.0f) ? oracle_e2m1_from_f32(v0) : oracle_e2m1_from_f32(v0 / scale);
            uint8_t c1 = (amax == 0.0f) ? oracle_e2m1_from_f32(v1) : oracle_e2m1_from_f32(v1 / scale);
            q[(b * 32 + i) / 2] = (uint8_t)(c0 | (c1 << 4));
        }
    }
}

void oracle_quant_tokens_fp4(int64_t n, int H, const uint16_t* x, uint8_t* q, float* scales) {
    for (int64_t i = 0; i < n; ++i)
        oracle_quant_row_fp4(H, x + i * H, q + i * (H / 2), scales + i * (H / 32));
}

/* ------------------------------------------------------- routing layout */

/* [Guide] s.2 num_experts_per_rank ("256 experts / 8 GPUs"), s.3 dispatch()
 * and get_dispatch_src_token_pos(); [Issue] one copy per distinct rank.
 * idx [R][Tmax][k]; outputs recv_num_token [R], src_pos [R][R*Tmax]
 * (-1 past the count), slot [R][Tmax][R] (-1 = token not sent to rank). */
int oracle_route(int R, int Tmax, int k, int E_r, const int32_t* ntok, const int32_t* idx,
                 int32_t* recv_num_token, int32_t* src_pos, int32_t* slot) {
    if (R < 1 || R > ORC_MAX_RANKS || Tmax < 0 || k < 1 || E_r < 1) return ORC_ERR_ARG;
    int64_t cap = (int64_t)R * Tmax;
    int32_t E = R * E_r;
    for (int s = 0; s < R; ++s) {
        if (ntok[s] < 0 || ntok[s] > Tmax) return ORC_ERR_ARG;
        for (int t = 0; t < ntok[s]; ++t)
            for (int j = 0; j < k; ++j) {
                int32_t e = idx[((int64_t)s * Tmax + t) * k + j];
                if (e < -1 || e >= E) return ORC_ERR_INDEX;
            }
    }
    for (int r = 0; r < R; ++r) {
        recv_num_token[r] = 0;
        for (int64_t i = 0; i < cap; ++i) src_pos[r * cap + i] = -1;
    }
    for (int64_t g = 0; g < cap; ++g)
        for (int r = 0; r < R; ++r) slot[g * R + r] = -1;

    /* visit source tokens in (rank asc, token asc) order: reading R1 */
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < ntok[s]; ++t) {
            int64_t g = (int64_t)s * Tmax + t;
            int dest[ORC_MAX_RANKS] = {0};
            for (int j = 0; j < k; ++j) {
                int32_t e = idx[g * k + j];
                if (e < 0) continue;               /* dropped slot */
                dest[e / E_r] = 1;                 /* owner rank */
            }
            for (int r = 0; r < R; ++r) {
                if (!dest[r]) continue;
                int32_t i = recv_num_token[r]++;
                slot[g * R + r] = i;
                src_pos[r * cap + i] = s * (R * Tmax) + t;   /* reading R2 */
            }
        }
    return ORC_OK;
}

/* Copy every source row [R][Tmax][row_bytes] to each receive slot it was
 * routed to; dst is [R][R*Tmax][row_bytes]. Used for payload, weights,
 * indices and pass-through scales alike: dispatch moves bits unchanged. */
void oracle_place_rows(int R, int Tmax, int64_t row_bytes, const int32_t* ntok,
                       const int32_t* slot, const uint8_t* src, uint8_t* dst) {
    int64_t cap = (int64_t)R * Tmax;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < ntok[s]; ++t) {
            int64_t g = (int64_t)s * Tmax + t;
            for (int r = 0; r < R; ++r) {
                int32_t i = slot[g * R + r];
                if (i < 0) continue;
                memcpy(dst + ((int64_t)r * cap + i) * row_bytes, src + g * row_bytes,
                       (size_t)row_bytes);
            }
        }
}

/* ---------------------------------------------------------------- combine */

/* [Guide] s.3 combine(): gather expert outputs back to the source token;
 * [Back] the combine is a gather, in bf16 or f32. y is [R][R*Tmax][H] (y_dtype),
 * w_recv [R][R*Tmax][k] or NULL, out [R][Tmax][H] (out_dtype),
 * out_w [R][Tmax][k] or NULL. Readings R5, R6. */
/* One source token g = s*Tmax + t of the 2D combine; out_row [H], out_w_row [k] or NULL. */
static void combine_token(int R, int Tmax, int k, int E_r, int H, int64_t g, const int32_t* idx,
                          const int32_t* slot, int y_dtype, const void* y, const float* w_recv,
                          int weighted, int out_dtype, void* out_row, float* out_w_row) {
    int64_t cap = (int64_t)R * Tmax;
    float wr[ORC_MAX_RANKS];
    for (int r = 0; r < R; ++r) {
        wr[r] = 0.0f;
        int32_t i = slot[g * R + r];
        if (i < 0 || !w_recv) continue;
        for (int j = 0; j < k; ++j) {
            int32_t e = idx[g * k + j];
            if (e >= 0 && e / E_r == r) wr[r] = wr[r] + w_recv[((int64_t)r * cap + i) * k + j];
        }
    }
    if (out_w_row) {
        int rmin = -1;
        for (int r = R - 1; r >= 0; --r)
            if (slot[g * R + r] >= 0) rmin = r;
        for (int j = 0; j < k; ++j)
            out_w_row[j] = (rmin >= 0 && w_recv)
                ? w_recv[((int64_t)rmin * cap + slot[g * R + rmin]) * k + j] : 0.0f;
    }
    for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int r = 0; r < R; ++r) {
            int32_t i = slot[g * R + r];
            if (i < 0) continue;
            float v = load_elem(y_dtype, y, ((int64_t)r * cap + i) * H + h);
            if (weighted) acc = fmaf(wr[r], v, acc);
            else acc = acc + v;
        }
        store_elem(out_dtype, out_row, h, acc);
    }
}

static int64_t dtype_bytes(int dt) { return dt == DT_BF16 ? 2 : 4; }

/* [Guide] s.3 combine(): gather expert outputs back to the source token;
 * [Back] the combine is a gather, in bf16 or f32. y is [R][R*Tmax][H] (y_dtype),
 * w_recv [R][R*Tmax][k] or NULL, out [R][Tmax][H] (out_dtype),
 * out_w [R][Tmax][k] or NULL. Readings R5, R6. */
int oracle_combine(int R, int Tmax, int k, int E_r, int H, const int32_t* ntok,
                   const int32_t* idx, const int32_t* slot, int y_dtype, const void* y,
                   const float* w_recv, int weighted, int out_dtype, void* out, float* out_w) {
    if (R < 1 || R > ORC_MAX_RANKS) return ORC_ERR_ARG;
    if (weighted && !w_recv) return ORC_ERR_ARG;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < ntok[s]; ++t) {
            int64_t g = (int64_t)s * Tmax + t;
            combine_token(R, Tmax, k, E_r, H, g, idx, slot, y_dtype, y, w_recv, weighted,
                          out_dtype, (uint8_t*)out + g * H * dtype_bytes(out_dtype),
                          out_w ? out_w + g * k : NULL);
        }
    return ORC_OK;
}

/* The same combine for a list of source tokens g only: out [n][H], out_w [n][k]. */
int oracle_combine_tokens(int R, int Tmax, int k, int E_r, int H, const int64_t* tokens,
                          int64_t n, const int32_t* idx, const int32_t* slot, int y_dtype,
                          const void* y, const float* w_recv, int weighted, int out_dtype,
                          void* out, float* out_w) {
    if (R < 1 || R > ORC_MAX_RANKS) return ORC_ERR_ARG;
    if (weighted && !w_recv) return ORC_ERR_ARG;
    for (int64_t q = 0; q < n; ++q)
        combine_token(R, Tmax, k, E_r, H, tokens[q], idx, slot, y_dtype, y, w_recv, weighted,
                      out_dtype, (uint8_t*)out + q * H * dtype_bytes(out_dtype),
                      out_w ? out_w + q * k : NULL);
    return ORC_OK;
}

/* ------------------------------------------------------- standard MoE */

static int64_t round_up_128(int64_t n) { return (n + 127) / 128 * 128; }

/* [Guide] s.4 dispatch_standard_moe() / convert_dispatch_output(), reading R7.
 * One packed row per valid (token, slot): no per-rank deduplication.
 * Outputs: count/seg_off [R][E_r], rank_rows [R] (padded rows used),
 * row_map [R][Tmax][k] (global packed row r*pcap+row, or -1),
 * src_info [R][pcap] (-1 for padding and unused rows),
 * layout_range [R][E_r][R]. Duplicate valid ids in one row are rejected. */
int oracle_std_layout(int R, int Tmax, int k, int E_r, int64_t pcap, const int32_t* ntok,
                      const int32_t* idx, int32_t* count, int32_t* seg_off, int32_t* rank_rows,
                      int32_t* row_map, int32_t* src_info, int64_t* layout_range) {
    if (R < 1 || R > ORC_MAX_RANKS || k < 1 || E_r < 1) return ORC_ERR_ARG;
    int32_t E = R * E_r;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < ntok[s]; ++t)
            for (int j = 0; j < k; ++j) {
                int32_t e = idx[((int64_t)s * Tmax + t) * k + j];
                if (e < -1 || e >= E) return ORC_ERR_INDEX;
                for (int jj = 0; jj < j; ++jj)
                    if (e >= 0 && idx[((int64_t)s * Tmax + t) * k + jj] == e) return ORC_ERR_INDEX;
            }
    for (int64_t g = 0; g < (int64_t)R * Tmax * k; ++g) row_map[g] = -1;
    for (int64_t i = 0; i < (int64_t)R * pcap; ++i) src_info[i] = -1;

    for (int r = 0; r < R; ++r) {
        int64_t off = 0;
        for (int el = 0; el < E_r; ++el) {
            int32_t e = r * E_r + el;
            int64_t pos = 0;
            seg_off[r * E_r + el] = (int32_t)off;
            for (int s = 0; s < R; ++s) {
                int64_t begin = pos;
                for (int t = 0; t < ntok[s]; ++t)
                    for (int j = 0; j < k; ++j) {
                        int64_t g = (int64_t)s * Tmax + t;
                        if (idx[g * k + j] != e) continue;
                        int64_t row = off + pos;
                        if (row >= pcap) return ORC_ERR_CAPACITY;
                        row_map[g * k + j] = (int32_t)(r * pcap + row);
                        src_info[r * pcap + row] = s * (R * Tmax) + t;
                        pos++;
                    }
                layout_range[((int64_t)r * E_r + el) * R + s] =
                    (int64_t)(((uint64_t)begin << 32) | (uint64_t)(pos - begin));
            }
            count[r * E_r + el] = (int32_t)pos;
            off += round_up_128(pos);
        }
        if (off > pcap) return ORC_ERR_CAPACITY;
        rank_rows[r] = (int32_t)off;
    }
    return ORC_OK;
}

/* Copy every source row to each packed row of its valid slots. */
void oracle_std_place_rows(int R, int Tmax, int k, int64_t row_bytes, const int32_t* ntok,
                           const int32_t* row_map, const uint8_t* src, uint8_t* dst) {
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < ntok[s]; ++t) {
            int64_t g = (int64_t)s * Tmax + t;
            for (int j = 0; j < k; ++j) {
                int32_t m = row_map[g * k + j];
                if (m < 0) continue;
                memcpy(dst + (int64_t)m * row_bytes, src + g * row_bytes, (size_t)row_bytes);
            }
        }
}

/* One source token of the standard-MoE combine; out_row [H]. */
static void std_combine_token(int R, int k, int E_r, int H, int64_t g, const int32_t* idx,
                              const int32_t* row_map, int y_dtype, const void* Y, const float* w,
                              int weighted, int out_dtype, void* out_row) {
    for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int r = 0; r < R; ++r)
            for (int j = 0; j < k; ++j) {
                int32_t e = idx[g * k + j];
                if (e < 0 || e / E_r != r) continue;
                float v = load_elem(y_dtype, Y, (int64_t)row_map[g * k + j] * H + h);
                if (weighted) acc = fmaf(w[g * k + j], v, acc);
                else acc = acc + v;
            }
        store_elem(out_dtype, out_row, h, acc);
    }
}

/* [Guide] s.4 combine_standard_moe(), reading R8. Y is the packed expert
 * output [R][pcap][H]; w [R][Tmax][k] source-side router weights. */
int oracle_std_combine(int R, int Tmax, int k, int E_r, int H, const int32_t* ntok,
                       const int32_t* idx, const int32_t* row_map, int y_dtype, const void* Y,
                       const float* w, int weighted, int out_dtype, void* out) {
    if (R < 1 || R > ORC_MAX_RANKS) return ORC_ERR_ARG;
    if (weighted && !w) return ORC_ERR_ARG;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < ntok[s]; ++t) {
            int64_t g = (int64_t)s * Tmax + t;
            std_combine_token(R, k, E_r, H, g, idx, row_map, y_dtype, Y, w, weighted, out_dtype,
                              (uint8_t*)out + g * H * dtype_bytes(out_dtype));
        }
    return ORC_OK;
}

/* The same for a list of source tokens g only: out [n][H]. */
int oracle_std_combine_tokens(int R, int k, int E_r, int H, const int64_t* tokens, int64_t n,
                              const int32_t* idx, const int32_t* row_map, int y_dtype,
                              const void* Y, const float* w, int weighted, int out_dtype,
                              void* out) {
    if (R < 1 || R > ORC_MAX_RANKS) return ORC_ERR_ARG;
    if (weighted && !w) return ORC_ERR_ARG;
    for (int64_t q = 0; q < n; ++q)
        std_combine_token(R, k, E_r, H, tokens[q], idx, row_map, y_dtype, Y, w, weighted,
                          out_dtype, (uint8_t*)out + q * H * dtype_bytes(out_dtype));
    return ORC_OK;
}

/* [Guide] s.4 convert_dispatch_output(): the per-expert packed layout built
 * from the 2D receive buffers (recv_x [R][cap][row_bytes], recv_idx
 * [R][cap][k], recv_src_pos [R][cap]) instead of from the source tokens.
 * Rows of a receive buffer are already in (src rank, token) order, so the
 * segment order is receive-row order. Also rebuilds row_map [R][Tmax][k]. */
int oracle_convert_dispatch_output(int R, int Tmax, int k, int E_r, int64_t pcap,
                                   int64_t row_bytes, const int32_t* recv_num_token,
                                   const uint8_t* recv_x, const int32_t* recv_idx,
                                   const int32_t* recv_src_pos, int32_t* count, int32_t* seg_off,
                                   int32_t* rank_rows, int32_t* row_map, uint8_t* packed_x,
                                   int32_t* src_info, int64_t* layout_range) {
    if (R < 1 || R > ORC_MAX_RANKS) return ORC_ERR_ARG;
    int64_t cap = (int64_t)R * Tmax;
    int64_t stride = (int64_t)R * Tmax;          /* src_token_pos rank stride */
    for (int64_t g = 0; g < (int64_t)R * Tmax * k; ++g) row_map[g] = -1;
    for (int64_t i = 0; i < (int64_t)R * pcap; ++i) src_info[i] = -1;
    for (int r = 0; r < R; ++r) {
        int64_t off = 0;
        for (int el = 0; el < E_r; ++el) {
            int32_t e = r * E_r + el;
            int64_t per_src[ORC_MAX_RANKS] = {0};
            for (int i = 0; i < recv_num_token[r]; ++i)
                for (int j = 0; j < k; ++j)
                    if (recv_idx[((int64_t)r * cap + i) * k + j] == e)
                        per_src[recv_src_pos[r * cap + i] / stride]++;
            int64_t begin = 0;
            for (int s = 0; s < R; ++s) {
                layout_range[((int64_t)r * E_r + el) * R + s] =
                    (int64_t)(((uint64_t)begin << 32) | (uint64_t)per_src[s]);
                begin += per_src[s];
            }
            seg_off[r * E_r + el] = (int32_t)off;
            int64_t pos = 0;
            for (int i = 0; i < recv_num_token[r]; ++i)
                for (int j = 0; j < k; ++j) {
                    if (recv_idx[((int64_t)r * cap + i) * k + j] != e) continue;
                    int64_t row = off + pos;
                    if (row >= pcap) return ORC_ERR_CAPACITY;
                    int32_t p = recv_src_pos[r * cap + i];
                    int64_t g = (int64_t)(p / stride) * Tmax + (p % stride);
                    memcpy(packed_x + ((int64_t)r * pcap + row) * row_bytes,
                           recv_x + ((int64_t)r * cap + i) * row_bytes, (size_t)row_bytes);
                    src_info[r * pcap + row] = p;
                    row_map[g * k + j] = (int32_t)(r * pcap + row);
                    pos++;
                }
            count[r * E_r + el] = (int32_t)pos;
            off += round_up_128(pos);
        }
        if (off > pcap) return ORC_ERR_CAPACITY;
        rank_rows[r] = (int32_t)off;
    }
    return ORC_OK;
}

/* [Guide] s.4 convert_combine_input(), reading R9: 2D combine input
 * y2d [R][cap][H] from the packed expert outputs Y [R][pcap][H]. */
int oracle_convert_combine_input(int R, int Tmax, int k, int E_r, int H,
                                 const int32_t* recv_num_token, const int32_t* recv_src_pos,
                                 const int32_t* idx, const int32_t* row_map, int y_dtype,
                                 const void* Y, int out_dtype, void* y2d) {
    if (R < 1 || R > ORC_MAX_RANKS) return ORC_ERR_ARG;
    int64_t cap = (int64_t)R * Tmax;
    int64_t stride = (int64_t)R * Tmax;
    for (int r = 0; r < R; ++r)
        for (int i = 0; i < recv_num_token[r]; ++i) {
            int32_t p = recv_src_pos[r * cap + i];
            int64_t g = (int64_t)(p / stride) * Tmax + (p % stride);
            for (int h = 0; h < H; ++h) {
                float acc = 0.0f;
                for (int j = 0; j < k; ++j) {
                    int32_t e = idx[g * k + j];
                    if (e < 0 || e / E_r != r) continue;
                    acc = acc + load_elem(y_dtype, Y, (int64_t)row_map[g * k + j] * H + h);
                }
                store_elem(out_dtype, y2d, ((int64_t)r * cap + i) * H + h, acc);
            }
        }
    return ORC_OK;
}
