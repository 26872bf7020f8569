/*
 * ds41_oracle.c - plain, slow CPU oracle for one layer's compressed sparse
 * attention forward (window ring, compressed latent rows, fp4 indexer top-k,
 * sparse attention with a per-head sink).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent definition the CUDA
 * path is checked against.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load it; the product library never links,
 * calls or falls back to it, and it shares no source, header, table or helper
 * with the CUDA path.
 *
 * Sources (page title, then the function or section on it):
 *   [compress]  metrale_model_arch/deepseek_v41_ref/compress.rs
 *               (DeepSeek-V4.1 compressed attention, CPU reference)
 *   [forward]   metrale_model_arch/attn_v41/forward.rs (AttnV41::forward)
 *
 * Build: any C11 compiler, -O2 -ffp-contract=off, no fast-math.  Contraction
 * of a*b+c into an FMA would change f32 results, so every f32 expression here
 * is meant to be evaluated exactly as written, one rounding per operation.
 *
 * Parity unpinned (the pages give no worked example, so these follow a
 * reading, not a value the pages fix): the indexer's score formula, which dims
 * apply_rotary rotates and how it pairs them, and the YaRN constants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Bit views                                                                 */
/* ------------------------------------------------------------------------- */
static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the upper half of an IEEE binary32 word. */
float ds41o_bf16_to_f32(uint16_t h) { return f_of((uint32_t)h << 16); }

/* to_bf16_rne (named in [compress], body not printed).  Reading: IEEE binary32
 * to bfloat16, round to nearest, ties to the even bfloat16.  The dropped half
 * word decides: above 0x8000 rounds up, below rounds down, exactly 0x8000
 * rounds to the neighbour whose last kept bit is 0.  A carry out of the
 * mantissa moves into the exponent, which is what the next bfloat16 is. */
uint16_t ds41o_f32_to_bf16_rne(float x) {
    uint32_t u = u_of(x);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a quiet NaN */
    uint32_t keep = u >> 16;
    uint32_t drop = u & 0xffffu;
    if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

static float bf16_round(float x) { return ds41o_bf16_to_f32(ds41o_f32_to_bf16_rne(x)); }

/* ------------------------------------------------------------------------- */
/* e2m1 (fp4) grid: [compress], constants FP4_MAX and E2M1, to_e2m1_rne.      */
/* ------------------------------------------------------------------------- */
static const float kGrid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
#define FP4_MAX 6.0f

/* Index (0..7) of the grid value nearest |y|; on a tie the even index wins.
 * Between neighbouring grid values g_i <= a <= g_{i+1} both differences are
 * exact in f32 (g_{i+1} <= 2 g_i, Sterbenz), so the tie test is exact. */
static int e2m1_index(float y) {
    float a = fabsf(y);
    int best = 0;
    float bestd = fabsf(a - kGrid[0]);
    for (int i = 1; i < 8; i++) {
        float d = fabsf(a - kGrid[i]);
        if (d < bestd || (d == bestd && (i % 2 == 0) && (best % 2 == 1))) {
            best = i;
            bestd = d;
        }
    }
    return best;
}

/* to_e2m1_rne: nearest grid value, ties to the even code, sign of y kept
 * (so a negative input that rounds to zero gives -0). */
float ds41o_to_e2m1_rne(float y) { return copysignf(kGrid[e2m1_index(y)], y); }

/* 4-bit code of to_e2m1_rne(y): bit 3 is the sign, bits 0..2 the grid index. */
static uint8_t e2m1_code(float y) {
    return (uint8_t)((signbit(y) ? 8 : 0) | e2m1_index(y));
}

/* pow2_ceil (named in [compress], body not printed).  Reading: the smallest
 * power of two >= x for x > 0.  frexp gives x = f * 2^e with f in [0.5, 1);
 * x is itself a power of two exactly when f == 0.5. */
float ds41o_pow2_ceil(float x) {
    int e;
    float f = frexpf(x, &e);
    if (f == 0.5f) return x;
    return ldexpf(1.0f, e);
}

/* f32_to_e4m3_rne / e4m3_to_f32 (named in [compress], imported from the
 * engram module, bodies not printed).  Reading: OCP FP8 E4M3 ("fn"): bias 7,
 * three mantissa bits, subnormals with step 2^-9, largest finite 448, no
 * infinities, 0x7f / 0xff are NaN.  Rounding is to nearest, ties to even, and
 * values beyond 448 saturate to 448.
 *
 * Method: inside one binade [2^E, 2^(E+1)) the representable values are
 * multiples of 2^(E-3); below 2^-6 they are multiples of 2^-9.  Divide by that
 * step (exact, a power of two), round to the nearest integer with ties to
 * even, and rebuild the code from exponent and integer. */
uint8_t ds41o_f32_to_e4m3_rne(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    float a = fabsf(x);
    if (isnan(x)) return (uint8_t)(sign | 0x7f);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7e); /* saturate */
    if (a < 0.015625f) {                            /* below 2^-6: subnormal step 2^-9 */
        float q = nearbyintf(a * 512.0f);           /* exact scaling, RNE */
        return (uint8_t)(sign | (uint8_t)q);        /* q == 8 is the code of 2^-6 */
    }
    int e;
    (void)frexpf(a, &e);      /* a = f * 2^e, f in [0.5,1): binade exponent e-1 */
    int eb = e - 1;           /* a in [2^eb, 2^(eb+1)) */
    float step = ldexpf(1.0f, eb - 3);
    float q = nearbyintf(a / step); /* in [8, 16] */
    if (q == 16.0f) { eb += 1; q = 8.0f; }
    int field = eb + 7;       /* biased exponent, 1..15 */
    uint8_t code = (uint8_t)((field << 3) | ((int)q - 8));
    if (code > 0x7e) code = 0x7e; /* beyond 448 after rounding: saturate */
    return (uint8_t)(sign | code);
}

float ds41o_e4m3_to_f32(uint8_t c) {
    int field = (c >> 3) & 15, man = c & 7;
    float v;
    if (field == 15 && man == 7) return NAN;
    if (field == 0) v = ldexpf((float)man, -9);
    else v = ldexpf((float)(8 + man), field - 10);
    return (c & 0x80) ? -v : v;
}

/* ------------------------------------------------------------------------- */
/* Block quantisers: [compress], fp4_quant_e8m0_inplace and                  */
/* fp4_quant_e4m3_inplace.                                                    */
/* x holds f32 values, rewritten in place with the dequantised, bf16-rounded  */
/* result.  codes (nullable) receives the 4-bit e2m1 codes, two per byte, the */
/* even element in the low nibble; scales (nullable) one byte per block: the  */
/* biased exponent (e8m0) or the e4m3 code.                                   */
/* ------------------------------------------------------------------------- */
static void quant_block_elems(float* blk, int64_t block, float s, uint8_t* codes, int64_t first) {
    for (int64_t i = 0; i < block; i++) {
        float t = blk[i] / s;                    /* IEEE f32 division */
        if (t < -FP4_MAX) t = -FP4_MAX;          /* clamp to the grid's range */
        if (t > FP4_MAX) t = FP4_MAX;
        float g = ds41o_to_e2m1_rne(t);
        float p = g * s;                         /* exact: <= 6 significant bits */
        if (codes) {
            int64_t j = first + i;
            uint8_t c = e2m1_code(t);
            if (j % 2 == 0) codes[j / 2] = (uint8_t)((codes[j / 2] & 0xf0) | c);
            else codes[j / 2] = (uint8_t)((codes[j / 2] & 0x0f) | (c << 4));
        }
        blk[i] = bf16_round(p);
    }
}

static float block_amax(const float* blk, int64_t block) {
    float m = 0.0f;
    for (int64_t i = 0; i < block; i++) {
        float a = fabsf(blk[i]);
        if (a > m) m = a;
    }
    return m;
}

void ds41o_fp4_quant_e8m0(float* x, int64_t n, int64_t block, uint8_t* codes, uint8_t* scales) {
    const float floor_amax = ldexpf(6.0f, -126);
    for (int64_t b = 0; b * block < n; b++) {
        float* blk = x + b * block;
        float amax = block_amax(blk, block);
        if (amax < floor_amax) amax = floor_amax;
        float s = ds41o_pow2_ceil(amax / FP4_MAX);
        if (scales) {
            int e;
            (void)frexpf(s, &e);                  /* s = 0.5 * 2^e = 2^(e-1) */
            scales[b] = (uint8_t)(e - 1 + 127);
        }
        quant_block_elems(blk, block, s, codes, b * block);
    }
}

void ds41o_fp4_quant_e4m3(float* x, int64_t n, int64_t block, uint8_t* codes, uint8_t* scales) {
    const float floor_amax = ldexpf(6.0f, -9);
    for (int64_t b = 0; b * block < n; b++) {
        float* blk = x + b * block;
        float amax = block_amax(blk, block);
        if (amax < floor_amax) amax = floor_amax;
        uint8_t sc = ds41o_f32_to_e4m3_rne(amax / FP4_MAX);
        float s = ds41o_e4m3_to_f32(sc);
        if (scales) scales[b] = sc;
        quant_block_elems(blk, block, s, codes, b * block);
    }
}

/* bf16 in, bf16 out wrappers of the two quantisers (rows x cols, row-major;
 * blocks run along each row). */
void ds41o_fp4_quant_bf16(const uint16_t* x, uint16_t* y, uint8_t* codes, uint8_t* scales,
                          int64_t rows, int64_t cols, int64_t block, int e4m3) {
    float* buf = (float*)malloc(sizeof(float) * (size_t)cols);
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t c = 0; c < cols; c++) buf[c] = ds41o_bf16_to_f32(x[r * cols + c]);
        uint8_t* cr = codes ? codes + r * (cols / 2) : NULL;
        uint8_t* sr = scales ? scales + r * (cols / block) : NULL;
        if (e4m3) ds41o_fp4_quant_e4m3(buf, cols, block, cr, sr);
        else ds41o_fp4_quant_e8m0(buf, cols, block, cr, sr);
        for (int64_t c = 0; c < cols; c++) y[r * cols + c] = ds41o_f32_to_bf16_rne(buf[c]);
    }
    free(buf);
}

/* ------------------------------------------------------------------------- */
/* RoPE table: [compress], yarn_freqs_cis.  out is [seqlen][dim/2][2] with    */
/* (cos, sin).  f32 where the page computes in f32, f64 for the correction    */
/* range, as the page does.                                                   */
/* ------------------------------------------------------------------------- */
static double yarn_corr(double rot, int64_t dim, int64_t orig, float base) {
    const double two_pi = 6.283185307179586476925286766559;
    return (double)dim * log((double)orig / (rot * two_pi)) / (2.0 * log((double)base));
}

void ds41o_yarn_inv_freqs(int64_t dim, int64_t orig, float base, float factor, float beta_fast,
                          float beta_slow, float* freqs /* [dim/2] */) {
    int64_t half = dim / 2;
    double lo_d = floor(yarn_corr((double)beta_fast, dim, orig, base));
    if (lo_d < 0.0) lo_d = 0.0;
    double hi_d = ceil(yarn_corr((double)beta_slow, dim, orig, base));
    if (hi_d > (double)(dim - 1)) hi_d = (double)(dim - 1);
    float lo = (float)lo_d, hi = (float)hi_d;
    float span = hi - lo;
    if (span < 1e-3f) span = 1e-3f;
    for (int64_t k = 0; k < half; k++) {
        float ex = (float)(2 * k) / (float)dim;
        float f = 1.0f / powf(base, ex);
        float ramp = ((float)k - lo) / span;
        if (ramp < 0.0f) ramp = 0.0f;
        if (ramp > 1.0f) ramp = 1.0f;
        float keep = 1.0f - ramp;               /* weight of the unscaled frequency */
        float scaled = f / factor;
        float a = scaled * (1.0f - keep);
        float b = f * keep;
        freqs[k] = a + b;
    }
}

void ds41o_yarn_freqs_cis(int64_t dim, int64_t seqlen, int64_t orig, float base, float factor,
                          float beta_fast, float beta_slow, float* out) {
    int64_t half = dim / 2;
    float* f = (float*)malloc(sizeof(float) * (size_t)half);
    ds41o_yarn_inv_freqs(dim, orig, base, factor, beta_fast, beta_slow, f);
    for (int64_t p = 0; p < seqlen; p++) {
        for (int64_t k = 0; k < half; k++) {
            float ang = (float)p * f[k];
            out[(p * half + k) * 2 + 0] = cosf(ang);
            out[(p * half + k) * 2 + 1] = sinf(ang);
        }
    }
    free(f);
}

/* apply_rotary (named in [compress], body not printed).  Reading: the last rd
 * dims of each hd-wide row are the rotary part; dims (2i, 2i+1) of that part
 * form a pair rotated by table column i of the row's position:
 *   y0 = x0*c - x1*s,  y1 = x0*s + x1*c   (each product rounded, then the sum);
 * the inverse rotation uses -s.  buf holds f32 values, rows x hd. */
void ds41o_apply_rotary(float* buf, int64_t rows, int64_t hd, int64_t rd, const int64_t* pos,
                        const float* fc, int inverse) {
    int64_t half = rd / 2;
    for (int64_t r = 0; r < rows; r++) {
        float* x = buf + r * hd + (hd - rd);
        const float* tab = fc + pos[r] * half * 2;
        for (int64_t i = 0; i < half; i++) {
            float c = tab[2 * i], s = tab[2 * i + 1];
            if (inverse) s = -s;
            float x0 = x[2 * i], x1 = x[2 * i + 1];
            float p00 = x0 * c, p11 = x1 * s, p01 = x0 * s, p10 = x1 * c;
            x[2 * i] = p00 - p11;
            x[2 * i + 1] = p01 + p10;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Window ring and window indices: [forward] "the window ring" block and     */
/* [compress] attention_any's ring update; window_topk_idxs is named there    */
/* but not printed.                                                           */
/*                                                                            */
/* Invariant of the printed ring updates: the row of position q sits in slot  */
/* q mod win.  rows_a, the rows the window indices point into, is             */
/*   start_pos == 0         : the m fresh rows (index = position);            */
/*   start_pos > 0, m == 1  : the ring after the write (index = q mod win);   */
/*   start_pos > 0, m > 1   : the ring as it was before the chunk, then the m */
/*                            fresh rows: q < start_pos -> q mod win,         */
/*                            q >= start_pos -> win + (q - start_pos).        */
/* (The pages print only the first two cases; the third is the reading that   */
/* reduces to both.)  A query at position p sees positions p-win+1 .. p that  */
/* are >= 0; the others are -1.                                               */
/* ------------------------------------------------------------------------- */
int64_t ds41o_rows_a_len(int64_t m, int64_t win, int64_t start_pos) {
    if (start_pos == 0) return m;
    if (m == 1) return win;
    return win + m;
}

void ds41o_window_ring_write(const uint16_t* kv, uint16_t* ring, uint16_t* rows_a, int64_t m,
                             int64_t hd, int64_t win, int64_t start_pos) {
    int64_t n_a = ds41o_rows_a_len(m, win, start_pos);
    if (rows_a && start_pos > 0 && m > 1) {
        memcpy(rows_a, ring, sizeof(uint16_t) * (size_t)(win * hd));
        memcpy(rows_a + win * hd, kv, sizeof(uint16_t) * (size_t)(m * hd));
    }
    /* Write positions in order, so a later position overwrites an earlier one
     * that maps to the same slot: the ring ends up holding the newest row of
     * every slot. */
    for (int64_t t = 0; t < m; t++) {
        int64_t q = start_pos + t;
        memcpy(ring + (q % win) * hd, kv + t * hd, sizeof(uint16_t) * (size_t)hd);
    }
    if (rows_a && start_pos == 0) memcpy(rows_a, kv, sizeof(uint16_t) * (size_t)(m * hd));
    if (rows_a && start_pos > 0 && m == 1) memcpy(rows_a, ring, sizeof(uint16_t) * (size_t)(n_a * hd));
}

void ds41o_window_topk_idxs(int64_t win, int64_t m, int64_t start_pos, int32_t* idx) {
    for (int64_t t = 0; t < m; t++) {
        int64_t p = start_pos + t;
        for (int64_t j = 0; j < win; j++) {
            int64_t q = p - win + 1 + j;
            int32_t v;
            if (q < 0) v = -1;
            else if (start_pos == 0) v = (int32_t)q;
            else if (m == 1) v = (int32_t)(q % win);
            else if (q < start_pos) v = (int32_t)(q % win);
            else v = (int32_t)(win + (q - start_pos));
            idx[t * win + j] = v;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Compressed latent write: [forward] "if let Some(groups) = latent_groups"   */
/* and [compress] attention_any's latent branch.  Group g of this call is the */
/* compressed row start_pos/r + g, built from positions                        */
/* (start_pos/r + g)*r .. +r-1; its RoPE position is the first of them        */
/* (g*r at start_pos 0, start_pos+1-r for the one decode group).  The row is  */
/* rotated, rounded to bf16, sent through the e4m3 fp4 round trip (block 16)  */
/* and stored.                                                                 */
/* ------------------------------------------------------------------------- */
/* compress_len ([forward] AttnV41::forward, [compress] attention_any): the  */
/* compressed rows that exist once positions 0 .. start_pos+m-1 are in, one   */
/* per complete group of ratio positions.                                     */
int64_t ds41o_compress_len(int64_t m, int64_t ratio, int64_t start_pos) {
    return (start_pos + m) / ratio;
}

/* Groups this call completes: those past the start_pos/ratio rows that were  */
/* complete before it (the cache row the latent copy starts at).              */
int64_t ds41o_new_groups(int64_t m, int64_t ratio, int64_t start_pos) {
    return ds41o_compress_len(m, ratio, start_pos) - start_pos / ratio;
}

/* Length of a merged index row: the win window indices, then                */
/* ctopk = min(topk, compress_len) compressed picks (0 when no compressed row */
/* exists yet, when the pages skip the indexer).                             */
/* scale = head_dim^-0.5 as [compress] attention_any computes it: an f32 pow. */
float ds41o_attn_scale(int64_t hd) { return powf((float)hd, -0.5f); }

int64_t ds41o_merged_len(int64_t win, int64_t topk, int64_t n_c) {
    int64_t ctopk = (n_c == 0) ? 0 : (topk < n_c ? topk : n_c);
    return win + ctopk;
}

void ds41o_compress_latent_write(const uint16_t* latent, const float* fc, uint16_t* cache,
                                 uint8_t* cache_codes, uint8_t* cache_scales, int64_t G,
                                 int64_t hd, int64_t rd, int64_t ratio, int64_t start_pos) {
    float* row = (float*)malloc(sizeof(float) * (size_t)hd);
    for (int64_t g = 0; g < G; g++) {
        int64_t crow = start_pos / ratio + g;
        int64_t lpos = crow * ratio;
        for (int64_t d = 0; d < hd; d++) row[d] = ds41o_bf16_to_f32(latent[g * hd + d]);
        ds41o_apply_rotary(row, 1, hd, rd, &lpos, fc, 0);
        for (int64_t d = 0; d < hd; d++) row[d] = bf16_round(row[d]);
        uint8_t* cr = cache_codes ? cache_codes + crow * (hd / 2) : NULL;
        uint8_t* sr = cache_scales ? cache_scales + crow * (hd / 16) : NULL;
        if (cr) memset(cr, 0, (size_t)(hd / 2));
        ds41o_fp4_quant_e4m3(row, hd, 16, cr, sr);
        for (int64_t d = 0; d < hd; d++) cache[crow * hd + d] = ds41o_f32_to_bf16_rne(row[d]);
    }
    free(row);
}

/* ------------------------------------------------------------------------- */
/* Indexer scores.  [compress] names the indexer but does not print it; its   */
/* header fixes the precision: q and k take the e2m1 round trip with          */
/* power-of-two scales per block of 32, and the scores are bf16.  Reading:    */
/*   qh = Q8(q_idx[t,h,:]),  kh = Q8(k_idx[s,:])                              */
/*   dot(t,h,s) = sum_d qh[d]*kh[d]      (f32, d ascending)                   */
/*   acc = 0; for h = 0..Hi-1: acc = fma(w[t,h], max(dot,0), acc)             */
/*   score(t,s) = bf16(acc), -0 written as +0                                 */
/* for the rows the query can see, s < (start_pos+t+1)/ratio; the others hold */
/* -inf.  acc32 (nullable) receives the f32 head sum before the bf16 rounding */
/* (0 for hidden rows).  Returns how many dots differ from the same sum taken */
/* in f64 (the dot is exact for the configs' inputs, which makes its order    */
/* irrelevant).                                                               */
/* ------------------------------------------------------------------------- */
int64_t ds41o_visible_rows(int64_t t, int64_t start_pos, int64_t ratio, int64_t n_c) {
    int64_t v = (start_pos + t + 1) / ratio;
    return v < n_c ? v : n_c;
}

int64_t ds41o_indexer_scores(const uint16_t* q_idx, const uint16_t* k_idx, const float* w,
                             uint16_t* scores, float* acc32, int64_t m, int64_t Hi, int64_t Di,
                             int64_t n_c,
                             int64_t ratio, int64_t start_pos, const int64_t* tokens,
                             int64_t n_tokens) {
    /* quantise every key row once */
    float* kq = (float*)malloc(sizeof(float) * (size_t)(n_c * Di));
    for (int64_t i = 0; i < n_c * Di; i++) kq[i] = ds41o_bf16_to_f32(k_idx[i]);
    for (int64_t s = 0; s < n_c; s++) ds41o_fp4_quant_e8m0(kq + s * Di, Di, 32, NULL, NULL);
    int64_t inexact = 0;
    #pragma omp parallel for schedule(dynamic, 1) reduction(+ : inexact)
    for (int64_t ti = 0; ti < n_tokens; ti++) {
        int64_t t = tokens[ti];
        float* qq = (float*)malloc(sizeof(float) * (size_t)(Hi * Di));
        for (int64_t i = 0; i < Hi * Di; i++) qq[i] = ds41o_bf16_to_f32(q_idx[t * Hi * Di + i]);
        for (int64_t h = 0; h < Hi; h++) ds41o_fp4_quant_e8m0(qq + h * Di, Di, 32, NULL, NULL);
        int64_t vis = ds41o_visible_rows(t, start_pos, ratio, n_c);
        for (int64_t s = 0; s < n_c; s++) {
            uint16_t out;
            float accv = 0.0f;
            if (s >= vis) {
                out = 0xff80u; /* -inf */
            } else {
                float acc = 0.0f;
                for (int64_t h = 0; h < Hi; h++) {
                    float d32 = 0.0f;
                    double d64 = 0.0;
                    for (int64_t d = 0; d < Di; d++) {
                        float pr = qq[h * Di + d] * kq[s * Di + d];
                        d32 = d32 + pr;
                        d64 += (double)qq[h * Di + d] * (double)kq[s * Di + d];
                    }
                    if ((double)d32 != d64) inexact++;
                    float r = d32 > 0.0f ? d32 : 0.0f;
                    acc = fmaf(w[t * Hi + h], r, acc);
                }
                out = ds41o_f32_to_bf16_rne(acc);
                if (out == 0x8000u) out = 0x0000u;
                accv = acc;
            }
            scores[ti * n_c + s] = out;
            if (acc32) acc32[ti * n_c + s] = accv;
        }
        free(qq);
    }
    free(kq);
    return inexact;
}

/* ------------------------------------------------------------------------- */
/* Per-query top-k and merge.  [forward] / [compress]: the indexer returns    */
/* ctopk row numbers per query, already offset by the rows_a length, and the  */
/* merged index row of a query is its window indices followed by them.        */
/* Reading: the top min(topk, visible) visible rows by score, ties to the     */
/* lower row, padded with -1 to ctopk = min(topk, n_c) entries.               */
/* ------------------------------------------------------------------------- */
typedef struct { float v; int64_t s; } key_t_;

static int key_cmp(const void* a, const void* b) {
    const key_t_* x = (const key_t_*)a;
    const key_t_* y = (const key_t_*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->s < y->s) ? -1 : (x->s > y->s);
}

void ds41o_topk_merge(const uint16_t* scores, const int32_t* win_idx, int32_t* idx, int64_t n_tokens,
                      const int64_t* tokens, int64_t n_c, int64_t win, int64_t ratio,
                      int64_t start_pos, int64_t topk, int64_t offset) {
    int64_t ctopk = (n_c == 0) ? 0 : (topk < n_c ? topk : n_c);
    int64_t K = win + ctopk;
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t ti = 0; ti < n_tokens; ti++) {
        int64_t t = tokens[ti];
        int32_t* row = idx + ti * K;
        memcpy(row, win_idx + ti * win, sizeof(int32_t) * (size_t)win);
        int64_t vis = ds41o_visible_rows(t, start_pos, ratio, n_c);
        key_t_* keys = (key_t_*)malloc(sizeof(key_t_) * (size_t)(vis > 0 ? vis : 1));
        for (int64_t s = 0; s < vis; s++) {
            keys[s].v = ds41o_bf16_to_f32(scores[ti * n_c + s]);
            keys[s].s = s;
        }
        qsort(keys, (size_t)vis, sizeof(key_t_), key_cmp);
        for (int64_t j = 0; j < ctopk; j++)
            row[win + j] = (j < vis) ? (int32_t)(offset + keys[j].s) : -1;
        free(keys);
    }
}

/* ------------------------------------------------------------------------- */
/* Sparse attention with a per-head sink.  [compress] attention_any calls     */
/* sparse_attn(q, kv_rows, sink, idx, ...) with scale = head_dim^-0.5; its    */
/* body is not printed.  Reading: one row per position serves as key and      */
/* value; for query t, head h, over the valid indices i of row t              */
/*   s_i = scale * <q[t,h,:], row_i>                                          */
/*   o   = sum_i e^{s_i} row_i / (e^{sink_h} + sum_i e^{s_i})                 */
/* (the sink enters the denominator only).  Index v < n_a names rows_a[v],    */
/* n_a <= v < n_a + n_c names rows_b[v - n_a]; -1 is padding.  Everything is  */
/* accumulated in f64.  o and lse are [n_tokens, nh, hd] and [n_tokens, nh]. */
/* Returns the number of out-of-range indices seen (they are skipped).        */
/* ------------------------------------------------------------------------- */
int64_t ds41o_sparse_attn(const uint16_t* q, const uint16_t* rows_a, int64_t n_a,
                          const uint16_t* rows_b, int64_t n_c, const int32_t* idx, int64_t K,
                          const float* sink, float scale, double* o, double* lse, int64_t nh,
                          int64_t hd, const int64_t* tokens, int64_t n_tokens) {
    int64_t bad = 0;
    #pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t ti = 0; ti < n_tokens; ti++) {
        for (int64_t h = 0; h < nh; h++) {
            int64_t t = tokens[ti];
            const uint16_t* qv = q + (t * nh + h) * hd;
            const int32_t* ir = idx + ti * K;
            double* s = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
            const uint16_t** rp = (const uint16_t**)malloc(sizeof(void*) * (size_t)(K > 0 ? K : 1));
            double mx = (double)sink[h];
            for (int64_t i = 0; i < K; i++) {
                int64_t v = ir[i];
                rp[i] = NULL;
                if (v < 0) continue;
                if (v < n_a) rp[i] = rows_a + v * hd;
                else if (v < n_a + n_c) rp[i] = rows_b + (v - n_a) * hd;
                else { bad++; continue; }
                double acc = 0.0;
                for (int64_t d = 0; d < hd; d++)
                    acc += (double)ds41o_bf16_to_f32(qv[d]) * (double)ds41o_bf16_to_f32(rp[i][d]);
                s[i] = (double)scale * acc;
                if (s[i] > mx) mx = s[i];
            }
            double den = exp((double)sink[h] - mx);
            double* ov = o + (ti * nh + h) * hd;
            for (int64_t d = 0; d < hd; d++) ov[d] = 0.0;
            for (int64_t i = 0; i < K; i++) {
                if (!rp[i]) continue;
                double e = exp(s[i] - mx);
                den += e;
                for (int64_t d = 0; d < hd; d++) ov[d] += e * (double)ds41o_bf16_to_f32(rp[i][d]);
            }
            for (int64_t d = 0; d < hd; d++) ov[d] = (den > 0.0) ? ov[d] / den : 0.0;
            if (lse) lse[ti * nh + h] = mx + log(den);
            free(s);
            free(rp);
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Output side of the layer.  [compress] attention_any, after sparse_attn:    */
/* o is rotated back (apply_rotary with inverse = true at each head's token   */
/* position), split into `groups` groups of gw = nh*hd/groups values, and     */
/* each group is projected by its own o_rank rows of wo_a, every result       */
/* rounded to bf16 (to_bf16_rne); the groups*o_rank values then go through    */
/* linear_bf16 with wo_b, [dim, groups*o_rank].  linear_bf16's body is not    */
/* printed: reading, out = og . wo_b^T with no rounding of the result.        */
/* Here the dot products are accumulated in f64; og is rounded to f32 and     */
/* then to bf16 (the pages round an f32 sum).  o is the attention output as   */
/* given ([n_tokens][nh*hd] bf16 bits, token tokens[i] at position            */
/* start_pos + tokens[i]); og is [n_tokens][groups*o_rank] bf16 bits and out  */
/* [n_tokens][dim].                                                           */
/* ------------------------------------------------------------------------- */
void ds41o_attn_out_proj(const uint16_t* o, const float* fc, const uint16_t* wo_a,
                         const uint16_t* wo_b, uint16_t* og, double* out, int64_t nh, int64_t hd,
                         int64_t rd, int64_t groups, int64_t o_rank, int64_t dim,
                         int64_t start_pos, const int64_t* tokens, int64_t n_tokens) {
    const int64_t gw = nh * hd / groups, gr = groups * o_rank;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ti = 0; ti < n_tokens; ti++) {
        const int64_t t = tokens[ti];
        float* x = (float*)malloc(sizeof(float) * (size_t)(nh * hd));
        int64_t* hp = (int64_t*)malloc(sizeof(int64_t) * (size_t)nh);
        for (int64_t i = 0; i < nh * hd; i++) x[i] = ds41o_bf16_to_f32(o[t * nh * hd + i]);
        for (int64_t h = 0; h < nh; h++) hp[h] = start_pos + t;
        ds41o_apply_rotary(x, nh, hd, rd, hp, fc, 1);
        uint16_t* gv = og + ti * gr;
        for (int64_t g = 0; g < groups; g++) {
            const float* xg = x + g * gw;
            for (int64_t r = 0; r < o_rank; r++) {
                const uint16_t* wr = wo_a + (g * o_rank + r) * gw;
                double acc = 0.0;
                for (int64_t i = 0; i < gw; i++) acc += (double)xg[i] * (double)ds41o_bf16_to_f32(wr[i]);
                gv[g * o_rank + r] = ds41o_f32_to_bf16_rne((float)acc);
            }
        }
        for (int64_t j = 0; j < dim; j++) {
            const uint16_t* wr = wo_b + j * gr;
            double acc = 0.0;
            for (int64_t k = 0; k < gr; k++)
                acc += (double)ds41o_bf16_to_f32(gv[k]) * (double)ds41o_bf16_to_f32(wr[k]);
            out[ti * dim + j] = acc;
        }
        free(x);
        free(hp);
    }
}

/* Number of threads OpenMP will use (1 without OpenMP). */
int ds41o_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ds41o_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Elementwise array forms of the scalar codecs (used by the exhaustive pins). */
void ds41o_to_e2m1_rne_array(const float* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = ds41o_to_e2m1_rne(in[i]);
}
void ds41o_f32_to_bf16_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = ds41o_f32_to_bf16_rne(in[i]);
}
void ds41o_f32_to_e4m3_array(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = ds41o_f32_to_e4m3_rne(in[i]);
}
void ds41o_e4m3_to_f32_array(const uint8_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = ds41o_e4m3_to_f32(in[i]);
}
void ds41o_pow2_ceil_array(const float* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = ds41o_pow2_ceil(in[i]);
}
