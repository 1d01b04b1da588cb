/*
 * CPU oracle for the BitNet b1.58 BitLinear hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library; both sides implement the same written
 * definitions independently.
 *
 * Plain, slow, obviously correct.  Each function cites the passage of the
 * source pages it follows.  Pages (by title):
 *   [P1] asi.tokyo, "マイクロソフトが偶然に作った史上最も効率的なAI" (2025-04-27),
 *        on BitNet B1.58 2B4T (no section headings: passages are named by
 *        their subject, e.g. the paragraph on running the model on a GPU)
 *   [P2] cheatsheet.md, "1ビットLarge Language Models時代：マイクロソフトがBitNet b1.58を紹介"
 *   [P3] lumen-it.ai, BitNet (original 1-bit BitNet) article
 *   [P4] vi.news.hada.io topic 20406 (and its Portuguese twin), comments
 *        on ternary packing: five ternary digits per byte, 3^5 = 243 <= 256
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fopenmp
 * (no -ffast-math: every float operation below must be one IEEE-754
 * correctly rounded operation, in the order written).
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32 (bit level)                                           */
/* ------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest-even fp32 -> bf16 (NaN kept quiet). */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

uint16_t bl_oracle_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

/* ------------------------------------------------------------------ */
/* Step 1: absmean scale gamma = mean |W|.                             */
/* [P2] section "BitNet b1.58とは？": weights are scaled by their mean   */
/* absolute value, then rounded to the nearest integer in {-1,0,+1}.   */
/* [P1]: the "absmean quantiser" picks the chip for every weight.      */
/*                                                                      */
/* The sum S = sum |W| is computed exactly with Shewchuk's adaptive     */
/* non-overlapping partials (Shewchuk 1997, "Adaptive precision         */
/* floating-point arithmetic"), the method behind Python's math.fsum,  */
/* and rounded once to double.  gamma = (float)(S_double / (N*K)).     */
/* ------------------------------------------------------------------ */

/* Exact sum of |w[i]| rounded once to the nearest double (ties to even). */
double bl_oracle_sum_abs(const float *w, int64_t n) {
    int cap = 64, np = 0;
    double *p = (double *)malloc(sizeof(double) * cap);
    for (int64_t i = 0; i < n; ++i) {
        double x = fabs((double)w[i]);
        int j = 0;
        for (int k = 0; k < np; ++k) {
            double y = p[k];
            if (fabs(x) < fabs(y)) { double t = x; x = y; y = t; }
            double hi = x + y;
            double lo = y - (hi - x);      /* exact error of hi (|x|>=|y|) */
            if (lo != 0.0) p[j++] = lo;
            x = hi;
        }
        if (j >= cap) { cap *= 2; p = (double *)realloc(p, sizeof(double) * cap); }
        p[j++] = x;
        np = j;
    }
    /* The partials are non-overlapping and increasing in magnitude; their
     * exact sum is the true sum.  Round it once to double: add from the
     * top until the first inexact addition, then correct the half-way
     * case using the sign of the remaining partials. */
    double hi = 0.0;
    if (np > 0) {
        int k = np - 1;
        hi = p[k];
        double lo = 0.0;
        while (k > 0) {
            double x = hi;
            double y = p[--k];
            hi = x + y;
            double yr = hi - x;
            lo = y - yr;
            if (lo != 0.0) break;
        }
        if (k > 0 && ((lo < 0.0 && p[k - 1] < 0.0) || (lo > 0.0 && p[k - 1] > 0.0))) {
            double y = lo * 2.0;
            double x = hi + y;
            double yr = x - hi;
            if (y == yr) hi = x;
        }
    }
    free(p);
    return hi;
}

/* gamma = mean|W| over the whole tensor (per-tensor scale). */
float bl_oracle_gamma(const float *w, int64_t N, int64_t K) {
    double s = bl_oracle_sum_abs(w, N * K);
    double m = s / (double)(N * K);
    return (float)m;
}

/* ------------------------------------------------------------------ */
/* Step 2: ternarise.  [P2] "BitNet b1.58とは？": divide by the mean    */
/* absolute value and round to the nearest integer, constrained to     */
/* {-1, 0, +1}.  Wq = clip(round(W / (gamma + eps)), -1, 1), computed   */
/* in fp32 (one rounded add, one rounded divide), round half to even.  */
/* ------------------------------------------------------------------ */
void bl_oracle_ternarize(const float *w, int64_t n, float gamma, float eps, int8_t *wq) {
    float d = gamma + eps;                 /* fp32 add, rounded once */
    for (int64_t i = 0; i < n; ++i) {
        float t = w[i] / d;                /* fp32 divide, rounded once */
        float r = rintf(t);                /* nearest, ties to even */
        int v = (r > 1.0f) ? 1 : (r < -1.0f) ? -1 : (int)r;
        wq[i] = (int8_t)v;
    }
}

/* ------------------------------------------------------------------ */
/* Step 3: pack four ternary weights per byte.  [P1]: the custom kernel */
/* packs four chips into one byte and unpacks them next to the math     */
/* units.  Code = Wq + 1 (00 = -1, 01 = 0, 10 = +1, 11 invalid).        */
/*                                                                      */
/* Layout (tiles of 16 rows x 128 k, 512 bytes each):                   */
/*   Np = 16*ceil(N/16), Kp = 128*ceil(K/128), KT = Kp/128              */
/*   r = n/16, i = n%16, c = k/128, kk = k%128                          */
/*   g = i%8, u = i/8              (row g+8u of the row group)          */
/*   t = kk/32, j = kk%32          (lane 4g+t owns k in [32t, 32t+32))  */
/*   P = j/16, m = (j%16)/4, sb = (j%4)/2, h = j%2                      */
/*   p = 2m + sb                   (bit pair inside a 16-bit half)      */
/*   lane = 4g + t, word = 2P + u, bit = 16h + 2p                       */
/*   byte = 512*(r*KT + c) + 16*lane + 4*word + bit/8, shift = bit%8    */
/* Positions with n >= N or k >= K hold code 01 (weight 0).             */
/* ------------------------------------------------------------------ */
int64_t bl_oracle_packed_bytes(int64_t N, int64_t K) {
    int64_t Np = (N + 15) / 16 * 16;
    int64_t Kp = (K + 127) / 128 * 128;
    return Np * Kp / 4;
}

static void position(int64_t n, int64_t k, int64_t KT, int64_t *byte, int *shift) {
    int64_t r = n / 16, c = k / 128;
    int i = (int)(n % 16), kk = (int)(k % 128);
    int g = i % 8, u = i / 8;
    int t = kk / 32, j = kk % 32;
    int P = j / 16, m = (j % 16) / 4, sb = (j % 4) / 2, h = j % 2;
    int p = 2 * m + sb;
    int lane = 4 * g + t, word = 2 * P + u, bit = 16 * h + 2 * p;
    *byte = 512 * (r * KT + c) + 16 * lane + 4 * word + bit / 8;
    *shift = bit % 8;
}

/* Byte offset and bit shift of weight (n, k); exported for the tests. */
void bl_oracle_position(int64_t n, int64_t k, int64_t K, int64_t *byte, int *shift) {
    position(n, k, (K + 127) / 128, byte, shift);
}

void bl_oracle_pack(const int8_t *wq, int64_t N, int64_t K, uint8_t *packed) {
    int64_t Np = (N + 15) / 16 * 16, Kp = (K + 127) / 128 * 128, KT = Kp / 128;
    memset(packed, 0, (size_t)(Np * Kp / 4));
    for (int64_t n = 0; n < Np; ++n)
        for (int64_t k = 0; k < Kp; ++k) {
            int code = (n < N && k < K) ? wq[n * K + k] + 1 : 1;
            int64_t byte; int shift;
            position(n, k, KT, &byte, &shift);
            packed[byte] |= (uint8_t)(code << shift);
        }
}

/* Inverse of bl_oracle_pack.  Returns the number of invalid codes (11)
 * plus the number of padding positions that do not hold code 01. */
int64_t bl_oracle_unpack(const uint8_t *packed, int64_t N, int64_t K, int8_t *wq) {
    int64_t Np = (N + 15) / 16 * 16, Kp = (K + 127) / 128 * 128, KT = Kp / 128;
    int64_t bad = 0;
    for (int64_t n = 0; n < Np; ++n)
        for (int64_t k = 0; k < Kp; ++k) {
            int64_t byte; int shift;
            position(n, k, KT, &byte, &shift);
            int code = (packed[byte] >> shift) & 3;
            if (code == 3) { ++bad; continue; }
            if (n < N && k < K) wq[n * K + k] = (int8_t)(code - 1);
            else if (code != 1) ++bad;
        }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Step 4: RMSNorm + per-token absmax int8.                             */
/* [P2] "BitNet b1.58とは？": activations are scaled per token into      */
/* [-Qb, Qb] (8 bit); the LLaMA parts include RMSNorm.  [P3]: absmax    */
/* quantisation of activations.  [P1]: 8-bit activations.              */
/*                                                                      */
/* Per token m, with v_k = x_k * g_k (fp32 product, exact for bf16):    */
/*   mx = max_k |v_k|  (clamped below at 1e-5)                          */
/*   c  = 127 / mx                    (fp32 divide)                     */
/*   q_k = clamp(rint(v_k * c), -128, 127)   (fp32 multiply)            */
/*   r  = 1 / sqrt(sum_k v_k^2 / K + eps)    (fp64)                     */
/*   s_tok = (float)(r * mx / 127)                                      */
/* RMSNorm's factor r > 0 cancels inside absmax, so q is computed from  */
/* v directly; s_tok carries r so that q * s_tok approximates the       */
/* normalised activation x * r * g.                                     */
/* ------------------------------------------------------------------ */
void bl_oracle_quant_act(const uint16_t *x, const uint16_t *gain, int64_t M, int64_t K,
                         float eps, int8_t *q, float *s_tok) {
    #pragma omp parallel for schedule(static)
    for (int64_t mi = 0; mi < M; ++mi) {
        const uint16_t *xr = x + mi * K;
        float mx = 0.0f;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            float v = bf16_to_f32(xr[k]);
            if (gain) v = v * bf16_to_f32(gain[k]);
            float a = fabsf(v);
            if (a > mx) mx = a;
            ss += (double)v * (double)v;
        }
        if (!(mx >= 1e-5f)) mx = 1e-5f;
        float c = 127.0f / mx;
        for (int64_t k = 0; k < K; ++k) {
            float v = bf16_to_f32(xr[k]);
            if (gain) v = v * bf16_to_f32(gain[k]);
            float y = v * c;
            float r = rintf(y);
            if (r > 127.0f) r = 127.0f;
            if (r < -128.0f) r = -128.0f;
            q[mi * K + k] = (int8_t)(int)r;
        }
        double rr = 1.0 / sqrt(ss / (double)K + (double)eps);
        s_tok[mi] = (float)(rr * (double)mx / 127.0);
    }
}

/* ------------------------------------------------------------------ */
/* Step 5: acc[m,n] = sum_k q[m,k] * Wq[n,k], exact.  [P1]: unpacked    */
/* weights are multiplied with the 8-bit blocks; [P2]: the matmul is    */
/* mostly additions.  Accumulated in int64; returns nonzero if a result */
/* does not fit int32.                                                  */
/* ------------------------------------------------------------------ */
int bl_oracle_matmul(const int8_t *q, const int8_t *wq, int64_t M, int64_t N, int64_t K,
                     int32_t *acc) {
    int overflow = 0;
    #pragma omp parallel for schedule(static) reduction(|:overflow)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t mi = 0; mi < M; ++mi) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)q[mi * K + k] * (int64_t)wq[n * K + k];
            if (s > INT32_MAX || s < INT32_MIN) overflow = 1;
            acc[mi * N + n] = (int32_t)s;
        }
    return overflow;
}

/* Same contraction for a list of (m, n) pairs only (for large shapes). */
void bl_oracle_matmul_pairs(const int8_t *q, const int8_t *wq, int64_t K, const int64_t *ms,
                            const int64_t *ns, int64_t cnt, int32_t *acc) {
    for (int64_t i = 0; i < cnt; ++i) {
        int64_t s = 0;
        for (int64_t k = 0; k < K; ++k) s += (int64_t)q[ms[i] * K + k] * (int64_t)wq[ns[i] * K + k];
        acc[i] = (int32_t)s;
    }
}

/* ------------------------------------------------------------------ */
/* Step 6: rescale.  The integer result is dequantised by the weight    */
/* scale gamma and the token scale s_tok:                               */
/*   f = gamma * s_tok[m]           (fp32 multiply)                     */
/*   out = bf16_rne((float)acc * f) (fp32 multiply, then RNE to bf16)   */
/* ------------------------------------------------------------------ */
void bl_oracle_epilogue(const int32_t *acc, const float *s_tok, float gamma, int64_t M,
                        int64_t N, uint16_t *out) {
    for (int64_t mi = 0; mi < M; ++mi) {
        float f = gamma * s_tok[mi];
        for (int64_t n = 0; n < N; ++n) {
            float y = (float)acc[mi * N + n] * f;
            out[mi * N + n] = f32_to_bf16_rne(y);
        }
    }
}

/* Sets the number of OpenMP threads of the parallel loops (timing of the
   single-threaded baseline); n <= 0 restores all cores. */
void bl_oracle_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}

/* Number of OpenMP threads the parallel loops above use. */
int bl_oracle_threads(void) {
    int t = 1;
    #pragma omp parallel
    {
        #pragma omp single
        {
#ifdef _OPENMP
            t = omp_get_num_threads();
#endif
        }
    }
    return t;
}

/* ------------------------------------------------------------------ */
/* Synthetic ternary weights by a counter-based generator (inputs, not */
/* the method).  The large stacked workloads draw their weights on the */
/* device, element by element, from SplitMix64 (Steele, Lea and Flood, */
/* "Fast splittable pseudorandom number generators", OOPSLA 2014): the */
/* i-th output (i = 0, 1, ...) of SplitMix64 seeded with s is          */
/* mix(s + (i+1)*0x9E3779B97F4A7C15).  A matrix keyed by `word` (its   */
/* workload seed, layer and projection) takes s = the first output of  */
/* SplitMix64 seeded with `word`; its element (n, k) is the output     */
/* i = n*K + k of SplitMix64 seeded with s, mapped to {-1, 0, +1} as   */
/* floor(hi32 * 3 / 2^32) - 1 (hi32: the output's upper 32 bits).      */
/* This implementation is written from that definition alone; the     */
/* device side has its own.                                            */
/* ------------------------------------------------------------------ */

static uint64_t splitmix_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* The first n outputs of SplitMix64 seeded with `seed`. */
void bl_oracle_splitmix64(uint64_t seed, int64_t n, uint64_t *out) {
    uint64_t x = seed;
    for (int64_t i = 0; i < n; ++i) {
        x += 0x9E3779B97F4A7C15ull;
        out[i] = splitmix_mix(x);
    }
}

/* Rows [n0, n1) of the [N, K] ternary matrix keyed by `word`, row-major. */
void bl_oracle_ternary_hash(uint64_t word, int64_t K, int64_t n0, int64_t n1, int8_t *out) {
    uint64_t s;
    bl_oracle_splitmix64(word, 1, &s);
    for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const uint64_t i = (uint64_t)n * (uint64_t)K + (uint64_t)k;
            const uint64_t v = splitmix_mix(s + (i + 1u) * 0x9E3779B97F4A7C15ull);
            out[(n - n0) * K + k] = (int8_t)((int)(((v >> 32) * 3u) >> 32) - 1);
        }
}

/* ------------------------------------------------------------------ */
/* Variant layout: five ternary digits per byte (1.6 bit per weight).   */
/* [P4], the Hacker News comments: five ternary digits fit one byte     */
/* because 3^5 = 243 <= 256, so b1.58 weights need log2(3) = 1.58 bits  */
/* rather than 2.  The pages give no digit order or byte encoding;     */
/* this reading: digits e = Wq + 1, most significant first,             */
/*   v = e0*81 + e1*27 + e2*9 + e3*3 + e4      (0 <= v <= 242)          */
/* and the byte holds v as a base-3 fraction scaled to 256,             */
/*   b = ceil(256 * v / 243),                                           */
/* the fixed-point form of the ternary-packing write-up the comment     */
/* links (its digits come back by repeated multiplication by 3).        */
/* Decoding here is plain arithmetic: v = floor(243 * b / 256), then   */
/* base-3 digits of v.                                                  */
/*                                                                      */
/* Layout (tiles of 16 rows x 160 k, 512 bytes each):                   */
/*   Np = 16*ceil(N/16), K5 = 160*ceil(K/160), KT5 = K5/160             */
/*   r = n/16, i = n%16, c = k/160, kk = k%160                          */
/*   g = i%8, u = i/8, t = kk/40, j = (kk%40)/5, d = kk%5               */
/*   byte = 512*(r*KT5 + c) + 16*(4g + t) + 8u + j, digit d of it       */
/* so lane 4g+t's 16 bytes hold rows g (bytes 0-7) and g+8 (8-15) over  */
/* k in [40t, 40t+40), five consecutive k per byte.  Padding positions  */
/* (n >= N or k >= K) hold digit 1 (weight 0).                          */
/* ------------------------------------------------------------------ */
int64_t bl_oracle_packed5_bytes(int64_t N, int64_t K) {
    int64_t Np = (N + 15) / 16 * 16;
    int64_t K5 = (K + 159) / 160 * 160;
    return Np * K5 / 5;
}

static void position5(int64_t n, int64_t k, int64_t KT5, int64_t *byte, int *digit) {
    int64_t r = n / 16, c = k / 160;
    int i = (int)(n % 16), kk = (int)(k % 160);
    int g = i % 8, u = i / 8, t = kk / 40, j = (kk % 40) / 5;
    *byte = 512 * (r * KT5 + c) + 16 * (4 * g + t) + 8 * u + j;
    *digit = kk % 5;
}

/* Byte offset and digit index (0 = most significant) of weight (n, k). */
void bl_oracle_position5(int64_t n, int64_t k, int64_t K, int64_t *byte, int *digit) {
    position5(n, k, (K + 159) / 160, byte, digit);
}

/* One byte from its five digits (each 0, 1 or 2). */
uint8_t bl_oracle_encode5(const int *e) {
    int v = 0;
    for (int d = 0; d < 5; ++d) v = 3 * v + e[d];
    return (uint8_t)((256 * v + 242) / 243);
}

/* The five digits of a byte; returns 0 if the byte is not an encoding. */
int bl_oracle_decode5(uint8_t b, int *e) {
    int v = (243 * (int)b) / 256;
    if ((256 * v + 242) / 243 != (int)b) return 0;
    for (int d = 4; d >= 0; --d) {
        e[d] = v % 3;
        v /= 3;
    }
    return 1;
}

void bl_oracle_pack5(const int8_t *wq, int64_t N, int64_t K, uint8_t *packed) {
    int64_t Np = (N + 15) / 16 * 16, K5 = (K + 159) / 160 * 160, KT5 = K5 / 160;
    for (int64_t n = 0; n < Np; ++n)
        for (int64_t k0 = 0; k0 < K5; k0 += 5) {
            int e[5];
            for (int d = 0; d < 5; ++d) {
                int64_t k = k0 + d;
                e[d] = (n < N && k < K) ? wq[n * K + k] + 1 : 1;
            }
            int64_t byte; int digit;
            position5(n, k0, KT5, &byte, &digit);
            packed[byte] = bl_oracle_encode5(e);
        }
}

/* Inverse of bl_oracle_pack5.  Returns the number of bytes that are not
 * encodings plus the number of padding digits that are not 1. */
int64_t bl_oracle_unpack5(const uint8_t *packed, int64_t N, int64_t K, int8_t *wq) {
    int64_t Np = (N + 15) / 16 * 16, K5 = (K + 159) / 160 * 160, KT5 = K5 / 160;
    int64_t bad = 0;
    for (int64_t n = 0; n < Np; ++n)
        for (int64_t k0 = 0; k0 < K5; k0 += 5) {
            int64_t byte; int digit;
            position5(n, k0, KT5, &byte, &digit);
            int e[5];
            if (!bl_oracle_decode5(packed[byte], e)) { ++bad; continue; }
            for (int d = 0; d < 5; ++d) {
                int64_t k = k0 + d;
                if (n < N && k < K) wq[n * K + k] = (int8_t)(e[d] - 1);
                else if (e[d] != 1) ++bad;
            }
        }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Variant: the original 1-bit BitNet.  [P3]: weights become binary     */
/* values (+1 or -1) through the signum function, activations are       */
/* absmax-quantised, and the weights are quantised and normalised in   */
/* groups (for model parallelism).  Readings (the page gives no more):  */
/*   - the groups are G equal blocks of consecutive output rows (the    */
/*     model-parallel split of a weight matrix), N % G == 0;            */
/*   - Wb = +1 where W > 0 and -1 elsewhere (a binary signum: zero has  */
/*     to go to one side; it goes to -1);                               */
/*   - each group's scale is its mean absolute weight,                  */
/*     beta_g = mean |W| over the group's rows (exact sum, rounded      */
/*     once, as gamma above), and the output is                         */
/*     bf16(acc * (beta_g * s_tok)), acc = sum_k Wb * q exact;          */
/*   - activations: the same per-token absmax int8 as above.            */
/* ------------------------------------------------------------------ */
void bl_oracle_beta(const float *w, int64_t N, int64_t K, int64_t G, float *beta) {
    int64_t rows = N / G;
    for (int64_t g = 0; g < G; ++g) {
        double s = bl_oracle_sum_abs(w + g * rows * K, rows * K);
        beta[g] = (float)(s / (double)(rows * K));
    }
}

void bl_oracle_binarize(const float *w, int64_t n, int8_t *wb) {
    for (int64_t i = 0; i < n; ++i) wb[i] = w[i] > 0.0f ? 1 : -1;
}

/* Packed binary layout (tiles of 16 rows x 256 k, 512 bytes each): one
 * bit per weight, 1 for +1 and 0 for -1.
 *   Np = 16*ceil(N/16), K1 = 256*ceil(K/256), KT1 = K1/256
 *   r = n/16, i = n%16, c = k/256, kk = k%256
 *   g = i%8, u = i/8, t = kk/64, j = kk%64
 *   P = j/32, s = (j%32)/4, sb = (j%4)/2, h = j%2, p = 2s + sb
 *   byte = 512*(r*KT1 + c) + 16*(4g + t) + 4*(2P + u) + (16h + p)/8,
 *   bit = (16h + p)%8
 * so lane 4g+t's 16 bytes hold rows g and g+8 over k in [64t, 64t+64),
 * one 32-bit word per (row, 32-k half).  Padding positions hold 0 (-1);
 * the matmul never reads them against a nonzero activation. */
int64_t bl_oracle_packed1_bytes(int64_t N, int64_t K) {
    int64_t Np = (N + 15) / 16 * 16;
    int64_t K1 = (K + 255) / 256 * 256;
    return Np * K1 / 8;
}

static void position1(int64_t n, int64_t k, int64_t KT1, int64_t *byte, int *bit) {
    int64_t r = n / 16, c = k / 256;
    int i = (int)(n % 16), kk = (int)(k % 256);
    int g = i % 8, u = i / 8, t = kk / 64, j = kk % 64;
    int P = j / 32, sidx = (j % 32) / 4, sb = (j % 4) / 2, h = j % 2;
    int p = 2 * sidx + sb, b = 16 * h + p;
    *byte = 512 * (r * KT1 + c) + 16 * (4 * g + t) + 4 * (2 * P + u) + b / 8;
    *bit = b % 8;
}

void bl_oracle_position1(int64_t n, int64_t k, int64_t K, int64_t *byte, int *bit) {
    position1(n, k, (K + 255) / 256, byte, bit);
}

void bl_oracle_pack1(const int8_t *wb, int64_t N, int64_t K, uint8_t *packed) {
    int64_t Np = (N + 15) / 16 * 16, K1 = (K + 255) / 256 * 256, KT1 = K1 / 256;
    memset(packed, 0, (size_t)(Np * K1 / 8));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            if (wb[n * K + k] > 0) {
                int64_t byte; int bit;
                position1(n, k, KT1, &byte, &bit);
                packed[byte] |= (uint8_t)(1u << bit);
            }
}

/* Inverse of bl_oracle_pack1 on [0, N) x [0, K); returns the number of set
 * padding bits. */
int64_t bl_oracle_unpack1(const uint8_t *packed, int64_t N, int64_t K, int8_t *wb) {
    int64_t Np = (N + 15) / 16 * 16, K1 = (K + 255) / 256 * 256, KT1 = K1 / 256;
    int64_t bad = 0;
    for (int64_t n = 0; n < Np; ++n)
        for (int64_t k = 0; k < K1; ++k) {
            int64_t byte; int bit;
            position1(n, k, KT1, &byte, &bit);
            int v = (packed[byte] >> bit) & 1;
            if (n < N && k < K) wb[n * K + k] = v ? 1 : -1;
            else if (v) ++bad;
        }
    return bad;
}

/* Rescale with one scale per group of N/G consecutive rows:
 *   f = beta[n / (N/G)] * s_tok[m], out = bf16_rne((float)acc * f). */
void bl_oracle_epilogue_groups(const int32_t *acc, const float *s_tok, const float *beta, int64_t G,
                               int64_t M, int64_t N, uint16_t *out) {
    int64_t rows = N / G;
    for (int64_t mi = 0; mi < M; ++mi)
        for (int64_t n = 0; n < N; ++n) {
            float f = beta[n / rows] * s_tok[mi];
            float y = (float)acc[mi * N + n] * f;
            out[mi * N + n] = f32_to_bf16_rne(y);
        }
}
