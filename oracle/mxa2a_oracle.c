/*
 * CPU oracle for the fused AllToAll + MXFP8 block-scaled GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, exact reference the
 * CUDA path is checked against.  Only the tests, the package's smoke check
 * and the benchmark's CPU-baseline leg may load it; the CUDA library never
 * links, includes or calls it, and it shares no code with it.
 *
 * What it computes (the all_to_all_matmul kernel, all_to_all_matmul_impl.h,
 * MatmulProcess + AllToAllComm::PutSegmentToRank): segment r of the exchange
 * lands at offset r*commMSize*kPerRank of a staging slot, and the GEMM runs
 * over all R segments with split-K = R accumulating into one output, so the
 * R segments are K-columns [r*kPerRank, (r+1)*kPerRank) of one operand A, and
 *
 *   C[m][n] = RNE_bf16( sum_r sum_k  dec(A_seg[r][m][k]) * 2^(A_scale_seg[r][m][k/32]-127)
 *                                  * dec(B[n][r*ka+k])  * 2^(B_scale[n][(r*ka+k)/32]-127) )
 *
 * with E4M3 "fn" codes (fp8_e4m3fn_t), E8M0 scales (fp8_e8m0_t) one per 32
 * elements along K, and a BF16 output (the kernel entry's third template
 * argument, bfloat16_t).
 *
 * How: the sum is formed EXACTLY and rounded to BF16 once.
 *   - every E4M3 value is an integer multiple of 2^-9 with magnitude at most
 *     448 = 229376 * 2^-9, so it is decoded to that integer;
 *   - the dot product of one 32-element block is then an exact int64
 *     (|sum| < 32 * 229376^2 < 2^41) in units of 2^-18;
 *   - the block's value is that integer times 2^(sa-127 + sb-127 - 18);
 *     all blocks are added into an exact fixed-point big integer whose unit is
 *     2^-272 (the smallest block exponent), kept as separate positive and
 *     negative magnitudes;
 *   - the difference is rounded once to BF16, round to nearest, ties to even,
 *     with BF16 subnormals and overflow to infinity.
 * No floating-point arithmetic touches the sum, so the result does not depend
 * on any summation order.  A NaN code (E4M3 0x7F/0xFF or E8M0 0xFF) anywhere
 * in a contributing block makes the output the canonical BF16 NaN 0x7FC0.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define MX_BLOCK 32
#define LIMBS 11               /* 704-bit magnitudes; the largest sum needs < 600 bits */
#define UNIT_EXP (-286)        /* value of bit 0 of the big integer: 2^-286, the smallest block
                                  quantum (E5M2 x E5M2: 2^-32 units times 2^(0-127) twice) */
#define FMT_E4M3 0
#define FMT_E5M2 1

/* E4M3 "fn": sign, 4-bit exponent (bias 7), 3-bit mantissa; exponent 0 is
 * subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity.
 * Returns the value in units of 2^-9. */
static int32_t e4m3_units(uint8_t code, int *nan)
{
    int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
    int32_t mag;
    if (e == 15 && m == 7) { *nan = 1; return 0; }
    if (e == 0) mag = m;                        /* m/8 * 2^-6 = m * 2^-9 */
    else mag = (int32_t)(8 + m) << (e - 1);     /* (8+m)/8 * 2^(e-7) = (8+m)*2^(e-1) * 2^-9 */
    return s ? -mag : mag;
}

/* E5M2: sign, 5-bit exponent (bias 15), 2-bit mantissa; exponent 0 is
 * subnormal (m/4 * 2^-14); exponent 31 is infinity (m == 0) or NaN (m != 0).
 * Returns the value in units of 2^-16 (the largest, 57344, is 7 * 2^29
 * units); *special = 1 for NaN, 2 for +inf, 3 for -inf, else untouched. */
static int64_t e5m2_units(uint8_t code, int *special)
{
    int s = code >> 7, e = (code >> 2) & 0x1F, m = code & 3;
    int64_t mag;
    if (e == 31) { *special = m ? 1 : (s ? 3 : 2); return 0; }
    if (e == 0) mag = (int64_t)m;                /* m/4 * 2^-14 = m * 2^-16 */
    else mag = (int64_t)(4 + m) << (e - 1);      /* (4+m)/4 * 2^(e-15) = (4+m)*2^(e-1) * 2^-16 */
    return s ? -mag : mag;
}

double mxa2a_oracle_decode_e5m2(uint8_t code)
{
    int special = 0;
    int64_t u = e5m2_units(code, &special);
    if (special == 1) return __builtin_nan("");
    if (special == 2) return __builtin_inf();
    if (special == 3) return -__builtin_inf();
    return (double)u / 65536.0;
}

double mxa2a_oracle_decode_e4m3(uint8_t code)
{
    int nan = 0;
    int32_t u = e4m3_units(code, &nan);
    if (nan) return __builtin_nan("");
    return (double)u / 512.0;
}

/* E8M0: unsigned biased exponent, value 2^(e-127); 0xFF is NaN. */
double mxa2a_oracle_decode_e8m0(uint8_t code)
{
    if (code == 0xFF) return __builtin_nan("");
    double v = 1.0;
    int e = (int)code - 127;
    while (e > 0) { v *= 2.0; --e; }
    while (e < 0) { v *= 0.5; ++e; }
    return v;
}

typedef struct { uint64_t w[LIMBS]; } big_t;

/* mag += v * 2^shift, for v < 2^63 and 0 <= shift < 64*(LIMBS-2) */
static void big_add_shifted(big_t *a, uint64_t v, int shift)
{
    int limb = shift / 64, b = shift % 64;
    uint64_t part[2];
    part[0] = v << b;
    part[1] = b ? (v >> (64 - b)) : 0;
    uint64_t carry = 0;
    for (int i = limb; i < LIMBS; ++i) {
        uint64_t add = (i - limb < 2) ? part[i - limb] : 0;
        if (i - limb >= 2 && carry == 0) break;
        uint64_t o = a->w[i];
        uint64_t t = o + add;
        uint64_t c1 = t < o;
        uint64_t t2 = t + carry;
        uint64_t c2 = t2 < t;
        a->w[i] = t2;
        carry = c1 | c2;
    }
}

static int big_cmp(const big_t *a, const big_t *b)
{
    for (int i = LIMBS - 1; i >= 0; --i) {
        if (a->w[i] != b->w[i]) return a->w[i] > b->w[i] ? 1 : -1;
    }
    return 0;
}

/* d = a - b, requires a >= b */
static void big_sub(big_t *d, const big_t *a, const big_t *b)
{
    uint64_t borrow = 0;
    for (int i = 0; i < LIMBS; ++i) {
        uint64_t x = a->w[i], y = b->w[i];
        uint64_t t = x - y;
        uint64_t b1 = x < y;
        uint64_t t2 = t - borrow;
        uint64_t b2 = t < borrow;
        d->w[i] = t2;
        borrow = b1 | b2;
    }
}

static int big_bit(const big_t *a, int i)
{
    if (i < 0 || i >= 64 * LIMBS) return 0;
    return (int)((a->w[i / 64] >> (i % 64)) & 1u);
}

static int big_msb(const big_t *a)
{
    for (int i = LIMBS - 1; i >= 0; --i)
        if (a->w[i]) return i * 64 + 63 - __builtin_clzll(a->w[i]);
    return -1;
}

/* any bit strictly below position i set? */
static int big_any_below(const big_t *a, int i)
{
    if (i <= 0) return 0;
    int full = i / 64, rem = i % 64;
    for (int k = 0; k < full && k < LIMBS; ++k)
        if (a->w[k]) return 1;
    if (rem && full < LIMBS && (a->w[full] & ((1ull << rem) - 1))) return 1;
    return 0;
}

/* bits [lo, lo+n) as an integer, n <= 16 */
static uint32_t big_field(const big_t *a, int lo, int n)
{
    uint32_t v = 0;
    for (int k = n - 1; k >= 0; --k) v = (v << 1) | (uint32_t)big_bit(a, lo + k);
    return v;
}

/* Round sign * mag * 2^UNIT_EXP to BF16 (1-8-7), nearest, ties to even. */
static uint16_t round_to_bf16(int negative, const big_t *mag)
{
    const int sub_shift = -133 - UNIT_EXP;        /* bit position of 2^-133, the BF16 subnormal quantum */
    int p = big_msb(mag);
    uint16_t sign = negative ? 0x8000 : 0;
    if (p < 0) return 0x0000;                      /* exact zero: +0 */
    /* Quantum of the result: 2^(e-7) for a normal result whose leading bit is
     * 2^e, 2^-133 below the normal range.  As a bit position: max(p-7, sub_shift). */
    int shift = p - 7;
    int subnormal = 0;
    if (shift < sub_shift) { shift = sub_shift; subnormal = 1; }
    uint32_t q = big_field(mag, shift, p - shift + 1);   /* kept significand */
    int round_bit = big_bit(mag, shift - 1);
    int sticky = big_any_below(mag, shift - 1);
    if (round_bit && (sticky || (q & 1u))) q += 1;
    if (subnormal) {
        /* value = q * 2^-133 with q in [0, 128]; q == 128 is the smallest
         * normal number, whose encoding is exactly 0x0080 */
        return (uint16_t)(sign | q);
    }
    int e = p + UNIT_EXP;                          /* q in [128, 256] times 2^(e-7) */
    if (q == 256) { q = 128; e += 1; }
    int field = e + 127;
    if (field >= 255) return (uint16_t)(sign | 0x7F80);   /* overflow: infinity */
    return (uint16_t)(sign | (field << 7) | (q - 128));
}

typedef struct {
    int R;
    int64_t M, ka, N, K;
    const uint8_t *const *A_seg;
    const uint8_t *const *A_sf;
    const uint8_t *B, *B_sf;
    const int64_t *rows, *cols;
    int64_t nrows, ncols;
    uint16_t *C;
    int64_t *Bu;          /* decoded B units [ncols][K] */
    uint8_t *Bnan;        /* per (col, block) NaN flag */
    int8_t *Binf;         /* E5M2 B: per element +1 / -1 for +-inf, else 0 */
    uint8_t *Binfb;       /* per (col, block): the block holds an infinity */
    int fmt_a, fmt_b;     /* FMT_E4M3 or FMT_E5M2 */
    int uexp_fix;         /* units exponent of a product beyond the E4M3 x E4M3 2^-18 */
    int64_t next_row;     /* work counter */
    pthread_mutex_t lock;
} job_t;

/* 128-bit magnitude v added at bit position shift (two 64-bit halves) */
static void big_add_shifted128(big_t *a, unsigned __int128 v, int shift)
{
    uint64_t lo = (uint64_t)v, hi = (uint64_t)(v >> 64);
    if (lo >> 63) {           /* keep each half below 2^63 for big_add_shifted */
        big_add_shifted(a, lo >> 1, shift + 1);
        big_add_shifted(a, lo & 1u, shift);
    } else {
        big_add_shifted(a, lo, shift);
    }
    if (hi) big_add_shifted(a, hi, shift + 64);
}

/* Infinity / NaN of one 32-block that holds an infinity (IEEE products and
 * sums): 1 NaN, 2 +inf, 3 -inf. */
static int block_special(const int64_t *au, const int8_t *ainf, const int64_t *bu, const int8_t *binf)
{
    int pos = 0, neg = 0;
    for (int k = 0; k < MX_BLOCK; ++k) {
        int ia = ainf ? ainf[k] : 0, ib = binf ? binf[k] : 0;
        if (!ia && !ib) continue;
        int sa = ia ? ia : (au[k] > 0 ? 1 : (au[k] < 0 ? -1 : 0));
        int sb = ib ? ib : (bu[k] > 0 ? 1 : (bu[k] < 0 ? -1 : 0));
        if (sa == 0 || sb == 0) return 1;      /* inf * 0 */
        if (sa * sb > 0) pos = 1; else neg = 1;
    }
    if (pos && neg) return 1;                  /* inf - inf */
    return pos ? 2 : 3;
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    const int64_t K = j->K, nb = K / MX_BLOCK, bpr = j->ka / MX_BLOCK;
    int64_t *Au = (int64_t *)malloc(sizeof(int64_t) * (size_t)K);
    uint8_t *Anan = (uint8_t *)malloc((size_t)nb);
    int8_t *Ainf = (int8_t *)malloc((size_t)K);
    uint8_t *Ainfb = (uint8_t *)malloc((size_t)nb);
    const int wide = j->fmt_a == FMT_E5M2 && j->fmt_b == FMT_E5M2;   /* products need > 64 bits */
    for (;;) {
        pthread_mutex_lock(&j->lock);
        int64_t i = j->next_row++;
        pthread_mutex_unlock(&j->lock);
        if (i >= j->nrows) break;
        int64_t m = j->rows ? j->rows[i] : i;
        /* decode row m of the K-concatenation of the R segments, and flag the
         * 32-blocks that hold a NaN code or a NaN scale (and, for E5M2, the
         * ones that hold an infinity) */
        memset(Anan, 0, (size_t)nb);
        memset(Ainf, 0, (size_t)K);
        memset(Ainfb, 0, (size_t)nb);
        for (int r = 0; r < j->R; ++r) {
            const uint8_t *src = j->A_seg[r] + m * j->ka;
            const uint8_t *sf = j->A_sf[r] + m * bpr;
            for (int64_t k = 0; k < j->ka; ++k) {
                int nan = 0;
                if (j->fmt_a == FMT_E5M2) {
                    int special = 0;
                    Au[r * j->ka + k] = e5m2_units(src[k], &special);
                    nan = special == 1;
                    if (special >= 2) {
                        Ainf[r * j->ka + k] = special == 2 ? 1 : -1;
                        Ainfb[(r * j->ka + k) / MX_BLOCK] = 1;
                    }
                } else {
                    Au[r * j->ka + k] = e4m3_units(src[k], &nan);
                }
                if (nan || sf[k / MX_BLOCK] == 0xFF) Anan[(r * j->ka + k) / MX_BLOCK] = 1;
            }
        }
        for (int64_t jc = 0; jc < j->ncols; ++jc) {
            int64_t n = j->cols ? j->cols[jc] : jc;
            const int64_t *bu = j->Bu + jc * K;
            big_t pos, neg;
            memset(&pos, 0, sizeof pos);
            memset(&neg, 0, sizeof neg);
            int is_nan = 0, pinf = 0, ninf = 0;
            for (int64_t b = 0; b < nb; ++b) {
                if (Anan[b] || j->Bnan[jc * nb + b]) { is_nan = 1; break; }
                if (Ainfb[b] || j->Binfb[jc * nb + b]) {
                    const int sp = block_special(Au + b * MX_BLOCK, Ainf + b * MX_BLOCK, bu + b * MX_BLOCK,
                                                 j->Binf + jc * K + b * MX_BLOCK);
                    if (sp == 1) { is_nan = 1; break; }
                    if (sp == 2) pinf = 1; else ninf = 1;
                    continue;
                }
                int r = (int)(b / bpr);
                if (wide) {
                    __int128 s = 0;                     /* exact, units of 2^-32 */
                    for (int64_t k = b * MX_BLOCK; k < (b + 1) * MX_BLOCK; ++k)
                        s += (__int128)Au[k] * (__int128)bu[k];
                    if (s == 0) continue;
                    int sa = j->A_sf[r][m * bpr + (b % bpr)];
                    int sb = j->B_sf[n * nb + b];
                    int shift = (sa - 127) + (sb - 127) - 32 - UNIT_EXP;
                    if (s > 0) big_add_shifted128(&pos, (unsigned __int128)s, shift);
                    else big_add_shifted128(&neg, (unsigned __int128)(-s), shift);
                    continue;
                }
                int64_t s = 0;                          /* exact, units of 2^-18 (E4M3 x E4M3) */
                for (int64_t k = b * MX_BLOCK; k < (b + 1) * MX_BLOCK; ++k)
                    s += (int64_t)Au[k] * (int64_t)bu[k];
                if (s == 0) continue;
                int sa = j->A_sf[r][m * bpr + (b % bpr)];
                int sb = j->B_sf[n * nb + b];
                /* value = s * 2^(sa-127 + sb-127 - 18); bit position relative to 2^UNIT_EXP */
                int shift = (sa - 127) + (sb - 127) - 18 - UNIT_EXP;
                shift -= j->uexp_fix;                   /* other element formats: finer units */
                if (s > 0) big_add_shifted(&pos, (uint64_t)s, shift);
                else big_add_shifted(&neg, (uint64_t)(-s), shift);
            }
            uint16_t out;
            if (is_nan || (pinf && ninf)) {
                out = 0x7FC0;
            } else if (pinf || ninf) {
                out = pinf ? 0x7F80 : 0xFF80;
            } else {
                int c = big_cmp(&pos, &neg);
                big_t d;
                if (c >= 0) { big_sub(&d, &pos, &neg); out = round_to_bf16(0, &d); }
                else { big_sub(&d, &neg, &pos); out = round_to_bf16(1, &d); }
            }
            j->C[i * j->ncols + jc] = out;
        }
    }
    free(Au);
    free(Anan);
    free(Ainf);
    free(Ainfb);
    return NULL;
}

/*
 * C_out[i][jc] = C[rows[i]][cols[jc]] as BF16 bits, with A and B elements in
 * the given formats (FMT_E4M3 = 0, FMT_E5M2 = 1; the four pairs are the
 * kernel entries E4M3E4M3, E5M2E5M2, E4M3E5M2 and E5M2E4M3).  rows/cols may
 * be NULL (all rows / all columns, in order).  nthreads <= 0 uses every
 * online core.  Returns 0 on success, -1 on bad arguments or allocation
 * failure.
 */
int mxa2a_oracle_gemm_fmt(int R, int64_t M, int64_t ka, int64_t N,
                          const uint8_t *const *A_seg, const uint8_t *const *A_scale_seg,
                          const uint8_t *B, const uint8_t *B_scale, int fmt_a, int fmt_b,
                          const int64_t *rows, int64_t nrows,
                          const int64_t *cols, int64_t ncols,
                          uint16_t *C_out, int nthreads)
{
    if (R < 1 || M < 0 || N < 0 || ka <= 0 || ka % MX_BLOCK) return -1;
    if (!A_seg || !A_scale_seg || !B || !B_scale || !C_out) return -1;
    if ((fmt_a != FMT_E4M3 && fmt_a != FMT_E5M2) || (fmt_b != FMT_E4M3 && fmt_b != FMT_E5M2)) return -1;
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    if (nrows == 0 || ncols == 0) return 0;
    job_t j;
    memset(&j, 0, sizeof j);
    j.R = R; j.M = M; j.ka = ka; j.N = N; j.K = (int64_t)R * ka;
    j.A_seg = A_seg; j.A_sf = A_scale_seg; j.B = B; j.B_sf = B_scale;
    j.rows = rows; j.cols = cols; j.nrows = nrows; j.ncols = ncols; j.C = C_out;
    j.fmt_a = fmt_a; j.fmt_b = fmt_b;
    /* units: E4M3 2^-9, E5M2 2^-16; the int64 block path is written for 2^-18 */
    j.uexp_fix = (fmt_a == FMT_E5M2 ? 7 : 0) + (fmt_b == FMT_E5M2 ? 7 : 0);
    for (int64_t i = 0; rows && i < nrows; ++i) if (rows[i] < 0 || rows[i] >= M) return -1;
    for (int64_t i = 0; cols && i < ncols; ++i) if (cols[i] < 0 || cols[i] >= N) return -1;
    const int64_t K = j.K, nb = K / MX_BLOCK;
    j.Bu = (int64_t *)malloc(sizeof(int64_t) * (size_t)(ncols * K));
    j.Bnan = (uint8_t *)calloc((size_t)(ncols * nb), 1);
    j.Binf = (int8_t *)calloc((size_t)(ncols * K), 1);
    j.Binfb = (uint8_t *)calloc((size_t)(ncols * nb), 1);
    if (!j.Bu || !j.Bnan || !j.Binf || !j.Binfb) {
        free(j.Bu); free(j.Bnan); free(j.Binf); free(j.Binfb);
        return -1;
    }
    for (int64_t jc = 0; jc < ncols; ++jc) {
        int64_t n = cols ? cols[jc] : jc;
        for (int64_t k = 0; k < K; ++k) {
            int nan = 0;
            if (fmt_b == FMT_E5M2) {
                int special = 0;
                j.Bu[jc * K + k] = e5m2_units(B[n * K + k], &special);
                nan = special == 1;
                if (special >= 2) {
                    j.Binf[jc * K + k] = special == 2 ? 1 : -1;
                    j.Binfb[jc * nb + k / MX_BLOCK] = 1;
                }
            } else {
                j.Bu[jc * K + k] = e4m3_units(B[n * K + k], &nan);
            }
            if (nan) j.Bnan[jc * nb + k / MX_BLOCK] = 1;
        }
        for (int64_t b = 0; b < nb; ++b)
            if (B_scale[n * nb + b] == 0xFF) j.Bnan[jc * nb + b] = 1;
    }
    pthread_mutex_init(&j.lock, NULL);
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, worker, &j) == 0) ++started;
    if (started == 0) worker(&j);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&j.lock);
    free(j.Bu);
    free(j.Bnan);
    free(j.Binf);
    free(j.Binfb);
    return 0;
}

/* The E4M3 x E4M3 product (the method's main entry). */
int mxa2a_oracle_gemm(int R, int64_t M, int64_t ka, int64_t N,
                      const uint8_t *const *A_seg, const uint8_t *const *A_scale_seg,
                      const uint8_t *B, const uint8_t *B_scale,
                      const int64_t *rows, int64_t nrows,
                      const int64_t *cols, int64_t ncols,
                      uint16_t *C_out, int nthreads)
{
    return mxa2a_oracle_gemm_fmt(R, M, ka, N, A_seg, A_scale_seg, B, B_scale, FMT_E4M3, FMT_E4M3, rows, nrows, cols,
                                 ncols, C_out, nthreads);
}

/* Round a value given exactly as  sign * sum_i digits[i] * 2^(exp0 + 31*i)
 * (digits < 2^31, i < ndigits) to BF16; exposed so the tests can check the
 * rounding step on its own against an independent rounding. */
uint16_t mxa2a_oracle_round_bf16(int negative, const uint32_t *digits, int ndigits, int exp0)
{
    big_t mag;
    memset(&mag, 0, sizeof mag);
    for (int i = 0; i < ndigits; ++i) {
        if (!digits[i]) continue;
        int shift = exp0 + 31 * i - UNIT_EXP;
        if (shift < 0 || shift >= 64 * (LIMBS - 2)) return 0xFFFF;  /* out of range */
        big_add_shifted(&mag, digits[i], shift);
    }
    return round_to_bf16(negative, &mag);
}
