/*
 * mmq_oracle.c -- the CPU oracle for block-quantized int8 matrix multiply (MMQ).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no header, helper, table or constant with the CUDA path.
 *
 * Plain, slow, obviously correct loops.  Floating point sums are taken in double
 * precision; integer block dots in int64.  Build with -ffp-contract=off so that no
 * multiply-add is fused (the q8_1 quantizer's f32 steps must round exactly once each).
 *
 * Sources (page title, then section / equation):
 *  [P1] "When the Product Won't Collapse: A Negative Result on int8 Tensor-Core MMQ",
 *       sec. "The obstruction: an opaque accumulator", display equation for out[m,n]
 *       (Q8_0 x q8_1 contraction; scale applied once per 32-element block).
 *  [P2] "13 . r7-r8 raw-byte MMQ kernel + wide tile + FA probe", sec. 2 (raw-byte
 *       staging: Q4KB super-block of 144 B per 256 weights), sec. 3.2 (the quantize
 *       pass: amax, scale, round to nearest, clamp, block sum; the Q4_K per-(row,
 *       chunk) scales d*sc and -dmin*m).
 *  [P3] "When Does a Kernel Win Surface? ...", sec. "Kept levers: Vulkan" (the
 *       Q4_K x q8_1 affine identity acc += d1*xs*dot(q4,xq) - m1*xsum).
 *
 * Readings taken where the pages are silent:
 *  - q8_1 block = 36 bytes: f16 d at byte 0, f16 s at byte 2, int8 q[32] at byte 4.
 *  - d = amax / 127 in f32 (one IEEE division); q = rint(x / d) (true division,
 *    round half to even), clamped to [-127, 127]; when d == 0 every q, d and s is 0.
 *  - s = f16( f32(d) * f32(S) ), S = sum of the 32 q: the unrounded f32 d, one f32
 *    multiply, then one rounding to f16.
 *  - Q8_0 block = 34 bytes: f16 d at byte 0, int8 q[32] at byte 2.
 *  - Q4_K super-block = 144 bytes: f16 d @0, f16 dmin @2, 12 packed scale bytes @4,
 *    128 nibble bytes @16.  The 12 bytes pack eight 6-bit sub-scales and eight 6-bit
 *    sub-mins in the common GGUF "K-quant" arrangement (see oracle_q4_k_scale_min).
 *    Nibble byte 32c+i holds element 64c+i in its low half (sub-block 2c) and element
 *    64c+32+i in its high half (sub-block 2c+1).
 *  - Q4_K weight value = d*sc_j*q - dmin*m_j, q in [0, 15]; the min term of the
 *    contraction uses the stored f16 block sum s of the activation block.
 *  - Q5_K ([P3] sec. "Architecture: three orthogonal axes" lists it among the wired GGUF
 *    K-quants; its bytes are not on the pages, so the GGUF arrangement is the reading):
 *    super-block = 176 bytes: f16 d @0, f16 dmin @2, the 12 scale bytes @4 packed as in
 *    Q4_K, 32 high-bit bytes qh @16, 128 nibble bytes qs @48 laid out as the Q4_K nibbles.
 *    Element 64c+i (i < 64) takes its low 4 bits from qs as in Q4_K and its fifth bit
 *    from bit 2c + (i >= 32) of qh[i % 32]; value = d*sc_j*q - dmin*m_j, q in [0, 31].
 *  - Q6_K ([P3] sec. "Architecture: three orthogonal axes" lists it; [P3] sec. "Unified
 *    dp4a decode cores" fixes its 16-element scale groups and the centring q - 32; the
 *    bytes are the GGUF arrangement): super-block = 210 bytes: 128 low-nibble bytes ql @0,
 *    64 bytes of 2-bit high parts qh @128, 16 int8 sub-scales @192, f16 d @208.  Element
 *    128h + 32t + l (h in 0..1, t in 0..3, l in 0..31) takes its low 4 bits from
 *    ql[64h + 32(t mod 2) + l] (low nibble for t < 2, high nibble for t >= 2) and its top
 *    2 bits from bits 2t, 2t+1 of qh[32h + l]; value = d * sc[e/16] * (q - 32), q in
 *    [0, 63].  Its scale changes every 16 elements, inside a q8_1 block, so the block dot
 *    of a 32-element block is taken with the sub-scales inside:
 *    D = sum_k u_k * (q_k - 32) * sc[k/16], and out = sum_b xd * d * D.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 32          /* elements per q8_1 / Q8_0 block, and per Q4_K sub-block */
#define QK_K 256       /* elements per Q4_K super-block */
#define Q8_1_BYTES 36
#define Q8_0_BYTES 34
#define Q4_K_BYTES 144
#define Q5_K_BYTES 176
#define Q6_K_BYTES 210

/* ---------------------------------------------------------------- binary16 */

/* Exact value of an IEEE binary16 bit pattern. */
double oracle_f16_to_f64(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return s ? -v : v;
}

/* Round a double to the nearest binary16, ties to even (IEEE 754 roundTiesToEven).
 * Used only on values that are exact f32 numbers, so this is also f32 -> f16. */
uint16_t oracle_f64_to_f16(double a) {
    uint16_t sign = signbit(a) ? 0x8000 : 0;
    if (isnan(a)) return 0x7e00;
    a = fabs(a);
    if (a >= 65520.0) return sign | 0x7c00; /* 65520 is the tie above 65504 */
    if (a < ldexp(1.0, -14)) {              /* subnormal range, step 2^-24 */
        double q = rint(ldexp(a, 24));      /* q <= 1024; 1024 is the least normal */
        return sign | (uint16_t)q;
    }
    int e;
    double fr = frexp(a, &e);               /* a = fr * 2^e, fr in [0.5, 1) */
    double m = rint(ldexp(fr, 11));         /* 11 significant bits */
    if (m == 2048.0) { m = 1024.0; e += 1; }
    int biased = e + 14;                    /* a = m * 2^(biased - 25) */
    return sign | (uint16_t)((biased << 10) | ((int)m - 1024));
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

/* ---------------------------------------------------------- q8_1 quantize */

/* One 32-element block: amax, d = amax/127, q = clamp(rint(x/d)), S = sum q,
 * stored d and s as f16.  [P2] sec. 3.2; [P1] sec. 1 (activation quantized to q8_1). */
static void quantize_block(const float* x, uint8_t* out) {
    float amax = 0.0f;
    for (int k = 0; k < QK; ++k) {
        float a = fabsf(x[k]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    int S = 0;
    int8_t q[QK];
    for (int k = 0; k < QK; ++k) {
        if (d == 0.0f) {
            q[k] = 0;
        } else {
            float r = rintf(x[k] / d);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[k] = (int8_t)r;
        }
        S += q[k];
    }
    float s = d * (float)S;
    wr16(out + 0, oracle_f64_to_f16((double)d));
    wr16(out + 2, oracle_f64_to_f16((double)s));
    memcpy(out + 4, q, QK);
}

/* x: f32 [M][K] row-major, K % 32 == 0.  out: [M][K/32] blocks of 36 bytes. */
void oracle_quantize_q8_1(const float* x, int64_t M, int64_t K, uint8_t* out) {
    int64_t nb = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b)
            quantize_block(x + m * K + b * QK, out + (m * nb + b) * Q8_1_BYTES);
}

/* ------------------------------------------------------------ Q4_K scales */

/* Sub-scale sc and sub-min m (6 bits each) of sub-block j in 0..7 from the 12
 * packed bytes p.  Sub-blocks 0..3 keep their values in the low 6 bits of bytes
 * j (scale) and j+4 (min).  Sub-blocks 4..7 keep their low 4 bits in byte j+4
 * (scale in the low nibble, min in the high nibble) and their top 2 bits in the
 * spare top bits of bytes j-4 (scale) and j (min). */
void oracle_q4_k_scale_min(const uint8_t* p, int j, int* sc, int* m) {
    if (j < 4) {
        *sc = p[j] & 63;
        *m = p[j + 4] & 63;
    } else {
        *sc = (p[j + 4] & 15) | ((p[j - 4] >> 6) << 4);
        *m = (p[j + 4] >> 4) | ((p[j] >> 6) << 4);
    }
}

/* Nibble code (0..15) of element e in 0..255 of a super-block's 128 nibble bytes. */
static int q4_code(const uint8_t* qs, int e) {
    int c = e / 64, i = e % 64;
    uint8_t byte = qs[32 * c + (i % 32)];
    return i < 32 ? (byte & 15) : (byte >> 4);
}

/* 5-bit code (0..31) of element e in 0..255 of a Q5_K super-block sbk. */
static int q5_code(const uint8_t* sbk, int e) {
    int c = e / 64, i = e % 64;
    int hi = (sbk[16 + (i % 32)] >> (2 * c + (i >= 32))) & 1;
    return q4_code(sbk + 48, e) | (hi << 4);
}

/* 6-bit code (0..63) of element e in 0..255 of a Q6_K super-block sbk, and the int8
 * sub-scale of its 16-element group. */
static int q6_code(const uint8_t* sbk, int e) {
    int h = e / 128, t = (e % 128) / 32, l = e % 32;
    uint8_t lo = sbk[64 * h + 32 * (t % 2) + l];
    int low4 = t < 2 ? (lo & 15) : (lo >> 4);
    int top2 = (sbk[128 + 32 * h + l] >> (2 * t)) & 3;
    return low4 | (top2 << 4);
}

static int q6_scale(const uint8_t* sbk, int e) { return (int)(int8_t)sbk[192 + e / 16]; }

/* --------------------------------------------------------------- block dots */

/* Integer dot of activation block (m, b) with weight block (n, b), exact. */
static int64_t dot_q8_0(const uint8_t* xq, const uint8_t* wq, int64_t m, int64_t n, int64_t nb, int64_t b) {
    const int8_t* xa = (const int8_t*)(xq + (m * nb + b) * Q8_1_BYTES + 4);
    const int8_t* wa = (const int8_t*)(wq + (n * nb + b) * Q8_0_BYTES + 2);
    int64_t s = 0;
    for (int k = 0; k < QK; ++k) s += (int64_t)xa[k] * (int64_t)wa[k];
    return s;
}

static int64_t dot_q4_k(const uint8_t* xq, const uint8_t* wq, int64_t m, int64_t n, int64_t nb, int64_t b) {
    int64_t nsb = nb / 8;
    const int8_t* xa = (const int8_t*)(xq + (m * nb + b) * Q8_1_BYTES + 4);
    const uint8_t* sbk = wq + (n * nsb + b / 8) * Q4_K_BYTES;
    int j = (int)(b % 8);
    int64_t s = 0;
    for (int k = 0; k < QK; ++k) s += (int64_t)xa[k] * (int64_t)q4_code(sbk + 16, 32 * j + k);
    return s;
}

static int64_t dot_q5_k(const uint8_t* xq, const uint8_t* wq, int64_t m, int64_t n, int64_t nb, int64_t b) {
    int64_t nsb = nb / 8;
    const int8_t* xa = (const int8_t*)(xq + (m * nb + b) * Q8_1_BYTES + 4);
    const uint8_t* sbk = wq + (n * nsb + b / 8) * Q5_K_BYTES;
    int j = (int)(b % 8);
    int64_t s = 0;
    for (int k = 0; k < QK; ++k) s += (int64_t)xa[k] * (int64_t)q5_code(sbk, 32 * j + k);
    return s;
}

/* Q6_K block b (elements 32j .. 32j+31 of super-block b/8, j = b mod 8), with the
 * centring and the two 16-element sub-scales inside. */
static int64_t dot_q6_k(const uint8_t* xq, const uint8_t* wq, int64_t m, int64_t n, int64_t nb, int64_t b) {
    int64_t nsb = nb / 8;
    const int8_t* xa = (const int8_t*)(xq + (m * nb + b) * Q8_1_BYTES + 4);
    const uint8_t* sbk = wq + (n * nsb + b / 8) * Q6_K_BYTES;
    int j = (int)(b % 8);
    int64_t s = 0;
    for (int k = 0; k < QK; ++k) {
        int e = 32 * j + k;
        s += (int64_t)xa[k] * (int64_t)(q6_code(sbk, e) - 32) * (int64_t)q6_scale(sbk, e);
    }
    return s;
}

/* dots: int32 [M][N][K/32].  D[m,n,b] = sum over the block of xq * wq. */
void oracle_block_dots_q8_0(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K, int32_t* dots) {
    int64_t nb = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < nb; ++b)
                dots[(m * N + n) * nb + b] = (int32_t)dot_q8_0(xq, wq, m, n, nb, b);
}

/* dots: int32 [M][N][K/32].  D[m,n,b] = sum over the block of xq * q4 (codes 0..15). */
void oracle_block_dots_q4_k(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K, int32_t* dots) {
    int64_t nb = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < nb; ++b)
                dots[(m * N + n) * nb + b] = (int32_t)dot_q4_k(xq, wq, m, n, nb, b);
}

/* dots: int32 [M][N][K/32].  D[m,n,b] = sum over the block of xq * q5 (codes 0..31). */
void oracle_block_dots_q5_k(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K, int32_t* dots) {
    int64_t nb = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < nb; ++b)
                dots[(m * N + n) * nb + b] = (int32_t)dot_q5_k(xq, wq, m, n, nb, b);
}

/* dots: int32 [M][N][K/32].  D[m,n,b] = sum over the block of xq * (q6 - 32) * sc. */
void oracle_block_dots_q6_k(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K, int32_t* dots) {
    int64_t nb = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < nb; ++b)
                dots[(m * N + n) * nb + b] = (int32_t)dot_q6_k(xq, wq, m, n, nb, b);
}

/* -------------------------------------------------------------- contractions */

/* out[m,n] = sum_b xd[m,b] * wd[n,b] * D[m,n,b]          ([P1] display equation)
 * norm[m,n] = sum_b |xd * wd * D|, the scale of the rounding error bound. */
static void entry_q8_0(const uint8_t* xq, const uint8_t* wq, int64_t m, int64_t n, int64_t K,
                       double* out, double* norm) {
    int64_t nb = K / QK;
    double acc = 0.0, t = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        double xd = oracle_f16_to_f64(rd16(xq + (m * nb + b) * Q8_1_BYTES));
        double wd = oracle_f16_to_f64(rd16(wq + (n * nb + b) * Q8_0_BYTES));
        double term = xd * wd * (double)dot_q8_0(xq, wq, m, n, nb, b);
        acc += term;
        t += fabs(term);
    }
    *out = acc;
    *norm = t;
}

/* out[m,n] = sum_b [ xd*d*sc_j*D[m,n,b] - dmin*m_j*xs ]   ([P3] affine identity;
 * [P2] sec. 3.2 per-(row, chunk) scales d*sc and -dmin*m), j = b mod 8.
 * norm[m,n] = sum_b |xd*d*sc_j*D| + |dmin*m_j*xs|. */
static void entry_q4_k(const uint8_t* xq, const uint8_t* wq, int64_t m, int64_t n, int64_t K,
                       double* out, double* norm) {
    int64_t nb = K / QK, nsb = K / QK_K;
    double acc = 0.0, t = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* xb = xq + (m * nb + b) * Q8_1_BYTES;
        const uint8_t* sbk = wq + (n * nsb + b / 8) * Q4_K_BYTES;
        double xd = oracle_f16_to_f64(rd16(xb));
        double xs = oracle_f16_to_f64(rd16(xb + 2));
        double d = oracle_f16_to_f64(rd16(sbk));
        double dmin = oracle_f16_to_f64(rd16(sbk + 2));
        int sc, mn;
        oracle_q4_k_scale_min(sbk + 4, (int)(b % 8), &sc, &mn);
        double t1 = xd * d * (double)sc * (double)dot_q4_k(xq, wq, m, n, nb, b);
        double t2 = dmin * (double)mn * xs;
        acc += t1 - t2;
        t += fabs(t1) + fabs(t2);
    }
    *out = acc;
    *norm = t;
}

/* Q5_K: the same affine identity as Q4_K, over 5-bit codes (j = b mod 8). */
static void entry_q5_k(const uint8_t* xq, const uint8_t* wq, int64_t m, int64_t n, int64_t K,
                       double* out, double* norm) {
    int64_t nb = K / QK, nsb = K / QK_K;
    double acc = 0.0, t = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* xb = xq + (m * nb + b) * Q8_1_BYTES;
        const uint8_t* sbk = wq + (n * nsb + b / 8) * Q5_K_BYTES;
        double xd = oracle_f16_to_f64(rd16(xb));
        double xs = oracle_f16_to_f64(rd16(xb + 2));
        double d = oracle_f16_to_f64(rd16(sbk));
        double dmin = oracle_f16_to_f64(rd16(sbk + 2));
        int sc, mn;
        oracle_q4_k_scale_min(sbk + 4, (int)(b % 8), &sc, &mn);
        double t1 = xd * d * (double)sc * (double)dot_q5_k(xq, wq, m, n, nb, b);
        double t2 = dmin * (double)mn * xs;
        acc += t1 - t2;
        t += fabs(t1) + fabs(t2);
    }
    *out = acc;
    *norm = t;
}

/* Q6_K: out[m,n] = sum_b xd * d * D[m,n,b] (the weight value d * sc * (q - 32) summed
 * against the activation value xd * u; the sub-scales are inside D). */
static void entry_q6_k(const uint8_t* xq, const uint8_t* wq, int64_t m, int64_t n, int64_t K,
                       double* out, double* norm) {
    int64_t nb = K / QK, nsb = K / QK_K;
    double acc = 0.0, t = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* sbk = wq + (n * nsb + b / 8) * Q6_K_BYTES;
        double xd = oracle_f16_to_f64(rd16(xq + (m * nb + b) * Q8_1_BYTES));
        double d = oracle_f16_to_f64(rd16(sbk + 208));
        double term = xd * d * (double)dot_q6_k(xq, wq, m, n, nb, b);
        acc += term;
        t += fabs(term);
    }
    *out = acc;
    *norm = t;
}

/* Full contraction: out, norm double [M][N]. */
void oracle_gemm_q8_0(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                      double* out, double* norm) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) entry_q8_0(xq, wq, m, n, K, out + m * N + n, norm + m * N + n);
}

void oracle_gemm_q4_k(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                      double* out, double* norm) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) entry_q4_k(xq, wq, m, n, K, out + m * N + n, norm + m * N + n);
}

void oracle_gemm_q5_k(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                      double* out, double* norm) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) entry_q5_k(xq, wq, m, n, K, out + m * N + n, norm + m * N + n);
}

void oracle_gemm_q6_k(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                      double* out, double* norm) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) entry_q6_k(xq, wq, m, n, K, out + m * N + n, norm + m * N + n);
}

/* Sampled contraction: entry i is (im[i], in[i]); out, norm double [cnt]. */
void oracle_gemm_q8_0_at(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                         const int64_t* im, const int64_t* in, int64_t cnt, double* out, double* norm) {
    (void)M; (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < cnt; ++i) entry_q8_0(xq, wq, im[i], in[i], K, out + i, norm + i);
}

void oracle_gemm_q4_k_at(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                         const int64_t* im, const int64_t* in, int64_t cnt, double* out, double* norm) {
    (void)M; (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < cnt; ++i) entry_q4_k(xq, wq, im[i], in[i], K, out + i, norm + i);
}

void oracle_gemm_q5_k_at(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                         const int64_t* im, const int64_t* in, int64_t cnt, double* out, double* norm) {
    (void)M; (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < cnt; ++i) entry_q5_k(xq, wq, im[i], in[i], K, out + i, norm + i);
}

void oracle_gemm_q6_k_at(const uint8_t* xq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                         const int64_t* im, const int64_t* in, int64_t cnt, double* out, double* norm) {
    (void)M; (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < cnt; ++i) entry_q6_k(xq, wq, im[i], in[i], K, out + i, norm + i);
}

/* Threads an OpenMP region of this library would use (the CPU baseline's core count). */
int oracle_num_threads(void) {
    int n = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
#endif
    return n;
}
