/*
 * exl3_oracle.c -- plain, slow, obviously-correct CPU reference for the EXL3
 * trellis linear layer, its merged-shard column-slice form, the grouped MoE
 * form and the int8 embedding gather.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links or calls
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA path.
 *
 * Arithmetic is fp64 throughout; fp16 / bf16 appear only where the method
 * stores a value in that format (decoded weights, scale vectors, inputs,
 * the final output), converted by hand-written round-to-nearest-even
 * routines below.
 *
 * Sources (web pages this reference restates):
 *   [escha]  radiance_escha.py (vLLM method for escha EXL3 trellis W2
 *            checkpoints): module docstring "THE FORWARD", the two mistakes
 *            it warns about, the per-shard rationale; process_weights_after_loading
 *            (code tensor [IC/16, OC/16, 16K], K = last dim / 16, rin per
 *            shard); escha_linear_into (M == 0 no-op, ldo / col0 slice).
 *   [linear] vllm-quantpack 0.1.0, exl3/linear.py: module docstring (the
 *            code is a packed, tail-biting trellis whose width gives the
 *            bitrate), Exl3LinearMethod._forward (one GEMM per shard).
 *   [embed]  vllm-quantpack 0.1.0, exl3/embedding.py: embedding() --
 *            q[ids] converted, times s[ids].
 *   [bank]   bank.py (one layer's EXL3 expert bank): w13 = [w1 | w3] per
 *            slot, w2, suh/svh vectors [E, ...], K-sorted slots.
 *
 * Readings where the pages are silent (the trellis bit layout and the
 * codebook are not on any page):
 *   - stream: a tile's 16K int16 words, in index order, each read as a uint16
 *     most-significant bit first; stream bit p is bit (15 - p%16) of word p/16.
 *   - state of weight t (0..255): the 16 stream bits ending at bit (t+1)K,
 *     i.e. bits [(t+1)K-16, (t+1)K) taken modulo 256K (tail-biting: the first
 *     windows wrap round to the end of the tile), first bit = MSB.
 *   - codebook: the 3INST hash family of QTIP (Tseng et al., 2024):
 *     z = 89226354*s + 64248484 (mod 2^32); z' = (z & 0x8FFF8FFF) ^ 0x3B603B60;
 *     weight = fp16(half(z' low 16 bits) + half(z' high 16 bits)), the sum
 *     formed exactly and rounded once.
 *   - weight t of tile code[a][b] is W[16a + t/16][16b + t%16]; the first
 *     tile index runs along the input channels.
 *   - Had128 is the Sylvester matrix H[i][j] = (-1)^popcount(i & j) scaled by
 *     1/sqrt(128), applied to each contiguous block of 128 channels.
 * Parity of these readings against real exllamav3 checkpoints: unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EXL3O_OK 0
#define EXL3O_EINVAL 1

/* ------------------------------------------------------------------------ */
/* IEEE binary16 / bfloat16 <-> double, written from the format definitions  */
/* ------------------------------------------------------------------------ */

double exl3o_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* zero / subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

double exl3o_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int m = b & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + m), e - 134);     /* (1 + m/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a finite |a| onto the grid of a binary format with `mant` explicit
 * mantissa bits and minimum normal exponent `emin`, ties to even.  Returns the
 * magnitude bits (exponent field << mant | mantissa), or -1 on overflow. */
static long round_to_format(double a, int mant, int emin, int emax)
{
    if (a == 0.0)
        return 0;
    int e2;
    frexp(a, &e2);                 /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;                /* a in [2^E, 2^(E+1)) */
    if (E < emin)
        E = emin;                  /* subnormal range shares emin's quantum */
    double n = ldexp(a, mant - E); /* a / quantum, exact (power-of-two scale) */
    double r = nearbyint(n);       /* default rounding mode: nearest, ties even */
    double diff = n - floor(n);
    if (diff == 0.5) {             /* make the tie rule explicit */
        double f = floor(n);
        r = (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
    }
    long m = (long)r;              /* in [0, 2^(mant+1)] */
    long bits;
    if (m < (1L << mant))
        bits = m;                  /* only reachable when E == emin: subnormal */
    else
        bits = ((long)(E - emin + 1) << mant) + (m - (1L << mant));
    long maxbits = ((long)(emax - emin + 2) << mant);  /* first infinite code */
    if (bits >= maxbits)
        return -1;
    return bits;
}

uint16_t exl3o_f16_from_f64(double v)
{
    if (isnan(v))
        return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7C00;
    long bits = round_to_format(a, 10, -14, 15);
    if (bits < 0)
        return sign | 0x7C00;
    return (uint16_t)(sign | bits);
}

uint16_t exl3o_bf16_from_f64(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7F80;
    long bits = round_to_format(a, 7, -126, 127);
    if (bits < 0)
        return sign | 0x7F80;
    return (uint16_t)(sign | bits);
}

/* ------------------------------------------------------------------------ */
/* Trellis decode                                                            */
/* ------------------------------------------------------------------------ */

/* 3INST codebook: 16-bit trellis state -> fp16 weight (bits). */
uint16_t exl3o_codebook(uint32_t state)
{
    uint32_t z = (uint32_t)(89226354u * (state & 0xFFFFu) + 64248484u);
    z = (z & 0x8FFF8FFFu) ^ 0x3B603B60u;
    double lo = exl3o_f16_to_f64((uint16_t)(z & 0xFFFFu));
    double hi = exl3o_f16_to_f64((uint16_t)(z >> 16));
    return exl3o_f16_from_f64(lo + hi);   /* exact sum, one rounding */
}

/* Stream bit p of a tile (p taken modulo the tile's 256K bits). */
static int stream_bit(const int16_t *tile, int K, long p)
{
    long n = 256L * K;
    p %= n;
    if (p < 0)
        p += n;
    uint16_t w = (uint16_t)tile[p / 16];
    return (w >> (15 - (p % 16))) & 1;
}

/* Trellis state of weight t: stream bits [(t+1)K-16, (t+1)K), MSB first. */
uint32_t exl3o_state(const int16_t *tile, int K, int t)
{
    uint32_t s = 0;
    long start = (long)(t + 1) * K - 16;
    for (int j = 0; j < 16; j++)
        s = (s << 1) | (uint32_t)stream_bit(tile, K, start + j);
    return s;
}

/* The 256 fp16 weights of one 16x16 tile, in trellis order t = 16r + c. */
void exl3o_decode_tile(const int16_t *tile, int K, uint16_t *w256)
{
    for (int t = 0; t < 256; t++)
        w256[t] = exl3o_codebook(exl3o_state(tile, K, t));
}

static int valid_k(int K) { return K >= 1 && K <= 8; }

/* Dense fp16 weights of output columns [oc0, oc0+noc) of a code tensor
 * [IC/16][OC/16][16K]: W[i][j] (row-major, IC rows, noc columns) is weight
 * (input i, output oc0 + j).  oc0 and noc must be multiples of 16. */
int exl3o_reconstruct_cols(const int16_t *code, int IC, int OC, int K,
                           int oc0, int noc, uint16_t *W)
{
    if (!valid_k(K) || IC % 16 || OC % 16 || oc0 % 16 || noc % 16 ||
        oc0 < 0 || oc0 + noc > OC)
        return EXL3O_EINVAL;
    int tiles_oc = OC / 16;
    long words = 16L * K;
#pragma omp parallel for schedule(static)
    for (int a = 0; a < IC / 16; a++) {
        uint16_t w256[256];
        for (int b = oc0 / 16; b < (oc0 + noc) / 16; b++) {
            const int16_t *tile = code + ((long)a * tiles_oc + b) * words;
            exl3o_decode_tile(tile, K, w256);
            for (int t = 0; t < 256; t++) {
                int r = t / 16, c = t % 16;
                W[(long)(16 * a + r) * noc + (16 * b + c - oc0)] = w256[t];
            }
        }
    }
    return EXL3O_OK;
}

int exl3o_reconstruct(const int16_t *code, int IC, int OC, int K, uint16_t *W)
{
    return exl3o_reconstruct_cols(code, IC, OC, K, 0, OC, W);
}

/* ------------------------------------------------------------------------ */
/* Hadamard-128                                                              */
/* ------------------------------------------------------------------------ */

/* Sylvester-ordered 128x128 Hadamard matrix (entries +-1, unnormalised). */
void exl3o_hadamard128(double *H)
{
    for (int i = 0; i < 128; i++)
        for (int j = 0; j < 128; j++)
            H[i * 128 + j] = (__builtin_popcount((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
}

/* y = Had128(v) blockwise on n (multiple of 128) values: each contiguous
 * block of 128 is multiplied by H / sqrt(128). */
static void had_blocks(const double *H, const double *v, double *y, long n)
{
    const double norm = 1.0 / sqrt(128.0);
    for (long b = 0; b < n; b += 128)
        for (int i = 0; i < 128; i++) {
            double acc = 0.0;
            for (int j = 0; j < 128; j++)
                acc += H[i * 128 + j] * v[b + j];
            y[b + i] = acc * norm;
        }
}

/* ------------------------------------------------------------------------ */
/* EXL3 linear                                                               */
/* ------------------------------------------------------------------------ */

/* [escha] THE FORWARD, first factor: u = Had128((x * s_in) * rin) per
 * 128-channel block, fp64.  x bf16 [M][IC]; u [M][IC]. */
int exl3o_pretransform_f64(const uint16_t *x, long M, int IC, const uint16_t *s_in,
                           const uint16_t *rin, double *u)
{
    if (IC % 128 || M < 0)
        return EXL3O_EINVAL;
    double *H = malloc(sizeof(double) * 128 * 128);
    double *xs = malloc(sizeof(double) * IC);
    exl3o_hadamard128(H);
    for (long m = 0; m < M; m++) {
        for (int c = 0; c < IC; c++)
            xs[c] = (exl3o_bf16_to_f64(x[m * IC + c]) * exl3o_f16_to_f64(s_in[c]))
                    * exl3o_f16_to_f64(rin[c]);
        had_blocks(H, xs, u + m * IC, IC);
    }
    free(H);
    free(xs);
    return EXL3O_OK;
}

/*
 * [escha] THE FORWARD, restated step by step:
 *   u = Had128((x * s_in) * rin)          rin is a pre-scale, before its Had
 *   v = u @ decode(code)
 *   y = (Had128(v) * rout) * s_out        rout is a post-scale, after its Had
 * No bias.  x is bf16 [M][IC]; the four scale vectors are fp16; y is returned
 * unrounded in fp64 for output columns [blk0*128, (blk0+nblk)*128):
 * y[m][j] is output column blk0*128 + j, row stride nblk*128.
 */
int exl3o_linear_f64(const uint16_t *x, long M, int IC,
                     const int16_t *code, int OC, int K,
                     const uint16_t *s_in, const uint16_t *rin,
                     const uint16_t *rout, const uint16_t *s_out,
                     int blk0, int nblk, double *y)
{
    if (!valid_k(K) || IC % 128 || OC % 128 || M < 0 || blk0 < 0 || nblk < 0 ||
        (long)(blk0 + nblk) * 128 > OC)
        return EXL3O_EINVAL;
    if (M == 0 || nblk == 0)
        return EXL3O_OK;
    int noc = nblk * 128, oc0 = blk0 * 128;

    uint16_t *Wh = malloc(sizeof(uint16_t) * (size_t)IC * noc);
    double *W = malloc(sizeof(double) * (size_t)IC * noc);
    double *H = malloc(sizeof(double) * 128 * 128);
    if (!Wh || !W || !H) {
        free(Wh); free(W); free(H);
        return EXL3O_EINVAL;
    }
    exl3o_hadamard128(H);

    /* step 1: decoded weights */
    exl3o_reconstruct_cols(code, IC, OC, K, oc0, noc, Wh);
    for (long i = 0; i < (long)IC * noc; i++)
        W[i] = exl3o_f16_to_f64(Wh[i]);
    free(Wh);

#pragma omp parallel for schedule(dynamic)
    for (long m = 0; m < M; m++) {
        double *xs = malloc(sizeof(double) * IC);
        double *u = malloc(sizeof(double) * IC);
        double *v = malloc(sizeof(double) * noc);
        double *hv = malloc(sizeof(double) * noc);
        /* step 2: pre-scale then input Hadamard */
        for (int c = 0; c < IC; c++)
            xs[c] = (exl3o_bf16_to_f64(x[m * IC + c]) * exl3o_f16_to_f64(s_in[c]))
                    * exl3o_f16_to_f64(rin[c]);
        had_blocks(H, xs, u, IC);
        /* step 3: GEMM against the decoded weights */
        for (int j = 0; j < noc; j++)
            v[j] = 0.0;
        for (int c = 0; c < IC; c++) {
            double uc = u[c];
            const double *wr = W + (long)c * noc;
            for (int j = 0; j < noc; j++)
                v[j] += uc * wr[j];
        }
        /* step 4: output Hadamard, then rout, then s_out */
        had_blocks(H, v, hv, noc);
        for (int j = 0; j < noc; j++)
            y[m * noc + j] = (hv[j] * exl3o_f16_to_f64(rout[oc0 + j]))
                             * exl3o_f16_to_f64(s_out[oc0 + j]);
        free(xs); free(u); free(v); free(hv);
    }
    free(W);
    free(H);
    return EXL3O_OK;
}

/*
 * [escha] escha_linear_into: the shard writes its own column slice
 * out[:, col0 : col0+OC] of a caller-owned bf16 [M][ldo] buffer; every other
 * column is left as it was.  Output rounded once to bf16 (round to nearest
 * even).
 */
int exl3o_linear_into(const uint16_t *x, long M, int IC,
                      const int16_t *code, int OC, int K,
                      const uint16_t *s_in, const uint16_t *rin,
                      const uint16_t *rout, const uint16_t *s_out,
                      uint16_t *out, long ldo, long col0)
{
    if (col0 < 0 || ldo < OC || col0 + OC > ldo)
        return EXL3O_EINVAL;
    if (M == 0)
        return EXL3O_OK;
    double *y = malloc(sizeof(double) * (size_t)M * OC);
    if (!y)
        return EXL3O_EINVAL;
    int rc = exl3o_linear_f64(x, M, IC, code, OC, K, s_in, rin, rout, s_out,
                              0, OC / 128, y);
    if (rc == EXL3O_OK)
        for (long m = 0; m < M; m++)
            for (int j = 0; j < OC; j++)
                out[m * ldo + col0 + j] = exl3o_bf16_from_f64(y[m * OC + j]);
    free(y);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* MoE routing and grouped experts                                           */
/* ------------------------------------------------------------------------ */

/* Top-k of each token's router logits (largest first, equal logits: lower
 * expert id first), weights = softmax over the k selected logits. */
int exl3o_topk_softmax(const float *logits, int T, int E, int topk,
                       int32_t *ids, float *w)
{
    if (T < 0 || E <= 0 || topk <= 0 || topk > E)
        return EXL3O_EINVAL;
    char *used = malloc((size_t)E);
    double *l = malloc(sizeof(double) * topk);
    for (int t = 0; t < T; t++) {
        memset(used, 0, (size_t)E);
        for (int k = 0; k < topk; k++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!used[e] && (best < 0 || logits[(long)t * E + e] > logits[(long)t * E + best]))
                    best = e;
            used[best] = 1;
            ids[(long)t * topk + k] = best;
            l[k] = logits[(long)t * E + best];
        }
        double mx = l[0], den = 0.0;
        for (int k = 0; k < topk; k++)
            den += exp(l[k] - mx);
        for (int k = 0; k < topk; k++)
            w[(long)t * topk + k] = (float)(exp(l[k] - mx) / den);
    }
    free(used);
    free(l);
    return EXL3O_OK;
}

/* y = Had(Had(x * pre) @ W) * post for one row; W is fp64 [IC][OC]. */
static void exl3_chain_row(const double *H, const double *xrow, int IC, int OC,
                           const double *W, const uint16_t *pre, const uint16_t *post,
                           double *out)
{
    double *xs = malloc(sizeof(double) * IC);
    double *u = malloc(sizeof(double) * IC);
    double *v = malloc(sizeof(double) * OC);
    double *hv = malloc(sizeof(double) * OC);
    for (int c = 0; c < IC; c++)
        xs[c] = xrow[c] * exl3o_f16_to_f64(pre[c]);
    had_blocks(H, xs, u, IC);
    for (int j = 0; j < OC; j++)
        v[j] = 0.0;
    for (int c = 0; c < IC; c++)
        for (int j = 0; j < OC; j++)
            v[j] += u[c] * W[(long)c * OC + j];
    had_blocks(H, v, hv, OC);
    for (int j = 0; j < OC; j++)
        out[j] = hv[j] * exl3o_f16_to_f64(post[j]);
    free(xs); free(u); free(v); free(hv);
}

static double *decode_dense(const int16_t *code, int IC, int OC, int K)
{
    uint16_t *Wh = malloc(sizeof(uint16_t) * (size_t)IC * OC);
    double *W = malloc(sizeof(double) * (size_t)IC * OC);
    exl3o_reconstruct(code, IC, OC, K, Wh);
    for (long i = 0; i < (long)IC * OC; i++)
        W[i] = exl3o_f16_to_f64(Wh[i]);
    free(Wh);
    return W;
}

/*
 * Grouped SiLU-gated MoE over an EXL3 expert bank ([bank] layout):
 *   slot p = perm[e] of logical expert e; its w1 / w3 code tensors
 *   [H/16][I/16][16*k_gu[p]] start at int16 word off_w1[p] / off_w3[p] of w13,
 *   its w2 code tensor [I/16][H/16][16*k_d[p]] at off_w2[p] of w2;
 *   w13_suh [E][2][H], w13_svh [E][2][I], w2_suh [E][I], w2_svh [E][H] (fp16,
 *   indexed by slot).
 * For each token t and each of its k = 0..topk-1 routes (e = ids[t][k]):
 *   g = Had(Had(x_t * w13_suh[p][0]) @ W1) * w13_svh[p][0]
 *   u = Had(Had(x_t * w13_suh[p][1]) @ W3) * w13_svh[p][1]
 *   h = silu(g) * u
 *   d = Had(Had(h * w2_suh[p]) @ W2) * w2_svh[p]
 * and y_t = sum over k in order 0..topk-1 of w[t][k] * d.  y is fp64 [T][H].
 * Rows are computed expert by expert (each expert decoded once); every (t, k)
 * term is independent, and the sum over k runs in k order afterwards.
 */
int exl3o_moe(const uint16_t *x, int T, int H, int I, int E, int topk,
              const int32_t *ids, const float *w,
              const int16_t *w13, const int16_t *w2,
              const int64_t *off_w1, const int64_t *off_w3, const int64_t *off_w2,
              const int32_t *perm, const int32_t *k_gu, const int32_t *k_d,
              const uint16_t *w13_suh, const uint16_t *w13_svh,
              const uint16_t *w2_suh, const uint16_t *w2_svh,
              double *y)
{
    if (T < 0 || H % 128 || I % 128 || E <= 0 || topk <= 0)
        return EXL3O_EINVAL;
    for (long i = 0; i < (long)T * topk; i++)
        if (ids[i] < 0 || ids[i] >= E)
            return EXL3O_EINVAL;
    double *H128 = malloc(sizeof(double) * 128 * 128);
    exl3o_hadamard128(H128);
    double *d = calloc((size_t)T * topk * H, sizeof(double));
    double *xd = malloc(sizeof(double) * (size_t)T * H);
    for (long i = 0; i < (long)T * H; i++)
        xd[i] = exl3o_bf16_to_f64(x[i]);

#pragma omp parallel for schedule(dynamic)
    for (int e = 0; e < E; e++) {
        int used = 0;
        for (long i = 0; i < (long)T * topk; i++)
            used |= (ids[i] == e);
        if (!used)
            continue;
        int p = perm[e];
        double *W1 = decode_dense(w13 + off_w1[p], H, I, k_gu[p]);
        double *W3 = decode_dense(w13 + off_w3[p], H, I, k_gu[p]);
        double *W2 = decode_dense(w2 + off_w2[p], I, H, k_d[p]);
        double *g = malloc(sizeof(double) * I);
        double *uu = malloc(sizeof(double) * I);
        for (long i = 0; i < (long)T * topk; i++) {
            if (ids[i] != e)
                continue;
            long t = i / topk;
            exl3_chain_row(H128, xd + t * H, H, I, W1, w13_suh + ((long)p * 2 + 0) * H,
                           w13_svh + ((long)p * 2 + 0) * I, g);
            exl3_chain_row(H128, xd + t * H, H, I, W3, w13_suh + ((long)p * 2 + 1) * H,
                           w13_svh + ((long)p * 2 + 1) * I, uu);
            for (int j = 0; j < I; j++)
                g[j] = (g[j] / (1.0 + exp(-g[j]))) * uu[j];
            exl3_chain_row(H128, g, I, H, W2, w2_suh + (long)p * I, w2_svh + (long)p * H,
                           d + i * H);
        }
        free(W1); free(W3); free(W2); free(g); free(uu);
    }
    for (long t = 0; t < T; t++)
        for (int j = 0; j < H; j++) {
            double acc = 0.0;
            for (int k = 0; k < topk; k++)
                acc += (double)w[t * topk + k] * d[(t * topk + k) * H + j];
            y[t * H + j] = acc;
        }
    free(d); free(xd); free(H128);
    return EXL3O_OK;
}

/* ------------------------------------------------------------------------ */
/* int8 embedding gather                                                     */
/* ------------------------------------------------------------------------ */

/*
 * [embed] out[i][:] = bf16(q[ids[i]][:] * s[ids[i]]): the int8 row converted
 * and multiplied by its fp16 scale on the gathered rows only.  The product of
 * an 8-bit integer and an fp16 scale is exact in fp64; it is rounded once.
 * An id outside [0, V) gives a row of zeros and is counted in *n_bad.
 */
int exl3o_gather(const int8_t *q, const uint16_t *s, long V, int H,
                 const int32_t *ids, long N, uint16_t *out, long *n_bad)
{
    if (V <= 0 || H <= 0 || N < 0)
        return EXL3O_EINVAL;
    long bad = 0;
    for (long i = 0; i < N; i++) {
        long id = ids[i];
        if (id < 0 || id >= V) {
            bad++;
            for (int j = 0; j < H; j++)
                out[i * H + j] = 0;
            continue;
        }
        double sc = exl3o_f16_to_f64(s[id]);
        for (int j = 0; j < H; j++)
            out[i * H + j] = exl3o_bf16_from_f64((double)q[id * H + j] * sc);
    }
    if (n_bad)
        *n_bad = bad;
    return EXL3O_OK;
}

/* ------------------------------------------------------------------ int8 output head
 * The int8 table used as the output projection (vllm-quantpack exl3/embedding.py,
 * Exl3EmbeddingMethod.apply: the linear layer's weight is the int8 table times its
 * per-row scale, w[v][h] = q[v][h] * s[v], and the head computes x @ w^T).
 * Reading: the per-row scale is factored out of the sum and the product is rounded
 * once, as the gather above does:
 *     y[m][v] = s[v] * sum_h x[m][h] * q[v][h]       (fp64, unrounded)
 * for vocabulary rows v in [v0, v0 + nv); y is [M][nv].  x is bf16 [M][H], q int8
 * [V][H] row-major, s fp16 [V].
 */
int exl3o_lm_head_f64(const uint16_t *x, long M, int H, const int8_t *q, const uint16_t *s, long V,
                      long v0, long nv, double *y)
{
    if (M < 0 || H <= 0 || V <= 0 || v0 < 0 || nv < 0 || v0 + nv > V)
        return EXL3O_EINVAL;
#pragma omp parallel for schedule(static)
    for (long v = v0; v < v0 + nv; v++) {
        const double sc = exl3o_f16_to_f64(s[v]);
        for (long m = 0; m < M; m++) {
            double acc = 0.0;
            for (int h = 0; h < H; h++)
                acc += exl3o_bf16_to_f64(x[m * H + h]) * (double)q[v * H + h];
            y[m * nv + (v - v0)] = sc * acc;
        }
    }
    return EXL3O_OK;
}

/* ------------------------------------------------------------------ 8-bit activations
 * The 8-bit activation variant ([escha] escha_linear_into: escha_pre_quant fills
 * an A buffer of uint8 [M][IC] with a float32 scale As [M] from a per-row amax
 * [M]; the pages give the buffers, not the encoding).  Reading: per row of the
 * pre-transformed activations u,
 *     amax = max_c |u[c]|,  As = amax / 127,
 *     q[c] = round_half_even(u[c] / As) clipped to [-127, 127]   (q = 0 if amax = 0)
 *     A[c] = q[c] + 128  (offset binary in a byte)
 * and the GEMM multiplies q * As in place of u:
 *     y = (Had128((q * As) @ decode(code)) * rout) * s_out.
 * Codes and scales are returned if the pointers are non-null (A [M][IC],
 * As [M]); y as in exl3o_linear_f64.
 */
int exl3o_quantize_a8(const double *u, long M, int IC, uint8_t *A, double *As)
{
    for (long m = 0; m < M; m++) {
        double amax = 0.0;
        for (int c = 0; c < IC; c++)
            if (fabs(u[m * IC + c]) > amax)
                amax = fabs(u[m * IC + c]);
        const double s = amax / 127.0;
        As[m] = s;
        for (int c = 0; c < IC; c++) {
            double q = 0.0;
            if (s > 0.0) {
                q = nearbyint(u[m * IC + c] / s);   /* default rounding mode: half to even */
                if (q > 127.0) q = 127.0;
                if (q < -127.0) q = -127.0;
            }
            A[m * IC + c] = (uint8_t)((int)q + 128);
        }
    }
    return EXL3O_OK;
}

int exl3o_linear_a8_f64(const uint16_t *x, long M, int IC,
                        const int16_t *code, int OC, int K,
                        const uint16_t *s_in, const uint16_t *rin,
                        const uint16_t *rout, const uint16_t *s_out,
                        int blk0, int nblk, double *y, uint8_t *A_out, double *As_out)
{
    if (!valid_k(K) || IC % 128 || OC % 128 || M < 0 || blk0 < 0 || nblk < 0 ||
        (long)(blk0 + nblk) * 128 > OC)
        return EXL3O_EINVAL;
    if (M == 0)
        return EXL3O_OK;
    int noc = nblk * 128, oc0 = blk0 * 128;
    double *u = malloc(sizeof(double) * (size_t)M * IC);
    uint8_t *A = malloc((size_t)M * IC);
    double *As = malloc(sizeof(double) * M);
    uint16_t *Wh = malloc(sizeof(uint16_t) * (size_t)IC * (noc > 0 ? noc : 1));
    double *W = malloc(sizeof(double) * (size_t)IC * (noc > 0 ? noc : 1));
    double *H = malloc(sizeof(double) * 128 * 128);
    if (!u || !A || !As || !Wh || !W || !H) {
        free(u); free(A); free(As); free(Wh); free(W); free(H);
        return EXL3O_EINVAL;
    }
    /* step 1: the activations, transformed, then quantized per row */
    exl3o_pretransform_f64(x, M, IC, s_in, rin, u);
    exl3o_quantize_a8(u, M, IC, A, As);
    if (A_out)
        memcpy(A_out, A, (size_t)M * IC);
    if (As_out)
        memcpy(As_out, As, sizeof(double) * M);
    if (noc > 0) {
        exl3o_hadamard128(H);
        exl3o_reconstruct_cols(code, IC, OC, K, oc0, noc, Wh);
        for (long i = 0; i < (long)IC * noc; i++)
            W[i] = exl3o_f16_to_f64(Wh[i]);
#pragma omp parallel for schedule(dynamic)
        for (long m = 0; m < M; m++) {
            double *v = malloc(sizeof(double) * noc);
            double *hv = malloc(sizeof(double) * noc);
            /* step 2: GEMM of the dequantized activations q * As */
            for (int j = 0; j < noc; j++)
                v[j] = 0.0;
            for (int c = 0; c < IC; c++) {
                const double uc = ((int)A[m * IC + c] - 128) * As[m];
                const double *wr = W + (long)c * noc;
                for (int j = 0; j < noc; j++)
                    v[j] += uc * wr[j];
            }
            /* step 3: output Hadamard, then rout, then s_out */
            had_blocks(H, v, hv, noc);
            for (int j = 0; j < noc; j++)
                y[m * noc + j] = (hv[j] * exl3o_f16_to_f64(rout[oc0 + j]))
                                 * exl3o_f16_to_f64(s_out[oc0 + j]);
            free(v); free(hv);
        }
    }
    free(u); free(A); free(As); free(Wh); free(W); free(H);
    return EXL3O_OK;
}
