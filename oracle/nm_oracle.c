/*
 * nm_oracle.c -- CPU oracle for batched inference of the fused FP16 MLP.
 *
 * TEST INFRASTRUCTURE. This file is the slow, plain, single-threaded
 * statement of what the GPU path computes. Only tests/, the smoke check in
 * __graft_entry__.py and the CPU-baseline leg of bench.py may load it. The
 * product library (libnmmlp.so) never links, loads or calls it, and it shares
 * no code, header, table or constant with the CUDA sources.
 *
 * What it follows (page titles and sections of the source pages):
 *  - "Profiling neural material inference", section "Experiment setup": one
 *    evaluation runs the complete eight-affine-layer network E1/E2/E3/F/S/D/H/O
 *    on one input.
 *  - same page, "Bad versus good activation": the activation works on a half
 *    (FP16) vector, value = max(value, value * half(0.01)); the branchy per-lane
 *    form (if value < 0: value *= half(0.01)) is the same operation written
 *    lane by lane.
 *  - same page, "Row-major versus InferencingOptimal weights": the network
 *    consumes FP16 row-major matrices; a one-time conversion into an opaque
 *    device layout changes neither the network nor the activation.
 *  - "Working with Cooperative Matrices", "Hardware Constraints and
 *    Capabilities" (Precision Trade-offs): FP16 operands, FP32 accumulation.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *  - W_l is [N_l][K_l] row-major (rows = outputs) and y = W_l x + b_l.
 *  - Each dot product is summed in FP32 in increasing k; the bias is added in
 *    FP32 after the whole sum; the sum is rounded once to FP16 (round to
 *    nearest even, subnormals kept).
 *  - The activation follows every layer except the last and is applied to the
 *    FP16 value with the FP16 slope half(0.01) = 0x211F.
 *
 * The narrow-precision variant (or_mlp_forward_fp8, or_pack_fp8) follows
 * "Optimization Techniques: Squeezing the Silicon", chapter introduction (the
 * FP16/Quantization pillar), and the ninfer pull request #160 page (narrow
 * weight codes streamed to the tensor cores through a TMA ring). Neither page
 * fixes a format; the reading taken here: the weights of layers 2..L and the
 * hidden activations that feed them are rounded to OCP E4M3 (round to
 * nearest even, saturating at +-448, no scale), the first layer keeps its
 * FP16 inputs and weights, sums stay FP32 and biases FP16.
 *
 * The weight-packing reference (or_pack / or_unpack) writes the packed-blob
 * byte layout from its definition (stated beside or_packed_layout) so that
 * the GPU packer can be checked byte for byte. That layout is this library's
 * own choice of device-private format; the pages leave it implementation
 * defined.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
/* ------------------------------------------------------------------------ */

/* binary16 -> binary32. Every binary16 value is exactly representable in
 * binary32, so this is exact; NaN payloads are carried into the top fraction
 * bits. */
float or_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t e = (uint32_t)(h >> 10) & 0x1Fu;
    uint32_t f = (uint32_t)h & 0x3FFu;
    float mag;
    if (e == 31u) {
        uint32_t bits = (sign << 31) | 0x7F800000u | (f << 13);
        float r;
        memcpy(&r, &bits, sizeof r);
        return r;                                 /* infinity or NaN */
    }
    if (e == 0u)
        mag = ldexpf((float)f, -24);              /* zero or subnormal: f * 2^-24 */
    else
        mag = ldexpf((float)(1024u + f), (int)e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* Encode a non-negative value that is known to be representable in binary16
 * (or is >= 2^16, which encodes as infinity). */
static uint16_t encode_f16_magnitude(double v)
{
    int ex;
    double fr;
    if (v == 0.0)
        return 0;
    if (v < 0x1p-14)                              /* subnormal: v = f * 2^-24 */
        return (uint16_t)(v * 0x1p24);
    fr = frexp(v, &ex);                           /* v = fr * 2^ex, fr in [0.5, 1) */
    if (ex - 1 + 15 >= 31)
        return 0x7C00;
    return (uint16_t)(((uint32_t)(ex - 1 + 15) << 10) | (uint32_t)((2.0 * fr - 1.0) * 1024.0));
}

/* binary32 -> binary16, round to nearest, ties to even, subnormals kept.
 * The float is widened to double (exact), divided by the binary16 quantum of
 * its binade (exact: a power of two), rounded to an integer with rint (the
 * default rounding mode is nearest-even) and scaled back. */
uint16_t or_f32_to_f16(float x)
{
    uint32_t bits;
    uint16_t sign;
    double a, q, m;
    memcpy(&bits, &x, sizeof bits);
    sign = (uint16_t)((bits >> 16) & 0x8000u);
    if ((bits & 0x7F800000u) == 0x7F800000u) {
        if ((bits & 0x007FFFFFu) == 0)
            return (uint16_t)(sign | 0x7C00u);    /* infinity */
        return (uint16_t)(sign | 0x7E00u | ((bits >> 13) & 0x3FFu)); /* quiet NaN */
    }
    a = fabs((double)x);
    if (a >= 65520.0)                             /* halfway between 65504 and 2^16 and up */
        return (uint16_t)(sign | 0x7C00u);
    if (a < 0x1p-14) {
        q = 0x1p-24;                              /* subnormal spacing */
    } else {
        int ex;
        (void)frexp(a, &ex);                      /* a in [2^(ex-1), 2^ex) */
        q = ldexp(1.0, ex - 1 - 10);              /* 10 fraction bits */
    }
    m = rint(a / q);
    return (uint16_t)(sign | encode_f16_magnitude(m * q));
}

/* ------------------------------------------------------------------------ */
/* Activation ("Bad versus good activation")                                 */
/* ------------------------------------------------------------------------ */

/* half(0.01): the slope literal of the page's expression, converted to FP16. */
uint16_t or_slope_f16(void)
{
    return or_f32_to_f16(0.01f);
}

static int f16_is_nan(uint16_t h)
{
    return ((h & 0x7C00u) == 0x7C00u) && (h & 0x3FFu);
}

/* FP16 product: both factors have 11 significant bits, so the binary32
 * product is exact and one rounding to binary16 gives the correctly rounded
 * FP16 product. */
static uint16_t f16_mul(uint16_t a, uint16_t b)
{
    return or_f32_to_f16(or_f16_to_f32(a) * or_f16_to_f32(b));
}

/* IEEE maxNum on FP16 values: a NaN operand loses to a number. */
static uint16_t f16_max(uint16_t a, uint16_t b)
{
    if (f16_is_nan(a))
        return b;
    if (f16_is_nan(b))
        return a;
    return or_f16_to_f32(b) > or_f16_to_f32(a) ? b : a;
}

/* The good form: value = max(value, value * half(0.01)). */
uint16_t or_leaky_max(uint16_t h)
{
    return f16_max(h, f16_mul(h, or_slope_f16()));
}

/* The bad form, lane by lane: if (value < half(0)) value *= half(0.01). */
uint16_t or_leaky_branchy(uint16_t h)
{
    if (or_f16_to_f32(h) < 0.0f)
        return f16_mul(h, or_slope_f16());
    return h;
}

/* ------------------------------------------------------------------------ */
/* The network ("Experiment setup": one evaluation = the full layer chain)   */
/* ------------------------------------------------------------------------ */

#define OR_MAX_LAYERS 16
#define OR_MAX_DIM 256

/* dims[0..n_layers]: d_0 (inputs) ... d_L (outputs). W[l] is [d_{l+1}][d_l]
 * row-major FP16 bits, b[l] has d_{l+1} FP16 entries. x is [n][d_0] row-major,
 * y is [n][d_L] row-major. Returns 0, or -1 for dims outside 1..256 or more
 * than 16 layers. */
int or_mlp_forward(const int32_t *dims, int32_t n_layers,
                   const uint16_t *const *W, const uint16_t *const *b,
                   const uint16_t *x, int64_t n, uint16_t *y)
{
    float *Wf[OR_MAX_LAYERS];
    float *bf[OR_MAX_LAYERS];
    float cur[OR_MAX_DIM];
    uint16_t nxt[OR_MAX_DIM];
    int32_t l;
    int64_t i;
    int rc = 0;

    if (n_layers < 1 || n_layers > OR_MAX_LAYERS)
        return -1;
    for (l = 0; l <= n_layers; ++l)
        if (dims[l] < 1 || dims[l] > OR_MAX_DIM)
            return -1;
    for (l = 0; l < n_layers; ++l)
        Wf[l] = bf[l] = NULL;

    /* Widen the weights and biases once (exact). */
    for (l = 0; l < n_layers; ++l) {
        int32_t K = dims[l], N = dims[l + 1], j;
        Wf[l] = (float *)malloc(sizeof(float) * (size_t)K * (size_t)N);
        bf[l] = (float *)malloc(sizeof(float) * (size_t)N);
        if (!Wf[l] || !bf[l]) {
            rc = -2;
            goto done;
        }
        for (j = 0; j < K * N; ++j)
            Wf[l][j] = or_f16_to_f32(W[l][j]);
        for (j = 0; j < N; ++j)
            bf[l][j] = or_f16_to_f32(b[l][j]);
    }

    for (i = 0; i < n; ++i) {
        int32_t k;
        for (k = 0; k < dims[0]; ++k)
            cur[k] = or_f16_to_f32(x[i * dims[0] + k]);
        for (l = 0; l < n_layers; ++l) {
            int32_t K = dims[l], N = dims[l + 1], o;
            for (o = 0; o < N; ++o) {
                const float *w = Wf[l] + (size_t)o * (size_t)K;
                float acc = 0.0f;
                float v;
                uint16_t h;
                for (k = 0; k < K; ++k)
                    acc = acc + cur[k] * w[k];    /* FP32, increasing k */
                v = acc + bf[l][o];               /* bias in FP32 after the sum */
                h = or_f32_to_f16(v);             /* one rounding to FP16 */
                if (l < n_layers - 1)
                    h = or_leaky_max(h);          /* no activation after the last */
                nxt[o] = h;
            }
            if (l < n_layers - 1)
                for (o = 0; o < N; ++o)
                    cur[o] = or_f16_to_f32(nxt[o]);
        }
        memcpy(y + i * dims[n_layers], nxt, sizeof(uint16_t) * (size_t)dims[n_layers]);
    }
done:
    for (l = 0; l < n_layers; ++l) {
        free(Wf[l]);
        free(bf[l]);
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* OCP 8-bit float E4M3 (the "FN" encoding): 1 sign bit, 4 exponent bits     */
/* (bias 7), 3 fraction bits; no infinities; S.1111.111 is NaN; the largest  */
/* finite magnitude is 1.75 * 2^8 = 448; exponent field 0 holds the          */
/* subnormals f * 2^-9.                                                      */
/* ------------------------------------------------------------------------ */

float or_e4m3_to_f32(uint8_t c)
{
    uint32_t sign = (uint32_t)(c >> 7) & 1u;
    uint32_t e = (uint32_t)(c >> 3) & 0xFu;
    uint32_t f = (uint32_t)c & 0x7u;
    float mag;
    if (e == 15u && f == 7u)
        return sign ? -NAN : NAN;
    if (e == 0u)
        mag = ldexpf((float)f, -9);                    /* f/8 * 2^-6 */
    else
        mag = ldexpf((float)(8u + f), (int)e - 10);    /* (1 + f/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* Encode a non-negative multiple of the E4M3 quantum of its binade, at most
 * 448. */
static uint8_t encode_e4m3_magnitude(double v)
{
    int ex;
    double fr;
    if (v < 0x1p-6)                                    /* subnormal (or zero) */
        return (uint8_t)(v * 0x1p9);
    fr = frexp(v, &ex);                                /* v = fr * 2^ex */
    return (uint8_t)(((uint32_t)(ex - 1 + 7) << 3) | (uint32_t)((2.0 * fr - 1.0) * 8.0));
}

/* binary16 -> E4M3: round to nearest, ties to even; magnitudes that round
 * above 448, and infinities (E4M3 has none), saturate to 448; NaN gives the
 * NaN code with the input's sign. Same quantum scaling as or_f32_to_f16. */
uint8_t or_f16_to_e4m3(uint16_t h)
{
    uint8_t sign = (uint8_t)((h >> 8) & 0x80u);
    double a, q, m;
    if ((h & 0x7C00u) == 0x7C00u)
        return (uint8_t)(sign | ((h & 0x3FFu) ? 0x7Fu : 0x7Eu));
    a = fabs((double)or_f16_to_f32(h));
    if (a < 0x1p-6) {
        q = 0x1p-9;                                    /* subnormal spacing */
    } else {
        int ex;
        (void)frexp(a, &ex);
        q = ldexp(1.0, ex - 1 - 3);                    /* 3 fraction bits */
    }
    m = rint(a / q) * q;
    if (m > 448.0)
        m = 448.0;
    return (uint8_t)(sign | encode_e4m3_magnitude(m));
}

/* The narrow-precision forward pass. Layer 1 is the FP16 layer of
 * or_mlp_forward. Every later layer l: the weights are E4M3(W_l); the
 * activation it reads is E4M3 of the FP16 activation of the layer before;
 * the dot product is summed in FP32 in increasing k (each E4M3 x E4M3
 * product is exact in FP32), the FP16 bias is added in FP32 after the sum,
 * and the result is rounded once to FP16 (then, for hidden layers, the FP16
 * activation as in or_mlp_forward). Requires n_layers >= 2. Returns 0, -1
 * for dims outside 1..256 or a depth outside 2..16, -2 on allocation
 * failure. */
int or_mlp_forward_fp8(const int32_t *dims, int32_t n_layers,
                       const uint16_t *const *W, const uint16_t *const *b,
                       const uint16_t *x, int64_t n, uint16_t *y)
{
    float *Wf[OR_MAX_LAYERS];
    float *bf[OR_MAX_LAYERS];
    float cur[OR_MAX_DIM];
    uint16_t nxt[OR_MAX_DIM];
    int32_t l;
    int64_t i;
    int rc = 0;

    if (n_layers < 2 || n_layers > OR_MAX_LAYERS)
        return -1;
    for (l = 0; l <= n_layers; ++l)
        if (dims[l] < 1 || dims[l] > OR_MAX_DIM)
            return -1;
    for (l = 0; l < n_layers; ++l)
        Wf[l] = bf[l] = NULL;

    for (l = 0; l < n_layers; ++l) {
        int32_t K = dims[l], N = dims[l + 1], j;
        Wf[l] = (float *)malloc(sizeof(float) * (size_t)K * (size_t)N);
        bf[l] = (float *)malloc(sizeof(float) * (size_t)N);
        if (!Wf[l] || !bf[l]) {
            rc = -2;
            goto done;
        }
        for (j = 0; j < K * N; ++j)
            Wf[l][j] = (l == 0) ? or_f16_to_f32(W[l][j]) : or_e4m3_to_f32(or_f16_to_e4m3(W[l][j]));
        for (j = 0; j < N; ++j)
            bf[l][j] = or_f16_to_f32(b[l][j]);
    }

    for (i = 0; i < n; ++i) {
        int32_t k;
        for (k = 0; k < dims[0]; ++k)
            cur[k] = or_f16_to_f32(x[i * dims[0] + k]);
        for (l = 0; l < n_layers; ++l) {
            int32_t K = dims[l], N = dims[l + 1], o;
            for (o = 0; o < N; ++o) {
                const float *w = Wf[l] + (size_t)o * (size_t)K;
                float acc = 0.0f;
                uint16_t h;
                for (k = 0; k < K; ++k)
                    acc = acc + cur[k] * w[k];         /* FP32, increasing k */
                h = or_f32_to_f16(acc + bf[l][o]);     /* bias, then one rounding */
                if (l < n_layers - 1)
                    h = or_leaky_max(h);
                nxt[o] = h;
            }
            if (l < n_layers - 1)                      /* the next layer reads E4M3 */
                for (o = 0; o < N; ++o)
                    cur[o] = or_e4m3_to_f32(or_f16_to_e4m3(nxt[o]));
        }
        memcpy(y + i * dims[n_layers], nxt, sizeof(uint16_t) * (size_t)dims[n_layers]);
    }
done:
    for (l = 0; l < n_layers; ++l) {
        free(Wf[l]);
        free(bf[l]);
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Packed weight blob: reference packer written from the layout definition  */
/* ------------------------------------------------------------------------ */
/*
 * Layout definition (device-private format of this library):
 *  - The blob holds one weight image per layer, then one bias block.
 *  - Layer l's image starts at a multiple of 1024 bytes. With K = d_l and
 *    N = d_{l+1}, the k range [0, K) is cut, from k = 0 upward, into segments
 *    of width 64 while at least 64 columns remain, then one of width 32 if at
 *    least 32 remain, then one of width 16 if 16 remain (K is a multiple of 16).
 *  - Each segment of width w and first column k0 starts at a multiple of 1024
 *    bytes and spans N * 2w bytes. Element W[n][k] (k0 <= k < k0 + w) has the
 *    plain offset p = n * 2w + 2 (k - k0) inside its segment and is stored at
 *    p XOR (((p >> 7) & m) << 4), with m = 7, 3, 1 for w = 64, 32, 16.
 *  - The bias block starts at the next multiple of 1024 bytes after the last
 *    image and holds b_0, b_1, ..., b_{L-1} back to back as FP16.
 *  - All other bytes are zero. The blob size is the end of the bias block.
 */

static int seg_count(int32_t K, int32_t *w_out, int32_t *k0_out)
{
    int32_t k0 = 0, ns = 0;
    while (K - k0 >= 64) {
        w_out[ns] = 64;
        k0_out[ns++] = k0;
        k0 += 64;
    }
    if (K - k0 >= 32) {
        w_out[ns] = 32;
        k0_out[ns++] = k0;
        k0 += 32;
    }
    if (K - k0 >= 16) {
        w_out[ns] = 16;
        k0_out[ns++] = k0;
        k0 += 16;
    }
    return (k0 == K) ? ns : -1;
}

static int64_t round_up(int64_t v, int64_t a)
{
    return (v + a - 1) / a * a;
}

/* Fills image_off[l] (byte offset of layer l's image), *bias_off and returns
 * the blob size, or -1 for dims that are not multiples of 16 in 16..256. */
int64_t or_packed_layout(const int32_t *dims, int32_t n_layers, int64_t *image_off, int64_t *bias_off)
{
    int64_t off = 0, nb = 0;
    int32_t l;
    if (n_layers < 1 || n_layers > OR_MAX_LAYERS)
        return -1;
    for (l = 0; l <= n_layers; ++l)
        if (dims[l] < 16 || dims[l] > OR_MAX_DIM || dims[l] % 16)
            return -1;
    for (l = 0; l < n_layers; ++l) {
        int32_t w[16], k0[16], ns, s;
        ns = seg_count(dims[l], w, k0);
        off = round_up(off, 1024);
        image_off[l] = off;
        for (s = 0; s < ns; ++s) {
            off = round_up(off, 1024);
            off += (int64_t)dims[l + 1] * 2 * w[s];
        }
        nb += dims[l + 1];
    }
    off = round_up(off, 1024);
    *bias_off = off;
    return off + 2 * nb;
}

static int64_t swizzle(int64_t p, int32_t w)
{
    int64_t m = (w == 64) ? 7 : (w == 32) ? 3 : 1;
    return p ^ (((p >> 7) & m) << 4);
}

/* Position of W_l[n][k] inside the blob. */
static int64_t packed_pos(const int32_t *dims, int64_t image_off, int32_t l, int32_t n, int32_t k)
{
    int32_t w[16], k0[16], ns, s;
    int64_t seg_off = image_off;
    ns = seg_count(dims[l], w, k0);
    for (s = 0; s < ns; ++s) {
        seg_off = round_up(seg_off, 1024);
        if (k < k0[s] + w[s])
            return seg_off + swizzle((int64_t)n * 2 * w[s] + 2 * (int64_t)(k - k0[s]), w[s]);
        seg_off += (int64_t)dims[l + 1] * 2 * w[s];
    }
    return -1;
}

int or_pack(const int32_t *dims, int32_t n_layers, const uint16_t *const *W,
            const uint16_t *const *b, uint8_t *blob)
{
    int64_t image_off[OR_MAX_LAYERS], bias_off, size, bpos;
    int32_t l;
    size = or_packed_layout(dims, n_layers, image_off, &bias_off);
    if (size < 0)
        return -1;
    memset(blob, 0, (size_t)size);
    bpos = bias_off;
    for (l = 0; l < n_layers; ++l) {
        int32_t K = dims[l], N = dims[l + 1], n, k;
        for (n = 0; n < N; ++n)
            for (k = 0; k < K; ++k) {
                int64_t p = packed_pos(dims, image_off[l], l, n, k);
                uint16_t v = W[l][(size_t)n * (size_t)K + (size_t)k];
                blob[p] = (uint8_t)(v & 0xFFu);   /* little-endian FP16 */
                blob[p + 1] = (uint8_t)(v >> 8);
            }
        for (n = 0; n < N; ++n) {
            blob[bpos] = (uint8_t)(b[l][n] & 0xFFu);
            blob[bpos + 1] = (uint8_t)(b[l][n] >> 8);
            bpos += 2;
        }
    }
    return 0;
}

int or_unpack(const int32_t *dims, int32_t n_layers, const uint8_t *blob,
              uint16_t *const *W, uint16_t *const *b)
{
    int64_t image_off[OR_MAX_LAYERS], bias_off, bpos;
    int32_t l;
    if (or_packed_layout(dims, n_layers, image_off, &bias_off) < 0)
        return -1;
    bpos = bias_off;
    for (l = 0; l < n_layers; ++l) {
        int32_t K = dims[l], N = dims[l + 1], n, k;
        for (n = 0; n < N; ++n)
            for (k = 0; k < K; ++k) {
                int64_t p = packed_pos(dims, image_off[l], l, n, k);
                W[l][(size_t)n * (size_t)K + (size_t)k] = (uint16_t)(blob[p] | (blob[p + 1] << 8));
            }
        for (n = 0; n < N; ++n) {
            b[l][n] = (uint16_t)(blob[bpos] | (blob[bpos + 1] << 8));
            bpos += 2;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* E4M3 weight images of the narrow-precision variant                        */
/* ------------------------------------------------------------------------ */
/*
 * Layout definition (device-private, separate from the FP16 blob):
 *  - One image per layer l = 1 .. L-1 (0-based; layer 0 has none), in that
 *    order, each starting at a multiple of 1024 bytes from the start of the
 *    region. With K = d_l and N = d_{l+1} (K a multiple of 32), the k range
 *    is cut from k = 0 upward into segments of width 128 while at least 128
 *    columns remain, then one of 64 if at least 64 remain, then one of 32 if
 *    32 remain.
 *  - Each segment of width w starts at a multiple of 1024 bytes and spans
 *    N * w bytes. E4M3(W[n][k]) (k0 <= k < k0 + w) has the plain offset
 *    p = n * w + (k - k0) inside its segment and is stored at
 *    p XOR (((p >> 7) & m) << 4), with m = 7, 3, 1 for w = 128, 64, 32.
 *  - All other bytes are zero; the region ends at the end of the last image.
 */

static int seg_count_fp8(int32_t K, int32_t *w_out, int32_t *k0_out)
{
    int32_t k0 = 0, ns = 0;
    while (K - k0 >= 128) {
        w_out[ns] = 128;
        k0_out[ns++] = k0;
        k0 += 128;
    }
    if (K - k0 >= 64) {
        w_out[ns] = 64;
        k0_out[ns++] = k0;
        k0 += 64;
    }
    if (K - k0 >= 32) {
        w_out[ns] = 32;
        k0_out[ns++] = k0;
        k0 += 32;
    }
    return (k0 == K) ? ns : -1;
}

/* Fills image_off[l] for l = 1 .. L-1 (image_off[0] = -1) and returns the
 * region size, or -1 for a depth outside 2..16 or widths that are not
 * multiples of 16 in 16..256 with hidden widths (d_1 .. d_{L-1}) multiples
 * of 32. */
int64_t or_fp8_layout(const int32_t *dims, int32_t n_layers, int64_t *image_off)
{
    int64_t off = 0;
    int32_t l;
    if (n_layers < 2 || n_layers > OR_MAX_LAYERS)
        return -1;
    for (l = 0; l <= n_layers; ++l)
        if (dims[l] < 16 || dims[l] > OR_MAX_DIM || dims[l] % 16)
            return -1;
    for (l = 1; l < n_layers; ++l)
        if (dims[l] % 32)
            return -1;
    image_off[0] = -1;
    for (l = 1; l < n_layers; ++l) {
        int32_t w[16], k0[16], ns, s;
        ns = seg_count_fp8(dims[l], w, k0);
        off = round_up(off, 1024);
        image_off[l] = off;
        for (s = 0; s < ns; ++s) {
            off = round_up(off, 1024);
            off += (int64_t)dims[l + 1] * w[s];
        }
    }
    return off;
}

static int64_t swizzle_fp8(int64_t p, int32_t w)
{
    int64_t m = (w == 128) ? 7 : (w == 64) ? 3 : 1;
    return p ^ (((p >> 7) & m) << 4);
}

int or_pack_fp8(const int32_t *dims, int32_t n_layers, const uint16_t *const *W, uint8_t *region)
{
    int64_t image_off[OR_MAX_LAYERS], size;
    int32_t l;
    size = or_fp8_layout(dims, n_layers, image_off);
    if (size < 0)
        return -1;
    memset(region, 0, (size_t)size);
    for (l = 1; l < n_layers; ++l) {
        int32_t K = dims[l], N = dims[l + 1], w[16], k0[16], ns, s, n, k;
        int64_t seg_off = image_off[l];
        ns = seg_count_fp8(K, w, k0);
        for (s = 0; s < ns; ++s) {
            seg_off = round_up(seg_off, 1024);
            for (n = 0; n < N; ++n)
                for (k = k0[s]; k < k0[s] + w[s]; ++k)
                    region[seg_off + swizzle_fp8((int64_t)n * w[s] + (k - k0[s]), w[s])] =
                        or_f16_to_e4m3(W[l][(size_t)n * (size_t)K + (size_t)k]);
            seg_off += (int64_t)N * w[s];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Array forms of the scalar functions above (plain loops, for tests).       */
/* ------------------------------------------------------------------------ */

void or_f16_to_f32_n(const uint16_t *h, int64_t n, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_f16_to_f32(h[i]);
}

void or_f32_to_f16_n(const float *x, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_f32_to_f16(x[i]);
}

void or_leaky_max_n(const uint16_t *h, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_leaky_max(h[i]);
}

void or_leaky_branchy_n(const uint16_t *h, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_leaky_branchy(h[i]);
}

void or_e4m3_to_f32_n(const uint8_t *c, int64_t n, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_e4m3_to_f32(c[i]);
}

void or_f16_to_e4m3_n(const uint16_t *h, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_f16_to_e4m3(h[i]);
}
