/*
 * Double-precision CPU oracle for the Mamba2 decode-step selective state update.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this file;
 * only the tests, the package's smoke check and the bench's CPU-baseline leg use it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (sglang PR #41223 "Mamba2 selective_state_update up to 2x faster on B200",
 * sections Summary and Details / Kernel measurement, give the operands: an fp32 state pool
 * [pool, H, headdim, dstate] gathered through state_batch_indices and updated in place,
 * x [bs, H, headdim], B and C [bs, ngroups, dstate], per-head dt, A, D and dt_bias; the pages
 * never print the arithmetic, so the plainest reading of the standard Mamba2 decode step is
 * written out here):
 *
 *   for each request b with slot s = idx[b] and each head h (group g = h / (H / G)):
 *     dtv   = softplus(dt[b,h] + dt_bias[h])
 *     dA    = exp(dtv * A[h])
 *     S'[p,n] = S[s,h,p,n] * dA + (dtv * x[b,h,p]) * B[b,g,n]      (written back to slot s)
 *     y[b,h,p] = sum_n S'[p,n] * C[b,g,n] + D[h] * x[b,h,p]
 *
 * Every input arrives already widened to double (bf16 and fp32 values widen exactly), so the
 * whole computation is one rounding chain in IEEE double.  A request whose slot lies outside
 * [0, pool_size) is skipped: its slot and its outputs are left alone and it is counted.
 *
 * Parity pins (tests/test_oracle_pins.py): hand-computed 1x1x2 cases, x = 0 pure decay,
 * C = e_k selection, linearity in x and B, T sequential steps against the unrolled closed
 * form, head-to-group mapping, untouched slots, and bf16 round-to-nearest-even special cases.
 */
#include <math.h>
#include <stdint.h>

/* softplus(z) = log(1 + e^z).  Above z = 20 the difference from z is below 2.1e-9, and
 * exp(z) would only lose precision there, so z itself is returned. */
static double oracle_softplus(double z)
{
    if (z > 20.0)
        return z;
    return log1p(exp(z));
}

/*
 * One decode step over a batch.  All arrays are dense, row-major, double:
 *   pool     [pool_size, H, P, N]   updated in place for the slots idx[] names
 *   idx      [bs]                   int64 slot ids
 *   x        [bs, H, P]
 *   dt       [bs, H]
 *   dt_bias  [H], A [H], D [H]
 *   B, C     [bs, G, N]
 *   y        [bs, H, P]             output; NaN for skipped requests
 * Returns the number of skipped requests, or -1 when the shape is not valid.
 */
int64_t oracle_ssu_step(double *pool, int64_t pool_size, const int64_t *idx,
                        const double *x, const double *dt, const double *dt_bias,
                        const double *A, const double *B, const double *C, const double *D,
                        int64_t bs, int64_t H, int64_t P, int64_t N, int64_t G, double *y)
{
    if (bs < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0 || pool_size < 0)
        return -1;
    const int64_t heads_per_group = H / G;
    int64_t skipped = 0;

    for (int64_t b = 0; b < bs; ++b) {
        const int64_t s = idx[b];
        if (s < 0 || s >= pool_size) {
            for (int64_t i = 0; i < H * P; ++i)
                y[b * H * P + i] = NAN;
            ++skipped;
            continue;
        }
        for (int64_t h = 0; h < H; ++h) {
            const int64_t g = h / heads_per_group;
            const double dtv = oracle_softplus(dt[b * H + h] + dt_bias[h]);
            const double dA = exp(dtv * A[h]);
            const double *Bv = B + (b * G + g) * N;
            const double *Cv = C + (b * G + g) * N;
            double *S = pool + (s * H + h) * P * N;
            for (int64_t p = 0; p < P; ++p) {
                const double xp = x[(b * H + h) * P + p];
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double updated = S[p * N + n] * dA + (dtv * xp) * Bv[n];
                    S[p * N + n] = updated;
                    acc += updated * Cv[n];
                }
                y[(b * H + h) * P + p] = acc + D[h] * xp;
            }
        }
    }
    return skipped;
}

/*
 * Round doubles to bfloat16 (1 sign, 8 exponent, 7 stored mantissa bits) with
 * round-to-nearest, ties to even, in one rounding step.  Writes the 16-bit patterns.
 *
 * A finite |v| lies in a binade [2^e, 2^(e+1)) whose bf16 spacing is 2^(e-7); below the
 * smallest normal (2^-126) the spacing stays at the subnormal step 2^-133.  Dividing by
 * the spacing is exact (a power of two), rint() rounds to the nearest integer with ties to
 * even under the default rounding mode, and the product is a bf16 value (or 2^128, which
 * overflows to infinity).  Its float32 pattern then carries the bf16 pattern in the top
 * half exactly.
 */
void oracle_bf16_rne(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        const double a = v[i];
        const uint16_t sign = signbit(a) ? 0x8000u : 0u;
        if (isnan(a)) {
            out[i] = (uint16_t)(sign | 0x7FC0u);
            continue;
        }
        const double mag = fabs(a);
        if (isinf(a) || mag == 0.0) {
            out[i] = (uint16_t)(sign | (isinf(a) ? 0x7F80u : 0u));
            continue;
        }
        int e2;
        (void)frexp(mag, &e2); /* mag = f * 2^e2 with f in [0.5, 1): binade exponent e2 - 1 */
        int binade = e2 - 1;
        if (binade < -126)
            binade = -126;
        const double spacing = ldexp(1.0, binade - 7);
        const double rounded = rint(mag / spacing) * spacing;
        if (rounded >= ldexp(1.0, 128)) {
            out[i] = (uint16_t)(sign | 0x7F80u);
            continue;
        }
        union {
            float f;
            uint32_t u;
        } pun;
        pun.f = (float)rounded; /* exact: rounded is representable in bf16, hence in fp32 */
        out[i] = (uint16_t)(sign | (pun.u >> 16));
    }
}
