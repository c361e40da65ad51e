/* Exhaustive check behind the GPU E4M3 quantiser's division.
 *
 * The blockwise FP8 recipe ("Scalable Training of Mixture-of-Experts Models
 * with Megatron Core", §5, blockwise FP8) stores a value v of a block with
 * maximum magnitude amax as q = E4M3(RN(v / s)), s = RN(amax / 448), all in
 * fp32 (E4M3: nearest code, ties to even, saturating at 448). The GPU forms
 * the quotient without a division, by Markstein's correction of the product
 * with the rounded reciprocal r = RN(1 / s) (P. Markstein, IBM J. Res. Dev.
 * 34(1), 1990):  y0 = RN(v r),  y1 = RN(y0 + r RN(v - s y0)).
 * The layer quantises bf16 tensors, so v and amax are bf16 numbers. This
 * program walks every positive finite bf16 amax with s >= 2^-112 and every
 * bf16 v in [0, amax] (the negative half is the mirror image: every step is
 * sign-symmetric) and counts the pairs where E4M3(y1) != E4M3(RN(v / s)).
 * Build with -ffp-contract=off (each multiply and add rounded as written;
 * fmaf is the correctly rounded fused multiply-add). Prints the counts and
 * exits 1 on any difference. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bf16(uint32_t h)
{
    uint32_t u = h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Nearest E4M3 value of y >= 0 (ties to the even mantissa), saturating at 448. */
static float e4m3_value(float y)
{
    if (y != y) return y;
    if (y >= 448.0f) return 448.0f;
    if (y < 0x1p-6f) return nearbyintf(y * 512.0f) / 512.0f; /* subnormal step 2^-9 */
    uint32_t b;
    memcpy(&b, &y, 4);
    b = (b + 0x7FFFFu + ((b >> 20) & 1u)) & ~0xFFFFFu;      /* keep 3 mantissa bits */
    float r;
    memcpy(&r, &b, 4);
    return r > 448.0f ? 448.0f : r;
}

int main(void)
{
    long long pairs = 0, diff = 0, blocks = 0;
    for (uint32_t ha = 1; ha < 0x7F80u; ++ha) {
        const float amax = from_bf16(ha);
        const float s = amax / 448.0f;
        if (s < 0x1p-112f) continue;
        const float r = 1.0f / s;
        ++blocks;
        for (uint32_t hv = 0; hv <= ha; ++hv) {
            const float v = from_bf16(hv);
            const float y0 = v * r;
            const float y1 = fmaf(fmaf(-s, y0, v), r, y0);
            const float q = v / s;
            ++pairs;
            if (e4m3_value(y1) != e4m3_value(q)) {
                if (diff < 5) printf("difference: amax=%a v=%a s=%a y1=%a v/s=%a\n", amax, v, s, y1, q);
                ++diff;
            }
        }
    }
    printf("block maxima %lld, pairs %lld, E4M3 differences %lld\n", blocks, pairs, diff);
    return diff == 0 ? 0 : 1;
}
