/* Checks, with IEEE binary32 arithmetic on the host (fmaf, no contraction),
 * the two division methods the fast quantizer kernel uses instead of div.rn:
 *   BMR: RN(y zh + RN(y zl)) with zh = RD(1/d), zl = RN(1/d - zh)
 *        (Brisebarre, Muller, Raina, IEEE Trans. Computers 2004)
 *   Markstein: q = RN(u r), e = RN(q S - u), RN(q - e r) with r = RN(1/S)
 * against the correctly rounded quotient y / d.  Arguments: the kernel's
 * table constants (hex), so the check runs on the values the kernel holds.
 * Usage: check <stride> <hi_1> <lo_1> ... <hi_15> <lo_15> <hi_21> <lo_21>  */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float bf(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t fb(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

int main(int argc, char **argv) {
  if (argc != 2 + 2 * 16) return 2;
  uint32_t stride = (uint32_t)strtoul(argv[1], 0, 10);
  long bad = 0, n = 0;
  for (int i = 0; i < 16; i++) {
    int M = i < 15 ? i + 1 : 21;
    uint32_t hi = (uint32_t)strtoul(argv[2 + 2 * i], 0, 16), lo = (uint32_t)strtoul(argv[3 + 2 * i], 0, 16);
    for (int ex = -17; ex <= 15; ex += 8) {          /* divisor M * 2^ex, table scaled by 2^-ex */
      float d = ldexpf((float)M, ex);
      float zh = ldexpf(bf(hi), -ex), zl = ldexpf(bf(lo), -ex);
      for (int ey = -2; ey <= 2; ey += 2) {
        for (uint32_t m = 0; m < (1u << 23); m += stride) {
          float y = ldexpf(bf(0x3F800000u | m), ex + ey);
          for (int sgn = 0; sgn < 2; sgn++, y = -y) {
            float q = fmaf(y, zh, y * zl);
            n++;
            if (fb(q) != fb(y / d)) bad++;
          }
        }
      }
    }
    float z = fmaf(-0.0f, bf(hi), -0.0f * bf(lo));
    if (fb(z) != 0x80000000u) { printf("sign of zero lost for M=%d\n", M); bad++; }
  }
  printf("bmr %ld of %ld wrong\n", bad, n);
  long bad2 = 0, n2 = 0;
  srand(12345);
  for (int k = 0; k < 64; k++) {
    uint32_t e = 2 + (uint32_t)(k % 16) * 15;
    float S = bf((e << 23) | (((uint32_t)rand() << 12 ^ (uint32_t)rand()) & 0x7FFFFFu));
    float r = 1.0f / S;
    for (int eu = -8; eu <= 8; eu += 8) {
      int ue = (int)e + eu;
      if (ue < 1 || ue > 254) continue;
      for (uint32_t m = 0; m < (1u << 23); m += stride) {
        float u = bf(((uint32_t)ue << 23) | m);
        float ref = u / S;
        if (isinf(ref) || fabsf(u) < ldexpf(1.0f, -100)) continue;
        for (int sgn = 0; sgn < 2; sgn++, u = -u, ref = -ref) {
          float q = u * r;
          float er = fmaf(q, S, -u);
          float x = fmaf(er, -r, q);
          n2++;
          if (fb(x) != fb(ref)) bad2++;
        }
      }
    }
    float zs = -0.0f, q = zs * r, er = fmaf(q, S, -zs), x = fmaf(er, -r, q);
    if (fb(x) != 0x80000000u) { printf("markstein lost the sign of -0\n"); bad2++; }
  }
  printf("markstein %ld of %ld wrong\n", bad2, n2);
  return (bad || bad2) ? 1 : 0;
}
