// Host driver for the fixed-point helpers of the filter kernels: reads
// "f <hex float bits>" and "t <hex float bits> <decimal S>" lines on stdin
// and prints f2ull_rn / mass_target results, one per line.
#include <cstdio>
#include <cstring>

#include "common.cuh"

int main() {
  char op[8];
  while (scanf("%7s", op) == 1) {
    unsigned int bits = 0;
    if (scanf("%x", &bits) != 1) return 1;
    float f;
    memcpy(&f, &bits, sizeof f);
    if (strcmp(op, "f") == 0) {
      printf("%llu\n", topkp::f2ull_rn(f));
    } else {
      unsigned long long S = 0;
      if (scanf("%llu", &S) != 1) return 1;
      printf("%llu\n", topkp::mass_target(f, S));
    }
  }
  return 0;
}
