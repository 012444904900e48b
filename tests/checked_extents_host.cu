// Host-side check of the extent arithmetic the checked library runs before each
// device access (row_in_range in csrc/common.cuh): built and run by
// tests/test_checked_mode.py with nvcc, no GPU needed.  Prints one line per
// failed expectation and exits non-zero if any failed.
#include <cstdio>

#include "common.cuh"

using gbattn::row_in_range;

static int fails = 0;
static void expect(bool got, bool want, const char* what) {
  if (got != want) {
    std::printf("FAIL %s: got %d, want %d\n", what, (int)got, (int)want);
    ++fails;
  }
}

int main() {
  // fixed length: batch 2, seqlen 300, 4 heads
  expect(row_in_range(0, 2, 300, 0, 4, 0, 0, 0, 0), true, "first row");
  expect(row_in_range(0, 2, 300, 0, 4, 1, 3, 0, 299), true, "last row of the last head and batch entry");
  expect(row_in_range(0, 2, 300, 0, 4, 1, 3, 0, 300), false, "one row past the sequence");
  expect(row_in_range(0, 2, 300, 0, 4, 2, 0, 0, 0), false, "batch entry past the batch");
  expect(row_in_range(0, 2, 300, 0, 4, -1, 0, 0, 0), false, "negative batch entry");
  expect(row_in_range(0, 2, 300, 0, 4, 0, 4, 0, 0), false, "head past the heads");
  expect(row_in_range(0, 2, 300, 0, 4, 0, -1, 0, 0), false, "negative head");
  expect(row_in_range(0, 2, 300, 0, 4, 0, 0, 0, -1), false, "negative position");
  expect(row_in_range(0, 0, 300, 0, 4, 0, 0, 0, 0), false, "empty batch");
  // packed variable length: 1000 tokens, 2 heads; the sequence at token 900 has 100 rows
  expect(row_in_range(1, 0, 512, 1000, 2, 0, 1, 900, 99), true, "last token of the packed tensor");
  expect(row_in_range(1, 0, 512, 1000, 2, 0, 1, 900, 100), false, "one token past the packed tensor");
  expect(row_in_range(1, 0, 512, 1000, 2, 1, 0, 0, 0), false, "packed tensors have one batch entry");
  expect(row_in_range(1, 0, 512, 1000, 2, 0, 0, 0, 999), true, "a row past seqlen is fine when packed");
  expect(row_in_range(1, 0, 512, 1000, 2, 0, 2, 0, 0), false, "head past the heads (packed)");
  // positions beyond 32 bits of tokens do not wrap
  expect(row_in_range(1, 0, 512, 3000000000LL, 1, 0, 0, 2999999999LL, 0), true, "64-bit token index");
  expect(row_in_range(1, 0, 512, 3000000000LL, 1, 0, 0, 2999999999LL, 1), false, "64-bit token index past the end");
  if (fails == 0) std::printf("ok\n");
  return fails == 0 ? 0 : 1;
}
