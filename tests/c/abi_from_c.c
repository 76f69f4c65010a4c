/* A C11 client of the TreeWY C ABI: checks that include/treewy.h compiles as
 * plain C and that the library's host-side validation answers through the
 * declared entry points.  It makes no call that reaches the GPU (every batch
 * below fails validation before any launch). */
#include <stdio.h>
#include <string.h>

#include "treewy.h"

static int fails = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    fprintf(stderr, "FAILED: %s (last error: %s)\n", what, treewy_last_error());
    ++fails;
  }
}

int main(void) {
  expect(strstr(treewy_version(), "sm_103a") != NULL, "version names sm_103a");
  expect(treewy_verify(NULL, 0) == TREEWY_ERR_INVALID_ARG, "NULL batch rejected");
  expect(treewy_selftest_wait_timeout(NULL, 1000, 0) == TREEWY_ERR_INVALID_ARG,
         "wait self-test without a status word rejected");

  treewy_batch b;
  memset(&b, 0, sizeof b);
  b.R = 2;
  b.H = 4;
  b.dk = 256; /* above the supported head size */
  b.dv = 128;
  b.max_nodes = 64;
  b.qkv_dtype = TREEWY_DTYPE_BF16;
  b.T = 10;
  b.num_slots = 2;
  expect(treewy_verify(&b, 0) == TREEWY_ERR_UNSUPPORTED, "dk = 256 unsupported");
  expect(strlen(treewy_last_error()) > 0, "error message set");

  b.dk = 128;
  expect(treewy_commit(&b, NULL, 0) == TREEWY_ERR_INVALID_ARG, "commit without pointers rejected");

  /* aligned placeholders: never dereferenced, every call below fails
     validation before any launch */
  void* fake = (void*)(size_t)0x10000;
  b.node_offset = (const int32_t*)fake;
  b.parent = (const int32_t*)fake;
  b.q = b.k = b.v = fake;
  b.alpha = b.beta = (const float*)fake;
  b.state = fake;
  b.state_slot = (const int32_t*)fake;
  b.o = b.U = (float*)fake;
  b.status = (int32_t*)fake;
  b.flags = TREEWY_FLAG_STATE_BF16;
  expect(treewy_storeall_verify(&b, (float*)fake, 0) == TREEWY_ERR_UNSUPPORTED,
         "storeall rejects a bf16 state pool");
  expect(treewy_commit(&b, NULL, 0) == TREEWY_ERR_INVALID_ARG, "commit without accepted rejected");
  b.flags = 4; /* no such flag */
  expect(treewy_verify(&b, 0) == TREEWY_ERR_INVALID_ARG, "unknown flag rejected");
  b.flags = 0;
  b.state = (void*)(size_t)0x10004; /* misaligned */
  expect(treewy_verify(&b, 0) == TREEWY_ERR_INVALID_ARG, "misaligned state rejected");

  b.R = 0; /* an empty batch is a no-op */
  b.flags = 0;
  expect(treewy_verify(&b, 0) == TREEWY_OK, "empty batch accepted");
  expect(treewy_last_error()[0] == '\0', "no error after success");

  if (fails == 0) printf("c abi ok\n");
  return fails ? 1 : 0;
}
