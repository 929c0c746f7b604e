/*
 * Host cost of libcsa's argument validation, measured from C (no Python in the loop).
 * Every call below passes every check but the last one (the workspace is one byte short),
 * so it runs the full validation and returns CSA_ERR_WORKSPACE without launching anything.
 * Prints the mean nanoseconds per call of csa_decode_step and of csa_sparse_attn.
 */
#include <stdio.h>
#include <stdint.h>
#include <time.h>

#include "csa.h"

static double now_ns(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return (double)ts.tv_sec * 1e9 + (double)ts.tv_nsec;
}

int main(void) {
  csa_config c = {4, 64, 512, 64, 128, 4, 512, 128, CSA_BF16, CSA_E4M3, 0.044194173824159216f};
  void *p = (void *)(uintptr_t)0x10000; /* aligned, never dereferenced: nothing is launched */
  csa_decode_args a = {0};
  a.E_cap = 262144;
  a.q_pos = p; a.q = p; a.qI = p; a.w = p; a.sink = p; a.kv_comp = p; a.kI = p; a.kscale = p;
  a.kv_tail = p; a.z_tail = p; a.kvI_tail = p; a.zI_tail = p; a.bias = p; a.biasI = p;
  a.kv_local = p; a.L = 128; a.local_base = p; a.out = p;
  const size_t need = csa_workspace_size(CSA_OP_DECODE, &c, 4, 262144);
  const size_t need_attn = csa_workspace_size(CSA_OP_ATTN, &c, 4, 1);
  /* both sizes must be non-zero: a call given need - 1 bytes must stop at the workspace check,
     since the pointers above are not device memory */
  if (need == (size_t)-1 || need_attn == (size_t)-1 || need < 16 || need_attn < 16) return 2;
  const int n = 200000;
  int bad = 0;
  for (int i = 0; i < 1000; ++i) bad |= csa_decode_step(&c, &a, p, need - 1, NULL) != CSA_ERR_WORKSPACE;
  double t0 = now_ns();
  for (int i = 0; i < n; ++i) bad |= csa_decode_step(&c, &a, p, need - 1, NULL) != CSA_ERR_WORKSPACE;
  const double dec = (now_ns() - t0) / n;
  for (int i = 0; i < 1000; ++i)
    bad |= csa_sparse_attn(&c, p, 1, p, 262144, p, p, 128, p, p, p, p, NULL, p, need_attn - 1, NULL) !=
           CSA_ERR_WORKSPACE;
  t0 = now_ns();
  for (int i = 0; i < n; ++i)
    bad |= csa_sparse_attn(&c, p, 1, p, 262144, p, p, 128, p, p, p, p, NULL, p, need_attn - 1, NULL) !=
           CSA_ERR_WORKSPACE;
  const double att = (now_ns() - t0) / n;
  printf("decode_step_ns %.1f\nsparse_attn_ns %.1f\n", dec, att);
  return bad ? 1 : 0;
}
