/*
 * abi_client.c -- a plain C99 user of include/gemm.h.
 *
 * Proves that the header is valid C (compiled with -std=c99 -pedantic
 * -Werror) and that the library is usable from C with nothing but the
 * header and the shared object: no CUDA headers, no C++ runtime of the
 * caller's own.
 *
 *   abi_client layout
 *       Host-only checks: version, status strings, the shared-memory
 *       formula, argument rejection, and the size and field offsets of
 *       gemm_tuning_t, gemm_plan_info_t and gemm_device_desc_t, printed one per line as
 *       "key value" for the Python test to compare with its ctypes mirrors.
 *
 *   abi_client run M N K dtype epi a.bin b.bin c.bin
 *       Reads A (M x K) and B (N x K) as raw 16-bit elements of `dtype`
 *       (0 fp16, 1 bf16), computes C = epi(A . B^T) through a plan and
 *       gemm_run_host (host buffers in and out), checks the device status
 *       and writes C (M x N, raw 16-bit) to c.bin.  Exit code 0 on success.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm.h"

#define OFF(T, tag, f) printf("offset %s.%s %lu\n", tag, #f, (unsigned long)offsetof(T, f))

static int layout(void) {
  gemm_plan_t* plan = (gemm_plan_t*)&plan; /* must be reset to NULL on failure */
  gemm_status_t s;

  printf("version %s\n", gemm_version());
  printf("status_ok %s\n", gemm_status_string(GEMM_OK));
  printf("status_timeout %s\n", gemm_status_string(GEMM_ERR_TIMEOUT));
  printf("smem %lu\n", (unsigned long)gemm_smem_bytes(128, 256, 64, 2, 4));

  s = gemm_plan_create(&plan, -1, 8, 8, GEMM_F16, GEMM_EPI_NONE, 4, GEMM_PIPELINED, 0);
  printf("bad_m %d %d\n", (int)s, plan == NULL);
  s = gemm_plan_create(&plan, 8, 8, 8, GEMM_F16, GEMM_EPI_NONE, 0, GEMM_PIPELINED, 0);
  printf("bad_stages %d %d\n", (int)s, plan == NULL);
  gemm_plan_destroy(NULL);
  printf("destroy_null ok\n");
  printf("wait_mma_full %s\n", gemm_wait_detail_string(GEMM_WAIT_MMA_FULL));

  printf("sizeof tuning %lu\n", (unsigned long)sizeof(gemm_tuning_t));
  OFF(gemm_tuning_t, "tuning", tile_n);
  OFF(gemm_tuning_t, "tuning", raster_group);
  OFF(gemm_tuning_t, "tuning", max_ctas);
  OFF(gemm_tuning_t, "tuning", cta_group);
  OFF(gemm_tuning_t, "tuning", tail_split);
  OFF(gemm_tuning_t, "tuning", timeout_ns);
  OFF(gemm_tuning_t, "tuning", b_kn);
  OFF(gemm_tuning_t, "tuning", out_f32);
  OFF(gemm_tuning_t, "tuning", debug_fault);
  OFF(gemm_tuning_t, "tuning", k_serpentine);
  OFF(gemm_tuning_t, "tuning", epi_groups);

  printf("sizeof info %lu\n", (unsigned long)sizeof(gemm_plan_info_t));
  OFF(gemm_plan_info_t, "info", tile_m);
  OFF(gemm_plan_info_t, "info", tile_n);
  OFF(gemm_plan_info_t, "info", tile_k);
  OFF(gemm_plan_info_t, "info", stages);
  OFF(gemm_plan_info_t, "info", accumulators);
  OFF(gemm_plan_info_t, "info", raster_group);
  OFF(gemm_plan_info_t, "info", grid);
  OFF(gemm_plan_info_t, "info", num_tiles);
  OFF(gemm_plan_info_t, "info", smem_bytes);
  OFF(gemm_plan_info_t, "info", pads_operands);
  OFF(gemm_plan_info_t, "info", tma_store);
  OFF(gemm_plan_info_t, "info", kernels_per_run);
  OFF(gemm_plan_info_t, "info", sm_count);
  OFF(gemm_plan_info_t, "info", cta_group);
  OFF(gemm_plan_info_t, "info", tail_tiles);
  OFF(gemm_plan_info_t, "info", tail_splits);
  OFF(gemm_plan_info_t, "info", work_units);
  OFF(gemm_plan_info_t, "info", stream_k);
  OFF(gemm_plan_info_t, "info", out_f32);
  OFF(gemm_plan_info_t, "info", b_kn);
  OFF(gemm_plan_info_t, "info", k_sub);
  OFF(gemm_plan_info_t, "info", host_panels);
  OFF(gemm_plan_info_t, "info", k_serpentine);
  OFF(gemm_plan_info_t, "info", l2_prefetch_first);
  OFF(gemm_plan_info_t, "info", sk_cluster);
  OFF(gemm_plan_info_t, "info", epi_groups);
  OFF(gemm_plan_info_t, "info", stream_k_first);

  printf("sizeof device %lu\n", (unsigned long)sizeof(gemm_device_desc_t));
  OFF(gemm_device_desc_t, "device", sm_count);
  OFF(gemm_device_desc_t, "device", smem_optin);
  OFF(gemm_device_desc_t, "device", l2_bytes);
  OFF(gemm_device_desc_t, "device", pair_clusters);
  return 0;
}

static void* read_file(const char* path, size_t bytes) {
  FILE* f = fopen(path, "rb");
  void* p = malloc(bytes ? bytes : 1);
  if (!f || !p || fread(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot read %lu bytes from %s\n", (unsigned long)bytes, path);
    if (f) fclose(f);
    free(p);
    return NULL;
  }
  fclose(f);
  return p;
}

static int run(int argc, char** argv) {
  int64_t M, N, K;
  int dtype, epi, rc = 1;
  void *a = NULL, *b = NULL, *c = NULL;
  gemm_plan_t* plan = NULL;
  gemm_status_t s;
  int32_t dev_status = -1, detail = -1;
  FILE* f;

  if (argc != 10) {
    fprintf(stderr, "usage: abi_client run M N K dtype epi a.bin b.bin c.bin\n");
    return 2;
  }
  M = strtoll(argv[2], NULL, 10);
  N = strtoll(argv[3], NULL, 10);
  K = strtoll(argv[4], NULL, 10);
  dtype = atoi(argv[5]);
  epi = atoi(argv[6]);
  if (M <= 0 || N <= 0 || K <= 0) {
    fprintf(stderr, "M, N, K must be positive\n");
    return 2;
  }
  a = read_file(argv[7], (size_t)(M * K * 2));
  b = read_file(argv[8], (size_t)(N * K * 2));
  c = malloc((size_t)(M * N * 2));
  if (!a || !b || !c) goto done;
  memset(c, 0xff, (size_t)(M * N * 2)); /* NaN pattern: every element must be written */

  s = gemm_plan_create(&plan, M, N, K, (gemm_dtype_t)dtype, (gemm_epilogue_t)epi, 4,
                       GEMM_PIPELINED, 0);
  if (s != GEMM_OK) {
    fprintf(stderr, "gemm_plan_create: %s (%s)\n", gemm_status_string(s), gemm_last_error());
    goto done;
  }
  /* stream NULL: the legacy default stream; gemm_run_host synchronises it */
  s = gemm_run_host(plan, a, b, c, M, N, K, (gemm_dtype_t)dtype, (gemm_epilogue_t)epi, 4, NULL);
  if (s != GEMM_OK) {
    fprintf(stderr, "gemm_run_host: %s (%s)\n", gemm_status_string(s), gemm_last_error());
    goto done;
  }
  s = gemm_plan_check(plan, &dev_status, &detail);
  if (s != GEMM_OK || dev_status != GEMM_OK) {
    fprintf(stderr, "gemm_plan_check: %s, device %s (%s)\n", gemm_status_string(s),
            gemm_status_string((gemm_status_t)dev_status), gemm_wait_detail_string(detail));
    goto done;
  }
  f = fopen(argv[9], "wb");
  if (!f || fwrite(c, 1, (size_t)(M * N * 2), f) != (size_t)(M * N * 2)) {
    fprintf(stderr, "cannot write %s\n", argv[9]);
    if (f) fclose(f);
    goto done;
  }
  fclose(f);
  printf("ran %lld x %lld x %lld\n", (long long)M, (long long)N, (long long)K);
  rc = 0;
done:
  gemm_plan_destroy(plan);
  free(a);
  free(b);
  free(c);
  return rc;
}

int main(int argc, char** argv) {
  if (argc >= 2 && strcmp(argv[1], "layout") == 0) return layout();
  if (argc >= 2 && strcmp(argv[1], "run") == 0) return run(argc, argv);
  fprintf(stderr, "usage: abi_client layout | run M N K dtype epi a.bin b.bin c.bin\n");
  return 2;
}
