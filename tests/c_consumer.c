/* A plain C program against the library's header: no Python, no torch.  It
 * exercises the host entry points (nothing here needs a GPU) and the
 * argument checks of a device entry point, and prints what it found. */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "spectree.h"

int main(void) {
  int failures = 0;
  if (spec_version() < 1) failures++;
  if (strcmp(spec_status_string(SPEC_OK), "ok") != 0) failures++;
  if (strcmp(spec_dev_status_string(SPEC_DEV_BAD_PATH), "bad commit path") != 0) failures++;

  /* goodput table: AL / ITL per batch size, K in {1, 2, 3} */
  const double al[2][3] = {{1.8, 2.4, 2.9}, {1.8, 2.4, 2.9}};
  const double itl[2][3] = {{10.0, 11.0, 12.0}, {10.0, 15.0, 22.0}};
  const int32_t ks[3] = {1, 2, 3};
  int32_t kopt[2];
  if (spec_dsd_optimal_k(&al[0][0], &itl[0][0], 2, 3, ks, kopt) != SPEC_OK) failures++;
  if (kopt[0] != 3 || kopt[1] != 1) failures++;
  const int32_t bs[2] = {1, 64};
  int32_t k = 0;
  if (spec_dsd_select_k(bs, kopt, 2, 100, &k) != SPEC_OK || k != 1) failures++;

  /* graph keys for 8 tokens and K <= 3 */
  int32_t t[64], kk[64], n = 0;
  if (spec_dsd_graph_keys(8, 3, t, kk, 64, &n) != SPEC_OK) failures++;
  int found = 0;
  for (int i = 0; i < n; ++i)
    if (t[i] == 8) found = found * 10 + kk[i];
  if (found != 13) failures++; /* K = 1 then K = 3 */

  /* a device entry point rejects bad sizes before any launch */
  if (spec_tree_expand_level(NULL, 1, 1, 100, 40, 0, 64, NULL, NULL, NULL) != SPEC_ERR_UNSUPPORTED) failures++;

  printf("c consumer: %s (k_opt %d %d, keys for 8 tokens %d)\n", failures ? "FAILED" : "ok", kopt[0], kopt[1], found);
  return failures ? 1 : 0;
}
