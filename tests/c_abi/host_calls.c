/* A plain C caller of the library's host calls: parse, print, compose,
 * zipped_divide, plan and describe, bank model and local_partition.  Built
 * by tests/test_c_abi.py with gcc against include/layoutmove.h and
 * liblayoutmove.so; prints one result per line for the test to check. */
#include <stdio.h>
#include <string.h>

#include "layoutmove.h"

static int check(int rc, const char* what) {
  if (rc != LM_OK) {
    printf("FAIL %s %s\n", what, lm_status_string(rc));
    return 1;
  }
  return 0;
}

int main(void) {
  lm_layout *a = NULL, *b = NULL, *r = NULL, *z = NULL, *part = NULL;
  lm_plan* plan = NULL;
  char buf[4096];
  int64_t v = 0, w = 0, base = 0;
  if (check(lm_layout_parse("(8,8):(1,9)", &a), "parse a")) return 1;
  if (check(lm_layout_parse("((4,8),2):((16,1),8)", &b), "parse b")) return 1;
  if (check(lm_layout_compose(a, b, &r), "compose")) return 1;
  if (check(lm_layout_to_string(r, buf, sizeof buf), "print")) return 1;
  printf("compose %s\n", buf);
  lm_layout* m = NULL;
  if (check(lm_layout_parse("(8192,8192):(8192,1)", &m), "parse m")) return 1;
  const int64_t tiler[2] = {64, 64};
  if (check(lm_layout_zipped_divide(m, 2, tiler, &z), "zipped_divide"))
    return 1;
  if (check(lm_layout_to_string(z, buf, sizeof buf), "print z")) return 1;
  printf("zipped_divide %s\n", buf);
  lm_layout *s = NULL, *d = NULL;
  if (check(lm_layout_parse("(4096,4096):(1,4096)", &s), "parse s")) return 1;
  if (check(lm_layout_parse("(4096,4096):(4096,1)", &d), "parse d")) return 1;
  if (check(lm_plan_copy(s, d, 4, &plan), "plan")) return 1;
  if (check(lm_plan_describe(plan, buf, sizeof buf), "describe")) return 1;
  printf("plan_path %s\n", strstr(buf, "\"path\":\"STAGED\"") ? "STAGED" : "?");
  lm_layout* col = NULL;
  if (check(lm_layout_parse("32:8", &col), "parse col")) return 1;
  if (check(lm_smem_wavefronts(col, 4, 4, &v, &w), "banks")) return 1;
  printf("banks %lld %lld\n", (long long)v, (long long)w);
  lm_layout *tile = NULL, *thr = NULL;
  if (check(lm_layout_parse("(8,8):(8,1)", &tile), "parse tile")) return 1;
  if (check(lm_layout_parse("(4,2):(1,4)", &thr), "parse thr")) return 1;
  if (check(lm_layout_local_partition(tile, thr, 5, &part, &base), "part"))
    return 1;
  if (check(lm_layout_to_string(part, buf, sizeof buf), "print part"))
    return 1;
  printf("local_partition %s %lld\n", buf, (long long)base);
  lm_layout_destroy(r);
  r = NULL;
  printf("bad %s\n", lm_status_string(lm_layout_parse("(3,", &r)));
  printf("bad_out_null %d\n", r == NULL);
  printf("version %s\n", lm_version());
  lm_plan_destroy(plan);
  lm_layout_destroy(a);
  lm_layout_destroy(b);
  lm_layout_destroy(m);
  lm_layout_destroy(z);
  lm_layout_destroy(s);
  lm_layout_destroy(d);
  lm_layout_destroy(col);
  lm_layout_destroy(tile);
  lm_layout_destroy(thr);
  lm_layout_destroy(part);
  return 0;
}
