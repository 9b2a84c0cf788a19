/* Host-only use of the C ABI from C (no GPU needed): build the chain Command
 * out = (a*b) - (c + a)*s, lower it, plan launches over fake device
 * addresses (aligned, one load off the alignment, a size mismatch), write and
 * read back its text form, and check the error paths. Prints "ok" on
 * success; any failed check prints its line and exits 1. */
#include <stdio.h>
#include <string.h>

#include "cmd.h"

#define CHECK(cond)                                                               \
  do {                                                                            \
    if (!(cond)) {                                                                \
      printf("FAILED line %d: %s (%s)\n", __LINE__, #cond, cmd_last_error());     \
      return 1;                                                                   \
    }                                                                             \
  } while (0)

static cmd_tensor_arg view1d(cmd_tag tag, uintptr_t addr, int64_t n) {
  cmd_tensor_arg t;
  memset(&t, 0, sizeof t);
  t.tag = tag;
  t.rank = 1;
  t.ptr = (void*)addr;
  t.sizes[0] = n;
  t.strides[0] = 1;
  return t;
}

int main(void) {
  CHECK(cmd_abi_version() == CMD_ABI_VERSION);

  cmd_command_t c;
  CHECK(cmd_create(&c) == CMD_OK);
  cmd_tag a, b, cc, s, r[4], out;
  CHECK(cmd_add_load_tensor(c, CMD_F32, 1, &a) == CMD_OK);
  CHECK(cmd_add_load_tensor(c, CMD_F32, 1, &b) == CMD_OK);
  CHECK(cmd_add_load_tensor(c, CMD_F32, 1, &cc) == CMD_OK);
  CHECK(cmd_add_load_scalar(c, CMD_F32, &s) == CMD_OK);
  cmd_xop ops[4] = {{CMD_E_MUL, a, b, -1, }, {CMD_E_ADD, cc, a, -1}, {CMD_E_MUL, CMD_LOCAL(1), s, -1},
                    {CMD_E_SUB, CMD_LOCAL(0), CMD_LOCAL(2), -1}};
  CHECK(cmd_add_execute(c, ops, 4, r) == CMD_OK);
  CHECK(cmd_add_store(c, r[3], CMD_F32, 1, &out) == CMD_OK);

  /* a T_Execute op naming a tag that does not exist */
  cmd_xop bad = {CMD_E_ADD, 999, a, -1};
  cmd_tag dummy;
  CHECK(cmd_add_execute(c, &bad, 1, &dummy) == CMD_ERR_BAD_TAG);
  CHECK(strlen(cmd_last_error()) > 0);

  cmd_program_info info;
  uint32_t words[256];
  CHECK(cmd_lower(c, &info, words, 256) == CMD_OK);
  CHECK(info.n_loads == 3 && info.n_scalars == 1 && info.n_stores == 1 && info.tier == 1 && info.extended == 0);

  cmd_kernel_t k;
  CHECK(cmd_lower_kernel(c, &k) == CMD_OK);
  const int64_t n = 100003;
  const uintptr_t base = (uintptr_t)1 << 40, gap = (uintptr_t)1 << 32;
  cmd_tensor_arg t[4] = {view1d(a, base, n), view1d(b, base + gap, n), view1d(cc, base + 2 * gap, n),
                         view1d(out, base + 3 * gap, n)};
  cmd_scalar_arg sv;
  sv.tag = s;
  sv.v.f32 = 0.75f;
  cmd_runtime_args args = {t, 4, &sv, 1};
  cmd_launch_plan p;
  CHECK(cmd_plan_launch(k, &args, &p) == CMD_OK);
  CHECK(p.path == CMD_PATH_CONTIG && p.n_elements == n && p.bytes == 16 * n && p.shifted_loads == 0);
  CHECK(p.head_elements == 0 && p.contig_elements == n - n % 256);

  t[0].ptr = (void*)(base + 4); /* a one element past a vector boundary: shifted */
  CHECK(cmd_plan_launch(k, &args, &p) == CMD_OK);
  CHECK(p.path == CMD_PATH_CONTIG && p.shifted_loads == 1 && p.head_elements == 4);
  CHECK(p.contig_elements % 256 == 0 && n - 4 - p.contig_elements >= 4);

  t[0].ptr = (void*)base;
  t[1].sizes[0] = n - 1; /* sizes that differ */
  CHECK(cmd_plan_launch(k, &args, &p) == CMD_ERR_SHAPE);
  t[1].sizes[0] = n;
  t[3].ptr = (void*)(base + 8); /* the store overlapping load a */
  CHECK(cmd_plan_launch(k, &args, &p) == CMD_ERR_ALIAS);
  cmd_kernel_destroy(k);

  /* the text form: write, read back, write again to the same text */
  int64_t need = 0;
  CHECK(cmd_to_yaml(c, NULL, 0, &need) == CMD_OK && need > 1);
  char text1[8192], text2[8192];
  CHECK(need <= (int64_t)sizeof text1);
  CHECK(cmd_to_yaml(c, text1, sizeof text1, NULL) == CMD_OK);
  cmd_command_t c2;
  CHECK(cmd_from_yaml(text1, (int64_t)strlen(text1), &c2) == CMD_OK);
  CHECK(cmd_to_yaml(c2, text2, sizeof text2, NULL) == CMD_OK);
  CHECK(strcmp(text1, text2) == 0);
  cmd_destroy(c2);
  cmd_destroy(c);
  printf("ok\n");
  return 0;
}
