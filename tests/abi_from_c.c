/* A plain C99 caller of the library: includes the public header, links the shared
 * library and exercises the calls that need no GPU (validation, layouts, argument
 * errors that return before any launch, host fault injection). Prints one
 * "name value" line per check; tests/test_abi_c.py compiles it, runs it and compares
 * the struct sizes it prints with those of the Python binding. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "magicpig.h"

static mp_config base_config(void) {
  mp_config c;
  memset(&c, 0, sizeof c);
  c.layers = 1;
  c.batch = 1;
  c.kv_heads = 2;
  c.q_heads = 4;
  c.head_dim = 128;
  c.K = 8;
  c.L = 75;
  c.n_sink = 4;
  c.window = 64;
  c.capacity = 4096;
  c.dtype = MP_DTYPE_BF16;
  c.threshold = 2;
  return c;
}

int main(void) {
  /* never dereferenced: every call below fails validation before touching memory */
  void* fake = (void*)(size_t)(1u << 20);
  mp_config c = base_config();
  mp_tables_layout tl;
  mp_decode_layout dl;

  printf("abi %d\n", mp_abi_version());
  printf("sizeof_config %u\n", (unsigned)sizeof(mp_config));
  printf("sizeof_tables_layout %u\n", (unsigned)sizeof(mp_tables_layout));
  printf("sizeof_decode_layout %u\n", (unsigned)sizeof(mp_decode_layout));
  printf("sizeof_kernel_time %u\n", (unsigned)sizeof(mp_kernel_time));
  printf("check_ok %d\n", mp_config_check(&c));
  printf("check_null %d\n", mp_config_check(NULL));
  c.q_heads = 3;
  printf("check_bad_group %d\n", mp_config_check(&c));
  c.q_heads = 4;
  c.head_dim = 96;
  printf("check_head_dim %d\n", mp_config_check(&c));
  c.head_dim = 128;
  printf("tables_layout %d\n", mp_tables_layout_get(&c, &tl));
  printf("tables_bytes %llu\n", (unsigned long long)tl.total_bytes);
  printf("tables_match_mode %d\n", tl.match_mode);
  printf("decode_layout %d\n", mp_decode_layout_get(&c, &dl));
  printf("decode_bytes %llu\n", (unsigned long long)dl.total_bytes);
  printf("build_capacity %d\n", mp_build_tables(&c, fake, 5000, (const float*)fake, fake, NULL));
  printf("build_null_keys %d\n", mp_build_tables(&c, NULL, 10, (const float*)fake, fake, NULL));
  printf("append_capacity %d\n", mp_append(&c, fake, fake, 4096, NULL));
  printf("decode_scratch %d\n",
         mp_decode_attention(&c, fake, fake, fake, 100, fake, (float*)fake, fake, dl.total_bytes - 1, NULL));
  printf("status_string %s\n", mp_status_string(MP_ERR_CAPACITY));
  return 0;
}
