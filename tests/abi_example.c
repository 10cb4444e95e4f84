/* A plain C caller of libdflash: the host-side part of the ABI (handle,
 * workspace sizes, validation, selector sizes) needs no GPU.  Built and run by
 * tests/test_abi_cpu.py with gcc against include/ and libdflash.so.  Device
 * pointers are placeholders: nothing here dereferences them. */
#include <stdint.h>
#include <stdio.h>

#include "dflash.h"

int main(void) {
  int32_t windows[2] = {0, 0};
  dflash_config c = {DFLASH_BF16, 256, 3, 512, 2, 8, 2, 128, 1024, 4096, 4095, 16, 64,
                     windows, 1e-6f, 1e6f, 4, 256, 4096};
  const void *fake = (const void *)0x10000;
  const void *per_layer[2] = {fake, fake};
  dflash_weights w = {fake, fake, fake, fake, fake, per_layer, per_layer, per_layer,
                      per_layer, per_layer, per_layer, per_layer, per_layer};
  dflash_handle *h = NULL;
  int st = dflash_create(&c, &w, &h);
  if (st != DFLASH_OK) {
    printf("create failed: %s\n", dflash_last_error());
    return 1;
  }
  size_t ws = 0, sel = 0;
  if (dflash_workspace_size(h, &ws) != DFLASH_OK || ws == 0) return 2;
  if (dflash_selector_workspace_size(h, 8, 128, &sel) != DFLASH_OK || sel == 0) return 3;
  /* validation: K above 8, a draft before any workspace */
  if (dflash_selector_workspace_size(h, 9, 128, &sel) != DFLASH_EUNSUPPORTED) return 4;
  int32_t ids[16];
  if (dflash_draft_block(h, NULL, 1, (const int32_t *)fake, ids, NULL, NULL) != DFLASH_ESTATE)
    return 5;
  dflash_destroy(h);
  /* a config the kernels do not implement */
  c.head_dim = 96;
  if (dflash_create(&c, &w, &h) != DFLASH_EUNSUPPORTED || h != NULL) return 6;
  printf("ok workspace=%zu selector=%zu last_error=\"%s\"\n", ws, sel, dflash_last_error());
  return 0;
}
