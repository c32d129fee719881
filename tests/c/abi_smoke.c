/* A plain C99 caller of libbeam.so: the header compiles as C and every call
 * below is answered on the host (argument checks), so it runs without a GPU.
 * Exits 0 when every answer is the documented one, else prints the first
 * mismatch and exits 1. */
#include <stdio.h>
#include <string.h>

#include "beam.h"

static int check(const char* what, int got, int want) {
  if (got != want) {
    printf("%s: got %d, want %d\n", what, got, want);
    return 1;
  }
  return 0;
}

int main(void) {
  beam_moe_config_t cfg = {5120, 256, 8, 4, 8, 2560, 2.5f, 1e-6f};
  beam_moe_config_t bad = cfg;
  beam_moe_weights_t w;
  beam_moe_uncombined_t out;
  uint16_t* p16 = (uint16_t*)(uintptr_t)0x10000; /* aligned, never dereferenced: rejected first */
  int fails = 0;
  memset(&w, 0, sizeof w);
  if (strncmp(beam_version(), "beam", 4) != 0) {
    printf("version: %s\n", beam_version());
    return 1;
  }
  if (strcmp(beam_status_string(BEAM_OK), "ok") != 0) return 1;
  fails += check("workspace size of a Beam layer is nonzero", beam_moe_workspace_size(&cfg, 64) > 0, 1);
  bad.d_ff = 2500; /* not a multiple of 64 */
  fails += check("workspace size of an unsupported shape", (int)beam_moe_workspace_size(&bad, 64), 0);
  fails += check("empty batch", beam_boundary_norm(NULL, NULL, NULL, NULL, 0, 5120, 1e-6f, 3, NULL, NULL, NULL),
                 BEAM_OK);
  fails += check("n = 0", beam_boundary_norm(p16, p16, p16, p16, 4, 5120, 1e-6f, 0, p16 + 32, p16 + 64, NULL),
                 BEAM_ERR_INVALID_ARG);
  fails += check("hidden size", beam_boundary_norm(p16, p16, p16, p16, 4, 5000, 1e-6f, 3, p16 + 32, p16 + 64, NULL),
                 BEAM_ERR_UNSUPPORTED_SHAPE);
  fails += check("misaligned h", beam_boundary_norm(p16 + 1, p16, p16, p16, 4, 5120, 1e-6f, 3, p16 + 32, p16 + 64,
                                                     NULL),
                 BEAM_ERR_MISALIGNED);
  fails += check("layer with null weights", beam_moe_layer(p16, p16, 3, &w, 4, &cfg, p16, p16, NULL, p16,
                                                           (size_t)1 << 40, NULL),
                 BEAM_ERR_INVALID_ARG);
  fails += check("uncombined layer without an output struct",
                 beam_moe_layer_uncombined(p16, p16, 3, &w, 4, &cfg, p16, NULL, p16, (size_t)1 << 40, NULL),
                 BEAM_ERR_INVALID_ARG);
  fails += check("uncombined layer, empty batch",
                 beam_moe_layer_uncombined(NULL, NULL, 3, &w, 0, &cfg, NULL, &out, NULL, 0, NULL), BEAM_OK);
  fails += check("device error query without an output", beam_get_device_error(NULL, NULL), BEAM_ERR_INVALID_ARG);
  fails += check("graph release", beam_release_host_graphs(), BEAM_OK);
  if (fails == 0) printf("ok\n");
  return fails == 0 ? 0 : 1;
}
