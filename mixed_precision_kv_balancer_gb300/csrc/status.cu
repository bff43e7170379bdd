// Thread-local status message behind mikv_last_error().
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"

namespace mikv {

static thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_msg[0] = '\0'; }

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MIKV_ECUDA, "%s: %s", what, cudaGetErrorString(e));
  return MIKV_OK;
}

}  // namespace mikv

extern "C" const char* mikv_last_error(void) { return mikv::g_msg; }

extern "C" int mikv_wait_status(unsigned* bits, int clear) {
  mikv::clear_error();
  if (!bits) return mikv::fail(MIKV_EINVAL, "wait_status: null pointer");
  unsigned v = 0;
  if (int e = mikv::scores_wait_giveups(&v, clear != 0)) return e;
  if (int e = mikv::select_wait_giveups(&v, clear != 0)) return e;
  if (int e = mikv::perturb_wait_giveups(&v, clear != 0)) return e;
  *bits = v;
  return MIKV_OK;
}
