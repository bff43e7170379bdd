// Thread-local status message behind mikv_last_error().
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"
#include "tcgen05.cuh"

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

namespace mikv {
// The give-up path of the tensor-core kernels' waits, run alone: one thread waits twice on an
// mbarrier of one arrival, which it makes itself only if `arrive`; with no arrival both
// waits give up (the first after `polls` polls, the second after the short limit) and the
// thread sets the probe's status bit.  Nothing is copied or issued.
__global__ void wait_probe_kernel(long polls, int arrive) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t mb = smem_u32(&bar);
  tc::mbar_init(mb, 1);
  tc::mbar_init_fence();
  if (arrive) tc::mbar_arrive(mb);
  tc::Waits w;
  w.polls = polls;
  w(mb, 0);
  w(mb, 0);
  if (!w.ok) tc::report_giveup(tc::kGiveupProbe);
}
}  // namespace mikv

extern "C" int mikv_wait_probe(int64_t polls, int arrive, void* stream) {
  mikv::clear_error();
  if (polls < 1 || polls > (1L << 24)) return mikv::fail(MIKV_EINVAL, "wait_probe: polls=%lld", (long long)polls);
  mikv::wait_probe_kernel<<<1, 32, 0, mikv::as_stream(stream)>>>(static_cast<long>(polls), arrive != 0);
  return mikv::check_launch("wait_probe_kernel");
}

extern "C" int mikv_wait_status(unsigned* bits, int clear) {
  mikv::clear_error();
  if (!bits) return mikv::fail(MIKV_EINVAL, "wait_status: null pointer");
  unsigned v = 0;
  if (int e = mikv::scores_wait_giveups(&v, clear != 0)) return e;
  if (int e = mikv::select_wait_giveups(&v, clear != 0)) return e;
  if (int e = mikv::perturb_wait_giveups(&v, clear != 0)) return e;
  if (int e = mikv::tc::wait_giveups(&v, clear != 0)) return e;  // the probe's word
  *bits = v;
  return MIKV_OK;
}
