// api.cu -- error text, sizes, shared host-side checks of the C ABI.
#include <cstdarg>
#include <cstdio>
#include <string>

#include "q2.cuh"

namespace q1 {

static thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return Q1_OK;
  // The runtime also keeps the error in the thread's last-error slot; read it
  // here, so that a later launch check does not report it as its own.
  (void)cudaGetLastError();
  return fail(Q1_ERR_CUDA, "%s: CUDA error %d (%s)", what, (int)e, cudaGetErrorString(e));
}

}  // namespace q1

extern "C" const char* q1_last_error(void) { return q1::g_last_error.c_str(); }

extern "C" int64_t q1_0_packed_bytes(int64_t rows, int64_t n) {
  if (rows < 1 || rows > (int64_t(1) << 26) || n < 128 || n > (int64_t(1) << 24) || n % 128)
    return q1::fail(Q1_ERR_ARG, "q1_0_packed_bytes: bad shape rows=%lld n=%lld (rows in 1..2^26, "
                                "n a multiple of 128 in 128..2^24)",
                    (long long)rows, (long long)n);
  q1::g_last_error.clear();
  return q1::layout_of(rows, n).total_bytes;
}

extern "C" int64_t q2_0_packed_bytes(int64_t rows, int64_t n) {
  if (rows < 1 || rows > (int64_t(1) << 26) || n < 128 || n > (int64_t(1) << 24) || n % 128)
    return q1::fail(Q1_ERR_ARG, "q2_0_packed_bytes: bad shape rows=%lld n=%lld (rows in 1..2^26, "
                                "n a multiple of 128 in 128..2^24)",
                    (long long)rows, (long long)n);
  q1::g_last_error.clear();
  return q1::layout_q2(rows, n).total_bytes;
}

extern "C" int q1_device_status(int clear) {
  unsigned v = 0, u = 0, t = 0;
  if (int e = q1::status_word_dp4a(&v, clear)) return e;
  if (int e = q1::status_word_prod(&u, clear)) return e;
  if (int e = q1::status_word_tc(&t, clear)) return e;
  return int(v | u | t);
}
