// Thread-local error messages behind pw_last_error().
#include <cstdarg>
#include <cstdio>
#include <string>

#include "pw_internal.h"

namespace {
thread_local std::string g_last_error;
}

namespace pw {

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

void clear_error() { g_last_error.clear(); }

int cuda_error(cudaError_t e, const char* what) {
  return set_error(PW_ERR_CUDA, "%s failed: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

}  // namespace pw

extern "C" const char* pw_last_error(void) { return g_last_error.c_str(); }
