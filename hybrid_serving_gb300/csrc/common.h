// common.h -- host-side helpers shared by the library's translation units.
#pragma once
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>

#include "hs.h"

namespace hs {

// Record the message of a failing call (thread-local) and return its code.
hs_status fail(hs_status code, const char* fmt, ...);
// Count one kernel launch (hs_launch_count()).
void count_launch(int n = 1);

}  // namespace hs

#define HS_CHECK_ARG(cond, ...)                         \
  do {                                                  \
    if (!(cond)) return hs::fail(HS_EINVAL, __VA_ARGS__); \
  } while (0)
