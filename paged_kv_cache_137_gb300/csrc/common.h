// Shared host-side helpers of libpkv: error reporting.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <string>

#include "pkv.h"

namespace pkv {

void set_error(const char* fmt, ...);
void clear_error();

inline pkv_status fail(pkv_status st, const char* msg) {
  set_error("%s", msg);
  return st;
}

}  // namespace pkv
