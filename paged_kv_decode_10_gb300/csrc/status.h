// Thread-local error reporting shared by every translation unit of the library.
#pragma once
#include <cstdarg>
#include <cstdio>

#include "pkv.h"

namespace pkv {

// Records a formatted message for pkv_last_error() and returns `code`.
int fail(int code, const char *fmt, ...);
// Clears the calling thread's message (called on entry of each API function).
void clear_error();

}  // namespace pkv

#define PKV_REQUIRE(cond, code, ...)          \
  do {                                        \
    if (!(cond)) return ::pkv::fail((code), __VA_ARGS__); \
  } while (0)
