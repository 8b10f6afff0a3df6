// Shared host-side helpers of libradixattn.so: error reporting and argument checks.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <string>

#include "radix_attn.h"

namespace rx {

// Thread-local message for rx_last_error(); defined in radix_tree.cpp.
void set_error(const char* fmt, ...);
void clear_error();

}  // namespace rx

#define RX_REQUIRE(cond, ...)          \
    do {                               \
        if (!(cond)) {                 \
            ::rx::set_error(__VA_ARGS__); \
            return RX_EINVAL;          \
        }                              \
    } while (0)
