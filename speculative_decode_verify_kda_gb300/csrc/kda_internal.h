// kda_internal.h -- helpers private to the CUDA library (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include "kda_spec.h"

namespace kda {

// Record the reason of a failing call for kda_last_error() and return `code`.
int fail(int code, const std::string &msg);
// Clear the calling thread's last error and return KDA_OK.
int ok();
// Map a CUDA error after a launch to KDA_ECUDA (with its text) or KDA_OK.
int check_launch(const char *what);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace kda
