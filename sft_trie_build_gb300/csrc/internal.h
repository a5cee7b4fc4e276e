// Internal helpers shared by the translation units of libstp.so.
#pragma once

#include <cstdarg>
#include <cstdint>

#include "stp.h"

namespace stp {

// Records a printf-style message as the thread's last error and returns `code`.
stp_status fail(stp_status code, const char* fmt, ...);

// Clears the thread's last error.
void clear_error();

// Validates an attention descriptor (records the reason and returns its code).
stp_status check_desc(const stp_attn_desc* d);

}  // namespace stp
