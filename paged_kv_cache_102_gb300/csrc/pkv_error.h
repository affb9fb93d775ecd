// Per-host-thread error message of the last failing C-ABI call.
#pragma once
#include <string>

namespace pkv {

void set_error(const std::string& msg);
inline int fail(int code, const std::string& msg) {
    set_error(msg);
    return code;
}

}  // namespace pkv
