// host_common.cuh -- shared host utilities of libsdt: error reporting, device
// properties, the device status word, environment switches.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "sdt.h"

namespace sdt {

// Record `msg` as this thread's last error and return `code`.
int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
void clear_error();

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int smem_optin = 0;      // max dynamic shared memory per block (opt-in)
    int smem_per_sm = 0;
    int cc_major = 0, cc_minor = 0;
    int l2_bytes = 0;
};

// Properties of the current device (cached per device).  Returns SDT_OK, or a
// negative status (with the last error set) when there is no usable device or
// it is not compute capability 10.3.
int current_device(DeviceInfo *out);

// Device address of the status word on the current device (cached per device).
int status_word(int **out);

// Default bound on any single wait inside a kernel, in nanoseconds (SDT_WAIT_TIMEOUT_MS).
unsigned long long wait_timeout_ns();

// 1 when the named environment variable is set to a true value ("1", "on", "true", "yes").
bool env_flag(const char *name);

}  // namespace sdt
