// Host-side helpers shared by the entry points: argument checks and device
// queries.  Host code only.
#pragma once

#include <cstdint>

#include "pa_kv.h"

namespace pa {

// bytes of one element of a storage dtype (0 for an unknown code)
int elem_bytes(int dtype);

// Checks a cache descriptor: non-null 16-byte-aligned pointers, positive
// sizes, a known dtype.
pa_status check_cache(const pa_kv_cache* cache);

// SM count of the current device (cached per device); 0 on failure.
int device_sm_count();

// Largest dynamic shared memory a block may opt into on the current device.
int device_max_smem_optin();

}  // namespace pa
