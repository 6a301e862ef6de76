// api_internal.h -- host helpers that api.cu shares with the other files that
// define entry points (noalloc.cu), so every entry point validates the same
// way, counts SMs the same way and reports its launches to the same
// measurement hook.
#pragma once
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe_api {

// The shape checks every entry point makes before any launch.  `routed`: the
// call selects k distinct experts per token, so k <= E.
moe_status check_dims(const moe_dims* d, bool routed);

// SMs of the current device (looked up once per device).
int num_sms();

// The measurement hook (moe_profile_events): records an event after a launch
// named `name` when the hook is armed.  False if recording failed.
bool note(cudaStream_t s, const char* name);

}  // namespace moe_api
