// debug_hooks.cuh -- test hooks of the tensor-core router's bounded waits
// (set through moe_debug_set; the state lives in abi.cu).
#pragma once

namespace moe {

// The router tile that, in the next tensor-core router launch, never issues
// its first stage's copies (-1: none); reading it clears it.
int debug_take_skip_router();

}  // namespace moe
