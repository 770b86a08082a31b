// The current device's context, for state the library keeps per device
// (kernel attributes it raised, split weights it uploaded, a scratch
// address): such state belongs to the context it was made in, and a
// cudaDeviceReset destroys that context and starts a new one on the next
// call.
#pragma once

namespace pkv {

// Unique id (for the life of the process) of the current device's context;
// false if there is none yet or the driver cannot say.  Defined in noalloc.cu.
bool current_context_id(unsigned long long *id);

}  // namespace pkv
