// profile.cuh - optional per-launch CUDA-event timing (measurement only).
#pragma once

#include <cuda_runtime.h>

namespace smol {

// Called around each kernel launch with its kind (SMOL_K_*).  Both are no-ops
// unless smol_profile_begin enabled the kind on this host thread.
void prof_before(int kind, cudaStream_t st);
void prof_after(int kind, cudaStream_t st);

}  // namespace smol
