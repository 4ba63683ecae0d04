// host.h -- per-context host state of the library.
//
// Kernels, their attributes and __device__ arrays belong to the module that is
// loaded into one CUDA context, not to a device: two contexts on one device
// (the runtime's primary context and a driver-API context, or the primary
// context before and after cudaDeviceReset) each hold their own copy.  State
// the host caches about them is therefore keyed by the current context's id.
#pragma once

#include <cuda_runtime.h>

namespace moe {

// Unique id (for the life of the process) of the CUDA context current on the
// calling thread; 0 when no context is current or it cannot be read.
unsigned long long current_context_id();

// Raise `func`'s dynamic shared-memory limit to at least `bytes` in the
// current context (cudaFuncSetAttribute once per context, kernel and size;
// it is not a stream operation, so calls captured later stay capturable).
cudaError_t ensure_dynamic_smem(const void* func, int bytes);

}  // namespace moe
