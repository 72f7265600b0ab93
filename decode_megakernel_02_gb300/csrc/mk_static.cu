// Fixed-size device scratch for mk_decode_static: a file-scope device array
// instead of a caller-provided workspace, so that call needs no allocation.
#include <cuda_runtime.h>

#include "mk.h"

namespace mk {

static __device__ __align__(256) unsigned char g_static_scratch[MK_STATIC_SCRATCH_BYTES];

// Address of the array in the current device's context.  The lookup loads
// this module on first use, so it must not run inside a stream capture.
cudaError_t static_scratch_address(void** ptr) { return cudaGetSymbolAddress(ptr, g_static_scratch); }

}  // namespace mk
