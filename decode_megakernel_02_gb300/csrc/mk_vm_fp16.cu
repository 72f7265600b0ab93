// Decode kernel instances for fp16 GEMV weights (head_dim 64 and 128).
#include "mk_vm.cuh"

namespace mk {

const void* vm_kernel_fp16(int hd) {
    return hd == 64 ? (const void*)vm_kernel<MK_W_FP16, MK_W_FP16, 64> : (const void*)vm_kernel<MK_W_FP16, MK_W_FP16, 128>;
}

}  // namespace mk
