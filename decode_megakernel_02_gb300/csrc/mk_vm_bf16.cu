// Decode kernel instances for bf16 GEMV weights (head_dim 64 and 128).
#include "mk_vm.cuh"

namespace mk {

const void* vm_kernel_bf16(int hd) {
    return hd == 64 ? (const void*)vm_kernel<MK_W_BF16, MK_W_BF16, 64> : (const void*)vm_kernel<MK_W_BF16, MK_W_BF16, 128>;
}

}  // namespace mk
