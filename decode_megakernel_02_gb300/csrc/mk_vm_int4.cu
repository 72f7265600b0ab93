// Decode kernel instances for int4 GEMV weights (head_dim 64 and 128).
#include "mk_vm.cuh"

namespace mk {

const void* vm_kernel_int4(int hd) {
    return hd == 64 ? (const void*)vm_kernel<MK_W_INT4_G128, MK_W_BF16, 64> : (const void*)vm_kernel<MK_W_INT4_G128, MK_W_BF16, 128>;
}

}  // namespace mk
