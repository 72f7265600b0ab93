// Decode kernel instances for int8 GEMV weights (head_dim 64 and 128).
#include "mk_vm.cuh"

namespace mk {

const void* vm_kernel_int8(int hd) {
    return hd == 64 ? (const void*)vm_kernel<MK_W_INT8_ROW, MK_W_BF16, 64> : (const void*)vm_kernel<MK_W_INT8_ROW, MK_W_BF16, 128>;
}

}  // namespace mk
