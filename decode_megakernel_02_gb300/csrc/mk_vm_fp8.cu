// Decode kernel instances for FP8 E4M3 block-scaled GEMV weights (head_dim 64 and 128, greedy and token-selection).
#include "mk_vm.cuh"

namespace mk {

// sel: the token-selection instance (sampling, EOS, the token-select task).
const void* vm_kernel_fp8(int hd, bool sel) {
    if (sel)
        return hd == 64 ? (const void*)vm_kernel<MK_W_FP8_E4M3, MK_W_BF16, 64, true>
                        : (const void*)vm_kernel<MK_W_FP8_E4M3, MK_W_BF16, 128, true>;
    return hd == 64 ? (const void*)vm_kernel<MK_W_FP8_E4M3, MK_W_BF16, 64, false>
                    : (const void*)vm_kernel<MK_W_FP8_E4M3, MK_W_BF16, 128, false>;
}

}  // namespace mk
