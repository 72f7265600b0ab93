// Kernel selection, shared-memory sizing and the test-support kernels.
#include "mk_vm.cuh"

namespace mk {

// ------------------------------------------------------------------ launch
const void* vm_kernel_bf16(int hd, bool sel);
const void* vm_kernel_fp16(int hd, bool sel);
const void* vm_kernel_int8(int hd, bool sel);
const void* vm_kernel_int4(int hd, bool sel);
const void* vm_kernel_fp8(int hd, bool sel);

// sel: the instance with token selection (sampling, EOS, the token-select task).
const void* vm_kernel_for(int wdtype, int base, int hd, bool sel) {
    if (hd != 64 && hd != 128) return nullptr;
    if (base == MK_W_FP16) return wdtype == MK_W_FP16 ? vm_kernel_fp16(hd, sel) : nullptr;
    switch (wdtype) {
        case MK_W_BF16: return vm_kernel_bf16(hd, sel);
        case MK_W_INT8_ROW: return vm_kernel_int8(hd, sel);
        case MK_W_INT4_G128: return vm_kernel_int4(hd, sel);
        case MK_W_FP8_E4M3: return vm_kernel_fp8(hd, sel);
        default: return nullptr;
    }
}

size_t vm_shared_bytes(int wdtype, int xs_floats, int tab_cap) {
    size_t ring = 0;
    switch (wdtype) {
        case MK_W_INT8_ROW: ring = (size_t)NW * ring_slots<MK_W_INT8_ROW>() * ring_slot_bytes<MK_W_INT8_ROW>(); break;
        case MK_W_INT4_G128: ring = (size_t)NW * ring_slots<MK_W_INT4_G128>() * ring_slot_bytes<MK_W_INT4_G128>(); break;
        case MK_W_FP8_E4M3: ring = (size_t)NW * ring_slots<MK_W_FP8_E4M3>() * ring_slot_bytes<MK_W_FP8_E4M3>(); break;
        default: ring = (size_t)NW * ring_slots<MK_W_BF16>() * ring_slot_bytes<MK_W_BF16>(); break;
    }
    return ring_offset(xs_floats, tab_cap) + ring;
}

// ------------------------------------------------------------------ test kernels
// Dequantise a packed tensor with the decode kernel's own code -> float path.
template <int WT>
__global__ void dequant_kernel(const uint8_t* rows, int64_t stride, int first, int step, int nrows, int K,
                               float* out) {
    const int r = blockIdx.x;
    if (r >= nrows) return;
    const uint8_t* row = rows + (int64_t)(first + (int64_t)r * step) * stride;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        float v;
        if constexpr (WT == MK_W_INT8_ROW) {
            const uint32_t word = *(const uint32_t*)(row + (k & ~3)) ^ 0x80808080u;
            v = i8_to_f32(word, k & 3) * half_bits_to_f32(*(const uint16_t*)(row + K));
        } else if constexpr (WT == MK_W_INT4_G128) {
            const uint32_t word = *(const uint32_t*)(row + (k >> 3) * 4) ^ 0x88888888u;
            v = i4_to_f32(word, k & 7) * half_bits_to_f32(*(const uint16_t*)(row + K / 2 + 2 * (k >> 7)));
        } else if constexpr (WT == MK_W_FP8_E4M3) {
            const uint32_t pair = *(const uint16_t*)(row + (k & ~1));
            const unsigned long long f = e4m3x2_pair(pair);
            v = __uint_as_float((uint32_t)(f >> (32 * (k & 1)))) * half_bits_to_f32(*(const uint16_t*)(row + K + 2 * (k >> 7)));
        } else if constexpr (WT == MK_W_FP16) {
            v = half_bits_to_f32(((const uint16_t*)row)[k]);
        } else {
            v = bf16_bits_to_f32(((const uint16_t*)row)[k]);
        }
        out[(int64_t)r * K + k] = v;
    }
}

// The same for a quantised down projection in 16-byte column blocks: the
// code of (row r, unit k) sits at ((k / BU) * nrows + r) * 16 + its place in
// the chunk, and the scales follow the blocks ([nrows] for int8, [K / 128]
// [nrows] for int4), as the fused FFN reads them.
template <int WT>
__global__ void dequant_cols_kernel(const uint8_t* base, int nrows, int K, float* out) {
    constexpr int BU = ffn_block(WT);
    const int r = blockIdx.x;
    if (r >= nrows) return;
    const uint16_t* scales = (const uint16_t*)(base + (int64_t)nrows * (K / BU) * 16);
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const uint8_t* chunk = base + ((int64_t)(k / BU) * nrows + r) * 16;
        const int j = k % BU;
        float v;
        if constexpr (WT == MK_W_INT8_ROW) {
            const uint32_t word = *(const uint32_t*)(chunk + (j & ~3)) ^ 0x80808080u;
            v = i8_to_f32(word, j & 3) * half_bits_to_f32(scales[r]);
        } else if constexpr (WT == MK_W_FP8_E4M3) {
            const unsigned long long f = e4m3x2_pair(*(const uint16_t*)(chunk + (j & ~1)));
            v = __uint_as_float((uint32_t)(f >> (32 * (j & 1)))) * half_bits_to_f32(scales[(int64_t)(k >> 7) * nrows + r]);
        } else {
            const uint32_t word = *(const uint32_t*)(chunk + (j >> 3) * 4) ^ 0x88888888u;
            v = i4_to_f32(word, j & 7) * half_bits_to_f32(scales[(int64_t)(k >> 7) * nrows + r]);
        }
        out[(int64_t)r * K + k] = v;
    }
}

cudaError_t launch_dequant(int wdtype, const uint8_t* rows, int64_t stride, int first, int step, int nrows,
                           int K, float* out, cudaStream_t st) {
    dim3 grid(nrows), block(256);
    if (stride == 0) {  // a quantised down projection in column blocks
        if (wdtype == MK_W_INT8_ROW) dequant_cols_kernel<MK_W_INT8_ROW><<<grid, block, 0, st>>>(rows, nrows, K, out);
        else if (wdtype == MK_W_FP8_E4M3) dequant_cols_kernel<MK_W_FP8_E4M3><<<grid, block, 0, st>>>(rows, nrows, K, out);
        else if (wdtype == MK_W_INT4_G128) dequant_cols_kernel<MK_W_INT4_G128><<<grid, block, 0, st>>>(rows, nrows, K, out);
        else return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    switch (wdtype) {
        case MK_W_INT8_ROW: dequant_kernel<MK_W_INT8_ROW><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
        case MK_W_INT4_G128: dequant_kernel<MK_W_INT4_G128><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
        case MK_W_FP8_E4M3: dequant_kernel<MK_W_FP8_E4M3><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
        case MK_W_FP16: dequant_kernel<MK_W_FP16><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
        default: dequant_kernel<MK_W_BF16><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
    }
    return cudaGetLastError();
}

// A wait that can never be satisfied, with the same watchdog as the VM: the
// kernel must give up, report DEV_TIMEOUT and return.
__global__ void watchdog_kernel(uint32_t* ctr, uint32_t* status, int64_t limit_ns) {
    if (threadIdx.x != 0) return;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if ((int32_t)(ld_acquire(ctr) - 1u) >= 0) {
            status[0] = DEV_OK;
            return;
        }
        if ((it & 63u) == 0u && gtimer() - t0 > (uint64_t)limit_ns) {
            status[0] = DEV_TIMEOUT;
            return;
        }
    }
}

cudaError_t launch_watchdog(uint32_t* ctr, uint32_t* status, int64_t limit_ns, cudaStream_t st) {
    watchdog_kernel<<<1, 32, 0, st>>>(ctr, status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mk
