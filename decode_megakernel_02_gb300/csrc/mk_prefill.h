// Tensor-core chunked prefill: internal interface between the runtime and
// mk_prefill.cu.  Not part of the public ABI.
#pragma once
#include <cuda.h>  // CUtensorMap and its encoder's types (no link against the driver library)
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk.h"

namespace mk {
namespace pf {

constexpr int BM = 128, BN = 128, BK = 64;  // GEMM tile (tokens x output columns x reduction)

// Epilogues of the prompt GEMMs.
enum Epi : int32_t {
    EPI_F32 = 0,     // out_f32[m][n] = C (tests)
    EPI_QKV = 1,     // q (roped) -> out_f32; k (roped), v -> the bf16 KV cache at position pos0 + m
    EPI_RESID = 2,   // out_f32[m][n] += C (the residual stream)
    EPI_SWIGLU = 3,  // columns (2j, 2j + 1) = (gate_j, up_j): out16[m][j] = silu(gate_j) * up_j
};

struct GemmArgs {
    int32_t M, N, K;       // rows launched (a multiple of BM), output columns, reduction length
    int32_t m_valid;       // rows that exist
    int32_t b_blocks;      // B is stored in column blocks of 8 (3-D map) instead of rows (2-D map)
    int32_t f16;           // operands are fp16 (else bf16)
    int32_t epi;
    float* out_f32;
    int32_t ldo;
    uint16_t* out16;       // EPI_SWIGLU: the hi and lo halves of the activations
    uint16_t* out16_lo;
    int32_t ld16;
    // EPI_QKV
    int32_t q_dim, kv_dim, hd, max_seq, pos0, layer, n_kv_heads;
    const float* inv_freq;
    uint16_t* kv;
    uint32_t* err;         // set when a wait gives up (the launch then leaves early)
};

// Encoder of tiled tensor maps (cuTensorMapEncodeTiled through the runtime's
// driver entry points).  Returns false when the driver has no such entry.
bool tensor_map_encoder_ready();
// 2-D K-major tile map of a [rows][k] 16-bit matrix with a row stride of
// row_bytes, box BK x box_rows, 128-byte swizzle.
bool make_map_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int64_t row_bytes, int box_rows,
                   bool f16);
// 3-D map of a [k/8][rows][8] column-block matrix (no swizzle): box 8 x box_rows x BK/8.
bool make_map_blocks(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int box_rows, bool f16);

// A is given as two maps, the hi and lo halves of the activations.
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& a_lo, const CUtensorMap& b, const GemmArgs& g,
                        cudaStream_t st);
// x[m][:] = E[tok[m]][:] (fp32) for m < m_valid.
cudaError_t launch_embed(const uint16_t* emb, const int32_t* tok, int m_valid, int d, bool f16, float* x,
                         cudaStream_t st);
// y = x[m][:] * (mean x^2 + eps)^(-1/2) * gain for m < m_valid, stored as the
// operand-type pair out16 = round(y), out16_lo = round(y - out16).
cudaError_t launch_rmsnorm(const float* x, const uint16_t* gain, int m_valid, int d, float eps, bool f16,
                           uint16_t* out16, uint16_t* out16_lo, cudaStream_t st);
// Causal GQA attention of the chunk's queries (q fp32 [m][q_dim], roped,
// unscaled) over the cache positions 0 .. pos0 + m -> (out16, out16_lo) [m][q_dim].
cudaError_t launch_attention(const float* q, const uint16_t* kv, int layer, int pos0, int m_valid, int n_q_heads,
                             int n_kv_heads, int hd, int max_seq, bool f16, uint16_t* out16, uint16_t* out16_lo,
                             cudaStream_t st);

}  // namespace pf
}  // namespace mk
