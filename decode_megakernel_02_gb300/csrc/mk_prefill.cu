// Tensor-core chunked prefill for sm_103a.
//
// Kog monokernel tutorial ("How the monokernel removes launch overhead"):
// prefill belongs to the same resident runtime as decode.  A prompt is a dense
// contraction (M = prompt tokens), so, unlike batch-1 decode, it runs on the
// 5th-generation tensor cores: each projection is a GEMM C = A . W^T with the
// activations A [tokens][K] and the packed weight rows W [N][K] both K-major.
//
// GEMM kernel (one 128 x 128 output tile per CTA):
//   warp 0   one thread streams the A tiles (hi and lo halves, below) and the
//            W tile (128 x 64 bf16/fp16 each) into a 4-stage shared-memory ring
//            with cp.async.bulk.tensor (TMA), the stage's mbarrier counting
//            the bytes;
//   warp 1   allocates 128 TMEM columns; one thread issues tcgen05.mma
//            (kind::f16, fp32 accumulators in TMEM, K = 16 per instruction)
//            and frees each stage with tcgen05.commit;
//   warps 2-5 read the accumulators with tcgen05.ld (warp w owns TMEM lanes
//            32 (w % 4) ..) and apply the fused epilogue: RoPE + KV-cache
//            append for QKV, residual add for O and down, SwiGLU for gate/up.
// Every wait is bounded by %globaltimer (1 s): on expiry the CTA records an
// error, stops issuing and leaves after freeing its TMEM.
//
// Operand layouts in shared memory: rows of 64 elements (128 B) with the
// 128-byte swizzle for row-major operands, and [8 chunks][128 rows][8 elems]
// without swizzle for the down projection, which the packer stores in column
// blocks of 8 (block b holds W[r][8b .. 8b+8) for every output row r).
//
// Precision: the weights are exact in their 16-bit type, the activations are
// not.  Each activation is stored as a pair hi = round16(a), lo = round16(a -
// hi), and every K step issues two MMAs (hi . W and lo . W) into the same fp32
// accumulators, so the products carry the activation to about 2^-16 of its
// size instead of 2^-9: the prompt's KV cache then differs from a float64
// forward pass by about one bf16 rounding of the stored values, as the decode
// kernel's does.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

#include "mk_internal.h"
#include "mk_prefill.h"

namespace mk {
namespace pf {

constexpr int STAGES = 4;
constexpr int TILE = BM * BK * 2;        // one operand tile (16 KB)
constexpr int STAGE_BYTES = 3 * TILE;    // A hi, A lo, B
constexpr int GEMM_THREADS = 192;
constexpr int GEMM_SMEM = STAGES * STAGE_BYTES + 1024 + 256;  // ring + alignment + barriers
constexpr uint64_t WAIT_NS = 1000000000ull;

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase of the given parity; false after WAIT_NS.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = gtimer();
    while (!mbar_try(b, parity))
        if (gtimer() - t0 > WAIT_NS) return false;
    return true;
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptors of tcgen05.mma (start address, leading and
// stride byte offsets, descriptor version 1, layout type).
// Rows of 128 B with the 128-byte swizzle: 8-row core groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// No swizzle, [chunks][rows][8 elems]: core matrices of 8 rows x 16 B, 128 B
// apart along the rows (stride offset) and rows x 16 B apart along K (leading
// offset).
__device__ __forceinline__ uint64_t desc_blocks(uint32_t saddr, uint32_t k_stride, uint32_t row_stride) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((k_stride >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((row_stride >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor, kind::f16: fp32 accumulators, A and B of one 16-bit
// type (format 1 = bf16, 0 = fp16), both K-major, M x N.
__device__ __forceinline__ uint32_t idesc_f16(int m, int n, bool f16) {
    const uint32_t fmt = f16 ? 0u : 1u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint16_t to16(float v, bool f16) {
    return f16 ? __half_as_ushort(__float2half_rn(v)) : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float from16(uint32_t b, bool f16) {
    return f16 ? __half2float(__ushort_as_half((unsigned short)b)) : __uint_as_float(b << 16);
}
// (a0, a1) -> packed hi pair and packed lo pair: hi = round16(a), lo = round16(a - hi).
__device__ __forceinline__ void split16(float a0, float a1, bool f16, uint32_t& hi, uint32_t& lo) {
    const uint16_t h0 = to16(a0, f16), h1 = to16(a1, f16);
    const uint16_t l0 = to16(a0 - from16(h0, f16), f16), l1 = to16(a1 - from16(h1, f16), f16);
    hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
    lo = (uint32_t)l0 | ((uint32_t)l1 << 16);
}

// 32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// QKV epilogue of one head (HD columns starting at tile column c0): RoPE for
// q and k (rotate-half pairs (i, i + HD/2), angle fp32(pos) * inv_freq_i, as in
// the decode kernel), then q -> the fp32 q buffer, k and v -> the bf16 cache.
template <int HD>
__device__ __forceinline__ void epi_qkv_head(const GemmArgs& g, uint32_t tmem_row, int c0, int n, int m) {
    float v[HD];
#pragma unroll
    for (int j = 0; j < HD / 32; ++j) {
        float t[32];
        tmem_ld32(tmem_row + (uint32_t)(c0 + 32 * j), t);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * j + i] = t[i];
    }
    if (m >= g.m_valid) return;
    const int pos = g.pos0 + m;
    const bool is_q = n < g.q_dim, is_k = !is_q && n < g.q_dim + g.kv_dim;
    if (is_q || is_k) {
#pragma unroll
        for (int i = 0; i < HD / 2; ++i) {
            const float ang = __fmul_rn((float)pos, __ldg(g.inv_freq + i));
            float sn, cs;
            sincosf(ang, &sn, &cs);
            const float x1 = v[i], x2 = v[i + HD / 2];
            v[i] = x1 * cs - x2 * sn;
            v[i + HD / 2] = x2 * cs + x1 * sn;
        }
    }
    if (is_q) {
        float4* dst = (float4*)(g.out_f32 + (size_t)m * g.ldo + n);
#pragma unroll
        for (int i = 0; i < HD / 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        return;
    }
    const int kvsel = is_k ? 0 : 1;
    const int h = (n - g.q_dim - kvsel * g.kv_dim) / HD;
    uint16_t* row = g.kv + ((((size_t)g.layer * 2 + kvsel) * g.n_kv_heads + h) * g.max_seq + pos) * HD;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
        uint4 w;
        uint32_t* wp = (uint32_t*)&w;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            wp[e] = (uint32_t)to16(v[8 * i + 2 * e], false) | ((uint32_t)to16(v[8 * i + 2 * e + 1], false) << 16);
        ((uint4*)row)[i] = w;
    }
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAl,
                const __grid_constant__ CUtensorMap tmB, const GemmArgs g) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* tiles = smem;
    uint64_t* full = (uint64_t*)(smem + STAGES * STAGE_BYTES);  // TMA -> MMA
    uint64_t* empty = full + STAGES;                            // MMA -> TMA
    uint64_t* done = empty + STAGES;                            // MMA -> epilogue
    uint32_t* tmem_slot = (uint32_t*)(done + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int kblocks = g.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {  // TMA producer
        for (int kb = 0; kb < kblocks; ++kb) {
            const int s = kb % STAGES;
            if (kb >= STAGES && !mbar_wait(&empty[s], ((kb / STAGES) - 1) & 1)) {
                atomicExch(g.err, 1u);
                break;
            }
            uint8_t* a = tiles + s * STAGE_BYTES;
            mbar_expect_tx(&full[s], STAGE_BYTES);
            tma_2d(a, &tmA, &full[s], kb * BK, m0);
            tma_2d(a + TILE, &tmAl, &full[s], kb * BK, m0);
            if (g.b_blocks) tma_3d(a + 2 * TILE, &tmB, &full[s], 0, n0, kb * (BK / 8));
            else tma_2d(a + 2 * TILE, &tmB, &full[s], kb * BK, n0);
        }
    } else if (warp == 1 && lane == 0) {  // MMA issuer
        const uint32_t idesc = idesc_f16(BM, BN, g.f16 != 0);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
            const int s = kb % STAGES;
            if (!mbar_wait(&full[s], (kb / STAGES) & 1)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t a = smem_u32(tiles + s * STAGE_BYTES), b = a + 2 * TILE;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
                const uint64_t db = g.b_blocks ? desc_blocks(b + 2 * k * BN * 16, BN * 16, 128) : desc_sw128(b + 32 * k);
#pragma unroll
                for (int part = 0; part < 2; ++part) {  // hi . W, then lo . W
                    const uint64_t da = desc_sw128(a + part * TILE + 32 * k);
                    const uint32_t acc = (kb > 0 || k > 0 || part > 0) ? 1u : 0u;
                    asm volatile(
                        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                        "l"(da), "l"(db), "r"(idesc), "r"(acc)
                        : "memory");
                }
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&empty[s]))
                         : "memory");
        }
        if (ok)
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(done))
                         : "memory");
        else
            atomicExch(g.err, 2u);
    } else if (warp >= 2) {  // epilogue
        const int q = warp & 3;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(done, 0) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) {
            if (lane == 0) atomicExch(g.err, 3u);
        } else {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int m = m0 + 32 * q + lane;
            const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
            if (g.epi == EPI_QKV) {
                if (g.hd == 64) {
                    for (int c0 = 0; c0 < BN; c0 += 64) epi_qkv_head<64>(g, trow, c0, n0 + c0, m);
                } else {
                    for (int c0 = 0; c0 < BN; c0 += 128) epi_qkv_head<128>(g, trow, c0, n0 + c0, m);
                }
            } else {
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    float v[32];
                    tmem_ld32(trow + (uint32_t)c0, v);
                    if (m >= g.m_valid || n0 + c0 >= g.N) continue;
                    if (g.epi == EPI_SWIGLU) {
                        uint32_t w[8], wl[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float a0 = v[4 * j] / (1.f + __expf(-v[4 * j])) * v[4 * j + 1];
                            const float a1 = v[4 * j + 2] / (1.f + __expf(-v[4 * j + 2])) * v[4 * j + 3];
                            split16(a0, a1, g.f16 != 0, w[j], wl[j]);
                        }
                        const size_t o = (size_t)m * g.ld16 + (n0 + c0) / 2;
                        uint4* dst = (uint4*)(g.out16 + o);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        uint4* dl = (uint4*)(g.out16_lo + o);
                        dl[0] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                        dl[1] = make_uint4(wl[4], wl[5], wl[6], wl[7]);
                    } else {
                        float4* dst = (float4*)(g.out_f32 + (size_t)m * g.ldo + n0 + c0);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float4 o = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                            if (g.epi == EPI_RESID) {
                                const float4 r = dst[j];
                                o.x += r.x;
                                o.y += r.y;
                                o.z += r.z;
                                o.w += r.w;
                            }
                            dst[j] = o;
                        }
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BN) : "memory");
    }
}

// ------------------------------------------------------------------ small kernels
__global__ void embed_kernel(const uint16_t* emb, const int32_t* tok, int m_valid, int d, int f16, float* x) {
    const int m = blockIdx.x;
    if (m >= m_valid) return;
    const uint16_t* row = emb + (size_t)tok[m] * d;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        const uint32_t b = row[i];
        x[(size_t)m * d + i] = f16 ? __half2float(__ushort_as_half((unsigned short)b)) : __uint_as_float(b << 16);
    }
}

// One warp per row.
__global__ void rmsnorm_kernel(const float* x, const uint16_t* gain, int m_valid, int d, float eps, int f16,
                               uint16_t* out, uint16_t* out_lo) {
    const int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (m >= m_valid) return;
    const float* xr = x + (size_t)m * d;
    float ss = 0.f;
    for (int i = lane * 4; i < d; i += 128) {
        const float4 v = *(const float4*)(xr + i);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    const float r = rsqrtf(ss / (float)d + eps);
    for (int i = lane * 4; i < d; i += 128) {
        const float4 v = *(const float4*)(xr + i);
        const uint2 gw = *(const uint2*)(gain + i);
        auto gf = [&](uint32_t b) {
            return f16 ? __half2float(__ushort_as_half((unsigned short)b)) : __uint_as_float(b << 16);
        };
        const float y0 = v.x * r * gf(gw.x & 0xFFFFu), y1 = v.y * r * gf(gw.x >> 16);
        const float y2 = v.z * r * gf(gw.y & 0xFFFFu), y3 = v.w * r * gf(gw.y >> 16);
        uint2 o, ol;
        split16(y0, y1, f16 != 0, o.x, ol.x);
        split16(y2, y3, f16 != 0, o.y, ol.y);
        *(uint2*)(out + (size_t)m * d + i) = o;
        *(uint2*)(out_lo + (size_t)m * d + i) = ol;
    }
}

// Causal GQA attention over the cache (CUDA cores, flash style).  A CTA takes
// one KV head and QB consecutive query positions of the chunk, i.e. QB * rep
// query rows (row r = query r / rep, head r % rep); warp w owns rows w, w + 8,
// ...  Key tiles of KT positions are staged in shared memory (K transposed so
// that lanes read consecutive keys); each lane scores keys lane and lane + 32
// of the tile and owns output dims lane + 32 i.
constexpr int QB = 16, KT = 64, ATT_THREADS = 256, ATT_WARPS = 8;
template <int HD, int RPW>  // RPW: rows per warp = QB * rep / 8
__global__ void __launch_bounds__(ATT_THREADS) attention_kernel(const float* q, const uint16_t* kv, int layer, int pos0,
                                                                 int m_valid, int Hq, int Hkv, int max_seq, int f16,
                                                                 uint16_t* out, uint16_t* out_lo) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int rep = Hq / Hkv, R = QB * rep;
    float* qs = (float*)smem;                                    // [R][HD], pre-scaled
    uint16_t* kt = (uint16_t*)(qs + (size_t)R * HD);             // [HD][KT]
    uint16_t* vs = kt + HD * KT;                                 // [KT][HD]
    float* ps = (float*)(vs + KT * HD);                          // [8][RPW][KT]
    const int g = blockIdx.x, qb0 = blockIdx.y * QB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q_dim = Hq * HD;
    const float scale = rsqrtf((float)HD);
    for (int i = tid; i < R * HD; i += ATT_THREADS) {
        const int r = i / HD, dd = i % HD, qi = qb0 + r / rep, h = g * rep + r % rep;
        qs[i] = qi < m_valid ? q[(size_t)qi * q_dim + h * HD + dd] * scale : 0.f;
    }
    const uint16_t* kbase = kv + (((size_t)layer * 2 + 0) * Hkv + g) * (size_t)max_seq * HD;
    const uint16_t* vbase = kv + (((size_t)layer * 2 + 1) * Hkv + g) * (size_t)max_seq * HD;
    float o[RPW][HD / 32], mrow[RPW], lrow[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        mrow[i] = -1.0e30f;
        lrow[i] = 0.f;
#pragma unroll
        for (int j = 0; j < HD / 32; ++j) o[i][j] = 0.f;
    }
    const int last = min(qb0 + QB, m_valid) - 1;  // last query of the block
    const int kend = pos0 + last + 1;               // keys 0 .. kend - 1
    for (int k0 = 0; k0 < kend; k0 += KT) {
        __syncthreads();  // the previous tile is consumed
        for (int i = tid; i < KT * (HD / 8); i += ATT_THREADS) {
            const int kk = i / (HD / 8), ch = i % (HD / 8), j = k0 + kk;
            uint4 kw = make_uint4(0, 0, 0, 0), vw = make_uint4(0, 0, 0, 0);
            if (j < kend) {
                kw = *(const uint4*)(kbase + (size_t)j * HD + ch * 8);
                vw = *(const uint4*)(vbase + (size_t)j * HD + ch * 8);
            }
            *(uint4*)(vs + kk * HD + ch * 8) = vw;
            const uint16_t* ke = (const uint16_t*)&kw;
#pragma unroll
            for (int e = 0; e < 8; ++e) kt[(ch * 8 + e) * KT + kk] = ke[e];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int r = warp + ATT_WARPS * i;
            const int qpos = pos0 + qb0 + r / rep;
            float s0 = 0.f, s1 = 0.f;
            const float* qr = qs + (size_t)r * HD;
#pragma unroll 8
            for (int dd = 0; dd < HD; ++dd) {
                const float qv = qr[dd];
                s0 = fmaf(qv, __uint_as_float((uint32_t)kt[dd * KT + lane] << 16), s0);
                s1 = fmaf(qv, __uint_as_float((uint32_t)kt[dd * KT + lane + 32] << 16), s1);
            }
            if (k0 + lane > qpos) s0 = -3.0e38f;
            if (k0 + lane + 32 > qpos) s1 = -3.0e38f;
            float mt = fmaxf(s0, s1);
#pragma unroll
            for (int off = 16; off; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, off));
            const float mn = fmaxf(mrow[i], mt);
            const float p0 = k0 + lane > qpos ? 0.f : expf(s0 - mn);
            const float p1 = k0 + lane + 32 > qpos ? 0.f : expf(s1 - mn);
            float ls = p0 + p1;
#pragma unroll
            for (int off = 16; off; off >>= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, off);
            const float al = expf(mrow[i] - mn);
            lrow[i] = lrow[i] * al + ls;
            mrow[i] = mn;
#pragma unroll
            for (int j = 0; j < HD / 32; ++j) o[i][j] *= al;
            float* pr = ps + ((size_t)warp * RPW + i) * KT;
            pr[lane] = p0;
            pr[lane + 32] = p1;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const float* pr = ps + ((size_t)warp * RPW + i) * KT;
            for (int kk = 0; kk < KT; ++kk) {
                const float pv = pr[kk];
#pragma unroll
                for (int j = 0; j < HD / 32; ++j)
                    o[i][j] = fmaf(pv, __uint_as_float((uint32_t)vs[kk * HD + lane + 32 * j] << 16), o[i][j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = warp + ATT_WARPS * i, qi = qb0 + r / rep, h = g * rep + r % rep;
        if (qi >= m_valid) continue;
        const float inv = 1.f / lrow[i];
#pragma unroll
        for (int j = 0; j < HD / 32; ++j) {
            const float a = o[i][j] * inv;
            const uint16_t hb = to16(a, f16 != 0);
            out[(size_t)qi * q_dim + h * HD + lane + 32 * j] = hb;
            out_lo[(size_t)qi * q_dim + h * HD + lane + 32 * j] = to16(a - from16(hb, f16 != 0), f16 != 0);
        }
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn g_encode = nullptr;
static std::once_flag g_encode_once;

bool tensor_map_encoder_ready() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = (EncodeTiledFn)fn;
    });
    return g_encode != nullptr;
}

bool make_map_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int64_t row_bytes, int box_rows,
                   bool f16) {
    if (!tensor_map_encoder_ready()) return false;
    cuuint64_t dim[2] = {(cuuint64_t)k, (cuuint64_t)rows}, str[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {BK, (cuuint32_t)box_rows}, es[2] = {1, 1};
    return g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)base, dim,
                    str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_blocks(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int box_rows, bool f16) {
    if (!tensor_map_encoder_ready()) return false;
    cuuint64_t dim[3] = {8, (cuuint64_t)rows, (cuuint64_t)(k / 8)}, str[2] = {16, (cuuint64_t)rows * 16};
    cuuint32_t box[3] = {8, (cuuint32_t)box_rows, BK / 8}, es[3] = {1, 1, 1};
    return g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)base, dim,
                    str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& a_lo, const CUtensorMap& b, const GemmArgs& g,
                        cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] { attr = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM); });
    if (attr != cudaSuccess) return attr;
    dim3 grid(g.M / BM, (g.N + BN - 1) / BN);
    gemm_kernel<<<grid, GEMM_THREADS, GEMM_SMEM, st>>>(a, a_lo, b, g);
    return cudaGetLastError();
}

cudaError_t launch_embed(const uint16_t* emb, const int32_t* tok, int m_valid, int d, bool f16, float* x,
                         cudaStream_t st) {
    embed_kernel<<<m_valid, 256, 0, st>>>(emb, tok, m_valid, d, f16 ? 1 : 0, x);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float* x, const uint16_t* gain, int m_valid, int d, float eps, bool f16,
                           uint16_t* out16, uint16_t* out16_lo, cudaStream_t st) {
    rmsnorm_kernel<<<(m_valid + 7) / 8, 256, 0, st>>>(x, gain, m_valid, d, eps, f16 ? 1 : 0, out16, out16_lo);
    return cudaGetLastError();
}

template <int HD, int RPW>
static cudaError_t launch_att(const float* q, const uint16_t* kv, int layer, int pos0, int m_valid, int Hq, int Hkv,
                              int max_seq, bool f16, uint16_t* out, uint16_t* out_lo, cudaStream_t st) {
    const int R = QB * (Hq / Hkv);
    const size_t smem = (size_t)R * HD * 4 + 2 * (size_t)KT * HD * 2 + (size_t)ATT_WARPS * RPW * KT * 4;
    cudaError_t e = cudaFuncSetAttribute(attention_kernel<HD, RPW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(Hkv, (m_valid + QB - 1) / QB);
    attention_kernel<HD, RPW><<<grid, ATT_THREADS, smem, st>>>(q, kv, layer, pos0, m_valid, Hq, Hkv, max_seq,
                                                               f16 ? 1 : 0, out, out_lo);
    return cudaGetLastError();
}

cudaError_t launch_attention(const float* q, const uint16_t* kv, int layer, int pos0, int m_valid, int n_q_heads,
                             int n_kv_heads, int hd, int max_seq, bool f16, uint16_t* out16, uint16_t* out16_lo,
                             cudaStream_t st) {
    const int rpw = QB * (n_q_heads / n_kv_heads) / ATT_WARPS;  // rep 1..8 -> 2..16 rows per warp
    auto go = [&](auto hdc) -> cudaError_t {
        constexpr int H = decltype(hdc)::value;
        switch (rpw) {
            case 2: return launch_att<H, 2>(q, kv, layer, pos0, m_valid, n_q_heads, n_kv_heads, max_seq, f16, out16, out16_lo, st);
            case 4: return launch_att<H, 4>(q, kv, layer, pos0, m_valid, n_q_heads, n_kv_heads, max_seq, f16, out16, out16_lo, st);
            case 6: return launch_att<H, 6>(q, kv, layer, pos0, m_valid, n_q_heads, n_kv_heads, max_seq, f16, out16, out16_lo, st);
            case 8: return launch_att<H, 8>(q, kv, layer, pos0, m_valid, n_q_heads, n_kv_heads, max_seq, f16, out16, out16_lo, st);
            case 10: return launch_att<H, 10>(q, kv, layer, pos0, m_valid, n_q_heads, n_kv_heads, max_seq, f16, out16, out16_lo, st);
            case 12: return launch_att<H, 12>(q, kv, layer, pos0, m_valid, n_q_heads, n_kv_heads, max_seq, f16, out16, out16_lo, st);
            case 14: return launch_att<H, 14>(q, kv, layer, pos0, m_valid, n_q_heads, n_kv_heads, max_seq, f16, out16, out16_lo, st);
            case 16: return launch_att<H, 16>(q, kv, layer, pos0, m_valid, n_q_heads, n_kv_heads, max_seq, f16, out16, out16_lo, st);
            default: return cudaErrorInvalidValue;
        }
    };
    if (hd == 64) return go(std::integral_constant<int, 64>{});
    if (hd == 128) return go(std::integral_constant<int, 128>{});
    return cudaErrorInvalidValue;
}

}  // namespace pf
}  // namespace mk
