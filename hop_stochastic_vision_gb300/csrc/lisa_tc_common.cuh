// lisa_tc_common.cuh -- pieces shared by the tensor-core kernel families of
// the LiSA forward layer (bf16, d_h = d_v = 64, sm_103a): ReLU on packed
// bf16, swizzled bf16 row images, thread-block-cluster helpers, the TF32
// recurrence step U_k^T = U_(k-1)^T M^T on the legacy tensor path, tensor-
// memory loads in the mma.sync fragment layout, and the host-side tensor-map
// and launch-attribute helpers.  Everything is internal to the translation
// unit that includes it.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "lisa_sm100.cuh"

namespace lisa {
namespace {

using namespace sm100;

constexpr int kD = 64;                         // head width of this family
constexpr int kRow = 128;                      // bytes of one token row (64 bf16)

__device__ __forceinline__ void record_error(int *err, int bits) { atomicOr(err, bits); }

__device__ __forceinline__ uint32_t relu2(uint32_t v) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&v);
    x = __hmax2(x, __float2bfloat162_rn(0.f));
    return *reinterpret_cast<uint32_t *>(&x);
}
__device__ __forceinline__ uint4 relu4(uint4 v) {
    return make_uint4(relu2(v.x), relu2(v.y), relu2(v.z), relu2(v.w));
}
// In-place ReLU of `bytes` (multiple of 16) of shared memory.
__device__ __forceinline__ void relu_smem(uint8_t *p, int bytes, int tid, int nthreads) {
    uint4 *v = reinterpret_cast<uint4 *>(p);
    for (int i = tid; i < bytes / 16; i += nthreads) v[i] = relu4(v[i]);
}

// Writes one 64-element fp32 row as bf16 into a 128-B-swizzled row image.
__device__ __forceinline__ void put_row_bf16(uint8_t *img, int row, const float *v, int chunk) {
    uint4 o;
    o.x = pack_bf16(v[0], v[1]);
    o.y = pack_bf16(v[2], v[3]);
    o.z = pack_bf16(v[4], v[5]);
    o.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4 *>(img + (size_t)row * kRow + ((chunk ^ (row & 7)) << 4)) = o;
}

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Remote shared-memory loads.  Volatile keeps them after the cluster barrier
// that precedes them; no memory clobber, so a run of them can be in flight
// together.
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ void st_dsmem4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Sum of one float4 over the CL <= 8 CTAs of the cluster, rank order 0..CL-1;
// all remote loads are issued before the first add.
__device__ __forceinline__ float4 cluster_sum4(uint32_t local_addr, int CL) {
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (q < CL) v[q] = ld_dsmem4(map_rank(local_addr, (uint32_t)q));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (q < CL) {
            acc.x += v[q].x; acc.y += v[q].y; acc.z += v[q].z; acc.w += v[q].w;
        }
    return acc;
}

// Row strides (floats) of the fused statistics kernel's recurrence buffers,
// chosen so the tensor-path fragment loads below are free of bank conflicts:
// U_k, U_next, the fold: 68 (rows g of a fragment land on banks 4 g + c);
// M^T: 72 (rows k = q, q + 4 land on banks 8 q + n).
constexpr int kUS = 68;
constexpr int kMS = 72;

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Un[i][a] = sum_b U[i][b] Mt[b][a] for `rows` rows on the tensor path in TF32
// (operands rounded to 10-bit mantissas, fp32 accumulation): U and Un with row
// stride kUS, M^T with row stride kMS.  Warp w of `nwarps` takes the 8-column
// tiles w, w + nwarps, ...; rows in tiles of 16 (missing rows read as zero and
// are not stored); when there are as many row tiles as warps, warp w takes
// row tile w whole instead.  The A fragments of a k-step are loaded once per row tile.
// With `fold`, also fold[i][a] += wk * Un[i][a] (stride kUS; each element is
// owned by the thread that computes it).
__device__ __forceinline__ void rows_times_mt_tf32(const float *U, const float *Mt, float *Un, int rows, int warp,
                                                   int lane, int nwarps, float *fold, float wk) {
    const int g = lane >> 2, q4 = lane & 3;
    if (rows > 16 * (nwarps - 1) && rows <= 16 * nwarps) {
        // one row tile per warp (a slice held by one CTA): all eight column
        // tiles of it, four independent accumulator chains at a time
        const int r0 = 16 * warp + g, r1 = r0 + 8;
        uint32_t a[8][4];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int b = 8 * ks + q4;
            a[ks][0] = r0 < rows ? to_tf32(U[r0 * kUS + b]) : 0u;
            a[ks][1] = r1 < rows ? to_tf32(U[r1 * kUS + b]) : 0u;
            a[ks][2] = r0 < rows ? to_tf32(U[r0 * kUS + b + 4]) : 0u;
            a[ks][3] = r1 < rows ? to_tf32(U[r1 * kUS + b + 4]) : 0u;
        }
#pragma unroll 1
        for (int n0 = 0; n0 < 8; n0 += 4) {
            float d[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int b = 8 * ks + q4;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_tf32_1688(d[j], a[ks][0], a[ks][1], a[ks][2], a[ks][3],
                                  to_tf32(Mt[b * kMS + 8 * (n0 + j) + g]), to_tf32(Mt[(b + 4) * kMS + 8 * (n0 + j) + g]));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 8 * (n0 + j) + 2 * q4;
                if (r0 < rows) {
                    Un[r0 * kUS + c] = d[j][0];
                    Un[r0 * kUS + c + 1] = d[j][1];
                    if (fold) {
                        fold[r0 * kUS + c] = fmaf(wk, d[j][0], fold[r0 * kUS + c]);
                        fold[r0 * kUS + c + 1] = fmaf(wk, d[j][1], fold[r0 * kUS + c + 1]);
                    }
                }
                if (r1 < rows) {
                    Un[r1 * kUS + c] = d[j][2];
                    Un[r1 * kUS + c + 1] = d[j][3];
                    if (fold) {
                        fold[r1 * kUS + c] = fmaf(wk, d[j][2], fold[r1 * kUS + c]);
                        fold[r1 * kUS + c + 1] = fmaf(wk, d[j][3], fold[r1 * kUS + c + 1]);
                    }
                }
            }
        }
        return;
    }
    for (int m0 = 0; m0 < rows; m0 += 16) {
        const int r0 = m0 + g, r1 = m0 + g + 8;
        uint32_t a[8][4];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int b = 8 * ks + q4;
            a[ks][0] = r0 < rows ? to_tf32(U[r0 * kUS + b]) : 0u;
            a[ks][1] = r1 < rows ? to_tf32(U[r1 * kUS + b]) : 0u;
            a[ks][2] = r0 < rows ? to_tf32(U[r0 * kUS + b + 4]) : 0u;
            a[ks][3] = r1 < rows ? to_tf32(U[r1 * kUS + b + 4]) : 0u;
        }
        for (int nt = warp; nt < 8; nt += nwarps) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int b = 8 * ks + q4;
                mma_tf32_1688(d, a[ks][0], a[ks][1], a[ks][2], a[ks][3], to_tf32(Mt[b * kMS + 8 * nt + g]),
                              to_tf32(Mt[(b + 4) * kMS + 8 * nt + g]));
            }
            const int c = 8 * nt + 2 * q4;
            if (r0 < rows) {
                Un[r0 * kUS + c] = d[0];
                Un[r0 * kUS + c + 1] = d[1];
                if (fold) {
                    fold[r0 * kUS + c] = fmaf(wk, d[0], fold[r0 * kUS + c]);
                    fold[r0 * kUS + c + 1] = fmaf(wk, d[1], fold[r0 * kUS + c + 1]);
                }
            }
            if (r1 < rows) {
                Un[r1 * kUS + c] = d[2];
                Un[r1 * kUS + c + 1] = d[3];
                if (fold) {
                    fold[r1 * kUS + c] = fmaf(wk, d[2], fold[r1 * kUS + c]);
                    fold[r1 * kUS + c + 1] = fmaf(wk, d[3], fold[r1 * kUS + c + 1]);
                }
            }
        }
    }
}

// B-operand rows of the s term: n_umat*64 + {0: s_hi, 1: s_lo, 2..15: 0}.
__device__ __forceinline__ void put_s_rows(uint8_t *img, int row0, const float *s, int tid) {
    if (tid < 128) {
        const int r16 = tid >> 3, chunk = tid & 7;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float x = s[chunk * 8 + e];
            const float hi = __bfloat162float(__float2bfloat16_rn(x));
            v[e] = r16 == 0 ? hi : (r16 == 1 ? x - hi : 0.f);
        }
        put_row_bf16(img, row0 + r16, v, chunk);
    }
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero); 2^-inf = +0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Column `col` of the sum over `count` rows (row stride `stride` floats) of a
// partial-sum array in global memory: eight loads in flight, eight
// accumulators, added in a fixed order.
__device__ __forceinline__ float sum_partials(const float *part, int count, int stride, int col) {
    float a[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) a[u] = 0.f;
    int r = 0;
    for (; r + 8 <= count; r += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = part[(size_t)(r + u) * stride + col];
#pragma unroll
        for (int u = 0; u < 8; ++u) a[u] += v[u];
    }
    for (; r < count; ++r) a[0] += part[(size_t)r * stride + col];
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

__device__ __forceinline__ float gelu_erf(float x) {
    return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
}

// GELU(x) = x (1 + erf(x / sqrt 2)) / 2 with erf from Abramowitz & Stegun,
// Handbook of Mathematical Functions, formula 7.1.26 (the formula's absolute
// error is at most 1.5e-7; the approximate reciprocal and 2^x below add a few
// fp32 ulps): for z >= 0, erf(z) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5))))
// exp(-z^2), t = 1 / (1 + p z); erf is odd.  Used by the adaptive-weight
// epilogue, where it replaces erff's longer evaluation on the per-token path.
__device__ __forceinline__ float gelu_as7126(float x) {
    const float z = fabsf(x) * 0.70710678118654752f;
    const float t = __fdividef(1.f, fmaf(0.3275911f, z, 1.f));
    const float poly =
        t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f), 0.254829592f);
    const float erf_abs = fmaf(-poly, ex2_approx(-z * z * 1.4426950408889634f), 1.f);
    return 0.5f * x * (1.f + copysignf(erf_abs, x));
}

// GELU'(x) = Phi(x) + x phi(x): Phi(x) = (1 + erf(x / sqrt 2)) / 2 from the same
// formula 7.1.26, whose exp(-z^2) = exp(-x^2 / 2) also gives the normal density
// phi(x) = exp(-x^2 / 2) / sqrt(2 pi).  Used by the adaptive-weight backward.
__device__ __forceinline__ float gelu_grad_as7126(float x) {
    const float z = fabsf(x) * 0.70710678118654752f;
    const float t = __fdividef(1.f, fmaf(0.3275911f, z, 1.f));
    const float poly =
        t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f), 0.254829592f);
    const float e = ex2_approx(-z * z * 1.4426950408889634f);
    const float erf_abs = fmaf(-poly, e, 1.f);
    return fmaf(x * 0.39894228040143268f, e, 0.5f * (1.f + copysignf(erf_abs, x)));
}

// 16 TMEM lanes x 8 consecutive fp32 columns per repetition, in mma.sync
// C-fragment layout: regs 4r+0,1 = (row g, cols 8r+2q, +1), 4r+2,3 = (row g+8, same).
__device__ __forceinline__ void tmem_ld_frag8_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_frag_nowait(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 3-D map over [S][n][64] bf16, box {64, box_tokens, 1}.
bool make_map_tokens(CUtensorMap *m, const void *ptr, int S, int n, int box_tokens) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)n, (cuuint64_t)S};
    cuuint64_t strides[2] = {(cuuint64_t)kRow, (cuuint64_t)n * kRow};
    cuuint32_t box[3] = {64, (cuuint32_t)box_tokens, 1}, es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over [S][H][W][64] bf16, box {64, bw, bh, 1}.
bool make_map_grid(CUtensorMap *m, const void *ptr, int S, int H, int W, int bh, int bw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)S};
    cuuint64_t strides[3] = {(cuuint64_t)kRow, (cuuint64_t)W * kRow, (cuuint64_t)H * W * kRow};
    cuuint32_t box[4] = {64, (cuuint32_t)bw, (cuuint32_t)bh, 1}, es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise a kernel's dynamic shared-memory limit once per device (and again
// only if a larger size is asked for), so calls made during stream capture
// do not touch function attributes.
template <typename Kern>
cudaError_t set_smem(Kern k, int slot, int bytes) {
    static std::mutex mu;
    static int done[8][64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[slot][dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[slot][dev] = bytes;
    return e;
}

uint32_t pow2_cols(int cols) {
    uint32_t c = 32;
    while ((int)c < cols) c <<= 1;
    return c;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
    return n;
}

}  // namespace
}  // namespace lisa
