// fp32 CUDA-core GEMMs for the Newton-Schulz accuracy-check mode
// (MUONH_FLAG_FP32_CHECK): the same three stages as the tensor-core path --
// Gram (X X^T, or X^T X for a tall matrix), polynomial b*A + c*A A, apply
// (a*X + B X, or a*X + X B) -- with fp32 operands and fp32 accumulation, so
// the result can be held to a 1e-4 relative tolerance against the float64
// oracle.  Plain 128x128 tiles, 8x8 outputs per thread, no symmetry
// shortcuts: this path is for checking, not speed.

#include "common.cuh"
#include "ns_gemm.h"

namespace muonh {

constexpr int SB = 128, SK = 8, ST = 256;

template <int MODE>
__global__ void __launch_bounds__(ST) simt_gemm_kernel(const SimtParams p) {
    __shared__ float As[SK][SB + 4];
    __shared__ float Bs[SK][SB + 4];
    const int g = blockIdx.z;
    const int m0 = blockIdx.y * SB, n0 = blockIdx.x * SB;
    const float* A = p.a + (size_t)g * p.a_bstride;
    const float* B = p.b + (size_t)g * p.b_bstride;
    const int t = threadIdx.x;
    const int tx = t & 15, ty = t >> 4;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < p.K; k0 += SK) {
        if (p.a_km) {
            // A stored [k][m]: 8 x 128; thread -> k t/32, m (t&31)*4 .. +3
            const int kk = t >> 5, mq = (t & 31) * 4;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int gk = k0 + kk, gi = m0 + mq + u;
                As[kk][mq + u] = (gk < p.K && gi < p.M) ? A[(size_t)gk * p.lda + gi] : 0.f;
            }
        } else {
            // A tile: 128 rows x 8 k; thread -> row t/2, k (t&1)*4 .. +3
            const int r = t >> 1, kq = (t & 1) * 4;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int gi = m0 + r, gk = k0 + kq + u;
                As[kq + u][r] = (gi < p.M && gk < p.K) ? A[(size_t)gi * p.lda + gk] : 0.f;
            }
        }
        if (p.b_kn) {
            // B rows are k: 8 x 128; thread -> k t/32, n (t&31)*4 .. +3
            const int kk = t >> 5, nq = (t & 31) * 4;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int gk = k0 + kk, gn = n0 + nq + u;
                Bs[kk][nq + u] = (gk < p.K && gn < p.N) ? B[(size_t)gk * p.ldb + gn] : 0.f;
            }
        } else {
            const int r = t >> 1, kq = (t & 1) * 4;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int gn = n0 + r, gk = k0 + kq + u;
                Bs[kq + u][r] = (gn < p.N && gk < p.K) ? B[(size_t)gn * p.ldb + gk] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < SK; ++k) {
            float a[8], b[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[k][ty * 4 + i];
                a[4 + i] = As[k][64 + ty * 4 + i];
                b[i] = Bs[k][tx * 4 + i];
                b[4 + i] = Bs[k][64 + tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

    const float sc = p.scale ? p.scale[g] : 1.f;
    const float* add = p.addend ? p.addend + (size_t)g * p.add_bstride : nullptr;
    float* out = p.out + (size_t)g * p.out_bstride;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gi = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (gi >= p.M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int gj = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (gj >= p.N) continue;
            float v = acc[i][j];
            if (MODE == NS_GRAM) {
                v *= sc;
            } else if (MODE == NS_POLY) {
                v = fmaf(p.cb, add[(size_t)gi * p.ld_add + gj], p.cc * v);
            } else {
                v = sc * fmaf(p.ca, add[(size_t)gi * p.ld_add + gj], v);
            }
            out[(size_t)gi * p.ldo + gj] = v;
        }
    }
}

cudaError_t launch_simt_gemm(const SimtParams& p, cudaStream_t st) {
    if (p.G <= 0 || p.M <= 0 || p.N <= 0) return cudaSuccess;
    dim3 grid((p.N + SB - 1) / SB, (p.M + SB - 1) / SB, p.G);
    if (grid.z > 65535) return cudaErrorInvalidConfiguration;
    switch (p.mode) {
        case NS_GRAM: simt_gemm_kernel<NS_GRAM><<<grid, ST, 0, st>>>(p); break;
        case NS_POLY: simt_gemm_kernel<NS_POLY><<<grid, ST, 0, st>>>(p); break;
        default: simt_gemm_kernel<NS_APPLY><<<grid, ST, 0, st>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace muonh
