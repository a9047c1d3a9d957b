// HBM-bound kernels of the MuonH step: momentum (+ ||M||^2 + the Newton-
// Schulz input X), the hyperball retraction (||W - lr*O||^2, then the
// rescale), and the initial-norm capture.
//
// Method: Puro-2B digest (jacksunwei.me), section "The load-bearing tricks
// aren't in the abstract" -- Muon momentum orthogonalised by Newton-Schulz,
// and every weight matrix held at its initial Frobenius norm.  Model card
// (axforge.ai), section "Training": fp32 master weights and optimizer state.
//
// Work split: a chunk is a band of rows of one matrix (64-row bands for
// tall matrices, whose X is the transpose).  Each CTA takes one chunk and
// writes one fp64 partial sum; a one-thread-per-matrix finalize kernel adds
// a matrix's partials in index order, so every norm is deterministic.

#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace muonh {

__device__ uint32_t g_status = 0;

constexpr int kThreads = 256;

__device__ __forceinline__ int find_matrix(const DescBatch& b, int chunk) {
    int lo = 0, hi = b.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (b.d[mid].chunk0 <= chunk) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

// ---------------------------------------------------------------------------
// K1: M <- beta*M + G; X_state = M and X_op = bf16(M) in X orientation
// (unscaled: the 1/(||M||+eps) factor is folded into the Newton-Schulz
// epilogues); partial ||M||^2 per chunk.  With D.m null the input G itself
// is the Newton-Schulz input (standalone orthogonalisation).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
momentum_kernel(const __grid_constant__ DescBatch b, float beta, double* __restrict__ partials) {
    __shared__ float tile[kTile][kTile + 1];
    __shared__ double red[kThreads / 32];
    const int chunk = b.chunk_begin + blockIdx.x;
    const MatDesc& D = b.d[find_matrix(b, chunk)];
    const int rows = D.rows, cols = D.cols, ld = D.ld;
    const int cr = chunk_rows_for(rows, cols);
    const int r_begin = (chunk - D.chunk0) * cr;
    const int r_end = min(rows, r_begin + cr);
    float acc = 0.f;

    if (!is_transposed(rows, cols)) {
        if (ld == cols && (cols & 3) == 0) {
            // flat float4 stream; four vectors per thread in flight
            const size_t e0 = (size_t)r_begin * cols, e1 = (size_t)r_end * cols;
            constexpr int U = 4;
            size_t e = e0 + 4 * (size_t)threadIdx.x;
            for (; e + 4 * kThreads * (U - 1) < e1; e += 4 * kThreads * U) {
                float4 g[U], m[U];
#pragma unroll
                for (int u = 0; u < U; ++u) g[u] = __ldcs(reinterpret_cast<const float4*>(D.g + e + 4 * kThreads * u));
                if (D.m) {
#pragma unroll
                    for (int u = 0; u < U; ++u) m[u] = __ldcs(reinterpret_cast<const float4*>(D.m + e + 4 * kThreads * u));
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const size_t f = e + 4 * kThreads * u;
                    float4 v = g[u];
                    if (D.m) {
                        v.x = fmaf(beta, m[u].x, v.x); v.y = fmaf(beta, m[u].y, v.y);
                        v.z = fmaf(beta, m[u].z, v.z); v.w = fmaf(beta, m[u].w, v.w);
                        *reinterpret_cast<float4*>(D.m + f) = v;
                    }
                    *reinterpret_cast<float4*>(D.xs + f) = v;
                    store_bf16x4(D.xo + f, v);
                    acc = fmaf(v.x, v.x, acc); acc = fmaf(v.y, v.y, acc);
                    acc = fmaf(v.z, v.z, acc); acc = fmaf(v.w, v.w, acc);
                }
            }
            for (; e < e1; e += 4 * kThreads) {
                float4 v = __ldcs(reinterpret_cast<const float4*>(D.g + e));
                if (D.m) {
                    const float4 m = *reinterpret_cast<const float4*>(D.m + e);
                    v.x = fmaf(beta, m.x, v.x); v.y = fmaf(beta, m.y, v.y);
                    v.z = fmaf(beta, m.z, v.z); v.w = fmaf(beta, m.w, v.w);
                    *reinterpret_cast<float4*>(D.m + e) = v;
                }
                *reinterpret_cast<float4*>(D.xs + e) = v;
                store_bf16x4(D.xo + e, v);
                acc = fmaf(v.x, v.x, acc); acc = fmaf(v.y, v.y, acc);
                acc = fmaf(v.z, v.z, acc); acc = fmaf(v.w, v.w, acc);
            }
        } else {
            for (int r = r_begin; r < r_end; ++r) {
                for (int c = threadIdx.x; c < cols; c += kThreads) {
                    const size_t e = (size_t)r * cols + c;
                    float m = D.g[e];
                    if (D.m) { m = fmaf(beta, D.m[e], m); D.m[e] = m; }
                    D.xs[(size_t)r * ld + c] = m;
                    D.xo[(size_t)r * ld + c] = __float2bfloat16_rn(m);
                    acc = fmaf(m, m, acc);
                }
            }
        }
    } else {
        // X = M^T: stage 64x64 tiles in shared memory, write them transposed.
        const bool vec_ok = (cols & 3) == 0;
        for (int c0 = 0; c0 < cols; c0 += kTile) {
            if (vec_ok && r_begin + kTile <= r_end && c0 + kTile <= cols) {
                // full tile: float4 along W rows, then float4 along X rows
                const int lr = threadIdx.x >> 4, lc = (threadIdx.x & 15) * 4;
                float4 g[4], m[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    g[k] = __ldcs(reinterpret_cast<const float4*>(D.g + (size_t)(r_begin + lr + 16 * k) * cols + c0 + lc));
                if (D.m) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        m[k] = __ldcs(reinterpret_cast<const float4*>(D.m + (size_t)(r_begin + lr + 16 * k) * cols + c0 + lc));
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float4 v = g[k];
                    if (D.m) {
                        v.x = fmaf(beta, m[k].x, v.x); v.y = fmaf(beta, m[k].y, v.y);
                        v.z = fmaf(beta, m[k].z, v.z); v.w = fmaf(beta, m[k].w, v.w);
                        *reinterpret_cast<float4*>(D.m + (size_t)(r_begin + lr + 16 * k) * cols + c0 + lc) = v;
                    }
                    acc = fmaf(v.x, v.x, acc); acc = fmaf(v.y, v.y, acc);
                    acc = fmaf(v.z, v.z, acc); acc = fmaf(v.w, v.w, acc);
                    float* tr = &tile[lr + 16 * k][lc];
                    tr[0] = v.x; tr[1] = v.y; tr[2] = v.z; tr[3] = v.w;
                }
                __syncthreads();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int cc = lr + 16 * k, rr = lc;   // X row c0+cc, X cols r_begin+rr..+3
                    const float4 v = make_float4(tile[rr][cc], tile[rr + 1][cc], tile[rr + 2][cc], tile[rr + 3][cc]);
                    const size_t o = (size_t)(c0 + cc) * ld + r_begin + rr;
                    *reinterpret_cast<float4*>(D.xs + o) = v;
                    store_bf16x4(D.xo + o, v);
                }
                __syncthreads();
                continue;
            }
            const int tr = threadIdx.x & 63, tq = threadIdx.x >> 6;   // 64 x 4
            for (int i = 0; i < kTile; i += 4) {
                const int r = r_begin + i + tq, c = c0 + tr;
                if (r < r_end && c < cols) {
                    const size_t e = (size_t)r * cols + c;
                    float m = D.g[e];
                    if (D.m) { m = fmaf(beta, D.m[e], m); D.m[e] = m; }
                    acc = fmaf(m, m, acc);
                    tile[i + tq][tr] = m;
                }
            }
            __syncthreads();
            for (int i = 0; i < kTile; i += 4) {
                const int c = c0 + i + tq, r = r_begin + tr;
                if (r < r_end && c < cols) {
                    const float v = tile[tr][i + tq];
                    D.xs[(size_t)c * ld + r] = v;
                    D.xo[(size_t)c * ld + r] = __float2bfloat16_rn(v);
                }
            }
            __syncthreads();
        }
    }
    double s = block_sum<kThreads>((double)acc, red);
    if (threadIdx.x == 0) partials[chunk] = s;
}

// Per matrix: nu^2 = sum of its partials (index order); 1/(nu+eps) factors.
__global__ void momentum_finalize(const __grid_constant__ DescBatch b, const double* __restrict__ partials,
                                  Scalars sc, float eps) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= b.n) return;
    const MatDesc& D = b.d[i];
    const int p = b.first + i;
    const int nch = chunks_for(D.rows, D.cols);
    double s = 0.0;
    for (int k = 0; k < nch; ++k) s += partials[D.chunk0 + k];
    sc.nu2[p] = s;
    uint32_t f = 0;
    float inv = 0.f;
    if (!isfinite(s)) {
        f = MUONH_STATUS_NONFINITE_INPUT;
        raise_status(&g_status, f);
    } else {
        inv = (float)(1.0 / (sqrt(s) + (double)eps));
    }
    sc.inv_nu[p] = inv;
    sc.inv_nu2[p] = inv * inv;
    sc.flags[p] = f;
}

// ---------------------------------------------------------------------------
// K3a: partial ||W - lr*O||^2 per chunk (O = X_state, read transposed for
// tall matrices).  K3b: W <- factor*(W - lr*O), W_bf16 = bf16(W).
// Both evaluate U = fma(-lr, O, W) identically.
// ---------------------------------------------------------------------------
template <bool APPLY>
__global__ void __launch_bounds__(kThreads)
hyperball_kernel(const __grid_constant__ DescBatch b, float lr, double* __restrict__ partials,
                 const float* __restrict__ factor, const uint32_t* __restrict__ flags,
                 const float* __restrict__ o_scale) {
    __shared__ float tile[kTile][kTile + 1];
    __shared__ double red[kThreads / 32];
    const int chunk = b.chunk_begin + blockIdx.x;
    const int mi = find_matrix(b, chunk);
    const MatDesc& D = b.d[mi];
    const int p = b.first + mi;
    const int rows = D.rows, cols = D.cols, ld = D.ld;
    const int cr = chunk_rows_for(rows, cols);
    const int r_begin = (chunk - D.chunk0) * cr;
    const int r_end = min(rows, r_begin + cr);
    float f = 0.f;
    if (APPLY) {
        if (flags[p] != 0) return;  // W stays as it was
        f = factor[p];
    }
    // O = o_scale * X_state (o_scale is 1/(||M||+eps) when no Newton-Schulz
    // iteration ran, X_state then holding the unscaled momentum)
    const float nlr = o_scale ? -lr * o_scale[p] : -lr;
    float acc = 0.f;

    // U = W - lr*O for four values; APPLY: W <- f*U (+ bf16 copy), else ||U||^2
    auto visit4 = [&](float4 w, float4 o, size_t widx) {
        float4 u;
        u.x = fmaf(nlr, o.x, w.x); u.y = fmaf(nlr, o.y, w.y);
        u.z = fmaf(nlr, o.z, w.z); u.w = fmaf(nlr, o.w, w.w);
        if (APPLY) {
            u.x *= f; u.y *= f; u.z *= f; u.w *= f;
            *reinterpret_cast<float4*>(D.w + widx) = u;
            if (D.wb) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(u.x, u.y);
                __nv_bfloat162 hi = __floats2bfloat162_rn(u.z, u.w);
                uint2 v;
                v.x = *reinterpret_cast<uint32_t*>(&lo);
                v.y = *reinterpret_cast<uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(D.wb + widx) = v;
            }
        } else {
            acc = fmaf(u.x, u.x, acc); acc = fmaf(u.y, u.y, acc);
            acc = fmaf(u.z, u.z, acc); acc = fmaf(u.w, u.w, acc);
        }
    };

    if (!is_transposed(rows, cols)) {
        if (ld == cols && (cols & 3) == 0) {
            const size_t e0 = (size_t)r_begin * cols, e1 = (size_t)r_end * cols;
            constexpr int U = 4;
            size_t e = e0 + 4 * (size_t)threadIdx.x;
            for (; e + 4 * kThreads * (U - 1) < e1; e += 4 * kThreads * U) {
                float4 w[U], o[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    w[u] = *reinterpret_cast<const float4*>(D.w + e + 4 * kThreads * u);
                    o[u] = __ldcs(reinterpret_cast<const float4*>(D.xs + e + 4 * kThreads * u));
                }
#pragma unroll
                for (int u = 0; u < U; ++u) visit4(w[u], o[u], e + 4 * kThreads * u);
            }
            for (; e < e1; e += 4 * kThreads)
                visit4(*reinterpret_cast<const float4*>(D.w + e), __ldcs(reinterpret_cast<const float4*>(D.xs + e)), e);
        } else {
            for (int r = r_begin; r < r_end; ++r) {
                for (int c = threadIdx.x; c < cols; c += kThreads) {
                    const size_t e = (size_t)r * cols + c;
                    float u = fmaf(nlr, D.xs[(size_t)r * ld + c], D.w[e]);
                    if (APPLY) {
                        u *= f;
                        D.w[e] = u;
                        if (D.wb) D.wb[e] = bf16_bits(u);
                    } else {
                        acc = fmaf(u, u, acc);
                    }
                }
            }
        }
    } else {
        const bool vec_ok = (cols & 3) == 0;
        for (int c0 = 0; c0 < cols; c0 += kTile) {
            if (vec_ok && r_begin + kTile <= r_end && c0 + kTile <= cols) {
                // full tile: X rows (W columns) loaded as float4 along W rows
                const int lr = threadIdx.x >> 4, lc = (threadIdx.x & 15) * 4;
                float4 x[4], w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    x[k] = __ldcs(reinterpret_cast<const float4*>(D.xs + (size_t)(c0 + lr + 16 * k) * ld + r_begin + lc));
                    w[k] = *reinterpret_cast<const float4*>(D.w + (size_t)(r_begin + lr + 16 * k) * cols + c0 + lc);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // tile[W row][W col]
                    tile[lc][lr + 16 * k] = x[k].x;
                    tile[lc + 1][lr + 16 * k] = x[k].y;
                    tile[lc + 2][lr + 16 * k] = x[k].z;
                    tile[lc + 3][lr + 16 * k] = x[k].w;
                }
                __syncthreads();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float* t = &tile[lr + 16 * k][lc];
                    visit4(w[k], make_float4(t[0], t[1], t[2], t[3]),
                           (size_t)(r_begin + lr + 16 * k) * cols + c0 + lc);
                }
                __syncthreads();
                continue;
            }
            const int tr = threadIdx.x & 63, tq = threadIdx.x >> 6;
            // X_state rows c (contiguous along r) -> tile[c - c0][r - r_begin]
            for (int i = 0; i < kTile; i += 4) {
                const int c = c0 + i + tq, r = r_begin + tr;
                if (r < r_end && c < cols) tile[i + tq][tr] = D.xs[(size_t)c * ld + r];
            }
            __syncthreads();
            for (int i = 0; i < kTile; i += 4) {
                const int r = r_begin + i + tq, c = c0 + tr;
                if (r < r_end && c < cols) {
                    const size_t e = (size_t)r * cols + c;
                    float u = fmaf(nlr, tile[tr][i + tq], D.w[e]);
                    if (APPLY) {
                        u *= f;
                        D.w[e] = u;
                        if (D.wb) D.wb[e] = bf16_bits(u);
                    } else {
                        acc = fmaf(u, u, acc);
                    }
                }
            }
            __syncthreads();
        }
    }
    if (!APPLY) {
        double s = block_sum<kThreads>((double)acc, red);
        if (threadIdx.x == 0) partials[chunk] = s;
    }
}

// Standalone orthogonalisation output: out (W orientation, D.w) = o_scale * X.
__global__ void __launch_bounds__(kThreads)
emit_kernel(const __grid_constant__ DescBatch b, const float* __restrict__ o_scale) {
    __shared__ float tile[kTile][kTile + 1];
    const int chunk = b.chunk_begin + blockIdx.x;
    const int mi = find_matrix(b, chunk);
    const MatDesc& D = b.d[mi];
    const int p = b.first + mi;
    const int rows = D.rows, cols = D.cols, ld = D.ld;
    const int cr = chunk_rows_for(rows, cols);
    const int r_begin = (chunk - D.chunk0) * cr;
    const int r_end = min(rows, r_begin + cr);
    const float os = o_scale ? o_scale[p] : 1.f;
    if (!is_transposed(rows, cols)) {
        for (int r = r_begin; r < r_end; ++r)
            for (int c = threadIdx.x; c < cols; c += kThreads)
                D.w[(size_t)r * cols + c] = os * D.xs[(size_t)r * ld + c];
    } else {
        const int tr = threadIdx.x & 63, tq = threadIdx.x >> 6;
        for (int c0 = 0; c0 < cols; c0 += kTile) {
            for (int i = 0; i < kTile; i += 4) {
                const int c = c0 + i + tq, r = r_begin + tr;
                if (r < r_end && c < cols) tile[i + tq][tr] = D.xs[(size_t)c * ld + r];
            }
            __syncthreads();
            for (int i = 0; i < kTile; i += 4) {
                const int r = r_begin + i + tq, c = c0 + tr;
                if (r < r_end && c < cols) D.w[(size_t)r * cols + c] = os * tile[tr][i + tq];
            }
            __syncthreads();
        }
    }
}

// Per matrix: rho^2 = sum of partials; factor = r0 / rho, or a status bit.
__global__ void hyperball_finalize(const __grid_constant__ DescBatch b, const double* __restrict__ partials,
                                   Scalars sc, const float* __restrict__ r0) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= b.n) return;
    const MatDesc& D = b.d[i];
    const int p = b.first + i;
    const int nch = chunks_for(D.rows, D.cols);
    double s = 0.0;
    for (int k = 0; k < nch; ++k) s += partials[D.chunk0 + k];
    sc.rho2[p] = s;
    uint32_t f = sc.flags[p];
    float fac = 0.f;
    if (f == 0) {
        if (!isfinite(s) || s == 0.0) {
            f = MUONH_STATUS_DEGENERATE_NORM;
            raise_status(&g_status, f);
        } else {
            fac = (float)((double)r0[D.user_index] / sqrt(s));
        }
    }
    sc.flags[p] = f;
    sc.factor[p] = fac;
}

// ---------------------------------------------------------------------------
// r0 capture: one 8-CTA cluster per matrix; each CTA sums the squares of one
// eighth of the matrix, rank 0 adds the eight block sums in rank order via
// distributed shared memory.  Needs no scratch memory.
// ---------------------------------------------------------------------------
constexpr int kCaptureCluster = 8;

__global__ void __cluster_dims__(kCaptureCluster, 1, 1) __launch_bounds__(kThreads)
capture_norms_kernel(const __grid_constant__ DescBatch b, float* __restrict__ r0) {
    __shared__ double red[kThreads / 32];
    __shared__ double block_total;
    cg::cluster_group cluster = cg::this_cluster();
    const int mi = blockIdx.x / kCaptureCluster;
    const int rank = (int)cluster.block_rank();
    const MatDesc& D = b.d[mi];
    const size_t total = (size_t)D.rows * D.cols;
    const size_t per = ((total + kCaptureCluster - 1) / kCaptureCluster + 3) & ~(size_t)3;
    const size_t e0 = min(total, per * rank), e1 = min(total, e0 + per);
    float acc = 0.f;
    // per and e0 are multiples of 4 and w is 16-byte aligned: vector body, scalar tail.
    const size_t v1 = e0 + ((e1 - e0) & ~(size_t)3);
    for (size_t e = e0 + 4 * (size_t)threadIdx.x; e < v1; e += 4 * kThreads) {
        float4 w = *reinterpret_cast<const float4*>(D.w + e);
        acc = fmaf(w.x, w.x, acc); acc = fmaf(w.y, w.y, acc);
        acc = fmaf(w.z, w.z, acc); acc = fmaf(w.w, w.w, acc);
    }
    for (size_t e = v1 + threadIdx.x; e < e1; e += kThreads) acc = fmaf(D.w[e], D.w[e], acc);
    double s = block_sum<kThreads>((double)acc, red);
    if (threadIdx.x == 0) block_total = s;
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0) {
        double t = 0.0;
        for (int k = 0; k < kCaptureCluster; ++k) t += *cluster.map_shared_rank(&block_total, k);
        r0[D.user_index] = (float)sqrt(t);
    }
    cluster.sync();
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
cudaError_t launch_momentum(const DescBatch& b, float beta, double* partials, cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    momentum_kernel<<<nblk, kThreads, 0, st>>>(b, beta, partials);
    return cudaGetLastError();
}

cudaError_t launch_momentum_finalize(const DescBatch& b, const double* partials, const Scalars& sc,
                                     float eps, cudaStream_t st) {
    momentum_finalize<<<(b.n + 127) / 128, 128, 0, st>>>(b, partials, sc, eps);
    return cudaGetLastError();
}

cudaError_t launch_hyperball_norm(const DescBatch& b, float lr, double* partials, const float* o_scale,
                                  cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    hyperball_kernel<false><<<nblk, kThreads, 0, st>>>(b, lr, partials, nullptr, nullptr, o_scale);
    return cudaGetLastError();
}

cudaError_t launch_hyperball_finalize(const DescBatch& b, const double* partials, const Scalars& sc,
                                      const float* r0, cudaStream_t st) {
    hyperball_finalize<<<(b.n + 127) / 128, 128, 0, st>>>(b, partials, sc, r0);
    return cudaGetLastError();
}

cudaError_t launch_hyperball_apply(const DescBatch& b, float lr, const Scalars& sc, const float* o_scale,
                                   cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    hyperball_kernel<true><<<nblk, kThreads, 0, st>>>(b, lr, nullptr, sc.factor, sc.flags, o_scale);
    return cudaGetLastError();
}

cudaError_t launch_emit(const DescBatch& b, const float* o_scale, cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    emit_kernel<<<nblk, kThreads, 0, st>>>(b, o_scale);
    return cudaGetLastError();
}

// Device address of this device's status word (cudaGetSymbolAddress; the
// calling thread's current device).
cudaError_t status_word(uint32_t** ptr) { return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_status); }

cudaError_t launch_capture_norms(const DescBatch& b, float* r0, cudaStream_t st) {
    capture_norms_kernel<<<b.n * kCaptureCluster, kThreads, 0, st>>>(b, r0);
    return cudaGetLastError();
}

}  // namespace muonh
