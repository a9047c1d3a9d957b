// HBM-bound kernels of the MuonH step: momentum (+ ||M||^2 + the Newton-
// Schulz input X), the hyperball retraction (||W - lr*O||^2 where the last
// apply GEMM has not already summed it, then the rescale), and the
// initial-norm capture.
//
// Method: Puro-2B digest (jacksunwei.me), section "The load-bearing tricks
// aren't in the abstract" -- Muon momentum orthogonalised by Newton-Schulz,
// and every weight matrix held at its initial Frobenius norm.  Model card
// (axforge.ai), section "Training": fp32 master weights and optimizer state.
//
// Work split: a chunk is a band of about 64 K elements (whole rows) of one
// matrix; every buffer keeps the matrix's own orientation, so each kernel
// streams row-major.  Each CTA takes one chunk and writes one fp64 partial
// sum; a one-warp-per-matrix finalize kernel adds a matrix's partials in a
// fixed order, so every norm is deterministic.

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
// K1: M <- beta*M + G; the Newton-Schulz input X is M (or with Nesterov
// momentum G + beta*M); X_op = bf16(X) and, unless D.fused has kFusedIn (the
// first apply GEMM then reads M itself), X_state = X, in the matrix's own
// orientation (unscaled: the 1/(||M||+eps) factor is folded into the
// Newton-Schulz epilogues); partial ||X||^2 per chunk.  With D.m null the
// input G itself is the Newton-Schulz input (standalone orthogonalisation).
// With `io` set, the CTA of each matrix's first chunk records where the
// matrix's input and weight are (NsIO, indexed by bucket-order position).
// ---------------------------------------------------------------------------
// Four gradient values at element e (a multiple of 4), fp32 or bf16 (the
// bf16 values widen exactly to fp32).
__device__ __forceinline__ float4 load_g4(const float* g, size_t e, bool bf16) {
    if (!bf16) return __ldcs(reinterpret_cast<const float4*>(g + e));
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(g) + e));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
}

__device__ __forceinline__ float load_g1(const float* g, size_t e, bool bf16) {
    if (!bf16) return g[e];
    return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(g)[e] << 16);
}

// The Newton-Schulz input of one element: the new momentum v, or with
// Nesterov momentum the look-ahead g + beta*v.
__device__ __forceinline__ float ns_in(float v, float g, float beta, bool nesterov) {
    return nesterov ? fmaf(beta, v, g) : v;
}

template <bool WRITE_XS>
__device__ __forceinline__ void momentum_chunk(const MatDesc& D, int r_begin, int r_end, float beta, bool nesterov,
                                               bool grad_bf16, float& acc) {
    const int cols = D.cols, ld = D.ld;
    if (ld == cols && (cols & 3) == 0) {
        // flat float4 stream; four vectors per thread in flight
        const size_t e0 = (size_t)r_begin * cols, e1 = (size_t)r_end * cols;
        constexpr int U = 4;
        size_t e = e0 + 4 * (size_t)threadIdx.x;
        for (; e + 4 * kThreads * (U - 1) < e1; e += 4 * kThreads * U) {
            float4 g[U], m[U];
#pragma unroll
            for (int u = 0; u < U; ++u) g[u] = load_g4(D.g, e + 4 * kThreads * u, grad_bf16);
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
                const float4 x = make_float4(ns_in(v.x, g[u].x, beta, nesterov), ns_in(v.y, g[u].y, beta, nesterov),
                                             ns_in(v.z, g[u].z, beta, nesterov), ns_in(v.w, g[u].w, beta, nesterov));
                if (WRITE_XS) *reinterpret_cast<float4*>(D.xs + f) = x;
                store_bf16x4(D.xo + f, x);
                acc = fmaf(x.x, x.x, acc); acc = fmaf(x.y, x.y, acc);
                acc = fmaf(x.z, x.z, acc); acc = fmaf(x.w, x.w, acc);
            }
        }
        for (; e < e1; e += 4 * kThreads) {
            const float4 g = load_g4(D.g, e, grad_bf16);
            float4 v = g;
            if (D.m) {
                const float4 m = *reinterpret_cast<const float4*>(D.m + e);
                v.x = fmaf(beta, m.x, v.x); v.y = fmaf(beta, m.y, v.y);
                v.z = fmaf(beta, m.z, v.z); v.w = fmaf(beta, m.w, v.w);
                *reinterpret_cast<float4*>(D.m + e) = v;
            }
            const float4 x = make_float4(ns_in(v.x, g.x, beta, nesterov), ns_in(v.y, g.y, beta, nesterov),
                                         ns_in(v.z, g.z, beta, nesterov), ns_in(v.w, g.w, beta, nesterov));
            if (WRITE_XS) *reinterpret_cast<float4*>(D.xs + e) = x;
            store_bf16x4(D.xo + e, x);
            acc = fmaf(x.x, x.x, acc); acc = fmaf(x.y, x.y, acc);
            acc = fmaf(x.z, x.z, acc); acc = fmaf(x.w, x.w, acc);
        }
    } else {
        // any row length: the chunk's elements in row-major order
        const size_t n = (size_t)(r_end - r_begin) * cols;
        for (size_t e = threadIdx.x; e < n; e += kThreads) {
            const size_t r = r_begin + e / cols, c = e % cols;
            const size_t wi = r * cols + c, xi = r * ld + c;
            const float g = load_g1(D.g, wi, grad_bf16);
            float m = g;
            if (D.m) { m = fmaf(beta, D.m[wi], m); D.m[wi] = m; }
            const float x = ns_in(m, g, beta, nesterov);
            if (WRITE_XS) D.xs[xi] = x;
            D.xo[xi] = __float2bfloat16_rn(x);
            acc = fmaf(x, x, acc);
        }
    }
}

__global__ void __launch_bounds__(kThreads)
momentum_kernel(const __grid_constant__ DescBatch b, float beta, double* __restrict__ partials, NsIO* io,
                bool nesterov, bool grad_bf16) {
    __shared__ double red[kThreads / 32];
    const int chunk = b.chunk_begin + blockIdx.x;
    const int mi = find_matrix(b, chunk);
    const MatDesc& D = b.d[mi];
    if (D.fused & kFusedAll) return;
    const int cols = D.cols;
    if (io && chunk == D.chunk0 && threadIdx.x == 0) {
        NsIO r;
        r.src = D.m ? D.m : D.g;
        r.w = D.w;
        r.wb = D.wb;
        io[b.first + mi] = r;
    }
    const int cr = chunk_rows_for(D.rows, cols);
    const int r_begin = (chunk - D.chunk0) * cr;
    const int r_end = min(D.rows, r_begin + cr);
    float acc = 0.f;
    if (D.fused & kFusedIn)
        momentum_chunk<false>(D, r_begin, r_end, beta, nesterov, grad_bf16, acc);
    else
        momentum_chunk<true>(D, r_begin, r_end, beta, nesterov, grad_bf16, acc);
    double s = block_sum<kThreads>((double)acc, red);
    if (threadIdx.x == 0) partials[chunk] = s;
}

// Per matrix: nu^2 = sum of its partials (index order); 1/(nu+eps) factors;
// oscale = the update scale (times 1/(nu+eps) when no Newton-Schulz
// iteration runs, X_state then holding the unscaled input).
__global__ void momentum_finalize(const __grid_constant__ DescBatch b, const double* __restrict__ partials,
                                  Scalars sc, float eps, int scale_mode, bool no_iterations) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= b.n) return;
    const MatDesc& D = b.d[i];
    if (D.fused & kFusedAll) return;
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
    const float us = update_scale(D.rows, D.cols, scale_mode);
    sc.oscale[p] = no_iterations ? us * inv : us;
}

// ---------------------------------------------------------------------------
// Hyperball retraction, W <- r0 * U / ||U||_F with U = W - lr*O.  One chunk
// in one of three forms (O = X_state, same orientation as W, row stride D.ld):
//   HB_NORM   partial ||U||^2 (U = fma(-lr, O, W))
//   HB_APPLY  W <- factor*U, W_bf16 = bf16(W)   (U recomputed identically)
//   HB_SCALE  W <- factor*U, W_bf16 = bf16(W), where X_state already holds U
//             (written by the last apply GEMM, which also summed ||U||^2)
// ---------------------------------------------------------------------------
enum { HB_NORM = 0, HB_APPLY = 1, HB_SCALE = 2, HB_MUON = 3 };

// HB_MUON is plain Muon's weight update on the same stream:
// W <- f*W - lr*O (f = 1 - lr*weight_decay), W_bf16 = bf16(W).
template <int HB>
__device__ __forceinline__ void hyperball_chunk(const MatDesc& D, int r_begin, int r_end, float nlr, float f,
                                                float& acc) {
    constexpr bool WRITE = HB != HB_NORM;
    constexpr bool READ_W = HB != HB_SCALE;
    const int cols = D.cols, ld = D.ld;
    if (ld == cols && (cols & 3) == 0) {
        const size_t e0 = (size_t)r_begin * cols, e1 = (size_t)r_end * cols;
        constexpr int U = 4;
        // U for four values (from W and O, or as read); write f*U or add ||U||^2
        auto visit4 = [&](float4 w, float4 o, size_t widx) {
            float4 u;
            if (HB == HB_MUON) {
                u.x = fmaf(nlr, o.x, f * w.x); u.y = fmaf(nlr, o.y, f * w.y);
                u.z = fmaf(nlr, o.z, f * w.z); u.w = fmaf(nlr, o.w, f * w.w);
            } else if (READ_W) {
                u.x = fmaf(nlr, o.x, w.x); u.y = fmaf(nlr, o.y, w.y);
                u.z = fmaf(nlr, o.z, w.z); u.w = fmaf(nlr, o.w, w.w);
            } else {
                u = o;
            }
            if (HB != HB_MUON && WRITE) {
                u.x *= f; u.y *= f; u.z *= f; u.w *= f;
            }
            if (WRITE) {
                *reinterpret_cast<float4*>(D.w + widx) = u;
                if (D.wb) store_bf16x4(reinterpret_cast<__nv_bfloat16*>(D.wb) + widx, u);
            } else {
                acc = fmaf(u.x, u.x, acc); acc = fmaf(u.y, u.y, acc);
                acc = fmaf(u.z, u.z, acc); acc = fmaf(u.w, u.w, acc);
            }
        };
        const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
        size_t e = e0 + 4 * (size_t)threadIdx.x;
        for (; e + 4 * kThreads * (U - 1) < e1; e += 4 * kThreads * U) {
            float4 w[U], o[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                w[u] = READ_W ? *reinterpret_cast<const float4*>(D.w + e + 4 * kThreads * u) : zero4;
                o[u] = __ldcs(reinterpret_cast<const float4*>(D.xs + e + 4 * kThreads * u));
            }
#pragma unroll
            for (int u = 0; u < U; ++u) visit4(w[u], o[u], e + 4 * kThreads * u);
        }
        for (; e < e1; e += 4 * kThreads)
            visit4(READ_W ? *reinterpret_cast<const float4*>(D.w + e) : zero4,
                   __ldcs(reinterpret_cast<const float4*>(D.xs + e)), e);
    } else {
        const size_t n = (size_t)(r_end - r_begin) * cols;
        for (size_t e = threadIdx.x; e < n; e += kThreads) {
            const size_t r = r_begin + e / cols, c = e % cols;
            const size_t wi = r * cols + c;
            const float o = D.xs[r * ld + c];
            const float u = HB == HB_MUON ? fmaf(nlr, o, f * D.w[wi]) : (READ_W ? fmaf(nlr, o, D.w[wi]) : o);
            if (WRITE) {
                const float y = HB == HB_MUON ? u : u * f;
                D.w[wi] = y;
                if (D.wb) D.wb[wi] = bf16_bits(y);
            } else {
                acc = fmaf(u, u, acc);
            }
        }
    }
}

// Partial ||W - lr*O||^2 per chunk, for the matrices without kFusedOut
// (their last apply GEMM left O in X_state).
__global__ void __launch_bounds__(kThreads)
hyperball_norm_kernel(const __grid_constant__ DescBatch b, float lr, double* __restrict__ partials,
                      const float* __restrict__ o_scale) {
    __shared__ double red[kThreads / 32];
    const int chunk = b.chunk_begin + blockIdx.x;
    const int mi = find_matrix(b, chunk);
    const MatDesc& D = b.d[mi];
    if (D.fused & (kFusedOut | kFusedAll)) return;
    const int p = b.first + mi;
    const int cr = chunk_rows_for(D.rows, D.cols);
    const int r_begin = (chunk - D.chunk0) * cr;
    const int r_end = min(D.rows, r_begin + cr);
    // O = o_scale * X_state (o_scale is 1/(||M||+eps) when no Newton-Schulz
    // iteration ran, X_state then holding the unscaled momentum)
    const float nlr = o_scale ? -lr * o_scale[p] : -lr;
    float acc = 0.f;
    hyperball_chunk<HB_NORM>(D, r_begin, r_end, nlr, 0.f, acc);
    double s = block_sum<kThreads>((double)acc, red);
    if (threadIdx.x == 0) partials[chunk] = s;
}

// W <- factor * U, W_bf16 = bf16(W): U from W - lr*O, or read from X_state
// for the matrices with kFusedOut.  Matrices with a status bit keep W.
__global__ void __launch_bounds__(kThreads)
hyperball_finish_kernel(const __grid_constant__ DescBatch b, float lr, const float* __restrict__ factor,
                        const uint32_t* __restrict__ flags, const float* __restrict__ o_scale) {
    const int chunk = b.chunk_begin + blockIdx.x;
    const int mi = find_matrix(b, chunk);
    const MatDesc& D = b.d[mi];
    const int p = b.first + mi;
    if ((D.fused & kFusedAll) || flags[p] != 0) return;  // W stays as it was
    const int cr = chunk_rows_for(D.rows, D.cols);
    const int r_begin = (chunk - D.chunk0) * cr;
    const int r_end = min(D.rows, r_begin + cr);
    float unused = 0.f;
    if (D.fused & kFusedOut) {
        hyperball_chunk<HB_SCALE>(D, r_begin, r_end, 0.f, factor[p], unused);
    } else {
        const float nlr = o_scale ? -lr * o_scale[p] : -lr;
        hyperball_chunk<HB_APPLY>(D, r_begin, r_end, nlr, factor[p], unused);
    }
}

// Plain Muon's weight update for the matrices whose last apply GEMM did not
// write it (no kFusedOutW): W <- (1 - lr*wd)*W - lr*O, W_bf16 = bf16(W).
// Matrices with a status bit keep W.
__global__ void __launch_bounds__(kThreads)
muon_finish_kernel(const __grid_constant__ DescBatch b, float lr, float wdecay, const uint32_t* __restrict__ flags,
                   const float* __restrict__ o_scale) {
    const int chunk = b.chunk_begin + blockIdx.x;
    const int mi = find_matrix(b, chunk);
    const MatDesc& D = b.d[mi];
    const int p = b.first + mi;
    if ((D.fused & (kFusedOutW | kFusedAll)) || flags[p] != 0) return;
    const int cr = chunk_rows_for(D.rows, D.cols);
    const int r_begin = (chunk - D.chunk0) * cr;
    const int r_end = min(D.rows, r_begin + cr);
    const float nlr = o_scale ? -lr * o_scale[p] : -lr;
    float unused = 0.f;
    hyperball_chunk<HB_MUON>(D, r_begin, r_end, nlr, wdecay, unused);
}

// Standalone orthogonalisation output: out (D.w) = o_scale * X_state, as
// fp32 or, with out_bf16, as bf16 (round to nearest even of that fp32 value).
__global__ void __launch_bounds__(kThreads)
emit_kernel(const __grid_constant__ DescBatch b, const float* __restrict__ o_scale, bool out_bf16) {
    const int chunk = b.chunk_begin + blockIdx.x;
    const int mi = find_matrix(b, chunk);
    const MatDesc& D = b.d[mi];
    const int p = b.first + mi;
    const int cols = D.cols, ld = D.ld;
    const int cr = chunk_rows_for(D.rows, cols);
    const int r_begin = (chunk - D.chunk0) * cr;
    const int r_end = min(D.rows, r_begin + cr);
    const float os = o_scale ? o_scale[p] : 1.f;
    const size_t n = (size_t)(r_end - r_begin) * cols;
    uint16_t* wb = reinterpret_cast<uint16_t*>(D.w);
    for (size_t e = threadIdx.x; e < n; e += kThreads) {
        const size_t r = r_begin + e / cols, c = e % cols;
        const float y = os * D.xs[r * ld + c];
        if (out_bf16)
            wb[r * cols + c] = bf16_bits(y);
        else
            D.w[r * cols + c] = y;
    }
}

// Per matrix: rho^2 = sum of partials in index order (the hyperball norm
// kernel's per-chunk partials, or, with kFusedOut, the last apply GEMM's
// per-warp partials at upart[D.part0..]); factor = r0 / rho, or a status bit.
// One warp per matrix: lane k adds partials k, k+32, ... in order, then a
// fixed shuffle tree combines the lanes, so the sum is deterministic.
__global__ void hyperball_finalize(const __grid_constant__ DescBatch b, const double* __restrict__ partials,
                                   const double* __restrict__ upart, Scalars sc, const float* __restrict__ r0) {
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= b.n) return;
    const MatDesc& D = b.d[i];
    if (D.fused & kFusedAll) return;
    const int p = b.first + i;
    const bool from_gemm = (D.fused & kFusedOut) != 0;
    const double* src = from_gemm ? upart + (size_t)D.part0 : partials + D.chunk0;
    const int cnt = from_gemm ? D.npart : chunks_for(D.rows, D.cols);
    double s = 0.0;
    for (int k = lane; k < cnt; k += 32) s += src[k];
    s = warp_sum(s);
    if (lane != 0) return;
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
cudaError_t launch_momentum(const DescBatch& b, float beta, double* partials, NsIO* io, bool nesterov,
                            bool grad_bf16, cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    momentum_kernel<<<nblk, kThreads, 0, st>>>(b, beta, partials, io, nesterov, grad_bf16);
    return cudaGetLastError();
}

cudaError_t launch_momentum_finalize(const DescBatch& b, const double* partials, const Scalars& sc,
                                     float eps, int scale_mode, bool no_iterations, cudaStream_t st) {
    momentum_finalize<<<(b.n + 127) / 128, 128, 0, st>>>(b, partials, sc, eps, scale_mode, no_iterations);
    return cudaGetLastError();
}

cudaError_t launch_hyperball_norm(const DescBatch& b, float lr, double* partials, const float* o_scale,
                                  cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    hyperball_norm_kernel<<<nblk, kThreads, 0, st>>>(b, lr, partials, o_scale);
    return cudaGetLastError();
}

cudaError_t launch_hyperball_finalize(const DescBatch& b, const double* partials, const double* upart,
                                      const Scalars& sc, const float* r0, cudaStream_t st) {
    hyperball_finalize<<<(b.n + 3) / 4, 128, 0, st>>>(b, partials, upart, sc, r0);
    return cudaGetLastError();
}

cudaError_t launch_hyperball_finish(const DescBatch& b, float lr, const Scalars& sc, const float* o_scale,
                                    cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    hyperball_finish_kernel<<<nblk, kThreads, 0, st>>>(b, lr, sc.factor, sc.flags, o_scale);
    return cudaGetLastError();
}

cudaError_t launch_muon_finish(const DescBatch& b, float lr, float wdecay, const Scalars& sc, const float* o_scale,
                               cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    muon_finish_kernel<<<nblk, kThreads, 0, st>>>(b, lr, wdecay, sc.flags, o_scale);
    return cudaGetLastError();
}

cudaError_t launch_emit(const DescBatch& b, const float* o_scale, bool out_bf16, cudaStream_t st) {
    const int nblk = b.chunk_end - b.chunk_begin;
    if (nblk <= 0) return cudaSuccess;
    emit_kernel<<<nblk, kThreads, 0, st>>>(b, o_scale, out_bf16);
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
