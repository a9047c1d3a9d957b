// The whole MuonH (or plain Muon) step for matrices whose sides are both at
// most 256, with every Newton-Schulz iteration on chip (Puro-2B digest,
// section "The load-bearing tricks aren't in the abstract": Muon's
// Newton-Schulz iterations, then the hyperball projection).
//
// One CTA pair (cluster of 2, tcgen05 cta_group::2) per matrix, persistent
// over a list of matrices.  X is held in its wide orientation s x l (a tall
// matrix is transposed while it is loaded and written back), zero-padded to
// 256 x 256; CTA r owns rows 128r..128r+127.
//
//   TMEM (512 columns, fp32):  [0, 256)   the state X (this CTA's 128 rows)
//                              [256, 512) the accumulator
//   shared memory, bf16, 128-byte swizzle (tensor-core operand layouts):
//     XR  this CTA's 128 rows of X, K-major        (Gram operand)
//     XC  all 256 rows x this CTA's 128 columns of X, MN-major (apply operand),
//         written by both CTAs through distributed shared memory
//     AR  this CTA's 128 rows of A, then of B, K-major
//
// One iteration (a, b, c the coefficients):
//   GRAM  acc = X X^T;  epilogue: A = sigma^2 acc,
//         AR = bf16(A), acc <- (b/c) A
//   POLY  acc += A A;   epilogue: B' = c acc / a, AR = bf16(B')
//   APPLY X += B' X;    epilogue: XR, XC = bf16(X) unless last
// so X_{k+1} = a X_k + (b A + c A^2) X_k.  TMEM holds X up to a scalar
// sigma (the iterate is sigma X): sigma starts at 1/(||X0|| + eps), the
// Gram's epilogue scales A by sigma^2, and the factor a goes into sigma
// instead of into a pass over X (sigma <- a sigma).  Should a sigma leave
// [2^-32, 2^32] (or a = 0), that iteration folds it into X instead:
// X <- (sigma a) X, B' = sigma B, sigma = 1.  The write-out scales O by sigma.
// The step reads G, M and W and writes M, W and the bf16 copy: 22 bytes per
// element.
//
// Every wait is bounded; after a timeout the CTA raises
// MUONH_STATUS_KERNEL_TIMEOUT and runs on through the same barrier sequence
// (with invalid results) so that the peer CTA is never left waiting, and
// before TMEM is freed the issuer waits (bounded) for its last MMAs.

#include "common.cuh"
#include "ns_gemm.h"
#include "tc_ptx.cuh"

namespace muonh {
namespace small {

using namespace ptx;

constexpr int S = 256;                       // padded side of X
constexpr int THREADS = 256;                 // 8 warps
constexpr int OP_BYTES = 128 * S * 2;        // 64 KB per operand buffer
constexpr int SMEM_BYTES = 3 * OP_BYTES + 1024 /*alignment*/ + 256 /*barrier, reduction slots*/;
constexpr int TMEM_COLS = 512;
constexpr int kMaxPerLaunch = 660;

struct SmallDesc {
    float* w;
    uint16_t* wb;
    const float* g;
    float* m;
    int rows, cols;
    int r0_index;
    int pad_;
};
static_assert(sizeof(SmallDesc) == 48, "SmallDesc layout");

struct SmallBatch {
    int n;
    int pad_[3];
    SmallDesc d[kMaxPerLaunch];
};
static_assert(sizeof(SmallBatch) <= 31744, "small-matrix batch exceeds kernel parameter space");

struct SmallParams {
    float lr, beta, eps, wdecay;   // wdecay: plain Muon's 1 - lr*weight_decay
    float ca, cb, cc;
    int ns_steps;
    int muon;                      // 1: plain Muon update, 0: MuonH (hyperball)
    int nesterov;
    int scale_mode;                // UpdateScale
    int grad_bf16;                 // gradients are bf16 bit patterns
    const float* r0;
    uint32_t* status;
};

// Byte offset of element (row, k) in a K-major 128-row operand: four 16 KB
// chunks of 64 K-elements; 8-row groups of 1024 B; 16-byte granules
// XOR-swizzled by row % 8.  k is a multiple of 8 here (one granule).
__device__ __forceinline__ uint32_t kmajor_off(int row, int k) {
    return (uint32_t)((k >> 6) * 16384 + (row >> 3) * 1024 + (row & 7) * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4));
}

// Byte offset of element (k, n) in an MN-major operand of 256 K-rows x 128
// columns: four 16 KB blocks of 64 K-rows, each two 8 KB chunks of 64
// columns; K-rows 128 B apart, granules XOR-swizzled by k % 8.  n is a
// multiple of 8 (one granule).
__device__ __forceinline__ uint32_t mnmajor_off(int k, int n) {
    return (uint32_t)((k >> 6) * 16384 + (n >> 6) * 8192 + ((k & 63) >> 3) * 1024 + (k & 7) * 128 +
                      ((((n & 63) >> 3) ^ (k & 7)) << 4));
}

__device__ __forceinline__ uint4 pack8(const float* v) {
    uint4 u;
    __nv_bfloat162 t;
    t = __floats2bfloat162_rn(v[0], v[1]); u.x = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(v[2], v[3]); u.y = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(v[4], v[5]); u.z = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(v[6], v[7]); u.w = *reinterpret_cast<uint32_t*>(&t);
    return u;
}

// This thread's 32 values of row `row` (local, 0..127), columns j0..j0+31,
// as bf16 into a K-major operand at shared address `base`.
__device__ __forceinline__ void put_kmajor(uint32_t base, int row, int j0, const float (&v)[32]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint4 p = pack8(v + 8 * u);
        const uint32_t a = base + kmajor_off(row, j0 + 8 * u);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(p.x), "r"(p.y), "r"(p.z), "r"(p.w)
                     : "memory");
    }
}

// The same values as row `k` (global X row, 0..255) of the MN-major column
// operand of the CTA that owns columns j0..j0+31 (shared::cluster base
// addresses of both CTAs' XC buffers in xc[]).
__device__ __forceinline__ void put_mnmajor(const uint32_t (&xc)[2], int k, int j0, const float (&v)[32]) {
    const uint32_t base = xc[j0 >> 7];
    const int n0 = j0 & 127;
#pragma unroll
    for (int u = 0; u < 4; ++u) st_cluster_v4(base + mnmajor_off(k, n0 + 8 * u), pack8(v + 8 * u));
}

// Cluster barrier without release semantics: prior memory accesses of this
// thread are not ordered before it (its global stores need not be performed).
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;\n\tbarrier.cluster.wait;" ::: "memory");
}

// Sum of one double per thread over both CTAs of the pair, the same value
// in every thread of both (fixed order: warps, then CTA 0 + CTA 1).
__device__ __forceinline__ double pair_sum(double v, double* red, double* peer, uint32_t peer_remote, int rank) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_sum(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int k = 0; k < THREADS / 32; ++k) t += red[k];
        peer[rank] = t;
        st_cluster_f64(peer_remote + 8 * rank, t);
    }
    cluster_sync();
    return peer[0] + peer[1];
}

// Element (i, j) of X (wide orientation) in the caller's row-major buffer.
__device__ __forceinline__ size_t widx(bool tall, int C, int i, int j) {
    return tall ? (size_t)j * C + i : (size_t)i * C + j;
}

// 32 values of W (X orientation: row i, columns j0..j0+31; zero outside the
// matrix), all loads issued before any use.
__device__ __forceinline__ void load_w(const SmallDesc& D, bool tall, int C, int i, int j0, bool row_ok, int l,
                                       float (&wv)[32]) {
    if (!tall && row_ok && j0 + 32 <= l && (C & 3) == 0) {
        const float4* q = reinterpret_cast<const float4*>(D.w + (size_t)i * C + j0);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 w = q[c];
            wv[4 * c] = w.x; wv[4 * c + 1] = w.y; wv[4 * c + 2] = w.z; wv[4 * c + 3] = w.w;
        }
        return;
    }
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        const bool ok = row_ok && j0 + t < l;
        wv[t] = ok ? D.w[widx(tall, C, i, ok ? j0 + t : 0)] : 0.f;
    }
}

// The new weight's 32 values (and their bf16 copy) back to the caller.
__device__ __forceinline__ void store_w(const SmallDesc& D, bool tall, int C, int i, int j0, bool row_ok, int l,
                                        const float (&y)[32]) {
    if (!tall && row_ok && j0 + 32 <= l && (C & 3) == 0) {
        float4* q = reinterpret_cast<float4*>(D.w + (size_t)i * C + j0);
#pragma unroll
        for (int c = 0; c < 8; ++c) q[c] = make_float4(y[4 * c], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3]);
        if (D.wb) {
            if ((C & 7) == 0) {
                // 16-byte stores: the row start i*C*2 bytes is a multiple of 16
                uint4* b = reinterpret_cast<uint4*>(D.wb + (size_t)i * C + j0);
#pragma unroll
                for (int u = 0; u < 4; ++u) b[u] = pack8(y + 8 * u);
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) D.wb[(size_t)i * C + j0 + t] = bf16_bits(y[t]);
            }
        }
        return;
    }
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        if (row_ok && j0 + t < l) {
            const size_t e = widx(tall, C, i, j0 + t);
            D.w[e] = y[t];
            if (D.wb) D.wb[e] = bf16_bits(y[t]);
        }
    }
}

// ---- coalesced HBM phases ---------------------------------------------------------
// The momentum and write-out phases move the matrix between HBM and the
// lane-per-row layout of TMEM through a per-warp 32 x 32 fp32 staging tile
// (in the A buffer, free in those phases), XOR-swizzled in 16-byte chunks
// (chunk c of row r at c ^ (r & 7)).  In global memory lane l then covers
// columns 4*(l%8)..+3 of rows 4*kk + l/8 (kk = 0..7): every warp access is
// four whole 128-byte row segments.
__device__ __forceinline__ float* stage_at(float* st, int r, int c) { return st + r * 32 + ((c ^ (r & 7)) << 2); }

// coalesced row / column of pass kk of this lane within the warp's block
__device__ __forceinline__ int co_row(int lane, int kk) { return 4 * kk + (lane >> 3); }
__device__ __forceinline__ int co_col(int lane) { return 4 * (lane & 7); }

// the lane-per-row view (lane = row) of the staged tile: 32 values
__device__ __forceinline__ void staged_row(const float* st, int lane, float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 q = *reinterpret_cast<const float4*>(stage_at(const_cast<float*>(st), lane, c));
        v[4 * c] = q.x; v[4 * c + 1] = q.y; v[4 * c + 2] = q.z; v[4 * c + 3] = q.w;
    }
}
__device__ __forceinline__ void stage_row(float* st, int lane, const float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(stage_at(st, lane, c)) = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// 8 coalesced float4 of a row-major fp32 (or bf16, widened) matrix: rows
// row0 + co_row, columns col0 + co_col; zero for rows >= nrows
__device__ __forceinline__ void load_co(const float* base, bool bf16, int C, int row0, int nrows, int col0, int lane,
                                        float4 (&o)[8], bool streaming) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int row = row0 + co_row(lane, kk);
        const size_t e = (size_t)row * C + col0 + co_col(lane);
        if (row >= nrows) {
            o[kk] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else if (bf16) {
            const uint2 u = __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(base) + e));
            o[kk] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                                __uint_as_float(u.y & 0xFFFF0000u));
        } else {
            o[kk] = streaming ? __ldcs(reinterpret_cast<const float4*>(base + e))
                              : *reinterpret_cast<const float4*>(base + e);
        }
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
small_step_kernel(const __grid_constant__ SmallBatch b, const __grid_constant__ SmallParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t xr = smem_u32(smem), xcl = smem_u32(smem + OP_BYTES), ar = smem_u32(smem + 2 * OP_BYTES);
    // staging tiles of the coalesced HBM phases (in the A buffer, free then)
    // and the write-out's U buffer (X's two buffers, 128 rows x 256 fp32)
    float* const stage_base = reinterpret_cast<float*>(smem + 2 * OP_BYTES);
    float* const ubuf = reinterpret_cast<float*>(smem);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 3 * OP_BYTES);
    double* red = reinterpret_cast<double*>(smem + 3 * OP_BYTES + 8);        // [8]
    double* peer = red + 8;                                                  // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(peer + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t drain_bar = smem_u32(tmem_slot + 2);                     // 8-byte aligned

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, h = warp >> 2;
    const uint32_t rank = cluster_rank();
    const uint32_t mbar = smem_u32(bar);

    if (threadIdx.x == 0) {
        mbar_init(mbar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t tx = lane_base, tacc = lane_base + 256;            // this warp's TMEM rows
    const uint32_t xc[2] = {map_to_rank(xcl, 0), map_to_rank(xcl, 1)};
    const uint32_t peer_remote = map_to_rank(smem_u32(peer), rank ^ 1u);
    const bool issuer = rank == 0 && threadIdx.x == 0;
    const uint32_t id_kk = idesc_f16(256, 256, false, false), id_kn = idesc_f16(256, 256, false, true);
    uint32_t phase = 0;
    const int row_l = 32 * q + lane;                 // local row (TMEM lane)
    const int i = 128 * (int)rank + row_l;           // global X row
    const float pre = p.cc != 0.f ? p.cb / p.cc : p.cb;

    // all threads of both CTAs: the MMA is issued, then everyone waits for it
    auto mma_gram = [&](uint32_t a_base, uint32_t d) {
        if (issuer) {
            tc_fence_after();
            for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t da = sdesc(a_base + kb * 16384 + kk * 32, 16, 1024);
                    mma_bf16_pair(d, da, da, id_kk, (kb | kk) ? 1u : 0u);
                }
            mma_commit_pair(mbar);
        }
    };
    auto mma_acc = [&](uint32_t a_base, uint32_t b_base, bool b_mn, uint32_t d) {
        if (issuer) {
            tc_fence_after();
            for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t da = sdesc(a_base + kb * 16384 + kk * 32, 16, 1024);
                    const uint64_t db = b_mn ? sdesc(b_base + kb * 16384 + kk * 2048, 8192, 1024)
                                             : sdesc(b_base + kb * 16384 + kk * 32, 16, 1024);
                    mma_bf16_pair(d, da, db, b_mn ? id_kn : id_kk, 1u);
                }
            mma_commit_pair(mbar);
        }
    };
    auto wait_mma = [&]() {
        if (!mbar_wait(mbar, phase, abort_flag, p.status)) { /* timed out: run on, results invalid */ }
        phase ^= 1;
        tc_fence_after();
    };
    // TMEM and shared-memory writes of this thread made visible to the next MMA
    auto publish = [&]() {
        tmem_st_wait();
        fence_proxy_async();
        tc_fence_before();
        cluster_sync();
    };

    for (int mi = (int)cluster_id(); mi < b.n; mi += (int)cluster_count()) {
        const SmallDesc& D = b.d[mi];
        const int R = D.rows, C = D.cols;
        const bool tall = R > C;
        const int s = tall ? C : R, l = tall ? R : C;
        const bool row_ok = i < s;
        const bool vec = !tall && (C & 3) == 0;

        // ---- momentum; the Newton-Schulz input into TMEM (fp32) and XR / XC (bf16) ----
        // Wide matrices with whole 32-column slices stream G and M coalesced
        // through the staging tile, the next slice's loads in flight while
        // the current one is processed; other shapes take element loads.
        double part = 0.0;
        float* st = stage_base + warp * (32 * 32);
        const int wrow0 = 128 * (int)rank + 32 * q;   // this warp's first X row
        const bool coal = !tall && C == 256;   // whole rows of 256 columns: every slice in range
        if (coal) {
            float4 gc[8], mc[8], gn[8], mn[8];
            load_co(D.g, p.grad_bf16, C, wrow0, s, 128 * h, lane, gc, true);
            load_co(D.m, false, C, wrow0, s, 128 * h, lane, mc, false);
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
                const int j0 = 128 * h + 32 * k;
                if (k + 1 < 4) {
                    load_co(D.g, p.grad_bf16, C, wrow0, s, j0 + 32, lane, gn, true);
                    load_co(D.m, false, C, wrow0, s, j0 + 32, lane, mn, false);
                }
                float acc = 0.f;
                __syncwarp();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int r = co_row(lane, kk);
                    float4 m = mc[kk];
                    const float4 g = gc[kk];
                    m.x = fmaf(p.beta, m.x, g.x); m.y = fmaf(p.beta, m.y, g.y);
                    m.z = fmaf(p.beta, m.z, g.z); m.w = fmaf(p.beta, m.w, g.w);
                    if (wrow0 + r < s)
                        *reinterpret_cast<float4*>(D.m + (size_t)(wrow0 + r) * C + j0 + co_col(lane)) = m;
                    float4 x = m;
                    if (p.nesterov) {
                        x.x = fmaf(p.beta, m.x, g.x); x.y = fmaf(p.beta, m.y, g.y);
                        x.z = fmaf(p.beta, m.z, g.z); x.w = fmaf(p.beta, m.w, g.w);
                    }
                    acc = fmaf(x.x, x.x, acc); acc = fmaf(x.y, x.y, acc);
                    acc = fmaf(x.z, x.z, acc); acc = fmaf(x.w, x.w, acc);
                    *reinterpret_cast<float4*>(stage_at(st, r, lane & 7)) = x;
                }
                __syncwarp();
                part += (double)acc;
                float x[32];
                staged_row(st, lane, x);
                tmem_st32(tx + j0, x);
                put_kmajor(xr, row_l, j0, x);
                put_mnmajor(xc, i, j0, x);
                if (k + 1 < 4) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) { gc[kk] = gn[kk]; mc[kk] = mn[kk]; }
                }
            }
        } else {
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
            const int j0 = 128 * h + 32 * k;
            // all loads of the slice first, then the stores: stores to M
            // would otherwise order (and serialise) the loads behind them
            float x[32], gv[32];
            float acc = 0.f;
            if (vec && row_ok && j0 + 32 <= l) {
                const size_t base = (size_t)i * C + j0;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float4 g;
                    if (p.grad_bf16) {
                        const uint2 u =
                            __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(D.g) + base) + c);
                        g = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                        __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
                    } else {
                        g = __ldcs(reinterpret_cast<const float4*>(D.g + base) + c);
                    }
                    const float4 mv = *reinterpret_cast<const float4*>(D.m + base + 4 * c);
                    gv[4 * c] = g.x; gv[4 * c + 1] = g.y; gv[4 * c + 2] = g.z; gv[4 * c + 3] = g.w;
                    x[4 * c] = mv.x; x[4 * c + 1] = mv.y; x[4 * c + 2] = mv.z; x[4 * c + 3] = mv.w;
                }
#pragma unroll
                for (int t = 0; t < 32; ++t) x[t] = fmaf(p.beta, x[t], gv[t]);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<float4*>(D.m + base + 4 * c) =
                        make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int j = j0 + t;
                    const bool ok = row_ok && j < l;
                    const size_t e = widx(tall, C, i, ok ? j : 0);
                    gv[t] = !ok ? 0.f
                                : p.grad_bf16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(D.g)[e] << 16)
                                              : __ldcs(D.g + e);
                    x[t] = ok ? D.m[e] : 0.f;
                }
#pragma unroll
                for (int t = 0; t < 32; ++t) x[t] = fmaf(p.beta, x[t], gv[t]);
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int j = j0 + t;
                    if (row_ok && j < l) D.m[widx(tall, C, i, j)] = x[t];
                }
            }
            if (p.nesterov) {
#pragma unroll
                for (int t = 0; t < 32; ++t) x[t] = fmaf(p.beta, x[t], gv[t]);
            }
#pragma unroll
            for (int t = 0; t < 32; ++t) acc = fmaf(x[t], x[t], acc);
            part += (double)acc;
            tmem_st32(tx + j0, x);
            put_kmajor(xr, row_l, j0, x);
            put_mnmajor(xc, i, j0, x);
        }
        }
        // ||M||^2 over the pair (the order of pair_sum: warps, then CTA 0 +
        // CTA 1), exchanged in the cluster barrier that publishes X
        {
            const double v = warp_sum(part);
            if (lane == 0) red[warp] = v;
        }
        tmem_st_wait();
        fence_proxy_async();
        __syncthreads();
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int k = 0; k < THREADS / 32; ++k) t += red[k];
            peer[rank] = t;
            st_cluster_f64(peer_remote + 8 * rank, t);
        }
        tc_fence_before();
        cluster_sync();
        const double nu2 = peer[0] + peer[1];
        const bool finite = isfinite(nu2);
        const float inv = finite ? (float)(1.0 / (sqrt(nu2) + (double)p.eps)) : 0.f;
        if (!finite && threadIdx.x == 0 && rank == 0) raise_status(p.status, MUONH_STATUS_NONFINITE_INPUT);

        // ---- Newton-Schulz iterations ----
        float sigma = inv;   // the iterate is sigma times the X held in TMEM
        for (int it = 0; it < p.ns_steps; ++it) {
            const bool last = it + 1 == p.ns_steps;
            if (it == (p.ns_steps > 2 ? p.ns_steps - 2 : 0) && threadIdx.x == 0) {
                // While the last two iterations run on chip, pull into L2 this
                // matrix's weight (read by the write-out) and the gradient and
                // momentum of this cluster's next matrix (read by its load
                // phase), so those phases read L2 instead of HBM (two
                // iterations ahead measured faster than one: 0.915 against
                // 0.920 ms for 1024 matrices of 256 x 256).
                if (rank == 1) {
                    prefetch_l2(D.w, (size_t)R * C * 4);
                } else if (mi + (int)cluster_count() < b.n) {
                    const SmallDesc& Dn = b.d[mi + (int)cluster_count()];
                    const size_t el = (size_t)Dn.rows * Dn.cols;
                    prefetch_l2(Dn.g, el * (p.grad_bf16 ? 2 : 4));
                    prefetch_l2(Dn.m, el * 4);
                }
            }
            mma_gram(xr, tmem + 256);
            wait_mma();
            const float sa = sigma * sigma;
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
                const int j0 = 128 * h + 32 * k;
                float v[32];
                tmem_ld32(tacc + j0, v);
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] *= sa;
                put_kmajor(ar, row_l, j0, v);
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] *= pre;
                tmem_st32(tacc + j0, v);
            }
            publish();
            if (p.cc != 0.f) {
                mma_acc(ar, ar, false, tmem + 256);   // acc += A A, onto the (b/c) A preload
                wait_mma();
            }
            // the a X term: a goes into sigma while sigma a stays in range;
            // otherwise X <- (sigma a) X here, B' = sigma B and sigma = 1
            const float sig_a = sigma * p.ca;
            const bool defer = p.ca != 0.f && fabsf(sig_a) <= 0x1p32f && fabsf(sig_a) >= 0x1p-32f;
            const float pb = (p.cc != 0.f ? p.cc : 1.f) * (defer ? 1.f / p.ca : sigma);
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
                const int j0 = 128 * h + 32 * k;
                float v[32];
                tmem_ld32(tacc + j0, v);
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] *= pb;
                put_kmajor(ar, row_l, j0, v);
                if (!defer) {
                    tmem_ld32(tx + j0, v);
#pragma unroll
                    for (int t = 0; t < 32; ++t) v[t] *= sig_a;
                    tmem_st32(tx + j0, v);
                }
            }
            sigma = defer ? sig_a : 1.f;
            publish();
            mma_acc(ar, xcl, true, tmem);   // X += B X
            wait_mma();
            if (!last) {
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    const int j0 = 128 * h + 32 * k;
                    float v[32];
                    tmem_ld32(tx + j0, v);
                    put_kmajor(xr, row_l, j0, v);
                    put_mnmajor(xc, i, j0, v);
                }
                publish();
            }
        }

        // ---- write-out: MuonH retraction or plain Muon update ----
        // Whole 256-column rows go coalesced: O through the staging tile, W
        // loaded one slice ahead, U kept in the U buffer (shared memory) for
        // the rescale.  Other shapes: element access, U in the accumulator.
        const float nlr = -p.lr * update_scale(R, C, p.scale_mode) * sigma;   // O = sigma X
        const bool keep = !finite || *abort_flag;
        auto o_coalesced = [&](int j0, float4 (&o4)[8]) {
            float o[32];
            tmem_ld32(tx + j0, o);
            __syncwarp();
            stage_row(st, lane, o);
            __syncwarp();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) o4[kk] = *reinterpret_cast<const float4*>(stage_at(st, co_row(lane, kk), lane & 7));
        };
        auto store_w_co = [&](int j0, int kk, float4 w) {
            const int row = wrow0 + co_row(lane, kk);
            if (row >= s) return;
            const size_t e = (size_t)row * C + j0 + co_col(lane);
            __stcs(reinterpret_cast<float4*>(D.w + e), w);
            if (D.wb) {
                const __nv_bfloat162 a = __floats2bfloat162_rn(w.x, w.y), b2 = __floats2bfloat162_rn(w.z, w.w);
                *reinterpret_cast<uint2*>(D.wb + e) =
                    make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b2));
            }
        };
        if (p.muon) {
            if (!keep && coal) {
                float4 wc[8], wn[8];
                load_co(D.w, false, C, wrow0, s, 128 * h, lane, wc, true);
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    const int j0 = 128 * h + 32 * k;
                    if (k + 1 < 4) load_co(D.w, false, C, wrow0, s, j0 + 32, lane, wn, true);
                    float4 o4[8];
                    o_coalesced(j0, o4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const float4 w = wc[kk], o = o4[kk];
                        store_w_co(j0, kk, make_float4(fmaf(nlr, o.x, p.wdecay * w.x), fmaf(nlr, o.y, p.wdecay * w.y),
                                                       fmaf(nlr, o.z, p.wdecay * w.z), fmaf(nlr, o.w, p.wdecay * w.w)));
                    }
                    if (k + 1 < 4) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) wc[kk] = wn[kk];
                    }
                }
            } else if (!keep) {
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    const int j0 = 128 * h + 32 * k;
                    float o[32], wv[32];
                    tmem_ld32(tx + j0, o);
                    load_w(D, tall, C, i, j0, row_ok, l, wv);
#pragma unroll
                    for (int t = 0; t < 32; ++t) wv[t] = fmaf(nlr, o[t], p.wdecay * wv[t]);
                    store_w(D, tall, C, i, j0, row_ok, l, wv);
                }
            }
            cluster_sync_relaxed();   // the stores of W need not be performed first
        } else {
            double up = 0.0;
            if (coal) {
                float4 wc[8], wn[8];
                load_co(D.w, false, C, wrow0, s, 128 * h, lane, wc, true);
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    const int j0 = 128 * h + 32 * k;
                    if (k + 1 < 4) load_co(D.w, false, C, wrow0, s, j0 + 32, lane, wn, true);
                    float4 o4[8];
                    o_coalesced(j0, o4);
                    float acc = 0.f;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const float4 w = wc[kk], o = o4[kk];
                        const float4 u = make_float4(fmaf(nlr, o.x, w.x), fmaf(nlr, o.y, w.y), fmaf(nlr, o.z, w.z),
                                                     fmaf(nlr, o.w, w.w));
                        const int r = co_row(lane, kk);
                        if (wrow0 + r < s) {
                            acc = fmaf(u.x, u.x, acc); acc = fmaf(u.y, u.y, acc);
                            acc = fmaf(u.z, u.z, acc); acc = fmaf(u.w, u.w, acc);
                        }
                        *reinterpret_cast<float4*>(ubuf + (32 * q + r) * 256 + j0 + co_col(lane)) = u;
                    }
                    up += (double)acc;
                    if (k + 1 < 4) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) wc[kk] = wn[kk];
                    }
                }
            } else {
                // U = W - lr*O goes to the accumulator columns (free now), so W
                // is read once
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    const int j0 = 128 * h + 32 * k;
                    float o[32], wv[32];
                    tmem_ld32(tx + j0, o);
                    load_w(D, tall, C, i, j0, row_ok, l, wv);
                    float acc = 0.f;
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        wv[t] = fmaf(nlr, o[t], wv[t]);
                        if (row_ok && j0 + t < l) acc = fmaf(wv[t], wv[t], acc);
                    }
                    up += (double)acc;
                    tmem_st32(tacc + j0, wv);
                }
                tmem_st_wait();
            }
            const double rho2 = pair_sum(up, red, peer, peer_remote, (int)rank);
            const bool degenerate = !isfinite(rho2) || rho2 == 0.0;
            if (!keep && degenerate && threadIdx.x == 0 && rank == 0)
                raise_status(p.status, MUONH_STATUS_DEGENERATE_NORM);
            if (!keep && !degenerate) {
                const float f = (float)((double)p.r0[D.r0_index] / sqrt(rho2));
                if (coal) {
#pragma unroll 1
                    for (int k = 0; k < 4; ++k) {
                        const int j0 = 128 * h + 32 * k;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const float4 u =
                                *reinterpret_cast<const float4*>(ubuf + (32 * q + co_row(lane, kk)) * 256 + j0 + co_col(lane));
                            store_w_co(j0, kk, make_float4(f * u.x, f * u.y, f * u.z, f * u.w));
                        }
                    }
                } else {
#pragma unroll 1
                    for (int k = 0; k < 4; ++k) {
                        const int j0 = 128 * h + 32 * k;
                        float u[32];
                        tmem_ld32(tacc + j0, u);
#pragma unroll
                        for (int t = 0; t < 32; ++t) u[t] = f * u[t];
                        store_w(D, tall, C, i, j0, row_ok, l, u);
                    }
                }
            }
            // the reduction slots, the accumulator and the U buffer are free
            // again (every read of them has returned: its value was stored);
            // the stores of W need not be performed first
            tc_fence_before();
            cluster_sync_relaxed();
            tc_fence_after();
        }
    }

    // after a wait gave up, MMAs may still be running: every MMA the issuer
    // started has completed before either CTA frees TMEM or exits
    if (issuer) {
        mma_commit_pair(drain_bar, 1);
        mbar_drain_wait(drain_bar, 0, p.status, kTimeoutNs);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace small
}  // namespace muonh

// ---- host side -------------------------------------------------------------------
namespace muonh {


namespace small {

static int max_clusters() {
    static int cached = 0;
    if (cached) return cached;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 148, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, small_step_kernel, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        n = sms > 1 ? sms / 2 : 1;
    }
    cached = n;
    return n;
}

}  // namespace small

// Launches small_step_kernel over matrices mats[idx[k]] (host array; every
// listed matrix has both sides <= 256), kMaxPerLaunch per launch.  `launches`
// counts the kernels launched.
cudaError_t launch_small_step(const muonh_matrix_t* mats, const int* idx, int n, const SmallStepArgs& a,
                              cudaStream_t st, int* launches) {
    using namespace small;
    *launches = 0;
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(small_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    SmallParams p{};
    p.lr = a.lr;
    p.beta = a.beta;
    p.eps = a.eps;
    p.wdecay = a.wdecay;
    p.ca = a.coeffs[0];
    p.cb = a.coeffs[1];
    p.cc = a.coeffs[2];
    p.ns_steps = a.ns_steps;
    p.muon = a.muon ? 1 : 0;
    p.nesterov = a.nesterov ? 1 : 0;
    p.scale_mode = a.scale_mode;
    p.grad_bf16 = a.grad_bf16 ? 1 : 0;
    p.r0 = a.r0;
    p.status = a.status;
    for (int b0 = 0; b0 < n; b0 += kMaxPerLaunch) {
        SmallBatch B;
        B.n = n - b0 < kMaxPerLaunch ? n - b0 : kMaxPerLaunch;
        B.pad_[0] = B.pad_[1] = B.pad_[2] = 0;
        for (int k = 0; k < B.n; ++k) {
            const muonh_matrix_t& m = mats[idx[b0 + k]];
            SmallDesc& D = B.d[k];
            D.w = m.w;
            D.wb = m.w_bf16;
            D.g = m.grad;
            D.m = m.mom;
            D.rows = (int)m.rows;
            D.cols = (int)m.cols;
            D.r0_index = idx[b0 + k];
            D.pad_ = 0;
        }
        const int clusters = B.n < max_clusters() ? B.n : max_clusters();
        small_step_kernel<<<2 * clusters, THREADS, SMEM_BYTES, st>>>(B, p);
        ++*launches;
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace muonh
