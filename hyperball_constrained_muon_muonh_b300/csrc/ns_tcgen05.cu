// Newton-Schulz GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged by TMA.  One iteration of the orthogonalisation (Puro-2B
// digest, section "The load-bearing tricks aren't in the abstract": Muon's
// Newton-Schulz iterations) on a bucket of G same-shape matrices X, each kept
// in its own orientation R x C (s = min(R, C), l = max(R, C)):
//
//   GRAM   A = X X^T (wide) or X^T X (tall)   (s x s, K = l)  symmetric: upper
//                                               tiles only; epilogue writes A
//                                               fp32, A bf16 and their mirrors
//   POLY   B = b*A + c*A A     (s x s, K = s)  symmetric (A A = A A^T):
//                                               upper tiles, B bf16 + mirror
//   APPLY  X <- a*X + B X (wide) or a*X + X B (tall)   (R x C, K = s): X fp32
//          state read/written in the epilogue, bf16 operand copy out
//
// A tall matrix is never transposed: its Gram reads both operands MN-major
// (the instruction descriptor's transpose bits), and its apply multiplies by
// B on the right, which reads both operands K-major.
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer (one thread) and TMEM allocator
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f16, bf16 in,
//               fp32 accumulate in TMEM, 128 x 256 tile, K step 16
//   warps 2..9  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)..+31), fused arithmetic, global stores
// Shared memory: 4-stage ring of (A 128x64, B 256x64) bf16 tiles, 128-byte
// swizzle.  TMEM: two 256-column fp32 accumulators so the epilogue of one
// tile overlaps the main loop of the next.  Every mbarrier wait gives up
// after a time limit, sets MUONH_STATUS_KERNEL_TIMEOUT and unwinds: copies
// and MMAs already issued are waited for (bounded) before the CTA frees its
// TMEM and exits (ExitState).

#include <cuda.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "ns_gemm.h"
#include "tc_ptx.cuh"

namespace muonh {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int TMEM_COLS = 2 * BN;               // 512
constexpr int EPI_WARPS = 8;                    // two per TMEM lane quarter
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int ST_FLOATS = 32 * 32;              // 4 KB staging tile per epilogue warp
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ +
                           EPI_WARPS * ST_FLOATS * 4;
using namespace ptx;

// Per-kk increment of an operand descriptor (start address field, 16-byte
// units): 32 B along K for K-major tiles, 16 K-rows = 2048 B for MN-major.
__device__ __forceinline__ uint64_t operand_desc_step(bool mn_major) { return mn_major ? (2048 >> 4) : (32 >> 4); }

// Descriptor of the kk-th K=16 slice of a staged operand tile.  K-major: rows
// of 64 K-elements (128 B, swizzled), 8-row groups 1024 B apart.  MN-major:
// 64-element MN chunks of 64 K-rows each (8 KB apart), K rows 128 B apart.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk, bool mn_major) {
    return mn_major ? sdesc(base + kk * 2048, 64 * BK * 2, 1024) : sdesc(base + kk * 32, 16, 1024);
}

// Bookkeeping for leaving the kernel after a wait gave up, kept after the
// pipeline barriers.  Copies and MMAs already issued must finish before the
// CTA gives up the shared memory they write or read and the TMEM they
// write: the producer counts the stage fills it issued (and the bytes of
// each stage's last fill), the MMA issuer the fills it consumed, and on the
// way out the fills issued but never consumed are waited for.
struct ExitState {
    uint64_t drain_bar;      // one MMA commit after the issuer's last MMA
    uint32_t tmem_slot;
    int abort_flag;
    int fills;               // stage fills this CTA's producer issued
    int consumed;            // stage fills the MMA issuer waited for
    uint32_t fill_bytes[8];  // per stage, its last fill: bytes this CTA loaded (the pair
                             // kernel's leader: the bytes it expected from both CTAs)
};
static_assert(sizeof(ExitState) == 56, "ExitState layout");

__device__ __forceinline__ unsigned long long wait_limit(const GemmParams& p) {
    return p.timeout_ns ? p.timeout_ns : kTimeoutNs;
}

__host__ __device__ constexpr uint32_t idesc_bf16(bool a_mn_major, bool b_mn_major) {
    return idesc_f16(BM, BN, a_mn_major, b_mn_major);
}

// ---- tile scheduling ---------------------------------------------------------
// Symmetric modes keep tile (mi, nj) iff it holds an element with col >= row:
// (nj+1)*BN > mi*BM, i.e. nj >= mi/2 (BN = 2*BM).
__device__ __forceinline__ void tile_coords(const GemmParams& p, int local, int& mi, int& nj) {
    if (p.mode == NS_APPLY) {
        // the panel of the large operand X_op outermost, so consecutive CTAs
        // share it: its column panel (wide, B operand) or row panel (tall, A)
        if (p.m_outer) {
            mi = local / p.tiles_n;
            nj = local - mi * p.tiles_n;
        } else {
            nj = local / p.tiles_m;
            mi = local - nj * p.tiles_m;
        }
        return;
    }
    int m = 0;
    for (;;) {
        const int cnt = p.tiles_n - (m >> 1);
        if (local < cnt) break;
        local -= cnt;
        ++m;
    }
    mi = m;
    nj = (m >> 1) + local;
}

// ---- epilogues, staged (one-K-step pipelines) -------------------------------------
// tcgen05.ld gives each lane one accumulator row (32 consecutive columns).
// Row-wise global access from that layout touches 32 rows per instruction,
// so each warp stages its 32 x 32 slice in shared memory and reads it back
// so that each lane holds 8 consecutive columns of one row: lane l takes
// columns 8*(l%4) .. +7 of rows 8k + l/4, k = 0..3.  Every global access is
// then one 16-byte vector per lane (8 bf16 values, or half of 8 fp32 values),
// which keeps the epilogue's memory instructions, not only its bytes, few.
// The staging tile is XOR-swizzled in 16-byte chunks (chunk c of row r sits
// at c ^ (r & 7)), which keeps the row-per-lane writes and the reads free of
// bank conflicts.  The mirror of a symmetric product is read back from the
// staged slice by columns (8 consecutive rows of one column per lane, one
// 16-byte store) where the slice lies wholly above the diagonal, and is
// written element by element elsewhere.  Operands the epilogue reads (X for
// APPLY, A for POLY) are loaded one slice ahead, as raw bits that are turned
// into values only where they are used, so that the loads stay in flight
// while the previous slice is processed.

__device__ __forceinline__ void stage_rows(float* st, int lane, const float (&v)[32]) {
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(st + lane * 32 + ((c ^ (lane & 7)) << 2)) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    __syncwarp();
}

// row r (0..31), chunk c (0..7) of the staged slice
__device__ __forceinline__ float4 staged(const float* st, int r, int c) {
    return *reinterpret_cast<const float4*>(st + r * 32 + ((c ^ (r & 7)) << 2));
}

// This lane's row (0..31) and first column (0..24) of the slice, pass k.
__device__ __forceinline__ int st_row(int lane, int k) { return 8 * k + (lane >> 2); }
__device__ __forceinline__ int st_col(int lane) { return 8 * (lane & 3); }

// 8 values as bf16 (round to nearest even), packed for one 16-byte store
__device__ __forceinline__ uint4 pack_bf16x8(float4 a, float4 b) {
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
    return make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                      *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
}

// two bf16 values of a 32-bit word as floats
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Raw bits of a 16-byte vector kept in a float4 register (a prefetch slot)
__device__ __forceinline__ float4 as_slot(uint4 u) {
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}
__device__ __forceinline__ uint4 slot_bits(float4 f) {
    return make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z), __float_as_uint(f.w));
}

// Prefetch of an fp32 row-major array (row stride `ld`) for pass k = 0..3:
// xp[2k], xp[2k+1] = X[i0 + 8k + lane/4][j0 + 8*(lane%4) .. +7].  A workspace
// array's row stride is a multiple of 8 elements, so the 8-wide access at a
// column < N stays inside the padded row (padding is never read back); a
// caller's buffer (row stride N, N % 4 == 0) is read only up to column N.
__device__ __forceinline__ void prefetch_rm(const float* base, int ld, int M, int N, int i0, int lane, int j0,
                                            float4 (&xp)[8], bool exact_cols = false) {
    const int col = j0 + st_col(lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = i0 + st_row(lane, k);
        const float4* q = reinterpret_cast<const float4*>(base + (size_t)row * ld + col);
        const bool ok = row < M && col < N;
        xp[2 * k] = ok ? __ldcs(q) : make_float4(0.f, 0.f, 0.f, 0.f);
        xp[2 * k + 1] = (ok && (!exact_cols || col + 4 < N)) ? __ldcs(q + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// The same for the two-part state X = hi + lo (bf16 each, row stride ld):
// xp[2k] holds hi's 8 values, xp[2k+1] lo's, as raw bits (hilo_values).
__device__ __forceinline__ void prefetch_hilo(const __nv_bfloat16* hi, const __nv_bfloat16* lo, int ld, int M, int N,
                                              int i0, int lane, int j0, float4 (&xp)[8]) {
    const int col = j0 + st_col(lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = i0 + st_row(lane, k);
        uint4 h = make_uint4(0u, 0u, 0u, 0u), l = h;
        if (row < M && col < N) {
            const size_t off = (size_t)row * ld + col;
            // hi is also this launch's operand, which neighbouring tiles still
            // fetch: a plain load, not an evict-first one
            h = *reinterpret_cast<const uint4*>(hi + off);
            l = __ldcs(reinterpret_cast<const uint4*>(lo + off));
        }
        xp[2 * k] = as_slot(h);
        xp[2 * k + 1] = as_slot(l);
    }
}

// L2 prefetch of what prefetch_rm / prefetch_hilo read for the slice at
// column j0: one lane per row (lanes 4r) touches the row's segment of each
// array; nothing is loaded into registers.
__device__ __forceinline__ void l2_prefetch(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void l2_prefetch_hilo(const __nv_bfloat16* hi, const __nv_bfloat16* lo, int ld, int M, int N,
                                                 int i0, int lane, int j0) {
    if ((lane & 3) != 0 || j0 >= N) return;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = i0 + st_row(lane, k);
        if (row < M) {
            const size_t off = (size_t)row * ld + j0;
            l2_prefetch(hi + off);
            l2_prefetch(lo + off);
        }
    }
}
__device__ __forceinline__ void l2_prefetch_rm(const float* base, int ld, int M, int N, int i0, int lane, int j0) {
    if ((lane & 3) != 0 || j0 >= N) return;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = i0 + st_row(lane, k);
        if (row < M) l2_prefetch(base + (size_t)row * ld + j0);
    }
}

// The 8 values hi + lo of pass k of a prefetch_hilo slot pair
__device__ __forceinline__ void hilo_values(float4 hs, float4 ls, float (&x)[8]) {
    const uint4 h = slot_bits(hs), l = slot_bits(ls);
    const uint32_t hw[4] = {h.x, h.y, h.z, h.w}, lw[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        x[2 * w] = bf_lo(hw[w]) + bf_lo(lw[w]);
        x[2 * w + 1] = bf_hi(hw[w]) + bf_hi(lw[w]);
    }
}

// hi = bf16(y) (round to nearest even), lo = bf16(y - hi): y's two-part
// form, exact to about 16 significant bits.
__device__ __forceinline__ void split_hilo8(const float (&y)[8], uint4& hi, uint4& lo) {
    hi = pack_bf16x8(make_float4(y[0], y[1], y[2], y[3]), make_float4(y[4], y[5], y[6], y[7]));
    const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
    float r[8];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        r[2 * w] = y[2 * w] - bf_lo(hw[w]);
        r[2 * w + 1] = y[2 * w + 1] - bf_hi(hw[w]);
    }
    lo = pack_bf16x8(make_float4(r[0], r[1], r[2], r[3]), make_float4(r[4], r[5], r[6], r[7]));
}

// Prefetch for POLY: A[i][j..j+7] for pass k from the bf16 operand copy A_op
// (both triangles written by the Gram; the b*A term uses the same rounded A
// as the A*A product), one 16-byte vector per pass, raw bits in ap[k].
__device__ __forceinline__ void prefetch_a_st(const GemmParams& p, int g, int i0, int lane, int j0, float4 (&ap)[8]) {
    const uint16_t* a = reinterpret_cast<const uint16_t*>(p.a_op) + (size_t)g * p.ld_s * p.M;
    const int col = j0 + st_col(lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = i0 + st_row(lane, k);
        ap[k] = (row < p.M && col < p.N && col + 7 >= row)
                    ? as_slot(*reinterpret_cast<const uint4*>(a + (size_t)row * p.ld_s + col))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// The 8 values of pass k of an fp32 prefetch slot pair
__device__ __forceinline__ void f32_values(float4 a, float4 b, float (&x)[8]) {
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// APPLY slice: X (prefetched by the caller: fp32, or the two-part state when
// in_hilo) and the accumulator give y = sc*(a*x + (B X)).  Output: with
// NS_OUT_U, u = W - lr*y goes to the fp32 state and u^2 is added to hacc for
// the elements inside the matrix; with NS_OUT_W the new weight goes to the
// caller's buffers; otherwise, when another iteration follows (x_op_out
// set), the two-part state hi -> x_op_out (also the next Gram's operand),
// lo -> x_lo; after the last iteration, y -> the fp32 state.
template <int VAR>
__device__ __forceinline__ void apply_slice_st(const GemmParams& p, const NsIO& io, bool keep_w, int g, int i0,
                                               int lane, int j0, const float (&v)[32], float* st,
                                               const float4 (&xp)[8], const float4 (&wp)[8], float sc, float& hacc) {
    stage_rows(st, lane, v);
    const int col = j0 + st_col(lane);
    const size_t moff = (size_t)g * p.ld_x * p.M;
    float* xs = p.x_state + moff;
    __nv_bfloat16* xo = p.x_op_out ? p.x_op_out + moff : nullptr;
    __nv_bfloat16* xlo = p.x_lo + moff;
    const bool hilo_in = !(VAR & NS_IN_SRC) && p.in_hilo;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = st_row(lane, k), row = i0 + r;
        if (row >= p.M || col >= p.N) continue;
        const float4 a0 = staged(st, r, 2 * (lane & 3)), a1 = staged(st, r, 2 * (lane & 3) + 1);
        const float acc[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float x[8];
        if (hilo_in) hilo_values(xp[2 * k], xp[2 * k + 1], x);
        else f32_values(xp[2 * k], xp[2 * k + 1], x);
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = sc * fmaf(p.ca, x[e], acc[e]);
        if (VAR & (NS_OUT_U | NS_OUT_W)) {
            float w[8];
            f32_values(wp[2 * k], wp[2 * k + 1], w);
            const int nv = p.N - col;   // >= 4: caller buffers have N % 4 == 0
            if (VAR & NS_OUT_U) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    y[e] = fmaf(p.nlr, y[e], w[e]);
                    if (e < nv) hacc = fmaf(y[e], y[e], hacc);
                }
            } else {
                // new weight, written to the caller's buffers (row stride N)
                if (!keep_w) {
                    float u[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) u[e] = fmaf(p.nlr, y[e], p.wdecay * w[e]);
                    const size_t woff = (size_t)row * p.N + col;
                    float4* wq = reinterpret_cast<float4*>(io.w + woff);
                    __stcs(wq, make_float4(u[0], u[1], u[2], u[3]));
                    if (nv > 4) __stcs(wq + 1, make_float4(u[4], u[5], u[6], u[7]));
                    if (io.wb) {
                        __nv_bfloat16* wb = reinterpret_cast<__nv_bfloat16*>(io.wb) + woff;
                        const uint4 pk = pack_bf16x8(make_float4(u[0], u[1], u[2], u[3]),
                                                     make_float4(u[4], u[5], u[6], u[7]));
                        if (nv > 4 && (woff & 7) == 0) {
                            *reinterpret_cast<uint4*>(wb) = pk;
                        } else {
                            *reinterpret_cast<uint2*>(wb) = make_uint2(pk.x, pk.y);
                            if (nv > 4) *reinterpret_cast<uint2*>(wb + 4) = make_uint2(pk.z, pk.w);
                        }
                    }
                }
                continue;
            }
        }
        const size_t off = (size_t)row * p.ld_x + col;
        if (!(VAR & NS_OUT_U) && xo) {
            uint4 hi, lo;
            split_hilo8(y, hi, lo);
            *reinterpret_cast<uint4*>(xo + off) = hi;
            // lo is read again only by the next apply's epilogue: streaming
            // store, so it does not push the GEMM operands out of L2
            __stcs(reinterpret_cast<uint4*>(xlo + off), lo);
        } else {
            float4* q = reinterpret_cast<float4*>(xs + off);
            __stcs(q, make_float4(y[0], y[1], y[2], y[3]));
            __stcs(q + 1, make_float4(y[4], y[5], y[6], y[7]));
        }
    }
}

// GRAM / POLY: element (i, j) is written when j >= i, its mirror (j, i) when
// j > i; tiles entirely below the diagonal are never scheduled.  The
// polynomial's b*A term comes from A_op (ap: raw bits, one 16-byte vector per
// pass), so both the element and its mirror get c*(A A) + b*A.
template <int MODE>
__device__ __forceinline__ void sym_slice_st(const GemmParams& p, int g, int i0, int lane, int j0, float (&v)[32],
                                             float* st, const float4 (&ap)[8], float sc) {
    const int M = p.M, N = p.N;
    const size_t mbase = (size_t)g * p.ld_s * M;
    if (MODE == NS_GRAM) {
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] *= sc;
    } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] *= p.cc;
    }
    __nv_bfloat16* ob = p.sym_bf16 + mbase;
    stage_rows(st, lane, v);
    const int col = j0 + st_col(lane);
    // a slice wholly above the diagonal and inside the matrix writes its
    // mirror through the staged slice, 16 bytes per lane; others element by
    // element
    const bool whole = j0 > i0 + 31 && i0 + 32 <= M && j0 + 32 <= N;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = st_row(lane, k), row = i0 + r;
        if (row >= M || col >= N || col + 7 < row) continue;
        const float4 a0 = staged(st, r, 2 * (lane & 3)), a1 = staged(st, r, 2 * (lane & 3) + 1);
        float y[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        if (MODE == NS_POLY) {
            const uint4 aw = slot_bits(ap[k]);
            const uint32_t w4[4] = {aw.x, aw.y, aw.z, aw.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                y[2 * w] = fmaf(p.cb, bf_lo(w4[w]), y[2 * w]);
                y[2 * w + 1] = fmaf(p.cb, bf_hi(w4[w]), y[2 * w + 1]);
            }
            if (whole) {
                // the final values back into the staged slice, for the mirror
                *reinterpret_cast<float4*>(st + r * 32 + (((2 * (lane & 3)) ^ (r & 7)) << 2)) =
                    make_float4(y[0], y[1], y[2], y[3]);
                *reinterpret_cast<float4*>(st + r * 32 + (((2 * (lane & 3) + 1) ^ (r & 7)) << 2)) =
                    make_float4(y[4], y[5], y[6], y[7]);
            }
        }
        const size_t off = (size_t)row * p.ld_s + col;
        if (col >= row && col + 8 <= N) {
            *reinterpret_cast<uint4*>(ob + off) =
                pack_bf16x8(make_float4(y[0], y[1], y[2], y[3]), make_float4(y[4], y[5], y[6], y[7]));
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (col + e >= row && col + e < N) ob[off + e] = __float2bfloat16_rn(y[e]);
        }
        if (!whole) {
            // mirrors (strictly above the diagonal): for each e, the warp's
            // lanes write 8 consecutive elements of 4 transposed rows
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (col + e > row && col + e < N) ob[(size_t)(col + e) * p.ld_s + row] = __float2bfloat16_rn(y[e]);
        }
    }
    if (whole) {
        // pass k: this lane's column c = 8k + lane/4 of the slice and rows
        // 8(lane%4)..+7, which are 8 consecutive elements of row j0 + c of the
        // mirror (i0 is a multiple of 32, ld_s of 8: 16-byte aligned)
        __syncwarp();
        const int r0 = 8 * (lane & 3);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = 8 * k + (lane >> 2);
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = r0 + e;
                y[e] = st[r * 32 + ((((c >> 2) ^ (r & 7))) << 2) + (c & 3)];
            }
            *reinterpret_cast<uint4*>(ob + (size_t)(j0 + c) * p.ld_s + i0 + r0) =
                pack_bf16x8(make_float4(y[0], y[1], y[2], y[3]), make_float4(y[4], y[5], y[6], y[7]));
        }
    }
}

// ---- epilogue, fragment layout (the Gram with two-K-step pipelines) ------------------
// The accumulator is read with tcgen05.ld.16x256b: two loads (TMEM lanes
// +0..15 and +16..31 of this warp's lane quarter) of four 8-column groups
// give each thread, for a 32 x 32 slice at (i0, j0), the values
//   v[8*rr + 2*j + e] = acc[i0 + 8*rr + lane/4][j0 + 8*j + 2*(lane%4) + e]
// for rr, j in 0..3 and e in 0..1: four rows and four column pairs.  Four
// consecutive lanes hold 8 consecutive columns (32 bytes) of one row, so
// every row-wise global access is in whole 32-byte sectors without staging
// the slice in shared memory; for the mirror, eight lanes with the same
// lane%4 hold 8 consecutive rows of one column, which are 8 consecutive
// elements of the transposed row.

__device__ __forceinline__ int quad_row(int lane, int rr) { return 8 * rr + (lane >> 2); }
__device__ __forceinline__ int quad_col(int lane, int j) { return 8 * j + 2 * (lane & 3); }

__device__ __forceinline__ void store_bf16x2(__nv_bfloat16* dst, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(a, b);
}

// GRAM slice: element (i, j) is written when j >= i, its mirror (j, i) when
// j > i; tiles entirely below the diagonal are never scheduled.
__device__ __forceinline__ void gram_slice(const GemmParams& p, int g, int i0, int lane, int j0, const float (&v)[32],
                                           float sc) {
    const int M = p.M, N = p.N;
    const size_t mbase = (size_t)g * p.ld_s * M;
    __nv_bfloat16* ob = p.sym_bf16 + mbase;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int row = i0 + quad_row(lane, rr);
        if (row >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = j0 + quad_col(lane, j);
            if (col >= N || col + 1 < row) continue;
            const int q = 4 * rr + j;
            const float y0 = sc * v[2 * q], y1 = sc * v[2 * q + 1];
            const size_t off = (size_t)row * p.ld_s + col;
            const bool in1 = col + 1 < N;
            if (col >= row && in1) {
                store_bf16x2(ob + off, y0, y1);
            } else {
                // col + 1 == row (only y1 is on or above the diagonal), or col + 1 == N
                if (col >= row) ob[off] = __float2bfloat16_rn(y0);
                if (in1 && col + 1 >= row) ob[off + 1] = __float2bfloat16_rn(y1);
            }
            // mirrors (strictly above the diagonal)
            if (col > row) ob[(size_t)col * p.ld_s + row] = __float2bfloat16_rn(y0);
            if (in1 && col + 1 > row) ob[(size_t)(col + 1) * p.ld_s + row] = __float2bfloat16_rn(y1);
        }
    }
}

// One accumulator tile's epilogue for one warp: rows i0..i0+31 (TMEM lane
// quarter of this warp), columns jb..jb+127 (four 32-column slices).  Loads
// the operands the epilogue reads one slice ahead, waits for the
// accumulator, releases it after the last TMEM read (`release`), and for
// NS_OUT_U writes this warp's ||U||^2 partial to *upart_slot (0 when the
// warp's rows or columns fall outside the matrix).  False if the wait gave up.
// FRAG (the Gram only) selects the fragment-layout epilogue; otherwise slices
// pass through the warp's 4 KB staging tile `st`.
//
// Split-K Gram (`kp0` set): this warp's partial for K range `split` goes to
// kp0 + split*kstride (a private layout: value i of slice k of lane l at
// (32k + i)*32 + l, so every store is one coalesced 128-byte row); after the
// stores, one arrival on *kcnt.  The warp that brings the count to `splits`
// resets it, sums the partials in range order and runs the epilogue.
template <int MODE, int VAR, bool FRAG, class Release>
__device__ __forceinline__ bool epilogue_tile(const GemmParams& p, int g, int i0, int jb, uint32_t tfull_bar,
                                              uint32_t acc_phase, uint32_t trow, float* st, int lane,
                                              volatile int* abort_flag, double* upart_slot, Release release,
                                              float* kp0 = nullptr, size_t kstride = 0, int split = 0,
                                              int* kcnt = nullptr) {
    static_assert(!FRAG || MODE == NS_GRAM, "the fragment-layout epilogue serves the Gram");
    const int nsl = max(0, min(BN / 64, (p.N - jb + 31) / 32));
    float sc = 1.f;
    if (MODE != NS_POLY && p.scale) sc = p.scale[g];
    auto load_slice = [&](uint32_t taddr, float (&v)[32]) {
        if constexpr (FRAG) tmem_ld_quad32(taddr, v);
        else tmem_ld32(taddr, v);
    };
    auto gram_out = [&](int j0, float (&v)[32]) {
        if constexpr (FRAG) {
            gram_slice(p, g, i0, lane, j0, v, sc);
        } else {
            const float4 unused[8] = {};
            sym_slice_st<NS_GRAM>(p, g, i0, lane, j0, v, st, unused, sc);
        }
    };
    if (MODE == NS_GRAM && kp0 != nullptr) {
        if (!mbar_wait(tfull_bar, acc_phase, abort_flag, p.status, wait_limit(p))) return false;
        tc_fence_after();
        if (nsl == 0) {   // no column of this warp's half lies inside the matrix, for any range
            release();
            return true;
        }
        float* mine = kp0 + (size_t)split * kstride;
#pragma unroll
        for (int k = 0; k < BN / 64; ++k) {
            if (k < nsl) {
                float v[32];
                load_slice(trow + 32 * k, v);
                if (k == nsl - 1) {
                    tc_fence_before();
                    release();
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) __stcg(mine + (32 * k + i) * 32 + lane, v[i]);
            }
        }
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atomicAdd(kcnt, 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev != p.splits - 1) return true;
        __threadfence();
        if (lane == 0) *kcnt = 0;   // every range has arrived: ready for the next launch
#pragma unroll
        for (int k = 0; k < BN / 64; ++k) {
            if (k < nsl) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __ldcg(kp0 + (32 * k + i) * 32 + lane);
                for (int sp = 1; sp < p.splits; ++sp) {
                    const float* part = kp0 + (size_t)sp * kstride;
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] += __ldcg(part + (32 * k + i) * 32 + lane);
                }
                gram_out(jb + 32 * k, v);
            }
        }
        return true;
    }
    if constexpr (FRAG) {
        if (!mbar_wait(tfull_bar, acc_phase, abort_flag, p.status, wait_limit(p))) return false;
        tc_fence_after();
        if (nsl == 0) release();
#pragma unroll
        for (int k = 0; k < BN / 64; ++k) {
            if (k < nsl) {
                float v[32];
                load_slice(trow + 32 * k, v);
                if (k == nsl - 1) {
                    tc_fence_before();
                    release();
                }
                gram_out(jb + 32 * k, v);
            }
        }
        return true;
    } else {
        // Where the apply epilogue reads X: the matrix's own input (NS_IN_SRC,
        // fp32, row stride N; the variants need N % 4 == 0), the two-part
        // state written by the previous apply (in_hilo), or the fp32 state
        // written by the momentum kernel.
        NsIO io{nullptr, nullptr, nullptr};
        if (MODE == NS_APPLY && VAR != 0) io = p.io[g];
        const size_t xoff = (size_t)g * p.ld_x * p.M;
        auto pre_x = [&](int j0, float4 (&dst)[8]) {
            if (VAR & NS_IN_SRC)
                prefetch_rm(io.src, p.N, p.M, p.N, i0, lane, j0, dst, true);
            else if (p.in_hilo)
                prefetch_hilo(p.x_hi + xoff, p.x_lo + xoff, p.ld_x, p.M, p.N, i0, lane, j0, dst);
            else
                prefetch_rm(p.x_state + xoff, p.ld_x, p.M, p.N, i0, lane, j0, dst);
        };
        // L2 prefetch of the epilogue's X (and W) for later slices (when
        // p.epi_l2pf): with one slice in registers per warp, a tile's later
        // slices otherwise wait for DRAM one after another
        auto l2_x = [&](int j0) {
            if (VAR & NS_IN_SRC)
                l2_prefetch_rm(io.src, p.N, p.M, p.N, i0, lane, j0);
            else if (p.in_hilo)
                l2_prefetch_hilo(p.x_hi + xoff, p.x_lo + xoff, p.ld_x, p.M, p.N, i0, lane, j0);
            else
                l2_prefetch_rm(p.x_state + xoff, p.ld_x, p.M, p.N, i0, lane, j0);
        };
        // Operands the epilogue reads are loaded one slice ahead.  With
        // NS_OUT_U / NS_OUT_W both X and W are read for the current slice
        // only, at its start (the register budget holds two 32-value slices,
        // not four).
        constexpr bool reads_w = MODE == NS_APPLY && (VAR & (NS_OUT_U | NS_OUT_W));
        constexpr bool ahead = !reads_w;
        const bool keep_w = (MODE == NS_APPLY && (VAR & NS_OUT_W)) ? p.mflags[g] != 0 : false;
        float4 xc[8], xn[8], wc[8];
        float4 ac[8], an[8];   // POLY: A_op, raw bits (4 of 8 used)
        if (nsl > 0) {
            if (MODE == NS_APPLY) pre_x(jb, xc);
            if (reads_w) prefetch_rm(io.w, p.N, p.M, p.N, i0, lane, jb, wc, true);
            if (MODE == NS_APPLY && p.epi_l2pf) {
                // the tile's other slices, into L2
                for (int k = 1; k < nsl; ++k) {
                    l2_x(jb + 32 * k);
                    if (reads_w) l2_prefetch_rm(io.w, p.N, p.M, p.N, i0, lane, jb + 32 * k);
                }
            }
            if (MODE == NS_POLY) prefetch_a_st(p, g, i0, lane, jb, ac);
        }
        if (!mbar_wait(tfull_bar, acc_phase, abort_flag, p.status, wait_limit(p))) return false;
        tc_fence_after();
        if (nsl == 0) release();
        float hacc = 0.f;
#pragma unroll
        for (int k = 0; k < BN / 64; ++k) {
            if (k < nsl) {
                const int j0 = jb + 32 * k;
                if (!ahead && k > 0) {
                    pre_x(j0, xc);
                    prefetch_rm(io.w, p.N, p.M, p.N, i0, lane, j0, wc, true);
                }
                float v[32];
                load_slice(trow + 32 * k, v);
                if (k == nsl - 1) {
                    // last read of this accumulator by this warp
                    tc_fence_before();
                    release();
                }
                if (k + 1 < nsl) {
                    if (MODE == NS_APPLY && ahead) pre_x(j0 + 32, xn);
                    if (MODE == NS_POLY) prefetch_a_st(p, g, i0, lane, j0 + 32, an);
                }
                if (MODE == NS_APPLY) {
                    apply_slice_st<VAR>(p, io, keep_w, g, i0, lane, j0, v, st, xc, wc, sc, hacc);
                    if (ahead) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) xc[u] = xn[u];
                    }
                } else {
                    sym_slice_st<MODE>(p, g, i0, lane, j0, v, st, ac, sc);
                    if (MODE == NS_POLY) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) ac[u] = an[u];
                    }
                }
            }
        }
        if (MODE == NS_APPLY && (VAR & NS_OUT_U)) {
            const double s = warp_sum((double)hacc);
            if (lane == 0 && upart_slot) *upart_slot = s;
        }
        return true;
    }
}

// ---- the kernel ----------------------------------------------------------------
template <int MODE, int VAR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ns_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* smem_a = smem;
    uint8_t* smem_b = smem + STAGES * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2]; then the exit state
    ExitState* ex = reinterpret_cast<ExitState*>(bars + 2 * STAGES + 4);
    static_assert((2 * STAGES + 4) * 8 + sizeof(ExitState) <= 256, "barrier region");
    uint32_t* tmem_slot = &ex->tmem_slot;
    volatile int* abort_flag = &ex->abort_flag;
    float* stage_base = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain_bar = smem_u32(&ex->drain_bar);
    const unsigned long long tlimit = wait_limit(p);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(tfull0 + 8 * s, 1);
            mbar_init(tempty0 + 8 * s, 32 * EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ex->fills = 0;
        ex->consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_b);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int total = p.G * p.tiles_per_mat;
    const int num_kb = (p.K + BK - 1) / BK;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = !p.test_no_loads;
        int fills = 0;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const int g = t / p.tiles_per_mat;
            int mi, nj;
            tile_coords(p, t - g * p.tiles_per_mat, mi, nj);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status, tlimit)) { ok = false; break; }
                const uint32_t fb = full0 + 8 * stage;
                mbar_expect_tx(fb, STAGE_BYTES);
                const uint32_t sa = smem_u32(smem_a + stage * A_BYTES);
                const uint32_t sb = smem_u32(smem_b + stage * B_BYTES);
                if (!p.a_mn) {
                    tma_load_3d(sa, &tm_a, fb, kb * BK, mi * BM, g);
                } else {
#pragma unroll
                    for (int c = 0; c < BM / 64; ++c) tma_load_3d(sa + c * (64 * BK * 2), &tm_a, fb, mi * BM + c * 64, kb * BK, g);
                }
                if (!p.b_mn) {
                    tma_load_3d(sb, &tm_b, fb, kb * BK, nj * BN, g);
                } else {
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c) tma_load_3d(sb + c * (64 * BK * 2), &tm_b, fb, nj * BN + c * 64, kb * BK, g);
                }
                ++fills;
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        ex->fills = fills;
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = idesc_bf16(p.a_mn != 0, p.b_mn != 0);
        const uint64_t a_desc0 = operand_desc(smem_u32(smem_a), 0, p.a_mn != 0);
        const uint64_t b_desc0 = operand_desc(smem_u32(smem_b), 0, p.b_mn != 0);
        const uint64_t a_step = operand_desc_step(p.a_mn != 0), b_step = operand_desc_step(p.b_mn != 0);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        int consumed = 0;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, p.status, tlimit)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status, tlimit)) { ok = false; break; }
                ++consumed;
                tc_fence_after();
                // descriptors: stage base plus add-only steps along K
                const uint64_t ad = a_desc0 + (uint64_t)(stage * (A_BYTES >> 4));
                const uint64_t bd = b_desc0 + (uint64_t)(stage * (B_BYTES >> 4));
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16(d_tmem, ad + kk * a_step, bd + kk * b_step, idesc, (kb | kk) ? 1u : 0u);
                mma_commit(empty0 + 8 * stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            mma_commit(tfull0 + 8 * acc);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        ex->consumed = consumed;
        // every MMA this thread issued has completed before TMEM is freed
        mma_commit(drain_bar);
        mbar_drain_wait(drain_bar, 0, p.status, tlimit);
    } else if (warp >= 2) {
        // ---------------- epilogue ----------------
        // warp w reads TMEM lane quarter w%4; warps 2..5 take accumulator
        // columns 0..127, warps 6..9 columns 128..255
        const int e = warp - 2;
        const int q = warp & 3;
        const int h = e >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t tempty_bar = tempty0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const int g = t / p.tiles_per_mat;
            int mi, nj;
            tile_coords(p, t - g * p.tiles_per_mat, mi, nj);
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + h * (BN / 2));
            const uint32_t te = tempty_bar + 8 * acc;
            double* slot = (VAR & NS_OUT_U) ? p.upart + (size_t)t * kUPartsPerTile1 + e : nullptr;
            if (!epilogue_tile<MODE, VAR, false>(p, g, mi * BM + q * 32, nj * BN + h * (BN / 2), tfull0 + 8 * acc,
                                                 acc_phase, trow, stage_base + e * ST_FLOATS, lane, abort_flag, slot,
                                                 [&]() { mbar_arrive(te); }))
                break;
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        // stage fills issued but never consumed (a wait gave up): their
        // copies land in this CTA's shared memory, so wait for them here
        for (int i = ex->consumed; i < ex->fills; ++i)
            mbar_drain_wait(full0 + 8 * (i % STAGES), (uint32_t)(i / STAGES) & 1u, p.status, tlimit);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// ---- 2-SM variant: one CTA pair (cluster of 2) per 256 x 256 tile -------------------
// tcgen05.mma.cta_group::2 issued by the even CTA of the pair computes a
// 256 x 256 tile: each CTA holds 128 rows of A and 128 rows (N) of B in its
// own shared memory and receives its 128 accumulator rows in its own TMEM.
// Per CTA and K step this moves 32 KB instead of 48 KB, so the ring is 6
// stages deep.  Both CTAs' TMA loads complete on the even CTA's full barrier;
// the MMA commits are multicast to both CTAs' empty / tmem-full barriers; the
// epilogue warps of both CTAs release an accumulator on the even CTA's
// tmem-empty barrier.
namespace pair {

constexpr int STAGES2 = 6;                            // one-K-step stages (32 KB each) of the ring
constexpr int A2_BYTES = BM * BK * 2;                 // 16 KB: this CTA's 128 rows of A
constexpr int B2_BYTES = (BN / 2) * BK * 2;           // 16 KB: this CTA's 128 rows of B
constexpr int STAGE2_BYTES = A2_BYTES + B2_BYTES;
// the ring, barriers and exit state, and the epilogue warps' staging tiles
// (used by the one-K-step pipeline's epilogue)
constexpr int SMEM2_BYTES = STAGES2 * STAGE2_BYTES + 1024 + 256 + EPI_WARPS * ST_FLOATS * 4;
static_assert(SMEM2_BYTES <= 232448, "shared memory per CTA");

// Pipeline shape of the pair kernel: KPS K steps of BK per stage.  Alone,
// TMA moves about 56 bytes per SM clock into shared memory with 16 KB boxes
// and about 80 with 32 KB boxes (8 KB boxes: about 40), while a 256 x 256
// pair tile consumes 64 bytes per clock per SM at the full MMA rate.  A
// two-step stage is loaded by one 32 KB box per operand (4-D view of a
// K-major operand, 5-D view of an MN-major one); within it, K step j sits at
// +j * 16 KB in the layout of a one-step stage, so the MMA descriptors are
// those of the one-step pipeline plus that offset.  Inside the GEMM the two
// shapes deliver about the same bytes per clock (the MMA's own shared-memory
// reads share the SM's bandwidth), and the three-stage ring holds less in
// flight, so the host takes two steps only where that measured faster.
template <int KPS>
struct PairPipe {
    static constexpr int STAGES = STAGES2 / KPS;
    static constexpr int A_STEP = BM * BK * 2;          // 16 KB: one K step of this CTA's A rows
    static constexpr int B_STEP = (BN / 2) * BK * 2;    // 16 KB: one K step of this CTA's B rows
    static constexpr int A_BYTES = KPS * A_STEP;
    static constexpr int B_BYTES = KPS * B_STEP;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
};
static_assert(PairPipe<1>::STAGES * PairPipe<1>::STAGE_BYTES == STAGES2 * STAGE2_BYTES, "pipelines share smem size");
static_assert(PairPipe<2>::STAGES * PairPipe<2>::STAGE_BYTES == STAGES2 * STAGE2_BYTES, "pipelines share smem size");
static_assert(PairPipe<1>::A_BYTES == PairPipe<1>::B_BYTES && PairPipe<2>::A_BYTES == PairPipe<2>::B_BYTES &&
                  PairPipe<1>::A_STEP == PairPipe<1>::B_STEP,
              "a diagonal tile reads B from A's buffer");

// TMA load into this CTA's shared memory, completing on a barrier that may
// belong to the peer CTA of the pair.
// MUONH_TMA_L2_HINT (build-time): 1 tags the operand loads with an L2
// evict_last cache policy (operand panels are re-read by the neighbouring
// tiles of a launch), 0 loads them with the default policy.
#ifndef MUONH_TMA_L2_HINT
#define MUONH_TMA_L2_HINT 0
#endif
__device__ __forceinline__ uint64_t operand_policy() {
    uint64_t pol = 0;
#if MUONH_TMA_L2_HINT
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
#endif
    return pol;
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cluster_bar, int x,
                                                 int y, int z, uint64_t pol = 0) {
#if MUONH_TMA_L2_HINT
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(x), "r"(y), "r"(z), "l"(pol)
        : "memory");
#else
    (void)pol;
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(x), "r"(y), "r"(z)
        : "memory");
#endif
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cluster_bar, int c0,
                                                 int c1, int c2, int c3, uint64_t pol = 0) {
#if MUONH_TMA_L2_HINT
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
        : "memory");
#else
    (void)pol;
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
#endif
}
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cluster_bar, int c0,
                                                 int c1, int c2, int c3, int c4, uint64_t pol = 0) {
#if MUONH_TMA_L2_HINT
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "l"(pol)
        : "memory");
#else
    (void)pol;
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
#endif
}
__host__ __device__ constexpr uint32_t idesc_pair(bool a_mn_major, bool b_mn_major) {
    return idesc_f16(2 * BM, BN, a_mn_major, b_mn_major);
}

// Pair tile (mp, nj): rows mp*256 .. +255, columns nj*256 .. +255.
// Symmetric modes keep nj >= mp.
__device__ __forceinline__ void pair_coords(const GemmParams& p, int local, int& mp, int& nj) {
    if (p.mode == NS_APPLY) {
        if (p.m_outer) {
            mp = local / p.tiles_n;
            nj = local - mp * p.tiles_n;
        } else {
            nj = local / p.tiles_m;
            mp = local - nj * p.tiles_m;
        }
        return;
    }
    int m = 0;
    for (;;) {
        const int cnt = p.tiles_n - m;
        if (local < cnt) break;
        local -= cnt;
        ++m;
    }
    mp = m;
    nj = m + local;
}

// KPS = 1: 3-D maps, K-major box 64 x 128, MN-major box 64 x 64 (two per
// operand and step).  KPS = 2: K-major 4-D map {64 k, rows, K/64, G}, box
// {64, 128, 2, 1}; MN-major 5-D map {64 m, 64 k, M/64, K/64, G}, box
// {64, 64, 2, 2, 1}.  Both give, per K step, 128 rows of 128 bytes in the
// 128B-swizzled layout (MN-major: two 64-wide chunks 8 KB apart).
template <int MODE, int VAR, int KPS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
ns_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ GemmParams p) {
    using Pipe = PairPipe<KPS>;
    constexpr int STAGES2 = Pipe::STAGES, A2_BYTES = Pipe::A_BYTES, B2_BYTES = Pipe::B_BYTES;
    constexpr int STAGE2_BYTES = Pipe::STAGE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* smem_a = smem;
    uint8_t* smem_b = smem + STAGES2 * A2_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES2 * STAGE2_BYTES);
    // bars: full[STAGES2], empty[STAGES2], tfull[2], tempty[2]; then the exit state
    ExitState* ex = reinterpret_cast<ExitState*>(bars + 2 * STAGES2 + 4);
    static_assert((2 * STAGES2 + 4) * 8 + sizeof(ExitState) <= 256 && STAGES2 <= 8, "barrier region");
    uint32_t* tmem_slot = &ex->tmem_slot;
    volatile int* abort_flag = &ex->abort_flag;
    float* stage_base = reinterpret_cast<float*>(smem + STAGES2 * STAGE2_BYTES + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES2);
    const uint32_t tfull0 = smem_u32(bars + 2 * STAGES2), tempty0 = smem_u32(bars + 2 * STAGES2 + 2);
    const uint32_t drain_bar = smem_u32(&ex->drain_bar);
    const unsigned long long tlimit = wait_limit(p);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(tfull0 + 8 * s, 1);
            mbar_init(tempty0 + 8 * s, 2 * EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ex->fills = 0;
        ex->consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_b);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // work units: (K range, tile), the range outermost; one range unless the
    // Gram is split (splits > 1)
    const int total = p.G * p.tiles_per_mat;
    const int units = total * p.splits;
    const int num_kb = (p.K + BK - 1) / BK;
    const int cid = (int)cluster_id(), ncl = (int)cluster_count();

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        const uint64_t pol = operand_policy();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = !p.test_no_loads;
        int fills = 0;
        for (int u = cid; u < units && ok; u += ncl) {
            const int split = u / total, t = u - split * total;
            const int kb0 = split * p.kb_per_split, kb1 = min(num_kb, kb0 + p.kb_per_split);
            const int g = t / p.tiles_per_mat;
            int mp, nj;
            pair_coords(p, t - g * p.tiles_per_mat, mp, nj);
            const int row_a = mp * 2 * BM + (int)rank * BM;       // this CTA's 128 rows of A
            const int row_b = nj * BN + (int)rank * (BN / 2);     // this CTA's 128 rows (N) of B
            // diagonal tile of a symmetric product: this CTA's B rows are its A
            // rows (same operand tensor), so B is not fetched
            const bool diag = MODE != NS_APPLY && mp == nj;
            for (int ks = kb0 / KPS; ks * KPS < kb1; ++ks) {
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status, tlimit)) { ok = false; break; }
                const uint32_t fb_local = full0 + 8 * stage;
                const uint32_t fb = map_to_rank(fb_local, 0);
                // the leader's full barrier expects both CTAs' bytes; each CTA loads half
                const uint32_t both = diag ? 2 * A2_BYTES : 2 * STAGE2_BYTES;
                ex->fill_bytes[stage] = leader ? both : both / 2;
                ++fills;
                if (leader) mbar_expect_tx(fb_local, both);
                const uint32_t sa = smem_u32(smem_a + stage * A2_BYTES);
                const uint32_t sb = smem_u32(smem_b + stage * B2_BYTES);
                if (KPS == 2) {
                    // K steps 2ks and 2ks+1 (the second is zero-filled past K)
                    if (!p.a_mn)
                        tma_load_4d_pair(sa, &tm_a, fb, 0, row_a, 2 * ks, g, pol);
                    else
                        tma_load_5d_pair(sa, &tm_a, fb, 0, 0, row_a / 64, 2 * ks, g, pol);
                    if (diag) {
                    } else if (!p.b_mn)
                        tma_load_4d_pair(sb, &tm_b, fb, 0, row_b, 2 * ks, g, pol);
                    else
                        tma_load_5d_pair(sb, &tm_b, fb, 0, 0, row_b / 64, 2 * ks, g, pol);
                    if (++stage == STAGES2) { stage = 0; phase ^= 1; }
                    continue;
                }
                const int kb = ks;
                if (!p.a_mn) {
                    tma_load_3d_pair(sa, &tm_a, fb, kb * BK, row_a, g, pol);
                } else {
#pragma unroll
                    for (int c = 0; c < BM / 64; ++c)
                        tma_load_3d_pair(sa + c * (64 * BK * 2), &tm_a, fb, row_a + c * 64, kb * BK, g, pol);
                }
                if (diag) {
                } else if (!p.b_mn) {
                    tma_load_3d_pair(sb, &tm_b, fb, kb * BK, row_b, g, pol);
                } else {
#pragma unroll
                    for (int c = 0; c < BN / 128; ++c)
                        tma_load_3d_pair(sb + c * (64 * BK * 2), &tm_b, fb, row_b + c * 64, kb * BK, g, pol);
                }
                if (++stage == STAGES2) { stage = 0; phase ^= 1; }
            }
        }
        ex->fills = fills;
    } else if (warp == 1 && lane == 0 && leader) {
        // ---------------- MMA issuer (even CTA only) ----------------
        const uint32_t idesc = idesc_pair(p.a_mn != 0, p.b_mn != 0);
        const uint64_t a_desc0 = operand_desc(smem_u32(smem_a), 0, p.a_mn != 0);
        const uint64_t b_desc0 = operand_desc(smem_u32(smem_b), 0, p.b_mn != 0);
        const uint64_t a_step = operand_desc_step(p.a_mn != 0), b_step = operand_desc_step(p.b_mn != 0);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        int consumed = 0;
        for (int u = cid; u < units && ok; u += ncl) {
            const int split = u / total, t = u - split * total;
            const int kb0 = split * p.kb_per_split, kb1 = min(num_kb, kb0 + p.kb_per_split);
            bool diag = false;
            if (MODE != NS_APPLY) {
                const int g = t / p.tiles_per_mat;
                int mp, nj;
                pair_coords(p, t - g * p.tiles_per_mat, mp, nj);
                diag = mp == nj;
            }
            // B of a diagonal tile is read from A's buffer (same layout and size)
            const uint64_t b_base = diag ? a_desc0 : b_desc0;
            const int b_stage = diag ? A2_BYTES : B2_BYTES;
            if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, p.status, tlimit)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int ks = kb0 / KPS; ks * KPS < kb1; ++ks) {
                if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status, tlimit)) { ok = false; break; }
                ++consumed;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < KPS; ++j) {
                    const int kb = ks * KPS + j;
                    if (KPS > 1 && kb >= kb1) break;
                    const uint64_t ad = a_desc0 + (uint64_t)((stage * A2_BYTES + j * Pipe::A_STEP) >> 4);
                    const uint64_t bd = b_base + (uint64_t)((stage * b_stage + j * Pipe::B_STEP) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16_pair(d_tmem, ad + kk * a_step, bd + kk * b_step, idesc,
                                      ((kb - kb0) | kk) ? 1u : 0u);
                }
                mma_commit_pair(empty0 + 8 * stage);
                if (++stage == STAGES2) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            mma_commit_pair(tfull0 + 8 * acc);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        ex->consumed = consumed;
        // every MMA this thread issued (they read both CTAs' shared memory and
        // write both CTAs' TMEM) has completed before either CTA moves on
        mma_commit_pair(drain_bar, 1);
        mbar_drain_wait(drain_bar, 0, p.status, tlimit);
    } else if (warp >= 2) {
        // ---------------- epilogue (both CTAs: 128 rows each) ----------------
        const int e = warp - 2;
        const int q = warp & 3;
        const int h = e >> 2;
        const uint32_t tempty_leader = map_to_rank(tempty0, 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        const bool split_k = MODE == NS_GRAM && p.splits > 1;
        const size_t kstride = (size_t)total * 2 * 8 * 4096;
        for (int u = cid; u < units; u += ncl) {
            const int split = u / total, t = u - split * total;
            const int g = t / p.tiles_per_mat;
            int mp, nj;
            pair_coords(p, t - g * p.tiles_per_mat, mp, nj);
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + h * (BN / 2));
            const uint32_t te = tempty_leader + 8 * acc;
            double* slot = (VAR & NS_OUT_U)
                               ? p.upart + ((size_t)t * 2 + rank) * (kUPartsPerTilePair / 2) + e
                               : nullptr;
            const size_t wslot = ((size_t)t * 2 + rank) * 8 + e;   // this warp's (tile, CTA, warp)
            // two-K-step stages take the fragment-layout epilogue (it measured
            // faster there), one-K-step stages the staged one
            if (!epilogue_tile<MODE, VAR, KPS == 2>(p, g, mp * 2 * BM + (int)rank * BM + q * 32,
                                          nj * BN + h * (BN / 2), tfull0 + 8 * acc, acc_phase, trow,
                                          stage_base + e * ST_FLOATS, lane, abort_flag, slot,
                                          [&]() {
                                              __syncwarp();
                                              if (lane == 0) remote_arrive(te);
                                          },
                                          split_k ? p.kpart + wslot * 4096 : nullptr, kstride, split,
                                          split_k ? p.kcount + wslot : nullptr))
                break;
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    cluster_sync();   // neither CTA issues another copy or MMA from here on
    if (leader && threadIdx.x == 0) {
        // Stage fills issued but never consumed (a wait gave up) still land in
        // either CTA's shared memory and complete on this CTA's full
        // barriers.  Both producers walk the same stage sequence, each fill
        // waits for the consumption of the fill one ring earlier, so every
        // unconsumed fill is the only one outstanding on its stage.  Fill i
        // is complete when its phase is: where only one producer issued it,
        // the missing half of the barrier's accounting is supplied first.
        const int C = ex->consumed, n_lead = ex->fills;
        const int n_peer = (int)ld_cluster_u32(map_to_rank(smem_u32(&ex->fills), 1));
        const int n_max = max(n_lead, n_peer);
        for (int i = C; i < n_max; ++i) {
            const int s = i % STAGES2;
            const uint32_t fb = full0 + 8 * s;
            if (i >= n_lead)        // the peer loaded, the leader never armed the barrier
                mbar_expect_tx(fb, ld_cluster_u32(map_to_rank(smem_u32(&ex->fill_bytes[s]), 1)));
            else if (i >= n_peer)   // the leader expected the peer's half, which never comes
                mbar_complete_tx(fb, ex->fill_bytes[s] / 2);
            mbar_drain_wait(fb, (uint32_t)(i / STAGES2) & 1u, p.status, tlimit);
        }
    }
    cluster_sync();   // no CTA leaves while its peer may still signal, read or receive into it
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

}  // namespace pair

// ---- host side -------------------------------------------------------------------
#ifndef MUONH_TMA_PROMOTION
#define MUONH_TMA_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// bf16 tensor [G][rows][ld] (cols valid), box {64, box_rows, 1}, 128B swizzle.
static bool encode_bf16_3d(CUtensorMap* map, const void* base, int cols, int rows, int G, int ld, int box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)G};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * 2 * (cuuint64_t)rows};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, MUONH_TMA_PROMOTION,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Two-K-step boxes (pair kernel, KPS = 2).  K-major operand [G][rows][ld],
// K valid columns (K % 64 == 0): {64 k, rows, K/64, G}, box {64, 128, 2, 1}.
// MN-major operand [G][K][ld], `cols` valid columns (cols % 64 == 0, K % 64
// == 0): {64 m, 64 k, cols/64, K/64, G}, box {64, 64, 2, 2, 1}.  Every
// coordinate past an extent reads zeros.
static bool encode_bf16_kmajor_2step(CUtensorMap* map, const void* base, int K, int rows, int G, int ld) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(K / 64), (cuuint64_t)G};
    cuuint64_t strides[3] = {(cuuint64_t)ld * 2, 128, (cuuint64_t)ld * 2 * (cuuint64_t)rows};
    cuuint32_t box[4] = {64, (cuuint32_t)BM, 2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, MUONH_TMA_PROMOTION,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
static bool encode_bf16_mnmajor_2step(CUtensorMap* map, const void* base, int cols, int K, int G, int ld) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[5] = {64, 64, (cuuint64_t)(cols / 64), (cuuint64_t)(K / 64), (cuuint64_t)G};
    cuuint64_t strides[4] = {(cuuint64_t)ld * 2, 128, (cuuint64_t)ld * 2 * 64, (cuuint64_t)ld * 2 * (cuuint64_t)K};
    cuuint32_t box[5] = {64, 64, 2, 2, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, MUONH_TMA_PROMOTION,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

int tiles_per_matrix(int mode, int M, int N) {
    const int tm = (M + BM - 1) / BM, tn = (N + BN - 1) / BN;
    if (mode == NS_APPLY) return tm * tn;
    int cnt = 0;
    for (int m = 0; m < tm; ++m) cnt += tn - (m >> 1) > 0 ? tn - (m >> 1) : 0;
    return cnt;
}

int pair_tiles_per_matrix(int mode, int M, int N) {
    const int tm = (M + 2 * BM - 1) / (2 * BM), tn = (N + BN - 1) / BN;
    if (mode == NS_APPLY) return tm * tn;
    int cnt = 0;
    for (int m = 0; m < tm; ++m) cnt += tn - m > 0 ? tn - m : 0;
    return cnt;
}

// A Gram launch with few pair tiles (<= 16; a B300 runs 74 CTA pairs)
// leaves most SMs idle for its whole duration: its K steps (>= 16 per range)
// are cut into ranges so that the units number about 148.  Measured on a
// lone 16384x1024 orthogonalisation (10 tiles): 1.09 -> 0.97 ms; launches
// with 36 tiles were 3-7 % slower split, so they are not.
#ifndef MUONH_SPLIT_MAX
#define MUONH_SPLIT_MAX 8
#endif
#ifndef MUONH_SPLIT_TARGET
#define MUONH_SPLIT_TARGET 148
#endif
#ifndef MUONH_SPLIT_MAX_TILES
#define MUONH_SPLIT_MAX_TILES 16
#endif
#ifndef MUONH_SPLIT_MIN_STEPS
#define MUONH_SPLIT_MIN_STEPS 16
#endif
int gram_splits(long long tiles, int K) {
    constexpr long long kTargetUnits = MUONH_SPLIT_TARGET;
    const int nkb = (K + BK - 1) / BK;
    if (tiles <= 0 || tiles > MUONH_SPLIT_MAX_TILES || tiles >= kTargetUnits) return 1;
    long long sp = (kTargetUnits + tiles - 1) / tiles;
    sp = std::min<long long>(sp, nkb / MUONH_SPLIT_MIN_STEPS);
    sp = std::min<long long>(sp, MUONH_SPLIT_MAX);
    return sp < 1 ? 1 : (int)sp;
}

template <int MODE, int VAR, int KPS>
static int max_pair_clusters() {
    static int cached = 0;
    if (cached) return cached;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 148, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = pair::SMEM2_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, pair::ns_gemm_pair_kernel<MODE, VAR, KPS>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        n = sm_count() / 2;
    }
    cached = n;
    return n;
}

template <int MODE, int VAR, int KPS>
static cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, long long total,
                               cudaStream_t st) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(pair::ns_gemm_pair_kernel<MODE, VAR, KPS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, pair::SMEM2_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int maxc = max_pair_clusters<MODE, VAR, KPS>();
    const long long clusters = total < maxc ? total : maxc;
    pair::ns_gemm_pair_kernel<MODE, VAR, KPS><<<(int)(2 * clusters), NUM_THREADS, pair::SMEM2_BYTES, st>>>(ta, tb, p);
    return cudaGetLastError();
}

template <int MODE, int VAR>
static cudaError_t launch_single(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, long long total,
                                 cudaStream_t st) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel<MODE, VAR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int grid = (int)(total < sm_count() ? total : sm_count());
    ns_gemm_kernel<MODE, VAR><<<grid, NUM_THREADS, SMEM_BYTES, st>>>(ta, tb, p);
    return cudaGetLastError();
}

int pair_cluster_capacity() { return max_pair_clusters<NS_GRAM, 0, 2>(); }

template <int KIND>
static cudaError_t dispatch(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, long long total,
                            cudaStream_t st) {
#define MUONH_LAUNCH(M_, V_)                                                                      \
    (KIND == kGemmPair || KIND == kGemmPairStep1 ? launch_pair<M_, V_, 1>(ta, tb, p, total, st)   \
                                                 : launch_single<M_, V_>(ta, tb, p, total, st))
    // two K steps per stage: the Gram only (the launcher picks the kind)
    if (p.mode == NS_GRAM)
        return KIND == kGemmPair ? launch_pair<NS_GRAM, 0, 2>(ta, tb, p, total, st) : MUONH_LAUNCH(NS_GRAM, 0);
    if (p.mode == NS_POLY) return MUONH_LAUNCH(NS_POLY, 0);
    switch (p.variant) {
        case 0: return MUONH_LAUNCH(NS_APPLY, 0);
        case NS_IN_SRC: return MUONH_LAUNCH(NS_APPLY, NS_IN_SRC);
        case NS_OUT_U: return MUONH_LAUNCH(NS_APPLY, NS_OUT_U);
        case NS_IN_SRC | NS_OUT_U: return MUONH_LAUNCH(NS_APPLY, NS_IN_SRC | NS_OUT_U);
        case NS_OUT_W: return MUONH_LAUNCH(NS_APPLY, NS_OUT_W);
        case NS_IN_SRC | NS_OUT_W: return MUONH_LAUNCH(NS_APPLY, NS_IN_SRC | NS_OUT_W);
        default: return cudaErrorInvalidValue;
    }
#undef MUONH_LAUNCH
}

// Operand tensors ([G][rows][ld] bf16, ld = a_ld / b_ld):
//   K-major operand:  rows = M (or N), cols = K; box 64 x 128 (A, and B in
//                     the pair kernel: 128 rows per CTA) or 64 x 256 (B in the
//                     1-SM kernel)
//   MN-major operand: rows = K, cols = M (or N); box 64 x 64
// GRAM wide: A = B = X_op (K-major);  GRAM tall: A = B = X_op (MN-major);
// POLY: A = B = A_op (K-major);  APPLY wide: A = B_op (K-major), B = X_op
// (MN-major);  APPLY tall: A = X_op, B = B_op (both K-major).
// `kind` selects the 1-SM or the 2-SM kernel.
cudaError_t launch_ns_gemm(GemmParams p, const void* a_op, int a_ld, const void* b_op, int b_ld, int kind,
                           cudaStream_t st, const char** why) {
    if (p.mode != NS_APPLY) p.variant = 0;
    if (p.variant != 0 && !p.io) { *why = "apply variant without per-matrix buffers"; return cudaErrorInvalidValue; }
    if ((p.variant & NS_OUT_U) && !p.upart) { *why = "apply variant without partial buffer"; return cudaErrorInvalidValue; }
    if ((p.variant & NS_OUT_W) && !p.mflags) { *why = "apply variant without status flags"; return cudaErrorInvalidValue; }
    if ((p.variant & NS_OUT_U) && (p.variant & NS_OUT_W)) { *why = "conflicting apply variants"; return cudaErrorInvalidValue; }
    if (p.variant != 0 && (p.N & 3) != 0) { *why = "apply variant needs a row length that is a multiple of 4"; return cudaErrorInvalidValue; }
    if (kind != kGemmSingle && kind != kGemmPair && kind != kGemmPairStep1) {
        *why = "unknown GEMM kernel";
        return cudaErrorInvalidValue;
    }
    // two-K-step stages need every box coordinate past the data to be an
    // extent of the view: K, and the contiguous extent of an MN-major operand,
    // multiples of 64
    // Measured on the 2B set (cycles per K step, two-step vs one-step
    // stages): tall Gram 595 vs 653, wide Gram 660 vs 663, polynomial 801
    // vs 745, apply 635-675 vs 636-669.  Three 64 KB stages keep less data
    // in flight than six 32 KB ones, which only the tall Gram's four 8 KB
    // MN-major boxes per step outweigh; the other launches keep one step.
    // Two-step stages for the tall Gram only (MN-major operands, whose one-
    // step stages take four 8 KB boxes); measured slower for every other
    // launch kind (see the comment above)
    const bool two_step_ok = (p.K % 64) == 0 && (p.M % 64) == 0 && (p.N % 64) == 0;
    const bool two_step_wanted = p.mode == NS_GRAM && p.a_mn;
    if (kind == kGemmPair && !(two_step_ok && two_step_wanted)) kind = kGemmPairStep1;
    const bool multi = kind != kGemmSingle;
    const int a_box = BM;
    const int b_box = kind == kGemmPairStep1 ? BN / 2 : BN;
    CUtensorMap ta, tb;
    bool oka, okb;
    if (kind == kGemmPair) {
        oka = p.a_mn ? encode_bf16_mnmajor_2step(&ta, a_op, p.M, p.K, p.G, a_ld)
                     : encode_bf16_kmajor_2step(&ta, a_op, p.K, p.M, p.G, a_ld);
        okb = p.b_mn ? encode_bf16_mnmajor_2step(&tb, b_op, p.N, p.K, p.G, b_ld)
                     : encode_bf16_kmajor_2step(&tb, b_op, p.K, p.N, p.G, b_ld);
    } else {
        oka = p.a_mn ? encode_bf16_3d(&ta, a_op, p.M, p.K, p.G, a_ld, 64)
                     : encode_bf16_3d(&ta, a_op, p.K, p.M, p.G, a_ld, a_box);
        okb = p.b_mn ? encode_bf16_3d(&tb, b_op, p.N, p.K, p.G, b_ld, 64)
                     : encode_bf16_3d(&tb, b_op, p.K, p.N, p.G, b_ld, b_box);
    }
    if (!oka) { *why = "cuTensorMapEncodeTiled (A) failed"; return cudaErrorInvalidValue; }
    if (!okb) { *why = "cuTensorMapEncodeTiled (B) failed"; return cudaErrorInvalidValue; }
    if (multi) {
        p.tiles_m = (p.M + 2 * BM - 1) / (2 * BM);
        p.tiles_n = (p.N + BN - 1) / BN;
        p.tiles_per_mat = pair_tiles_per_matrix(p.mode, p.M, p.N);
    } else {
        p.tiles_m = (p.M + BM - 1) / BM;
        p.tiles_n = (p.N + BN - 1) / BN;
        p.tiles_per_mat = tiles_per_matrix(p.mode, p.M, p.N);
    }
    long long total = (long long)p.G * p.tiles_per_mat;
    if (total <= 0) return cudaSuccess;
    // split K: pair kernel, Gram only; ranges of an even number of K steps, so
    // one- and two-step pipeline stages cut K at the same places
    const int num_kb = (p.K + BK - 1) / BK;
    if (p.splits > 1 && multi && p.mode == NS_GRAM) {
        if (!p.kpart || !p.kcount) { *why = "split-K Gram without partial buffers"; return cudaErrorInvalidValue; }
        int len = (num_kb + p.splits - 1) / p.splits;
        len += len & 1;
        p.kb_per_split = len;
        p.splits = (num_kb + len - 1) / len;
    } else {
        p.splits = 1;
        p.kb_per_split = num_kb;
    }
    total *= p.splits;
    cudaError_t e = kind == kGemmPair        ? dispatch<kGemmPair>(ta, tb, p, total, st)
                    : kind == kGemmPairStep1 ? dispatch<kGemmPairStep1>(ta, tb, p, total, st)
                                             : dispatch<kGemmSingle>(ta, tb, p, total, st);
    if (e != cudaSuccess)
        *why = kind == kGemmSingle ? "GEMM launch failed" : "2-SM GEMM launch failed";
    return e;
}

}  // namespace tc
}  // namespace muonh
