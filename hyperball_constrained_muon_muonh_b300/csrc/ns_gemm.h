// Internal interface of the Newton-Schulz GEMM kernels (tcgen05 and fp32).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/muonh.h"

namespace muonh {

enum NsMode { NS_GRAM = 0, NS_POLY = 1, NS_APPLY = 2 };

// Variants of the apply stage (bit set):
//   NS_IN_SRC   X is read from the matrix's own unscaled input (NsIO::src, W
//               orientation) instead of the fp32 state: the first iteration
//   NS_OUT_U    the epilogue finishes O = X and writes U = W - lr*O into
//               the fp32 state, plus deterministic per-warp partial sums of
//               ||U||^2: the last iteration of a MuonH step
//   NS_OUT_W    the epilogue finishes O = X and writes the new weight
//               wdecay*W - lr*O (fp32, and bf16 when NsIO::wb is set) into
//               the caller's buffers, unless the matrix's status flag is set:
//               the last iteration of a plain Muon step
enum NsApplyVariant { NS_IN_SRC = 1, NS_OUT_U = 2, NS_OUT_W = 4 };

struct NsIO;

// One launch = one Newton-Schulz stage over a bucket of G same-shape
// matrices.  X keeps the matrix's own orientation, R x C (row stride ld_x);
// s = min(R, C), l = max(R, C); ld_s = row stride of the s x s buffers.
//   GRAM : M = N = s, K = l.  sym_bf16 <- bf16(scale*Gram) (both triangles),
//          Gram = X X^T (wide, R <= C) or X^T X (tall, R > C)
//   POLY : M = N = K = s.     sym_bf16 <- bf16(cb*A + cc*(A A)), with A the
//          Gram's bf16 copy a_op in both terms
//   APPLY: M = R, N = C, K = s.  X <- scale*(ca*X + P), with P = B X (wide)
//          or X B (tall); the new X goes to (x_op_out, x_lo) as hi + lo
//          when x_op_out is set, else to x_state (fp32).  `variant`
//          (NS_IN_SRC, NS_OUT_U, NS_OUT_W) and in_hilo select where X comes
//          from and what is written.
// Operand tiles are K-major (rows of the operand run along M or N, K
// contiguous) unless a_mn / b_mn say MN-major (K runs along the rows).
struct GemmParams {
    int mode;
    int variant;            // apply only: NsApplyVariant bits
    int a_mn, b_mn;         // operand A / B stored MN-major
    int m_outer;            // apply: tiles ordered row panels outermost (consecutive tiles
                            // share their A panel) instead of column panels outermost
    int epi_l2pf;           // apply: the epilogue prefetches a tile's later slices of X (and W)
                            // into L2 when it starts the tile
    int G, M, N, K;
    int tiles_m, tiles_n, tiles_per_mat;   // filled by the launcher
    int ld_x, ld_s;
    float* x_state;
    __nv_bfloat16* x_op_out;
    // APPLY: the two-part state X = hi + lo (bf16 each, [G][M][ld_x]) that
    // every apply with another iteration after it writes (hi to x_op_out, lo
    // to x_lo, in place) and that in_hilo applies read (hi from x_hi, the
    // current operand copy of X).  The momentum kernel's fp32 state is read
    // by the first apply of unfused matrices; the last apply writes fp32.
    const __nv_bfloat16* x_hi;
    __nv_bfloat16* x_lo;
    int in_hilo;
    const __nv_bfloat16* a_op;   // POLY: the Gram's bf16 output (read for the b*A term)
    __nv_bfloat16* sym_bf16;
    const float* scale;     // per-matrix factor (bucket-local index) or null
    const NsIO* io;         // NS_IN_SRC / NS_OUT_U: per-matrix buffers (bucket-local index)
    double* upart;          // NS_OUT_U: ||U||^2 partials, warps_per_tile per tile, tile order
    const uint32_t* mflags; // NS_OUT_W: per-matrix status bits (bucket-local); set = keep W
    float nlr;              // NS_OUT_U / NS_OUT_W: -lr
    float wdecay;           // NS_OUT_W: 1 - lr*weight_decay
    float ca, cb, cc;
    uint32_t* status;       // device status word
    // Split K (the Gram in the pair kernel, when a launch has few tiles): the
    // K steps are cut into `splits` ranges of kb_per_split 64-wide steps
    // (even); each (tile, range) is a work unit.  Every unit writes its
    // partial product to kpart; the last unit of a tile to finish sums the
    // partials in range order and runs the epilogue, so the result does not
    // depend on which finishes last.
    int splits;             // 1: no split
    int kb_per_split;
    float* kpart;           // [splits][tiles][2 CTAs][8 warps][4096] fp32
    int* kcount;            // [tiles][2][8] arrivals: zero before a launch, and again after it
    unsigned long long timeout_ns;   // limit of every pipeline wait (0: the default, 4 s)
    int test_no_loads;      // test hook: the TMA producer issues nothing, so the first wait of the
                            // MMA issuer runs out (nothing is in flight when the kernel gives up)
};

namespace tc {
// GEMM kernels: one SM per 128 x 256 tile; one CTA pair per 256 x 256
// tile, with two K steps per pipeline stage where the shape allows (else
// one) or always one (kGemmPairStep1).
enum GemmKind { kGemmSingle = 0, kGemmPair = 1, kGemmPairStep1 = 3 };
cudaError_t launch_ns_gemm(GemmParams p, const void* a_op, int a_ld, const void* b_op, int b_ld, int kind,
                           cudaStream_t st, const char** why);
// CTA pairs of the pair kernel that fit on the device at once
int pair_cluster_capacity();
int tiles_per_matrix(int mode, int M, int N);
int pair_tiles_per_matrix(int mode, int M, int N);
// K ranges a pair-kernel Gram launch of `tiles` tiles with K = `K` is split
// into, and the workspace it needs (partials and arrival counters).
int gram_splits(long long tiles, int K);
constexpr size_t kSplitPartialBytesPerTile = 2 * 8 * 4096 * sizeof(float);
constexpr size_t kSplitCountBytesPerTile = 2 * 8 * sizeof(int);
// ||U||^2 partials one apply tile writes: one per epilogue warp (8 per CTA,
// two CTAs per tile in the pair kernel).
constexpr int kUPartsPerTile1 = 8, kUPartsPerTilePair = 16;
}  // namespace tc

// The whole step of matrices with both sides <= 256 in one on-chip kernel
// per CTA pair (ns_small.cu): MuonH (muon = false, r0 read) or plain Muon.
struct SmallStepArgs {
    float lr, beta, eps, wdecay;   // wdecay: plain Muon's 1 - lr*weight_decay
    const float* coeffs;           // host array {a, b, c}
    int ns_steps;
    bool muon, nesterov;
    bool grad_bf16;                // gradients are bf16 bit patterns
    int scale_mode;                // UpdateScale
    const float* r0;               // device, indexed by caller position (MuonH)
    uint32_t* status;
};
cudaError_t launch_small_step(const muonh_matrix_t* mats, const int* idx, int n, const SmallStepArgs& a,
                              cudaStream_t st, int* launches);

// fp32 CUDA-core GEMM for the accuracy-check mode: out = epilogue(A B) with
// A M x K and B K x N.  a stored [m][k] (or [k][m] with a_km), b stored
// [n][k] (or [k][n] with b_kn).  Epilogues:
//   GRAM : out = scale*(A B)           (full s x s, ld_s)
//   POLY : out = cb*addend + cc*(A B)
//   APPLY: out = scale*(ca*addend + A B)
struct SimtParams {
    int mode;
    int a_km, b_kn;
    int G, M, N, K;
    const float* a; int lda; long long a_bstride;
    const float* b; int ldb; long long b_bstride;
    const float* addend; int ld_add; long long add_bstride;  // POLY: A; APPLY: X
    float* out; int ldo; long long out_bstride;
    const float* scale;
    float ca, cb, cc;
};
cudaError_t launch_simt_gemm(const SimtParams& p, cudaStream_t st);

}  // namespace muonh
