// Internal interface of the Newton-Schulz GEMM kernels (tcgen05 and fp32).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace muonh {

enum NsMode { NS_GRAM = 0, NS_POLY = 1, NS_APPLY = 2 };

// One launch = one Newton-Schulz stage over a bucket of G matrices, all
// s x l (ld_x = row stride of X buffers, ld_s = row stride of s x s buffers).
//   GRAM : M = N = s, K = l.  a_f32 <- scale*X X^T, sym_bf16 <- bf16 of it
//   POLY : M = N = K = s.     sym_bf16 <- cb*a_f32 + cc*(A A)
//   APPLY: M = s, N = l, K = s.  x_state <- scale*(ca*x_state + B X);
//          x_op_out <- bf16(x_state) unless null
struct GemmParams {
    int mode;
    int G, M, N, K;
    int tiles_m, tiles_n, tiles_per_mat;   // filled by the launcher
    int ld_x, ld_s;
    float* x_state;
    __nv_bfloat16* x_op_out;
    float* a_f32;
    __nv_bfloat16* sym_bf16;
    const float* scale;     // per-matrix factor (bucket-local index) or null
    float ca, cb, cc;
    uint32_t* status;       // device status word
};

namespace tc {
cudaError_t launch_ns_gemm(GemmParams p, const void* a_op, int a_ld, const void* b_op, int b_ld, bool pair,
                           cudaStream_t st, const char** why);
int tiles_per_matrix(int mode, int M, int N);
}  // namespace tc

// fp32 CUDA-core GEMM for the accuracy-check mode.  Operands fp32:
//   GRAM : a = X [G][s][ld_x]                 -> out = scale*X X^T (full s x s, ld_s)
//   POLY : a = A [G][s][ld_s]                 -> out = cb*A + cc*A A
//   APPLY: a = B [G][s][ld_s], x = X [G][s][ld_x] -> out = scale*(ca*X + B X) (ld_x)
struct SimtParams {
    int mode;
    int G, M, N, K;
    const float* a; int lda; long long a_bstride;
    const float* b; int ldb; long long b_bstride;   // GRAM/POLY: [N][K] rows; APPLY: [K][N] rows
    const float* addend; int ld_add; long long add_bstride;  // POLY: A; APPLY: X
    float* out; int ldo; long long out_bstride;
    const float* scale;
    float ca, cb, cc;
};
cudaError_t launch_simt_gemm(const SimtParams& p, cudaStream_t st);

}  // namespace muonh
