// Internal definitions shared by the CUDA translation units of libmuonh.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "../../include/muonh.h"

namespace muonh {

// ---- per-matrix record handed to the elementwise kernels by value ----------
// W-orientation pointers plus where the matrix's Newton-Schulz state lives in
// the workspace (X orientation: s x l, row stride ld).
struct MatDesc {
    float* w;             // fp32 master weight, rows x cols
    uint16_t* wb;         // bf16 copy or nullptr
    const float* g;       // gradient
    float* m;             // momentum
    float* xs;            // fp32 NS state X (rows x ld, the matrix's own orientation)
    __nv_bfloat16* xo;    // bf16 NS operand X (rows x ld)
    int rows, cols;
    int ld;               // row stride of xs / xo, elements
    int chunk0;           // first chunk index of this matrix
    int user_index;       // position in the caller's list (indexes r0)
    int part0;            // first ||U||^2 partial written by the last apply GEMM
    int npart;            // number of those partials
    int fused;            // kFused* bits: how this matrix meets the Newton-Schulz GEMMs
};

// MatDesc::fused bits.
//   kFusedIn   the first apply GEMM reads X from the momentum (or input)
//              itself, so the momentum kernel writes no fp32 copy of X
//   kFusedOut  the last apply GEMM writes U = W - lr*O and the partials of
//              ||U||^2 (part0, npart), so the hyperball step only rescales
//   kFusedOutW the last apply GEMM of a plain Muon step writes the new
//              weight (1 - lr*wd)*W - lr*O and its bf16 copy itself
//   kFusedAll  the whole step runs in the small-matrix kernel (both sides
//              <= 256): every other kernel of the step skips the matrix
constexpr int kFusedIn = 1, kFusedOut = 2, kFusedOutW = 4, kFusedAll = 8;
static_assert(sizeof(MatDesc) == 80, "MatDesc layout");

// Largest descriptor batch one launch carries in its parameter space
// (sm_90+ kernels take up to 32764 bytes of parameters).
constexpr int kMaxDescPerLaunch = 396;

// Where the Newton-Schulz apply epilogue finds a matrix's own buffers (row-
// major, row stride = cols; the state X has the matrix's own orientation).
// Written by the momentum kernel into the workspace, one record per
// bucket-order position.
//   src: the unscaled Newton-Schulz input (the momentum M, or the input of a
//        standalone orthogonalisation), read by the first apply in place of
//        an fp32 copy of X
//   w:   the master weight, read by the last apply of a MuonH step (and
//        written by the last apply of a plain Muon step)
//   wb:  the bf16 weight copy (or null), written by the last apply of a
//        plain Muon step
struct NsIO {
    const float* src;
    float* w;
    uint16_t* wb;
};
static_assert(sizeof(NsIO) == 24, "NsIO layout");

struct DescBatch {
    int n;                // matrices in this batch
    int first;            // global (bucket-order) index of d[0]
    int chunk_begin;      // first chunk of this batch
    int chunk_end;        // one past the last chunk of this batch
    int bucket;           // plan bucket of every matrix in this batch (host side)
    MatDesc d[kMaxDescPerLaunch];
};
static_assert(sizeof(DescBatch) <= 32000, "descriptor batch exceeds kernel parameter space");

// Rows per chunk: a chunk is rows [r, r + chunk_rows) of one matrix, about
// kChunkElems elements.  Every matrix keeps its own orientation throughout
// (the Newton-Schulz state of a tall matrix is tall too), so the HBM-bound
// kernels stream each matrix row-major.
constexpr int kChunkElems = 65536;

__host__ __device__ inline int chunk_rows_for(int rows, int cols) {
    (void)rows;
    int cr = kChunkElems / (cols > 0 ? cols : 1);
    return cr < 1 ? 1 : cr;
}

__host__ __device__ inline int chunks_for(int rows, int cols) {
    int cr = chunk_rows_for(rows, cols);
    return (rows + cr - 1) / cr;
}

// Update scale of a rows x cols matrix (MUONH_FLAG_SCALE_*), in float, the
// same on host and device (IEEE division and square root).
enum UpdateScale { kScaleNone = 0, kScaleShape = 1, kScaleRms = 2 };

__host__ __device__ inline float update_scale(int rows, int cols, int mode) {
    if (mode == kScaleShape) return sqrtf(fmaxf(1.f, (float)rows / (float)cols));
    if (mode == kScaleRms) return 0.2f * sqrtf((float)(rows > cols ? rows : cols));
    return 1.f;
}

// Per-matrix scalars in the workspace, indexed by bucket-order position.
struct Scalars {
    double* nu2;          // ||M||_F^2
    double* rho2;         // ||W - lr*O||_F^2
    float* inv_nu;        // 1 / (||M||_F + eps)
    float* inv_nu2;       // inv_nu^2
    float* factor;        // r0 / ||W - lr*O||_F
    float* oscale;        // factor on X_state that gives O: the update scale, times
                          // inv_nu when no Newton-Schulz iteration ran
    uint32_t* flags;      // per-matrix status bits
};

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bits) { atomicOr(status, bits); }

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Deterministic block sum (fixed tree); result valid in thread 0.
template <int THREADS>
__device__ __forceinline__ double block_sum(double v, double* smem) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    double r = 0.0;
    if (warp == 0) {
        r = lane < THREADS / 32 ? smem[lane] : 0.0;
        r = warp_sum(r);
    }
    __syncthreads();
    return r;
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

}  // namespace muonh
