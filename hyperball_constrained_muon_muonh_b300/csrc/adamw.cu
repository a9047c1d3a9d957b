// AdamW for the parameters outside the MuonH group (Puro-2B model card,
// section "Training": AdamW with weight decay 0.1 for the remaining
// parameters).  Decoupled weight decay and bias-corrected moments:
//
//   m <- beta1*m + (1 - beta1)*g
//   v <- beta2*v + (1 - beta2)*g^2
//   p <- (1 - lr*wd)*p - (lr / (1 - beta1^t)) * m / (sqrt(v) / sqrt(1 - beta2^t) + eps)
//
// One HBM-bound pass over a list of tensors: read p, g, m, v and write p, m,
// v (28 bytes per element, 30 with the bf16 copy).  A chunk is about 64 K
// elements of one tensor; one CTA per chunk, float4 accesses.

#include <algorithm>
#include <cmath>
#include <string>
#include <vector>

#include "common.cuh"

namespace muonh {

int report_error(int code, const char* msg);

namespace {

constexpr int kAdamThreads = 256;
constexpr int kAdamChunk = 65536;          // elements per chunk (a multiple of 4)
constexpr int kMaxAdamPerLaunch = 560;

struct AdamDesc {
    float* p;
    uint16_t* pb;
    const float* g;
    float* m;
    float* v;
    long long numel;
    int chunk0;
    int pad_;
};
static_assert(sizeof(AdamDesc) == 56, "AdamDesc layout");

struct AdamBatch {
    int n;
    int chunk_begin, chunk_end;
    int pad_;
    AdamDesc d[kMaxAdamPerLaunch];
};
static_assert(sizeof(AdamBatch) <= 32000, "AdamW descriptor batch exceeds kernel parameter space");

struct AdamScalars {
    float beta1, beta2, omb1, omb2;   // omb = 1 - beta
    float step_size;                   // lr / (1 - beta1^t)
    float inv_sqrt_bc2;                // 1 / sqrt(1 - beta2^t)
    float eps, decay;                  // decay = 1 - lr*wd
};

__device__ __forceinline__ int find_tensor(const AdamBatch& b, int chunk) {
    int lo = 0, hi = b.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (b.d[mid].chunk0 <= chunk) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float adam_one(float& p, float g, float& m, float& v, const AdamScalars& s) {
    m = fmaf(s.beta1, m, s.omb1 * g);
    v = fmaf(s.beta2, v, s.omb2 * (g * g));
    const float denom = sqrtf(v) * s.inv_sqrt_bc2 + s.eps;
    p = fmaf(-s.step_size, m / denom, p * s.decay);
    return p;
}

__global__ void __launch_bounds__(kAdamThreads)
adamw_kernel(const __grid_constant__ AdamBatch b, const AdamScalars s) {
    const int chunk = b.chunk_begin + blockIdx.x;
    const AdamDesc& D = b.d[find_tensor(b, chunk)];
    const long long e0 = (long long)(chunk - D.chunk0) * kAdamChunk;
    const long long e1 = min(D.numel, e0 + kAdamChunk);
    // float4 body (e0 is a multiple of 4 and the pointers are 16-byte aligned), scalar tail
    const long long v1 = e0 + ((e1 - e0) & ~3ll);
    for (long long e = e0 + 4 * (long long)threadIdx.x; e < v1; e += 4 * kAdamThreads) {
        float4 p = *reinterpret_cast<const float4*>(D.p + e);
        const float4 g = __ldcs(reinterpret_cast<const float4*>(D.g + e));
        float4 m = *reinterpret_cast<const float4*>(D.m + e);
        float4 v = *reinterpret_cast<const float4*>(D.v + e);
        adam_one(p.x, g.x, m.x, v.x, s);
        adam_one(p.y, g.y, m.y, v.y, s);
        adam_one(p.z, g.z, m.z, v.z, s);
        adam_one(p.w, g.w, m.w, v.w, s);
        *reinterpret_cast<float4*>(D.p + e) = p;
        *reinterpret_cast<float4*>(D.m + e) = m;
        *reinterpret_cast<float4*>(D.v + e) = v;
        if (D.pb) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(p.x, p.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(p.z, p.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t*>(&lo);
            u.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(D.pb + e) = u;
        }
    }
    for (long long e = v1 + threadIdx.x; e < e1; e += kAdamThreads) {
        float p = D.p[e], m = D.m[e], v = D.v[e];
        adam_one(p, D.g[e], m, v, s);
        D.p[e] = p;
        D.m[e] = m;
        D.v[e] = v;
        if (D.pb) D.pb[e] = bf16_bits(p);
    }
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Launches over all tensors, kMaxAdamPerLaunch per launch.  Returns a
// MUONH_* code; `launches` counts the kernels launched.
int adamw_launch(const adamw_param_t* params, int n, int step, float lr, float beta1, float beta2, float eps,
                 float weight_decay, cudaStream_t st, int* launches, double* bytes) {
    *launches = 0;
    *bytes = 0;
    if (!params) return report_error(MUONH_ERR_INVALID_ARG, "params is NULL");
    if (n <= 0 || n > (1 << 22)) return report_error(MUONH_ERR_INVALID_ARG, "n must be in [1, 4194304]");
    if (step < 1) return report_error(MUONH_ERR_INVALID_ARG, "step is 1-based and must be >= 1");
    if (!std::isfinite(lr) || !std::isfinite(weight_decay) || !std::isfinite(eps) || eps < 0.f)
        return report_error(MUONH_ERR_INVALID_ARG, "lr and weight_decay must be finite, eps finite and >= 0");
    if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f))
        return report_error(MUONH_ERR_INVALID_ARG, "beta1 and beta2 must be in [0, 1)");
    for (int i = 0; i < n; ++i) {
        const adamw_param_t& a = params[i];
        if (a.numel < 1 || a.numel > (1ll << 40))
            return report_error(MUONH_ERR_INVALID_ARG, ("tensor " + std::to_string(i) + ": numel out of range").c_str());
        if (!a.p || !a.grad || !a.exp_avg || !a.exp_avg_sq || !aligned16(a.p) || !aligned16(a.grad) ||
            !aligned16(a.exp_avg) || !aligned16(a.exp_avg_sq) || (a.p_bf16 && !aligned16(a.p_bf16)))
            return report_error(MUONH_ERR_INVALID_ARG,
                                ("tensor " + std::to_string(i) + ": pointer NULL or not 16-byte aligned").c_str());
    }
    AdamScalars s;
    s.beta1 = beta1;
    s.beta2 = beta2;
    s.omb1 = 1.f - beta1;
    s.omb2 = 1.f - beta2;
    const double bc1 = 1.0 - std::pow((double)beta1, (double)step);
    const double bc2 = 1.0 - std::pow((double)beta2, (double)step);
    s.step_size = (float)((double)lr / bc1);
    s.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
    s.eps = eps;
    s.decay = 1.f - lr * weight_decay;

    std::vector<AdamBatch> batches;
    for (int b0 = 0; b0 < n; b0 += kMaxAdamPerLaunch) {
        batches.emplace_back();
        AdamBatch& B = batches.back();
        B.n = std::min(kMaxAdamPerLaunch, n - b0);
        B.pad_ = 0;
        long long chunk = 0;
        for (int k = 0; k < B.n; ++k) {
            const adamw_param_t& a = params[b0 + k];
            AdamDesc& D = B.d[k];
            D.p = a.p;
            D.pb = a.p_bf16;
            D.g = a.grad;
            D.m = a.exp_avg;
            D.v = a.exp_avg_sq;
            D.numel = a.numel;
            D.chunk0 = (int)chunk;
            D.pad_ = 0;
            chunk += (a.numel + kAdamChunk - 1) / kAdamChunk;
            *bytes += (double)a.numel * (28 + (a.p_bf16 ? 2 : 0));
        }
        if (chunk > (1ll << 30)) return report_error(MUONH_ERR_UNSUPPORTED, "too many elements in one call");
        B.chunk_begin = 0;
        B.chunk_end = (int)chunk;
    }
    for (const AdamBatch& B : batches) {
        adamw_kernel<<<B.chunk_end - B.chunk_begin, kAdamThreads, 0, st>>>(B, s);
        ++*launches;
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return report_error(MUONH_ERR_CUDA, cudaGetErrorString(e));
    }
    return MUONH_OK;
}

}  // namespace muonh
