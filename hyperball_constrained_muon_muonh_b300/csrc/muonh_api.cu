// C ABI of libmuonh: argument checks, the shape planner, workspace layout and
// the launch sequence of one MuonH step.
//
// Step (Puro-2B digest, section "The load-bearing tricks aren't in the
// abstract"; model card, section "Training"): momentum, Newton-Schulz
// orthogonalisation of the momentum, then retraction of W - lr*O onto the
// sphere of radius r0 = ||W0||_F.
//
// Planner: matrices are grouped into buckets of equal shape (R, C).  Each
// matrix keeps its own orientation throughout: a tall matrix (R > C) is
// orthogonalised through its Gram X^T X and X <- a X + X B rather than
// through a transposed copy.  Each bucket's Newton-Schulz state lives
// contiguously in the workspace ([G][R][ld_x] and [G][s][ld_s] tensors), so
// one GEMM launch covers the whole bucket through 3-D TMA descriptors.

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "ns_gemm.h"
#include "../../include/muonh_test.h"

namespace muonh {

cudaError_t launch_momentum(const DescBatch& b, float beta, double* partials, NsIO* io, bool nesterov,
                            bool grad_bf16, cudaStream_t st);
cudaError_t launch_momentum_finalize(const DescBatch& b, const double* partials, const Scalars& sc, float eps,
                                     int scale_mode, bool no_iterations, cudaStream_t st);
cudaError_t launch_hyperball_norm(const DescBatch& b, float lr, double* partials, const float* o_scale,
                                  cudaStream_t st);
cudaError_t launch_hyperball_finalize(const DescBatch& b, const double* partials, const double* upart,
                                      const Scalars& sc, const float* r0, cudaStream_t st);
cudaError_t launch_hyperball_finish(const DescBatch& b, float lr, const Scalars& sc, const float* o_scale,
                                    cudaStream_t st);
cudaError_t launch_muon_finish(const DescBatch& b, float lr, float wdecay, const Scalars& sc, const float* o_scale,
                               cudaStream_t st);
cudaError_t launch_emit(const DescBatch& b, const float* o_scale, bool out_bf16, cudaStream_t st);
cudaError_t launch_capture_norms(const DescBatch& b, float* r0, cudaStream_t st);
cudaError_t status_word(uint32_t** ptr);
int adamw_launch(const adamw_param_t* params, int n, int step, float lr, float beta1, float beta2, float eps,
                 float weight_decay, cudaStream_t st, int* launches, double* bytes);


namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

int cuda_fail(cudaError_t e, const char* where) {
    g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
    return MUONH_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- tracing: per-kernel CUDA-event timing ---------------------------------
// ns_apply_in / _out / _in_out: the apply launches that read X from the
// matrices' own input, write U = W - lr*O, or both (first / last iteration);
// ns_apply_outw / _in_outw: the last apply of a plain Muon step, which writes
// the new weight
enum Kind { K_MOMENTUM, K_MOM_FIN, K_GRAM, K_POLY, K_APPLY, K_APPLY_IN, K_APPLY_OUT, K_APPLY_IN_OUT,
            K_APPLY_OUTW, K_APPLY_IN_OUTW, K_HB_NORM, K_HB_FIN, K_HB_APPLY, K_HB_SCALE, K_MUON_FIN, K_EMIT,
            K_CAPTURE, K_SIMT_GRAM, K_SIMT_POLY, K_SIMT_APPLY, K_ADAMW, K_SMALL, K_NS_BUSY, K_COUNT };
const char* const kKindName[K_COUNT] = {"momentum", "momentum_finalize", "ns_gram", "ns_poly", "ns_apply",
                                        "ns_apply_in", "ns_apply_out", "ns_apply_in_out", "ns_apply_outw",
                                        "ns_apply_in_outw", "hyperball_norm", "hyperball_finalize",
                                        "hyperball_apply", "hyperball_scale", "muon_finish", "emit",
                                        "capture_norms", "fp32_gram", "fp32_poly", "fp32_apply", "adamw",
                                        "small_step", "ns_busy"};
// A kind's ms is the length of the union of its launches' event intervals,
// so launches that overlap on the side streams are not counted twice.
// ns_busy: all Newton-Schulz GEMM launches (tensor-core and fp32) together.
inline bool is_ns_kind(int k) {
    return (k >= K_GRAM && k <= K_APPLY_IN_OUTW) || (k >= K_SIMT_GRAM && k <= K_SIMT_APPLY);
}

int apply_kind(int variant) {
    switch (variant) {
        case NS_IN_SRC: return K_APPLY_IN;
        case NS_OUT_U: return K_APPLY_OUT;
        case NS_IN_SRC | NS_OUT_U: return K_APPLY_IN_OUT;
        case NS_OUT_W: return K_APPLY_OUTW;
        case NS_IN_SRC | NS_OUT_W: return K_APPLY_IN_OUTW;
        default: return K_APPLY;
    }
}

std::atomic<long long> g_launches{0};

struct Pending {
    int kind;
    cudaEvent_t a, b;
    double flops, bytes;
};

struct Profiler {
    std::mutex mu;
    bool on = false;
    std::vector<Pending> pending;
    std::vector<cudaEvent_t> pool;
    long long launches[K_COUNT] = {};
    double ms[K_COUNT] = {}, flops[K_COUNT] = {}, bytes[K_COUNT] = {};
    cudaEvent_t get() {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
};
Profiler g_prof;

// Brackets one launch: records the start event (when tracing) on construction
// and the end event plus the work on done().
struct Trace {
    int kind;
    cudaStream_t st;
    cudaEvent_t a = nullptr;
    Trace(int k, cudaStream_t s) : kind(k), st(s) {
        ++g_launches;
        std::lock_guard<std::mutex> lk(g_prof.mu);
        if (g_prof.on) {
            a = g_prof.get();
            cudaEventRecord(a, st);
        }
    }
    cudaError_t done(cudaError_t e, double flops, double bytes) {
        if (!a) return e;
        std::lock_guard<std::mutex> lk(g_prof.mu);
        cudaEvent_t b = g_prof.get();
        cudaEventRecord(b, st);
        g_prof.pending.push_back({kind, a, b, flops, bytes});
        return e;
    }
};
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Matrices whose short side is at most this run Newton-Schulz on fp32 CUDA
// cores.  With few singular values the bf16 rounding of the tensor-core
// operands is not averaged out (B ~ -2.7 against a per-step result ~0.7 is a
// near-cancellation): emulating the bf16 path in NumPy on Gaussian inputs
// gives a median error in O of 3.2 % at 36 x 100, 2.7 % at 64 x 200 and
// 1.9 % at 96 x 256 (14 % worst case on rank-1 inputs), against 1e-6 in fp32.
// These matrices are small, so fp32 costs little.
constexpr int kSmallSide = 80;

// Matrices with both sides at most this (and a short side above kSmallSide)
// can take the whole step in one on-chip kernel (csrc/ns_small.cu).
constexpr int kSmallStepSide = 256;

struct Bucket {
    int R, C;             // matrix shape (rows, cols)
    int s, l, G;          // short side, long side, matrices
    bool tall;            // R > C
    bool small;           // s <= kSmallSide: Newton-Schulz on fp32 CUDA cores
    bool fusable;         // tensor-core bucket with C % 4 == 0: the apply GEMM can read and write the
                          // matrices' own buffers
    int first;            // bucket-order index of its first matrix
    int ld_x, ld_s;
    size_t off_xs, off_xo;                    // byte offsets in the workspace
    size_t off_xlo;                           // bf16 lo part of the two-part Newton-Schulz state
    size_t off_af, off_aop, off_bop;          // this bucket's slice of its s-group's s x s buffers
    size_t off_bf32;                          // fp32 check mode: its slice of the group's fp32 B
    int sgroup;                               // index of its s-group
    long long upart0;                         // first ||U||^2 partial of this bucket (index into the
                                              // plan's partial region; written by the last apply GEMM)
    int tiles1, tiles2;                       // apply tiles per matrix: 1-SM and pair kernel
    int gsplits = 1;                          // K ranges of its pair-kernel Gram (tc::gram_splits)
    size_t off_kpart = 0, off_kcount = 0;     // split-K Gram partials and arrival counters
    size_t x_elems() const { return (size_t)G * R * ld_x; }
};

// Buckets with the same short side s share one set of s x s buffers (Gram
// A fp32, A_op and B_op bf16, [G][s][ld_s] each), so one polynomial launch
// covers all of them.
struct SGroup {
    int s, ld_s, G;
    bool small_step;      // every matrix has both sides in (kSmallSide, kSmallStepSide]: the whole
                          // step can run in the small-matrix kernel
    int b_begin, b_end;   // its buckets, contiguous in Plan::buckets
    size_t off_af, off_aop, off_bop;
    size_t elems() const { return (size_t)G * s * ld_s; }
};

struct Plan {
    int n = 0;
    std::vector<Bucket> buckets;
    std::vector<SGroup> sgroups;
    std::vector<int> order;       // bucket-order position -> caller index
    std::vector<int> slot;        // bucket-order position -> slot in its bucket
    std::vector<int> bucket_of;   // bucket-order position -> bucket index
    std::vector<int> chunk0;      // bucket-order position -> first chunk
    int total_chunks = 0;
    size_t off_nu2, off_rho2, off_inv, off_inv2, off_fac, off_oscale, off_flags, off_partials, off_io, off_upart;
    long long n_upart = 0;        // ||U||^2 partials of the last apply GEMM, all buckets
    size_t bytes = 0;
};

std::mutex g_plan_mu;
std::map<std::string, Plan> g_plans;

std::string plan_key(const int64_t* rc, int n, uint32_t flags) {
    std::string k;
    k.reserve(16 * n + 8);
    k.append(reinterpret_cast<const char*>(&flags), sizeof flags);
    k.append(reinterpret_cast<const char*>(rc), sizeof(int64_t) * 2 * n);
    return k;
}

// Buckets whose pair-kernel Gram has few tiles get split-K partial buffers
// (tc::gram_splits).
Plan build_plan(const int64_t* rc, int n, uint32_t flags) {
    (void)flags;
    Plan P;
    P.n = n;
    std::map<std::pair<int, int>, std::vector<int>> groups;  // (rows, cols) -> caller indices
    for (int i = 0; i < n; ++i) groups[{(int)rc[2 * i], (int)rc[2 * i + 1]}].push_back(i);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        off = align_up(off, 256);
        const size_t o = off;
        off += bytes;
        return o;
    };
    P.off_nu2 = take(sizeof(double) * n);
    P.off_rho2 = take(sizeof(double) * n);
    P.off_inv = take(sizeof(float) * n);
    P.off_inv2 = take(sizeof(float) * n);
    P.off_fac = take(sizeof(float) * n);
    P.off_oscale = take(sizeof(float) * n);
    P.off_flags = take(sizeof(uint32_t) * n);
    P.off_io = take(sizeof(NsIO) * n);
    // s-groups with the most Newton-Schulz work first, and within one the
    // largest buckets first: their GEMMs are the longest launches
    struct Shape { int R, C; std::vector<int> idx; double work; };
    std::map<int, std::vector<Shape>> by_s;
    for (auto& kv : groups) {
        const int R = kv.first.first, C = kv.first.second, sd = std::min(R, C), ld = std::max(R, C);
        by_s[sd].push_back({R, C, kv.second, (double)sd * sd * ld * kv.second.size()});
    }
    std::vector<std::vector<Shape>> sl_list;
    for (auto& kv : by_s) {
        std::stable_sort(kv.second.begin(), kv.second.end(), [](const Shape& a, const Shape& b) { return a.work > b.work; });
        sl_list.push_back(kv.second);
    }
    std::stable_sort(sl_list.begin(), sl_list.end(), [](const std::vector<Shape>& a, const std::vector<Shape>& b) {
        double wa = 0, wb = 0;
        for (auto& x : a) wa += x.work;
        for (auto& x : b) wb += x.work;
        return wa > wb;
    });
    int chunk = 0;
    long long n_upart = 0;
    for (auto& shapes : sl_list) {
        SGroup S;
        S.s = std::min(shapes[0].R, shapes[0].C);
        S.ld_s = (int)align_up(S.s, 8);
        S.G = 0;
        S.b_begin = (int)P.buckets.size();
        S.small_step = S.s > kSmallSide;
        for (auto& sh : shapes) {
            S.G += (int)sh.idx.size();
            if (sh.R > kSmallStepSide || sh.C > kSmallStepSide) S.small_step = false;
        }
        // the fp32 Gram A: for Newton-Schulz on CUDA cores only (the fp32
        // check mode, short sides <= kSmallSide); the tensor-core path keeps A
        // in bf16 (A_op) alone
        const bool simt_group = (flags & MUONH_FLAG_FP32_CHECK) || S.s <= kSmallSide;
        S.off_af = simt_group ? take(sizeof(float) * S.elems()) : 0;
        S.off_aop = take(sizeof(__nv_bfloat16) * S.elems());
        // fp32 check mode keeps an fp32 B at off_aop, spanning A_op and B_op
        S.off_bop = take(sizeof(__nv_bfloat16) * S.elems());
        int g_in_group = 0;
        for (auto& sh : shapes) {
            Bucket B;
            B.R = sh.R;
            B.C = sh.C;
            B.s = S.s;
            B.l = std::max(B.R, B.C);
            B.tall = B.R > B.C;
            B.small = B.s <= kSmallSide;
            B.fusable = !B.small && (B.C & 3) == 0;
            B.G = (int)sh.idx.size();
            B.first = (int)P.order.size();
            B.ld_x = (int)align_up(B.C, 8);
            B.ld_s = S.ld_s;
            B.off_xs = take(sizeof(float) * B.x_elems());
            B.off_xo = take(2 * sizeof(__nv_bfloat16) * B.x_elems());    // two bf16 buffers (ping-pong)
            B.off_xlo = take(sizeof(__nv_bfloat16) * B.x_elems());
            const size_t so = (size_t)g_in_group * S.s * S.ld_s;
            B.off_af = S.off_af + sizeof(float) * so;
            B.off_aop = S.off_aop + sizeof(__nv_bfloat16) * so;
            B.off_bop = S.off_bop + sizeof(__nv_bfloat16) * so;
            B.off_bf32 = S.off_aop + sizeof(float) * so;
            B.sgroup = (int)P.sgroups.size();
            g_in_group += B.G;
            B.tiles1 = tc::tiles_per_matrix(NS_APPLY, B.R, B.C);
            B.tiles2 = tc::pair_tiles_per_matrix(NS_APPLY, B.R, B.C);
            // split K only for a lone bucket (a standalone orthogonalisation,
            // or a step over one shape) with few Gram tiles: beside other
            // buckets on the side streams, the SMs it would fill are busy anyway
            if (!B.small && groups.size() == 1) {
                const long long gtiles = (long long)B.G * tc::pair_tiles_per_matrix(NS_GRAM, B.s, B.s);
                B.gsplits = tc::gram_splits(gtiles, B.l);
                if (B.gsplits > 1) {
                    B.off_kpart = take(tc::kSplitPartialBytesPerTile * (size_t)gtiles * B.gsplits);
                    B.off_kcount = take(tc::kSplitCountBytesPerTile * (size_t)gtiles);
                }
            }
            B.upart0 = n_upart;
            n_upart += (long long)B.G * std::max((long long)B.tiles1 * tc::kUPartsPerTile1,
                                                 (long long)B.tiles2 * tc::kUPartsPerTilePair);
            int sl = 0;
            for (int i : sh.idx) {
                P.order.push_back(i);
                P.slot.push_back(sl++);
                P.bucket_of.push_back((int)P.buckets.size());
                P.chunk0.push_back(chunk);
                chunk += chunks_for((int)rc[2 * i], (int)rc[2 * i + 1]);
            }
            P.buckets.push_back(B);
        }
        S.b_end = (int)P.buckets.size();
        P.sgroups.push_back(S);
    }
    P.total_chunks = chunk;
    P.off_partials = take(sizeof(double) * std::max(chunk, 1));
    P.n_upart = n_upart;
    P.off_upart = take(sizeof(double) * (size_t)std::max(n_upart, 1LL));
    P.bytes = align_up(off, 256);
    return P;
}

const Plan& get_plan(const int64_t* rc, int n, uint32_t flags) {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    const std::string key = plan_key(rc, n, flags & MUONH_FLAG_FP32_CHECK);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) return it->second;
    if (g_plans.size() > 64) g_plans.clear();
    return g_plans.emplace(key, build_plan(rc, n, flags)).first->second;
}

int check_shapes(const muonh_matrix_t* mats, int n, std::vector<int64_t>& rc, bool need_state) {
    if (!mats) return fail(MUONH_ERR_INVALID_ARG, "mats is NULL");
    if (n <= 0 || n > (1 << 22)) return fail(MUONH_ERR_INVALID_ARG, "n must be in [1, 4194304]");
    rc.resize(2 * (size_t)n);
    for (int i = 0; i < n; ++i) {
        const muonh_matrix_t& m = mats[i];
        char buf[160];
        if (m.rows < 1 || m.cols < 1 || m.rows > MUONH_MAX_SIDE || m.cols > MUONH_MAX_SIDE) {
            snprintf(buf, sizeof buf, "matrix %d: rows/cols must be in [1, %d]", i, MUONH_MAX_SIDE);
            return fail(MUONH_ERR_INVALID_ARG, buf);
        }
        if (!m.w || !aligned16(m.w)) {
            snprintf(buf, sizeof buf, "matrix %d: w is NULL or not 16-byte aligned", i);
            return fail(MUONH_ERR_INVALID_ARG, buf);
        }
        if (need_state) {
            if (!m.grad || !aligned16(m.grad) || !m.mom || !aligned16(m.mom)) {
                snprintf(buf, sizeof buf, "matrix %d: grad/mom NULL or not 16-byte aligned", i);
                return fail(MUONH_ERR_INVALID_ARG, buf);
            }
            if (m.w_bf16 && !aligned16(m.w_bf16)) {
                snprintf(buf, sizeof buf, "matrix %d: w_bf16 not 16-byte aligned", i);
                return fail(MUONH_ERR_INVALID_ARG, buf);
            }
        }
        rc[2 * i] = m.rows;
        rc[2 * i + 1] = m.cols;
    }
    return MUONH_OK;
}

Scalars scalars_of(const Plan& P, uint8_t* ws) {
    Scalars sc;
    sc.nu2 = reinterpret_cast<double*>(ws + P.off_nu2);
    sc.rho2 = reinterpret_cast<double*>(ws + P.off_rho2);
    sc.inv_nu = reinterpret_cast<float*>(ws + P.off_inv);
    sc.inv_nu2 = reinterpret_cast<float*>(ws + P.off_inv2);
    sc.factor = reinterpret_cast<float*>(ws + P.off_fac);
    sc.oscale = reinterpret_cast<float*>(ws + P.off_oscale);
    sc.flags = reinterpret_cast<uint32_t*>(ws + P.off_flags);
    return sc;
}

// How the tensor-core Newton-Schulz path meets its neighbours, for the
// matrices of fusable buckets (row length a multiple of 4):
//   in   the first apply reads X from each matrix's own input (the
//        momentum kernel writes the NsIO table and no fp32 copy of X)
//   out  the last apply writes U = W - lr*O and its ||U||^2 partials
//   out_w the last apply writes Muon's new weight (1 - lr*wd)*W - lr*O
//   pair the partials' layout is the pair kernel's (else the 1-SM kernel's)
struct NsFuse {
    bool in = false;
    bool out = false;
    bool out_w = false;   // plain Muon: the last apply writes the new weight
    bool pair = true;
    bool check = false;   // fp32 check mode: every bucket on CUDA cores
    bool small = false;   // s-groups marked small_step take the whole step in the small-matrix kernel
    int scale_mode = kScaleNone;   // update scale of O (UpdateScale)
    float lr = 0.f;
    float wdecay = 1.f;   // out_w: 1 - lr*weight_decay
};

// Descriptor batches in bucket order.  With `x_in_alt`, the hyperball /
// emit view of X of every bucket that ran Newton-Schulz on CUDA cores (all
// of them in the fp32 check mode, else the small ones) points at the second
// fp32 buffer, where an odd number of those iterations leaves the result.
std::vector<DescBatch> make_batches(const Plan& P, const muonh_matrix_t* mats, uint8_t* ws, bool x_in_alt,
                                    bool with_momentum, const NsFuse& fuse = NsFuse()) {
    std::vector<DescBatch> out;
    const int n = P.n;
    // a batch never spans two buckets, so each bucket's elementwise passes
    // can go to that bucket's stream
    for (int b0 = 0; b0 < n;) {
        int len = 1;
        while (len < kMaxDescPerLaunch && b0 + len < n && P.bucket_of[b0 + len] == P.bucket_of[b0]) ++len;
        out.emplace_back();
        DescBatch& B = out.back();
        B.n = len;
        B.first = b0;
        B.bucket = P.bucket_of[b0];
        b0 += len;
        for (int k = 0; k < B.n; ++k) {
            const int p = B.first + k;
            const int u = P.order[p];
            const Bucket& bk = P.buckets[P.bucket_of[p]];
            const muonh_matrix_t& m = mats[u];
            MatDesc& D = B.d[k];
            D.w = m.w;
            D.wb = with_momentum ? m.w_bf16 : nullptr;
            D.g = with_momentum ? m.grad : m.w;
            D.m = with_momentum ? m.mom : nullptr;
            const size_t xoff = (size_t)P.slot[p] * bk.R * bk.ld_x;
            float* xs = reinterpret_cast<float*>(ws + bk.off_xs);
            float* x2 = reinterpret_cast<float*>(ws + bk.off_xo);
            D.xs = ((x_in_alt && (fuse.check || bk.small)) ? x2 : xs) + xoff;
            D.xo = reinterpret_cast<__nv_bfloat16*>(ws + bk.off_xo) + xoff;
            D.rows = (int)m.rows;
            D.cols = (int)m.cols;
            D.ld = bk.ld_x;
            D.chunk0 = P.chunk0[p];
            D.user_index = u;
            D.part0 = 0;
            D.npart = 0;
            D.fused = 0;
            if (fuse.small && P.sgroups[bk.sgroup].small_step) {
                D.fused = kFusedAll;
            } else if (bk.fusable) {
                if (fuse.in) D.fused |= kFusedIn;
                if (fuse.out_w) D.fused |= kFusedOutW;
                if (fuse.out) {
                    const int per = fuse.pair ? bk.tiles2 * tc::kUPartsPerTilePair : bk.tiles1 * tc::kUPartsPerTile1;
                    D.fused |= kFusedOut;
                    D.part0 = (int)(bk.upart0 + (long long)P.slot[p] * per);
                    D.npart = per;
                }
            }
        }
        B.chunk_begin = P.chunk0[B.first];
        B.chunk_end = (B.first + B.n < n) ? P.chunk0[B.first + B.n] : P.total_chunks;
    }
    return out;
}

double batch_elems(const DescBatch& b) {
    double e = 0;
    for (int k = 0; k < b.n; ++k) e += (double)b.d[k].rows * b.d[k].cols;
    return e;
}

struct Sync {
    bool on;
    cudaStream_t st;
    int check(cudaError_t e, const char* where) { return check_on(st, e, where); }
    int check_on(cudaStream_t s, cudaError_t e, const char* where) {
        if (e != cudaSuccess) return cuda_fail(e, where);
        if (on) {
            e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) return cuda_fail(e, where);
        }
        return MUONH_OK;
    }
};

// Side streams for Newton-Schulz.  The buckets of a step are independent
// until the polynomial of their s-group, and s-groups are independent
// throughout, so their launches go to up to kNsStreams streams (the
// caller's first): a launch's tail of partly filled waves overlaps the next
// bucket's launch instead of idling SMs.  Events fork the side streams from
// the caller's stream and join them back; events are handed out in order
// within a call, under a per-device lock so that concurrent calls cannot
// re-record an event another call has yet to wait on.
constexpr int kNsStreams = 4;
struct NsStreams {
    std::mutex mu;
    cudaStream_t side[kNsStreams - 1] = {};
    std::vector<cudaEvent_t> events;
    size_t next = 0;
    bool ready = false;
    cudaError_t init() {
        if (ready) return cudaSuccess;
        for (auto& st : side) {
            cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
            if (e != cudaSuccess) return e;
        }
        ready = true;
        return cudaSuccess;
    }
    cudaError_t event(cudaEvent_t* out) {
        if (next == events.size()) {
            cudaEvent_t e = nullptr;
            cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
            if (r != cudaSuccess) return r;
            events.push_back(e);
        }
        *out = events[next++];
        return cudaSuccess;
    }
};
NsStreams& ns_streams_for_device() {
    static std::mutex mu;
    static std::map<int, std::unique_ptr<NsStreams>> by_dev;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    auto& p = by_dev[dev];
    if (!p) p.reset(new NsStreams);
    return *p;
}
// `to` waits for the work enqueued so far on `from`
cudaError_t stream_after(NsStreams& ns, cudaStream_t to, cudaStream_t from) {
    if (to == from) return cudaSuccess;
    cudaEvent_t ev;
    cudaError_t e = ns.event(&ev);
    if (e == cudaSuccess) e = cudaEventRecord(ev, from);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
    return e;
}

// The stream of every bucket for one call.  Bucket k of the step (plan
// order, small-step groups left out) goes to stream k % kNsStreams, the
// caller's stream first.  open() forks the side streams from the caller's
// stream; close() (or the destructor, on an error path) joins them back.
struct Schedule {
    cudaStream_t st = nullptr;
    std::vector<cudaStream_t> bst;    // per bucket
    std::vector<cudaStream_t> used;   // used[0] = the caller's stream
    NsStreams* ns = nullptr;
    std::unique_lock<std::mutex> lock;
    bool joined = false;

    int open(const Plan& P, uint32_t flags, bool skip_small_groups, cudaStream_t caller) {
        st = caller;
        bst.assign(P.buckets.size(), caller);
        used.assign(1, caller);
        int active = 0;
        for (const SGroup& Q : P.sgroups)
            if (!(skip_small_groups && Q.small_step)) active += Q.b_end - Q.b_begin;
        if (active <= 1 || (flags & MUONH_FLAG_ONE_STREAM)) return MUONH_OK;
        ns = &ns_streams_for_device();
        lock = std::unique_lock<std::mutex>(ns->mu);
        ns->next = 0;
        cudaError_t e = ns->init();
        if (e != cudaSuccess) return cuda_fail(e, "side streams");
        int k = 0;
        for (const SGroup& Q : P.sgroups) {
            if (skip_small_groups && Q.small_step) continue;
            for (int b = Q.b_begin; b < Q.b_end; ++b, ++k) {
                const int slot = k % kNsStreams;
                bst[b] = slot == 0 ? caller : ns->side[slot - 1];
                if (std::find(used.begin(), used.end(), bst[b]) == used.end()) used.push_back(bst[b]);
            }
        }
        for (size_t u = 1; u < used.size(); ++u) {
            e = stream_after(*ns, used[u], caller);
            if (e != cudaSuccess) return cuda_fail(e, "fork of the side streams");
        }
        return MUONH_OK;
    }
    int close() {
        joined = true;
        if (!ns) return MUONH_OK;
        for (size_t u = 1; u < used.size(); ++u) {
            cudaError_t e = stream_after(*ns, st, used[u]);
            if (e != cudaSuccess) return cuda_fail(e, "join of the side streams");
        }
        return MUONH_OK;
    }
    ~Schedule() {
        if (!joined) (void)close();
    }
};

// Newton-Schulz over every bucket: per iteration and s-group, the Gram of
// each bucket, one polynomial launch for the group, the apply of each bucket.
// Returns MUONH_OK or an error code; *x_in_alt tells whether the buckets
// that ran on CUDA cores left their result in the second fp32 buffer.
int run_newton_schulz(const Plan& P, uint8_t* ws, const Scalars& sc, int ns_steps, const float* coeffs,
                      uint32_t flags, uint32_t* status, Sync& sy, bool* x_in_alt, const NsFuse& fuse,
                      const Schedule& S) {
    const bool check = (flags & MUONH_FLAG_FP32_CHECK) != 0;
    const int pair = (flags & MUONH_FLAG_GEMM_1SM)        ? tc::kGemmSingle
                     : (flags & MUONH_FLAG_GEMM_ONE_STEP) ? tc::kGemmPairStep1
                                                          : tc::kGemmPair;
    *x_in_alt = false;
    cudaStream_t cur = sy.st;   // stream of the launch being enqueued

    // ---- fp32 check mode (CUDA cores) ----
    auto simt_gram = [&](const Bucket& B, int it) {
        float* xs = reinterpret_cast<float*>(ws + B.off_xs);
        float* x2 = reinterpret_cast<float*>(ws + B.off_xo);
        float* xc = (it & 1) ? x2 : xs;
        const long long xstr = (long long)B.R * B.ld_x, sstr = (long long)B.s * B.ld_s;
        // X X^T (wide) reads X rows as [m][k]; X^T X (tall) reads them as [k][m]
        SimtParams g{};
        g.mode = NS_GRAM; g.G = B.G; g.M = B.s; g.N = B.s; g.K = B.l;
        g.a_km = B.tall; g.b_kn = B.tall;
        g.a = xc; g.lda = B.ld_x; g.a_bstride = xstr;
        g.b = xc; g.ldb = B.ld_x; g.b_bstride = xstr;
        g.out = reinterpret_cast<float*>(ws + B.off_af); g.ldo = B.ld_s; g.out_bstride = sstr;
        g.scale = it == 0 ? sc.inv_nu2 + B.first : nullptr;
        const double G = B.G, S = B.s, L = B.l;
        Trace tr(K_SIMT_GRAM, cur);
        return sy.check_on(cur, tr.done(launch_simt_gemm(g, cur), G * S * S * L, G * S * L * 4 + G * S * S * 4),
                        "fp32 Gram launch");
    };
    auto simt_poly = [&](const SGroup& Q) {
        const long long sstr = (long long)Q.s * Q.ld_s;
        float* af = reinterpret_cast<float*>(ws + Q.off_af);
        SimtParams q{};
        q.mode = NS_POLY; q.G = Q.G; q.M = Q.s; q.N = Q.s; q.K = Q.s;
        q.a = af; q.lda = Q.ld_s; q.a_bstride = sstr;
        q.b = af; q.ldb = Q.ld_s; q.b_bstride = sstr;
        q.addend = af; q.ld_add = Q.ld_s; q.add_bstride = sstr;
        q.out = reinterpret_cast<float*>(ws + Q.off_aop); q.ldo = Q.ld_s; q.out_bstride = sstr;
        q.cb = coeffs[1]; q.cc = coeffs[2];
        const double G = Q.G, S = Q.s;
        Trace tr(K_SIMT_POLY, cur);
        return sy.check_on(cur, tr.done(launch_simt_gemm(q, cur), G * S * S * S, G * S * S * 12), "fp32 polynomial launch");
    };
    auto simt_apply = [&](const Bucket& B, int it) {
        float* xs = reinterpret_cast<float*>(ws + B.off_xs);
        float* x2 = reinterpret_cast<float*>(ws + B.off_xo);
        float* xc = (it & 1) ? x2 : xs;
        float* xn = (it & 1) ? xs : x2;
        const long long xstr = (long long)B.R * B.ld_x, sstr = (long long)B.s * B.ld_s;
        float* bf = reinterpret_cast<float*>(ws + B.off_bf32);
        // B X (wide: A = B, B = X rows [k][n]) or X B (tall: A = X rows [m][k],
        // B = B, symmetric, read as [k][n])
        SimtParams a{};
        a.mode = NS_APPLY; a.G = B.G; a.M = B.R; a.N = B.C; a.K = B.s;
        a.b_kn = 1;
        if (B.tall) {
            a.a = xc; a.lda = B.ld_x; a.a_bstride = xstr;
            a.b = bf; a.ldb = B.ld_s; a.b_bstride = sstr;
        } else {
            a.a = bf; a.lda = B.ld_s; a.a_bstride = sstr;
            a.b = xc; a.ldb = B.ld_x; a.b_bstride = xstr;
        }
        a.addend = xc; a.ld_add = B.ld_x; a.add_bstride = xstr;
        a.out = xn; a.ldo = B.ld_x; a.out_bstride = xstr;
        a.scale = it == 0 ? sc.inv_nu + B.first : nullptr;
        a.ca = coeffs[0];
        const double G = B.G, S = B.s, L = B.l;
        Trace tr(K_SIMT_APPLY, cur);
        return sy.check_on(cur, tr.done(launch_simt_gemm(a, cur), 2 * G * S * S * L, G * S * S * 4 + G * S * L * 12),
                        "fp32 apply launch");
    };

    // ---- tensor cores ----
    auto x_ops = [&](const Bucket& B, int it, __nv_bfloat16** xc, __nv_bfloat16** xn) {
        __nv_bfloat16* xo0 = reinterpret_cast<__nv_bfloat16*>(ws + B.off_xo);
        __nv_bfloat16* xo1 = xo0 + B.x_elems();
        *xc = (it & 1) ? xo1 : xo0;
        *xn = (it & 1) ? xo0 : xo1;
    };
    auto tc_gram = [&](const Bucket& B, int it) {
        __nv_bfloat16 *xc, *xn;
        x_ops(B, it, &xc, &xn);
        const char* why = "";
        // K-major rows of X (wide) or MN-major columns (tall)
        GemmParams g{};
        g.mode = NS_GRAM; g.G = B.G; g.M = B.s; g.N = B.s; g.K = B.l;
        g.a_mn = g.b_mn = B.tall;
        g.ld_x = B.ld_x; g.ld_s = B.ld_s;
        g.sym_bf16 = reinterpret_cast<__nv_bfloat16*>(ws + B.off_aop);
        g.scale = it == 0 ? sc.inv_nu2 + B.first : nullptr;
        g.status = status;
        if (B.gsplits > 1 && pair != tc::kGemmSingle) {
            // split K: the arrival counters start at zero (each launch leaves them at zero)
            g.splits = B.gsplits;
            g.kpart = reinterpret_cast<float*>(ws + B.off_kpart);
            g.kcount = reinterpret_cast<int*>(ws + B.off_kcount);
            if (it == 0) {
                const size_t cnt_bytes =
                    tc::kSplitCountBytesPerTile * (size_t)B.G * tc::pair_tiles_per_matrix(NS_GRAM, B.s, B.s);
                const int r = sy.check_on(cur, cudaMemsetAsync(g.kcount, 0, cnt_bytes, cur), "split-K counters");
                if (r) return r;
            }
        }
        const double G = B.G, S = B.s, L = B.l;
        cudaError_t e;
        {
            Trace tr(K_GRAM, cur);
            e = tr.done(tc::launch_ns_gemm(g, xc, B.ld_x, xc, B.ld_x, pair, cur, &why), G * S * S * L,
                        G * S * L * 2 + G * S * S * 2);
        }
        return sy.check_on(cur, e, e == cudaErrorInvalidValue ? why : "tcgen05 Gram launch");
    };
    auto tc_poly = [&](const SGroup& Q) {
        const char* why = "";
        __nv_bfloat16* aop = reinterpret_cast<__nv_bfloat16*>(ws + Q.off_aop);
        GemmParams q{};
        q.mode = NS_POLY; q.G = Q.G; q.M = Q.s; q.N = Q.s; q.K = Q.s;
        q.ld_s = Q.ld_s;
        q.a_op = aop;
        q.sym_bf16 = reinterpret_cast<__nv_bfloat16*>(ws + Q.off_bop);
        q.cb = coeffs[1]; q.cc = coeffs[2];
        q.status = status;
        const double G = Q.G, S = Q.s;
        cudaError_t e;
        {
            Trace tr(K_POLY, cur);
            e = tr.done(tc::launch_ns_gemm(q, aop, Q.ld_s, aop, Q.ld_s, pair, cur, &why), G * S * S * S,
                        G * S * S * 6);
        }
        return sy.check_on(cur, e, e == cudaErrorInvalidValue ? why : "tcgen05 polynomial launch");
    };
    auto tc_apply = [&](const Bucket& B, int it) {
        __nv_bfloat16 *xc, *xn;
        x_ops(B, it, &xc, &xn);
        __nv_bfloat16* bop = reinterpret_cast<__nv_bfloat16*>(ws + B.off_bop);
        const char* why = "";
        // B X (wide: A = B_op, B = X_op MN-major) or X B (tall: A = X_op,
        // B = B_op, both K-major; B is symmetric)
        GemmParams a{};
        a.mode = NS_APPLY; a.G = B.G; a.M = B.R; a.N = B.C; a.K = B.s;
        a.b_mn = !B.tall;
        a.m_outer = B.tall;
        // Elongated matrices with a short side of at most 1024: a tile's
        // mainloop (K = s) is short and its epilogue's reads of X are the
        // slower side, so the epilogue prefetches them into L2.  Measured:
        // the 16384 x 1024 set +3.4 %; enabled for every s <= 1024 it cost
        // the 2B set 0.5 % (its 1024 x 2048 bucket), for every s 1.2 %.
        a.epi_l2pf = B.s <= 1024 && B.l >= 4 * B.s;
        a.ld_x = B.ld_x; a.ld_s = B.ld_s;
        a.x_state = reinterpret_cast<float*>(ws + B.off_xs);
        a.x_op_out = (it + 1 < ns_steps) ? xn : nullptr;
        // two-part state: written by every apply but the last, read from the
        // second iteration on (hi is the current operand copy of X)
        a.x_hi = xc;
        a.x_lo = reinterpret_cast<__nv_bfloat16*>(ws + B.off_xlo);
        a.in_hilo = it > 0;
        a.scale = it == 0 ? sc.inv_nu + B.first : nullptr;
        a.ca = coeffs[0];
        a.status = status;
        if (B.fusable) {
            const bool last = it + 1 == ns_steps;
            a.variant = (fuse.in && it == 0 ? NS_IN_SRC : 0) | (fuse.out && last ? NS_OUT_U : 0) |
                        (fuse.out_w && last ? NS_OUT_W : 0);
        }
        a.io = reinterpret_cast<const NsIO*>(ws + P.off_io) + B.first;
        a.upart = reinterpret_cast<double*>(ws + P.off_upart) + B.upart0;
        a.mflags = sc.flags + B.first;
        a.nlr = -fuse.lr * update_scale(B.R, B.C, fuse.scale_mode);
        a.wdecay = fuse.wdecay;
        const double G = B.G, S = B.s, L = B.l;
        cudaError_t e;
        {
            // bytes per element: X read (fp32 4, or hi + lo 2 + 2), X written (hi + lo 2 + 2
            // unless last, else fp32 4), W read when fused (4); NS_OUT_W writes the weight
            // (fp32 and bf16) in place of X
            double per_el = 4.0 + 4.0 + ((a.variant & NS_OUT_U) ? 4.0 : 0.0);
            if (a.variant & NS_OUT_W) per_el = 4.0 + 4.0 + 4.0 + 2.0;
            Trace tr(apply_kind(a.variant), cur);
            e = tr.done(B.tall ? tc::launch_ns_gemm(a, xc, B.ld_x, bop, B.ld_s, pair, cur, &why)
                               : tc::launch_ns_gemm(a, bop, B.ld_s, xc, B.ld_x, pair, cur, &why),
                        2 * G * S * S * L, G * S * S * 2 + G * S * L * per_el);
        }
        return sy.check_on(cur, e, e == cudaErrorInvalidValue ? why : "tcgen05 apply launch");
    };

    // Streams (Schedule): an s-group's polynomial runs on its first
    // bucket's stream, after every Gram of the group, and the group's applies
    // run after it.  The next iteration's Gram of a bucket follows its apply
    // on the same stream, so the polynomial of iteration it+1 (which rewrites
    // the group's A and B buffers) comes after every apply of iteration it.
    const std::vector<cudaStream_t>& bst = S.bst;
    NsStreams* ns = S.ns;
    // group stream waits for / releases the streams of the group's buckets
    auto join_group = [&](const SGroup& Q, cudaStream_t gs, bool to_group) {
        std::vector<cudaStream_t> seen;
        for (int b = Q.b_begin; b < Q.b_end; ++b) {
            if (bst[b] == gs || std::find(seen.begin(), seen.end(), bst[b]) != seen.end()) continue;
            seen.push_back(bst[b]);
            cudaError_t e = to_group ? stream_after(*ns, gs, bst[b]) : stream_after(*ns, bst[b], gs);
            if (e != cudaSuccess) return cuda_fail(e, "Newton-Schulz stream ordering");
        }
        return (int)MUONH_OK;
    };

    for (int it = 0; it < ns_steps; ++it) {
        for (const SGroup& Q : P.sgroups) {
            if (fuse.small && Q.small_step) continue;   // done by the small-matrix kernel
            // every bucket of an s-group has the same s, so the same path
            const bool simt = check || Q.s <= kSmallSide;
            for (int b = Q.b_begin; b < Q.b_end; ++b) {
                cur = bst[b];
                const int r = simt ? simt_gram(P.buckets[b], it) : tc_gram(P.buckets[b], it);
                if (r) return r;
            }
            const cudaStream_t gs = bst[Q.b_begin];
            int r = ns ? join_group(Q, gs, true) : MUONH_OK;
            if (r) return r;
            cur = gs;
            r = simt ? simt_poly(Q) : tc_poly(Q);
            if (r) return r;
            r = ns ? join_group(Q, gs, false) : MUONH_OK;
            if (r) return r;
            for (int b = Q.b_begin; b < Q.b_end; ++b) {
                cur = bst[b];
                r = simt ? simt_apply(P.buckets[b], it) : tc_apply(P.buckets[b], it);
                if (r) return r;
            }
        }
    }
    *x_in_alt = (ns_steps & 1) != 0;
    return MUONH_OK;
}

int check_scalars(int ns_steps, const float* coeffs, float eps, uint32_t flags) {
    if (ns_steps < 0 || ns_steps > 64) return fail(MUONH_ERR_INVALID_ARG, "ns_steps must be in [0, 64]");
    if (!coeffs) return fail(MUONH_ERR_INVALID_ARG, "ns_coeffs is NULL");
    for (int i = 0; i < 3; ++i)
        if (!std::isfinite(coeffs[i])) return fail(MUONH_ERR_INVALID_ARG, "ns_coeffs must be finite");
    if (!std::isfinite(eps) || eps < 0.f) return fail(MUONH_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (flags & ~(uint32_t)(MUONH_FLAG_FP32_CHECK | MUONH_FLAG_SYNC_DEBUG | MUONH_FLAG_GEMM_1SM |
                            MUONH_FLAG_GEMM_ONE_STEP | MUONH_FLAG_ONE_STREAM | MUONH_FLAG_NESTEROV | MUONH_FLAG_SCALE_SHAPE | MUONH_FLAG_SCALE_RMS |
                            MUONH_FLAG_GRAD_BF16))
        return fail(MUONH_ERR_UNSUPPORTED, "unknown flag bits");
    if ((flags & MUONH_FLAG_SCALE_SHAPE) && (flags & MUONH_FLAG_SCALE_RMS))
        return fail(MUONH_ERR_UNSUPPORTED, "MUONH_FLAG_SCALE_SHAPE and MUONH_FLAG_SCALE_RMS exclude each other");
    return MUONH_OK;
}

// True when every matrix of the batch takes its whole step in the
// small-matrix kernel (the batch's other kernels would do nothing).
bool all_small(const DescBatch& b) {
    for (int k = 0; k < b.n; ++k)
        if (!(b.d[k].fused & kFusedAll)) return false;
    return true;
}

// The matrices of small-step s-groups (caller indices, bucket order).
std::vector<int> small_step_matrices(const Plan& P) {
    std::vector<int> idx;
    for (int p = 0; p < P.n; ++p)
        if (P.sgroups[P.buckets[P.bucket_of[p]].sgroup].small_step) idx.push_back(P.order[p]);
    return idx;
}

// One launch sequence of the small-matrix kernel for a step (no-op if the
// step has none of its matrices).
int run_small_step(const Plan& P, const muonh_matrix_t* mats, const SmallStepArgs& a, Sync& sy) {
    const std::vector<int> idx = small_step_matrices(P);
    if (idx.empty()) return MUONH_OK;
    double flops = 0, bytes = 0;
    for (int u : idx) {
        const double r = (double)mats[u].rows, c = (double)mats[u].cols, sd = std::min(r, c), ld = std::max(r, c);
        flops += a.ns_steps * (3 * sd * sd * ld + sd * sd * sd);
        bytes += r * c * (22 + (mats[u].w_bf16 ? 0 : -2));
    }
    Trace tr(K_SMALL, sy.st);
    int launches = 0;
    const cudaError_t e = launch_small_step(mats, idx.data(), (int)idx.size(), a, sy.st, &launches);
    if (launches > 1) g_launches += launches - 1;
    return sy.check(tr.done(e, flops, bytes), "small-matrix step launch");
}

int scale_mode_of(uint32_t flags) {
    if (flags & MUONH_FLAG_SCALE_SHAPE) return kScaleShape;
    if (flags & MUONH_FLAG_SCALE_RMS) return kScaleRms;
    return kScaleNone;
}

int check_workspace(void* ws, size_t ws_bytes, size_t need) {
    if (!ws) return fail(MUONH_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(MUONH_ERR_WORKSPACE, "workspace not 256-byte aligned");
    if (ws_bytes < need) {
        char buf[128];
        snprintf(buf, sizeof buf, "workspace too small: %zu < %zu bytes", ws_bytes, need);
        return fail(MUONH_ERR_WORKSPACE, buf);
    }
    return MUONH_OK;
}

int get_status_ptr(uint32_t** p) {
    cudaError_t e = status_word(p);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    return MUONH_OK;
}

}  // namespace

// Lets other translation units of the library report an error text.
int report_error(int code, const char* msg) { return fail(code, msg); }

int orthogonalize_impl(const void* in, int in_dtype, void* out, int out_dtype, int64_t rows, int64_t cols,
                       int ns_steps, const float ns_coeffs[3], float eps, uint32_t flags, void* workspace,
                       size_t ws_bytes, void* stream);

}  // namespace muonh

using namespace muonh;

extern "C" {

int muonh_version(void) { return 100; }

const char* muonh_last_error(void) { return g_last_error.c_str(); }

const char* muonh_status_string(int code) {
    switch (code) {
        case MUONH_OK: return "ok";
        case MUONH_ERR_INVALID_ARG: return "invalid argument";
        case MUONH_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MUONH_ERR_UNSUPPORTED: return "unsupported flag or shape";
        case MUONH_ERR_CUDA: return "CUDA error";
        default: return "unknown code";
    }
}

int muonh_capture_norms(const muonh_matrix_t* mats, int n, float* r0_dev, void* stream) {
    g_last_error.clear();
    std::vector<int64_t> rc;
    int r = check_shapes(mats, n, rc, false);
    if (r) return r;
    if (!r0_dev || (reinterpret_cast<uintptr_t>(r0_dev) & 3u))
        return fail(MUONH_ERR_INVALID_ARG, "r0_dev is NULL or not 4-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int b0 = 0; b0 < n; b0 += kMaxDescPerLaunch) {
        DescBatch B;
        memset(&B, 0, sizeof B);
        B.n = std::min(kMaxDescPerLaunch, n - b0);
        B.first = b0;
        for (int k = 0; k < B.n; ++k) {
            B.d[k].w = mats[b0 + k].w;
            B.d[k].rows = (int)mats[b0 + k].rows;
            B.d[k].cols = (int)mats[b0 + k].cols;
            B.d[k].user_index = b0 + k;
        }
        Trace tr(K_CAPTURE, st);
        cudaError_t e = tr.done(launch_capture_norms(B, r0_dev, st), 0, batch_elems(B) * 4);
        if (e != cudaSuccess) return cuda_fail(e, "capture_norms launch");
    }
    return MUONH_OK;
}

int muonh_workspace_size(const muonh_matrix_t* mats, int n, uint32_t flags, size_t* bytes) {
    g_last_error.clear();
    if (!bytes) return fail(MUONH_ERR_INVALID_ARG, "bytes is NULL");
    std::vector<int64_t> rc;
    int r = check_shapes(mats, n, rc, false);
    if (r) return r;
    *bytes = get_plan(rc.data(), n, flags).bytes;
    return MUONH_OK;
}

int muonh_step(const muonh_matrix_t* mats, int n, const float* r0_dev, float lr, float beta, int ns_steps,
               const float ns_coeffs[3], float eps, uint32_t flags, void* workspace, size_t ws_bytes,
               void* stream) {
    g_last_error.clear();
    std::vector<int64_t> rc;
    int r = check_shapes(mats, n, rc, true);
    if (r) return r;
    if (!r0_dev || (reinterpret_cast<uintptr_t>(r0_dev) & 3u))
        return fail(MUONH_ERR_INVALID_ARG, "r0_dev is NULL or not 4-byte aligned");
    if (!std::isfinite(lr) || !std::isfinite(beta)) return fail(MUONH_ERR_INVALID_ARG, "lr and beta must be finite");
    r = check_scalars(ns_steps, ns_coeffs, eps, flags);
    if (r) return r;
    const Plan& P = get_plan(rc.data(), n, flags);
    r = check_workspace(workspace, ws_bytes, P.bytes);
    if (r) return r;
    uint32_t* status = nullptr;
    r = get_status_ptr(&status);
    if (r) return r;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Sync sy{(flags & MUONH_FLAG_SYNC_DEBUG) != 0, st};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const Scalars sc = scalars_of(P, ws);
    double* partials = reinterpret_cast<double*>(ws + P.off_partials);

    // Tensor-core path with at least one iteration, for the matrices whose
    // row length is a multiple of 4: momentum writes no fp32 copy of X (the
    // first apply reads M), and the last apply writes U = W - lr*O with its
    // ||U||^2 partials, so their hyperball step is one finalize plus a
    // rescale.  Other matrices, the fp32 check mode and ns_steps = 0 keep the
    // separate norm and apply passes.
    const bool check = (flags & MUONH_FLAG_FP32_CHECK) != 0;
    const bool nesterov = (flags & MUONH_FLAG_NESTEROV) != 0;
    const bool grad_bf16 = (flags & MUONH_FLAG_GRAD_BF16) != 0;
    NsFuse fuse;
    // with Nesterov momentum the Newton-Schulz input is not M, so it is stored
    fuse.in = !check && !nesterov && ns_steps >= 1;
    fuse.out = !check && ns_steps >= 1;
    fuse.pair = (flags & MUONH_FLAG_GEMM_1SM) == 0;
    fuse.check = check;
    fuse.small = !check && ns_steps >= 1;
    fuse.scale_mode = scale_mode_of(flags);
    fuse.lr = lr;
    // every bucket's momentum, Newton-Schulz and hyperball passes run on its
    // stream (Schedule); the small-matrix kernel runs on the caller's stream
    Schedule S;
    r = S.open(P, flags, fuse.small, st);
    if (r) return r;
    if (fuse.small) {
        SmallStepArgs sa{lr, beta, eps, 1.f, ns_coeffs, ns_steps, false, nesterov, grad_bf16, fuse.scale_mode, r0_dev,
                         status};
        r = run_small_step(P, mats, sa, sy);
        if (r) return r;
    }
    if (fuse.out && P.n_upart > INT32_MAX)
        return fail(MUONH_ERR_UNSUPPORTED, "too many matrices/tiles for one step: split the list");
    // the table of the matrices' own buffers, read by every fused apply variant
    NsIO* io = (fuse.in || fuse.out) ? reinterpret_cast<NsIO*>(ws + P.off_io) : nullptr;
    const double* upart = reinterpret_cast<const double*>(ws + P.off_upart);

    std::vector<DescBatch> batches = make_batches(P, mats, ws, false, true, fuse);
    // elements of the batch's matrices with and without a fusion bit
    auto elems = [](const DescBatch& b, int bit, bool with) {
        double e = 0;
        for (int k = 0; k < b.n; ++k)
            if (((b.d[k].fused & bit) != 0) == with) e += (double)b.d[k].rows * b.d[k].cols;
        return e;
    };
    for (const DescBatch& B : batches) {
        if (all_small(B)) continue;
        const double bytes = 14 * elems(B, kFusedIn, true) +
                             18 * (elems(B, kFusedIn, false) - elems(B, kFusedAll, true));
        const cudaStream_t bs = S.bst[B.bucket];
        {
            Trace tr(K_MOMENTUM, bs);
            r = sy.check_on(bs, tr.done(launch_momentum(B, beta, partials, io, nesterov, grad_bf16, bs), 0,
                                        bytes - (grad_bf16 ? 2 * (elems(B, 0, false) - elems(B, kFusedAll, true)) : 0)),
                            "momentum launch");
        }
        if (r) return r;
        {
            Trace tr(K_MOM_FIN, bs);
            r = sy.check_on(bs, tr.done(launch_momentum_finalize(B, partials, sc, eps, fuse.scale_mode, ns_steps == 0, bs),
                                        0, 0),
                            "momentum finalize launch");
        }
        if (r) return r;
    }
    bool x_alt = false;
    r = run_newton_schulz(P, ws, sc, ns_steps, ns_coeffs, flags, status, sy, &x_alt, fuse, S);
    if (r) return r;
    if (x_alt) batches = make_batches(P, mats, ws, true, true, fuse);
    const float* o_scale = sc.oscale;
    for (const DescBatch& B : batches) {
        if (all_small(B)) continue;
        const double e_sep = elems(B, kFusedOut, false) - elems(B, kFusedAll, true);
        const double e_fused = elems(B, kFusedOut, true);
        const cudaStream_t bs = S.bst[B.bucket];
        if (e_sep > 0) {
            Trace tr(K_HB_NORM, bs);
            r = sy.check_on(bs, tr.done(launch_hyperball_norm(B, lr, partials, o_scale, bs), 0, e_sep * 8),
                            "hyperball norm launch");
            if (r) return r;
        }
        {
            Trace tr(K_HB_FIN, bs);
            r = sy.check_on(bs, tr.done(launch_hyperball_finalize(B, partials, upart, sc, r0_dev, bs), 0, 0),
                            "hyperball finalize launch");
        }
        if (r) return r;
        {
            Trace tr(e_sep > 0 ? K_HB_APPLY : K_HB_SCALE, bs);
            r = sy.check_on(bs, tr.done(launch_hyperball_finish(B, lr, sc, o_scale, bs), 0, e_sep * 14 + e_fused * 10),
                            "hyperball finish launch");
        }
        if (r) return r;
    }
    return S.close();
}

int muon_step(const muonh_matrix_t* mats, int n, float lr, float beta, float weight_decay, int ns_steps,
              const float ns_coeffs[3], float eps, uint32_t flags, void* workspace, size_t ws_bytes, void* stream) {
    g_last_error.clear();
    std::vector<int64_t> rc;
    int r = check_shapes(mats, n, rc, true);
    if (r) return r;
    if (!std::isfinite(lr) || !std::isfinite(beta) || !std::isfinite(weight_decay))
        return fail(MUONH_ERR_INVALID_ARG, "lr, beta and weight_decay must be finite");
    r = check_scalars(ns_steps, ns_coeffs, eps, flags);
    if (r) return r;
    const Plan& P = get_plan(rc.data(), n, flags);
    r = check_workspace(workspace, ws_bytes, P.bytes);
    if (r) return r;
    uint32_t* status = nullptr;
    r = get_status_ptr(&status);
    if (r) return r;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Sync sy{(flags & MUONH_FLAG_SYNC_DEBUG) != 0, st};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const Scalars sc = scalars_of(P, ws);
    double* partials = reinterpret_cast<double*>(ws + P.off_partials);

    // Same momentum and Newton-Schulz as muonh_step; for the matrices of
    // fusable buckets the last apply writes the new weight itself, the rest
    // get it from muon_finish_kernel.
    const bool check = (flags & MUONH_FLAG_FP32_CHECK) != 0;
    const bool nesterov = (flags & MUONH_FLAG_NESTEROV) != 0;
    const bool grad_bf16 = (flags & MUONH_FLAG_GRAD_BF16) != 0;
    NsFuse fuse;
    fuse.in = !check && !nesterov && ns_steps >= 1;
    fuse.out_w = !check && ns_steps >= 1;
    fuse.pair = (flags & MUONH_FLAG_GEMM_1SM) == 0;
    fuse.check = check;
    fuse.small = !check && ns_steps >= 1;
    fuse.scale_mode = scale_mode_of(flags);
    fuse.lr = lr;
    fuse.wdecay = 1.f - lr * weight_decay;
    Schedule S;
    r = S.open(P, flags, fuse.small, st);
    if (r) return r;
    if (fuse.small) {
        SmallStepArgs sa{lr, beta, eps, fuse.wdecay, ns_coeffs, ns_steps, true, nesterov, grad_bf16, fuse.scale_mode,
                         nullptr, status};
        r = run_small_step(P, mats, sa, sy);
        if (r) return r;
    }
    // the table of the matrices' own buffers, read by every fused apply variant
    NsIO* io = (fuse.in || fuse.out_w) ? reinterpret_cast<NsIO*>(ws + P.off_io) : nullptr;

    std::vector<DescBatch> batches = make_batches(P, mats, ws, false, true, fuse);
    for (const DescBatch& B : batches) {
        if (all_small(B)) continue;
        double e_in = 0, e_all = 0;
        for (int k = 0; k < B.n; ++k) {
            if (B.d[k].fused & kFusedAll) continue;
            const double e = (double)B.d[k].rows * B.d[k].cols;
            e_all += e;
            if (B.d[k].fused & kFusedIn) e_in += e;
        }
        const cudaStream_t bs = S.bst[B.bucket];
        {
            Trace tr(K_MOMENTUM, bs);
            r = sy.check_on(bs, tr.done(launch_momentum(B, beta, partials, io, nesterov, grad_bf16, bs), 0,
                                        14 * e_in + 18 * (e_all - e_in) - (grad_bf16 ? 2 * e_all : 0)),
                            "momentum launch");
        }
        if (r) return r;
        {
            Trace tr(K_MOM_FIN, bs);
            r = sy.check_on(bs, tr.done(launch_momentum_finalize(B, partials, sc, eps, fuse.scale_mode, ns_steps == 0, bs),
                                        0, 0),
                            "momentum finalize launch");
        }
        if (r) return r;
    }
    bool x_alt = false;
    r = run_newton_schulz(P, ws, sc, ns_steps, ns_coeffs, flags, status, sy, &x_alt, fuse, S);
    if (r) return r;
    if (x_alt) batches = make_batches(P, mats, ws, true, true, fuse);
    const float* o_scale = sc.oscale;
    for (const DescBatch& B : batches) {
        double e_sep = 0;
        for (int k = 0; k < B.n; ++k)
            if (!(B.d[k].fused & (kFusedOutW | kFusedAll))) e_sep += (double)B.d[k].rows * B.d[k].cols;
        if (e_sep == 0) continue;
        const cudaStream_t bs = S.bst[B.bucket];
        Trace tr(K_MUON_FIN, bs);
        r = sy.check_on(bs, tr.done(launch_muon_finish(B, lr, fuse.wdecay, sc, o_scale, bs), 0, e_sep * 14),
                        "muon finish launch");
        if (r) return r;
    }
    return S.close();
}

int adamw_step(const adamw_param_t* params, int n, int step, float lr, float beta1, float beta2, float eps,
               float weight_decay, void* stream) {
    g_last_error.clear();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Trace tr(K_ADAMW, st);
    int launches = 0;
    double bytes = 0;
    const int r = adamw_launch(params, n, step, lr, beta1, beta2, eps, weight_decay, st, &launches, &bytes);
    if (launches > 1) g_launches += launches - 1;
    if (launches == 0) --g_launches;
    tr.done(cudaSuccess, 0, bytes);
    return r;
}

int muonh_orthogonalize_workspace_size(int64_t rows, int64_t cols, uint32_t flags, size_t* bytes) {
    g_last_error.clear();
    if (!bytes) return fail(MUONH_ERR_INVALID_ARG, "bytes is NULL");
    if (rows < 1 || cols < 1 || rows > MUONH_MAX_SIDE || cols > MUONH_MAX_SIDE)
        return fail(MUONH_ERR_INVALID_ARG, "rows/cols out of range");
    const int64_t rc[2] = {rows, cols};
    *bytes = get_plan(rc, 1, flags).bytes;
    return MUONH_OK;
}

int muonh_orthogonalize(const void* in, int in_dtype, void* out, int out_dtype, int64_t rows, int64_t cols,
                        int ns_steps, const float ns_coeffs[3], float eps, uint32_t flags, void* workspace,
                        size_t ws_bytes, void* stream) {
    g_last_error.clear();
    return muonh::orthogonalize_impl(in, in_dtype, out, out_dtype, rows, cols, ns_steps, ns_coeffs, eps, flags,
                                     workspace, ws_bytes, stream);
}

}  // extern "C"

namespace muonh {

// Newton-Schulz of one matrix (muonh_orthogonalize).
int orthogonalize_impl(const void* in, int in_dtype, void* out, int out_dtype, int64_t rows, int64_t cols,
                       int ns_steps, const float ns_coeffs[3], float eps, uint32_t flags, void* workspace,
                       size_t ws_bytes, void* stream) {
    g_last_error.clear();
    if (!in || !out || !aligned16(in) || !aligned16(out))
        return fail(MUONH_ERR_INVALID_ARG, "in/out NULL or not 16-byte aligned");
    if ((in_dtype != MUONH_DTYPE_F32 && in_dtype != MUONH_DTYPE_BF16) ||
        (out_dtype != MUONH_DTYPE_F32 && out_dtype != MUONH_DTYPE_BF16))
        return fail(MUONH_ERR_UNSUPPORTED, "in_dtype/out_dtype must be MUONH_DTYPE_F32 or MUONH_DTYPE_BF16");
    if (rows < 1 || cols < 1 || rows > MUONH_MAX_SIDE || cols > MUONH_MAX_SIDE)
        return fail(MUONH_ERR_INVALID_ARG, "rows/cols out of range");
    int r = check_scalars(ns_steps, ns_coeffs, eps, flags);
    if (r) return r;
    const int64_t rc[2] = {rows, cols};
    const Plan& P = get_plan(rc, 1, flags);
    r = check_workspace(workspace, ws_bytes, P.bytes);
    if (r) return r;
    uint32_t* status = nullptr;
    r = get_status_ptr(&status);
    if (r) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Sync sy{(flags & MUONH_FLAG_SYNC_DEBUG) != 0, st};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const Scalars sc = scalars_of(P, ws);
    double* partials = reinterpret_cast<double*>(ws + P.off_partials);
    const bool in_bf16 = in_dtype == MUONH_DTYPE_BF16, out_bf16 = out_dtype == MUONH_DTYPE_BF16;
    muonh_matrix_t m{};
    m.w = static_cast<float*>(const_cast<void*>(in));   // read by the first kernel as the input
    m.rows = rows;
    m.cols = cols;
    const double el = (double)rows * cols;
    NsFuse fuse;
    fuse.check = (flags & MUONH_FLAG_FP32_CHECK) != 0;
    // the first apply can read an fp32 input in place of an fp32 copy of X;
    // a bf16 input is widened into the fp32 state by the first kernel
    fuse.in = !fuse.check && ns_steps >= 1 && !in_bf16;
    NsIO* io = fuse.in ? reinterpret_cast<NsIO*>(ws + P.off_io) : nullptr;
    std::vector<DescBatch> batches = make_batches(P, &m, ws, false, false, fuse);
    const bool in_fused = (batches[0].d[0].fused & kFusedIn) != 0;
    {
        // bytes: the input read (4 or 2), X_op written (2), and the fp32 state (4) unless fused
        Trace tr(K_MOMENTUM, st);
        r = sy.check(tr.done(launch_momentum(batches[0], 0.f, partials, io, false, in_bf16, st), 0,
                             el * ((in_bf16 ? 2 : 4) + 2 + (in_fused ? 0 : 4))),
                     "momentum launch");
    }
    if (r) return r;
    {
        Trace tr(K_MOM_FIN, st);
        r = sy.check(tr.done(launch_momentum_finalize(batches[0], partials, sc, eps, kScaleNone, ns_steps == 0, st), 0, 0),
                     "momentum finalize launch");
    }
    if (r) return r;
    bool x_alt = false;
    Schedule S;   // one matrix, one bucket: the caller's stream only
    r = S.open(P, flags, fuse.small, st);
    if (r) return r;
    r = run_newton_schulz(P, ws, sc, ns_steps, ns_coeffs, flags, status, sy, &x_alt, fuse, S);
    if (r) return r;
    r = S.close();
    if (r) return r;
    m.w = static_cast<float*>(out);
    batches = make_batches(P, &m, ws, x_alt, false, fuse);
    {
        Trace tr(K_EMIT, st);
        r = sy.check(tr.done(launch_emit(batches[0], ns_steps == 0 ? sc.inv_nu : nullptr, out_bf16, st), 0,
                             el * (4 + (out_bf16 ? 2 : 4))),
                     "emit launch");
    }
    return r;
}

}  // namespace muonh

extern "C" {

int muonh_partition(const muonh_matrix_t* mats, int n, int world_size, int* owner_out) {
    g_last_error.clear();
    std::vector<int64_t> rc;
    int r = check_shapes(mats, n, rc, false);
    if (r) return r;
    if (world_size < 1 || world_size > 65536) return fail(MUONH_ERR_INVALID_ARG, "world_size must be in [1, 65536]");
    if (!owner_out) return fail(MUONH_ERR_INVALID_ARG, "owner_out is NULL");
    std::vector<std::pair<double, int>> cost(n);
    for (int i = 0; i < n; ++i) {
        const double a = (double)rc[2 * i], b = (double)rc[2 * i + 1];
        const double sd = std::min(a, b), ld = std::max(a, b);
        cost[i] = {3 * sd * sd * ld + sd * sd * sd, i};
    }
    std::stable_sort(cost.begin(), cost.end(), [](const std::pair<double, int>& x, const std::pair<double, int>& y) {
        return x.first > y.first;
    });
    std::vector<double> load(world_size, 0.0);
    for (const auto& c : cost) {
        int best = 0;
        for (int k = 1; k < world_size; ++k)
            if (load[k] < load[best]) best = k;
        load[best] += c.first;
        owner_out[c.second] = best;
    }
    return MUONH_OK;
}

int muonh_get_status(uint32_t* status_out, void* stream) {
    g_last_error.clear();
    if (!status_out) return fail(MUONH_ERR_INVALID_ARG, "status_out is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t* dev = nullptr;
    int r = get_status_ptr(&dev);
    if (r) return r;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpy(status_out, dev, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    e = cudaMemset(dev, 0, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    return MUONH_OK;
}

int muonh_profile_enable(int on) {
    g_last_error.clear();
    std::vector<Pending> drop;
    {
        std::lock_guard<std::mutex> lk(g_prof.mu);
        g_prof.on = on != 0;
        if (on) {
            drop.swap(g_prof.pending);
            for (int k = 0; k < K_COUNT; ++k) {
                g_prof.launches[k] = 0;
                g_prof.ms[k] = g_prof.flops[k] = g_prof.bytes[k] = 0;
            }
        }
    }
    for (Pending& q : drop) {
        cudaEventSynchronize(q.b);
        std::lock_guard<std::mutex> lk(g_prof.mu);
        g_prof.pool.push_back(q.a);
        g_prof.pool.push_back(q.b);
    }
    return MUONH_OK;
}

int muonh_profile_read(muonh_profile_entry_t* out, int max_entries, int* n_out) {
    g_last_error.clear();
    if (!out || !n_out || max_entries < 0) return fail(MUONH_ERR_INVALID_ARG, "out/n_out NULL");
    std::lock_guard<std::mutex> lk(g_prof.mu);
    // per kind, the launch intervals in ms from the first recorded start;
    // a kind's time is the length of their union (launches of one kind on
    // different streams may overlap)
    std::vector<std::vector<std::pair<float, float>>> iv(K_COUNT);
    const cudaEvent_t ref = g_prof.pending.empty() ? nullptr : g_prof.pending.front().a;
    for (Pending& q : g_prof.pending) {
        cudaError_t e = cudaEventSynchronize(q.b);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
        float ms = 0.f, t0 = 0.f;
        e = cudaEventElapsedTime(&ms, q.a, q.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t0, ref, q.a);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
        iv[q.kind].push_back({t0, t0 + ms});
        g_prof.launches[q.kind] += 1;
        g_prof.flops[q.kind] += q.flops;
        g_prof.bytes[q.kind] += q.bytes;
        if (is_ns_kind(q.kind)) {
            iv[K_NS_BUSY].push_back({t0, t0 + ms});
            g_prof.launches[K_NS_BUSY] += 1;
            g_prof.flops[K_NS_BUSY] += q.flops;
            g_prof.bytes[K_NS_BUSY] += q.bytes;
        }
    }
    for (Pending& q : g_prof.pending) {
        g_prof.pool.push_back(q.a);
        g_prof.pool.push_back(q.b);
    }
    g_prof.pending.clear();
    for (int k = 0; k < K_COUNT; ++k) {
        std::vector<std::pair<float, float>>& v = iv[k];
        std::sort(v.begin(), v.end());
        double busy = 0.0;
        for (size_t i = 0; i < v.size();) {
            float lo = v[i].first, hi = v[i].second;
            size_t j = i + 1;
            for (; j < v.size() && v[j].first <= hi; ++j) hi = std::max(hi, v[j].second);
            busy += hi - lo;
            i = j;
        }
        g_prof.ms[k] += busy;
    }
    int n = 0;
    for (int k = 0; k < K_COUNT && n < max_entries; ++k) {
        if (g_prof.launches[k] == 0) continue;
        out[n].name = kKindName[k];
        out[n].launches = g_prof.launches[k];
        out[n].ms = g_prof.ms[k];
        out[n].flops = g_prof.flops[k];
        out[n].bytes = g_prof.bytes[k];
        ++n;
    }
    *n_out = n;
    return MUONH_OK;
}

int64_t muonh_launch_count(void) { return g_launches.load(); }

int muonh_test_gemm_timeout(uint32_t flags, uint64_t timeout_ns, void* workspace, size_t ws_bytes, void* stream) {
    g_last_error.clear();
    if (flags & ~(uint32_t)MUONH_FLAG_GEMM_1SM) return fail(MUONH_ERR_UNSUPPORTED, "flags: only MUONH_FLAG_GEMM_1SM");
    if (timeout_ns < 1000ull || timeout_ns > 10000000000ull)
        return fail(MUONH_ERR_INVALID_ARG, "timeout_ns must be in [1e3, 1e10]");
    int r = check_workspace(workspace, ws_bytes, MUONH_TEST_TIMEOUT_WS_BYTES);
    if (r) return r;
    uint32_t* status = nullptr;
    r = get_status_ptr(&status);
    if (r) return r;
    // a 256 x 256 Gram: X_op bf16 [256][256], A fp32 [256][256], A_op bf16 [256][256]
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    GemmParams g{};
    g.mode = NS_GRAM; g.G = 1; g.M = 256; g.N = 256; g.K = 256;
    g.ld_x = 256; g.ld_s = 256;

    g.sym_bf16 = reinterpret_cast<__nv_bfloat16*>(ws + 384 * 1024);
    g.status = status;
    g.timeout_ns = timeout_ns;
    g.test_no_loads = 1;
    const char* why = "";
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Trace tr(K_GRAM, st);
    cudaError_t e = tr.done(tc::launch_ns_gemm(g, ws, 256, ws, 256,
                                               (flags & MUONH_FLAG_GEMM_1SM) ? tc::kGemmSingle : tc::kGemmPair, st,
                                               &why),
                            0, 0);
    if (e != cudaSuccess) return e == cudaErrorInvalidValue ? fail(MUONH_ERR_CUDA, why) : cuda_fail(e, "test GEMM launch");
    return MUONH_OK;
}

}  // extern "C"
