// lisa_api.cu -- the C ABI of liblisa.so: argument checks, the split-K plan,
// the workspace carve-up, host-side walk weights, and dispatch to the kernel
// families.  Every check runs on the host before the first launch.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "lisa.h"
#include "lisa_backward_mlp.h"
#include "lisa_bwd.h"
#include "lisa_internal.h"
#include "lisa_testing.h"

namespace lisa {
namespace {

constexpr int kTargetCtas = 2 * 152;  // two resident CTAs on each of the 152 SMs
constexpr int kTcTargetCtas = 228;     // about 1.5 waves of the 152 SMs
constexpr int kTcOneWaveCtas = 304;    // statistics CTAs resident at once for chunks <= 256 tokens (2 per SM)
constexpr int kMinChunk = 64;         // smallest split-K chunk, in tokens
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool supported_dim(int d) { return d == 16 || d == 32 || d == 64; }

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

}  // namespace

int choose_family(int dtype, int D, int T, int wmode, int hidden) {
    if (dtype != LISA_BF16 || D != 64) return kFamilySimt;
    if (wmode == LISA_W_MLP) {
        // TMEM holds Q [U_1..U_(T-1) | s] (64 (T-1) + 16 columns) and the MLP
        // hidden layer (hidden rounded up to 16) side by side: 512 columns.
        const int cols = 64 * (T - 1) + 16 + (hidden + 15) / 16 * 16;
        if (T < 2 || cols > 512) return kFamilySimt;
    }
    return kFamilyTc;
}

Plan make_plan(int slices, int n, int D, int T, int dtype, int wmode, int hidden) {
    Plan pl{};
    pl.family = choose_family(dtype, D, T, wmode, hidden);
    int chunks, chunk;
    if (pl.family == kFamilyTc) {
        // chunks of whole 64-token pipeline stages, about 1.5 waves of CTAs,
        // and a chunk count a cluster of at most 8 CTAs divides evenly
        chunks = (kTcTargetCtas + slices - 1) / slices;
        const int max_chunks = (n + 63) / 64;
        if (chunks > max_chunks) chunks = max_chunks;
        if (chunks < 1) chunks = 1;
        if (chunks > 8) chunks = (chunks + 7) / 8 * 8;
        // short slices: rather one chunk per slice in a single wave than two
        // half-length chunks in more than one (the per-CTA latency barely
        // depends on the chunk's length there)
        if (chunks > 1 && n <= 256 && (long long)slices * chunks > kTcOneWaveCtas)
            chunks = std::max(1, kTcOneWaveCtas / slices);
        chunk = ((n + chunks - 1) / chunks + 63) / 64 * 64;
        chunks = (n + chunk - 1) / chunk;
        int cl = 1;
        for (int d = 8; d >= 1; --d)
            if (chunks % d == 0) { cl = d; break; }
        pl.cluster = cl;
    } else {
        chunks = (kTargetCtas + slices - 1) / slices;
        const int max_chunks = (n + kMinChunk - 1) / kMinChunk;
        if (chunks > max_chunks) chunks = max_chunks;
        if (chunks < 1) chunks = 1;
        chunk = (n + chunks - 1) / chunks;
        chunk = (chunk + 15) / 16 * 16;
        chunks = (n + chunk - 1) / chunk;
        pl.cluster = 1;
    }
    pl.chunks = chunks;
    pl.chunk = chunk;
    const size_t S = (size_t)slices, C = (size_t)chunks, d = (size_t)D;
    size_t off = 0;
    pl.off_err = off;    off = align_up(off + sizeof(int));   // must stay at 0: lisa_query_status reads it there
    pl.off_s_part = off; off = align_up(off + S * C * d * sizeof(float));
    if (pl.family == kFamilySimt) {
        const size_t nmat = (size_t)(T > 1 ? T - 1 : 1);
        pl.off_u_part = off; off = align_up(off + S * C * d * d * sizeof(float));
        pl.off_m_part = off; off = align_up(off + S * C * d * d * sizeof(float));
        pl.off_s_red = off;  off = align_up(off + S * d * sizeof(float));
        pl.off_ucat = off;   off = align_up(off + S * nmat * d * d * sizeof(float));
    } else {
        const size_t parts = C / (size_t)pl.cluster;
        const size_t n_umat = (wmode == LISA_W_MLP) ? (size_t)(T - 1) : 1;
        pl.off_tc_part = off;  off = align_up(off + S * parts * 128 * 64 * sizeof(float));
        pl.off_tc_bepi = off;  off = align_up(off + S * (64 * n_umat + 16) * 128);
        pl.off_tc_w1img = off; off = align_up(off + 2 * 64 * 128);
    }
    pl.total = off;
    return pl;
}

namespace {

// Shared validation of lisa_forward / lisa_forward_host / lisa_workspace_bytes
// scalars.  Returns LISA_OK, or the status to report.
lisa_status check_sizes(int B, int heads, int H, int W, int d_h, int d_v, int T, int dtype) {
    if (B < 0 || heads < 0 || H < 0 || W < 0) return LISA_ERR_INVALID_ARG;
    if (dtype != LISA_F32 && dtype != LISA_BF16) return LISA_ERR_INVALID_ARG;
    if (d_h < 1 || d_v < 1 || T < 0) return LISA_ERR_INVALID_ARG;   // T = 0: untruncated walk
    if (!supported_dim(d_h) || d_v != d_h) return LISA_ERR_UNSUPPORTED;
    if (T > LISA_MAX_T) return LISA_ERR_UNSUPPORTED;
    const long long slices = (long long)B * heads, n = (long long)H * W;
    if (n > (1LL << 30) || slices > (1LL << 30) || slices * n > (1LL << 31) - 1)
        return LISA_ERR_UNSUPPORTED;
    return LISA_OK;
}

// The untruncated walk (T = 0) runs the kernels of a T = 2 fixed-weight walk
// whose single hop matrix comes from the d x d solve.
int effective_T(int T) { return T == 0 ? 2 : T; }

// The dtype that picks the kernel family: the ELU + 1 feature map
// (relu_inputs = 2) runs the SIMT chain whatever the data type, since the
// tensor-core kernels apply ReLU in their bf16 staging.
int family_dtype(int dtype, int relu_inputs) { return relu_inputs == 2 ? (int)LISA_F32 : dtype; }

// Walk weights of a call into p (T, w, wmode, the untruncated flag).
lisa_status resolve_weights(Problem &p, const lisa_weights *wts, int T) {
    p.T = effective_T(T);
    if (T == 0 && wts->mode != LISA_W_GEOMETRIC) return LISA_ERR_INVALID_ARG;
    switch (wts->mode) {
        case LISA_W_GEOMETRIC: {
            const double beta = (double)wts->beta;
            if (!(beta >= 0.0 && beta < 1.0)) return LISA_ERR_INVALID_ARG;
            if (T == 0) {
                // untruncated: w_0 = 1 - beta on V; the hop terms sum to
                // beta (1-beta) Q~ (I - beta M)^-1 U_1, so w_1 = beta (1-beta)
                // scales the solved matrix
                p.w[0] = (float)(1.0 - beta);
                p.w[1] = (float)(beta * (1.0 - beta));
                p.untruncated = 1;
                p.beta = (float)beta;
                p.wmode = LISA_W_FIXED;
                break;
            }
            // paper Eq. 4: (1-beta) beta^k renormalised over k < T, in double
            const double norm = 1.0 - std::pow(beta, (double)T);
            for (int k = 0; k < T; ++k)
                p.w[k] = (float)((1.0 - beta) * std::pow(beta, (double)k) / norm);
            p.wmode = LISA_W_FIXED;
            break;
        }
        case LISA_W_FIXED:
            if (!wts->w) return LISA_ERR_INVALID_ARG;
            for (int k = 0; k < T; ++k) {
                if (!std::isfinite(wts->w[k])) return LISA_ERR_INVALID_ARG;
                p.w[k] = wts->w[k];
            }
            p.wmode = LISA_W_FIXED;
            break;
        case LISA_W_MLP:
            if (!wts->W1 || !wts->b1 || !wts->W2 || !wts->b2) return LISA_ERR_INVALID_ARG;
            if (wts->hidden < 1) return LISA_ERR_INVALID_ARG;
            if (wts->hidden > LISA_MAX_HIDDEN || T > LISA_MAX_T_MLP) return LISA_ERR_UNSUPPORTED;
            p.wmode = LISA_W_MLP;
            p.W1 = wts->W1; p.b1 = wts->b1; p.W2 = wts->W2; p.b2 = wts->b2;
            p.hidden = wts->hidden;
            break;
        default:
            return LISA_ERR_INVALID_ARG;
    }
    return LISA_OK;
}

// Sizes, inputs and workspace views of a checked call.
void fill_problem(Problem &p, const Plan &pl, const void *Q, const void *K, const void *V, void *O, int slices,
                  int heads, int H, int W, int d_h, int relu_inputs, float eps, const float *alpha, int dtype,
                  void *workspace) {
    p.Q = Q; p.K = K; p.V = V; p.O = O;
    p.slices = slices;
    p.heads = heads;
    p.H = H; p.W = W; p.n = H * W;
    p.D = d_h;
    p.relu = relu_inputs;
    p.eps = eps;
    p.alpha = alpha;
    p.dtype = dtype;
    p.chunks = pl.chunks;
    p.chunk = pl.chunk;
    p.family = pl.family;
    p.tc_cluster = pl.cluster;
    char *ws = static_cast<char *>(workspace);
    p.err = reinterpret_cast<int *>(ws + pl.off_err);
    p.s_part = reinterpret_cast<float *>(ws + pl.off_s_part);
    if (pl.family == kFamilySimt) {
        p.u_part = reinterpret_cast<float *>(ws + pl.off_u_part);
        p.m_part = reinterpret_cast<float *>(ws + pl.off_m_part);
        p.s_red = reinterpret_cast<float *>(ws + pl.off_s_red);
        p.ucat = reinterpret_cast<float *>(ws + pl.off_ucat);
    } else {
        p.tc_part = reinterpret_cast<float *>(ws + pl.off_tc_part);
        p.tc_bepi = reinterpret_cast<uint8_t *>(ws + pl.off_tc_bepi);
        p.tc_w1img = reinterpret_cast<uint8_t *>(ws + pl.off_tc_w1img);
    }
}

}  // namespace
}  // namespace lisa

using namespace lisa;

extern "C" size_t lisa_workspace_bytes(int B, int heads, int H, int W, int d_h, int d_v, int T,
                                       int dtype) {
    if (check_sizes(B, heads, H, W, d_h, d_v, T, dtype) != LISA_OK) return 0;
    const long long slices = (long long)B * heads, n = (long long)H * W;
    if (slices == 0 || n == 0) return 0;
    T = effective_T(T);
    // neither the weight mode nor the feature map is known here: size for
    // whichever needs more (the ELU map runs the SIMT chain for every dtype)
    size_t need = 0;
    for (int fam_dtype : {dtype, (int)LISA_F32}) {
        need = std::max(need, make_plan((int)slices, (int)n, d_h, T, fam_dtype, LISA_W_FIXED, 0).total);
        for (int hidden : {16, LISA_MAX_HIDDEN})
            need = std::max(need, make_plan((int)slices, (int)n, d_h, T, fam_dtype, LISA_W_MLP, hidden).total);
    }
    return need;
}

namespace {

// Checks every argument of a forward call and fills the Problem.  Sets
// *empty when there is nothing to compute.  Launches nothing.
lisa_status prepare(Problem &p, bool &empty, const void *Q, const void *K, const void *V, void *O,
                    int B, int heads, int H, int W, int d_h, int d_v, int T,
                    const lisa_weights *wts, const float *alpha, float eps, int relu_inputs,
                    int dtype, void *workspace, size_t workspace_bytes) {
    empty = false;
    lisa_status st = check_sizes(B, heads, H, W, d_h, d_v, T, dtype);
    if (st != LISA_OK) return st;
    if (!wts) return LISA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !std::isfinite(eps)) return LISA_ERR_INVALID_ARG;
    if (relu_inputs < 0 || relu_inputs > 2) return LISA_ERR_INVALID_ARG;

    p = Problem{};
    st = resolve_weights(p, wts, T);
    if (st != LISA_OK) return st;

    const long long slices = (long long)B * heads, n = (long long)H * W;
    if (slices == 0 || n == 0) {  // empty problem: nothing to launch
        empty = true;
        return LISA_OK;
    }
    if (!Q || !K || !V || !O || !alpha) return LISA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
        return LISA_ERR_INVALID_ARG;
    const size_t esz = (dtype == LISA_BF16) ? 2 : 4;
    const size_t bytes = (size_t)slices * (size_t)n * (size_t)d_h * esz;
    if (overlaps(O, bytes, Q, bytes) || overlaps(O, bytes, K, bytes) || overlaps(O, bytes, V, bytes))
        return LISA_ERR_INVALID_ARG;

    const Plan pl = make_plan((int)slices, (int)n, d_h, p.T, family_dtype(dtype, relu_inputs), p.wmode, p.hidden);
    if (!workspace || workspace_bytes < pl.total) return LISA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return LISA_ERR_INVALID_ARG;
    fill_problem(p, pl, Q, K, V, O, (int)slices, heads, H, W, d_h, relu_inputs, eps, alpha, dtype, workspace);
    return LISA_OK;
}

lisa_status launch(const Problem &p, cudaStream_t cs, int stage = -1) {
    cudaError_t err = (p.family == kFamilyTc) ? launch_tc(p, cs, stage) : launch_simt(p, cs, stage);
    return err == cudaSuccess ? LISA_OK : LISA_ERR_CUDA;
}

int weights_mode(const lisa_weights *wts) {
    if (!wts) return -1;
    return wts->mode == LISA_W_MLP ? LISA_W_MLP : LISA_W_FIXED;
}

}  // namespace

extern "C" lisa_status lisa_forward(const void *Q, const void *K, const void *V, void *O, int B,
                                    int heads, int H, int W, int d_h, int d_v, int T,
                                    const lisa_weights *wts, const float *alpha, float eps,
                                    int relu_inputs, int dtype, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    Problem p;
    bool empty;
    lisa_status st = prepare(p, empty, Q, K, V, O, B, heads, H, W, d_h, d_v, T, wts, alpha, eps,
                             relu_inputs, dtype, workspace, workspace_bytes);
    if (st != LISA_OK || empty) return st;
    return launch(p, static_cast<cudaStream_t>(stream));
}

extern "C" lisa_status lisa_forward_host(const void *hQ, const void *hK, const void *hV, void *hO,
                                         void *dQ, void *dK, void *dV, void *dO, int B, int heads,
                                         int H, int W, int d_h, int d_v, int T,
                                         const lisa_weights *wts, const float *alpha, float eps,
                                         int relu_inputs, int dtype, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    Problem p;
    bool empty;
    lisa_status st = prepare(p, empty, dQ, dK, dV, dO, B, heads, H, W, d_h, d_v, T, wts, alpha,
                             eps, relu_inputs, dtype, workspace, workspace_bytes);
    if (st != LISA_OK || empty) return st;
    if (!hQ || !hK || !hV || !hO) return LISA_ERR_INVALID_ARG;
    const size_t esz = (dtype == LISA_BF16) ? 2 : 4;
    const size_t bytes = (size_t)p.slices * (size_t)p.n * (size_t)p.D * esz;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(dQ, hQ, bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(dK, hK, bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(dV, hV, bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return LISA_ERR_CUDA;
    st = launch(p, cs);
    if (st != LISA_OK) return st;
    if (cudaMemcpyAsync(hO, dO, bytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return LISA_ERR_CUDA;
    return LISA_OK;
}

namespace {

// Number of kernels and their names for one problem; 0 / NULL for sizes or
// weights lisa_forward would reject.
int stage_info(int B, int heads, int H, int W, int d_h, int T, int dtype, const lisa_weights *wts,
               int stage, const char **name) {
    if (name) *name = nullptr;
    if (!wts || check_sizes(B, heads, H, W, d_h, d_h, T, dtype) != LISA_OK) return 0;
    const long long slices = (long long)B * heads, n = (long long)H * W;
    if (slices == 0 || n == 0) return 0;
    const Plan pl = make_plan((int)slices, (int)n, d_h, effective_T(T), dtype, weights_mode(wts), wts->hidden);
    if (pl.family == kFamilyTc) {
        if (name) *name = tc_stage_name(pl.chunks, pl.cluster, pl.chunk, stage);
        return tc_num_stages(pl.chunks, pl.cluster, pl.chunk);
    }
    if (name && stage >= 0 && stage < kSimtStages) *name = kSimtStageNames[stage];
    return kSimtStages;
}

}  // namespace

extern "C" int lisa_num_stages(int B, int heads, int H, int W, int d_h, int T, int dtype,
                               const lisa_weights *wts) {
    return stage_info(B, heads, H, W, d_h, T, dtype, wts, -1, nullptr);
}

extern "C" const char *lisa_stage_name(int B, int heads, int H, int W, int d_h, int T, int dtype,
                                       const lisa_weights *wts, int stage) {
    const char *name = nullptr;
    stage_info(B, heads, H, W, d_h, T, dtype, wts, stage, &name);
    return name;
}

extern "C" lisa_status lisa_forward_stage(int stage, const void *Q, const void *K, const void *V,
                                          void *O, int B, int heads, int H, int W, int d_h,
                                          int d_v, int T, const lisa_weights *wts,
                                          const float *alpha, float eps, int relu_inputs,
                                          int dtype, void *workspace, size_t workspace_bytes,
                                          void *stream) {
    Problem p;
    bool empty;
    lisa_status st = prepare(p, empty, Q, K, V, O, B, heads, H, W, d_h, d_v, T, wts, alpha, eps,
                             relu_inputs, dtype, workspace, workspace_bytes);
    if (st != LISA_OK) return st;
    if (relu_inputs == 2) return LISA_ERR_INVALID_ARG;   // the stage list describes the ReLU chains
    if (stage < 0 || stage >= lisa_num_stages(B, heads, H, W, d_h, T, dtype, wts))
        return LISA_ERR_INVALID_ARG;
    if (empty) return LISA_OK;
    return launch(p, static_cast<cudaStream_t>(stream), stage);
}

extern "C" const char *lisa_status_string(int status) {
    switch (status) {
        case LISA_OK: return "LISA_OK";
        case LISA_ERR_INVALID_ARG: return "LISA_ERR_INVALID_ARG: invalid argument";
        case LISA_ERR_UNSUPPORTED: return "LISA_ERR_UNSUPPORTED: unsupported size or mode";
        case LISA_ERR_WORKSPACE: return "LISA_ERR_WORKSPACE: workspace missing or too small";
        case LISA_ERR_CUDA: return "LISA_ERR_CUDA: CUDA launch or runtime error";
        case LISA_ERR_TIMEOUT: return "LISA_ERR_TIMEOUT: a bounded device wait gave up";
        default: return "unknown lisa_status";
    }
}

extern "C" int lisa_abi_version(void) { return 104; }

extern "C" lisa_status lisa_query_status(const void *workspace, void *stream) {
    if (!workspace || !aligned16(workspace)) return LISA_ERR_INVALID_ARG;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int word = 0;
    // the error word is the first int of every forward workspace (Plan::off_err == 0)
    if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess)
        return LISA_ERR_CUDA;
    return word == 0 ? LISA_OK : LISA_ERR_TIMEOUT;
}

extern "C" lisa_status lisa_forward_resident(const void *Q, const void *K, const void *V, void *O,
                                             int B, int heads, int H, int W, int d_h, int d_v, int T,
                                             const lisa_weights *wts, const float *alpha, float eps,
                                             int relu_inputs, int dtype, void *workspace,
                                             size_t workspace_bytes, void *stream) {
    Problem p;
    bool empty;
    lisa_status st = prepare(p, empty, Q, K, V, O, B, heads, H, W, d_h, d_v, T, wts, alpha, eps,
                             relu_inputs, dtype, workspace, workspace_bytes);
    if (st != LISA_OK || empty) return st;
    if (p.family != kFamilyTc ||
        !tc_resident_applies(p.slices, H, W, d_h, dtype, p.wmode, p.untruncated, p.relu))
        return LISA_ERR_UNSUPPORTED;
    p.resident = 1;
    return launch(p, static_cast<cudaStream_t>(stream));
}

extern "C" lisa_status lisa_selftest_wait_timeout(long long cycles, void *workspace, size_t workspace_bytes,
                                                  void *stream) {
    if (cycles < 0 || !workspace || !aligned16(workspace) || workspace_bytes < sizeof(int))
        return LISA_ERR_INVALID_ARG;
    return launch_wait_selftest(static_cast<int *>(workspace), cycles, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? LISA_OK
               : LISA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// lisa_forward_noalloc -- the layer for callers that may not allocate device
// memory.  Some hosts of this code cannot call cudaMalloc when they run it:
// an operator plugged into an inference engine or framework that owns all
// device memory through its own pool and plans it before execution, or a
// serving loop that cannot afford the device-wide synchronisation cudaFree
// implies.  This entry point needs no workspace from them: it runs in a
// scratch array compiled into the library (LISA_NOALLOC_SCRATCH_BYTES on
// every device that loads the library, held until the process exits).  The
// array's device address is looked up once per device, on the first call
// with that device current, and kept for the life of the process.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[LISA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// In host code g_noalloc_scratch names a host-side shadow, not device memory;
// its device address comes from the runtime, looked up once per device with
// that device current.
lisa_status noalloc_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LISA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LISA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LISA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return LISA_OK;
}

}  // namespace

extern "C" lisa_status lisa_forward_noalloc(const void *Q, const void *K, const void *V, void *O,
                                            int B, int heads, int H, int W, int d_h, int d_v,
                                            int T, const lisa_weights *wts, const float *alpha,
                                            float eps, int relu_inputs, int dtype, void *stream) {
    lisa_status st = check_sizes(B, heads, H, W, d_h, d_v, T, dtype);
    if (st != LISA_OK) return st;
    const long long slices = (long long)B * heads, n = (long long)H * W;
    const size_t need = (slices == 0 || n == 0 || !wts)
                            ? 0
                            : make_plan((int)slices, (int)n, d_h, effective_T(T),
                                        family_dtype(dtype, relu_inputs), weights_mode(wts), wts->hidden)
                                  .total;
    if (need > (size_t)LISA_NOALLOC_SCRATCH_BYTES) return LISA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        st = noalloc_scratch(&scratch);
        if (st != LISA_OK) return st;
    }
    return lisa_forward(Q, K, V, O, B, heads, H, W, d_h, d_v, T, wts, alpha, eps, relu_inputs, dtype,
                        scratch, (size_t)LISA_NOALLOC_SCRATCH_BYTES, stream);
}

// ---------------------------------------------------------------------------
// lisa_backward -- gradients of the layer (see include/lisa.h).
// ---------------------------------------------------------------------------
namespace {

constexpr int kBwdTokensPerBlock = 32;   // per-token kernels: 8 warps x 4 tokens

struct BwdPlan {
    Plan fwd;   // SIMT statistics partials (s, K^T V, K^T Q~) and s
    int ntile;  // 8 x 8 tiles per slice (the tiled token pass)
    Plan tc;    // bf16, d = 64: the tensor-core split statistics' own region (tc.total == 0 otherwise)
    size_t off_tc, off_tcdub;
    int nh, nblk;
    size_t off_mred, off_uk, off_ubar, off_ubart, off_dub, off_lstat, off_dalp, off_dsp, off_dm, off_du1,
        off_dmt, off_du1t, off_dsr, off_dals, off_dkp, off_bimg, off_ubimg;
    // adaptive weights only
    size_t off_ukn, off_wtok, off_dz, off_h, off_da, off_dxm, off_dukp, off_pw1, off_pb1, off_pw2, off_pb2,
        off_ukimg, off_w1img, off_ukimgt;
    size_t total;
};

// The backward always runs the SIMT statistics kernels; its own buffers
// follow the forward plan's.  hidden > 0: the adaptive weights' buffers too.
BwdPlan make_bwd_plan(int slices, int H, int W, int D, int T, int hidden, int dtype) {
    const int n = H * W;
    BwdPlan b{};
    b.fwd = make_plan(slices, n, D, T, LISA_F32, LISA_W_FIXED, 0);   // SIMT family, any dtype
    b.nh = T > 1 ? T - 1 : 1;
    b.nblk = (n + kBwdTokensPerBlock - 1) / kBwdTokensPerBlock;
    b.ntile = ((H + 7) / 8) * ((W + 7) / 8);
    const size_t nparts = (size_t)(b.nblk > b.ntile ? b.nblk : b.ntile);   // ds partials of either token pass
    const size_t S = (size_t)slices, C = (size_t)b.fwd.chunks, d = (size_t)D, dd = d * d, N = (size_t)n;
    size_t off = b.fwd.total;
    b.off_mred = off;  off = align_up(off + S * dd * sizeof(float));
    b.off_uk = off;    off = align_up(off + S * b.nh * dd * sizeof(float));
    b.off_ubar = off;  off = align_up(off + S * dd * sizeof(float));
    b.off_ubart = off; off = align_up(off + S * dd * sizeof(float));
    b.off_dub = off;   off = align_up(off + S * C * dd * sizeof(float));
    b.off_lstat = off; off = align_up(off + S * N * 4 * sizeof(float));
    b.off_dalp = off;  off = align_up(off + S * b.nblk * sizeof(float));
    b.off_dsp = off;   off = align_up(off + S * nparts * d * sizeof(float));
    b.off_dm = off;    off = align_up(off + S * dd * sizeof(float));
    b.off_du1 = off;   off = align_up(off + S * dd * sizeof(float));
    b.off_dmt = off;   off = align_up(off + S * dd * sizeof(float));
    b.off_du1t = off;  off = align_up(off + S * dd * sizeof(float));
    b.off_dsr = off;   off = align_up(off + S * d * sizeof(float));
    b.off_dals = off;  off = align_up(off + S * sizeof(float));
    b.off_dkp = off;   off = align_up(off + S * N * d * sizeof(float));
    b.off_bimg = off;  off = align_up(off + S * 5 * dd * sizeof(uint16_t));
    b.off_ubimg = off; off = align_up(off + S * 2 * dd * sizeof(uint16_t));
    if (dtype == LISA_BF16 && D == 64) {
        b.tc = make_plan(slices, n, D, T, LISA_BF16, LISA_W_FIXED, 0);
        b.off_tc = off;
        off = align_up(off + b.tc.total);
        b.off_tcdub = off;   // dUbar's cluster partials, laid out like tc_part
        off = align_up(off + S * (size_t)(b.tc.chunks / b.tc.cluster) * 128 * 64 * sizeof(float));
    }
    if (hidden > 0) {
        const size_t Tz = (size_t)T, Hd = (size_t)hidden, nk = (size_t)b.nh;
        b.off_ukn = off;  off = align_up(off + S * nk * dd * sizeof(float));
        b.off_wtok = off; off = align_up(off + S * N * Tz * sizeof(float));
        b.off_dz = off;   off = align_up(off + S * N * Tz * sizeof(float));
        b.off_h = off;    off = align_up(off + S * N * Hd * sizeof(float));
        b.off_da = off;   off = align_up(off + S * N * Hd * sizeof(float));
        b.off_dxm = off;  off = align_up(off + S * N * 2 * d * sizeof(float));
        b.off_dukp = off; off = align_up(off + S * C * nk * dd * sizeof(float));
        b.off_pw1 = off;  off = align_up(off + S * C * Hd * 2 * d * sizeof(float));
        b.off_pb1 = off;  off = align_up(off + S * C * Hd * sizeof(float));
        b.off_pw2 = off;  off = align_up(off + S * C * Tz * Hd * sizeof(float));
        b.off_pb2 = off;  off = align_up(off + S * C * Tz * sizeof(float));
        b.off_ukimg = off; off = align_up(off + S * nk * 2 * 64 * 72 * sizeof(uint16_t));
        b.off_w1img = off; off = align_up(off + 2 * LISA_MAX_HIDDEN * 136 * sizeof(uint16_t));
        b.off_ukimgt = off; off = align_up(off + S * nk * 64 * 72 * sizeof(uint16_t));
    }
    b.total = off;
    return b;
}

// Everything lisa_backward and lisa_backward_mlp share: checks, plan,
// workspace views, launch.  mg is non-null exactly for the adaptive weights.
lisa_status run_backward(const void *Q, const void *K, const void *V, const void *dO, void *dQ, void *dK,
                         void *dV, float *dalpha, const lisa_mlp_grads *mg, int B, int heads, int H, int W,
                         int d_h, int d_v, int T, const lisa_weights *wts, const float *alpha, float eps,
                         int relu_inputs, int dtype, void *workspace, size_t workspace_bytes, void *stream) {
    lisa_status st = check_sizes(B, heads, H, W, d_h, d_v, T, dtype);
    if (st != LISA_OK) return st;
    if (!(eps > 0.f) || !std::isfinite(eps)) return LISA_ERR_INVALID_ARG;
    if (relu_inputs < 0 || relu_inputs > 2) return LISA_ERR_INVALID_ARG;
    BwdProblem b{};
    st = resolve_weights(b.fwd, wts, T);
    if (st != LISA_OK) return st;
    const bool mlp = mg != nullptr;
    if (mlp && (!mg->dW1 || !mg->db1 || !mg->dW2 || !mg->db2)) return LISA_ERR_INVALID_ARG;
    const long long slices = (long long)B * heads, n = (long long)H * W;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (slices == 0 || n == 0) {   // nothing to differentiate: dalpha (and the MLP's gradients) = 0
        if (heads > 0) {
            if (!dalpha) return LISA_ERR_INVALID_ARG;
            if (cudaMemsetAsync(dalpha, 0, (size_t)heads * sizeof(float), cs) != cudaSuccess)
                return LISA_ERR_CUDA;
        }
        if (mlp) {
            const size_t hd = (size_t)b.fwd.hidden;
            if (cudaMemsetAsync(mg->dW1, 0, hd * 2 * d_h * sizeof(float), cs) != cudaSuccess ||
                cudaMemsetAsync(mg->db1, 0, hd * sizeof(float), cs) != cudaSuccess ||
                cudaMemsetAsync(mg->dW2, 0, (size_t)T * hd * sizeof(float), cs) != cudaSuccess ||
                cudaMemsetAsync(mg->db2, 0, (size_t)T * sizeof(float), cs) != cudaSuccess)
                return LISA_ERR_CUDA;
        }
        return LISA_OK;
    }
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV || !dalpha || !alpha) return LISA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) || !aligned16(dQ) ||
        !aligned16(dK) || !aligned16(dV))
        return LISA_ERR_INVALID_ARG;
    const size_t esz = (dtype == LISA_BF16) ? 2 : 4;
    const size_t bytes = (size_t)slices * (size_t)n * (size_t)d_h * esz;
    const void *ins[4] = {Q, K, V, dO};
    void *outs[3] = {dQ, dK, dV};
    for (void *o : outs) {
        for (const void *in : ins)
            if (overlaps(o, bytes, in, bytes)) return LISA_ERR_INVALID_ARG;
        if (overlaps(o, bytes, dalpha, (size_t)heads * sizeof(float))) return LISA_ERR_INVALID_ARG;
    }
    if (overlaps(dQ, bytes, dK, bytes) || overlaps(dQ, bytes, dV, bytes) || overlaps(dK, bytes, dV, bytes))
        return LISA_ERR_INVALID_ARG;
    if (overlaps(dalpha, (size_t)heads * sizeof(float), alpha, (size_t)heads * sizeof(float)))
        return LISA_ERR_INVALID_ARG;

    const BwdPlan pl = make_bwd_plan((int)slices, H, W, d_h, b.fwd.T, mlp ? b.fwd.hidden : 0, dtype);
    if (!workspace || workspace_bytes < pl.total) return LISA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return LISA_ERR_INVALID_ARG;
    fill_problem(b.fwd, pl.fwd, Q, K, V, nullptr, (int)slices, heads, H, W, d_h, relu_inputs, eps, alpha, dtype,
                 workspace);
    b.fwd.dtype = dtype;
    b.dO = dO;
    b.dQ = dQ;
    b.dK = dK;
    b.dV = dV;
    b.dalpha = dalpha;
    b.tpb = kBwdTokensPerBlock;
    b.nblk = pl.nblk;
    b.nh = pl.nh;
    char *ws = static_cast<char *>(workspace);
    auto f32 = [ws](size_t off) { return reinterpret_cast<float *>(ws + off); };
    b.Mred = f32(pl.off_mred);
    b.Uk = f32(pl.off_uk);
    b.Ubar = f32(pl.off_ubar);
    b.UbarT = f32(pl.off_ubart);
    b.dub_part = f32(pl.off_dub);
    b.lstat = f32(pl.off_lstat);
    b.dal_part = f32(pl.off_dalp);
    b.ds_part = f32(pl.off_dsp);
    b.dM = f32(pl.off_dm);
    b.dU1 = f32(pl.off_du1);
    b.dMT = f32(pl.off_dmt);
    b.dU1T = f32(pl.off_du1t);
    b.ds_red = f32(pl.off_dsr);
    b.dal_slice = f32(pl.off_dals);
    b.dk_part = f32(pl.off_dkp);
    b.bimg = reinterpret_cast<uint16_t *>(ws + pl.off_bimg);
    b.ubimg = reinterpret_cast<uint16_t *>(ws + pl.off_ubimg);
    if (pl.tc.total > 0 && relu_inputs != 2) {
        // the statistics on the tensor cores; their kernels report into the
        // backward's own error word
        b.tc_stats = 1;
        b.tcfwd = b.fwd;
        fill_problem(b.tcfwd, pl.tc, Q, K, V, nullptr, (int)slices, heads, H, W, d_h, relu_inputs, eps, alpha,
                     dtype, ws + pl.off_tc);
        b.tcfwd.err = b.fwd.err;
        b.tcfwd.wmode = LISA_W_FIXED;   // statistics only: the walk weights play no part
        b.tcdub = f32(pl.off_tcdub);
        b.tc_dub = (!mlp && !b.fwd.untruncated) ? 1 : 0;
        b.ntile = pl.ntile;   // the tiled token pass
    }
    if (mlp) {
        b.mlp = 1;
        b.Ukn = f32(pl.off_ukn);
        b.wtok = f32(pl.off_wtok);
        b.dzbuf = f32(pl.off_dz);
        b.hbuf = f32(pl.off_h);
        b.dabuf = f32(pl.off_da);
        b.dxm = f32(pl.off_dxm);
        b.dukp = f32(pl.off_dukp);
        b.pw1 = f32(pl.off_pw1);
        b.pb1 = f32(pl.off_pb1);
        b.pw2 = f32(pl.off_pw2);
        b.pb2 = f32(pl.off_pb2);
        b.ukimg = reinterpret_cast<uint16_t *>(ws + pl.off_ukimg);
        b.w1img = reinterpret_cast<uint16_t *>(ws + pl.off_w1img);
        b.ukimgT = reinterpret_cast<uint16_t *>(ws + pl.off_ukimgt);
        b.dW1 = mg->dW1;
        b.db1 = mg->db1;
        b.dW2 = mg->dW2;
        b.db2 = mg->db2;
    }
    return launch_bwd(b, cs) == cudaSuccess ? LISA_OK : LISA_ERR_CUDA;
}

}  // namespace

extern "C" size_t lisa_backward_workspace_bytes(int B, int heads, int H, int W, int d_h, int d_v, int T,
                                                int dtype) {
    if (check_sizes(B, heads, H, W, d_h, d_v, T, dtype) != LISA_OK) return 0;
    const long long slices = (long long)B * heads, n = (long long)H * W;
    if (slices == 0 || n == 0) return 0;
    return make_bwd_plan((int)slices, H, W, d_h, effective_T(T), 0, dtype).total;
}

extern "C" lisa_status lisa_backward(const void *Q, const void *K, const void *V, const void *dO, void *dQ,
                                     void *dK, void *dV, float *dalpha, int B, int heads, int H, int W,
                                     int d_h, int d_v, int T, const lisa_weights *wts, const float *alpha,
                                     float eps, int relu_inputs, int dtype, void *workspace,
                                     size_t workspace_bytes, void *stream) {
    if (!wts) return LISA_ERR_INVALID_ARG;
    if (wts->mode == LISA_W_MLP) {   // sizes still checked first: T or d out of range stays UNSUPPORTED
        const lisa_status st = check_sizes(B, heads, H, W, d_h, d_v, T, dtype);
        return st != LISA_OK ? st : LISA_ERR_UNSUPPORTED;
    }
    return run_backward(Q, K, V, dO, dQ, dK, dV, dalpha, nullptr, B, heads, H, W, d_h, d_v, T, wts, alpha, eps,
                        relu_inputs, dtype, workspace, workspace_bytes, stream);
}

extern "C" size_t lisa_backward_mlp_workspace_bytes(int B, int heads, int H, int W, int d_h, int d_v, int T,
                                                    int hidden, int dtype) {
    if (check_sizes(B, heads, H, W, d_h, d_v, T, dtype) != LISA_OK) return 0;
    if (T < 1 || T > LISA_MAX_T_MLP || hidden < 1 || hidden > LISA_MAX_HIDDEN) return 0;
    const long long slices = (long long)B * heads, n = (long long)H * W;
    if (slices == 0 || n == 0) return 0;
    return make_bwd_plan((int)slices, H, W, d_h, T, hidden, dtype).total;
}

extern "C" lisa_status lisa_backward_mlp(const void *Q, const void *K, const void *V, const void *dO, void *dQ,
                                         void *dK, void *dV, float *dalpha, const lisa_mlp_grads *mgrads,
                                         int B, int heads, int H, int W, int d_h, int d_v, int T,
                                         const lisa_weights *wts, const float *alpha, float eps,
                                         int relu_inputs, int dtype, void *workspace, size_t workspace_bytes,
                                         void *stream) {
    if (!wts || wts->mode != LISA_W_MLP || !mgrads) return LISA_ERR_INVALID_ARG;
    return run_backward(Q, K, V, dO, dQ, dK, dV, dalpha, mgrads, B, heads, H, W, d_h, d_v, T, wts, alpha, eps,
                        relu_inputs, dtype, workspace, workspace_bytes, stream);
}
