// gma_api.cu -- the C ABI of libgma.so: argument validation, workspace
// sizing and dispatch to the kernel families.  Declarations and the contract
// of every entry point are in include/gma.h.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "gma_internal.h"

namespace {

using gma::Problem;

bool valid_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

bool shape_ok(int B, int H, int N, int d_r, int d_v, int K, bool need_dv) {
    if (B < 1 || H < 1 || N < 1 || K < 1 || K > 128) return false;
    if (!valid_dim(d_r)) return false;
    if (need_dv && !valid_dim(d_v)) return false;
    // element offsets must fit the 64-bit index arithmetic comfortably and
    // B*H must fit a grid dimension
    if ((long long)B * H > 65535LL) return false;
    if ((long long)B * H * N > (1LL << 40)) return false;
    return true;
}

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    auto pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

int choose_path(const Problem &p, int causal, const gma_options *opt) {
    int path = opt ? opt->path : GMA_PATH_AUTO;
    if (path == GMA_PATH_SIMT) return GMA_PATH_SIMT;
    const bool tc64 = causal >= 0 && gma::tc_supported(p, causal);
    const bool tc = tc64 || (causal >= 0 && gma::tc128_supported(p, causal));
    if (path == GMA_PATH_TC) return tc ? GMA_PATH_TC : -1;
    // the single-pass kernel is a causal kernel of the 64-wide family; the
    // bidirectional tensor-core calls already keep Gamma on chip
    if (path == GMA_PATH_TC_SINGLE_PASS) {
        if (causal == 1) return tc64 ? GMA_PATH_TC_SINGLE_PASS : -1;
        return tc ? GMA_PATH_TC : -1;
    }
    if (path != GMA_PATH_AUTO) return -1;
    return tc ? GMA_PATH_TC : GMA_PATH_SIMT;
}

// The causal chunk length of a kernel family: the tensor-core scan runs in
// chunks of 128 tokens (its tile), the CUDA-core scan in chunks of
// kSimtCausalChunk.  options->chunk must be 0 (the family's value) or exactly
// that value; other lengths are not built.
int family_chunk(int path) { return path == GMA_PATH_SIMT ? gma::kSimtCausalChunk : 128; }
bool chunk_ok(int path, int causal, const gma_options *opt) {
    if (!opt || opt->chunk == 0 || causal != 1) return true;
    return opt->chunk == family_chunk(path);
}

size_t workspace_for(const Problem &p, int causal, const gma_options *opt, int path) {
    int splits = opt ? opt->splits : 0;
    if (path == GMA_PATH_TC_SINGLE_PASS) return gma::tc_scan_workspace(p, splits);
    if (path == GMA_PATH_TC)
        return gma::tc128_supported(p, causal) ? gma::tc128_workspace(p, splits) : gma::tc_workspace(p, causal, splits);
    return gma::simt_layout(p, causal, splits).total;
}

// The decode step and the routing statistics have only a CUDA-core implementation.
bool simt_only(const gma_options *opt) {
    return !opt || opt->path == GMA_PATH_AUTO || opt->path == GMA_PATH_SIMT;
}

// Kernel family of the latent-memory calls (latent memory, read from a memory,
// carried-prefix causal forward): GMA_PATH_AUTO and GMA_PATH_SIMT keep them on
// the CUDA cores (fp32 accuracy for state carried from call to call);
// GMA_PATH_TC runs them on the tensor-core kernels where those support the
// sizes, else -1.
int memory_path(const Problem &p, int causal, const gma_options *opt) {
    const int path = opt ? opt->path : GMA_PATH_AUTO;
    if (path == GMA_PATH_AUTO || path == GMA_PATH_SIMT) return GMA_PATH_SIMT;
    if (path == GMA_PATH_TC) return gma::tc_supported(p, causal) ? GMA_PATH_TC : -1;
    if (path == GMA_PATH_TC_SINGLE_PASS)
        return !gma::tc_supported(p, causal) ? -1 : causal == 1 ? GMA_PATH_TC_SINGLE_PASS : GMA_PATH_TC;
    return -1;
}

gma::StageClock clock_for(const gma_options *opt, cudaStream_t s) {
    gma::StageClock c;
    if (opt && opt->stage_events && opt->n_stage_events > 0) {
        c.events = opt->stage_events;
        c.n = opt->n_stage_events;
    }
    c.stream = s;
    return c;
}

gma_status finish(cudaError_t err, const gma_options *opt, void *ws, cudaStream_t s) {
    if (err != cudaSuccess) {
        (void)cudaGetLastError();  // clear a sticky launch error for the caller
        return GMA_ERR_CUDA;
    }
    if (opt && opt->sync_status) return gma_last_device_status(ws, s);
    return GMA_OK;
}

gma_status forward(const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype,
                   const float *mu, const float *sigma2, const float *log_pi, float eps,
                   void *O, int B, int H, int N, int d_r, int d_v, int K,
                   const gma_options *options, void *workspace, size_t workspace_bytes,
                   void *stream, int causal) {
    if (!Q_X || !K_X || !V_X || !mu || !sigma2 || !log_pi || !O || !workspace)
        return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    if (!aligned16(Q_X) || !aligned16(K_X) || !aligned16(V_X) || !aligned16(O) || !aligned16(mu) ||
        !aligned16(sigma2))
        return GMA_ERR_INVALID_ARG;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (options && (options->chunk < 0 || options->splits < 0)) return GMA_ERR_INVALID_ARG;

    Problem p;
    p.Q = Q_X; p.Kx = K_X; p.V = V_X; p.mu = mu; p.sigma2 = sigma2; p.log_pi = log_pi;
    p.O = O; p.dtype = dtype; p.eps = eps;
    p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    p.o_bf16 = options && options->o_bf16;
    p.test_stall = options && options->test_stall;

    const size_t es = dtype == GMA_F32 ? 4 : 2;
    const size_t nr = es * (size_t)B * H * N * d_r, nv = es * (size_t)B * H * N * d_v;
    const size_t no = (p.o_bf16 ? 2 : 4) * (size_t)B * H * N * d_v;
    const int path = choose_path(p, causal, options);
    if (path < 0 || !chunk_ok(path, causal, options)) return GMA_ERR_UNSUPPORTED_SHAPE;
    const size_t need = workspace_for(p, causal, options, path);
    if (workspace_bytes < need) return GMA_ERR_WORKSPACE_TOO_SMALL;
    if (overlaps(O, no, Q_X, nr) || overlaps(O, no, K_X, nr) || overlaps(O, no, V_X, nv) ||
        overlaps(O, no, workspace, need) || overlaps(workspace, need, Q_X, nr) ||
        overlaps(workspace, need, K_X, nr) || overlaps(workspace, need, V_X, nv))
        return GMA_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int splits = options ? options->splits : 0;
    gma::StageClock clk = clock_for(options, s);
    cudaError_t err;
    if (path == GMA_PATH_TC_SINGLE_PASS)
        err = gma::tc_causal_1pass(p, splits, workspace, s, clk);
    else if (path == GMA_PATH_TC && gma::tc128_supported(p, causal))
        err = causal ? gma::tc128_causal(p, splits, workspace, s, clk) : gma::tc128_bidir(p, splits, workspace, s, clk);
    else if (path == GMA_PATH_TC)
        err = causal ? gma::tc_causal(p, splits, workspace, s, clk) : gma::tc_bidir(p, splits, workspace, s, clk);
    else
        err = causal ? gma::simt_causal(p, workspace, s, clk) : gma::simt_bidir(p, splits, workspace, s, clk);
    return finish(err, options, workspace, s);
}

gma_status backward(const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype, const float *mu,
                    const float *sigma2, const float *log_pi, float eps, const float *dO, float *dQ_X,
                    float *dK_X, float *dV_X, float *dmu, float *dsigma2, float *dlog_pi, int B, int H, int N,
                    int d_r, int d_v, int K, const gma_options *options, void *workspace,
                    size_t workspace_bytes, void *stream, int causal) {
    if (!Q_X || !K_X || !V_X || !mu || !sigma2 || !log_pi || !dO || !dQ_X || !dK_X || !dV_X || !dmu ||
        !dsigma2 || !dlog_pi || !workspace)
        return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    if (!aligned16(Q_X) || !aligned16(K_X) || !aligned16(V_X) || !aligned16(mu) || !aligned16(sigma2) ||
        !aligned16(dO) || !aligned16(dQ_X) || !aligned16(dK_X) || !aligned16(dV_X) || !aligned16(dmu) ||
        !aligned16(dsigma2) || reinterpret_cast<uintptr_t>(dlog_pi) % 4 != 0)
        return GMA_ERR_INVALID_ARG;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (options && options->splits < 0) return GMA_ERR_INVALID_ARG;
    if (options && (options->o_bf16 || (options->path != GMA_PATH_AUTO && options->path != GMA_PATH_SIMT)))
        return GMA_ERR_UNSUPPORTED_SHAPE;
    if (options && options->chunk < 0) return GMA_ERR_INVALID_ARG;
    if (!chunk_ok(GMA_PATH_SIMT, causal, options)) return GMA_ERR_UNSUPPORTED_SHAPE;

    Problem p;
    p.Q = Q_X; p.Kx = K_X; p.V = V_X; p.mu = mu; p.sigma2 = sigma2; p.log_pi = log_pi;
    p.dtype = dtype; p.eps = eps;
    p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    const int splits = options ? options->splits : 0;
    const size_t need = gma::backward_workspace(p, causal, splits);
    if (workspace_bytes < need) return GMA_ERR_WORKSPACE_TOO_SMALL;

    const size_t es = dtype == GMA_F32 ? 4 : 2;
    const size_t rows = (size_t)B * H * N;
    const size_t nr = es * rows * d_r, nv = es * rows * d_v;
    const size_t fr = 4 * rows * d_r, fv = 4 * rows * d_v, fp = 4 * (size_t)H * K * d_r, fl = 4 * (size_t)H * K;
    const void *in[] = {Q_X, K_X, V_X, dO, mu, sigma2, log_pi, workspace};
    const size_t nin[] = {nr, nr, nv, fv, fp, fp, fl, need};
    const void *out[] = {dQ_X, dK_X, dV_X, dmu, dsigma2, dlog_pi};
    const size_t nout[] = {fr, fr, fv, fp, fp, fl};
    for (int a = 0; a < 6; ++a) {
        for (int b = 0; b < 8; ++b)
            if (overlaps(out[a], nout[a], in[b], nin[b])) return GMA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 6; ++b)
            if (overlaps(out[a], nout[a], out[b], nout[b])) return GMA_ERR_INVALID_ARG;
    }
    if (overlaps(workspace, need, Q_X, nr) || overlaps(workspace, need, K_X, nr) ||
        overlaps(workspace, need, V_X, nv) || overlaps(workspace, need, dO, fv))
        return GMA_ERR_INVALID_ARG;

    gma::BackwardArgs g;
    g.dO = dO; g.dQ = dQ_X; g.dK = dK_X; g.dV = dV_X; g.dmu = dmu; g.dsigma2 = dsigma2; g.dlog_pi = dlog_pi;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gma::StageClock clk = clock_for(options, s);
    const cudaError_t err = causal ? gma::simt_backward_causal(p, g, workspace, s, clk)
                                   : gma::simt_backward_bidir(p, g, splits, workspace, s, clk);
    return finish(err, options, workspace, s);
}

}  // namespace

extern "C" {

size_t gma_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype,
                          int causal, const gma_options *options) {
    if (causal < -1 || causal > 1) return 0;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return 0;
    if (!shape_ok(B, H, N, d_r, d_v, K, causal >= 0)) return 0;
    Problem p;
    p.dtype = dtype; p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = causal >= 0 ? d_v : 16; p.K = K;
    int path = choose_path(p, causal, options);
    if (path < 0 || !chunk_ok(path, causal, options)) return 0;
    return workspace_for(p, causal, options, path);
}

gma_status gma_responsibilities(const void *X, gma_dtype dtype, const float *mu,
                                const float *sigma2, const float *log_pi, float *Gamma,
                                int B, int H, int N, int d_r, int K,
                                const gma_options *options, void *workspace,
                                size_t workspace_bytes, void *stream) {
    if (!X || !mu || !sigma2 || !log_pi || !Gamma || !workspace) return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    if (!shape_ok(B, H, N, d_r, 16, K, false)) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (options && (options->path != GMA_PATH_AUTO && options->path != GMA_PATH_SIMT))
        return GMA_ERR_UNSUPPORTED_SHAPE;
    Problem p;
    p.Q = X; p.mu = mu; p.sigma2 = sigma2; p.log_pi = log_pi; p.O = Gamma; p.dtype = dtype;
    p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = 16; p.K = K;
    const size_t need = gma::simt_layout(p, -1, 0).total;
    if (workspace_bytes < need) return GMA_ERR_WORKSPACE_TOO_SMALL;
    const size_t es = dtype == GMA_F32 ? 4 : 2;
    const size_t nx = es * (size_t)B * H * N * d_r, ng = sizeof(float) * (size_t)B * H * N * K;
    if (overlaps(Gamma, ng, X, nx) || overlaps(Gamma, ng, workspace, need) ||
        overlaps(workspace, need, X, nx))
        return GMA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gma::StageClock clk = clock_for(options, s);
    return finish(gma::simt_responsibilities(p, workspace, s, clk), options, workspace, s);
}

gma_status gma_forward_bidir(const void *Q_X, const void *K_X, const void *V_X,
                             gma_dtype dtype, const float *mu, const float *sigma2,
                             const float *log_pi, float eps, void *O,
                             int B, int H, int N, int d_r, int d_v, int K,
                             const gma_options *options, void *workspace,
                             size_t workspace_bytes, void *stream) {
    return forward(Q_X, K_X, V_X, dtype, mu, sigma2, log_pi, eps, O, B, H, N, d_r, d_v, K,
                   options, workspace, workspace_bytes, stream, 0);
}

gma_status gma_forward_causal(const void *Q_X, const void *K_X, const void *V_X,
                              gma_dtype dtype, const float *mu, const float *sigma2,
                              const float *log_pi, float eps, void *O,
                              int B, int H, int N, int d_r, int d_v, int K,
                              const gma_options *options, void *workspace,
                              size_t workspace_bytes, void *stream) {
    return forward(Q_X, K_X, V_X, dtype, mu, sigma2, log_pi, eps, O, B, H, N, d_r, d_v, K,
                   options, workspace, workspace_bytes, stream, 1);
}

size_t gma_backward_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype,
                                   int causal, const gma_options *options) {
    if ((causal != 0 && causal != 1) || (dtype != GMA_F32 && dtype != GMA_BF16)) return 0;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return 0;
    if (options && (options->splits < 0 || options->chunk < 0 || options->o_bf16 ||
                    (options->path != GMA_PATH_AUTO && options->path != GMA_PATH_SIMT)))
        return 0;
    if (!chunk_ok(GMA_PATH_SIMT, causal, options)) return 0;
    Problem p;
    p.dtype = dtype; p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    return gma::backward_workspace(p, causal, options ? options->splits : 0);
}

gma_status gma_backward_bidir(const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype,
                              const float *mu, const float *sigma2, const float *log_pi, float eps,
                              const float *dO, float *dQ_X, float *dK_X, float *dV_X, float *dmu,
                              float *dsigma2, float *dlog_pi, int B, int H, int N, int d_r, int d_v,
                              int K, const gma_options *options, void *workspace,
                              size_t workspace_bytes, void *stream) {
    return backward(Q_X, K_X, V_X, dtype, mu, sigma2, log_pi, eps, dO, dQ_X, dK_X, dV_X, dmu, dsigma2, dlog_pi,
                    B, H, N, d_r, d_v, K, options, workspace, workspace_bytes, stream, 0);
}

gma_status gma_backward_causal(const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype,
                               const float *mu, const float *sigma2, const float *log_pi, float eps,
                               const float *dO, float *dQ_X, float *dK_X, float *dV_X, float *dmu,
                               float *dsigma2, float *dlog_pi, int B, int H, int N, int d_r, int d_v,
                               int K, const gma_options *options, void *workspace,
                               size_t workspace_bytes, void *stream) {
    return backward(Q_X, K_X, V_X, dtype, mu, sigma2, log_pi, eps, dO, dQ_X, dK_X, dV_X, dmu, dsigma2, dlog_pi,
                    B, H, N, d_r, d_v, K, options, workspace, workspace_bytes, stream, 1);
}

size_t gma_latent_memory_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype,
                                        const gma_options *options) {
    if (dtype != GMA_F32 && dtype != GMA_BF16) return 0;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return 0;
    if (options && options->splits < 0) return 0;
    Problem p;
    p.dtype = dtype; p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    const int path = memory_path(p, 0, options), splits = options ? options->splits : 0;
    if (path < 0) return 0;
    return path == GMA_PATH_TC ? gma::tc_workspace(p, 0, splits) : gma::simt_layout(p, 2, splits).total;
}

gma_status gma_latent_memory(const void *K_X, const void *V_X, gma_dtype dtype, const float *mu,
                             const float *sigma2, const float *log_pi, float *Vt, float *Z,
                             int B, int H, int N, int d_r, int d_v, int K,
                             const gma_options *options, void *workspace, size_t workspace_bytes,
                             void *stream) {
    if (!K_X || !V_X || !mu || !sigma2 || !log_pi || !Vt || !Z || !workspace) return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    if (!aligned16(K_X) || !aligned16(V_X) || !aligned16(Vt) || !aligned16(Z) || !aligned16(mu) ||
        !aligned16(sigma2))
        return GMA_ERR_INVALID_ARG;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (options && options->splits < 0) return GMA_ERR_INVALID_ARG;
    Problem p;
    p.Kx = K_X; p.V = V_X; p.mu = mu; p.sigma2 = sigma2; p.log_pi = log_pi; p.dtype = dtype;
    p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    const int splits = options ? options->splits : 0;
    const int path = memory_path(p, 0, options);
    if (path < 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    const size_t need = path == GMA_PATH_TC ? gma::tc_workspace(p, 0, splits) : gma::simt_layout(p, 2, splits).total;
    if (workspace_bytes < need) return GMA_ERR_WORKSPACE_TOO_SMALL;
    const size_t es = dtype == GMA_F32 ? 4 : 2, rows = (size_t)B * H * N;
    const size_t nvt = 4 * (size_t)B * H * K * d_v, nz = 4 * (size_t)B * H * K;
    const void *in[] = {K_X, V_X, mu, sigma2, log_pi, workspace};
    const size_t nin[] = {es * rows * d_r, es * rows * d_v, 4 * (size_t)H * K * d_r, 4 * (size_t)H * K * d_r,
                          4 * (size_t)H * K, need};
    for (int a = 0; a < 6; ++a)
        if (overlaps(Vt, nvt, in[a], nin[a]) || overlaps(Z, nz, in[a], nin[a])) return GMA_ERR_INVALID_ARG;
    if (overlaps(Vt, nvt, Z, nz) || overlaps(workspace, need, K_X, nin[0]) || overlaps(workspace, need, V_X, nin[1]))
        return GMA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gma::StageClock clk = clock_for(options, s);
    const cudaError_t err = path == GMA_PATH_TC ? gma::tc_latent_memory(p, splits, Vt, Z, workspace, s, clk)
                                               : gma::simt_latent_memory(p, splits, Vt, Z, workspace, s, clk);
    return finish(err, options, workspace, s);
}

size_t gma_decode_workspace_size(int H, int d_r, int K) {
    if (!shape_ok(1, H, 1, d_r, 16, K, false)) return 0;
    return gma::decode_workspace(H, K, d_r);
}

gma_status gma_decode_step(const void *q, const void *k, const void *v, gma_dtype dtype,
                           const float *mu, const float *sigma2, const float *log_pi, float eps,
                           float *Vt, float *Z, float *o, int B, int H, int d_r, int d_v, int K,
                           const gma_options *options, void *workspace, size_t workspace_bytes,
                           void *stream) {
    if (!q || !k || !v || !mu || !sigma2 || !log_pi || !Vt || !Z || !o || !workspace) return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    const size_t es = dtype == GMA_F32 ? 4 : 2;
    // q, k, v are read element by element, Vt and o as float4
    const void *elem[] = {q, k, v};
    for (const void *ptr : elem)
        if (reinterpret_cast<uintptr_t>(ptr) % es != 0) return GMA_ERR_INVALID_ARG;
    const void *word[] = {mu, sigma2, log_pi, Z};
    for (const void *ptr : word)
        if (reinterpret_cast<uintptr_t>(ptr) % 4 != 0) return GMA_ERR_INVALID_ARG;
    if (!aligned16(Vt) || !aligned16(o)) return GMA_ERR_INVALID_ARG;
    if (!shape_ok(B, H, 1, d_r, d_v, K, true) || !simt_only(options) || (options && options->o_bf16))
        return GMA_ERR_UNSUPPORTED_SHAPE;
    Problem p;
    p.Q = q; p.Kx = k; p.V = v; p.mu = mu; p.sigma2 = sigma2; p.log_pi = log_pi; p.O = o;
    p.dtype = dtype; p.eps = eps;
    p.B = B; p.H = H; p.N = 1; p.d_r = d_r; p.d_v = d_v; p.K = K;
    const size_t need = gma::decode_workspace(H, K, d_r);
    if (workspace_bytes < need) return GMA_ERR_WORKSPACE_TOO_SMALL;
    const size_t bh = (size_t)B * H;
    const size_t nvt = 4 * bh * K * d_v, nz = 4 * bh * K, no = 4 * bh * d_v;
    const void *in[] = {q, k, v, mu, sigma2, log_pi, workspace};
    const size_t nin[] = {es * bh * d_r, es * bh * d_r, es * bh * d_v, 4 * (size_t)H * K * d_r,
                          4 * (size_t)H * K * d_r, 4 * (size_t)H * K, need};
    const void *out[] = {Vt, Z, o};
    const size_t nout[] = {nvt, nz, no};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 7; ++b)
            if (overlaps(out[a], nout[a], in[b], nin[b])) return GMA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlaps(out[a], nout[a], out[b], nout[b])) return GMA_ERR_INVALID_ARG;
    }
    for (int b = 0; b < 3; ++b)
        if (overlaps(workspace, need, in[b], nin[b])) return GMA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gma::StageClock clk = clock_for(options, s);
    return finish(gma::simt_decode_step(p, Vt, Z, workspace, s, clk), options, workspace, s);
}

size_t gma_routing_stats_workspace_size(int B, int H, int N, int d_r, int K, gma_dtype dtype) {
    if (dtype != GMA_F32 && dtype != GMA_BF16) return 0;
    if (!shape_ok(B, H, N, d_r, 16, K, false)) return 0;
    Problem p;
    p.dtype = dtype; p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = 16; p.K = K;
    return gma::stats_workspace(p);
}

gma_status gma_routing_stats(const void *X, gma_dtype dtype, const float *mu, const float *sigma2,
                             const float *log_pi, float *usage, int *counts, int *z, float *entropy,
                             int B, int H, int N, int d_r, int K, const gma_options *options,
                             void *workspace, size_t workspace_bytes, void *stream) {
    if (!X || !mu || !sigma2 || !log_pi || !usage || !counts || !workspace) return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(usage) || !aligned16(counts) || !aligned16(mu) || !aligned16(sigma2) ||
        reinterpret_cast<uintptr_t>(z) % 4 || reinterpret_cast<uintptr_t>(entropy) % 4)
        return GMA_ERR_INVALID_ARG;
    if (!shape_ok(B, H, N, d_r, 16, K, false) || !simt_only(options)) return GMA_ERR_UNSUPPORTED_SHAPE;
    Problem p;
    p.Q = X; p.mu = mu; p.sigma2 = sigma2; p.log_pi = log_pi; p.dtype = dtype;
    p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = 16; p.K = K;
    const size_t need = gma::stats_workspace(p);
    if (workspace_bytes < need) return GMA_ERR_WORKSPACE_TOO_SMALL;
    const size_t es = dtype == GMA_F32 ? 4 : 2, bh = (size_t)B * H;
    const void *in[] = {X, mu, sigma2, log_pi, workspace};
    const size_t nin[] = {es * bh * N * d_r, 4 * (size_t)H * K * d_r, 4 * (size_t)H * K * d_r, 4 * (size_t)H * K,
                          need};
    const void *out[] = {usage, counts, z, entropy};
    const size_t nout[] = {4 * bh * K, 4 * bh * K, z ? 4 * bh * N : 0, entropy ? 4 * bh : 0};
    for (int a = 0; a < 4; ++a) {
        if (!out[a]) continue;
        for (int b = 0; b < 5; ++b)
            if (overlaps(out[a], nout[a], in[b], nin[b])) return GMA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 4; ++b)
            if (out[b] && overlaps(out[a], nout[a], out[b], nout[b])) return GMA_ERR_INVALID_ARG;
    }
    if (overlaps(workspace, need, X, nin[0])) return GMA_ERR_INVALID_ARG;
    gma::StatsArgs a;
    a.usage = usage; a.counts = counts; a.z = z; a.entropy = entropy;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gma::StageClock clk = clock_for(options, s);
    return finish(gma::simt_routing_stats(p, a, workspace, s, clk), options, workspace, s);
}

size_t gma_read_memory_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype) {
    if (dtype != GMA_F32 && dtype != GMA_BF16) return 0;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return 0;
    Problem p;
    p.dtype = dtype; p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    const size_t simt = gma::simt_layout(p, 3, 0).total;
    const size_t tc = gma::tc_supported(p, 0) ? gma::tc_workspace(p, 0, 0) : 0;
    return simt > tc ? simt : tc;  // enough for either kernel family
}

gma_status gma_read_memory(const void *Q_X, gma_dtype dtype, const float *mu, const float *sigma2,
                           const float *log_pi, float eps, const float *Vt, const float *Z, void *O,
                           int B, int H, int N, int d_r, int d_v, int K, const gma_options *options,
                           void *workspace, size_t workspace_bytes, void *stream) {
    if (!Q_X || !mu || !sigma2 || !log_pi || !Vt || !Z || !O || !workspace) return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    if (!aligned16(Q_X) || !aligned16(Vt) || !aligned16(Z) || !aligned16(O) || !aligned16(mu) || !aligned16(sigma2))
        return GMA_ERR_INVALID_ARG;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return GMA_ERR_UNSUPPORTED_SHAPE;
    Problem p;
    p.Q = Q_X; p.mu = mu; p.sigma2 = sigma2; p.log_pi = log_pi; p.O = O; p.dtype = dtype; p.eps = eps;
    p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    p.o_bf16 = options && options->o_bf16;
    const int path = memory_path(p, 0, options);
    if (path < 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    const size_t need = path == GMA_PATH_TC ? gma::tc_workspace(p, 0, 0) : gma::simt_layout(p, 3, 0).total;
    if (workspace_bytes < need) return GMA_ERR_WORKSPACE_TOO_SMALL;
    const size_t es = dtype == GMA_F32 ? 4 : 2, rows = (size_t)B * H * N;
    const size_t no = (p.o_bf16 ? 2 : 4) * rows * d_v;
    const void *in[] = {Q_X, Vt, Z, mu, sigma2, log_pi, workspace};
    const size_t nin[] = {es * rows * d_r, 4 * (size_t)B * H * K * d_v, 4 * (size_t)B * H * K,
                          4 * (size_t)H * K * d_r, 4 * (size_t)H * K * d_r, 4 * (size_t)H * K, need};
    for (int a = 0; a < 7; ++a)
        if (overlaps(O, no, in[a], nin[a])) return GMA_ERR_INVALID_ARG;
    for (int a = 0; a < 3; ++a)
        if (overlaps(workspace, need, in[a], nin[a])) return GMA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gma::StageClock clk = clock_for(options, s);
    const cudaError_t err = path == GMA_PATH_TC ? gma::tc_read_memory(p, Vt, Z, workspace, s, clk)
                                               : gma::simt_read_memory(p, Vt, Z, workspace, s, clk);
    return finish(err, options, workspace, s);
}

size_t gma_causal_carry_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype) {
    if (dtype != GMA_F32 && dtype != GMA_BF16) return 0;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return 0;
    Problem p;
    p.dtype = dtype; p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    const size_t simt = gma::simt_layout(p, 1, 0).total;
    size_t tc = gma::tc_supported(p, 1) ? gma::tc_carry_workspace(p) : 0;
    const size_t tc1 = gma::tc_supported(p, 1) ? gma::tc_scan_workspace(p, 0) : 0;
    tc = tc > tc1 ? tc : tc1;
    return simt > tc ? simt : tc;  // enough for any kernel family
}

gma_status gma_forward_causal_carry(const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype,
                                    const float *mu, const float *sigma2, const float *log_pi, float eps,
                                    const float *Vt_in, const float *Z_in, float *Vt_out, float *Z_out,
                                    void *O, int B, int H, int N, int d_r, int d_v, int K,
                                    const gma_options *options, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    if (!Q_X || !K_X || !V_X || !mu || !sigma2 || !log_pi || !O || !workspace) return GMA_ERR_INVALID_ARG;
    if (!Vt_in != !Z_in || !Vt_out != !Z_out) return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    const void *al[] = {Q_X, K_X, V_X, O, mu, sigma2, Vt_in, Z_in, Vt_out, Z_out};
    for (const void *ptr : al)
        if (ptr && !aligned16(ptr)) return GMA_ERR_INVALID_ARG;
    if (!shape_ok(B, H, N, d_r, d_v, K, true)) return GMA_ERR_UNSUPPORTED_SHAPE;
    Problem p;
    p.Q = Q_X; p.Kx = K_X; p.V = V_X; p.mu = mu; p.sigma2 = sigma2; p.log_pi = log_pi; p.O = O;
    p.dtype = dtype; p.eps = eps;
    p.B = B; p.H = H; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    p.o_bf16 = options && options->o_bf16;
    if (options && options->chunk < 0) return GMA_ERR_INVALID_ARG;
    const int path = memory_path(p, 1, options);
    if (path < 0 || !chunk_ok(path, 1, options)) return GMA_ERR_UNSUPPORTED_SHAPE;
    const size_t need = path == GMA_PATH_TC_SINGLE_PASS ? gma::tc_scan_workspace(p, 0)
                        : path == GMA_PATH_TC            ? gma::tc_carry_workspace(p)
                                                         : gma::simt_layout(p, 1, 0).total;
    if (workspace_bytes < need) return GMA_ERR_WORKSPACE_TOO_SMALL;
    const size_t es = dtype == GMA_F32 ? 4 : 2, rows = (size_t)B * H * N;
    const size_t nvt = 4 * (size_t)B * H * K * d_v, nz = 4 * (size_t)B * H * K;
    const void *in[] = {Q_X, K_X, V_X, Vt_in, Z_in, mu, sigma2, log_pi, workspace};
    const size_t nin[] = {es * rows * d_r, es * rows * d_r, es * rows * d_v, Vt_in ? nvt : 0, Z_in ? nz : 0,
                          4 * (size_t)H * K * d_r, 4 * (size_t)H * K * d_r, 4 * (size_t)H * K, need};
    const void *out[] = {O, Vt_out, Z_out};
    const size_t nout[] = {(p.o_bf16 ? 2 : 4) * rows * d_v, Vt_out ? nvt : 0, Z_out ? nz : 0};
    for (int a = 0; a < 3; ++a) {
        if (!out[a]) continue;
        for (int b = 0; b < 9; ++b)
            if (in[b] && overlaps(out[a], nout[a], in[b], nin[b])) return GMA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (out[b] && overlaps(out[a], nout[a], out[b], nout[b])) return GMA_ERR_INVALID_ARG;
    }
    for (int b = 0; b < 5; ++b)
        if (in[b] && overlaps(workspace, need, in[b], nin[b])) return GMA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gma::StageClock clk = clock_for(options, s);
    const cudaError_t err =
        path == GMA_PATH_TC_SINGLE_PASS
            ? gma::tc_causal_carry_1pass(p, 0, Vt_in, Z_in, Vt_out, Z_out, workspace, s, clk)
        : path == GMA_PATH_TC ? gma::tc_causal_carry(p, 0, Vt_in, Z_in, Vt_out, Z_out, workspace, s, clk)
                            : gma::simt_causal_carry(p, Vt_in, Z_in, Vt_out, Z_out, workspace, s, clk);
    return finish(err, options, workspace, s);
}

gma_status gma_reparameterize(const float *omega, const float *alpha, int H, int K, int d_r, float eps_sigma,
                              float *sigma2, float *log_pi, void *stream) {
    if (!omega || !alpha || !sigma2 || !log_pi) return GMA_ERR_INVALID_ARG;
    if (!(eps_sigma > 0.f) || !std::isfinite(eps_sigma)) return GMA_ERR_INVALID_ARG;
    const void *al[] = {omega, alpha, sigma2, log_pi};
    for (const void *ptr : al)
        if (reinterpret_cast<uintptr_t>(ptr) % 4 != 0) return GMA_ERR_INVALID_ARG;
    if (!shape_ok(1, H, 1, d_r, 16, K, false)) return GMA_ERR_UNSUPPORTED_SHAPE;
    const size_t np = 4 * (size_t)H * K * d_r, nl = 4 * (size_t)H * K;
    if (overlaps(sigma2, np, omega, np) || overlaps(sigma2, np, alpha, nl) || overlaps(log_pi, nl, omega, np) ||
        overlaps(log_pi, nl, alpha, nl) || overlaps(sigma2, np, log_pi, nl))
        return GMA_ERR_INVALID_ARG;
    if (gma::reparameterize(omega, alpha, H, K, d_r, eps_sigma, sigma2, log_pi, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return GMA_ERR_CUDA;
    }
    return GMA_OK;
}

gma_status gma_reparameterize_backward(const float *omega, const float *alpha, const float *dsigma2,
                                       const float *dlog_pi, int H, int K, int d_r, float *domega,
                                       float *dalpha, void *stream) {
    if (!omega || !alpha || !dsigma2 || !dlog_pi || !domega || !dalpha) return GMA_ERR_INVALID_ARG;
    const void *al[] = {omega, alpha, dsigma2, dlog_pi, domega, dalpha};
    for (const void *ptr : al)
        if (reinterpret_cast<uintptr_t>(ptr) % 4 != 0) return GMA_ERR_INVALID_ARG;
    if (!shape_ok(1, H, 1, d_r, 16, K, false)) return GMA_ERR_UNSUPPORTED_SHAPE;
    const size_t np = 4 * (size_t)H * K * d_r, nl = 4 * (size_t)H * K;
    const void *in[] = {omega, alpha, dsigma2, dlog_pi};
    const size_t nin[] = {np, nl, np, nl};
    for (int b = 0; b < 4; ++b)
        if (overlaps(domega, np, in[b], nin[b]) || overlaps(dalpha, nl, in[b], nin[b])) return GMA_ERR_INVALID_ARG;
    if (overlaps(domega, np, dalpha, nl)) return GMA_ERR_INVALID_ARG;
    if (gma::reparameterize_backward(omega, alpha, dsigma2, dlog_pi, H, K, d_r, domega, dalpha,
                                     static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return GMA_ERR_CUDA;
    }
    return GMA_OK;
}

size_t gma_project_workspace_size(void) { return gma::proj_workspace(); }

gma_status gma_project_qkv(const void *X, const void *W_Q, const void *W_K, const void *W_V, void *Q_X, void *K_X,
                           void *V_X, gma_dtype out_dtype, int B, int N, int D, int H, int d_r, int d_v,
                           const gma_options *options, void *workspace, size_t workspace_bytes, void *stream) {
    if (!X || !W_Q || !W_K || !W_V || !Q_X || !K_X || !V_X || !workspace) return GMA_ERR_INVALID_ARG;
    if (out_dtype != GMA_F32 && out_dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GMA_ERR_INVALID_ARG;
    const void *al[] = {X, W_Q, W_K, W_V, Q_X, K_X, V_X};
    for (const void *ptr : al)
        if (!aligned16(ptr)) return GMA_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || H < 1 || D < 8 || D % 8 != 0 || !valid_dim(d_r) || !valid_dim(d_v))
        return GMA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * N > 65535LL * 128 || (long long)H * (d_r > d_v ? d_r : d_v) > (1LL << 24) ||
        (long long)B * N * D > (1LL << 40))
        return GMA_ERR_UNSUPPORTED_SHAPE;
    if (workspace_bytes < gma::proj_workspace()) return GMA_ERR_WORKSPACE_TOO_SMALL;
    const size_t oe = out_dtype == GMA_BF16 ? 2 : 4, rows = (size_t)B * N;
    const void *in[] = {X, W_Q, W_K, W_V, workspace};
    const size_t nin[] = {2 * rows * D, 2 * (size_t)H * d_r * D, 2 * (size_t)H * d_r * D, 2 * (size_t)H * d_v * D,
                          gma::proj_workspace()};
    void *out[] = {Q_X, K_X, V_X};
    const size_t nout[] = {oe * rows * H * d_r, oe * rows * H * d_r, oe * rows * H * d_v};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 5; ++b)
            if (overlaps(out[a], nout[a], in[b], nin[b])) return GMA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlaps(out[a], nout[a], out[b], nout[b])) return GMA_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t err = gma::tc_project_qkv(X, W_Q, W_K, W_V, Q_X, K_X, V_X, out_dtype == GMA_BF16, B, N, D, H,
                                                d_r, d_v, options && options->test_stall, workspace, s);
    return finish(err, options, workspace, s);
}

gma_status gma_last_device_status(const void *workspace, void *stream) {
    if (!workspace) return GMA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned st = 0;
    if (cudaMemcpyAsync(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        (void)cudaGetLastError();
        return GMA_ERR_CUDA;
    }
    return static_cast<gma_status>(st);
}

const char *gma_status_string(gma_status status) {
    switch (status) {
        case GMA_OK: return "ok";
        case GMA_ERR_INVALID_ARG: return "invalid argument";
        case GMA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case GMA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case GMA_ERR_CUDA: return "CUDA error";
        case GMA_ERR_TIMEOUT: return "device-side wait timed out";
        case GMA_ERR_NONFINITE_PARAM: return "invalid mixture parameter (sigma2 <= 0 or non-finite)";
    }
    return "unknown status";
}

int gma_selected_path(int N, int d_r, int d_v, int K, gma_dtype dtype, int causal,
                      const gma_options *options) {
    if (causal < 0 || causal > 1 || (dtype != GMA_F32 && dtype != GMA_BF16)) return -1;
    if (!shape_ok(1, 1, N, d_r, d_v, K, true)) return -1;
    Problem p;
    p.dtype = dtype; p.B = 1; p.H = 1; p.N = N; p.d_r = d_r; p.d_v = d_v; p.K = K;
    const int path = choose_path(p, causal, options);
    return path >= 0 && chunk_ok(path, causal, options) ? path : -1;
}

int gma_tc_partition(int tiles_per_head, int total_tiles, int max_ctas, int *starts, int starts_len,
                     int *switch_tiles) {
    return gma::tc_partition(tiles_per_head, total_tiles, max_ctas, starts, starts_len, switch_tiles);
}

int gma_stage_count(int path, int variant) {
    if (path == GMA_PATH_TC_SINGLE_PASS) {
        if (variant == 1 || variant == 8) return 2;
        if (variant == 0 || variant == 4 || variant == 7) path = GMA_PATH_TC;  // as GMA_PATH_TC
        else return 0;
    }
    const bool tc_aux = path == GMA_PATH_TC && (variant == 4 || variant == 7 || variant == 8);
    if (variant < -1 || variant > 8 || (variant >= 2 && path != GMA_PATH_SIMT && !tc_aux)) return 0;
    const char *const *names;
    if (tc_aux) names = gma::kAuxTcStages[variant - 4];
    else if (variant >= 4) names = gma::kAuxStages[variant - 4];
    else if (variant >= 2) names = gma::kBackwardStages[variant - 2];
    else if (path == GMA_PATH_SIMT) names = gma::kSimtStages[variant + 1];
    else if (path == GMA_PATH_TC) names = gma::kTcStages[variant + 1];
    else return 0;
    int n = 0;
    while (n < 8 && names[n]) ++n;
    return n;
}

const char *gma_stage_name(int path, int variant, int j) {
    int n = gma_stage_count(path, variant);
    if (j < 0 || j >= n) return nullptr;
    if (path == GMA_PATH_TC_SINGLE_PASS) {
        if (variant == 1 || variant == 8) return gma::kTcScanStages[j];
        path = GMA_PATH_TC;
    }
    if (variant >= 4) return path == GMA_PATH_TC ? gma::kAuxTcStages[variant - 4][j] : gma::kAuxStages[variant - 4][j];
    if (variant >= 2) return gma::kBackwardStages[variant - 2][j];
    return path == GMA_PATH_SIMT ? gma::kSimtStages[variant + 1][j] : gma::kTcStages[variant + 1][j];
}

}  // extern "C"
