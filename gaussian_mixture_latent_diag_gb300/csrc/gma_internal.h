// gma_internal.h -- declarations shared by the host API (gma_api.cu) and the
// kernel translation units of libgma.so.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gma.h"

namespace gma {

struct Problem {
    const void *Q = nullptr;   // or X for the responsibilities entry point
    const void *Kx = nullptr;
    const void *V = nullptr;
    const float *mu = nullptr, *sigma2 = nullptr, *log_pi = nullptr;
    void *O = nullptr;         // or Gamma (fp32) for the responsibilities entry point
    gma_dtype dtype = GMA_F32;  // inputs
    bool o_bf16 = false;        // output O in bf16 instead of fp32
    bool test_stall = false;    // gma_options.test_stall (failure-path test hook)
    float eps = 0.f;
    int B = 0, H = 0, N = 0, d_r = 0, d_v = 0, K = 0;
    int BH() const { return B * H; }
};

// Records stage boundaries on the caller's events (gma_options.stage_events).
struct StageClock {
    void **events = nullptr;
    int n = 0, next = 0;
    cudaStream_t stream = nullptr;
    void mark() {
        if (events && next < n && events[next]) {
            // a failed record (e.g. a destroyed event) must not be reported as a
            // launch failure of the next stage
            if (cudaEventRecord(static_cast<cudaEvent_t>(events[next]), stream) != cudaSuccess)
                (void)cudaGetLastError();
        }
        ++next;
    }
};

// Every workspace region starts on a 256-byte boundary.
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Device status word lives in the first 256 bytes of every workspace.
constexpr size_t kStatusBytes = 256;

// ---------------------------------------------------------------- SIMT path
struct SimtLayout {
    size_t inv_s2 = 0, cprime = 0;   // [H][K][d_r], [H][K] fp32
    size_t gq = 0, gk = 0;           // [BH][K][N] fp32 (component-major)
    size_t partial = 0;              // [BH][nsplit][K][d_v + 1] fp32
    size_t mem = 0;                  // [BH][K][d_v + 1] fp32 (bidirectional only)
    size_t total = 0;
    int nsplit = 0, tokens_per_split = 0;
};
constexpr int kSimtCausalChunk = 64;
SimtLayout simt_layout(const Problem &p,
                       int mode /* -1 resp, 0 bidir, 1 causal, 2 latent memory, 3 read from a memory */,
                       int splits);
// Clears the status word and writes 1/sigma2 and c' (with parameter validation)
// into the simt_layout(p, -1, 0) regions of ws.
cudaError_t simt_prep(const Problem &p, void *ws, cudaStream_t s);
// Latent memory of (p.Kx, p.V) into the caller's Vt [BH][K][d_v] and Z [BH][K]
// (stages prep, resp_k, write, reduce; workspace simt_layout(p, 2, splits)).
cudaError_t simt_latent_memory(const Problem &p, int splits, float *Vt, float *Z, void *ws, cudaStream_t s,
                               StageClock &clk);

// Eq. (7) from the caller's memory Vt [BH][K][d_v], Z [BH][K] (stages prep,
// resp_q, pack, read; workspace simt_layout(p, 3, 0)).
cudaError_t simt_read_memory(const Problem &p, const float *Vt, const float *Z, void *ws, cudaStream_t s,
                             StageClock &clk);
// Causal forward whose prefix starts from (Vt_in, Z_in) (zero when null); the
// prefix after the last position goes to (Vt_out, Z_out) when given (stages as
// simt_causal; workspace simt_layout(p, 1, 0)).
cudaError_t simt_causal_carry(const Problem &p, const float *Vt_in, const float *Z_in, float *Vt_out, float *Z_out,
                              void *ws, cudaStream_t s, StageClock &clk);
cudaError_t simt_responsibilities(const Problem &p, void *ws, cudaStream_t s, StageClock &clk);
cudaError_t simt_bidir(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk);
cudaError_t simt_causal(const Problem &p, void *ws, cudaStream_t s, StageClock &clk);
extern const char *const kSimtStages[3][8];  // [variant + 1][j], NULL-terminated
// Everything of the bidirectional SIMT forward before the read: 1/sigma2, c',
// Gamma^Q, Gamma^K and the latent memory [Vt | Z] in the simt_layout(p, 0, splits)
// regions of ws.
cudaError_t simt_bidir_state(const Problem &p, int splits, void *ws, cudaStream_t s);
// The causal SIMT forward before its output kernel: 1/sigma2, c', Gamma^Q, Gamma^K
// and the exclusive prefix memory at the start of every chunk of kSimtCausalChunk
// tokens (the `partial` region of simt_layout(p, 1, 0)).
cudaError_t simt_causal_state(const Problem &p, void *ws, cudaStream_t s);

// ---------------------------------------------------------------- backward (gma_backward.cu)
struct BackwardArgs {
    const float *dO = nullptr;                       // [BH][N][d_v]
    float *dQ = nullptr, *dK = nullptr, *dV = nullptr;  // [BH][N][d_r] / [BH][N][d_v]
    float *dmu = nullptr, *dsigma2 = nullptr;        // [H][K][d_r]
    float *dlog_pi = nullptr;                        // [H][K]
};
size_t backward_workspace(const Problem &p, int causal, int splits);
cudaError_t simt_backward_bidir(const Problem &p, const BackwardArgs &g, int splits, void *ws, cudaStream_t s,
                                StageClock &clk);
cudaError_t simt_backward_causal(const Problem &p, const BackwardArgs &g, void *ws, cudaStream_t s,
                                 StageClock &clk);
extern const char *const kBackwardStages[2][8];  // [causal][j], NULL-terminated

// ---------------------------------------------------------------- decode step (gma_decode.cu)
// One causal position for every (b, h): q, k [BH][d_r], v [BH][d_v] (p.Q, p.Kx,
// p.V), carried state Vt [BH][K][d_v], Z [BH][K] updated in place, output p.O
// [BH][d_v].  Workspace: decode_workspace(H, K, d_r) bytes (the status word and
// the per-head constants of the log-density).  Stages: prep (per-head
// constants, validation, status reset), step.
size_t decode_workspace(int H, int K, int d_r);
cudaError_t simt_decode_step(const Problem &p, float *Vt, float *Z, void *ws, cudaStream_t s, StageClock &clk);

// ---------------------------------------------------------------- usage diagnostics (gma_stats.cu)
struct StatsArgs {
    float *usage = nullptr;    // [BH][K]
    int *counts = nullptr;     // [BH][K]
    int *z = nullptr;          // [BH][N] or null
    float *entropy = nullptr;  // [BH] or null (normalised usage entropy)
};
size_t stats_workspace(const Problem &p);
cudaError_t simt_routing_stats(const Problem &p, const StatsArgs &a, void *ws, cudaStream_t s, StageClock &clk);

// Stage names of the auxiliary entry points: [0] latent memory, [1] decode step,
// [2] routing statistics, [3] read from a memory, [4] causal forward with a
// carried-in prefix; NULL-terminated.
extern const char *const kAuxStages[5][8];

// ---------------------------------------------------------------- parameters (gma_param.cu)
cudaError_t reparameterize(const float *omega, const float *alpha, int H, int K, int d_r, float eps_sigma,
                           float *sigma2, float *log_pi, cudaStream_t s);
cudaError_t reparameterize_backward(const float *omega, const float *alpha, const float *dsigma2,
                                    const float *dlog_pi, int H, int K, int d_r, float *domega, float *dalpha,
                                    cudaStream_t s);

// ---------------------------------------------------------------- projections (gma_proj.cu)
// Q_X, K_X, V_X [B][H][N][d] (bf16 or fp32) = X [B N][D] W^T, W [H d][D], all
// bf16; tcgen05 GEMM.  Workspace: proj_workspace() bytes (the status word).
size_t proj_workspace();
cudaError_t tc_project_qkv(const void *X, const void *Wq, const void *Wk, const void *Wv, void *Q, void *Kx, void *V,
                           bool out_bf16, int B, int N, int D, int H, int d_r, int d_v, bool stall, void *ws,
                           cudaStream_t s);

// ---------------------------------------------------------------- tensor-core path
bool tc_supported(const Problem &p, int causal);
size_t tc_workspace(const Problem &p, int causal, int splits);
// The per-CTA tile ranges of the 64-wide kernels (gma_tc_partition).
int tc_partition(int ntiles, int total, int max_ctas, int *starts, int starts_len, int *switch_tiles);
size_t tc_carry_workspace(const Problem &p);  // the carried-prefix causal forward (tc_causal_carry)
// The single-pass causal forward (GMA_PATH_TC_SINGLE_PASS): one kernel after the
// coefficient prep, key responsibilities kept on chip, prefix memories chained
// between chunks through global memory (tc_supported(p, 1) sizes).
size_t tc_scan_workspace(const Problem &p, int splits);
cudaError_t tc_causal_1pass(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk);
cudaError_t tc_causal_carry_1pass(const Problem &p, int splits, const float *Vt_in, const float *Z_in,
                                  float *Vt_out, float *Z_out, void *ws, cudaStream_t s, StageClock &clk);
extern const char *const kTcScanStages[8];  // stage names of both, NULL-terminated
cudaError_t tc_bidir(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk);
cudaError_t tc_causal(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk);
extern const char *const kTcStages[3][8];    // [variant + 1][j], NULL-terminated
// The latent memory, the read from a caller's memory and the carried-prefix
// causal forward on the tensor-core kernels (tc_supported sizes; workspace
// tc_workspace(p, 0 | 0 | 1, splits)).
cudaError_t tc_latent_memory(const Problem &p, int splits, float *Vt, float *Z, void *ws, cudaStream_t s,
                             StageClock &clk);
cudaError_t tc_read_memory(const Problem &p, const float *Vt, const float *Z, void *ws, cudaStream_t s,
                           StageClock &clk);
cudaError_t tc_causal_carry(const Problem &p, int splits, const float *Vt_in, const float *Z_in, float *Vt_out,
                            float *Z_out, void *ws, cudaStream_t s, StageClock &clk);
extern const char *const kAuxTcStages[5][8];  // as kAuxStages, tensor-core path (entries 0, 3, 4)

// ---------------------------------------------------------------- tensor-core path, d_r = d_v = 128 (gma_tc128.cu)
// The forward at d_r = d_v = 128, K <= 128, bf16: causal (stages as kTcStages[2]:
// prep, aggregation, chunk scan) and bidirectional (kTcStages[1]: prep, key side,
// query side); workspace tc128_workspace(p, splits) for both.
bool tc128_supported(const Problem &p, int causal);
size_t tc128_workspace(const Problem &p, int splits);
cudaError_t tc128_causal(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk);
cudaError_t tc128_bidir(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk);

}  // namespace gma
