/*
 * gma.h -- C ABI of libgma.so: the forward hot path of Gaussian Mixture
 * Attention (GMA) on NVIDIA GB300 (sm_103a).
 *
 * Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
 * Probabilistic Latent Routing" (arXiv 2606.18283), cited [GMA, ...].
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are dense, contiguous, row-major:
 *     X, Q_X, K_X : [B, H, N, d_r]   V_X, O : [B, H, N, d_v]   Gamma : [B, H, N, K]
 *   O is fp32 (the value of the fp32 accumulation, not rounded further)
 *   unless gma_options.o_bf16 asks for bfloat16 output.
 *     mu, sigma2  : [H, K, d_r] fp32 log_pi : [H, K] fp32
 *   One mixture (mu, sigma2, pi) per head h, shared by every batch entry and
 *   by the query and key side of that head ([GMA, "a shared Gaussian
 *   mixture", applied separately to Q_X and K_X]).
 * - Every pointer argument except the host-side `options` is a DEVICE pointer
 *   on the current CUDA device.  The caller owns all buffers, including the
 *   workspace; the library never allocates or frees device memory and keeps
 *   no state between calls.  One exception: gma_forward_bidir_noalloc keeps
 *   its scratch in a fixed device array of the library (see there).
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Calls are asynchronous on that stream.
 * - Host-detectable errors (null pointers, bad sizes, aliasing, short
 *   workspace) are returned before anything is launched.  Invalid parameter
 *   VALUES (sigma2 <= 0 or non-finite, non-finite mu or log_pi) and device
 *   timeouts are detected on the device: they are written to a status word
 *   at the start of the workspace, the remaining kernels of the call skip
 *   their work (O / Gamma are then left unwritten), and the status is
 *   returned by gma_last_device_status() -- or directly, when
 *   options->sync_status is set.
 * - Inputs must not overlap O / Gamma or the workspace.  Q_X, K_X, V_X and O
 *   (and mu, sigma2) must start on a 16-byte boundary, the workspace on a 256-byte boundary
 *   (GMA_ERR_INVALID_ARG otherwise).
 * - Results are deterministic: the same inputs, sizes and options give
 *   bitwise-identical outputs (fixed-order reductions, no atomics on data).
 * - Supported sizes: B, H, N >= 1; d_r, d_v in {16, 32, 64, 128};
 *   1 <= K <= 128.  Anything else returns GMA_ERR_UNSUPPORTED_SHAPE.
 */
#ifndef GMA_H_
#define GMA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of X / Q_X / K_X / V_X (Gamma and, by default, O are fp32). */
typedef enum gma_dtype {
    GMA_F32 = 0,  /* IEEE binary32 */
    GMA_BF16 = 1  /* bfloat16 */
} gma_dtype;

typedef enum gma_status {
    GMA_OK = 0,
    GMA_ERR_INVALID_ARG = 1,        /* null pointer, eps <= 0 or non-finite, aliasing, bad option */
    GMA_ERR_UNSUPPORTED_SHAPE = 2,  /* sizes outside the supported set */
    GMA_ERR_WORKSPACE_TOO_SMALL = 3,
    GMA_ERR_CUDA = 4,               /* a CUDA runtime call failed (launch, attribute, ...) */
    GMA_ERR_TIMEOUT = 5,            /* a bounded device-side wait ran out */
    GMA_ERR_NONFINITE_PARAM = 6     /* sigma2 <= 0 or non-finite, or non-finite mu / log_pi */
} gma_status;

/* Kernel family selector (gma_options.path). */
enum {
    GMA_PATH_AUTO = 0,   /* tensor-core path when the dtype/sizes allow it, else SIMT */
    GMA_PATH_SIMT = 1,   /* fp32 CUDA-core kernels (every supported size, fp32 or bf16 input) */
    /* tcgen05 tensor-core kernels, bf16 inputs: the forward calls at d_r in {32, 64},
     * d_v = 64, K <= 64 or at d_r = d_v = 128, K <= 128; the latent-memory calls
     * at the first of those sizes.  GMA_ERR_UNSUPPORTED_SHAPE if not eligible. */
    GMA_PATH_TC = 2,
    /* Causal calls (gma_forward_causal, gma_forward_causal_carry): the single-pass
     * tensor-core kernel, at d_r in {32, 64}, d_v = 64, K <= 64 (other sizes:
     * GMA_ERR_UNSUPPORTED_SHAPE).  Each 128-token chunk computes
     * its key responsibilities in shared memory next to its query side, so
     * Gamma^K never goes to device memory and Q_X, K_X, V_X are read once; the
     * prefix memory before a chunk is the fixed-order sum of the published
     * memories of earlier chunks (bitwise reproducible).  GMA_PATH_TC's two
     * kernels instead store Gamma^K between an aggregation pass and the chunk
     * scan; they are the faster of the two on GB300 (measured) and the
     * default.  Other calls: as GMA_PATH_TC. */
    GMA_PATH_TC_SINGLE_PASS = 3
};

/* Optional knobs; pass NULL for all defaults.  Zero in a field = default. */
typedef struct gma_options {
    int path;         /* GMA_PATH_* */
    int chunk;        /* causal chunk length in tokens: 0 or the kernel family's length (tensor cores 128,
                       * CUDA cores 64); any other value makes a causal call (forward, carried-prefix
                       * forward, backward) return GMA_ERR_UNSUPPORTED_SHAPE (negative:
                       * GMA_ERR_INVALID_ARG); ignored by the other calls */
    int splits;       /* number of N-splits of the key pass per head (0 = chosen from the grid) */
    int sync_status;  /* nonzero: synchronise `stream` before returning and return the device status */
    int o_bf16;       /* nonzero: O is bfloat16, rounded to nearest even from fp32 (default fp32) */
    /* Optional profiling hook: an array of n_stage_events cudaEvent_t (passed
     * as void*).  When non-NULL, event 0 is recorded on `stream` before the
     * first stage of the call and event j+1 after stage j, for as many
     * events as are given; the stages of a call are named by
     * gma_stage_name().  The events are owned by the caller. */
    void **stage_events;
    int n_stage_events;
    /* Test hook for the failure path, leave 0.  Nonzero: the tensor-core key
     * pass never loads its first key tile, so the first bounded device wait on
     * it runs out (after 4 s) and the call reports GMA_ERR_TIMEOUT through the
     * status word; every kernel still finishes and frees what it holds, and the
     * stream and workspace stay usable.  No effect on the SIMT path. */
    int test_stall;
} gma_options;

/*
 * Bytes of device workspace that a call with these sizes needs (256-byte
 * aligned start required).  causal: 0 for gma_forward_bidir, 1 for
 * gma_forward_causal, -1 for gma_responsibilities.  Returns 0 for sizes that
 * are not supported.
 */
size_t gma_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype,
                          int causal, const gma_options *options);

/*
 * Gamma[b,h,i,k] = p(z = k | x_i), the posterior responsibility of
 * component k of head h for row i of X ([GMA, Eqs. (2)-(3)]): a softmax over
 * k of log N(x_i; mu_k, diag sigma2_k) + log pi_k.  log_pi need not be
 * normalised (the softmax is invariant to a shift).  Gamma is fp32.
 */
gma_status gma_responsibilities(const void *X, gma_dtype dtype, const float *mu,
                                const float *sigma2, const float *log_pi, float *Gamma,
                                int B, int H, int N, int d_r, int K,
                                const gma_options *options, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Bidirectional GMA forward ([GMA, Eqs. (5)-(7), footnote 4]):
 *   Vt = (Gamma^K)^T V_X,  Z = (Gamma^K)^T 1,  O = Gamma^Q Vt / (Gamma^Q Z + eps)
 * per (b, h), with Gamma^Q / Gamma^K the responsibilities of Q_X / K_X.
 * eps > 0 is added after the sum over components.  O is fp32 (bf16 with
 * options->o_bf16).
 */
gma_status gma_forward_bidir(const void *Q_X, const void *K_X, const void *V_X,
                             gma_dtype dtype, const float *mu, const float *sigma2,
                             const float *log_pi, float eps, void *O,
                             int B, int H, int N, int d_r, int d_v, int K,
                             const gma_options *options, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * Causal GMA forward ([GMA, causal variant, Eq. (8b)]): as above with the
 * prefix memories Vt^(i) = sum_{j<=i} gamma^K_j V_j, Z^(i) = sum_{j<=i}
 * gamma^K_j (j <= i inclusive):
 *   O_i = Gamma^Q_i Vt^(i) / (Gamma^Q_i Z^(i) + eps).
 */
gma_status gma_forward_causal(const void *Q_X, const void *K_X, const void *V_X,
                              gma_dtype dtype, const float *mu, const float *sigma2,
                              const float *log_pi, float eps, void *O,
                              int B, int H, int N, int d_r, int d_v, int K,
                              const gma_options *options, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * Synchronises `stream` and returns the device-side status recorded in the
 * workspace by the last call that used it (GMA_OK, GMA_ERR_NONFINITE_PARAM,
 * GMA_ERR_TIMEOUT), or GMA_ERR_CUDA if the synchronisation itself failed.
 */
gma_status gma_last_device_status(const void *workspace, void *stream);

/* Static, human-readable name of a status code. */
const char *gma_status_string(gma_status status);

/*
 * Which kernel family a call with these arguments would run
 * (GMA_PATH_SIMT or GMA_PATH_TC), or -1 if the call would be rejected.
 */
int gma_selected_path(int N, int d_r, int d_v, int K, gma_dtype dtype, int causal,
                      const gma_options *options);

/*
 * Diagnostic, host only (no device work, no CUDA call): how the 64-wide
 * tensor-core kernels (GMA_PATH_TC at d_r, d_v <= 64) cut a call's tiles into
 * one contiguous range per CTA.  The call's B*H*ceil(N/128) tiles of 128 tokens
 * are taken in (head, tile) order: total_tiles of them, tiles_per_head per head
 * (total_tiles a multiple of tiles_per_head).  At most max_ctas ranges (the
 * kernels pass the SM count, or options->splits when set); the library caps
 * this at its own limit.  A range costs its tiles plus *switch_tiles for every
 * head boundary inside it (the job end and job start it pays), and the cuts
 * minimise the largest range cost.  Writes the first tile of every range, then
 * total_tiles, into starts[0 .. n] and returns n, the number of ranges; writes
 * the per-boundary cost to *switch_tiles when that pointer is not NULL.
 * Returns -1 for an argument out of range or starts_len < n + 1.
 */
int gma_tc_partition(int tiles_per_head, int total_tiles, int max_ctas, int *starts, int starts_len,
                     int *switch_tiles);

/*
 * Allocation-free variant of gma_forward_bidir.  The paper has no
 * counterpart: this is a deployment convenience.
 *
 * Some callers cannot allocate device memory at all: code that runs inside
 * another framework whose device memory is fully owned by that framework's
 * allocator, real-time or embedded code that must not call cudaMalloc after
 * start-up (it can fail at any time and it synchronises the whole device),
 * and plug-ins that receive only input and output buffers.  This entry point
 * takes no workspace: its scratch is a file-scope device array of
 * GMA_NOALLOC_SCRATCH_BYTES inside libgma.so, which every GPU that loads the
 * library holds until the process exits.  It calls no cudaMalloc, cudaFree
 * or allocating library routine.  The caller still passes the inputs and O.
 *
 * - Arguments and results are those of gma_forward_bidir.  Argument errors
 *   (null pointers, a bad dtype, negative options->chunk or splits) are
 *   checked first (GMA_ERR_INVALID_ARG), then the sizes: unsupported sizes
 *   return GMA_ERR_UNSUPPORTED_SHAPE, and sizes whose workspace
 *   (gma_workspace_size(..., causal = 0, options)) exceeds
 *   GMA_NOALLOC_SCRATCH_BYTES return GMA_ERR_WORKSPACE_TOO_SMALL, in both
 *   cases without touching the device.
 * - Every call looks up the array's device address in the CUDA context
 *   current on the calling thread (cudaGetSymbolAddress, which allocates
 *   nothing), so a call made after cudaDeviceReset, or with another context
 *   current, uses that context's copy of the array.  The first call in a
 *   context may load the library's device code, array included, into it:
 *   make that first call before any stream capture in that context.
 * - Every call on a device shares the one array, which keeps the last call's
 *   contents.  Calls whose work overlaps on the GPU (different streams, or
 *   different host threads without ordering) race on it: order them, e.g. on
 *   one stream.  The device status word lives at its start, as for
 *   gma_forward_bidir; read it with options->sync_status.
 */
#define GMA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
gma_status gma_forward_bidir_noalloc(const void *Q_X, const void *K_X, const void *V_X,
                                     gma_dtype dtype, const float *mu, const float *sigma2,
                                     const float *log_pi, float eps, void *O,
                                     int B, int H, int N, int d_r, int d_v, int K,
                                     const gma_options *options, void *stream);

/*
 * Gradients of gma_forward_bidir / gma_forward_causal ([GMA, gradient section]: the upstream
 * gradient of a responsibility row, the softmax Jacobian (Eq. (17)) and the
 * gradient entering the score (Eq. (18)), then the chain rule through the
 * score into the routing rows and the mixture parameters).  Given
 * dO = dL/dO of the forward with the same arguments:
 *   dO          : [B, H, N, d_v] fp32 (input)
 *   dQ_X, dK_X  : [B, H, N, d_r] fp32     dV_X : [B, H, N, d_v] fp32
 *   dmu, dsigma2: [H, K, d_r] fp32        dlog_pi : [H, K] fp32
 * The parameter gradients are summed over the batch and over the query and
 * key rows (one mixture per head).  Every output is written, none is
 * accumulated into.  The forward's responsibilities and latent memory are
 * recomputed; everything runs on the CUDA cores in fp32
 * (options->path must be GMA_PATH_AUTO or GMA_PATH_SIMT, o_bf16 must be 0).
 * Inputs as for gma_forward_bidir; dO and every output but dlog_pi must start
 * on a 16-byte boundary, and no output may overlap an input, another output
 * or the workspace (GMA_ERR_INVALID_ARG).  Device-side parameter errors and
 * the status word behave as for the forward.
 *
 * The causal variant differentiates Eq. (8b): the query side reads the
 * prefix memories, and a key j collects the suffix sums over the queries
 * i >= j; it runs in chunks of 64 tokens (options->splits is ignored).
 *
 * gma_backward_workspace_size: bytes of workspace for these sizes (causal 0
 * for gma_backward_bidir, 1 for gma_backward_causal; 0 is returned for
 * unsupported arguments).
 */
size_t gma_backward_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype,
                                   int causal, const gma_options *options);
gma_status gma_backward_bidir(const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype,
                              const float *mu, const float *sigma2, const float *log_pi, float eps,
                              const float *dO, float *dQ_X, float *dK_X, float *dV_X, float *dmu,
                              float *dsigma2, float *dlog_pi, int B, int H, int N, int d_r, int d_v,
                              int K, const gma_options *options, void *workspace,
                              size_t workspace_bytes, void *stream);
gma_status gma_backward_causal(const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype,
                               const float *mu, const float *sigma2, const float *log_pi, float eps,
                               const float *dO, float *dQ_X, float *dK_X, float *dV_X, float *dmu,
                               float *dsigma2, float *dlog_pi, int B, int H, int N, int d_r, int d_v,
                               int K, const gma_options *options, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Latent memory of a key/value sequence ([GMA, Eqs. (5)-(6), latent
 * aggregation]):
 *   Vt[b,h] = (Gamma^K)^T V_X  : [B, H, K, d_v] fp32
 *   Z[b,h]  = (Gamma^K)^T 1    : [B, H, K] fp32
 * with Gamma^K the responsibilities of K_X.  This is also the carried state
 * of the causal variant after the last position (the prefix memories of
 * Eq. (8b) at i = N - 1): it primes gma_decode_step with a prompt of N tokens.
 * Kernel family (options->path): GMA_PATH_AUTO and GMA_PATH_SIMT run it on
 * the CUDA cores (fp32 responsibilities, any supported size); GMA_PATH_TC on
 * the tensor-core write kernel of the bidirectional forward (bf16 inputs,
 * d_r in {32, 64}, d_v = 64, K <= 64; other sizes GMA_ERR_UNSUPPORTED_SHAPE),
 * whose fp32 memory is the sum of per-job partials in job order.
 * options->splits sets the number of N-splits (0 = default).
 * K_X, V_X, Vt, Z must start on a 16-byte boundary, the workspace on a
 * 256-byte boundary; Vt and Z may not overlap an input, each other or the
 * workspace (GMA_ERR_INVALID_ARG).  Parameter errors and the status word
 * behave as for the forward.  Workspace bytes:
 * gma_latent_memory_workspace_size for the same options (0 for unsupported
 * arguments or a kernel family that does not take them).
 */
size_t gma_latent_memory_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype,
                                        const gma_options *options);
gma_status gma_latent_memory(const void *K_X, const void *V_X, gma_dtype dtype, const float *mu,
                             const float *sigma2, const float *log_pi, float *Vt, float *Z,
                             int B, int H, int N, int d_r, int d_v, int K,
                             const gma_options *options, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * One autoregressive position of the causal GMA for every (b, h) ([GMA, causal
 * variant, Eq. (8b)], prefix memories carried as running sums).  The new
 * position's key enters its own prefix before its query reads it (j <= i):
 *   Vt[b,h,k,:] += gamma^K_k v[b,h,:],   Z[b,h,k] += gamma^K_k
 *   o[b,h,:]     = sum_k gamma^Q_k Vt[b,h,k,:] / (sum_k gamma^Q_k Z[b,h,k] + eps)
 *   q, k : [B, H, d_r]   v : [B, H, d_v]   (dtype)
 *   Vt   : [B, H, K, d_v] fp32, Z : [B, H, K] fp32 -- read and updated in place
 *   o    : [B, H, d_v] fp32
 * Start from zeros (an empty prefix) or from gma_latent_memory of a prompt.
 * Calling it for positions 0..N-1 in order reproduces gma_forward_causal row by
 * row.  Runs on the CUDA cores (options->path GMA_PATH_AUTO or GMA_PATH_SIMT;
 * options->o_bf16 is not supported, GMA_ERR_UNSUPPORTED_SHAPE).  Vt and o must
 * start on a 16-byte boundary and the workspace on a 256-byte boundary; Vt, Z and o
 * may not overlap an input, each other or the workspace (GMA_ERR_INVALID_ARG).
 * Invalid parameter values are reported through the status word as for the
 * forward; the (b, h) rows of a head with an invalid value are left unchanged
 * (Vt, Z and o), the other heads are updated.  The workspace
 * (gma_decode_workspace_size bytes, independent of B) holds the status word and
 * the per-head constants of the log-density.
 */
size_t gma_decode_workspace_size(int H, int d_r, int K);
gma_status gma_decode_step(const void *q, const void *k, const void *v, gma_dtype dtype,
                           const float *mu, const float *sigma2, const float *log_pi, float eps,
                           float *Vt, float *Z, float *o, int B, int H, int d_r, int d_v, int K,
                           const gma_options *options, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * Component-usage diagnostics of the responsibilities of X ([GMA,
 * introduction: the marginal usage of the components and the hard assignment
 * z_i = argmax_k gamma_ik; the interpretability results' components-used count
 * and usage entropy]), per (b, h), computed beside the responsibilities
 * without writing Gamma:
 *   usage   : [B, H, K] fp32   usage_k = sum_i gamma_ik
 *   counts  : [B, H, K] int32  number of rows whose hard assignment is k
 *   z       : [B, H, N] int32  hard assignment of each row: the smallest k
 *             that maximises the row's score (and so gamma); may be NULL
 *   entropy : [B, H] fp32      -sum_k p_k log p_k / log K with p = usage / N
 *             (1 when K = 1); may be NULL
 * The number of components used is the number of non-zero counts.  Runs on the
 * CUDA cores (options->path GMA_PATH_AUTO or GMA_PATH_SIMT).  X, usage and
 * counts must start on a 16-byte boundary, the workspace on a 256-byte
 * boundary; no output may overlap an input, another output or the workspace
 * (GMA_ERR_INVALID_ARG).  Parameter errors and the status word behave as for
 * the forward.  Workspace bytes: gma_routing_stats_workspace_size.
 */
size_t gma_routing_stats_workspace_size(int B, int H, int N, int d_r, int K, gma_dtype dtype);
gma_status gma_routing_stats(const void *X, gma_dtype dtype, const float *mu, const float *sigma2,
                             const float *log_pi, float *usage, int *counts, int *z, float *entropy,
                             int B, int H, int N, int d_r, int K, const gma_options *options,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Normalized broadcasting from a given latent memory ([GMA, Eq. (7),
 * footnote 4]):
 *   O[b,h,i,:] = sum_k gamma^Q_ik Vt[b,h,k,:] / (sum_k gamma^Q_ik Z[b,h,k] + eps)
 *   Q_X : [B, H, N, d_r] (dtype)   Vt : [B, H, K, d_v] fp32   Z : [B, H, K] fp32
 *   O   : [B, H, N, d_v] fp32 (bf16 with options->o_bf16)
 * With gma_latent_memory this splits the bidirectional forward at the latent
 * memory: the memories of several key/value shards add up (the sums of
 * Eqs. (5)-(6) split over N), so a sequence sharded over N needs one sum of
 * [K, d_v + 1] per head between the two calls.  Kernel family
 * (options->path): GMA_PATH_AUTO and GMA_PATH_SIMT run it on the CUDA cores;
 * GMA_PATH_TC packs the memory into the tensor-core read kernel's operand
 * (each fp32 value as a bf16 high part plus a bf16 low part) and runs the
 * read of the bidirectional forward (bf16 inputs, d_r in {32, 64}, d_v = 64,
 * K <= 64; other sizes GMA_ERR_UNSUPPORTED_SHAPE).  A GMA_PATH_TC memory from
 * gma_latent_memory read this way gives the GMA_PATH_TC bidirectional
 * forward's O bit for bit.  Q_X, Vt, Z and O must start
 * on a 16-byte boundary, the workspace on a 256-byte boundary; O may not
 * overlap an input or the workspace (GMA_ERR_INVALID_ARG).  Workspace bytes:
 * gma_read_memory_workspace_size (enough for either kernel family).
 */
size_t gma_read_memory_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype);
gma_status gma_read_memory(const void *Q_X, gma_dtype dtype, const float *mu, const float *sigma2,
                           const float *log_pi, float eps, const float *Vt, const float *Z, void *O,
                           int B, int H, int N, int d_r, int d_v, int K, const gma_options *options,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Causal GMA forward that continues a prefix ([GMA, causal variant, Eq. (8b)]):
 * the prefix memories start from a carried-in memory instead of zero,
 *   Vt^(i) = Vt_in + sum_{j<=i} gamma^K_j V_j,  Z^(i) = Z_in + sum_{j<=i} gamma^K_j,
 *   O_i    = Gamma^Q_i Vt^(i) / (Gamma^Q_i Z^(i) + eps),
 * and the prefix after the last position (Vt^(N-1), Z^(N-1)) is written to
 * (Vt_out, Z_out) when they are given.  Vt_in / Vt_out : [B, H, K, d_v] fp32,
 * Z_in / Z_out : [B, H, K] fp32; Vt_in and Z_in are both NULL (an empty prefix)
 * or both given, and so are Vt_out and Z_out.  Uses: a sequence sharded over N
 * (shard r starts from the sum of the memories of shards 0..r-1), a long prompt
 * processed in pieces, and priming gma_decode_step.  Kernel family
 * (options->path): GMA_PATH_AUTO and GMA_PATH_SIMT run it on the CUDA cores;
 * GMA_PATH_TC on the tensor-core causal forward, whose per-head prefix
 * combine starts at the carried-in memory and writes the final prefix
 * (bf16 inputs, d_r in {32, 64}, d_v = 64, K <= 64; other sizes
 * GMA_ERR_UNSUPPORTED_SHAPE); with an empty carried-in prefix it gives the
 * GMA_PATH_TC causal forward's O bit for bit.  Alignment and overlap rules
 * as for gma_forward_causal, plus: the carry buffers start on a 16-byte
 * boundary and the outputs (O, Vt_out, Z_out) overlap no input, each other or
 * the workspace.  Workspace bytes: gma_causal_carry_workspace_size (enough
 * for either kernel family).
 */
size_t gma_causal_carry_workspace_size(int B, int H, int N, int d_r, int d_v, int K, gma_dtype dtype);
gma_status gma_forward_causal_carry(const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype,
                                    const float *mu, const float *sigma2, const float *log_pi, float eps,
                                    const float *Vt_in, const float *Z_in, float *Vt_out, float *Z_out,
                                    void *O, int B, int H, int N, int d_r, int d_v, int K,
                                    const gma_options *options, void *workspace, size_t workspace_bytes,
                                    void *stream);

/*
 * Rank-order sum of latent memories ([GMA, Eqs. (5)-(6)]: the memory is a sum
 * over positions, so the memories of consecutive blocks of a sequence add up;
 * [GMA, causal variant, Eq. (8b)]: the prefix memory at a block boundary is
 * the sum of every earlier block's memory).  parts is a [P, n] fp32 device
 * array, one row per block in sequence order (e.g. each rank's packed
 * [Vt | Z] after an all-gather); out[e] = sum_{r < count} parts[r * n + e],
 * summed in fp32 one row after another from row 0, so every holder of the same
 * rows gets bitwise the same result.  count = P gives the whole sequence's
 * memory (the bidirectional read of every block), count = r the exclusive
 * prefix of block r (its causal carry-in).  1 <= count <= P, n >= 1
 * (GMA_ERR_UNSUPPORTED_SHAPE otherwise); both pointers 4-byte aligned and out
 * not overlapping parts (GMA_ERR_INVALID_ARG).  One kernel launch on `stream`;
 * no workspace.
 */
gma_status gma_combine_memories(const float *parts, int P, long long n, int count, float *out, void *stream);

/*
 * Reparameterised mixture parameters ([GMA, Eqs. (14)-(15)]), per head h:
 *   sigma2[h,k,j] = log(1 + exp(omega[h,k,j])) + eps_sigma   (softplus: positive covariances)
 *   log_pi[h,k]   = alpha[h,k] - log sum_l exp(alpha[h,l])   (log of the softmax priors)
 *   omega, sigma2 : [H, K, d_r] fp32   alpha, log_pi : [H, K] fp32
 * and the chain rule through them, for upstream gradients dsigma2, dlog_pi
 * (e.g. from gma_backward_bidir / gma_backward_causal):
 *   domega = dsigma2 * sigmoid(omega),  dalpha_k = dlog_pi_k - pi_k sum_l dlog_pi_l.
 * The outputs feed the forward entry points directly.  Device pointers, 4-byte
 * aligned; outputs may not overlap inputs (GMA_ERR_INVALID_ARG); eps_sigma must
 * be finite and > 0.  No workspace.  Sizes: H >= 1, 1 <= K <= 128, d_r in
 * {16, 32, 64, 128}.  Non-finite omega or alpha give non-finite outputs, which
 * the forward entry points then reject (GMA_ERR_NONFINITE_PARAM).
 */
gma_status gma_reparameterize(const float *omega, const float *alpha, int H, int K, int d_r, float eps_sigma,
                              float *sigma2, float *log_pi, void *stream);
gma_status gma_reparameterize_backward(const float *omega, const float *alpha, const float *dsigma2,
                                       const float *dlog_pi, int H, int K, int d_r, float *domega,
                                       float *dalpha, void *stream);

/*
 * The Q/K/V projections in front of the hot path ([GMA, Eq. (4)]: the layer
 * input X is mapped linearly to the routing rows and the values), as one
 * tensor-core GEMM per call that writes the head-major layouts the forward
 * entry points read:
 *   Q_X[b,h,n,c] = sum_i X[b,n,i] W_Q[h*d_r + c, i]   (K_X with W_K, V_X with W_V, d_v)
 *   X   : [B, N, D] bf16      W_Q, W_K : [H*d_r, D] bf16   W_V : [H*d_v, D] bf16
 *         (weights stored one output feature per row)
 *   Q_X, K_X : [B, H, N, d_r], V_X : [B, H, N, d_v] in out_dtype (GMA_BF16, rounded
 *         to nearest even from the fp32 accumulator, or GMA_F32)
 * D must be a multiple of 8 (1 <= D); B*N <= 65535*128; d_r, d_v in {16, 32, 64,
 * 128}; H >= 1.  Every pointer starts on a 16-byte boundary (the workspace on a
 * 256-byte one); outputs may not overlap inputs, each other or the workspace
 * (GMA_ERR_INVALID_ARG).  The workspace (gma_project_workspace_size bytes) holds
 * the status word; a bounded device wait that runs out reports GMA_ERR_TIMEOUT
 * there.  options: sync_status, and test_stall (the first stage of the first
 * tile is never loaded, so the MMA issuer's bounded wait runs out after 4 s).
 */
size_t gma_project_workspace_size(void);
gma_status gma_project_qkv(const void *X, const void *W_Q, const void *W_K, const void *W_V, void *Q_X, void *K_X,
                           void *V_X, gma_dtype out_dtype, int B, int N, int D, int H, int d_r, int d_v,
                           const gma_options *options, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Number of stages (kernel launches, plus the status reset of the first) of
 * a call on kernel family `path` (GMA_PATH_SIMT / GMA_PATH_TC) for
 * `variant` (-1 responsibilities, 0 bidirectional, 1 causal, 2 bidirectional
 * backward, 3 causal backward, 4 latent memory, 5 decode step, 6 routing
 * statistics, 7 read from a memory, 8 causal forward with a carried-in prefix
 * -- variants 2, 3, 5 and 6 SIMT only), and the name of
 * stage j (NULL if out of range).
 * Used with gma_options.stage_events.
 */
int gma_stage_count(int path, int variant);
const char *gma_stage_name(int path, int variant, int j);

#ifdef __cplusplus
}
#endif

#endif /* GMA_H_ */
