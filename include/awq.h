/*
 * awq.h - C ABI of libawq: the AWQ per-linear-layer step and the W4A16 matmul on one GPU
 * (B300, sm_103a).
 *
 * What the calls compute, with the passages they follow (page title, section):
 *
 *   awq_calib_stats    m_j = mean over calibration tokens of |x_j|
 *                      ("AWQ Math", "Saliency is an activation property, not a weight property")
 *   awq_search_scale   s = max(m, 1e-6)^alpha for each alpha of a grid; W' = W diag(s) quantised
 *                      group-wise to 4 bits; E(alpha) = mean over tokens and outputs of
 *                      (W x - Q(W') diag(s)^-1 x)^2; alpha* = the first minimiser
 *                      ("AWQ Math", "The equivalent transform", "Searching the scale")
 *   awq_quantize_pack  4-bit codes of W diag(s) (3- or 2-bit codes with cfg.bits, in the same
 *                      nibbles), one step and one zero point per group of input channels
 *                      ("AWQ Math", "Weight-only quantization and where it breaks" and
 *                      "Shapes, granularity, and complexity")
 *   awq_w4a16_gemm     Y = X (dequant(Q) diag(inv_s))^T without materialising fp16 weights
 *                      ("AWQ > Benefits and Practical Considerations": unpack the 4-bit
 *                      integers, apply the group scale and zero point and, optionally, the
 *                      per-channel inverse scale, fused with the matmul)
 *
 * Quantiser (fp32, IEEE rounding, no FMA contraction; rint = round half to even):
 *   asymmetric: hi = max(max w', 0), lo = min(min w', 0), step = (hi - lo) / 15 (1 if 0),
 *               z = clamp(rint(-lo / step), 0, 15), q = clamp(rint(w' / step) + z, 0, 15)
 *   symmetric:  step = max|w'| / 8 (1 if 0), q = clamp(rint(w' / step), -8, 7) + 8, z = 8
 *   w' = fp32(W * s). Stored step = fp16 (round to nearest even) of the fp32 step.
 *
 * Packed format (the one every call reads and writes):
 *   qweight [N, K/8] uint32, row-major: nibble i (bits 4i..4i+3) of qweight[n][w] is the
 *           code of input channel k = 8w + i.
 *   scales  [K/G, N] fp16: step of group g (channels gG .. gG+G-1) of output row n at g*N + n.
 *   zeros   [K/G, N] uint8: zero point, same indexing; not read or written in symmetric mode
 *           (the zero point is 8 there).
 *
 * Conventions for every call:
 *   - Pointers are device pointers owned by the caller, except `alphas`, a host array. Every
 *     device pointer must be 16-byte aligned. The library allocates no device memory; scratch
 *     for the search comes from the caller's workspace.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and is
 *     asynchronous: results are valid once the stream has been synchronised.
 *   - Arguments are checked on the host before anything is enqueued; a failed check returns
 *     an error code and enqueues nothing. Kernel launch failures return AWQ_ERR_CUDA.
 *   - The pipelined tensor-core kernels bound every wait; a kernel that gives up records
 *     AWQ_ERR_TIMEOUT in a device status word that awq_stream_status reports.
 *   - Shapes: G (group size) is 32, 64 or 128, K % G == 0, all sizes >= 1, and N * K, T * K and
 *     M * max(N, K) below 2^31 elements.
 */
#ifndef AWQ_H_
#define AWQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* awq_stream_t; /* same object as cudaStream_t */

typedef enum {
  AWQ_OK = 0,
  AWQ_ERR_INVALID_ARG = 1,       /* NULL pointer, non-positive size, bad group size/alpha count */
  AWQ_ERR_UNSUPPORTED_SHAPE = 2, /* K % G != 0, ldx < K or not a multiple of 8, size limits */
  AWQ_ERR_MISALIGNED = 3,        /* a device pointer is not 16-byte aligned */
  AWQ_ERR_WORKSPACE = 4,         /* workspace NULL or below the one-buffer search workspace */
  AWQ_ERR_CUDA = 5,              /* a CUDA runtime/driver call or kernel launch failed */
  AWQ_ERR_TIMEOUT = 6,           /* a device-side bounded wait gave up (see awq_stream_status) */
  AWQ_ERR_NO_DEVICE = 7          /* no usable device, or the device is not sm_103 */
} awq_status_t;

typedef struct {
  int32_t group_size; /* 32, 64 or 128 input channels per (step, zero point) */
  int32_t symmetric;  /* 0: asymmetric with zero point; 1: step = max|w| / 2^(bits-1) */
  int32_t bits;       /* code width N of "Weight-only quantization" (D = max|w| / 2^(N-1)):
                         0 or 4 for 4-bit codes, 3 or 2 for the narrower variants. Codes of
                         every width are stored in the 4-bit nibbles of the packed format, so
                         the matmul reads them unchanged: asymmetric codes 0 .. 2^N - 1 with a
                         zero point in that range; symmetric q in [-2^(N-1), 2^(N-1) - 1]
                         stored as q + 8 (implicit zero point 8 for every width) */
} awq_qcfg_t;

/*
 * Per-input-channel calibration statistic.
 *   X_f16    [T, ldx] fp16 row-major, the first K columns are used (calibration activations)
 *   mean_abs [K] fp32 out: (1/T) sum_t |X[t, j]| (fp32 accumulation, deterministic order)
 * Requires ldx >= K and ldx % 8 == 0, K % 8 == 0.
 */
awq_status_t awq_calib_stats(const void* X_f16, int64_t T, int64_t K, int64_t ldx,
                             float* mean_abs, awq_stream_t stream);

/*
 * How awq_search_scale computes E(alpha) (process-wide setting, default AWQ_SCORE_AUTO):
 *   DIRECT  sum of squares of X D^T per candidate (D = W - w_hat): 2 T N K flops each.
 *   GRAM    E = 1/(T N) sum_n d_n^T H d_n with H = X^T X formed once per call (about T K^2
 *           flops) and stored as fp16 after a power-of-two scale; each candidate then takes
 *           about 2 N K^2 / 2 flops over the lower triangle of H. Equal to DIRECT in exact
 *           arithmetic, so the errors agree to rounding (fp16 H: relative 2^-11 per entry).
 *           Runs as one persistent cooperative launch (one CTA per SM) over H and every
 *           candidate; if the device refuses the cooperative launch, as GRAM_LAUNCHES.
 *   GRAM_LAUNCHES  the same arithmetic with one launch for H and one per candidate (same
 *           results, bit for bit).
 *   AUTO    GRAM when it takes fewer tensor-core steps (long calibration sets, T > K / 2 or
 *           so), the workspace holds it, K % 64 == 0 and K T, K K < 2^31; DIRECT otherwise.
 *           Forcing GRAM on another shape returns AWQ_ERR_UNSUPPORTED_SHAPE.
 * Returns AWQ_ERR_INVALID_ARG for any other value.
 */
typedef enum {
  AWQ_SCORE_AUTO = 0,
  AWQ_SCORE_DIRECT = 1,
  AWQ_SCORE_GRAM = 2,
  AWQ_SCORE_GRAM_LAUNCHES = 3
} awq_score_mode_t;
awq_status_t awq_set_score_mode(awq_score_mode_t mode);

/*
 * Bytes of device workspace for awq_search_scale's fastest schedule under the current score
 * mode (0 on invalid input). Schedules, from the most workspace to the least:
 *   GRAM     two residual buffers plus X^T ([K, Tp] fp16, Tp = T rounded up to 64), the fp16
 *            triangle of H ([K, K]) and K Tp / 16 bytes of column sums: returned when the
 *            mode is GRAM, or AUTO and GRAM pays for this shape.
 *   OVERLAP  two residual buffers, so the next candidate's residual is built while the
 *            current one is scored (DIRECT scoring).
 *   SERIAL   one residual buffer (the OVERLAP size minus 2 N K bytes rounded up to 256): the
 *            candidates run strictly one after the other, with the same results as OVERLAP,
 *            bit for bit.
 * awq_search_scale takes the first schedule the given workspace holds (in AUTO, GRAM only
 * where it pays). Every schedule is deterministic; GRAM and the DIRECT schedules agree to
 * rounding, not bit for bit.
 */
size_t awq_search_workspace_bytes(int64_t N, int64_t K, int64_t T, int32_t n_alpha,
                                  awq_qcfg_t cfg);

/*
 * The alpha search of one linear layer.
 *   W_f16    [N, K] fp16 row-major: the layer weight W [C_out, C_in]
 *   X_f16    [T, K] fp16 row-major: calibration activations
 *   mean_abs [K] fp32 statistic from awq_calib_stats, or NULL to compute it here
 *   alphas   host [n_alpha] fp32 exponents (1 <= n_alpha <= 64), e.g. i/20 for i < 20
 *   workspace / ws_bytes   device scratch: awq_search_workspace_bytes(...) bytes, or at least
 *                          the one-buffer size given there
 *   err_out  [n_alpha] fp32 out: E(alpha_i)
 *   best_idx [1] int32 out: first i with the smallest E (computed in fp64)
 *   s_out    [K] fp32 out (may be NULL): s = max(m, 1e-6)^alpha* as used for the codes
 *   inv_s_out[K] fp32 out (may be NULL): 1 / s (IEEE division), the GEMM's inv_s
 * The scales are computed in fp64 and rounded to fp32; the codes behind E(alpha_i) are exactly
 * those awq_quantize_pack produces for s_i.
 * In the OVERLAP schedule (see awq_search_workspace_bytes) the residual kernels run on a second
 * stream owned by the library (one per device, created on the first call on that device
 * together with the events that order it); it forks from `stream` and rejoins it before the
 * call's last kernel, so the whole sequence can be captured in a CUDA graph once that first
 * call has been made. Searches issued concurrently on one device serialise their residual
 * kernels on that stream. GRAM uses that stream only for the scale grid and max|W|, which run
 * beside the transpose of X (same fork and join); it builds each next residual inside the
 * scoring launch. SERIAL uses `stream` alone.
 */
awq_status_t awq_search_scale(const void* W_f16, int64_t N, int64_t K, const void* X_f16,
                              int64_t T, const float* mean_abs, const float* alphas,
                              int32_t n_alpha, awq_qcfg_t cfg, void* workspace,
                              size_t ws_bytes, float* err_out, int32_t* best_idx,
                              float* s_out, float* inv_s_out, awq_stream_t stream);

/*
 * Group-wise 4-bit quantisation of W diag(s) into the packed format above.
 *   W_f16   [N, K] fp16;  s [K] fp32 per-input-channel scale, or NULL for s = 1 (plain RTN)
 *   qweight [N, K/8] uint32 out; scales_f16 [K/G, N] fp16 out; zeros [K/G, N] uint8 out
 *   (zeros may be NULL in symmetric mode).
 */
awq_status_t awq_quantize_pack(const void* W_f16, int64_t N, int64_t K, const float* s,
                               awq_qcfg_t cfg, uint32_t* qweight, void* scales_f16,
                               uint8_t* zeros, awq_stream_t stream);

/*
 * Per-group clipping search, run after the alpha search (the pages print no clipping step, so
 * the rule is a reading: "AWQ Math", "CPU-SLM implications and common pitfalls" only warns to
 * watch the group size). For each group of each output row and each ratio c of `ratios`, the
 * group's magnitudes are bounded by b = fp32(c max|w'|), w' = fp32(W s): the asymmetric range
 * ends become min(hi, b) and max(lo, -b) (hi and lo widened to hold 0 as usual), the symmetric
 * max|w'| becomes b, and weights beyond take the end codes. The group's error is
 * e(c) = sum_k h_k (W - w_hat)^2 over its channels, h_k = sum_t X[t, k]^2 (the layer's output
 * error on the calibration set with the cross-channel terms dropped), w_hat the dequantised
 * weight (q - z) step16 / s; the first ratio with the smallest e (fp32) wins.
 *   W_f16   [N, K] fp16;  X_f16 [T, K] fp16;  s [K] fp32 (the searched scale) or NULL (s = 1)
 *   ratios  host [n_ratio] fp32 in (0, 1], 1 <= n_ratio <= 32 (e.g. 1 - j/20 for j < 10;
 *           with ratios[0] = 1 a group is clipped only where that strictly lowers its error)
 *   energy  [K] fp32 device out: h (written by the call, fixed summation order)
 *   clip_out [K/G, N] fp32 device out: the chosen ratio of each group (indexed like scales)
 * Two kernels on `stream`. awq_quantize_pack_clip then packs with those ratios.
 */
awq_status_t awq_clip_search(const void* W_f16, int64_t N, int64_t K, const void* X_f16,
                             int64_t T, const float* s, const float* ratios, int32_t n_ratio,
                             awq_qcfg_t cfg, float* energy, float* clip_out, awq_stream_t stream);

/*
 * awq_quantize_pack with each group's magnitudes bounded as awq_clip_search describes:
 *   clip [K/G, N] fp32 ratios in (0, 1] (required; all ones gives awq_quantize_pack's output).
 * Every other argument as for awq_quantize_pack; the packed format is unchanged.
 */
awq_status_t awq_quantize_pack_clip(const void* W_f16, int64_t N, int64_t K, const float* s,
                                    const float* clip, awq_qcfg_t cfg, uint32_t* qweight,
                                    void* scales_f16, uint8_t* zeros, awq_stream_t stream);

/*
 * The quantisation residual of one scale vector: the operand the search scores, one candidate
 * of "AWQ Math", "Searching the scale" (the output error of that candidate is the mean of
 * (X D^T)^2 / 2^(2p) over tokens and outputs).
 *   D = 2^p (W - w_hat),  w_hat = (q - z) step16 / s  element by element,
 * with q, z and step the codes, zero points and fp32 steps awq_quantize_pack produces for s,
 * step16 = fp16(step), the products and the difference IEEE fp32 operations in that order and
 * the result rounded once to fp16; p = 14 - e where max|W| < 2^e <= 2 max|W| (p = 0 for an
 * all-zero W), so that every |D| < 2^14 (|W - w_hat| <= |W| for every weight).
 *   W_f16       [N, K] fp16 row-major
 *   s, inv_s    [K] fp32, both required: the scale and 1 / s (IEEE division), 16-byte aligned
 *   absmax_bits [1] device uint32 out: the fp32 bit pattern of max|W|, from which the caller
 *               reads p; it is also the call's scratch
 *   D_f16       [N, K] fp16 out
 * Two kernels on `stream` (max|W|, then the residual); the search builds the same residual.
 */
awq_status_t awq_quant_residual(const void* W_f16, int64_t N, int64_t K, const float* s,
                                const float* inv_s, awq_qcfg_t cfg, uint32_t* absmax_bits,
                                void* D_f16, awq_stream_t stream);

/*
 * W4A16 dequant-fused matmul: Y [M, N] fp16 = X [M, K] fp16 @ (dequant(Q) diag(inv_s))^T,
 * fp32 accumulation. inv_s [K] fp32 or NULL (1/s already folded into the previous layer).
 * M <= 4 runs a CUDA-core GEMV (integer inner products on block fixed-point activations)
 * where its K parts fit its 15 consumer warps and its shared memory (K up to 61440, 30720 and
 * 15360 channels at M = 1, 2 and 3-4); otherwise M <= 16 with G >= 64 the tcgen05 grouped
 * kernel, and every other M the tcgen05 dequant kernel. With inv_s,
 * X * inv_s must stay inside the fp16 range (as the folded activation would).
 */
awq_status_t awq_w4a16_gemm(const void* X_f16, int64_t M, int64_t N, int64_t K,
                            const uint32_t* qweight, const void* scales_f16,
                            const uint8_t* zeros, const float* inv_s, awq_qcfg_t cfg,
                            void* Y_f16, awq_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* awq_status_string(awq_status_t status);

/*
 * Synchronises `stream`, then reads and clears the device status word of the current device:
 * AWQ_ERR_TIMEOUT if a kernel gave up a bounded wait since the last call, AWQ_ERR_CUDA if the
 * synchronisation failed, else AWQ_OK.
 */
awq_status_t awq_stream_status(awq_stream_t stream);

/* Number of kernels this library has launched in this process (diagnostic counter). */
uint64_t awq_launch_count(void);

/*
 * Limit, in nanoseconds, of every bounded device-side wait in later launches (default 2e9).
 * Returns the previous value. A kernel that gives up records AWQ_ERR_TIMEOUT (see
 * awq_stream_status); its outputs are then undefined, the context stays usable. The waits by
 * which a giving-up CTA lets its own copies and MMAs in flight finish before it exits keep a
 * floor of 0.5 s, so even 0 exercises the give-up path safely: with 0 a wait that is not
 * already met gives up at once (in practice every pipelined kernel then reports a timeout).
 */
uint64_t awq_set_wait_limit_ns(uint64_t limit_ns);

/*
 * The alpha search without any device allocation, for callers that cannot allocate device
 * memory where they run it (a fixed memory budget set at start-up, a plug-in handed a device
 * but no allocator, a process whose allocations belong to another runtime). The pages have no
 * counterpart to this call; it exists only for such callers.
 *
 * Same arguments and results as awq_search_scale without the workspace: the scratch is a static
 * device array of AWQ_SEARCH_STATIC_SCRATCH_BYTES (40 MiB) inside this library, which every GPU
 * that loads the library holds until the process exits. Shapes whose smallest workspace (one
 * residual buffer, see awq_search_workspace_bytes) exceeds it return AWQ_ERR_WORKSPACE without
 * launching (the 4096 x 4096 layer with 20 alphas needs about 33 MiB); shapes that fit twice
 * over use the overlapped schedule. Arguments are checked exactly as awq_search_scale checks
 * them (same error codes, in the same order) before the size of the shape is compared with the
 * array. The call allocates no device memory.
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress, which
 * may load this library's device code on that device); like the first call of any search entry
 * point on a device, it also creates the library's second stream and the events that order it
 * (see awq_search_scale). Make that first call before any stream capture. Every call shares the one array and leaves its contents behind; the search writes
 * everything it later reads and clears its own max|W| word, so no clearing is needed between
 * calls. Calls whose work overlaps on the GPU (for example on two streams at once) race on the
 * array: serialise them.
 */
#define AWQ_SEARCH_STATIC_SCRATCH_BYTES (40u * 1024u * 1024u)
awq_status_t awq_search_scale_static(const void* W_f16, int64_t N, int64_t K, const void* X_f16,
                                     int64_t T, const float* mean_abs, const float* alphas,
                                     int32_t n_alpha, awq_qcfg_t cfg, float* err_out,
                                     int32_t* best_idx, float* s_out, float* inv_s_out,
                                     awq_stream_t stream);

/*
 * Folding 1/s into the operation that produces the layer's input ("AWQ Math", "The equivalent
 * transform": W' = W diag(s) on x' = diag(s)^-1 x gives the same output, so the quantised
 * layer can run with inv_s = NULL once the previous operation emits x / s; "AWQ > Benefits and
 * Practical Considerations": the scale folds into the previous layer).
 *   A_f16 [rows, cols] fp16 row-major, row stride lda >= cols, modified in place:
 *         A[r][c] = fp16_rne(fl32(A[r][c] * row_scale[r]))   (one IEEE fp32 multiply)
 *   row_scale [rows] fp32 (pass inv_s).
 * For the previous linear, A is its weight [C_out = K, C_in] (row k = output channel k); for a
 * norm's weight vector, rows = K and cols = lda = 1.
 */
awq_status_t awq_scale_rows(void* A_f16, int64_t rows, int64_t cols, int64_t lda,
                            const float* row_scale, awq_stream_t stream);

/*
 * The two elementwise operations of a Llama-style MLP block (RMSNorm -> gate/up -> SiLU(gate) *
 * up -> down), for running the block end to end around the quantised linears. They are the
 * block's own operations, not part of AWQ.
 *   awq_rmsnorm:  Y[t][j] = fp16(X[t][j] * r_t * gamma[j]), r_t = 1 / sqrt(mean_j X[t][j]^2 +
 *                 eps); X, Y [T, D] fp16 (D % 8 == 0), gamma [D] fp16; fp32 arithmetic, the
 *                 sum of squares in a fixed order (deterministic).
 *   awq_silu_mul: H[i] = fp16(silu(G[i]) * U[i]), silu(g) = g / (1 + e^-g); n % 8 == 0; fp32.
 */
awq_status_t awq_rmsnorm(const void* X_f16, int64_t T, int64_t D, const void* gamma_f16,
                         float eps, void* Y_f16, awq_stream_t stream);
awq_status_t awq_silu_mul(const void* G_f16, const void* U_f16, int64_t n, void* H_f16,
                          awq_stream_t stream);

/* Kernels of this library, as counted by the profiling calls below. */
typedef enum {
  AWQ_K_CALIB_STATS = 0, /* awq_calib_stats (and the search when mean_abs is NULL) */
  AWQ_K_SCALE_GRID = 1,  /* search: s and 1/s for every alpha */
  AWQ_K_ABSMAX = 2,      /* search: max|W| for the residual's power-of-two scale */
  AWQ_K_RESIDUAL = 3,    /* search: W - Q(W diag s) diag(s)^-1 of one alpha, fp16 */
  AWQ_K_SCORE = 4,       /* search, DIRECT: tcgen05 sum of squares of X D^T of one alpha */
  AWQ_K_FINALIZE = 5,    /* search: errors, argmin, winning scales */
  AWQ_K_QUANTIZE_PACK = 6,
  AWQ_K_GEMV = 7,        /* awq_w4a16_gemm, CUDA-core kernel for M <= 4 */
  AWQ_K_GEMM_TC = 8,     /* awq_w4a16_gemm, tcgen05 kernels for larger M */
  AWQ_K_GRAM_PREP = 9,   /* search, GRAM: X^T, column sums of squares and their maximum */
  AWQ_K_GRAM = 10,       /* search, GRAM_LAUNCHES: tcgen05 lower triangle of H = X^T X, fp16 */
  AWQ_K_SCORE_GRAM = 11, /* search, GRAM_LAUNCHES: tcgen05 sum_n d_n^T H d_n of one alpha */
  AWQ_K_GRAM_SEARCH = 12, /* search, GRAM: persistent launch over H and every alpha */
  AWQ_K_SCALE_ROWS = 13,  /* awq_scale_rows */
  AWQ_K_RMSNORM = 14,     /* awq_rmsnorm */
  AWQ_K_SILU_MUL = 15,    /* awq_silu_mul */
  AWQ_K_CLIP_SEARCH = 16, /* awq_clip_search (its channel-energy kernel counts as calib_stats) */
  AWQ_K_COUNT = 17
} awq_kernel_id_t;

/*
 * Profiling aid. After awq_profile_begin, every launch of this library (any thread, any
 * stream) is bracketed by a CUDA event pair recorded on its own stream. awq_profile_end
 * synchronises those events, stops recording and writes, per awq_kernel_id_t, the summed
 * kernel time in ms (total_ms[AWQ_K_COUNT]) and the launch count (launches[AWQ_K_COUNT]);
 * either output may be NULL. Events are created on first use and reused.
 */
awq_status_t awq_profile_begin(void);
awq_status_t awq_profile_end(double* total_ms, uint64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_H_ */
