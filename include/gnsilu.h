/*
 * gnsilu.h -- C ABI of libgnsilu: channels-last GroupNorm (+SiLU) on GB300,
 * and the decoder operations next to it.
 *
 * The operation (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
 * quality=high", section "Modifications", item 1): x is bf16 in (N, L, C)
 * rows with C innermost -- a channels_last (N, C, H, W) tensor seen through a
 * free permute view, L = H*W.  For each batch entry n and each of the G
 * channel groups g (Cg = C/G consecutive channels), over the L*Cg elements:
 *
 *     mean[n,g] = average of x          var[n,g] = biased variance of x
 *     rstd[n,g] = 1 / sqrt(var[n,g] + eps)
 *     scale[n,c] = gamma[c] * rstd[n,g]          (affine folded per channel)
 *     shift[n,c] = beta[c] - mean[n,g] * scale[n,c]
 *     y = x * scale + shift, then y = y * sigmoid(y) when apply_silu != 0
 *
 * computed as a pass-1 partial reduction, a finalize step and a pass-2
 * elementwise apply (the two-pass structure on that page), with fp32
 * statistics and one round-to-nearest-even rounding of y to bf16.
 *
 * Supported inputs (the page's "unsupported inputs are rejected" contract,
 * same section, item 1, second bullet): C a power of two in [8, 2048],
 * G >= 1 dividing C,
 * N, L >= 1.  Unsupported inputs return a non-zero status and touch nothing.
 * Two further entry points, gn_silu_rows_any() and gn_silu_ndhwc(), widen C
 * to any multiple of 8 up to 2048 (any channels per group, e.g. C = 320 or
 * 960) and add 5D channels-last input: the range the page's existing
 * general kernel serves (same section, item 1, third bullet).
 *
 * The library also carries the neighbouring decoder operations the pages
 * describe, each declared further down with its own definition and
 * contract: the residual-gate update residual + gate * update
 * (gn_residual_gate_add), the fused nearest-2x upsample + 3x3 convolution
 * (gn_upconv_fold, gn_upconv_nhwc) and the single-head attention with its
 * output projection folded into V (gn_attn_fold, gn_attn_folded); the last
 * two run on the tensor cores.
 *
 * Memory and streams: every pointer argument is a DEVICE pointer owned by
 * the caller; the library never frees caller memory.  x and y are bf16
 * (uint16 bit patterns) [N][L][C] contiguous, 16-byte aligned; gamma and
 * beta are fp32 [C], 4-byte aligned.  y may equal x exactly (in place) but
 * must not overlap it otherwise, nor overlap gamma or beta.  Work is
 * enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream)
 * and the call returns without synchronising: a return of GN_OK means the
 * arguments were valid and the kernels were launched.  Faults that happen
 * later surface at the caller's next synchronisation.  Every wait inside a
 * kernel is bounded; a kernel that gives up one records a sticky status in
 * device memory and in a word of page-locked host memory mapped into the
 * device.  From the moment that host word is set, every entry point that
 * launches kernels returns GN_ERR_KERNEL without launching, until
 * gn_device_status(1) clears it (calls enqueued before then return GN_OK,
 * and their kernels return at once without writing any output).
 *
 * Thread safety: calls from several host threads are safe.  Calls on
 * different streams of one device that use the library's own workspace are
 * safe (the workspace is kept per device and stream, for up to eight streams
 * per device; a further stream takes the place of the least recently used
 * one, whose workspace is freed after a device synchronisation); two calls
 * that share one caller-provided workspace must not overlap on the GPU.
 *
 * Device reset: the library keeps per-device state (kernel attributes, its
 * workspaces, the mapped status word, the static scratch address).
 * cudaDeviceReset() destroys what that state refers to; a process that
 * resets a device must not call the library on that device afterwards.
 */
#ifndef GNSILU_H
#define GNSILU_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum gn_status_code {
    GN_OK = 0,
    GN_ERR_NULL = 1,       /* a required pointer is NULL */
    GN_ERR_SHAPE = 2,      /* N, L (or H, W) < 1, or the element count overflows */
    GN_ERR_CHANNELS = 3,   /* C not a power of two in [8, 2048] (for gn_silu_rows_any and
                              gn_silu_ndhwc: not a multiple of 8 in [8, 2048]),
                              G < 1 or C % G != 0 */
    GN_ERR_ALIGN = 4,      /* x or y not 16-byte aligned; gamma, beta, mean/rstd outputs
                              not 4-byte aligned; workspace not 256-byte aligned */
    GN_ERR_EPS = 5,        /* eps not finite or negative */
    GN_ERR_ALIAS = 6,      /* y overlaps x without being equal to it, or overlaps
                              gamma, beta or a statistics output */
    GN_ERR_WORKSPACE = 7,  /* caller workspace smaller than gn_silu_workspace_bytes() */
    GN_ERR_CUDA = 8,       /* a CUDA runtime call or kernel launch failed */
    GN_ERR_DEVICE = 9,     /* no CUDA device, or the current device is not sm_103 */
    GN_ERR_VARIANT = 10,   /* unknown variant, or the fused variant cannot be
                              launched cooperatively for this shape, or the
                              cluster variant does not fit it */
    GN_ERR_KERNEL = 11,    /* a kernel gave up a bounded wait and the status has not
                              been cleared (gn_device_status(1)) since; nothing ran */
    GN_ERR_FORMAT = 12     /* gn_residual_gate_add(): unknown half format */
};

/* Element formats of gn_residual_gate_add(). */
enum gn_half_format {
    GN_FORMAT_BF16 = 0,
    GN_FORMAT_FP16 = 1
};

/* Kernel schedules selectable through gn_silu_rows_ex(). */
enum gn_variant {
    GN_VARIANT_AUTO = 0,      /* the library picks (fused when it can launch) */
    GN_VARIANT_TWO_PASS = 1,  /* three launches: pass 1, finalize, pass 2 */
    GN_VARIANT_FUSED = 2,     /* one cooperative launch: pass 1, grid barrier,
                                 finalize, grid barrier, pass 2; x re-read from
                                 shared memory / L2 where it still sits there */
    GN_VARIANT_CLUSTER = 3    /* one launch of thread-block clusters, each owning
                                 a slice of whole groups of one batch entry: its
                                 CTAs keep their rows in shared memory, merge the
                                 group statistics over distributed shared memory
                                 and write y; x is read from HBM once and no
                                 workspace is used.  Only for tensors whose
                                 slices fit the clusters' shared memory (about
                                 2 MiB of one batch entry's slice per cluster):
                                 GN_ERR_VARIANT otherwise.  GN_VARIANT_AUTO picks
                                 it for small tensors (up to a few MiB), where it
                                 is the fastest schedule */
};

/*
 * GroupNorm(+SiLU) of a channels_last (N, C, H, W) bf16 tensor, whose memory
 * is [N][H][W][C].  Identical to gn_silu_rows() with L = H * W (the page's
 * 4D entry served "via a free permute view").
 */
int gn_silu_nhwc(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16,
                 int64_t N, int64_t H, int64_t W, int64_t C, int64_t G,
                 float eps, int apply_silu, void *stream);

/*
 * GroupNorm(+SiLU) of (N, L, C) bf16 rows, channels innermost (the page's
 * rows entry, "as used by attention").  Uses a workspace the library
 * allocates on first use for each (device, stream) and grows when a larger
 * shape arrives; that first call allocates (cudaMalloc) and so should come
 * before any CUDA graph capture on the stream.  gn_release_workspaces()
 * frees these workspaces.
 */
int gn_silu_rows(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16,
                 int64_t N, int64_t L, int64_t C, int64_t G,
                 float eps, int apply_silu, void *stream);

/*
 * gn_silu_rows() with the statistics exported and the schedule and the
 * workspace chosen by the caller.
 *   mean_out, rstd_out : device fp32 [N * G] (index n * G + g), or NULL.
 *   workspace          : device memory of at least
 *                        gn_silu_workspace_bytes(N, L, C, G) bytes, 256-byte
 *                        aligned, whose first 256 bytes are zero before its
 *                        first use (cudaMemset once; the kernels leave them
 *                        zero again after every successful call).  NULL
 *                        selects the library's own workspace.
 *   variant            : enum gn_variant.
 */
int gn_silu_rows_ex(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16,
                    int64_t N, int64_t L, int64_t C, int64_t G,
                    float eps, int apply_silu,
                    float *mean_out, float *rstd_out,
                    void *workspace, size_t workspace_bytes, int variant, void *stream);

/*
 * gn_silu_rows_ex() for any channel count C that is a multiple of 8 in
 * [8, 2048] and any G dividing C -- every channels-per-group Cg = C / G,
 * including the non-power-of-two C of the page's existing general kernel
 * ("any channels-per-group", sglang PR #33451, section "Modifications",
 * item 1, third bullet).  The operation, arguments, alignment, aliasing,
 * workspace and status codes are those of gn_silu_rows_ex(); the kernels are
 * the same, with the per-vector channel bookkeeping done by division instead
 * of shifts.  For a power-of-two C the results equal gn_silu_rows_ex()'s
 * bit for bit.  C not a multiple of 8 (a row that is not whole 16-byte
 * vectors) gives GN_ERR_CHANNELS.
 */
int gn_silu_rows_any(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16,
                     int64_t N, int64_t L, int64_t C, int64_t G,
                     float eps, int apply_silu,
                     float *mean_out, float *rstd_out,
                     void *workspace, size_t workspace_bytes, int variant, void *stream);

/*
 * GroupNorm(+SiLU) of a 5D channels-last bf16 tensor (N, C, D, H, W) whose
 * memory is [N][D][H][W][C] (torch.channels_last_3d), such as the
 * HunyuanVAE-style video latents the page's general kernel serves (same
 * section, item 1, third bullet; "Speedup", note under the kernel table).
 * Statistics run over all D*H*W positions and the Cg channels of a group;
 * identical to gn_silu_rows_any() with L = D * H * W, the library's own
 * workspace and the automatic schedule.  C: a multiple of 8 in [8, 2048].
 */
int gn_silu_ndhwc(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16,
                  int64_t N, int64_t D, int64_t H, int64_t W, int64_t C, int64_t G,
                  float eps, int apply_silu, void *stream);

/* Workspace bytes gn_silu_rows_ex() / gn_silu_rows_any() need for this shape
 * on the CURRENT device (any variant).  Accepts any C that is a multiple of
 * 8 in [8, 2048].  Returns 0 if the shape is unsupported or there is no
 * usable device. */
size_t gn_silu_workspace_bytes(int64_t N, int64_t L, int64_t C, int64_t G);

/* The variant GN_VARIANT_AUTO resolves to for this shape on the current
 * device, or a negative status code. */
int gn_silu_pick_variant(int64_t N, int64_t L, int64_t C, int64_t G);

/* Number of CUDA kernels this library launched since the process started
 * (all devices, all streams). */
uint64_t gn_kernel_launch_count(void);

/* Synchronises the current device, then returns GN_OK or GN_ERR_KERNEL if
 * one of this library's kernels gave up a bounded wait since the last clear
 * (GN_ERR_CUDA / GN_ERR_DEVICE if the device itself reports an error).
 * While that flag is set the entry points return GN_ERR_KERNEL, and kernels
 * enqueued before it was set return at once without writing any output.
 * clear != 0 resets the flag (on the device and in host memory) and
 * re-zeroes the library's own workspaces on this device; a caller-provided
 * workspace must then be re-zeroed by the caller. */
int gn_device_status(int clear);

/* Synchronises the current device and frees every workspace the library
 * allocated on it (those of gn_silu_rows, gn_silu_nhwc, gn_silu_ndhwc and of
 * gn_silu_rows_ex / gn_silu_rows_any called without a workspace).  Later
 * calls allocate again.  Must not be called while a stream of the device is
 * being captured.  Returns GN_OK, GN_ERR_DEVICE or GN_ERR_CUDA. */
int gn_release_workspaces(void);

/* Number of workspaces the library currently holds on the current device
 * (at most eight), or a negative status code. */
int gn_library_workspaces(void);

/* Diagnostic of the kernels' failure handling: launches `blocks` CTAs that
 * each wait for something nothing will ever do -- mode 0: an mbarrier phase
 * no thread arrives on; mode 1: a barrier count no CTA reaches -- bounded by
 * timeout_ms (0..10000).  Each CTA must give up, record the sticky status
 * that gn_device_status() reports as GN_ERR_KERNEL, write 1 to
 * done[blockIdx] (device int array) and return.  The caller clears the
 * status afterwards with gn_device_status(1).  Asynchronous on `stream`. */
int gn_selftest_bounded_wait(int mode, int timeout_ms, int *done, int blocks, void *stream);

/* Size of the fixed scratch array used by gn_silu_rows_static(): 8 MiB. */
#define GN_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * gn_silu_rows_ex() for callers that cannot allocate device memory.  (This
 * entry point has no counterpart on the sglang PR #33451 page; it is a
 * deployment convenience of this library.)
 *
 * Who needs it: a plug-in inside a host framework that owns every byte of
 * device memory through its own pool and accounting, and so may not
 * allocate behind the framework's back; a latency-critical path that cannot
 * afford the device-wide synchronisation and unbounded time of an
 * allocation or a free; a process under a fixed device-memory budget that
 * cannot count on an allocation succeeding mid-run.  gn_silu_rows()
 * allocates its workspace on first use, and gn_silu_rows_ex() needs one from
 * the caller; this entry point needs neither.
 *
 * The scratch (partial statistics and grid-barrier words) comes from one
 * fixed array of GN_STATIC_SCRATCH_BYTES compiled into the library, which
 * every GPU that loads the library holds until the process exits.  No call
 * to cudaMalloc, cudaFree or any other allocating routine is made.
 *   - Shapes whose scratch need (gn_silu_workspace_bytes) exceeds
 *     GN_STATIC_SCRATCH_BYTES are refused with GN_ERR_WORKSPACE and nothing
 *     runs.  The need is about 8 C N + 16 G N + 8 G max(N, 152) + 2 KB
 *     on a GB300 (152 SMs): with C = 2048 and G = 32 that covers N up to
 *     about 490.
 *   - Every argument check runs before the array is touched: a refused
 *     call (any non-zero status) writes nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and the first call
 *     of the library on a device sets the device up (kernel attributes, the
 *     mapped status word), which takes device-wide CUDA calls.
 *   - All calls on a device share the one array, which keeps the previous
 *     call's contents; each call clears the words that must start at zero
 *     (an asynchronous memset on `stream`).  Calls whose GPU work overlaps
 *     -- on different streams, or from different host threads -- race on
 *     the array and must be serialised by the caller.
 * Arguments, outputs, statistics and status codes are those of
 * gn_silu_rows_ex() with the automatic schedule.
 */
int gn_silu_rows_static(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16,
                        int64_t N, int64_t L, int64_t C, int64_t G,
                        float eps, int apply_silu,
                        float *mean_out, float *rstd_out, void *stream);

/*
 * Residual-gate update of a transformer's residual stream (the prhub digest
 * of sglang PR #33823, FLUX.2 bit-exact residual-gate fusion, sections
 * "Functions and motivation" and "Implementation breakdown", items 1-3):
 *
 *     out[r, d] = residual[r, d] + gate[d] * update[r, d]
 *
 * in half precision, bit for bit equal to the eager two-kernel evaluation
 * (the product rounded to the half format, then the sum rounded to it;
 * round to nearest even, no fused multiply-add).  NaN results may carry any
 * NaN payload.
 *   residual, update, out : DEVICE [rows][D] bf16 or fp16 bit patterns
 *                           (format: enum gn_half_format), contiguous,
 *                           16-byte aligned.
 *   gate                  : DEVICE [D] of the same format, 16-byte aligned:
 *                           one row broadcast over all rows (a [1, ..., 1, D]
 *                           modulation vector; per-batch gates are not
 *                           taken, as on the page).
 *   rows >= 0 (0: nothing to do), D a multiple of 8 (whole 16-byte vectors).
 * out may equal residual or update exactly (in place) but must not overlap
 * them otherwise, nor overlap gate.  Asynchronous on `stream`, like the
 * other entry points; the caller owns every buffer.  Errors: GN_ERR_NULL,
 * GN_ERR_SHAPE (rows < 0 or the element count overflows), GN_ERR_CHANNELS
 * (D < 8 or not a multiple of 8), GN_ERR_ALIGN, GN_ERR_ALIAS, GN_ERR_FORMAT,
 * GN_ERR_DEVICE, GN_ERR_CUDA.
 */
int gn_residual_gate_add(const void *residual, const void *update, const void *gate, void *out,
                         int64_t rows, int64_t D, int format, void *stream);

/* ---- fused nearest-2x upsample + 3x3 convolution ---------------------------
 * The decoder's up-sampler (sglang PR #33451, "FLUX.2 VAE decoder fast path
 * behind quality=high", section "Modifications", item 2): a nearest-neighbour
 * 2x upsample followed by a 3x3 convolution with padding 1,
 *
 *   y[n][P][Q][co] = bias[co] + sum_{ky,kx,ci} u[n][P+ky-1][Q+kx-1][ci] * w[co][ci][ky][kx]
 *   u[n][p][q][ci] = x[n][p/2][q/2][ci] inside the 2H x 2W image, 0 outside,
 *
 * evaluated without materialising u: an output pixel of parity (P mod 2,
 * Q mod 2) sees a 2x2 input window whose taps are sums of the 3x3 taps (the
 * transposed convolution with kernel 4, stride 2, padding 1 that the page
 * names).  Two calls: gn_upconv_fold() turns the weight into those summed
 * taps once (fp32 sums rounded to bf16), gn_upconv_nhwc() runs the
 * convolution on the tensor cores (fp32 accumulation, bf16 output).  The
 * summed taps are rounded to bf16, so the result differs from the unfused
 * evaluation by rounding: per output less than 2^-7 of the sum of
 * |x * w| over its 9 Cin terms plus 2^-7 |y|.
 */

/* Bytes of the folded weight: [4 parities][Cout][4 taps][Cin] bf16
 * (16 Cin Cout 2 bytes), or -1 if Cin or Cout is out of range. */
int64_t gn_upconv_folded_bytes(int64_t Cin, int64_t Cout);

/* Fold the convolution weight.
 *   w  : DEVICE [Cout][Cin][3][3] bf16 (the convolution's own layout),
 *        2-byte aligned.
 *   wf : DEVICE, gn_upconv_folded_bytes(Cin, Cout) bytes, 16-byte aligned,
 *        not overlapping w; row p Cout + co holds the 4 Cin summed taps of
 *        output channel co for parity p = 2 (P mod 2) + (Q mod 2), taps
 *        ordered (r, s, ci) with window row r and column s in {0, 1}.
 *   Cin a multiple of 64 in [64, 8192]; Cout a multiple of 128 in [128, 8192].
 * Asynchronous on `stream`.  Errors: GN_ERR_NULL, GN_ERR_CHANNELS,
 * GN_ERR_ALIGN, GN_ERR_ALIAS, GN_ERR_DEVICE, GN_ERR_CUDA. */
int gn_upconv_fold(const void *w_bf16, void *wf_bf16, int64_t Cin, int64_t Cout, void *stream);

/* The upsample + convolution.
 *   x    : DEVICE [N][H][W][Cin] bf16 (channels-last), 16-byte aligned.
 *   wf   : DEVICE folded weight from gn_upconv_fold(), 16-byte aligned.
 *   bias : DEVICE [Cout] bf16, 4-byte aligned, or NULL for none.
 *   y    : DEVICE [N][2H][2W][Cout] bf16 (channels-last), 16-byte aligned,
 *          overlapping none of the inputs.
 *   N >= 0 (0: nothing to do); Cin and Cout as for gn_upconv_fold();
 *   W a multiple of 128, or a power of two below 128 with H either a
 *   multiple of 128 / W or a power of two below it (tiles of 128 output
 *   pixels of one parity never straddle a row or image edge).
 * Asynchronous on `stream`; the caller owns every buffer.  Errors:
 * GN_ERR_NULL, GN_ERR_SHAPE (N < 0, H or W < 1 or not tileable as above,
 * sizes overflow), GN_ERR_CHANNELS, GN_ERR_ALIGN, GN_ERR_ALIAS,
 * GN_ERR_DEVICE, GN_ERR_CUDA.  A bounded wait that expires inside the kernel
 * is reported by gn_device_status() as GN_ERR_KERNEL. */
int gn_upconv_nhwc(const void *x_bf16, const void *wf_bf16, const void *bias_bf16, void *y_bf16, int64_t N,
                   int64_t H, int64_t W, int64_t Cin, int64_t Cout, void *stream);

/* ---- single-head attention with the output projection folded into V -------
 * The VAE mid-block attention after its GroupNorm and its query / key
 * projections (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
 * quality=high", section "Modifications", item 2, attention bullet):
 *
 *   out = softmax(q k^T / sqrt(D)) (xn wv^T + bv) wo^T + bo + residual
 *       = softmax(q k^T / sqrt(D)) (xn W'^T + b') + residual,
 *   W' = wo wv,  b' = wo bv + bo
 *
 * (exact because every softmax row sums to 1).  gn_attn_fold() forms W'
 * (fp32 sums rounded once to bf16) and b' (fp32) once per weight;
 * gn_attn_folded() evaluates the second form on the tensor cores (fp32
 * accumulation), first the folded value rows, then the softmax and the
 * weighted sum by one of two schedules:
 *   GN_ATTN_ONE_PASS: one pass over the keys per tile of 128 query rows,
 *     on pairs of CTAs (D <= 512): the scores stay on chip (tensor memory),
 *     the weights go from one CTA of the pair to the other through
 *     distributed shared memory; a running row maximum rescales the output
 *     when it moves.  The pairs share the (query tile, key block) units
 *     equally; a tile split between pairs leaves its pieces (unnormalised
 *     output, row maxima and sums) in the workspace, and a third kernel
 *     merges them.
 *   GN_ATTN_STORED_WEIGHTS: the fp32 scores twice -- once reduced to each
 *     row's softmax maximum and sum, once written to the workspace as
 *     softmax weights rounded to bf16 -- then the weighted sum as a GEMM.
 * Both round the weights to bf16 before the weighted sum.  GN_ATTN_AUTO
 * takes the one-pass schedule when D <= 512 and there are at least 32 query
 * tiles (S >= 4096): with fewer tiles it leaves most SMs idle and the
 * stored-weights schedule is faster.
 */

/* Schedules of gn_attn_folded_ex(). */
enum { GN_ATTN_AUTO = 0, GN_ATTN_ONE_PASS = 1, GN_ATTN_STORED_WEIGHTS = 2 };

/* Fold the value projection (wv [D][D], bv [D]) and the output projection
 * (wo [D][D], bo [D]) -- DEVICE bf16, PyTorch Linear layout [out][in],
 * 2-byte aligned -- into wf (DEVICE bf16 [D][D], 16-byte aligned) and bf
 * (DEVICE fp32 [D], 16-byte aligned); the outputs overlap no input.
 * D a multiple of 128 in [128, 1024].  Asynchronous on `stream`.  Errors:
 * GN_ERR_NULL, GN_ERR_CHANNELS, GN_ERR_ALIGN, GN_ERR_ALIAS, GN_ERR_DEVICE,
 * GN_ERR_CUDA. */
int gn_attn_fold(const void *wv_bf16, const void *bv_bf16, const void *wo_bf16, const void *bo_bf16,
                 void *wf_bf16, float *bf, int64_t D, void *stream);

/* Workspace bytes gn_attn_folded() needs for S tokens of width D, whatever
 * the schedule: the folded value rows (2 D S bytes), per-row-segment softmax
 * records (16 S^2 / 128 bytes), the rows' softmax statistics (8 S) and the
 * bf16 softmax weights (2 S^2), each rounded up to 256 bytes (the one-pass
 * schedule keeps the pieces of split tiles where the others would be);
 * 0 if S or D is out of range. */
size_t gn_attn_workspace_bytes(int64_t S, int64_t D);

/* The folded attention.
 *   q, k, xn  : DEVICE bf16 [S][D], 16-byte aligned (query / key
 *               projections and the GroupNorm output).
 *   wf, bf    : from gn_attn_fold().
 *   residual  : DEVICE bf16 [S][D] added to the result, or NULL; may equal
 *               out (in place) but not overlap it otherwise.
 *   out       : DEVICE bf16 [S][D], 16-byte aligned, overlapping no input.
 *   workspace : DEVICE, workspace_bytes >= gn_attn_workspace_bytes(S, D),
 *               256-byte aligned, caller-owned, overlapping nothing else;
 *               all workspace_bytes of it may be used (the one-pass
 *               schedule keeps there the pieces of query tiles it splits
 *               between CTA pairs, and splits more finely when given more).
 *   S a multiple of 128 in [128, 32768]; D as for gn_attn_fold().
 * Asynchronous on `stream`.  Errors: GN_ERR_NULL, GN_ERR_SHAPE (S),
 * GN_ERR_CHANNELS (D), GN_ERR_ALIGN, GN_ERR_ALIAS, GN_ERR_WORKSPACE,
 * GN_ERR_DEVICE, GN_ERR_CUDA; a bounded wait that expires inside a kernel
 * is reported by gn_device_status() as GN_ERR_KERNEL. */
int gn_attn_folded(const void *q_bf16, const void *k_bf16, const void *xn_bf16, const void *wf_bf16, const float *bf,
                   const void *residual_bf16, void *out_bf16, int64_t S, int64_t D, void *workspace,
                   size_t workspace_bytes, void *stream);

/* gn_attn_folded() with the schedule named (GN_ATTN_*).  Errors as for
 * gn_attn_folded(), and GN_ERR_VARIANT for an unknown schedule or
 * GN_ATTN_ONE_PASS with D > 512. */
int gn_attn_folded_ex(const void *q_bf16, const void *k_bf16, const void *xn_bf16, const void *wf_bf16,
                      const float *bf, const void *residual_bf16, void *out_bf16, int64_t S, int64_t D,
                      void *workspace, size_t workspace_bytes, int schedule, void *stream);

/* Human-readable name of a status code (static storage). */
const char *gn_status_string(int status);

/* ABI version of this header: 7 (6 lacked gn_attn_folded_ex; 5 also lacked
 * gn_release_workspaces and gn_library_workspaces, and its entry points did
 * not return GN_ERR_KERNEL;
 * 4 also lacked the gn_attn_* calls; 3 also the gn_upconv_* calls; 2 also
 * gn_residual_gate_add; 1 also gn_silu_rows_any and gn_silu_ndhwc). */
int gn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GNSILU_H */
