/*
 * coda.h -- C ABI of libcoda.so: the GEMM -> residual -> RMSNorm -> GEMM chain
 *
 *     h = x @ W0 + z                      (new residual stream)
 *     r = 1 / sqrt(mean_j h^2 + eps)      (one float per row)
 *     y = RMSNorm(h, gamma) @ W1 = r * ((h * gamma) @ W1)
 *
 * computed as two GEMM-epilogue programs on an sm_103a GPU, and its
 * data-gradient twin grad_h = RMSNormBackward(grad_y @ W1^T).
 *
 * Source of the method: "CODA：将 Transformer 块重写为 GEMM-Epilogue 程序以消除显存瓶颈"
 * (blog.hotdry.top), section "GEMM-Residual-RMSNorm-GEMM 重参数化" (the
 * reparameterisation and its three steps) and section
 * "反向传播的 GEMM-Epilogue 结构" (the backward keeps the GEMM-epilogue shape; the
 * row statistic s = sum_cols(grad_h2 * h2) = sum_cols(grad_y * y) is formed at
 * the GEMM boundary).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor pointers are DEVICE pointers (memory of the current CUDA
 *    device), row-major and densely packed.  bf16 tensors hold IEEE bfloat16
 *    bit patterns (coda_bf16).  Weights are stored [in, out]:
 *    W0 is [d, d], W1 is [d, N1].
 *  - Every pointer must be 16-byte aligned.  Outputs must not alias inputs or
 *    each other.
 *  - Shapes: M >= 0 rows (M == 0 is a no-op that returns CODA_OK), d and N1
 *    positive multiples of 8 (rows must start on 16-byte boundaries), all
 *    below 2^31.
 *  - The caller owns every buffer, including the workspace; the library never
 *    allocates, frees or synchronises inside coda_fwd / coda_bwd_dgrad.  Work
 *    is enqueued asynchronously on `stream` (0 = legacy default stream).
 *  - Workspaces need no clearing and one buffer may serve any sequence of
 *    calls, of any shape and entry point, as long as calls sharing it do not
 *    run concurrently.  Its first 256 bytes hold a launch counter that no
 *    layout puts data into; launches whose blocks exchange completion flags
 *    tag them with the counter's next value mixed with a random 64-bit salt
 *    drawn for each call (kept by a call captured in a CUDA graph, whose
 *    replays the counter tells apart).  Flags of earlier launches on the same
 *    counter never match, and other contents of the buffer (earlier data,
 *    another buffer's flags recycled by an allocator) match only by a 2^-64
 *    coincidence.
 *  - Argument checks happen before anything is enqueued; on any error nothing
 *    is launched.  Device-side failures (a bounded wait that ran out) are
 *    reported later by coda_get_device_status().
 *  - Every kernel is launched with programmatic stream serialisation: it may
 *    begin its prologue while the kernel before it in `stream` is finishing,
 *    and it reads no memory before that kernel has completed.  Stream order is
 *    kept as for ordinary launches, whatever kernel precedes it.
 *  - Numerics: bf16 operands, fp32 accumulation in tensor memory, fp32
 *    epilogue arithmetic, bf16 round-to-nearest-even stores.
 */
#ifndef CODA_H_
#define CODA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define CODA_API __attribute__((visibility("default")))
#else
#define CODA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t coda_bf16; /* IEEE bfloat16 bit pattern */

typedef enum {
  CODA_OK = 0,
  CODA_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad eps */
  CODA_ERR_UNSUPPORTED_SHAPE = 2,  /* d or N1 not a positive multiple of 8, or too large */
  CODA_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
  CODA_ERR_WORKSPACE_TOO_SMALL = 4,
  CODA_ERR_LAUNCH = 5,             /* a CUDA launch or tensor-map encode failed */
  CODA_ERR_DEVICE_TIMEOUT = 6,     /* a bounded device-side wait ran out */
  CODA_ERR_NO_DEVICE = 7,          /* no CUDA device is current */
  CODA_ERR_UNSUPPORTED_DEVICE = 8, /* the current device is not compute capability 10.3 */
  CODA_ERR_DEVICE_BOUNDS = 9       /* checked build only: a device-side bounds or alignment check failed */
} coda_status_t;

/* Bytes of device workspace coda_fwd needs: the 256-byte slot of the launch
 * counter, the bf16 GEMM1 operand hg = h * gamma ([M, d]) and the fp32
 * partial sums of h^2, two per row and 256-column tile, then the split-tail
 * region of the two GEMMs: up to min(T, 160) partial accumulators of
 * 256 x 256 fp32 (T = the larger GEMM's count of 256 x 256 tiles) and one
 * 64-bit flag per 128-row half of each.  Returns 0 for M == 0. */
CODA_API size_t coda_fwd_workspace_bytes(int64_t M, int64_t d, int64_t N1);

/* Bytes of device workspace coda_bwd_dgrad needs: the 256-byte slot holding
 * the launch counter and its arrival word, fp32 partial row statistics (two
 * per row and column tile), one 64-bit completion flag per 128-row slab and
 * column tile, and min(3 T, 192) fp32 partial accumulators of 256 x 256 with
 * their flags for the pieces of the last row blocks (T = the count of
 * 256 x 256 tiles; see coda_set_dgrad_pieces). */
CODA_API size_t coda_bwd_dgrad_workspace_bytes(int64_t M, int64_t d, int64_t N1);

/*
 * Forward of the chain, the method's three steps ("CODA：将 Transformer 块重写为
 * GEMM-Epilogue 程序以消除显存瓶颈", blog.hotdry.top, section
 * "GEMM-Residual-RMSNorm-GEMM 重参数化": GEMM0 does the residual add and the
 * gamma scaling and emits partial sums of squares, a light auxiliary pass forms
 * the inverse RMS r, and GEMM1's epilogue multiplies its output rows by r):
 *   1. GEMM0 epilogue: h = x @ W0 + z (fp32), stores h and hg = h * gamma as
 *      bf16, and writes partial sums of h^2 (fp32, taken before rounding h;
 *      two per row and 256-column tile).
 *   2. auxiliary row reduction: r[m] = 1 / sqrt(sum of partials / d + eps).
 *   3. GEMM1 epilogue: y = r[m] * (hg @ W1), stored bf16.
 * No normalised [M, d] tensor is ever written.
 *
 *   x      [M, d]   bf16 in     z     [M, d]  bf16 in (residual)
 *   W0     [d, d]   bf16 in     gamma [d]     bf16 in (RMSNorm weight)
 *   W1     [d, N1]  bf16 in     eps   >= 0, finite
 *   h_out  [M, d]   bf16 out    (new residual stream; saved for backward)
 *   r_out  [M]      fp32 out    (inverse RMS per row; saved for backward)
 *   y_out  [M, N1]  bf16 out
 *   workspace: device memory of at least coda_fwd_workspace_bytes(M, d, N1)
 *   bytes (the launch counter, hg, the partial sums and the split-tail
 *   region).  Any initial contents work and the call clobbers them, except
 *   that two calls sharing a workspace must not run concurrently.
 * Split tail: when a GEMM's 256 x 256 tiles do not fill whole waves of CTA
 * pairs, its last U + R tiles (U pairs, R tiles past the last full wave) are
 * shared out along K so that every pair ends together; a tile cut in two is
 * finished by the pair holding its first K block, which adds the other pair's
 * fp32 partial (published with a flag whose token comes from the launch
 * counter in the workspace) before the epilogue.  Such a launch is
 * cooperative.  Results then differ from the whole-tile order only in fp32
 * summation order; coda_set_split_tail(0) turns it off.
 */
CODA_API coda_status_t coda_fwd(const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                       const coda_bf16* gamma, const coda_bf16* W1, float eps,
                       int64_t M, int64_t d, int64_t N1,
                       coda_bf16* h_out, float* r_out, coda_bf16* y_out,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Forward of the chain with the SwiGLU gated activation fused into GEMM1's
 * epilogue ("CODA：将 Transformer 块重写为 GEMM-Epilogue 程序以消除显存瓶颈",
 * blog.hotdry.top: SwiGLU gating is one of the section "五类 Epilogue 原语",
 * and section "成对激活的寄存器级融合" fuses the gate/up pair in the epilogue):
 *   steps 1 and 2 as coda_fwd, then GEMM1 with W1 = [W_gate | W_up] ([d, N1],
 *   the usual concatenated layout; no interleaving needed) and epilogue
 *   g = r * (hg @ W_gate),  u = r * (hg @ W_up),  a = silu(g) * u.
 * One accumulator tile holds 128 gate columns and the matching 128 up columns,
 * so each thread, which owns a whole tile row in tensor memory, has both
 * members of every pair; the gated output is the only [M, N1/2] tensor written.
 *   a_out  [M, N1/2] bf16 out   (required)
 *   y_out  [M, N1]   bf16 out   pre-activation [g | u]; may be NULL
 * Other arguments and the workspace as coda_fwd.  N1 must be a multiple of 16.
 */
CODA_API coda_status_t coda_fwd_swiglu(const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                                       const coda_bf16* gamma, const coda_bf16* W1, float eps,
                                       int64_t M, int64_t d, int64_t N1,
                                       coda_bf16* h_out, float* r_out, coda_bf16* y_out,
                                       coda_bf16* a_out, void* workspace, size_t workspace_bytes,
                                       cudaStream_t stream);

/*
 * Forward of the chain with FP8 (E4M3) GEMM operands.  The method's benefit
 * grows as GEMMs get cheaper with low precision ("CODA：将 Transformer 块重写为
 * GEMM-Epilogue 程序以消除显存瓶颈", blog.hotdry.top, opening section; section
 * "实践要点": FP8/FP4 shifts the cost to memory traffic).  Values of FP8 tensors
 * are code * scale (per-tensor fp32 scales > 0):
 *   1. GEMM0 (tcgen05 kind::f8f6f4): h = (x_q @ W0_q) * sx * sW0 + z, stored
 *      bf16; partial sums of h^2; GEMM1's operand quantised once in the
 *      epilogue: hq = E4M3(h * gamma / s_hg), round to nearest even,
 *      saturating at +-448 (the caller picks s_hg, e.g. from a previous amax);
 *   2. r = 1 / sqrt(sum / d + eps);
 *   3. GEMM1: y = r * (s_hg * sW1) * (hq @ W1_q), stored bf16.
 *   x_q [M, d], W0_q [d, d], W1_q [d, N1]: E4M3 codes (1 byte), row-major.
 *   z [M, d], gamma [d] bf16; h_out [M, d] bf16, r_out [M] fp32, y_out [M, N1] bf16.
 *   workspace: at least coda_fwd_fp8_workspace_bytes(M, d, N1) (the launch
 *   counter's slot, hq and the partial sums).
 * d and N1 must be multiples of 16.  Always runs CTA-pair tiles.
 */
CODA_API size_t coda_fwd_fp8_workspace_bytes(int64_t M, int64_t d, int64_t N1);
CODA_API coda_status_t coda_fwd_fp8(const uint8_t* x_q, float sx, const uint8_t* W0_q, float sW0,
                                    const coda_bf16* z, const coda_bf16* gamma,
                                    const uint8_t* W1_q, float sW1, float s_hg, float eps,
                                    int64_t M, int64_t d, int64_t N1,
                                    coda_bf16* h_out, float* r_out, coda_bf16* y_out,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Data gradient through the RMSNorm branch, as one GEMM-epilogue program
 * ("CODA：将 Transformer 块重写为 GEMM-Epilogue 程序以消除显存瓶颈",
 * blog.hotdry.top, section "反向传播的 GEMM-Epilogue 结构": the backward keeps
 * the GEMM-epilogue shape, and the row statistic s = sum_cols(grad_h2 * h2) =
 * sum_cols(grad_y * y) is accumulated in a GEMM's epilogue):
 *   grad_h2 = grad_y @ W1^T  accumulated in tensor memory, then in the epilogue
 *   q[m]    = sum_j grad_h2[m,j] * gamma[j] * h[m,j]  (so s = r * q equals
 *             sum_j grad_h2 * h2 = sum_n grad_y * y), completed across the
 *             row's column tiles through the workspace, and
 *   grad_h  = r * gamma * grad_h2 - (r^3 * q / d) * h,  stored bf16.
 * No separate norm-backward kernel runs and grad_h2 never reaches memory.
 *
 *   dy      [M, N1] bf16 in     W1    [d, N1] bf16 in
 *   h       [M, d]  bf16 in     r     [M]     fp32 in   (both as saved by coda_fwd)
 *   gamma   [d]     bf16 in
 *   dh_out  [M, d]  bf16 out
 *   workspace: at least coda_bwd_dgrad_workspace_bytes(M, d, N1) bytes.  The
 *   completion flags carry a token taken from the launch counter at the
 *   workspace's start, which every launch advances once all its blocks are
 *   done, mixed with the call's salt (see the conventions above): the
 *   workspace needs no clearing, and a call captured in a CUDA graph draws a
 *   fresh token at every replay.  Two calls that share a workspace must not
 *   run concurrently.
 * The kernel is a cooperative launch (all its blocks are resident at once):
 * every column tile of a row block must be in flight together, so d is limited
 * to 256 * (CTA pairs resident on the device) columns, 19456 on a 152-SM GB300
 * (256 * SMs with coda_set_mma_mode(0)); larger d returns
 * CODA_ERR_UNSUPPORTED_SHAPE without launching.  coda_bwd has the same limit.
 */
CODA_API coda_status_t coda_bwd_dgrad(const coda_bf16* dy, const coda_bf16* W1, const coda_bf16* h,
                             const float* r, const coda_bf16* gamma,
                             int64_t M, int64_t d, int64_t N1,
                             coda_bf16* dh_out, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/*
 * Backward of a = silu(g) * u, out = a @ W2, through to grad_h, with the
 * RMSNorm row statistic formed where grad_y and y meet ("CODA：将 Transformer
 * 块重写为 GEMM-Epilogue 程序以消除显存瓶颈", blog.hotdry.top, section
 * "反向传播的 GEMM-Epilogue 结构": s = sum_cols(grad_y * y) accumulated in the
 * epilogue of the GEMM that produces grad_y).  Three launches:
 *   1. da = dout @ W2^T, epilogue: with the saved pre-activation y = [g | u],
 *      dg = da * u * silu'(g), du = da * silu(g) -> dy_out = [dg | du], and
 *      per-tile partial sums of dy * y;
 *   2. s[m] = sum of the partials (light auxiliary reduction) -> s_out;
 *   3. grad_h2 = dy @ W1^T, epilogue: grad_h = r * gamma * grad_h2
 *      - (r^2 * s / d) * h, purely tile-local (no cross-tile exchange).
 *   dout   [M, Dout]  bf16 in     W2    [N1/2, Dout] bf16 in (down projection, [in, out])
 *   y      [M, N1]    bf16 in     (pre-activation [g | u] saved by coda_fwd_swiglu)
 *   W1     [d, N1]    bf16 in     h [M, d] bf16, r [M] fp32, gamma [d] bf16 in
 *   dy_out [M, N1]    bf16 out    s_out [M] fp32 out     dh_out [M, d] bf16 out
 *   workspace: at least coda_bwd_swiglu_dgrad_workspace_bytes(M, d, N1, Dout): the
 *   launch counter's slot, the partial sums of s, and the piece slots of launch 3
 *   as in coda_bwd_dgrad.
 * N1 must be a multiple of 16 and Dout of 8.  Conventions as coda_bwd_dgrad.
 */
CODA_API size_t coda_bwd_swiglu_dgrad_workspace_bytes(int64_t M, int64_t d, int64_t N1,
                                                      int64_t Dout);
CODA_API coda_status_t coda_bwd_swiglu_dgrad(const coda_bf16* dout, const coda_bf16* W2,
                                             const coda_bf16* y, const coda_bf16* W1,
                                             const coda_bf16* h, const float* r,
                                             const coda_bf16* gamma, int64_t M, int64_t d,
                                             int64_t N1, int64_t Dout, coda_bf16* dy_out,
                                             float* s_out, coda_bf16* dh_out, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream);

/*
 * All gradients of the chain h = x @ W0 + z, y = RMSNorm(h, gamma) @ W1 for
 * one training step, as GEMM-epilogue programs ("CODA：将 Transformer 块重写为
 * GEMM-Epilogue 程序以消除显存瓶颈", blog.hotdry.top, section
 * "反向传播的 GEMM-Epilogue 结构": with a GEMM + tile-local-epilogue forward the
 * backward keeps the same structure, the linear maps staying GEMMs).  Five
 * launches on `stream`:
 *   1. grad_h2 = dy @ W1^T; epilogue: the RMSNorm backward of coda_bwd_dgrad,
 *      plus dh_res (the gradient that reaches h through the residual stream,
 *      may be NULL), plus h2 = r * h * gamma (stored to the workspace) and
 *      per-warp column partials of dgamma = sum_m grad_h2 * r * h;
 *   2. dgamma = column sums of the partials (light auxiliary reduction);
 *   3. dW1 = h2^T dy          (K = M tokens; operands read transposed by TMA);
 *   4. dx  = dh @ W0^T;
 *   5. dW0 = x^T dh           (K = M tokens).
 *   dy [M, N1] bf16, x [M, d] bf16, W0 [d, d] bf16, W1 [d, N1] bf16,
 *   h [M, d] bf16 and r [M] fp32 (saved by coda_fwd), gamma [d] bf16,
 *   dh_res [M, d] bf16 or NULL                                   (inputs)
 *   dh_out [M, d] bf16 (= dz), dx_out [M, d] bf16, dgamma_out [d] fp32,
 *   dW0_out [d, d] fp32, dW1_out [d, N1] fp32                    (outputs)
 *   workspace: at least coda_bwd_workspace_bytes(M, d, N1) bytes: the
 *   coda_bwd_dgrad workspace (its launch counter serves every launch of the
 *   call), h2, the dgamma partials and a split-tail region as in coda_fwd,
 *   sized for the largest of launches 3-5.
 * Launch 1 is cooperative, as in coda_bwd_dgrad; launches 3-5 split their tail
 * (and are then cooperative) under the same conditions as coda_fwd's GEMMs.
 * Conventions as coda_fwd.
 */
CODA_API size_t coda_bwd_workspace_bytes(int64_t M, int64_t d, int64_t N1);
CODA_API coda_status_t coda_bwd(const coda_bf16* dy, const coda_bf16* x, const coda_bf16* W0,
                                const coda_bf16* W1, const coda_bf16* h, const float* r,
                                const coda_bf16* gamma, const coda_bf16* dh_res,
                                int64_t M, int64_t d, int64_t N1,
                                coda_bf16* dh_out, coda_bf16* dx_out, float* dgamma_out,
                                float* dW0_out, float* dW1_out, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/* Synchronises `stream`, then reports and clears the library's device-side
 * status word: CODA_OK, CODA_ERR_DEVICE_TIMEOUT if a bounded wait in any
 * kernel of this library ran out since the last call (raw code 0x100 | which
 * wait), or, in the checked build (libcoda_checked.so, compiled with
 * -DCODA_CHECKED: every staged epilogue load and store, gamma load, TMA box
 * start and workspace index checked on the device), CODA_ERR_DEVICE_BOUNDS if a check failed and
 * its access was skipped (raw code 0x200 | which check).  The first failure
 * since the last call is kept.  If `detail` is not NULL it receives the raw
 * code (0 = none).  Returns CODA_ERR_LAUNCH if the stream itself reports a
 * CUDA error. */
CODA_API coda_status_t coda_get_device_status(cudaStream_t stream, uint32_t* detail);

/* Tile shape of the tensor-core GEMMs used by every following call:
 *   0  one CTA per 128 x 256 output tile (tcgen05 .cta_group::1)
 *   1  a pair of CTAs on two SMs per 256 x 256 tile (tcgen05 .cta_group::2);
 *      each SM loads half of B, which halves operand traffic per SM (default).
 * Results are identical up to the fp32 summation order inside the tensor
 * cores.  Returns CODA_ERR_INVALID_ARG for any other value.  Process-wide. */
CODA_API coda_status_t coda_set_mma_mode(int mode);
CODA_API int coda_get_mma_mode(void);

/* Forward variant: 1 folds the row reduction (step 2) into GEMM1's epilogue,
 * which then forms r from the partial sums itself (each tile of column block
 * 0 also stores it), so coda_fwd and coda_fwd_swiglu launch 2 kernels instead
 * of 3.  r is bit-identical either way (same summation order and arithmetic).
 * 0 (the default) keeps the separate light auxiliary reduction.  Returns
 * CODA_ERR_INVALID_ARG for any other value.  Process-wide. */
CODA_API coda_status_t coda_set_fold_rowreduce(int enable);

/* 1 (the default) splits the tail of the CTA-pair GEMMs of coda_fwd,
 * coda_fwd_swiglu and coda_bwd (launches 3-5) along K when their tiles do not
 * fill whole waves (see coda_fwd); 0 hands out whole tiles only.  Returns
 * CODA_ERR_INVALID_ARG for any other value.  Process-wide. */
CODA_API coda_status_t coda_set_split_tail(int enable);

/* 1 or 2 lets the CTA-pair data gradients (coda_bwd_dgrad and launch 1 of
 * coda_bwd) cut each 256-row block into tiles narrower than 256 columns (two
 * widths w and w + step, between 128 and 256, at most 2 * ceil(d / 256) tiles;
 * 1: w and step multiples of 16, 2: multiples of 64) when that spreads the tiles
 * more evenly over the CTA pairs than 256-column tiles do: at d = 4096 and
 * M = 8192, 19 tiles per row block fill 8 whole waves of 76 pairs where 16 tiles
 * leave the seventh wave 74 % full.  The plan is chosen per shape and device on
 * the host; results differ from 256-column tiles only in fp32 summation order.
 * Measured on GB300 both are slower at every Llama shape (more tiles per row
 * block read the grad_y rows more often), so 0, 256-column tiles, is the
 * default.  Returns CODA_ERR_INVALID_ARG for any other value.  Process-wide. */
CODA_API coda_status_t coda_set_col_plan(int enable);

/* 1 makes the CTA-pair data gradients (coda_bwd_dgrad and launch 1 of
 * coda_bwd) load the K blocks of every other wave of tiles in reverse order, so
 * that a wave starts on the slices of W1 that the wave before it read last
 * (each wave streams all of W1, 235 MB at llama7b, through the 129 MB L2).
 * Results differ only in fp32 summation order.  Measured on GB300 with calls
 * of both orders interleaved one by one, it makes no difference (within
 * +-0.5 % at the llama1b, llama7b and llama70b shapes), so 0, K forwards, is
 * the default.  Returns CODA_ERR_INVALID_ARG for any other value.
 * coda_get_serpentine_k returns the current setting.  Process-wide. */
CODA_API coda_status_t coda_set_serpentine_k(int enable);
CODA_API int coda_get_serpentine_k(void);

/* 1 (the default): the CTA-pair data gradients (coda_bwd_dgrad, launch 1 of
 * coda_bwd and launch 3 of coda_bwd_swiglu_dgrad) may cut the tiles of their
 * last row blocks (for the tile-local launch 3: any last tiles) into P pieces
 * along K when whole 256 x 256 tiles would leave the last wave of CTA pairs
 * partly idle.  The pieces are dealt so that the pairs keep walking K in step, every
 * piece but the last of a tile writes an fp32 partial to the workspace, and
 * the pair holding the last piece adds them before the epilogue.  A host-side
 * model, fitted to GB300 measurements (a piece runs about 1.5 times its share
 * of K), picks the row blocks and P, and keeps whole tiles unless the cut
 * saves at least 3 % (llama1b's data gradient: the last 4 row blocks in 2
 * pieces, 8.9 % faster; llama7b and llama70b keep whole tiles).  Launch 3 of
 * coda_bwd_swiglu_dgrad waits on no other tile, so there a piece counts its
 * share of K and a 1 % saving suffices (llama7b: the last 56 tiles in 4
 * pieces, 3.5 % faster).  Results differ from whole tiles only in fp32
 * summation order.  0: whole tiles.
 * Returns CODA_ERR_INVALID_ARG for any other value; coda_get_dgrad_pieces
 * returns the current setting.  Process-wide. */
CODA_API coda_status_t coda_set_dgrad_pieces(int enable);
CODA_API int coda_get_dgrad_pieces(void);

/* The piece plan the CTA-pair data gradient would use for the shape on `npairs`
 * CTA pairs (the device has SMs / 2 of them), whatever coda_set_dgrad_pieces
 * says; host-only, no device needed.  tile_local = 0: the row-statistic launch
 * (coda_bwd_dgrad, launch 1 of coda_bwd); 1: launch 3 of coda_bwd_swiglu_dgrad.
 * Writes plan[4] = {tiles handed out whole (the cut tiles follow them in the
 * launch's tile order), pieces per cut tile, first of the pairs that hold one
 * whole tile fewer and take levelling pieces, levelling pieces per such pair}.
 * Returns 1 when a plan is taken, 0 when the launch keeps whole tiles (plan
 * zeroed) and -1 for invalid arguments. */
CODA_API int coda_dgrad_piece_plan(int64_t M, int64_t d, int64_t N1, int npairs, int tile_local,
                                   int32_t* plan);

/* Upper bound, in nanoseconds, of every device-side wait launched after this
 * call (default 1e9 = 1 s).  A wait that runs out records
 * CODA_ERR_DEVICE_TIMEOUT and lets its kernel finish without hanging. */
CODA_API void coda_set_wait_timeout_ns(uint64_t ns);

/* Human-readable name of a status code (static storage). */
CODA_API const char* coda_status_string(coda_status_t status);

/*
 * Measurement-only unfused reference sequence, built from the same GEMM
 * mainloop: GEMM0 with a plain epilogue (h = x @ W0 + z), a standalone
 * RMSNorm kernel that writes hn = r * h * gamma ([M, d] bf16) and r, then GEMM1
 * with a plain epilogue (y = hn @ W1).  It exists to show, with hardware
 * counters, the [M, d] round trip and the extra kernel that coda_fwd removes.
 * Same arguments and conventions as coda_fwd; workspace of at least
 * coda_fwd_unfused_workspace_bytes(M, d, N1) bytes.
 */
CODA_API size_t coda_fwd_unfused_workspace_bytes(int64_t M, int64_t d, int64_t N1);
CODA_API coda_status_t coda_fwd_unfused(const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                               const coda_bf16* gamma, const coda_bf16* W1, float eps,
                               int64_t M, int64_t d, int64_t N1,
                               coda_bf16* h_out, float* r_out, coda_bf16* y_out,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Measurement hook.  While `events` is non-NULL, every kernel launch k
 * (0-based, counted within one call of any entry point above except
 * coda_bwd_dgrad_noalloc) is followed by cudaEventRecord(events[k], stream)
 * for k < n, so that a caller that records its own event before the call can
 * time each launch on the launching stream.  coda_fwd, coda_fwd_swiglu,
 * coda_fwd_unfused, coda_fwd_fp8 and coda_bwd_swiglu_dgrad launch 3 kernels
 * (2 for the forwards with the folded row reduction), coda_bwd 5,
 * coda_bwd_dgrad 1.  The events are caller-owned; pass NULL to stop.
 * Process-wide setting, not thread-safe; no effect on results.
 */
CODA_API void coda_set_launch_events(cudaEvent_t* events, int n);

/*
 * Self-test of the device-side watchdog: launches one block whose waits (on
 * an mbarrier that nobody arrives on, and on a global flag that nobody sets)
 * are bounded by `timeout_ns`.  Both waits run out by construction, so a
 * following coda_get_device_status() must report CODA_ERR_DEVICE_TIMEOUT.
 * No other work is affected and the CUDA context stays usable.
 */
CODA_API coda_status_t coda_watchdog_selftest(uint64_t timeout_ns, cudaStream_t stream);

/*
 * coda_bwd_dgrad without a workspace, for callers that cannot allocate.
 *
 * The method's pages have no counterpart to this entry point; it exists for
 * callers that must not allocate device memory when they run the backward:
 * code running inside an allocator or memory-pool callback, runtimes that
 * forbid allocation mid-step (an allocation can synchronise the device or
 * fragment a pool sized up front), and embedders whose device memory is fully
 * reserved in advance.  It computes what coda_bwd_dgrad computes, with the same
 * epilogue program on single-CTA tiles (the coda_set_mma_mode(0) kernel; the
 * result equals the default CTA-pair kernel's bit for bit in the tests), but
 * takes only inputs and outputs: the per-tile partial row
 * statistics and the completion flags live in a fixed array inside the
 * library (2 * CODA_NOALLOC_MAX_PARTIALS floats + CODA_NOALLOC_MAX_TILES 64-bit
 * flags, about 4.1 MiB), which every GPU that loads the library holds until
 * the process exits.  It allocates nothing and calls no allocating routine.
 *
 *  - Size limit: ceil(d/256) * M <= CODA_NOALLOC_MAX_PARTIALS and
 *    ceil(M/128) * ceil(d/256) <= CODA_NOALLOC_MAX_TILES, otherwise it returns
 *    CODA_ERR_UNSUPPORTED_SHAPE without launching (e.g. M = 32768 rows at
 *    d = 4096, or 16384 rows at d = 8192, fit).
 *  - The library's device code, this array with it, is loaded on a device by
 *    the first call of any entry point on that device (CUDA loads modules
 *    lazily), and that first call also looks up the array's device address
 *    (cudaGetSymbolAddress) with the device current.  Loading the module
 *    reserves device memory for the array and the kernels, so the guarantee
 *    that a call allocates nothing holds from the second library call on a
 *    device on: make one call of any entry point that launches work (this one
 *    included) on each device outside the region where allocation is
 *    forbidden, and before any stream capture.
 *  - Every call uses the same array.  Nothing in it needs clearing (each
 *    launch tags its flags with a fresh token from a launch counter kept in
 *    the array, mixed with the call's salt), but calls whose kernels
 *    overlap on the GPU, on different streams or from different host threads,
 *    race on it and give wrong results: order them (one stream, or events).
 *  - Otherwise the arguments, checks and errors are those of coda_bwd_dgrad.
 */
#define CODA_NOALLOC_MAX_PARTIALS 524288
#define CODA_NOALLOC_MAX_TILES 16384
CODA_API coda_status_t coda_bwd_dgrad_noalloc(const coda_bf16* dy, const coda_bf16* W1,
                                              const coda_bf16* h, const float* r,
                                              const coda_bf16* gamma,
                                              int64_t M, int64_t d, int64_t N1,
                                              coda_bf16* dh_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CODA_H_ */
