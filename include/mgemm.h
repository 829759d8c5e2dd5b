/*
 * mgemm.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts grouped GEMM.
 *
 * The hot path computes gmm(x, w, group_sizes): M token rows of x, stored
 * contiguously by expert (group e owns rows [offsets[e], offsets[e+1])), are
 * multiplied by per-expert weights w[E, K, N]; the group sizes stay in device
 * memory and no call ever waits on the host.  Sources, cited per entry point
 * below:
 *   [GRB]  "Support GPU-resident batch sizes" (tgale96/grouped_gemm PR #21):
 *          description and benchmark script; review of
 *          csrc/fill_arguments.cuh and csrc/grouped_gemm.cu.
 *   [SPM]  "F8I4 Grouped Gemm Optimization for Sparse M" (pytorch/FBGEMM PR
 *          #3854), Summary.
 *   [FP8]  "[moe training] Optimize FP8 MoE backward pass: fused colwise
 *          kernel + AMD tuning" (pytorch/ao commit 34322b5): commit message and
 *          bench_colwise_block_configs.py (_colwise_kernel, run_experiment).
 *   [CMM]  pytorch-labs/applied-ai issue 24, the column-major fused MoE script
 *          (built on vLLM's fused_moe.py): moe_align_block_size (docstring and
 *          worked example), fused_moe_kernel, fused_moe.
 *
 * Conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer owned by the caller; the
 *     library allocates nothing, keeps no reference after the call returns and
 *     never synchronizes: work is enqueued on `stream` (0 = legacy default).
 *   - Return value: MGEMM_OK (0) when the work was enqueued, or a negative
 *     MGEMM_E* code when a host-side check failed; then nothing is launched.
 *   - Errors found on the device (bad group sizes, a wait that timed out) are
 *     written to the int32 `status` word at the start of the args block (see
 *     below).  Every kernel that takes an args block reads `status` first and
 *     writes nothing when it is non-zero.  The caller reads the word whenever
 *     it chooses to synchronize.
 *   - Matrices are dense and row-major unless stated; "[R, C]" means R rows of
 *     C elements with row stride C.  bf16 is IEEE bfloat16 (2 bytes), fp8 is
 *     OCP/NVIDIA e4m3fn (1 byte, max 448, no infinities), scales are float32.
 *   - Base pointers must be 16-byte aligned and row strides multiples of 16
 *     bytes (the tensor-memory-accelerator rule): K and N multiples of 8 for
 *     bf16 operands, of 16 for fp8 operands.  1 <= E <= MGEMM_MAX_EXPERTS.
 *     M < 2^31.  Violations return MGEMM_EALIGN / MGEMM_EINVAL.
 */
#ifndef MGEMM_H_
#define MGEMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st *mgemm_stream_t;

/* Host-side return codes. */
#define MGEMM_OK 0
#define MGEMM_EINVAL (-1)   /* null pointer, bad size, bad dtype/flag */
#define MGEMM_EALIGN (-2)   /* pointer or stride breaks the 16-byte rule */
#define MGEMM_ETOOMANY (-3) /* E > MGEMM_MAX_EXPERTS */
#define MGEMM_ECUDA (-4)    /* a CUDA runtime/driver call failed (launch, tensor map) */
#define MGEMM_ENOTSUP (-5)  /* combination not provided (e.g. fp8 with w stored [E,K,N] in mgemm_fwd) */

/* Device-side status codes, written to args->status. */
#define MGEMM_STATUS_OK 0
#define MGEMM_STATUS_NEGATIVE_SIZE 1 /* some group_sizes[e] < 0 */
#define MGEMM_STATUS_SUM_MISMATCH 2  /* sum of group_sizes != M */
#define MGEMM_STATUS_TIMEOUT 4       /* a pipeline wait in a GEMM gave up (about 1 s) */

/* Operand types for the GEMM entry points. */
#define MGEMM_BF16 0
#define MGEMM_FP8_E4M3 1

/* One thread per expert in the single-CTA fill kernel [GRB description]. */
#define MGEMM_MAX_EXPERTS 1024
/* Rows per output tile; the fill kernel's tile prefix counts tiles of this height. */
#define MGEMM_TILE_M 128
/* Row padding of each group in the column-major FP8 layout (see mgemm_colwise_ld). */
#define MGEMM_COL_PAD 128

/*
 * Args block: a device buffer of mgemm_args_bytes(E) bytes, 16-byte aligned,
 * written by mgemm_fill_args and read by every other entry point that takes
 * `args`.  Byte layout (E = number of experts):
 *   [0]   int32  status        MGEMM_STATUS_*
 *   [4]   int32  n_active      number of non-empty groups (<= min(M, E))
 *   [8]   int32  E
 *   [12]  int32  work counter: mgemm_fill_args writes 0; mgemm_quant_colwise_grouped
 *                hands out its work items from it and leaves it at 0 again when it
 *                completes (calls that share an args block must not overlap on the GPU)
 *   [16]  int64  M
 *   [24]  int64  offsets[E+1]  exclusive prefix sum of group_sizes
 *   [A]   int32  active[E]     ids of the non-empty groups, ascending (first n_active valid)
 *   [T]   int32  mtile_start[E+1]  prefix over active groups of ceil(m_e / MGEMM_TILE_M)
 *   [W]   int32  wgrad_order[E]    all experts by m_e descending, ties by ascending id
 *   [P]   int64  poffsets[E+1] exclusive prefix sum of group_sizes each rounded up to
 *                MGEMM_COL_PAD: where group e starts in the padded column-major
 *                FP8 layout of mgemm_quant_colwise_grouped / mgemm_wgrad
 *   [Q]   int32  ptile_start[E+1]  prefix over active groups of ceil(m_e / (2 MGEMM_TILE_M))
 *                (the row-tile pairs of the FP8 GEMMs that run on CTA pairs)
 * with A = 24 + 8(E+1), T = A + 4E, W = T + 4(E+1), P = W + 4E rounded up to a
 * multiple of 8, Q = P + 8(E+1); mgemm_args_layout returns A, T and W.
 */
size_t mgemm_args_bytes(int E);
int mgemm_args_layout(int E, size_t *off_offsets, size_t *off_active, size_t *off_mtile_start,
                      size_t *off_wgrad_order);

/*
 * mgemm_fill_args -- turn device-resident group sizes into the args block.
 * [GRB description]: a single-threadblock kernel converts the batch sizes that
 * live on the GPU into GEMM arguments, removing the GPU->CPU->GPU roundtrip;
 * [GRB review, fill_arguments.cuh]: the block scan, and the sort of problems
 * by k descending when k is dynamic (wgrad_order here); [SPM Summary]: only
 * the min(total_M, groups) non-empty groups are scheduled (active, mtile_start).
 *   group_sizes  int64[E], device; group_sizes[e] rows belong to expert e
 *   E            number of experts, 1..MGEMM_MAX_EXPERTS
 *   M            total rows the caller expects (checked on the device), or -1:
 *                the rows are the sum of the sizes, which only the device
 *                knows (sizes written by another kernel, e.g. the padded
 *                group sizes of mgemm_moe_align); status 2 if it reaches 2^31
 *   args         device buffer of mgemm_args_bytes(E) bytes (output)
 * One launch of one CTA.  Invalid sizes set status 1 or 2 (the other fields
 * are then unspecified).
 */
int mgemm_fill_args(const int64_t *group_sizes, int E, int64_t M, void *args, mgemm_stream_t stream);

/*
 * mgemm_quant_rowwise -- fused per-row absmax scale and saturating e4m3 cast.
 * [FP8 commit message]: replaces tensor_to_scale(A, axiswise_dim=-1),
 * A_scaled = A.to(float32) * A_scales, A_fp8 = to_fp8_saturated(A_scaled) by
 * one launch.  Per row r: amax = max_c |in[r, c]|;
 * s = 2^floor(log2(fp32(448 / max(amax, 1e-12)))) (the scale rule of
 * _colwise_kernel, applied per row); out[r, c] = e4m3_rne_sat(in[r, c] * s).
 *   in      bf16 [R, C] with row stride ld_in elements (ld_in >= C, ld_in % 8 == 0)
 *   out     fp8  [R, C] with row stride ld_out bytes (ld_out >= C, ld_out % 16 == 0)
 *   scales  float32 [R]
 * C % 8 == 0.  R == 0 or C == 0 launches nothing.
 */
int mgemm_quant_rowwise(const void *in, int64_t R, int64_t C, int64_t ld_in, uint8_t *out, int64_t ld_out,
                        float *scales, mgemm_stream_t stream);

/*
 * mgemm_quant_mx -- MXFP8 block quantize: e4m3 codes with one e8m0 scale per
 * 32 consecutive elements of a row.  [FP8 commit message]: the MXFP8 grouped
 * MM path beside the FP8 one, with its token groups padded to 32; the page
 * prints no arithmetic.  Reading: per block b of row r (columns 32b..32b+31),
 * amax = max |in|; s = the power-of-two rule of mgemm_quant_rowwise applied to
 * that amax; out = e4m3_rne_sat(in * s); sf[r, b] = 127 - log2(s) (the e8m0
 * byte of the decode factor 1/s, always in 79..254).
 *   in   bf16 [R, C] with row stride ld_in elements (ld_in >= C, ld_in % 8 == 0)
 *   out  e4m3 [R, C] with row stride ld_out bytes (ld_out >= C, ld_out % 16 == 0)
 *   sf   e8m0 [R, ld_sf] bytes, ld_sf >= C / 32, ld_sf % 16 == 0 (bytes past
 *        C / 32 in each row are not written)
 * C % 32 == 0.  R == 0 or C == 0 launches nothing.  Errors: -1 (sizes), -2
 * (alignment).
 */
int mgemm_quant_mx(const void *in, int64_t R, int64_t C, int64_t ld_in, uint8_t *out, int64_t ld_out, uint8_t *sf,
                   int64_t ld_sf, mgemm_stream_t stream);

/*
 * mgemm_colwise_ld -- the smallest leading dimension (bytes per column) of the
 * padded column-major FP8 layout for M rows in E groups: M plus the padding of
 * up to min(M, E) non-empty groups, rounded up to MGEMM_COL_PAD.  Known on the
 * host without the group sizes.  Returns -1 for M < 0 or E outside 1..MGEMM_MAX_EXPERTS.
 * (An implementation choice, not in [FP8]: it sizes the layout below.)
 */
int64_t mgemm_colwise_ld(int64_t M, int E);

/*
 * mgemm_quant_colwise_grouped -- per-group, per-column scale and e4m3 cast,
 * column-major output; optionally two tensors in one launch (dual form).
 * [FP8 _colwise_kernel]: for group g (rows offsets[g]..offsets[g+1]) and
 * column c, amax over the group's rows, the same power-of-two scale rule, the
 * scale stored at index c + C * g, the cast clamp(x * s) -> e4m3;
 * [FP8 run_experiment]: the output is column-major;
 * [FP8 commit message]: the dual kernel quantizes grad_output and A together.
 *   args        args block from mgemm_fill_args (group offsets, status)
 *   E, M        experts and rows (must match the args block)
 *   in1         bf16 [M, C1] row-major
 *   out1        fp8, padded column-major: column c of group g occupies bytes
 *               out1[c * ld + poffsets[g] ...], m_g codes followed by zeros up
 *               to the next multiple of MGEMM_COL_PAD (C1 * ld bytes; bytes past
 *               poffsets[E] in a column are not written)
 *   sc1         float32 [E * C1], sc1[c + C1 * g]
 *   in2/out2/sc2/C2  the second tensor; in2 == NULL selects the single form
 *   ld          bytes per output column: >= mgemm_colwise_ld(M, E), % 16 == 0
 * C1, C2 % 8 == 0; out1, out2 16-byte aligned.  Empty groups get scale 2^48
 * (amax 0) and no data.  The padding keeps every group's codes aligned and
 * lets mgemm_wgrad contract whole 128-row blocks without masking (an
 * implementation choice; [FP8 run_experiment]'s layout is unpadded, strides (1, M)).
 */
int mgemm_quant_colwise_grouped(const void *args, int E, int64_t M, const void *in1, int64_t C1,
                                uint8_t *out1, float *sc1, const void *in2, int64_t C2, uint8_t *out2,
                                float *sc2, int64_t ld, mgemm_stream_t stream);

/*
 * mgemm_fwd -- out[r, :] = x[r, :] . w[e(r)] for every row r of every non-empty group.
 * [GRB benchmark script]: gmm(x, w, batch_sizes) with x[M, K], w[E, K, N];
 * [GRB review, grouped_gemm.cu]: the trans_b variant (w stored [E, N, K]);
 * [SPM Summary]: only non-empty groups are visited; [FP8 commit message]:
 * FP8 operands are A * scale, so the product is divided by the scales.
 *   dtype == MGEMM_BF16:
 *     x bf16 [M, K]; w bf16 [E, K, N] (trans_b = 0) or [E, N, K] (trans_b = 1);
 *     sx, sw ignored (may be NULL); out bf16 [M, N] (fp32 accumulation, RNE).
 *   dtype == MGEMM_FP8_E4M3 (trans_b must be 1):
 *     x fp8 [M, K] + sx float32 [M]; w fp8 [E, N, K] + sw float32 [E * N];
 *     out[r, n] = bf16( sum_k x[r,k] w[e,n,k] / (sx[r] * sw[e*N + n]) ).
 * Rows of empty groups do not exist; no other memory is written.
 */
int mgemm_fwd(const void *args, int dtype, int trans_b, const void *x, const float *sx, const void *w,
              const float *sw, void *out, int64_t M, int K, int N, int E, mgemm_stream_t stream);

/*
 * mgemm_fwd_fp8_strided -- mgemm_fwd (dtype MGEMM_FP8_E4M3, w [E, N, K]) with
 * the e4m3 weights addressed through strides: w[e, n, k] at byte
 * e * ld_we + n * ld_wn + k.  With the weights' master copy stored [E, K, N]
 * (the layout of the GRIN benchmark script), the forward operand (one scale
 * per (e, n) over K) is mgemm_quant_colwise_grouped of w viewed [E * K, N]
 * with E groups of K rows ([FP8 commit message]: the per-group colwise
 * kernel): its padded column-major codes hold w[e, n, k] at
 * n * ld + e * ceil(K / 128) * 128 + k, i.e. ld_wn = ld (as passed to it),
 * ld_we = K rounded up to 128, and its scales [E * N] are this call's sw.  No
 * transposed copy of the weights is needed.
 *   ld_wn  >= K, % 16 == 0;  ld_we >= K (any value when E == 1), % 16 == 0
 *   the other arguments: as mgemm_fwd with dtype MGEMM_FP8_E4M3, trans_b = 1.
 * Errors as mgemm_fwd.
 */
int mgemm_fwd_fp8_strided(const void *args, const void *x, const float *sx, const void *w, int64_t ld_wn,
                          int64_t ld_we, const float *sw, void *out, int64_t M, int K, int N, int E,
                          mgemm_stream_t stream);

/*
 * mgemm_dgrad -- grad_x[r, :] = grad_out[r, :] . w[e(r)]^T (the backward pass
 * of gmm w.r.t. x).  [GRB benchmark script]: out.sum().backward();
 * [GRB review, grouped_gemm.cu]: the trans_b template; [FP8 commit message]:
 * grad_output is quantized rowwise for grad_A.
 *   grad_out  bf16 [M, N] (or fp8 [M, N] + sgo float32 [M])
 *   w         bf16 [E, K, N] (or fp8 [E, K, N] + sw float32 [E * K], one scale per (e, k))
 *   grad_x    bf16 [M, K]
 */
int mgemm_dgrad(const void *args, int dtype, const void *grad_out, const float *sgo, const void *w,
                const float *sw, void *grad_x, int64_t M, int K, int N, int E, mgemm_stream_t stream);

/*
 * mgemm_fwd_mx -- the MXFP8 grouped GEMM: out[r, n] = sum_k xv[r, k] wv[e(r), n, k]
 * where xv, wv are the decoded block-scaled values (e4m3 value times
 * 2^(sf - 127) of its 32-element block; see mgemm_quant_mx).  [FP8 commit
 * message]: the MXFP8 grouped MM path; the block scales are applied by the
 * tensor cores (block-scaled MMA, one e8m0 scale per 32 contraction elements
 * of each row of either operand), accumulation in fp32, bf16 output (RNE).
 * The same call computes the MXFP8 dgrad: pass grad_out as x (contraction N)
 * and w stored [E, K, N] quantized along N as w.
 *   x    e4m3 [M, K] (row stride K bytes); sx e8m0 [M, ld_sf]
 *   w    e4m3 [E, N, K]; sw e8m0 [E * N, ld_sf]
 *   ld_sf  bytes per scale row, >= K / 32, % 16 == 0 (as written by mgemm_quant_mx)
 *   out  bf16 [M, N]
 * K % 128 == 0, N % 8 == 0.  Groups of any size (the blocks run along K).
 * Errors: -1 (sizes or NULL), -2 (alignment), -3 (E), -4 (CUDA).
 */
int mgemm_fwd_mx(const void *args, const uint8_t *x, const uint8_t *sx, const uint8_t *w, const uint8_t *sw,
                 int64_t ld_sf, void *out, int64_t M, int K, int N, int E, mgemm_stream_t stream);

/*
 * mgemm_quant_colwise_mx -- per-group colwise MX blocks, the MXFP8 wgrad
 * operands (one or two tensors per launch).  Reading of [FP8]'s MXFP8 path
 * (groups padded to 32 rows): in group g and column c, blocks of 32
 * consecutive rows counted from the group's first row (a group's last block
 * may be short; its missing rows count as zeros); each block's scale and codes
 * follow mgemm_quant_mx.
 *   in1   bf16 [M, C1] row-major (C1 % 8 == 0); optionally in2 [M, C2] (dual)
 *   out1  e4m3 [C1, ld]: the padded column-major layout of
 *         mgemm_quant_colwise_grouped (group g's codes at column offset
 *         poffsets[g], zeros after them up to a multiple of MGEMM_COL_PAD)
 *   sf1   e8m0 [ld / 128][C1][4]: for padded row block j (rows 128 j .. 128 j +
 *         127) and column c, the 4 bytes of its four 32-row blocks
 *         ((ld / 128) * C1 * 4 bytes, 16-byte aligned)
 *   ld    bytes per column: >= mgemm_colwise_ld(M, E), % 128 == 0
 * Only bytes inside the padded total (poffsets[E]) are written.
 * Errors: -1 (sizes, NULL), -2 (alignment), -3 (E).
 */
int mgemm_quant_colwise_mx(const void *args, int E, int64_t M, const void *in1, int64_t C1, uint8_t *out1,
                           uint8_t *sf1, const void *in2, int64_t C2, uint8_t *out2, uint8_t *sf2, int64_t ld,
                           mgemm_stream_t stream);

/*
 * mgemm_wgrad_mx -- the MXFP8 wgrad: grad_w[e] = sum over the rows r of group e
 * of xv[r, :]^T gov[r, :], with the decoded block-scaled values of
 * mgemm_quant_colwise_mx (blocks of 32 rows of a group); zero for an empty
 * group.  Block-scaled tensor-core MMAs, fp32 accumulation, bf16 output.
 *   x, sx    x's codes [K, ld] and scale rows [ld / 128][K][4] (mgemm_quant_colwise_mx)
 *   grad_out, sgo   likewise [N, ld] and [ld / 128][N][4]
 *   grad_w   bf16 [E, K, N]; every element is written
 *   ld       as passed to mgemm_quant_colwise_mx
 * K % 16 == 0, N % 16 == 0.  Errors: -1, -2, -3, -4 as mgemm_wgrad.
 */
int mgemm_wgrad_mx(const void *args, const uint8_t *x, const uint8_t *sx, const uint8_t *grad_out,
                   const uint8_t *sgo, void *grad_w, int64_t M, int K, int N, int E, int64_t ld,
                   mgemm_stream_t stream);

/*
 * mgemm_wgrad -- grad_w[e] = x_e^T . grad_out_e, contracting over the m_e rows
 * of group e ("dynamic k"); grad_w[e] = 0 when m_e = 0.
 * [GRB review, fill_arguments.cuh]: problems sorted by k descending;
 * [GRB review, ZeroOutK0Outputs]: k = 0 problems produce zeros;
 * [FP8 commit message]: grad_B uses per-group colwise scales of grad_output and A.
 *   dtype == MGEMM_BF16: x bf16 [M, K], grad_out bf16 [M, N] (row-major).
 *   dtype == MGEMM_FP8_E4M3: x fp8 [K, ld] and grad_out fp8 [N, ld] in the
 *     padded column-major layout of mgemm_quant_colwise_grouped (rows of group
 *     e at poffsets[e], zero padding after them), sx float32 [E * K] and sgo
 *     float32 [E * N] its scales; ld as passed to it.
 *   ld        FP8: bytes per column of x and grad_out (% 16 == 0,
 *             >= mgemm_colwise_ld(M, E)); ignored for MGEMM_BF16.
 *   grad_w    bf16 [E, K, N]; every element is written.
 */
int mgemm_wgrad(const void *args, int dtype, const void *x, const float *sx, const void *grad_out,
                const float *sgo, void *grad_w, int64_t M, int K, int N, int E, int64_t ld, mgemm_stream_t stream);

/*
 * mgemm_dgrad_wgrad -- the bf16 backward of the grouped GEMM, both gradients:
 * grad_x exactly as mgemm_dgrad(MGEMM_BF16, grad_out, w [E, K, N]) and grad_w
 * exactly as mgemm_wgrad(MGEMM_BF16, x, grad_out), bit for bit ("Support
 * GPU-resident batch sizes", benchmark script: the backward of gmm after
 * out.sum()).  Where the groups are small enough that dgrad streams the
 * weights from HBM while wgrad is bound by its grad_w stores, both run in one
 * launch on disjoint sets of CTAs (a host-side model of the two sizes picks
 * the split) and overlap; otherwise the two calls run one after the other on
 * the stream.  Same args block as both; no other device memory.
 *   grad_out bf16 [M, N]; w bf16 [E, K, N]; x bf16 [M, K] (row-major)
 *   grad_x   bf16 [M, K]; grad_w bf16 [E, K, N] (every element written)
 * With M == 0 only grad_w is written (zeros) and grad_out, x, grad_x may be
 * NULL.  Errors as for the two calls (K % 8 == 0, N % 8 == 0, 16-byte aligned
 * pointers).
 */
int mgemm_dgrad_wgrad(const void *args, const void *grad_out, const void *w, const void *x, void *grad_x,
                      void *grad_w, int64_t M, int K, int N, int E, mgemm_stream_t stream);

/* The number of CTAs mgemm_dgrad_wgrad gives to dgrad in its one-launch form
 * for these sizes (the rest of the SMs run wgrad), or 0 when it makes the two
 * calls in turn; negative MGEMM_E* for invalid sizes.  Host-side (reads the
 * current device's SM count once). */
int mgemm_dgrad_wgrad_split(int64_t M, int K, int N, int E);

/*
 * mgemm_fill_args_quant_rowwise -- mgemm_fill_args and mgemm_quant_rowwise of
 * the token rows in one launch (the two independent steps before an FP8
 * forward: "Support GPU-resident batch sizes", the argument fill; "[moe
 * training] Optimize FP8 MoE backward pass" commit message, the fused rowwise
 * scale + cast).  The args block is exactly mgemm_fill_args(group_sizes, E, M,
 * args); xq and sx exactly mgemm_quant_rowwise(x [M, K]).  One CTA fills the
 * args block while the others cast rows, so at sparse M the pair costs about
 * one launch instead of two.
 *   group_sizes int64[E], device; args as for mgemm_fill_args (M >= 0 here)
 *   x     bf16 [M, K], row stride ld_x elements; xq e4m3 [M, K], row stride ld_q
 *         bytes; sx fp32 [M]
 * K % 8 == 0, ld_x % 8 == 0, ld_q % 8 == 0.  Errors as for the two calls.
 */
int mgemm_fill_args_quant_rowwise(const int64_t *group_sizes, int E, int64_t M, void *args, const void *x, int64_t K,
                                  int64_t ld_x, uint8_t *xq, int64_t ld_q, float *sx, mgemm_stream_t stream);

/*
 * mgemm_fwd_fp8_sparse -- the FP8 forward for few token rows in one launch:
 * mgemm_fill_args + mgemm_quant_rowwise of x + mgemm_fwd (MGEMM_FP8_E4M3,
 * w [E, N, K]) ("F8I4 Grouped Gemm Optimization for Sparse M", Summary:
 * work only for the min(total_M, groups) non-empty groups; "[moe training]
 * Optimize FP8 MoE backward pass" commit message: the fused rowwise scale +
 * cast).  Every CTA scans the group sizes itself, casts the token rows it
 * needs (the rowwise rule: power-of-two scale from the row's magnitude
 * maximum, saturating e4m3) into shared memory and streams its share of the
 * touched experts' weights.  When the tiles of 128 output columns cover at
 * most half of the SMs (one token), pairs of CTAs split each tile's
 * contraction in two halves and add the second half's fp32 partial sums to
 * the first's; otherwise every output equals mgemm_fwd's bit for bit.
 *   group_sizes int64[E], device, summing to M
 *   x        bf16 [M, K] token rows sorted by expert, row stride ld_x elements
 *   w, sw    e4m3 [E, N, K] and fp32 [E * N] (as for mgemm_fwd)
 *   out      bf16 [M, N]; only the M rows are written
 *   status   int32, device, holding 0 or a negative value on entry (zeroed
 *            once, it stays 0 while calls succeed): the call raises it to
 *            MGEMM_STATUS_NEGATIVE_SIZE or MGEMM_STATUS_SUM_MISMATCH (then
 *            nothing else is written) or MGEMM_STATUS_TIMEOUT, else to 0; a
 *            caller that reads a nonzero status resets it before the next call
 * 1 <= M <= 16, E <= 1024, K % 128 == 0, N % 8 == 0, ld_x % 8 == 0, and the
 * token rows must fit on chip: ceil(M / 8) * 8 * K <= 150 KiB (else -1; use
 * the three calls).  Errors: -1 (sizes or NULL), -2 (alignment), -3 (E),
 * -4 (CUDA).
 */
int mgemm_fwd_fp8_sparse(const int64_t *group_sizes, int E, const void *x, int64_t ld_x, const void *w,
                         const float *sw, void *out, int *status, int64_t M, int K, int N, mgemm_stream_t stream);



/*
 * mgemm_quant_int4 -- the INT4 weights of the FP8 x INT4 grouped GEMM.
 * "F8I4 Grouped Gemm Optimization for Sparse M" (FBGEMM PR #3854), title and
 * Summary, names FP8 activations times INT4 weights and gives no format; this
 * library's reading: per row (e, n) of w [E, N, K] and block of 32 consecutive
 * k, s = 2^floor(log2(fp32(7 / max(amax, 1e-12)))) (the FP8 power-of-two rule
 * at the INT4 range), q = clamp(round_half_even(w * s), -8, 7).
 *   w       bf16 [E, N, K], row stride ld_in elements (>= K, % 8 == 0), device
 *   packed  uint8 [E, N, K / 2]: two's-complement nibbles, element 2i in the low
 *           nibble of byte i of its row (rows of K / 2 bytes, no padding)
 *   sf      uint8, E * (K / 128) * N * 4 bytes: the e8m0 byte 127 - log2(s) of
 *           each block (the decode factor 1 / s), contraction-block major:
 *           block j of row (e, n) at ((e * (K / 128) + j / 4) * N + n) * 4 + j % 4
 * K % 128 == 0.  Codes and bytes are unique (bit-exact against the oracle).
 * Errors: -1 (sizes or NULL), -2 (alignment), -4 (CUDA).
 */
int mgemm_quant_int4(const void *w, int E, int N, int K, int64_t ld_in, uint8_t *packed, uint8_t *sf,
                     mgemm_stream_t stream);

/*
 * mgemm_fwd_f8i4 -- the FP8 x INT4 grouped forward GEMM ("F8I4 Grouped Gemm
 * Optimization for Sparse M", FBGEMM PR #3854, Summary: tiles only for the
 * min(total_M, groups) non-empty groups):
 *   out[r, n] = sum_k (e4m3(x[r, k]) / sx[r]) * q[e(r), n, k] * 2^(b[e, n, k / 32] - 127)
 * in fp32 on the tensor cores (block-scaled MMA: x's row scale and the weight
 * blocks' bytes are both applied inside it), rounded once to bf16 (RNE).
 *   args     filled by mgemm_fill_args for these E group sizes and M
 *   x, sx    e4m3 [M, K] and fp32 [M] row scales (mgemm_quant_rowwise)
 *   w_packed, w_scales  as written by mgemm_quant_int4 for w [E, N, K]
 *   out      bf16 [M, N]; rows of empty groups do not exist, nothing else is written
 * K % 128 == 0, N % 8 == 0 (else -2).  Errors: -1 (sizes or NULL), -2
 * (alignment), -3 (E), -4 (CUDA); device-side errors in the args status word.
 */
int mgemm_fwd_f8i4(const void *args, const uint8_t *x, const float *sx, const uint8_t *w_packed,
                   const uint8_t *w_scales, void *out, int64_t M, int K, int N, int E, mgemm_stream_t stream);

/*
 * mgemm_fwd_noalloc -- mgemm_fwd for callers that cannot allocate device memory.
 * The source pages have no counterpart to this call; it exists for callers
 * that may not call cudaMalloc (or any allocator) at the point where they run
 * the forward pass -- for example code inside another framework's launch
 * callback that has no allocator of its own, loops where an allocation could
 * synchronize the device, or runtimes that only provide a fixed workspace
 * chosen in advance.  Instead of a caller-provided args block it uses one held
 * in a static device array of this library, sized for MGEMM_NOALLOC_MAX_EXPERTS
 * experts (about 33 KB, kept on every GPU that loads the library until exit).
 *   group_sizes  int64[E], device (as for mgemm_fill_args)
 *   the other arguments are those of mgemm_fwd.
 * Makes every host check of mgemm_fill_args and mgemm_fwd first (same codes;
 * a rejected call launches nothing and leaves the array untouched; M must be
 * >= 0, and M == 0 returns MGEMM_OK at once), then runs mgemm_fill_args into
 * the static array and mgemm_fwd.  Allocates nothing.
 * E > MGEMM_NOALLOC_MAX_EXPERTS returns MGEMM_ETOOMANY.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.  The
 * address is kept for the life of the process: do not use this call on a
 * device after cudaDeviceReset.
 * All calls share the array: calls whose work overlaps on the GPU race on it.
 * Device-side errors go to the status word of the static args block, which the
 * caller cannot read; check the group sizes beforehand when that matters.
 */
#define MGEMM_NOALLOC_MAX_EXPERTS 1024
int mgemm_fwd_noalloc(const int64_t *group_sizes, int E, int dtype, int trans_b, const void *x, const float *sx,
                      const void *w, const float *sw, void *out, int64_t M, int K, int N, mgemm_stream_t stream);

/*
 * mgemm_moe_align -- moe_align_block_size on the device [CMM]: the flat
 * (token, slot) entries of topk_ids are grouped by expert, each expert's list
 * padded up to a multiple of block_size, so that every block of the sorted list
 * belongs to one expert.
 *   topk_ids      int32 [numel]: expert of flat entry i (token i / top_k when
 *                 topk_ids is [T, top_k] row-major).  Entries outside [0, E)
 *                 are not placed.
 *   sorted_ids    int32 [numel + E * (block_size - 1)]: expert by expert in
 *                 ascending id, the expert's flat indices in ascending order,
 *                 then the pad id numel up to the expert's padded count; every
 *                 position from num_post_padded to the end also holds numel.
 *   expert_ids    int32 [(numel + E * (block_size - 1)) / block_size]: the
 *                 expert of each block of block_size positions; -1 past the
 *                 last block.
 *   num_post_padded  int32 [1]: the padded total (a multiple of block_size).
 *   group_sizes   int64 [E] or NULL: each expert's padded count (the group
 *                 sizes for mgemm_fill_args over the sorted, padded rows).
 *   workspace     mgemm_moe_align_workspace_bytes(numel, E) bytes, 16-byte
 *                 aligned, scratch for the duration of the call's kernels.
 * Limits: 1 <= E <= MGEMM_MAX_EXPERTS, 1 <= block_size <= 4096,
 * numel + E * (block_size - 1) < 2^31.  The result is unique (stable order), so
 * it is bit-for-bit reproducible.  Three kernels: per-chunk counts, one CTA
 * that turns them into positions and writes the padding and block experts,
 * and the stable placement.
 */
int64_t mgemm_moe_align_workspace_bytes(int64_t numel, int E);
int mgemm_moe_align(const int32_t *topk_ids, int64_t numel, int E, int block_size, int32_t *sorted_ids,
                    int32_t *expert_ids, int32_t *num_post_padded, int64_t *group_sizes, void *workspace,
                    mgemm_stream_t stream);

/*
 * mgemm_moe_route_align -- for decode-size batches, one launch doing the work
 * of mgemm_topk_softmax, mgemm_moe_align and mgemm_fill_args (M = -1) in
 * sequence [CMM]: every output is what those three calls write, bit for bit.
 *   gating        float32 [T, E] (as for mgemm_topk_softmax), or NULL: the
 *                 routing is skipped and topk_ids is read as the input ids
 *                 (as for mgemm_moe_align, entries outside [0, E) are not
 *                 placed); topk_weights is then not used
 *   topk_weights  float32 [T, top_k], written when gating is given
 *   topk_ids      int32 [T, top_k]: written when gating is given, read otherwise
 *   sorted_ids, expert_ids, num_post_padded, group_sizes (may be NULL):
 *                 as from mgemm_moe_align with numel = T * top_k
 *   args          mgemm_args_bytes(E) bytes, 16-byte aligned: the args block of
 *                 the padded group sizes (the sorted rows' grouped GEMMs)
 * Limits: 1 <= E <= MGEMM_MAX_EXPERTS; 1 <= top_k (<= E when gating is given);
 * T * top_k <= MGEMM_ROUTE_ALIGN_MAX_ENTRIES; 1 <= block_size <= 4096.  Larger
 * batches return MGEMM_EINVAL: use the three calls, whose kernels spread over
 * the SMs.  With T = 0 the gating, weights and ids may be NULL; the other
 * outputs are still written (no entries: padding ids, empty groups).  One CTA
 * of 1024 threads.
 */
#define MGEMM_ROUTE_ALIGN_MAX_ENTRIES 4096
int mgemm_moe_route_align(const float *gating, int64_t T, int E, int top_k, int renormalize, int block_size,
                          float *topk_weights, int32_t *topk_ids, int32_t *sorted_ids, int32_t *expert_ids,
                          int32_t *num_post_padded, int64_t *group_sizes, void *args, mgemm_stream_t stream);

/*
 * The routed (fused_moe) layer [CMM], built from mgemm_moe_align and these
 * calls: x rows are gathered into expert order, the grouped GEMM runs over the
 * sorted rows, and its epilogue scatters each row to its flat (token, slot)
 * entry, optionally times the routed weight -- the work of fused_moe_kernel,
 * whose masked loads read padding entries as zero rows and whose masked stores
 * skip them; then silu_and_mul, the second GEMM with MUL_ROUTED_WEIGHT, and the
 * sum over the top_k slots of each token.
 *
 * mgemm_gather_rows -- dst row s = src row sorted_ids[s] / top_k for every s
 * below min(*num_post_padded, dst_rows); zeros when sorted_ids[s] >= numel (a
 * padding entry) or names a row outside src.  Rows from *num_post_padded on
 * are not written.
 *   src  [src_rows] rows of row_bytes bytes, src_ld_bytes apart
 *   dst  [dst_rows] rows, dst_ld_bytes apart (row_bytes and both strides
 *        multiples of 16; src and dst 16-byte aligned)
 *   sorted_ids, num_post_padded, numel: as from mgemm_moe_align
 */
int mgemm_gather_rows(const void *src, int64_t src_rows, int64_t row_bytes, int64_t src_ld_bytes,
                      const int32_t *sorted_ids, const int32_t *num_post_padded, int64_t numel, int top_k,
                      void *dst, int64_t dst_rows, int64_t dst_ld_bytes, mgemm_stream_t stream);

/*
 * mgemm_fwd_scatter -- mgemm_fwd over rows sorted by expert, with each output
 * row stored at the row row_map names (fused_moe_kernel's c_ptrs), optionally
 * multiplied by its routed weight (MUL_ROUTED_WEIGHT: the fp32 accumulator row
 * times the weight, then one rounding to bf16).
 *   args        args block of the sorted rows: mgemm_fill_args over the padded
 *               group sizes of mgemm_moe_align, with M = -1
 *   x           bf16 [M, K]: the sorted rows (mgemm_gather_rows); M >= the
 *               padded total (e.g. the sorted_ids capacity)
 *   w           bf16 [E, N, K] (trans_b = 1, the layout of fused_moe) or [E, K, N]
 *   out         bf16 [map_limit, N]
 *   row_map     int32 [M]: output row of sorted row i (sorted_ids: flat entry
 *               ids); a row with row_map[i] < 0 or >= map_limit (padding) is
 *               not stored
 *   map_limit   rows of out (numel of topk_ids)
 *   row_weight  float32 [map_limit] or NULL
 * bf16 only (fp8 returns MGEMM_ENOTSUP).  Output rows no sorted row names are
 * left as they were.  With map_limit < 128 (decode-size batches: a group has
 * at most map_limit routed rows, at the start of its block) only those rows of
 * each block are loaded.
 */
int mgemm_fwd_scatter(const void *args, int dtype, int trans_b, const void *x, const void *w, void *out,
                      const int32_t *row_map, int64_t map_limit, const float *row_weight, int64_t M, int K, int N,
                      int E, mgemm_stream_t stream);

/*
 * mgemm_fwd_gated -- the first GEMM of fused_moe with silu_and_mul in its
 * epilogue: out[r, j] = silu(g) * u with g = x[r, :] . w[e(r), j, :] and
 * u = x[r, :] . w[e(r), F + j, :] (the gate and up halves of w1 [E, 2F, K],
 * vLLM's silu_and_mul convention), g and u in fp32, silu(g) = g / (1 + exp(-g)),
 * one rounding to bf16.  Each tile's weight stage holds matching gate and up
 * rows, so both halves of an output column meet in one accumulator.
 *   args, x [M, K], M, K, E: as for mgemm_fwd (bf16)
 *   w    bf16 [E, 2F, K];  out  bf16 [M, F] (F % 8 == 0)
 *   group_rows_max  an upper bound on the rows of any group that are not
 *        padding (the routed entries; they come first in each 128-row block,
 *        as mgemm_moe_align places them), or 0 if unknown.  Below 128 (decode-
 *        size batches) only those rows of each block are loaded and stored:
 *        the padding rows of out are then left as they were.
 */
int mgemm_fwd_gated(const void *args, const void *x, const void *w, void *out, int64_t M, int K, int F, int E,
                    int64_t group_rows_max, mgemm_stream_t stream);

/*
 * mgemm_fwd_gated_gather -- mgemm_fwd_gated whose sorted rows are read from
 * the token rows through the sorted entry ids, as fused_moe_kernel loads A
 * through sorted_token_ids [CMM]: sorted row i is x row sorted_ids[i] / top_k,
 * or a row of zeros when sorted_ids[i] >= numel (padding), so the gathered
 * copy of mgemm_gather_rows is not needed.  The outputs equal those of
 * mgemm_gather_rows followed by mgemm_fwd_gated, bit for bit.
 *   x           bf16 [x_rows, K] (the token rows), 16-byte aligned
 *   sorted_ids, numel, top_k: as from mgemm_moe_align (sorted_ids holds at
 *               least M entries)
 *   args, w, out, M, K, F, E, group_rows_max: as for mgemm_fwd_gated
 * For decode-size batches only: 1 <= group_rows_max <= 32 and K % 64 == 0;
 * other shapes return MGEMM_ENOTSUP.  The GEMM's producer copies the rows
 * itself (16-byte asynchronous copies into the swizzled operand layout).
 */
int mgemm_fwd_gated_gather(const void *args, const void *x, int64_t x_rows, const int32_t *sorted_ids, int64_t numel,
                           int top_k, const void *w, void *out, int64_t M, int K, int F, int E,
                           int64_t group_rows_max, mgemm_stream_t stream);

/*
 * mgemm_silu_and_mul -- out[r, j] = silu(in[r, j]) * in[r, F + j] for in bf16
 * [R, 2F] and out bf16 [R, F] (vLLM's silu_and_mul as fused_moe applies it to
 * the first GEMM's output), silu(v) = v / (1 + exp(-v)), computed in fp32 and
 * rounded to bf16 once.  F % 8 == 0; pointers 16-byte aligned.
 */
int mgemm_silu_and_mul(const void *in, int64_t R, int64_t F, void *out, mgemm_stream_t stream);

/*
 * mgemm_topk_sum -- out[t, :] = sum_j in[t * top_k + j, :] for in bf16
 * [T * top_k, H] and out bf16 [T, H] (fused_moe's final sum over the top_k
 * slots), accumulated in fp32 in ascending j and rounded to bf16 once.
 * H % 8 == 0; pointers 16-byte aligned.
 */
int mgemm_topk_sum(const void *in, int64_t T, int top_k, int64_t H, void *out, mgemm_stream_t stream);

/*
 * mgemm_topk_softmax -- fused_moe's routing [CMM] (its topk_softmax call and
 * renormalize step): per token t, p = softmax(gating[t, :]) over the E
 * experts; topk_ids[t, :] = the top_k experts, largest probability first;
 * topk_weights[t, :] = their probabilities, divided by their sum when
 * renormalize != 0.
 *   gating        float32 [T, E], finite
 *   topk_weights  float32 [T, top_k];  topk_ids  int32 [T, top_k]
 * The selection compares logits (softmax is increasing in each, so the same
 * experts, with no rounding ties); equal logits go to the lower id.  The
 * weights are exp(l - max) / sum in fp32.  1 <= top_k <= E <= MGEMM_MAX_EXPERTS.
 * One warp per token.
 */
int mgemm_topk_softmax(const float *gating, int64_t T, int E, int top_k, int renormalize, float *topk_weights,
                       int32_t *topk_ids, mgemm_stream_t stream);

/* Number of SMs of the current device (the persistent GEMM grid size), or < 0 on error. */
int mgemm_num_sms(void);
/* Static string naming a MGEMM_E* or MGEMM_STATUS_* code. */
const char *mgemm_error_string(int code);
/* Text describing the last CUDA failure that made a call return MGEMM_ECUDA
 * in the calling thread ("" if none); static per-thread storage, valid until
 * the next failing call from the same thread. */
const char *mgemm_last_error(void);
/* Library ABI version (major * 100 + minor). */
int mgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MGEMM_H_ */
