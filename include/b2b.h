/*
 * b2b.h -- C ABI of libb2b.so: fused GEMM/conv operator chains for one GB300 (sm_103a).
 *
 * Each fused entry point runs a whole operator chain in ONE kernel launch and keeps the
 * chain's intermediate on chip:
 *
 *   b2b_gemm           GEMM0 -> bias + activation -> GEMM1 -> bias + activation
 *   b2b_conv_nhwc      conv RxS (implicit GEMM) -> bias + act -> conv1x1 -> bias + act
 *   conv_relu_maxpool  conv3x3 -> bias -> ReLU -> maxpool 2x2/2
 *
 * Sources (page title, section):
 *   BOLT notes, "Enabling deeper operator fusion" / "Persistent kernel (GEMM/Conv)
 *     fusion": several GEMMs/convs in one kernel, no load/store of the intermediate
 *     through global memory, no second launch (Figure 4a/4b).
 *   BOLT notes, "Threadblock residence": the block that computes a GEMM0 output tile also
 *     computes the GEMM1 tile that consumes it, which needs ThreadBlock_N = GEMM_N (for a
 *     conv: = output channels).  Here one CTA owns all N0 and N1 columns of its 128 rows,
 *     hence the N0, N1 <= 256 limits below.
 *   BOLT notes, "Shared-memory-resident fusion": GEMM0's accumulator tile is converted
 *     and staged in shared memory, where GEMM1 reads it (Figure 7).
 *   BOLT notes, "Prerequisite: Epilogue fusion" and "Graph Level" (Conv2D + BiasAdd +
 *     Hardswish): column-broadcast bias, element-wise activation, dtype conversion.
 *   BOLT notes, "Templated code generation": all convs in NHWC; tensors padded to an
 *     alignment of 8 fp16 elements = 128 bits (errata note: "8 bit" means 8 elements).
 *   Welder notes, "Operator-tile and Tile-graph" / "Tile-graph Scheduling" (Figure 5):
 *     Conv + ReLU + MaxPool as one tile-graph; the (2,2,F) reuse tile stays on chip.
 *   AI-Infra interview notes, "Conv optimisation": implicit GEMM (addresses computed on
 *     the fly, no im2col buffer); a 1x1 conv is a GEMM.
 *
 * Conventions shared by every entry point
 *   - Element type: dt selects fp16 or bf16 for every tensor argument (inputs, weights,
 *     biases and outputs).  Products accumulate in fp32; bias and activation are applied
 *     in fp32; each stored tensor (the on-chip intermediate included) is rounded to nearest
 *     even into dt.
 *   - Layouts are row-major / NHWC and dense (no strides): see each function.
 *   - Pointers: tensor pointers are DEVICE pointers, 16-byte aligned.  Bias pointers are
 *     device pointers (2-byte aligned) or NULL for "no bias".
 *   - Channel / inner sizes (K0, N0, N1, C, C0, C1, Cin, Cout) are multiples of 8
 *     elements (16 bytes).  Callers with other sizes zero-pad channels, weights and
 *     biases up to the next multiple of 8; the padded output channels are then exactly 0.
 *   - Ownership: the caller owns every buffer.  The library allocates no device memory per
 *     call; its only state is a host-side cache of TMA tensor maps, a per-device record of
 *     kernel attributes, and one small device error word per device.
 *   - Asynchrony: calls enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and return without synchronising.  Outputs must not alias inputs.
 *   - Errors: argument errors are detected on the host before anything is launched and
 *     returned as a status; launch failures return B2B_ERR_CUDA.  A kernel that waits
 *     longer than the wait limit (b2b_set_wait_limit_ns) for an on-chip event gives up,
 *     leaves its output incomplete and records B2B_ERR_TIMEOUT in the device error word,
 *     read with b2b_get_device_error.  No call aborts, traps or throws.
 *   - Empty problems (M == 0, N == 0) return B2B_OK and launch nothing.
 */
#ifndef B2B_H
#define B2B_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum b2b_status {
    B2B_OK = 0,
    B2B_ERR_NULL = 1,         /* a required pointer is NULL */
    B2B_ERR_SHAPE = 2,        /* a size is negative, or the output would be empty/invalid */
    B2B_ERR_ALIGN = 3,        /* pointer not 16-byte aligned, or a channel size not % 8 */
    B2B_ERR_UNSUPPORTED = 4,  /* outside the kernels' limits (e.g. N0 > 512) */
    B2B_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed (no device, launch...) */
    B2B_ERR_TIMEOUT = 6       /* a kernel gave up waiting (from b2b_get_device_error) */
} b2b_status;

typedef enum b2b_dtype { B2B_F16 = 0, B2B_BF16 = 1 } b2b_dtype;

/* Element-wise operator of an epilogue, applied after the bias:
 *   NONE: y = z;  RELU: y = max(z, 0);  HARDSWISH: y = z * min(max(z + 3, 0), 6) / 6. */
typedef enum b2b_epilogue { B2B_EPI_NONE = 0, B2B_EPI_RELU = 1, B2B_EPI_HARDSWISH = 2 } b2b_epilogue;

/* ------------------------------------------------------------------------------------ */
/* Fused chains                                                                          */
/* ------------------------------------------------------------------------------------ */

/* D[M,N1] = e1( e0( A[M,K0] . W0[K0,N0] + b0 ) . W1[N0,N1] + b1 )
 * (BOLT notes: "Persistent kernel (GEMM/Conv) fusion", "Threadblock residence",
 *  "Shared-memory-resident fusion").
 *   A  [M][K0]  row-major      W0 [K0][N0] row-major     b0 [N0] or NULL
 *   W1 [N0][N1] row-major      b1 [N1] or NULL           D  [M][N1] row-major (output)
 * Limits: M >= 0; K0 >= 8; 8 <= N0 <= 512; 8 <= N1 <= 256, and N1 <= 128 when N0 > 256;
 * K0, N0, N1 multiples of 8.  The GEMM0 result tile (128 rows x N0) is rounded to dt and
 * kept on chip: in shared memory, or in TMEM over the GEMM0 columns already read (wide
 * N0).  For 256 < N0 <= 512 GEMM0 runs as two MMAs per K step over the two halves of the
 * 512 TMEM columns, one tile in flight per CTA (the Blackwell form of wider
 * threadblock-resident chains: the CTA still owns all N0 columns of its rows). */
b2b_status b2b_gemm(b2b_dtype dt, int64_t M, int32_t K0, int32_t N0, int32_t N1,
                    const void* A, const void* W0, const void* b0, b2b_epilogue e0,
                    const void* W1, const void* b1, b2b_epilogue e1,
                    void* D, void* stream);

/* D[M,N2] = e2( e1( e0( A . W0 + b0 ) . W1 + b1 ) . W2 + b2 ): three operators in one
 * persistent kernel (BOLT notes, "Enabling deeper operator fusion": more GEMMs fused into
 * one operator, no load or store of the intermediates).  Both intermediates are rounded
 * to dt and kept in shared memory; the three weights stay resident in shared memory.
 *   A  [M][K0]  row-major      W0 [K0][N0] row-major     b0 [N0] or NULL
 *   W1 [N0][N1] row-major      b1 [N1] or NULL
 *   W2 [N1][N2] row-major      b2 [N2] or NULL           D  [M][N2] row-major (output)
 * Limits as b2b_gemm for each size, and two tiles of D0, D1, D2 accumulators must fit the
 * 512 TMEM columns (N0 + N1 + N2 <= 256 once each is rounded up to 32) and the resident
 * weights beside two ring stages of A: B2B_ERR_UNSUPPORTED otherwise. */
b2b_status b2b_gemm3(b2b_dtype dt, int64_t M, int32_t K0, int32_t N0, int32_t N1, int32_t N2,
                     const void* A, const void* W0, const void* b0, b2b_epilogue e0,
                     const void* W1, const void* b1, b2b_epilogue e1, const void* W2,
                     const void* b2, b2b_epilogue e2, void* D, void* stream);

/* y = conv1x1_{W1,b1,e1}( conv_{W0,b0,e0}(x) ), stride 1, dilation 1, zero padding `pad`,
 * cross-correlation (implicit GEMM; interview notes "Conv optimisation", item 2; BOLT
 * notes "Persistent kernel fusion" for the conv case, ThreadBlock_N = output channels).
 *   x  [N][H][W][C]             W0 [C0][R][S][C]          b0 [C0] or NULL
 *   W1 [C1][C0]  (the 1x1 filter, output-channel major)   b1 [C1] or NULL
 *   y  [N][Ho][Wo][C1] with Ho = H + 2*pad - R + 1, Wo = W + 2*pad - S + 1 (output)
 * Limits: N, H, W >= 0; Ho, Wo >= 1 when N*H*W > 0; 1 <= R, S <= 7; 0 <= pad <= 3;
 * C >= 8, 8 <= C0 <= 256, 8 <= C1 <= 256, all multiples of 8. */
b2b_status b2b_conv_nhwc(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                         const void* x, const void* W0, int32_t C0, int32_t R, int32_t S,
                         int32_t pad, const void* b0, b2b_epilogue e0,
                         const void* W1, int32_t C1, const void* b1, b2b_epilogue e1,
                         void* y, void* stream);

/* b2b_conv_nhwc with the first conv at spatial stride `stride` in both dimensions (Welder
 * notes, "Operator-tile and Tile-graph", tile propagation: a strided conv reads a strided
 * input region, so each output tile's input tile is (8 - 1) * stride + R rows by
 * (16 - 1) * stride + S columns, of which every stride-th pixel is used):
 *   h[n,ho,wo,:] = e0( sum_{r,s} x[n, stride*ho + r - pad, stride*wo + s - pad, :] . W0 + b0 )
 * with Ho = (H + 2 pad - R) / stride + 1, Wo = (W + 2 pad - S) / stride + 1 (floor); the
 * 1x1 conv that follows has stride 1.  y [N][Ho][Wo][C1].  1 <= stride <= 4
 * (B2B_ERR_UNSUPPORTED above); other arguments and limits as b2b_conv_nhwc, which is this
 * call with stride 1.  A strided 1x1 conv (pad 0) runs as an implicit GEMM, not as a GEMM
 * over the pixel rows. */
b2b_status b2b_conv_nhwc_strided(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                                 const void* x, const void* W0, int32_t C0, int32_t R,
                                 int32_t S, int32_t pad, int32_t stride, const void* b0,
                                 b2b_epilogue e0, const void* W1, int32_t C1, const void* b1,
                                 b2b_epilogue e1, void* y, void* stream);

/* y = maxpool2x2_stride2( ReLU( conv3x3_pad1(x, Wt) + b ) ), floor mode
 * (Welder notes, "Tile-graph Scheduling", Figure 5: Conv+ReLU at registers, ReLU->MaxPool
 * through the (2,2,F) reuse tile; the conv output never reaches global memory).
 *   x  [N][H][W][Cin]     Wt [Cout][3][3][Cin]     b [Cout] or NULL
 *   y  [N][H/2][W/2][Cout] (output; an odd last row/column of the conv is dropped)
 * Limits: N >= 0; H, W >= 2; Cin >= 8; 8 <= Cout <= 256; Cin, Cout multiples of 8.
 * For Cout <= 128 one more launch layout runs over CTA pairs (clusters of two CTAs, each
 * MMA of 256 rows covering one 8 x 16 output tile per CTA, each CTA holding half of the
 * filters, up to three MMA issuers; the bias is then added in fp32 after the sums rather
 * than as a last MMA step, so that on non-integer data its outputs may differ from the
 * single-CTA layout's in the last place, within the tolerance; the last layout index, see
 * b2b_debug_plan); the tile-graph model takes it where its bounds are lower and every pair
 * runs three or more pairs of tiles. */
b2b_status conv_relu_maxpool(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t Cin,
                             const void* x, const void* Wt, const void* b, int32_t Cout,
                             void* y, void* stream);

/* ------------------------------------------------------------------------------------ */
/* Single operators: the unfused two-kernel path the fused chains are measured against   */
/* ------------------------------------------------------------------------------------ */

/* D[M,N] = e( A[M,K] . W[K,N] + b ); layouts and limits as GEMM0 of b2b_gemm. */
b2b_status gemm_bias_act(b2b_dtype dt, int64_t M, int32_t K, int32_t N,
                         const void* A, const void* W, const void* b, b2b_epilogue e,
                         void* D, void* stream);

/* y[N,Ho,Wo,Co] = e( conv_{R x S, pad}(x[N,H,W,C], Wt[Co][R][S][C]) + b );
 * layouts and limits as the first conv of b2b_conv_nhwc. */
b2b_status conv_bias_act_nhwc(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                              const void* x, const void* Wt, int32_t Co, int32_t R, int32_t S,
                              int32_t pad, const void* b, b2b_epilogue e,
                              void* y, void* stream);

/* conv_bias_act_nhwc at spatial stride `stride` (1 to 4), as the first conv of
 * b2b_conv_nhwc_strided. */
b2b_status conv_bias_act_nhwc_strided(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                                      const void* x, const void* Wt, int32_t Co, int32_t R,
                                      int32_t S, int32_t pad, int32_t stride, const void* b,
                                      b2b_epilogue e, void* y, void* stream);

/* Batch normalisation folded into the weights and bias of the operator before it
 * (interview notes, "阿里巴巴 AI Infra (2)", TVM Relay scheduling primitives,
 * SimplifyInference: at inference BN is a per-channel scale and bias, which folded into
 * the preceding conv or GEMM makes the chain's bias epilogue):
 *   s[co]  = gamma[co] / sqrt(var[co] + eps)
 *   W'[..] = rnd(W[..] * s[co]),   b'[co] = rnd((b[co] - mean[co]) * s[co] + beta[co])
 * in fp32, one round-to-nearest-even per stored value.  W is [Co][K] (out_inner = 0: conv
 * filters [Co][R][S][Cin], K = R*S*Cin; b2b_conv_nhwc's W1 [C1][C0]) or [K][Co]
 * (out_inner = 1: b2b_gemm's row-major W0/W1).  gamma, beta, mean, var: fp32 device
 * arrays [Co]; b [Co] or NULL (0); W_out / b_out may be W / b (in place).  Device
 * pointers; asynchronous on `stream`.  Errors: B2B_ERR_SHAPE (Co or K < 1, eps < 0),
 * B2B_ERR_NULL, B2B_ERR_ALIGN (fp16/bf16 arrays 2-byte, fp32 arrays 4-byte aligned),
 * B2B_ERR_UNSUPPORTED (dtype, out_inner), B2B_ERR_CUDA. */
b2b_status b2b_fold_batchnorm(b2b_dtype dt, int64_t Co, int64_t K, int32_t out_inner,
                              const void* Wt, const void* b, const float* gamma,
                              const float* beta, const float* mean, const float* var, float eps,
                              void* W_out, void* b_out, void* stream);

/* y[N,H/2,W/2,C] = max over each 2x2 window (stride 2, floor mode) of x[N,H,W,C].
 * Limits: H, W >= 2; C multiple of 8. */
b2b_status maxpool2x2_nhwc(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                           const void* x, void* y, void* stream);

/* ------------------------------------------------------------------------------------ */
/* Diagnostics                                                                           */
/* ------------------------------------------------------------------------------------ */

/* Static string naming a status. */
const char* b2b_status_str(b2b_status s);

/* Library version, e.g. "0.1.0". */
const char* b2b_version(void);

/* Number of SMs of the current device (the persistent grid size), or -1 on error. */
int32_t b2b_num_sms(void);

/* Wait limit, in nanoseconds, that later launches give each of their on-chip waits
 * (default 1e9 = 1 s).  0 restores the default.  Host-side setting, not per stream. */
void b2b_set_wait_limit_ns(uint64_t ns);

/* Event trace for performance analysis.  When buf is not NULL, every later launch of a
 * chain kernel records, for its CTA number `cta` only, the time (%globaltimer, ns) at
 * which each role reached each step of each tile.  buf is a caller-owned, zero-filled
 * device array of 2 * capacity uint64 words split into four equal regions (producer,
 * MMA issuer, epilogue group 0, epilogue group 1); each role appends its events to its
 * region: word 2i = time, word 2i+1 = event code | group << 8 | tile index << 16 |
 * 1 << 63 (codes: TraceEvent in kernel_params.h); unused words stay 0.  buf = NULL turns
 * tracing off.  buf must be 8-byte aligned and stay valid while traced launches run.
 * Traced launches run a separate build of the kernels with the recording compiled in;
 * untraced launches carry none of it, so timings taken under a trace run a little slow. */
b2b_status b2b_set_trace(void* buf, uint32_t capacity, uint32_t cta);

/* Reads and clears the current device's error word.  Synchronises the current device.
 * Returns B2B_OK if no kernel recorded an error, B2B_ERR_TIMEOUT if one gave up waiting
 * (then info[0] = code, info[1] = kernel id, info[2] = wait site, info[3] = tile index),
 * or B2B_ERR_CUDA if the word could not be read.  info may be NULL. */
b2b_status b2b_get_device_error(uint32_t info[4]);

/* Launches a one-CTA kernel that waits, with the given limit, on an on-chip barrier that
 * nothing will ever signal, so that it takes its timeout path and records
 * B2B_ERR_TIMEOUT.  Used by tests of the failure-detection path. */
b2b_status b2b_probe_timeout(uint64_t limit_ns, void* stream);

/* Describes, without any CUDA call, the launch an entry point would make for the given
 * sizes: its shared-memory plan and TMEM use.  For tests and tuning.
 *   kind 0 b2b_gemm            dims = {M, K0, N0, N1}
 *   kind 1 gemm_bias_act       dims = {M, K, N}
 *   kind 2 b2b_conv_nhwc       dims = {N, H, W, C, C0, R, S, pad, C1[, stride]}
 *   kind 3 conv_bias_act_nhwc  dims = {N, H, W, C, Co, R, S, pad[, stride]}
 *   kind 4 conv_relu_maxpool   dims = {N, H, W, Cin, Cout}
 *   kind 5 b2b_gemm3           dims = {M, K0, N0, N1, N2}
 * The sizes may be followed (for the convs, after the stride, which must then be given) by
 * the call's variant: its dtype (b2b_dtype), then each of its epilogue kinds (b2b_epilogue:
 * e0, e1 for kinds 0 and 2, e for 1 and 3, e0, e1, e2 for 5, none for 4).  Launch choices are
 * filed per variant, since each dtype and epilogue pair runs its own kernel instantiation;
 * sizes alone address every variant (see b2b_set_choice).  Any other count of dims, or a
 * variant value out of range, returns B2B_ERR_SHAPE.
 * out (out_len >= 64) receives, in order: dynamic smem bytes, ring stages, stage bytes,
 * weights resident (0/1), output staging aliases P (0/1), ring offset, ring bytes,
 * resident-weight offset, W1 offset, resident bytes, W0 chunk bytes, W1 chunk bytes,
 * P offsets [2], bytes per P buffer, staging offsets [2], bytes per staging buffer,
 * bias offset, bias bytes, barrier offset, barrier bytes, TMEM columns, GEMM0 accumulator
 * columns [2], GEMM1 accumulator columns [2], two tiles in flight (0/1), epilogue groups
 * (1/2), tiles, GEMM0 K chunks, GEMM1 K chunks, padded N0, padded N1, kernel mode
 * (0 chain, 1 single, 2 pool), 1 if the chain's intermediate is kept in TMEM instead
 * of shared memory (wide N0: GEMM1 then reads its A operand from TMEM), 1 if W1 is then
 * loaded once per pair of tiles into shared ring stages, the W1 chunks per stage, 1 if a
 * conv loads one halo box per column tap for all row taps, the A bytes per ring stage, the
 * number of accumulator buffers (tiles in flight: 1, 2, 4, or 6 for the conv + pool over
 * CTA pairs with three MMA issuers), P offsets [2..3], GEMM0
 * accumulator columns [2..3], GEMM1 accumulator columns [2..3], the layout taken (an
 * index into the feasible layouts, in the planner's order of preference), the number of
 * feasible layouts, and the pinned or measured grid and second-tile-prefetch choices
 * (b2b_set_choice; -1, as a two's-complement word, for the default), and the ring stages
 * a launch adds over the output staging when no CTA gets more than two tiles (P in TMEM,
 * streamed weights; the staging is first written after the pair's last GEMM0), then, for
 * the three-operator chain, the resident W2 offset, P1 offsets [2] and GEMM2 accumulator
 * columns [2] (0 otherwise), the TMEM column split of a wide chain's two GEMM0 passes (256,
 * else 0), and 1 if W0 alone stays resident while A and W1 stream through the ring (P in
 * TMEM, tile pairs; the output is then stored from registers, with no staging tile), and
 * 1 if the launch runs over CTA pairs (clusters of two CTAs sharing each MMA of 256 rows,
 * each holding half of W0 (and W1); for the b2b GEMM chain tiles then count 256 rows, for
 * the conv + pool they still count 8 x 16 tiles, two per MMA), the MMA issuers beyond the
 * first: 1 if two warps issue the MMAs of alternate tiles, each from its own half of the
 * ring (the single-CTA conv + pool kernel with N0 <= 64 when half the ring holds a tile's
 * stages; conv chains with halo boxes and N0 <= 64 in their two-issuer layout), and for
 * the conv + pool over CTA pairs 0, 1 or 2 (one issuer per tile's stages the ring holds,
 * up to three; three only when their six accumulators fit TMEM), 1 if each epilogue
 * warp stages its output 16 columns at a time in a 1 KiB slot of its own (that two-issuer
 * layout), and the TMEM columns of the two P buffers when P is kept in TMEM (else 0).  A
 * choice pinned,
 * measured or ranked for these sizes is reflected; without one, the layout is the
 * tile-graph model's pick, as the entry point takes it (see b2b_set_autotune).
 * Returns the status the entry point would return for these sizes (B2B_OK if it would
 * launch). */
b2b_status b2b_debug_plan(int32_t kind, const int64_t* dims, int32_t ndims, uint32_t* out,
                          int32_t out_len);

/* As b2b_debug_plan, with the layout forced to feasible candidate `cand` (0 = the
 * planner's most preferred) whatever is pinned or measured: the plan each candidate
 * would make, for a host-side model to rank (Welder notes, "Scheduling policy": candidate
 * tile graphs are enumerated, checked against the memory footprint and ranked by their
 * traffic before any is profiled).  B2B_ERR_UNSUPPORTED if cand is not feasible,
 * B2B_ERR_SHAPE if it is negative. */
b2b_status b2b_debug_plan_candidate(int32_t kind, const int64_t* dims, int32_t ndims,
                                    int32_t cand, uint32_t* out, int32_t out_len);

/* Launch choices and the light-weight profiler (BOLT notes, "Light-weight performance
 * profiler" under "Automating templated code generation": a profiler picks among
 * template configurations by timing them; here the configurations are launch choices of
 * one kernel, which compute the same products with the same
 * roundings: results are bit-identical, except that an R x S conv (R > 1) sums its taps
 * in another fp32 order when its filters are resident (halo loads) than when they are
 * streamed, and that the conv + pool over CTA pairs adds the bias in fp32 after the sums,
 * not as a last MMA step).
 * The default layout of a problem is the pick of a tile-graph cost model (Welder notes,
 * "Scheduling policy": candidates are ordered by their traffic before any is profiled):
 * for each feasible layout it bounds the launch from below by HBM (the problem's
 * irreducible bytes), L2 -> SM (the busiest CTA's loads) and the tensor pipe (the busiest
 * CTA's MMAs).  Where every CTA of the compared plans runs three or more tiles, the plan
 * with the lower bounds wins, resource by resource from the binding one (within 2 % they
 * tie); otherwise, or on a tie, the planner's order of preference decides (more tiles in
 * flight, resident weights, separate staging, rings of three or more stages first).  The
 * profiler times the model's best three layouts and every later one the bounds do not
 * order against the third.
 * A problem is an entry point (kind, as for b2b_debug_plan), its sizes and its variant
 * (dtype and epilogue kinds; dims as for b2b_debug_plan).  A call looks up its own
 * variant's choice first, then one recorded for the sizes alone; the profiler files what
 * it measures under the call's variant.  Its
 * launch may vary: the shared-memory / TMEM layout (cand: an index into the feasible
 * layouts, 0 = most preferred), the grid (0: one CTA per SM, or per tile when there are
 * fewer tiles; 1: the fewest CTAs that give no CTA more tiles than grid 0 does; 2: one
 * CTA per tile, in as many waves as it takes) and
 * whether each CTA also prefetches its second tile's A rows into L2 at the start
 * (prefetch_second 0/1; 2-D A operands only).  -1 leaves a field to the default.
 *
 * b2b_set_autotune(1): from then on, the first call of an entry point for a problem with
 * no pinned or measured choice times the default and every choice over the ranked
 * layouts (2 warm-up launches,
 * then the fastest of 3 rounds of 10, CUDA events on the caller's stream, which it
 * synchronises; the outputs are overwritten with the same values each time; the inputs
 * are the caller's, so a problem smaller than L2 is timed with its inputs in L2), keeps
 * the fastest for later calls of that problem -- the default unless another choice is
 * more than 2 % faster -- and then runs it for the caller.  Calls on a stream being captured into a
 * CUDA graph use the current choice or the default and never time.  Off by default.
 * b2b_autotune_reset forgets every pinned and measured choice.  Host state shared by all
 * devices and threads of the process. */
void b2b_set_autotune(int32_t on);
void b2b_autotune_reset(void);

/* Pins a launch choice for a problem (no CUDA call); dims without a variant pin it for
 * every dtype and epilogue of those sizes.  B2B_ERR_UNSUPPORTED if cand is not
 * a feasible layout for these sizes, B2B_ERR_SHAPE for a field out of range, otherwise the
 * status b2b_debug_plan would return. */
b2b_status b2b_set_choice(int32_t kind, const int64_t* dims, int32_t ndims, int32_t cand,
                          int32_t grid, int32_t prefetch_second);

/* The choice recorded for a problem (no CUDA call): out (out_len >= 7) = {source (0 none,
 * 1 pinned, 2 measured, 3 ranked by b2b_set_candidates and not yet measured), cand, grid,
 * prefetch_second, fastest time in ns, default's time in ns, choices timed} (times 0
 * unless measured).  dims with a variant read that variant's entry, else the one pinned for
 * its sizes alone (the choice its calls take); dims without one read the most recently
 * recorded entry of those sizes, for every variant or for one. */
b2b_status b2b_get_choice(int32_t kind, const int64_t* dims, int32_t ndims, int32_t* out,
                          int32_t out_len);

/* Hands the profiler a model's ranking of layouts for a problem (no CUDA call; Welder
 * notes, "Scheduling policy": the cost model keeps the top candidates and hardware
 * profiling picks among them).  cands (n in [1, 64], distinct feasible layout indices as
 * b2b_debug_plan_candidate numbers them) replaces any pinned or measured choice of the
 * problem: calls launch cands[0] with the default grid and prefetch, and with the profiler
 * on, the first call times only these layouts (each with every grid and prefetch choice),
 * cands[0] standing as the default that another must beat by the profiler's margin.
 * B2B_ERR_SHAPE (n out of range, a negative or repeated index), B2B_ERR_NULL,
 * B2B_ERR_UNSUPPORTED (an infeasible index), otherwise the status of b2b_debug_plan. */
b2b_status b2b_set_candidates(int32_t kind, const int64_t* dims, int32_t ndims,
                              const int32_t* cands, int32_t n);

/* Why the profiler chose what it chose (no CUDA call): every launch choice it timed for a
 * problem, the default first, as rows of five int32 in out (room for max_rows rows):
 * {layout index, grid mode, CTAs launched (clusters for CTA pairs), prefetch_second (-1:
 * the default rule), fastest round's time per launch in ns}.  *rows receives the number of
 * rows recorded (0 unless measured), which may exceed max_rows.  dims as for
 * b2b_get_choice.  B2B_ERR_NULL (rows NULL, or out NULL with max_rows > 0),
 * B2B_ERR_SHAPE (max_rows < 0). */
b2b_status b2b_get_tune_record(int32_t kind, const int64_t* dims, int32_t ndims, int32_t* out,
                               int32_t max_rows, int32_t* rows);

#ifdef __cplusplus
}
#endif

#endif /* B2B_H */
