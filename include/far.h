/*
 * far.h -- C ABI of the GB300 fused residual-add + RMSNorm library.
 *
 * The operation is the one the case study "Aligning fused RMSNorm rounding
 * across vLLM backends" pins down (sections "Finding the rounding boundary"
 * and "Implementation and tradeoffs"), per row t of a [tokens, hidden]
 * row-major matrix:
 *
 *   s_i            = fl32(x_i + r_i)          binary32 add, never rounded before use
 *   residual_out_i = RNE_act(s_i)             rounded only when stored
 *   var            = fl32(S / hidden),        S = the binary32 sum of fl32(s_i * s_i)
 *   rstd           = fl32(1 / fl32(sqrt(fl32(var + eps))))
 *   out_i          = RNE_od(fl32(RNE_wd(fl32(s_i * rstd)) * w_i))
 *                                             cast to the weight dtype, then multiply
 *
 * The dtype policy is the one of the LyCORIS page "Precision", section
 * "Dtype policy": activations (x, residual, residual_out: dtype `act`) and the
 * weight (dtype `wd`) may each be fp16, bf16 or fp32, except fp16 together with
 * bf16, which is a caller error; out has the promoted dtype od (fp32 if either
 * is fp32, else the common 16-bit type).  Accumulation is binary32 throughout.
 *
 * Every entry point validates its arguments on the host first and returns a
 * status without touching memory when they are wrong.  0 means the work was
 * enqueued on `stream`; device faults surface at the caller's next
 * synchronisation (CUDA convention).  There is no CPU fallback: a pointer the
 * GPU cannot reach is a CUDA error, not a slow path.
 *
 * Memory: all tensors are caller-owned, contiguous and row-major (row stride =
 * hidden elements).  By default the device entry points allocate nothing and
 * keep no state from one call to the next: they only enqueue on the stream
 * they are given.  What the library holds is fixed at load time or created
 * once per device: a 4-byte device error word (far_device_status); the
 * host-buffer entry points' two internal streams and four events (created on
 * their first call on a device); the allocation-free entry point's 16 MiB
 * staging array (FAR_NOALLOC_SCRATCH_BYTES).  One opt-in mode keeps state
 * across calls: claimed rows (far_set_row_schedule(0) or (2)) use a 1 KB
 * device array of 64 row counters, create 64 CUDA events on a device's first
 * claimed launch, and remember which stream last used each counter; see
 * far_set_row_schedule.  The default, far_set_row_schedule(1), keeps none.
 *
 * Aliasing: an output may be the very same buffer as an input of the same
 * element size (in-place use: out == x, residual_out == residual, ...).  Any
 * other overlap between an output and any buffer is FAR_ERR_ALIAS.
 */
#ifndef FAR_H
#define FAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes */
typedef enum { FAR_F32 = 0, FAR_F16 = 1, FAR_BF16 = 2 } far_dtype;

/* the single `dtype` argument packs the activation and weight dtypes */
#define FAR_DTYPES(act, w) ((int)(act) | ((int)(w) << 4))

/* status codes */
#define FAR_OK 0
#define FAR_ERR_DTYPE_MIX 1  /* fp16 with bf16: a caller error under the dtype policy */
#define FAR_ERR_DTYPE 2      /* an unknown dtype code */
#define FAR_ERR_NULL 3       /* a required pointer is NULL (tokens > 0) */
#define FAR_ERR_SHAPE 4      /* hidden <= 0 or > 2^24, tokens < 0, or byte sizes overflow */
#define FAR_ERR_ALIAS 5      /* an output overlaps another buffer other than exactly */
#define FAR_ERR_EPS 6        /* eps is negative or not finite */
#define FAR_ERR_CUDA 7       /* a CUDA call failed; far_status_string gives its text */
#define FAR_ERR_TIMEOUT 8    /* a bounded wait inside a kernel ran out (far_device_status) */
#define FAR_ERR_WORKSPACE 9  /* the host-buffer entry points got too small a workspace */
#define FAR_ERR_SCRATCH 10   /* a row does not fit the allocation-free entry point's fixed scratch */

/*
 * Fused residual add + RMSNorm.
 *   x, residual     [tokens, hidden] act, device memory (read)
 *   weight          [hidden] wd, device memory (read)
 *   eps             added to the mean square inside the root (binary32)
 *   out             [tokens, hidden] od, device memory (written)
 *   residual_out    [tokens, hidden] act, device memory (written): RNE_act(x + r)
 *   tokens, hidden  tokens >= 0 (0 is a no-op), 1 <= hidden <= 2^24
 *   dtype           FAR_DTYPES(act, wd)
 *   stream          cudaStream_t to enqueue on; NULL is the legacy default stream
 * Returns FAR_OK or a status above.
 */
int fused_add_rmsnorm(const void* x, const void* residual, const void* weight, float eps,
                      void* out, void* residual_out, int64_t tokens, int64_t hidden,
                      int dtype, void* stream);

/*
 * RMSNorm without a residual: the same contract with s_i = x_i (exact
 * widening) and no residual_out.  Arguments as for fused_add_rmsnorm.
 */
int rmsnorm(const void* x, const void* weight, float eps, void* out,
            int64_t tokens, int64_t hidden, int dtype, void* stream);

/*
 * Strided rows: the same two operations on matrices whose consecutive rows are
 * *_row_stride ELEMENTS apart (each >= hidden; elements within a row stay
 * contiguous), e.g. column slices of wider matrices.  Rows whose starts are all
 * 16-byte aligned take the bulk-copy path; others the generic kernel, with the
 * same results.  Aliasing: an output may be exactly an input (same pointer,
 * stride and element size); otherwise no byte may be shared.  Regions with equal
 * strides are checked exactly (interleaved column slices of one buffer are
 * fine); regions with different strides must not even share their spanned
 * ranges.  FAR_ERR_SHAPE for a stride below hidden.
 */
int fused_add_rmsnorm_strided(const void* x, int64_t x_row_stride, const void* residual,
                              int64_t residual_row_stride, const void* weight, float eps, void* out,
                              int64_t out_row_stride, void* residual_out, int64_t residual_out_row_stride,
                              int64_t tokens, int64_t hidden, int dtype, void* stream);

int rmsnorm_strided(const void* x, int64_t x_row_stride, const void* weight, float eps, void* out,
                    int64_t out_row_stride, int64_t tokens, int64_t hidden, int dtype, void* stream);

/*
 * The argument checks of the strided entry points alone (no CUDA call, no memory
 * access): the status fused_add_rmsnorm_strided (has_residual = 1) or
 * rmsnorm_strided (has_residual = 0, residual arguments ignored) would return
 * before launching anything.
 */
int far_validate_strided(const void* x, int64_t x_row_stride, const void* residual, int64_t residual_row_stride,
                         const void* weight, float eps, const void* out, int64_t out_row_stride,
                         const void* residual_out, int64_t residual_out_row_stride, int64_t tokens, int64_t hidden,
                         int dtype, int has_residual);

/*
 * Quantised output: the same two operations followed by a per-token symmetric
 * quantisation of out (the "Mixed-Precision Kernels" page, section "Quantised
 * Kernels: INT8 and FP8 Inference": scale = max_abs / 127), applied to the
 * values out would have, so the result equals normalising and quantising apart:
 *   amax_t = max_i |out_ti|,  scale[t] = fl32(amax_t / QMAX),
 *   q_ti = Q(fl32(out_ti * fl32(QMAX / amax_t)))   (q = 0 for an all-zero row)
 *   FAR_Q_INT8:     QMAX = 127; nearest integer, ties to even, within +-127; NaN -> 0
 *   FAR_Q_FP8_E4M3: QMAX = 448; nearest E4M3 value, ties to even, finite values
 *                   saturated to +-448; NaN stays NaN
 *   q              [tokens, hidden] one byte an element (int8, or E4M3 codes), device
 *   scale          [tokens] binary32, device; dequantise as q * scale
 *   residual_out   as for fused_add_rmsnorm
 * q and scale may not overlap any other buffer.  FAR_ERR_DTYPE for an unknown qtype.
 */
#define FAR_Q_INT8 1
#define FAR_Q_FP8_E4M3 2

int fused_add_rmsnorm_quant(const void* x, const void* residual, const void* weight, float eps, void* q,
                            float* scale, void* residual_out, int64_t tokens, int64_t hidden, int dtype, int qtype,
                            void* stream);

int rmsnorm_quant(const void* x, const void* weight, float eps, void* q, float* scale, int64_t tokens,
                  int64_t hidden, int dtype, int qtype, void* stream);

/*
 * LayerNorm under the same rounding contract (the "Mixed-Precision Kernels" page,
 * section "Kernel-Level Mechanics: Cast Placement and Fusion": activations widened
 * on load, mean and variance accumulated in binary32, the result narrowed on store),
 * with the variance taken about the mean in a second pass over s instead of the
 * section's E[s^2] - mean^2 form:
 *   s_i           = fl32(x_i + residual_i)          (s_i = x_i for layernorm)
 *   residual_out_i = RNE_act(s_i)                    (fused_add_layernorm only)
 *   mean          = fl32(RN32(sum_i s_i) / hidden)
 *   d_i           = fl32(s_i - mean)
 *   var           = fl32(RN32(sum_i fl32(d_i * d_i)) / hidden)
 *   rstd          = fl32(1 / fl32(sqrt(fl32(var + eps))))
 *   n_i           = RNE_wd(fl32(d_i * rstd))         (cast to the weight dtype first)
 *   out_i         = RNE_od(fl32(fl32(n_i * gamma_i) + beta_i))
 * gamma and beta are [hidden] device vectors in the weight dtype wd; everything else
 * (dtype codes, layout, ownership, aliasing, asynchrony, statuses) is as for
 * fused_add_rmsnorm / rmsnorm with gamma in the weight's place.  beta is read-only:
 * FAR_ERR_NULL when it is NULL (tokens > 0), FAR_ERR_ALIAS when an output overlaps it.
 */
int fused_add_layernorm(const void* x, const void* residual, const void* gamma, const void* beta, float eps,
                        void* out, void* residual_out, int64_t tokens, int64_t hidden, int dtype, void* stream);

int layernorm(const void* x, const void* gamma, const void* beta, float eps, void* out, int64_t tokens,
              int64_t hidden, int dtype, void* stream);

/*
 * The consumer GEMM with fp16 storage and fp32 compute (the Luminal page "Luminal FP16
 * Backend Repair and H100 Evidence", section "What Was Fixed": the fp16 operands widened
 * exactly, products and sums in fp32, the result cast to fp16, then the fp16 bias add):
 *   x    [m, k] fp16, row-major, device
 *   wt   [n, k] fp16, row-major, device: the transposed weight (y = x @ wt^T)
 *   bias [n] fp16, device, or NULL
 *   out  [m, n] row-major, device:
 *     out_dtype FAR_F16: out = RNE_f16(RNE_f16(sum_k x[i,k] * wt[j,k]) + bias[j])
 *     out_dtype FAR_F32: out = the binary32 sum (bias must be NULL)
 * The order of the binary32 additions is not specified (tensor cores accumulate in
 * their own order); each product of two fp16 values is exact in binary32.  Tensor
 * cores (tcgen05) are used when k is a positive multiple of 8, n a multiple of 8 and
 * every pointer 16-byte aligned; any other shape takes a plain kernel with the same
 * contract.  out may not overlap x, wt or bias.  Statuses: FAR_ERR_DTYPE (out_dtype,
 * or a bias with FAR_F32), FAR_ERR_SHAPE (a negative size or one above 2^31 - 1),
 * FAR_ERR_NULL, FAR_ERR_ALIAS, FAR_ERR_CUDA.  Enqueued on `stream`; m == 0 or n == 0
 * is a no-op; k == 0 gives RNE_f16(0 + bias).
 */
int gemm_f16_f32acc(const void* x, const void* wt, const void* bias, void* out, int64_t m, int64_t n, int64_t k,
                    int out_dtype, void* stream);

/* the GEMM's plan for a device with `sms` SMs (host logic only, aligned operands):
   out6 = {kind (0 tensor cores, 1 plain, 2 tensor cores over CTA pairs), tile width, grid, threads,
   dynamic shared bytes, stages} */
int far_plan_gemm_for_sms(int64_t m, int64_t n, int64_t k, int has_bias, int out_dtype, int sms, int* out6);
/* process-wide override of the GEMM plan, for measurements and tests: kind -1 automatic,
   0 tensor cores, one CTA a tile, where feasible; 1 the plain kernel; 2 tensor cores over CTA
   pairs (256 x 256 tiles) where feasible; bn 0 automatic, else 64, 128 or 256 (kind 0) */
int far_set_gemm_override(int kind, int bn);

/*
 * Strided forms of LayerNorm and of the quantised output: as fused_add_rmsnorm_strided,
 * each activation tensor has its own row stride in elements (>= hidden; elements within a
 * row contiguous); an output may be exactly its input, no other byte may be shared.  q
 * and scale stay contiguous ([tokens, hidden] bytes and [tokens] binary32).
 */
int fused_add_layernorm_strided(const void* x, int64_t x_row_stride, const void* residual,
                                int64_t residual_row_stride, const void* gamma, const void* beta, float eps, void* out,
                                int64_t out_row_stride, void* residual_out, int64_t residual_out_row_stride,
                                int64_t tokens, int64_t hidden, int dtype, void* stream);

int layernorm_strided(const void* x, int64_t x_row_stride, const void* gamma, const void* beta, float eps, void* out,
                      int64_t out_row_stride, int64_t tokens, int64_t hidden, int dtype, void* stream);

int fused_add_rmsnorm_quant_strided(const void* x, int64_t x_row_stride, const void* residual,
                                    int64_t residual_row_stride, const void* weight, float eps, void* q, float* scale,
                                    void* residual_out, int64_t residual_out_row_stride, int64_t tokens,
                                    int64_t hidden, int dtype, int qtype, void* stream);

int rmsnorm_quant_strided(const void* x, int64_t x_row_stride, const void* weight, float eps, void* q, float* scale,
                          int64_t tokens, int64_t hidden, int dtype, int qtype, void* stream);

/* the output dtype od of FAR_DTYPES(act, wd), or -status when the pair is rejected */
int far_output_dtype(int dtype);

/* a static, human-readable text for a status (FAR_ERR_CUDA: the last CUDA error on this thread) */
const char* far_status_string(int status);

/*
 * Synchronises `stream`, then reports and clears the device-side error word of
 * the current device: FAR_ERR_TIMEOUT when a kernel gave up a bounded wait
 * since the last call (its outputs are then incomplete), FAR_ERR_CUDA when the
 * synchronisation itself failed, FAR_OK otherwise.
 */
int far_device_status(void* stream);

/*
 * End-to-end variants on HOST buffers: x, residual, weight, out and
 * residual_out are host pointers (pinned memory for asynchronous copies;
 * pageable memory works but the copies then block the calling thread).  The
 * call streams row chunks through `workspace` (caller-owned device memory of
 * `workspace_bytes`): host-to-device copy, kernel, device-to-host copy, with
 * two internal streams so that copies in both directions overlap the kernels.
 * Everything is ordered after the work already on `stream`, and work later
 * enqueued on `stream` is ordered after all of it.  Returns FAR_OK once
 * enqueued; the host outputs are valid after `stream` is synchronised.  Calls
 * on one device are serialised by a lock (they share the internal streams).
 */
int64_t far_host_workspace_bytes(int64_t chunk_tokens, int64_t hidden, int dtype, int has_residual);

int fused_add_rmsnorm_host(const void* x, const void* residual, const void* weight, float eps,
                           void* out, void* residual_out, int64_t tokens, int64_t hidden,
                           int dtype, void* workspace, int64_t workspace_bytes, void* stream);

int rmsnorm_host(const void* x, const void* weight, float eps, void* out, int64_t tokens,
                 int64_t hidden, int dtype, void* workspace, int64_t workspace_bytes, void* stream);

/*
 * The same host-buffer pipeline for LayerNorm and for the quantised outputs (arguments as
 * their device forms, every buffer on the host).  far_host_workspace_bytes_op sizes the
 * workspace for `chunk_tokens` rows of an op: 0 RMSNorm (as far_host_workspace_bytes),
 * 1 LayerNorm (gamma and beta kept once), 2 a quantised output (q and the per-row scales
 * in place of out).  Negative -status on bad arguments.
 */
int64_t far_host_workspace_bytes_op(int64_t chunk_tokens, int64_t hidden, int dtype, int has_residual, int op);

int fused_add_layernorm_host(const void* x, const void* residual, const void* gamma, const void* beta, float eps,
                             void* out, void* residual_out, int64_t tokens, int64_t hidden, int dtype,
                             void* workspace, int64_t workspace_bytes, void* stream);

int layernorm_host(const void* x, const void* gamma, const void* beta, float eps, void* out, int64_t tokens,
                   int64_t hidden, int dtype, void* workspace, int64_t workspace_bytes, void* stream);

int fused_add_rmsnorm_quant_host(const void* x, const void* residual, const void* weight, float eps, void* q,
                                 float* scale, void* residual_out, int64_t tokens, int64_t hidden, int dtype,
                                 int qtype, void* workspace, int64_t workspace_bytes, void* stream);

int rmsnorm_quant_host(const void* x, const void* weight, float eps, void* q, float* scale, int64_t tokens,
                       int64_t hidden, int dtype, int qtype, void* workspace, int64_t workspace_bytes,
                       void* stream);

/*
 * fused_add_rmsnorm_host on host buffers WITHOUT any allocation: no workspace
 * argument, no cudaMalloc or cudaFree, no stream or event creation.  (The pages
 * describe no such entry point: it is an addition of this library.)
 *
 * For callers that cannot allocate device memory themselves: code embedded in a
 * host program that owns all device memory through its own pool and forbids
 * other allocations, or code bound by a rule of no device allocation after
 * start-up.  They pass host buffers only, with the same meaning, layout and
 * checks as fused_add_rmsnorm_host.
 *
 * The device staging area is one fixed array inside the library,
 * FAR_NOALLOC_SCRATCH_BYTES (16 MiB) per GPU, held by every GPU that has
 * loaded it until the process exits.  Rows are streamed through it in chunks
 * on `stream` alone (copy in, kernel, copy out).  FAR_ERR_SCRATCH when a single
 * row of x, residual, out and residual_out plus the weight does not fit it
 * (a row of about 1.6 million elements when every dtype is 16-bit, 0.8 million
 * when every dtype is fp32).  Every byte the kernel reads from
 * the array is copied in by the same call, so nothing in it needs clearing;
 * the array keeps the last call's contents.  All calls share the one array:
 * calls that overlap on the GPU (on different streams, or from several host
 * threads) race on it and must be serialised by the caller.  The first call on
 * a device looks up the array's device address (once per device) and should
 * come before any stream capture on that device.
 */
#define FAR_NOALLOC_SCRATCH_BYTES (16ll << 20)

int fused_add_rmsnorm_host_noalloc(const void* x, const void* residual, const void* weight, float eps,
                                   void* out, void* residual_out, int64_t tokens, int64_t hidden, int dtype,
                                   void* stream);

/*
 * Failure-detection self test: launches one tiny kernel that waits on a
 * barrier nothing ever completes, with the same bounded wait the kernels use,
 * limited to `timeout_us` microseconds (1 .. 10^7).  The wait runs out, the
 * kernel records FAR_ERR_TIMEOUT in the device error word and returns, so a
 * following far_device_status(stream) reports it and the context stays usable.
 */
int far_selftest_wait_timeout(uint32_t timeout_us, void* stream);

/*
 * Tuning hooks (the library's own choice is used when they are not called).
 *
 * far_set_launch_override: process-wide override of the launch plan, for
 * measurements: kind -1 automatic, 0 staged kernel, 1 generic kernel; nch (16-byte
 * chunks per thread: 1, 2, 4, 8), groups (rows in flight per CTA) and stages
 * (shared-memory ring slots, 2..32) override the automatic choice when non-zero
 * and feasible.  Returns FAR_ERR_SHAPE for out-of-range values.
 *
 * far_describe_launch: the plan the library would use for a call with
 * 16-byte-aligned, non-overlapping buffers of this shape on the current device:
 * out6 = {kind, nch, warps per row, groups, stages, grid}.
 *
 * far_plan_for_sms: the same plan for a device with `sms` SMs, computed on the
 * host alone (no CUDA call): out8 = {kind, nch, warps per row, groups, stages,
 * grid, threads per CTA, dynamic shared-memory bytes}.
 */
int far_set_launch_override(int kind, int nch, int groups, int stages);
int far_describe_launch(int64_t tokens, int64_t hidden, int dtype, int has_residual, int* out6);
int far_plan_for_sms(int64_t tokens, int64_t hidden, int dtype, int has_residual, int sms, int* out8);
/* the same for the quantised entry points (qtype FAR_Q_INT8 or FAR_Q_FP8_E4M3) */
int far_plan_quant_for_sms(int64_t tokens, int64_t hidden, int dtype, int has_residual, int qtype, int sms,
                           int* out8);
/* the same for the LayerNorm entry points, with beta `beta_offset` bytes (0..15) past a
   16-byte boundary (every other buffer aligned) */
int far_plan_ln_for_sms(int64_t tokens, int64_t hidden, int dtype, int has_residual, int beta_offset, int sms,
                        int* out8);

/*
 * far_set_row_schedule: process-wide choice of how the staged kernel's CTAs share
 * rows.  Each CTA first takes rows at a fixed stride (its own index, plus the grid size
 * each time), as many as its shared-memory ring holds; after that it either keeps the
 * stride or claims the next free rows, a few at a time, from a counter of the launch.
 * Claimed rows keep the CTAs that the memory system serves faster busy until the last
 * rows, instead of idling them while slower ones finish (measured 2.5-4.4 % less time on
 * launches whose rows move 23 KB or more).  A claim takes as many rows as keep the claims
 * below ~150 M/s at the copy rate (one row where a row moves 45 KB or more).
 *   mode 1 (the default): the fixed stride always.  No state is kept between calls.
 *   mode 0: claimed rows where a claim takes one or two rows, the rows left after the
 *           first ring-full of every CTA are at least three times as many, the stream is
 *           not capturing a graph and a counter is free; also three rows a claim for the
 *           no-residual RMSNorm (16-bit out) and quantised kernels on 16-bit rows that
 *           are not a whole number of 256 16-byte chunks, with at least eight ring-fulls
 *           of rows; else the fixed stride.
 *   mode 2: claimed rows whenever there are rows left to claim (and a counter is free,
 *           and the stream is not capturing).
 * State of modes 0 and 2: the counters are a library-owned device array of 64 pairs a
 * device, each zero between launches (a launch's last CTA zeroes its pair).  A launch
 * takes the pair last used on its own stream (earlier launches there run before it), or
 * a pair with no launch pending whose CUDA event, recorded after its last launch, has
 * completed; so launches that can run side by side never share one.  The 64 events are
 * created on a device's first claimed launch and kept until exit.  A launch finding no
 * free pair, or a capturing stream, takes the fixed stride.  A stream must not begin a
 * capture while another host thread is launching on it in these modes (a pair whose
 * event record fell into a capture is retired for good).  The allocation-free entry
 * point always keeps the fixed stride.  The results are the same bits in every mode
 * (each row is computed the same way by whichever CTA takes it).  Returns FAR_ERR_SHAPE
 * for another mode.
 */
int far_set_row_schedule(int mode);
/* rows_per_claim: the rows a claim would take for such a call on a device with `sms` SMs
   under the current mode, or 0 where it keeps the fixed stride (host logic only: whether
   a counter is free or the stream capturing is decided at launch); op as
   far_host_workspace_bytes_op (0 RMSNorm, 1 LayerNorm, 2 a quantised output).
   FAR_ERR_SHAPE for tokens 0, sms < 1 or another op. */
int far_row_schedule_for_sms(int64_t tokens, int64_t hidden, int dtype, int has_residual, int op, int sms,
                             int* rows_per_claim);
/* the current mode of far_set_row_schedule */
int far_get_row_schedule(void);

/*
 * far_set_programmatic_launch: process-wide choice of how the normalisation kernels are
 * launched.  1 (the default): as programmatic dependent launches, so that a kernel is
 * dispatched while the kernel ahead of it on the stream finishes, and its CTAs take SMs as
 * that kernel's CTAs leave them; every kernel of this library first waits until the
 * kernels ahead of it have completed and their memory operations are visible, before it
 * touches any global memory, and it allows the next programmatic launch on the stream to
 * be dispatched as soon as it starts.  Stream order therefore holds as for a plain launch;
 * a stream of launches (this library's, or a caller's kernels launched the same way and
 * waiting the same way) loses less time between kernels.  A caller's kernel launched on
 * the same stream with the programmatic-stream-serialization attribute right after one of
 * these may start before it finishes: it must wait (griddepcontrol.wait, or
 * cudaGridDependencySynchronize) before it reads their outputs, as with any programmatic
 * launch; kernels launched without the attribute are ordered as usual.  0: plain launches.
 * The results are the same bits either way.  Returns FAR_ERR_SHAPE for another value.
 */
int far_set_programmatic_launch(int enable);
/* the current choice of far_set_programmatic_launch */
int far_get_programmatic_launch(void);
/* 1 if the calling thread's last kernel launch by this library claimed rows from a
   counter, else 0 (fixed-stride rows, the generic kernel, or no launch) */
int far_last_launch_claimed_rows(void);
/*
 * The counter pool's bookkeeping run alone, as host logic (no CUDA call), on a fresh pool
 * of 64 pairs: n operations of three int64 each, {op, a, b}:
 *   op 1  a launch on the stream with id a asks for a pair; b is a bit mask of the pairs
 *         whose event (recorded after their last launch) has completed, bit s for pair s;
 *         results[i] = the pair handed out, or -1 (the launch keeps the fixed stride);
 *   op 2  pair a is given back after its launch; b bit 0: the kernel was enqueued, bit 1:
 *         an event was recorded after it; results[i] = 0.
 * FAR_ERR_SHAPE for an unknown op, or for giving back a pair that is not handed out.
 */
int far_sched_pool_model(const int64_t* ops, int n, int* results);

#ifdef __cplusplus
}
#endif

#endif /* FAR_H */
