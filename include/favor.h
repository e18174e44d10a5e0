/*
 * favor.h -- C ABI of libfavor, the GB300 (sm_103a) FAVOR+ attention forward pass.
 *
 * What is computed (per head h, b):
 *
 *   positive random features (FAVOR+)
 *     phi(x) = exp(-|x|^2/2)/sqrt(m) [exp(w_1.x), ..., exp(w_m.x)]          (r = m)
 *       -- "Linear Attention > Performer: Unbiased Softmax Approximation", the
 *          phi(x) equation; "Linear Attention > Kernel Feature Maps", section 4.
 *   random Fourier features
 *     phi(x) = 1/sqrt(m) [sin(w_1.x), cos(w_1.x), ..., sin(w_m.x), cos(w_m.x)]  (r = 2m)
 *       -- "Kernel Feature Maps", section 3.
 *   ELU + 1
 *     phi(x)_j = x_j + 1 (x_j > 0), exp(x_j) (x_j <= 0), no projection     (r = d, m must equal d)
 *       -- "Kernel Feature Maps", section 1.
 *   ReLU
 *     phi(x)_j = max(0, x_j), no projection                                 (r = d, m must equal d)
 *       -- "Kernel Feature Maps", section 2.  A query whose features meet no
 *          key mass has a zero denominator: its row is 0/0 (NaN).
 *   softmax-scaled random Fourier features
 *     phi(x) = exp(|x|^2/2) x the sin/cos map above, so that
 *     E[phi(q).phi(k)] = exp(q.k)                                             (r = 2m)
 *       -- "Kernel Feature Maps", section 3 (the additional scaling that turns
 *          the Gaussian-kernel estimate into a softmax-kernel estimate).
 *   ReLU and the softmax-scaled map run on the fp32 SIMT kernels.  A head of
 *   r = 64 features (positive m = 64, sin/cos m = 32, ELU+1 d = 64) runs on
 *   the tensor-core kernels as one of 128 with every projection taken twice:
 *   numerator and denominator both double, so out is the same.
 *
 *   non-causal:  out_i = phi(q_i)^T (sum_j phi(k_j) v_j^T) / phi(q_i)^T (sum_j phi(k_j))
 *       -- Performer page In[25] (performer_attention, with eps = 0) and the
 *          Performer study notes, "Core points" steps 4-5.
 *   causal:      S_i = sum_{j<=i} phi(k_j) v_j^T,  z_i = sum_{j<=i} phi(k_j),
 *                out_i = phi(q_i)^T S_i / phi(q_i)^T z_i   (diagonal included)
 *       -- Performer study notes, "Case 2: the causal version" (prefix sum),
 *          with the linear denominator of "Core points" step 5.
 *
 * Every kernel stabilises the exponentials (a per-row query maximum and a
 * per-head running key maximum); both cancel exactly in the ratio.
 *
 * Range of the tensor-core path (favor_attn_forward and its variants; the
 * fp32 entry points compute every feature in fp32, where the same underflow
 * comes only for a key some e^80 below the head's largest key feature).
 * Its MMA operands are fp16, whose finite range is 2^-24 .. 65504:
 *   - q, k and v values must be finite with |x| <= 65280 (the largest bf16
 *     value below fp16's 65504);
 *   - a key's largest feature is scaled to at most e^10 against the head's
 *     running key maximum; a key whose largest feature would land below
 *     2^-14 there (about e^-18 or more below the largest key feature of the
 *     head so far) would lose its features to fp16 underflow.
 * Isotropic inputs stay far inside both bounds (the largest feature of every
 * key of N(0,1) d^-1/4 inputs lands within [e^0, e^10]).  The kernels check
 * both on the device; an input outside them still completes, and the
 * device status word (favor_get_device_status) then reads FAVOR_ERR_RANGE:
 * the result is unreliable and favor_attn_forward_f32 on the same values
 * (bf16 widened to fp32) computes it within the fp32 bound.  Inside the
 * range the result is the definition above within fp16 operand rounding.
 *
 * Conventions common to all entry points
 *   - All tensors are dense, row-major, contiguous:
 *       q, k   [B][H][L][d]
 *       v      [B][H][L][dv]
 *       omega  [H][m][d]  fp32, one random projection per head, shared by the
 *              batch (rows w_i; drawn by the caller, iid N(0,I) or
 *              block-orthogonal).  Ignored (may be NULL) for FAVOR_MAP_ELU1 and
 *              FAVOR_MAP_RELU.
 *       out    [B][H][L][dv] fp32.
 *   - Device pointers must be 16-byte aligned; out must not alias an input.
 *   - The caller owns every buffer and the stream.  The library owns a
 *     per-device workspace that it grows on demand (cudaMalloc outside any
 *     stream capture) and frees in favor_release_workspace().  Every call on
 *     a device uses that one workspace: calls whose kernels can overlap on
 *     the GPU (streams with no ordering between them) race on it, so order
 *     such calls with events or issue them on one stream.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) unless
 *     stated otherwise.  Argument errors are detected on the host and
 *     returned before anything is launched.  A launch failure returns
 *     FAVOR_ERR_CUDA.  Kernels that wait on an mbarrier give up after a
 *     bounded number of polls and record FAVOR_ERR_TIMEOUT in a device status
 *     word that favor_get_device_status() reads.
 *   - Supported: B, H, L >= 1; d, dv in {32, 64, 128}; m >= 1 and m % 16 == 0
 *     (positive, trig, softmax-scaled trig); m == d (elu1, relu).  B*H*L*max(d,dv) must fit in int32
 *     element offsets per tensor (checked).
 */
#ifndef FAVOR_H
#define FAVOR_H

#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FAVOR_OK = 0,
    FAVOR_ERR_INVALID_ARG = -1, /* null pointer, bad size, misalignment, aliasing */
    FAVOR_ERR_UNSUPPORTED = -2, /* valid but outside the supported shapes       */
    FAVOR_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed          */
    FAVOR_ERR_TIMEOUT = -4,     /* a bounded device-side wait expired            */
    FAVOR_ERR_NOMEM = -5,       /* workspace allocation failed                   */
    FAVOR_ERR_RANGE = -6        /* device status only: an input left the range
                                   the fp16 tensor-core operands represent (see
                                   "Range of the tensor-core path" above); the
                                   call completed but its result is unreliable */
} favor_status_t;

typedef enum {
    FAVOR_MAP_POSITIVE = 0,     /* FAVOR+ positive random features, r = m            */
    FAVOR_MAP_TRIG = 1,         /* sin/cos random Fourier features, r = 2m           */
    FAVOR_MAP_ELU1 = 2,         /* elu(x) + 1, r = d (m must equal d)                */
    FAVOR_MAP_RELU = 3,         /* max(0, x), r = d (m must equal d)                 */
    FAVOR_MAP_TRIG_SOFTMAX = 4  /* exp(|x|^2/2) x the sin/cos map, r = 2m: unbiased
                                   for the softmax kernel exp(q.k)                   */
} favor_feature_map_t;

/* FAVOR attention forward, bf16 q/k/v (raw bf16 bit patterns), fp32 omega
 * and fp32 out, all device pointers.  causal: 0 = non-causal contraction,
 * 1 = causal prefix-state form.  feature_map: favor_feature_map_t.
 * The hot path: tcgen05 tensor-core kernels with fp16 operands and fp32
 * accumulation.  Returns favor_status_t. */
int favor_attn_forward(const void *q, const void *k, const void *v, const float *omega,
                       float *out, int B, int H, int L, int d, int dv, int m, int causal,
                       int feature_map, cudaStream_t stream);

/* No counterpart on the pages: favor_attn_forward for callers that must not
 * allocate device memory on the call path -- a process whose framework has
 * reserved the GPU's memory in its own caching pool (a further cudaMalloc
 * fails), or a serving loop that cannot take the device-wide synchronisation
 * of cudaMalloc/cudaFree mid-request.  Same parameters and result as
 * favor_attn_forward; it never calls cudaMalloc, cudaFree or an allocating
 * routine.  Its scratch is a fixed 32 MiB array in the library's device
 * memory, held on every GPU that loads the library until the process exits.
 * Returns FAVOR_ERR_UNSUPPORTED for a shape the tensor-core kernels do not
 * cover or whose scratch (per-head fp16 W image, segment or piece states,
 * the non-causal state image) exceeds 32 MiB.  The benchmark shapes fit:
 * with d=dv=64, m=256, B=4, H=16, L=8192 causal (about 9 MB), B=8, H=12,
 * L=4096 non-causal (about 26 MB) and B=1, H=8, L=65536 either way (about
 * 20 MB: 19 segments per head, their states and the combined states); with
 * d=dv=128, m=256, B=2, H=8, L=16384 causal.  256 heads of L=65536 do not
 * (their segment states alone take hundreds of MB).  The first
 * call on a device looks the array's device address up (make it before any
 * stream capture).  All calls share the array: calls whose kernels overlap
 * on the GPU race on it.  Nothing in it needs clearing between calls. */
int favor_attn_forward_noalloc(const void *q, const void *k, const void *v, const float *omega,
                               float *out, int B, int H, int L, int d, int dv, int m, int causal,
                               int feature_map, cudaStream_t stream);

/* favor_attn_forward with out stored as bf16 bits [B][H][L][dv] (round to
 * nearest even from the fp32 result): half the output traffic.  No
 * counterpart on the pages (they do not state an output type; the default
 * entry keeps fp32).  Same inputs, conventions and result codes. */
int favor_attn_forward_bf16out(const void *q, const void *k, const void *v, const float *omega,
                               void *out, int B, int H, int L, int d, int dv, int m, int causal,
                               int feature_map, cudaStream_t stream);

/* Same operation and parameters with fp32 q/k/v: computed entirely in fp32
 * (FFMA, accurate expf/sincosf) by SIMT kernels.  Returns favor_status_t. */
int favor_attn_forward_f32(const float *q, const float *k, const float *v, const float *omega,
                           float *out, int B, int H, int L, int d, int dv, int m, int causal,
                           int feature_map, cudaStream_t stream);

/* End-to-end variant of favor_attn_forward on HOST buffers (q/k/v bf16 bits,
 * omega and out fp32; pinned memory gives the fastest copies).  Copies the
 * inputs to a library-owned device staging area, runs the forward pass and
 * copies out back, in up to ten groups of whole heads (whole batches, or
 * head ranges of one batch; the last group small) whose copies run on two
 * library-owned streams while the caller's `stream` computes the neighbouring
 * groups; each group is a separate forward pass (its rows agree with one
 * device-buffer call to within the bf16 parity bar, not bit for bit).  Starts
 * after the work queued on `stream`, synchronises `stream` before returning.
 * Not for use inside a stream capture, nor from two threads at once on one
 * device.  The host buffers must hold the full [B][H][L][...] extents the
 * sizes name, like memcpy's: the copies read and write exactly that much, and
 * on a system where the GPU reaches pageable host memory through the CPU's
 * page tables a short buffer faults the copy engine, not just the process.
 * Returns favor_status_t. */
int favor_attn_forward_host(const void *q, const void *k, const void *v, const float *omega,
                            float *out, int B, int H, int L, int d, int dv, int m, int causal,
                            int feature_map, cudaStream_t stream);

/* The feature map alone (test and inspection aid), bf16 x [B][H][L][d]:
 * phi [B][H][L][r] fp32 and log_scale [B][H][L] fp32 such that the exact
 * feature is phi * exp(log_scale) (phi is the stabilised feature: for the
 * positive map the row maximum of phi is 1).  r follows feature_map; the trig
 * features come in the printed interleaved order.  is_key is accepted for
 * symmetry and does not change the result.  Returns favor_status_t. */
int favor_feature_map(const void *x, const float *omega, float *phi, float *log_scale, int B,
                      int H, int L, int d, int m, int feature_map, int is_key,
                      cudaStream_t stream);

/* Synchronises `stream`, returns and clears the device status word
 * (FAVOR_OK or FAVOR_ERR_TIMEOUT), or FAVOR_ERR_CUDA if the sync failed. */
int favor_get_device_status(cudaStream_t stream);

/* No counterpart on the pages: a check of the library's failure detection.
 * Launches one thread that waits, with the same bounded mbarrier wait the
 * pipelines use, for a barrier phase that nothing completes.  After
 * limit_cycles SM clock cycles (1 .. 2^31; 2^21 is about a millisecond) the
 * wait gives up and records FAVOR_ERR_TIMEOUT in the device status word, as a
 * stalled pipeline would; nothing faults, traps or hangs, and the context
 * stays usable.  favor_get_device_status(stream) then returns (and clears)
 * FAVOR_ERR_TIMEOUT.  Asynchronous on `stream`.  Returns FAVOR_OK,
 * FAVOR_ERR_INVALID_ARG for a limit out of range (before any CUDA call), or
 * FAVOR_ERR_CUDA. */
int favor_wait_expiry_check(long long limit_cycles, cudaStream_t stream);

/* Human-readable name of a favor_status_t value (static string). */
const char *favor_strerror(int status);

/* Frees the workspace of every device this process used (synchronises the
 * device first).  The next forward call re-allocates. */
void favor_release_workspace(void);

/* Number of feature columns r for a map, or -1 if the arguments are invalid. */
int favor_feature_dim(int feature_map, int d, int m);

/* ---- backward pass ----------------------------------------------------------
 * Gradients of a loss through the forward pass, given dout = dloss/dout
 * [B][H][L][dv] fp32 (the prefix sums of the Performer study notes, "Case 2",
 * accumulated in reverse for the keys and values):
 *   dnum_i = dout_i / den_i,  dden_i = -(dout_i . out_i) / den_i
 *   dphi(q_i) = S_i dnum_i + z_i dden_i
 *   dphi(k_j) = R_j v_j + rho_j,  dv_j = R_j^T phi(k_j),
 *   R_j = sum_{i >= j} phi(q_i) dnum_i^T,  rho_j = sum_{i >= j} phi(q_i) dden_i
 * (non-causal: all rows), then each feature map's derivative to dq and dk,
 * and to domega [H][m][d] summed over the batch.  Outputs dq, dk
 * [B][H][L][d], dv [B][H][L][dv] fp32; domega may be NULL (not computed; it
 * is never written for elu1 and relu).  No output may overlap an input or
 * another output.  fp32 SIMT kernels (out is recomputed, not passed in).
 * Asynchronous on `stream`; returns favor_status_t. */
int favor_attn_backward(const void *q, const void *k, const void *v, const float *omega,
                        const float *dout, float *dq, float *dk, float *dv, float *domega, int B, int H,
                        int L, int d, int dv_, int m, int causal, int feature_map, cudaStream_t stream);

/* Same with fp32 q/k/v. */
int favor_attn_backward_f32(const float *q, const float *k, const float *v, const float *omega,
                            const float *dout, float *dq, float *dk, float *dv, float *domega, int B,
                            int H, int L, int d, int dv_, int m, int causal, int feature_map,
                            cudaStream_t stream);

/* ---- carried state and the one-token decode step --------------------------
 * The causal form keeps running sums (Performer study notes, "Case 2"):
 *   S_i = S_{i-1} + phi(k_i) v_i^T,  z_i = z_{i-1} + phi(k_i),
 *   out_i = phi(q_i)^T S_i / phi(q_i)^T z_i,
 * so generation continues a prefix one token at a time at O(r d) per head.
 *
 * Decode state of one head (b, h): favor_state_floats() = r (dv + 2) fp32
 * values laid out as  S^ [r][dv] | z^ [r] | rho [r],  state buffer
 * [B][H][r (dv + 2)], 16-byte aligned, owned by the caller.  The carried sums
 * are S_f = S^_f 2^rho_f and z_f = z^_f 2^rho_f with phi the map above
 * (1/sqrt(m) included; trig features interleaved (sin, cos) per projection);
 * rho_f is a per-feature log2 reference that keeps every stored value in
 * fp32 range.  The empty state (no tokens) is S^ = z^ = 0, rho = -inf. */

/* Values per head of the decode state, r (dv + 2), or -1 if the arguments are
 * invalid. */
int favor_state_floats(int d, int dv, int m, int feature_map);

/* The decode state after the L keys of each head: k [B][H][L][d] and
 * v [B][H][L][dv] bf16 bits, omega as for the forward pass -> state.
 * L = 0 writes the empty state (k, v may then be NULL).  bf16 inputs run the
 * tensor-core state pass (fp16 features, fp32 sums) where the shape allows,
 * else fp32 SIMT kernels.  state must not overlap k, v or omega.
 * Asynchronous on `stream`; returns favor_status_t. */
int favor_attn_state(const void *k, const void *v, const float *omega, float *state, int B, int H,
                     int L, int d, int dv, int m, int feature_map, cudaStream_t stream);

/* Same with fp32 k/v, computed in fp32 SIMT kernels. */
int favor_attn_state_f32(const float *k, const float *v, const float *omega, float *state, int B,
                         int H, int L, int d, int dv, int m, int feature_map, cudaStream_t stream);

/* One decode step for every head: q, k [B][H][d] and v [B][H][dv] (bf16
 * bits) of the new token; state is read and updated in place (S += phi(k)
 * v^T, z += phi(k)), then out [B][H][dv] fp32 = phi(q)^T S / phi(q)^T z on
 * the updated state (the new token attends to itself, as in the causal
 * forward pass).  Supports r <= 1024.  out and state must not overlap each
 * other or an input.  fp32 SIMT arithmetic throughout (one thread-block
 * cluster per head).  Asynchronous on `stream`; returns favor_status_t. */
int favor_attn_decode(const void *q, const void *k, const void *v, const float *omega, float *state,
                      float *out, int B, int H, int d, int dv, int m, int feature_map,
                      cudaStream_t stream);

/* Same with fp32 q/k/v. */
int favor_attn_decode_f32(const float *q, const float *k, const float *v, const float *omega,
                          float *state, float *out, int B, int H, int d, int dv, int m,
                          int feature_map, cudaStream_t stream);

/* ---- random projections drawn on the device --------------------------------
 * omega [H][m][d] fp32 for the forward pass, drawn without a host round trip
 * (a redraw per step or per layer).  The pages draw w ~ N(0, I_d) ("Performer:
 * Unbiased Softmax Approximation") and name orthogonal random features as the
 * lower-variance variant (Performer study notes); the generator is fixed here
 * so that the draw is reproducible anywhere:
 *   Philox4x64-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2,
 *   3", SC 2011) under key (seed, 0); normal number e of stream s comes from
 *   the block at counter (e / 4, s, 0, 0) by Box-Muller on word pairs
 *   (x0, x1) and (x2, x3), u = (x / 2^11 + 1/2) 2^-53.
 *   kind 0 (iid):        omega[h][i][j] = normal (h m + i) d + j of stream 0.
 *   kind 1 (orthogonal): per head ceil(m/d) blocks; block b holds normals
 *     ((h nb + b) d + i) d + j of stream 0, its rows are orthonormalised by
 *     modified Gram-Schmidt in row order and row i is scaled by the norm of
 *     normals ((h nb + b) d + i) d + t, t < d, of stream 1; the last block is
 *     truncated.
 * Computed in fp64, rounded to fp32 once.  d in {32, 64, 128}, m >= 1,
 * H >= 1.  Asynchronous on `stream`; returns favor_status_t. */
int favor_draw_omega(float *omega, int H, int m, int d, int kind, unsigned long long seed,
                     cudaStream_t stream);

/* Measurement hook (no counterpart on the pages): while enabled, every
 * forward call records a CUDA event pair on its stream around its dominant
 * kernel (the causal scan, or the non-causal output kernel), and every
 * kernel launch of the library is counted.  favor_stats_enable(1) starts a
 * fresh recording, favor_stats_enable(0) stops it.  favor_stats_read()
 * synchronises the recorded events and reports the summed dominant-kernel
 * time (ms), the number of timed launches and the kernel launches counted
 * since recording started.  Host-side state, one recorder per process. */
typedef struct {
    double dominant_ms;
    int dominant_launches;
    long long kernel_launches;
    const char *dominant_kernel; /* name of the kernel the events bracket */
} favor_stats_t;
int favor_stats_enable(int enable);
int favor_stats_read(favor_stats_t *out);

/* Measurement hook, no counterpart on the pages: the exponential throughput
 * of the current device, the MUFU term of the roofline (the positive map
 * takes 2 m exponentials per token).  Launches one kernel in which every
 * thread of (SMs x 2048 / 256) blocks of 256 threads runs eight independent
 * chains of ex2.approx.ftz.f32 (the instruction the feature epilogues use),
 * times it with CUDA events on `stream`, and stores the rate in
 * *ex2_per_second (exponentials per second, whole device).  Synchronous:
 * it waits for the timing to finish.  Returns favor_status_t. */
int favor_probe_ex2_rate(double *ex2_per_second, cudaStream_t stream);

/* Test hook, no counterpart on the pages: the launch plan the tensor-core
 * path takes for a forward pass of this shape on a device of `sms` SMs,
 * computed on the host without touching a device.  plan[7] receives:
 *   [0] causal: scan segments per head; non-causal: key pieces per head
 *   [1] causal: piece states per segment
 *   [2] piece states per head (the state pass's pieces; 0 for a causal head
 *       of one segment)
 *   [3] CTAs of a cluster that split a head's features (1: whole heads)
 *   [4] value tiles of 64 columns
 *   [5] causal: CTAs of the scan; non-causal: CTAs of the persistent output
 *       kernel
 *   [6] CTAs of the state pass
 * Returns FAVOR_ERR_INVALID_ARG / FAVOR_ERR_UNSUPPORTED as favor_attn_forward
 * would for the shape, FAVOR_ERR_UNSUPPORTED as well for a shape the
 * tensor-core kernels do not take (favor_attn_forward then runs the fp32 SIMT
 * kernels), FAVOR_ERR_INVALID_ARG for a NULL plan or sms < 1. */
int favor_plan_info(int B, int H, int L, int d, int dv, int m, int causal, int feature_map, int sms, int *plan);

/* Test hook, no counterpart on the pages: the sine and cosine the
 * tensor-core kernels use for the sin/cos features (FAVOR_MAP_TRIG), on n
 * device values x[i] -> s[i], c[i] (fp32, device pointers, 16-byte aligned,
 * not overlapping).  The argument is reduced by 2 pi in three parts
 * (Cody-Waite: n = rint(x / 2 pi), then x - n p1 - n p2 - n p3 with p1 holding
 * 8 significant bits, so n p1 is exact for |n| < 2^16) and the fast sincos of the remainder
 * in [-pi, pi] follows.  Asynchronous on `stream`.  Returns favor_status_t. */
int favor_check_sincos(const float *x, float *s, float *c, int n, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FAVOR_H */
