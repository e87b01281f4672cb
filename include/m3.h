/*
 * m3 -- Mamba-3 SSM layer recurrence on NVIDIA B300 (sm_103a).
 *
 * C ABI of libm3.so.  All tensor arguments are DEVICE pointers owned by the
 * caller; the library never allocates or frees device memory and never
 * synchronises.  Every call is validated on the host first; on any violation
 * it returns an error code and launches nothing.  Work is enqueued on the
 * given stream (a cudaStream_t passed as void*; NULL = the legacy default
 * stream); a launch failure is returned as M3_ERR_CUDA, execution errors show
 * up at the caller's next synchronisation.
 *
 * What is computed follows "Mamba-3: Improved Sequence Modeling using State
 * Space Principles" (abhik.ai/papers/mamba3; thelatestinai.com/papers/2603.15569):
 *
 *   alpha_t = exp(dt_t A_h), beta_t = (1 - lambda_t) dt_t alpha_t, gamma_t = lambda_t dt_t
 *                                       (Proposition 1, Eq. 6; Table 1)
 *   h_t = R(phi_t) (alpha_t h_{t-1} + beta_t B_{t-1} X_{t-1}^T) + gamma_t B_t X_t^T
 *   Y_t = h_t^T C_t                     (section 3.3, Eqs. 12-14: MIMO rank R)
 *
 * where h_t is the N x P state of one (batch, head), phi_{t,j} = dt_t omega_{t,j}
 * rotates state pair j = rows (2j, 2j+1) counter-clockwise (Propositions 2-4,
 * Eq. 11: the complex state realised as data-dependent rotary), and
 * R(theta)(a, b) = (a cos theta - b sin theta, a sin theta + b cos theta).
 * lambda_t = 1 is Mamba-2's exponential-Euler update.
 *
 * Layouts (row-major, contiguous, time-major):
 *   x, y          [batch, T, H, R, P]   io dtype
 *   B, C          [batch, T, H, R, N]   io dtype
 *   dt, lambda    [batch, T, H]         fp32  (dt >= 0, lambda in [0,1])
 *   A             [H]                   fp32  (A <= 0)
 *   omega         [batch, T, H, N/2]    fp32
 *   state         [batch, H, N, P]      fp32, physical (unrotated) frame
 * The preconditions dt >= 0, A <= 0, 0 <= lambda <= 1 are documented, not
 * checked per element.
 *
 * io dtype: M3_DTYPE_BF16 (inputs bf16, fp32 accumulation, bf16 y) or
 * M3_DTYPE_F32 (fp32 everywhere).  Every pointer must be 16-byte aligned.
 */
#ifndef M3_H
#define M3_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define M3_API __attribute__((visibility("default")))
#else
#define M3_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    M3_OK = 0,
    M3_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad size or dtype */
    M3_ERR_UNSUPPORTED = -2,   /* valid arguments outside what the kernels implement */
    M3_ERR_WORKSPACE = -3,     /* workspace missing or smaller than *_workspace_size */
    M3_ERR_CUDA = -4,          /* a CUDA call or kernel launch failed */
    M3_ERR_TIMEOUT = -5        /* a bounded device-side wait gave up */
} m3_status;

typedef enum { M3_DTYPE_BF16 = 0, M3_DTYPE_F32 = 1 } m3_dtype;

/* Human-readable name of a status code (static string, never NULL). */
M3_API const char* m3_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
M3_API int m3_version(void);

/*
 * Bytes of device workspace m3_scan_fwd needs for these sizes (0 if none).
 * Returns 0 too for sizes m3_scan_fwd would reject; call it to size the
 * buffer, then pass the buffer and this size.
 */
M3_API size_t m3_scan_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                  int64_t dstate, int R, int chunk, int io_dtype);

/*
 * How m3_scan_fwd would run for these sizes, without running it.
 *   path      out: 0 = CUDA-core kernels (fp32 arithmetic; the fp32 io mode
 *             and the fallback), 1 = tensor-core kernels (bf16 MMA with
 *             fp32 accumulation)
 *   launches  out: number of kernel launches one m3_scan_fwd call makes
 *             (besides a 4-byte memset of the workspace's status word)
 * Returns M3_OK, or the error m3_scan_fwd would return for these sizes.
 */
M3_API int m3_scan_fwd_plan(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                            int R, int chunk, int io_dtype, int* path, int* launches);

/*
 * Chunked parallel prefill over T = seqlen tokens from a zero state
 * (h_{-1} = 0 and no delayed write before the first token, as in the
 * page's scalar scan helper, panel 1).
 *
 *   x, B, C, dt, A, lambda, omega : inputs, layouts above
 *   R        MIMO rank, one of 1, 2, 4, 8
 *   chunk    tokens per chunk Q of the chunked algorithm (section 3.3):
 *            intra-chunk masked scores (decay x two-band mask, Eq. 7)
 *            plus inter-chunk state passing; 16 <= chunk <= 256 and a
 *            multiple of 16.  The result does not depend on it beyond rounding.
 *            The tensor-core path runs every chunk as sub-chunks of 64 / R
 *            tokens (64-row score tiles), the MIMO chunk-length reduction of
 *            section 3.3 taken to one tile shape.  With at most 148 (batch, head)
 *            sequences (half the 296 CTA slots of a B300) it also cuts every
 *            sequence at the same places into at most 296 / sequences segments
 *            (a state pass, the segment scan of m3_state_passing, a full pass:
 *            3 launches).
 *   y        out [batch, T, H, R, P], io dtype
 *   final_state  out (nullable) [batch, H, N, P] fp32: h_{T-1}, the state a
 *            decode step continues from (its delayed-write cache is
 *            B_{T-1}, X_{T-1}, taken by the caller from B and x).
 *   Sizes: batch >= 0, seqlen >= 0 (0 writes nothing except a zero
 *   final_state), nheads >= 1, dstate N even with 2 <= N <= 256,
 *   headdim P a multiple of 4 with 4 <= P <= 256.
 *   workspace / workspace_bytes: device scratch of at least
 *   m3_scan_fwd_workspace_size(...) bytes, 256-byte aligned; contents on
 *   entry are ignored.  On the tensor-core path (m3_scan_fwd_plan path 1)
 *   the first int of the workspace is the call's device status once the
 *   stream's work is done: M3_OK, or M3_ERR_TIMEOUT when a bounded wait in
 *   the kernel gave up (y and final_state are then not valid).
 * Returns M3_OK or an error code; launches nothing on error.
 */
M3_API int m3_scan_fwd(const void* x, const void* B, const void* C, const float* dt, const float* A,
                const float* lambda, const float* omega, int R, int chunk,
                void* y, float* final_state,
                int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                int io_dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of the fixed scratch array behind m3_scan_fwd_noalloc (16 MiB). */
#define M3_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * m3_scan_fwd for callers that cannot allocate device memory.  The paper has
 * no counterpart: this is a library convenience, not part of the method.
 *
 * Some callers cannot call cudaMalloc or hand the library a workspace: an
 * application that owns every device allocation and passes only inputs and
 * outputs, a serving loop that forbids allocation once it runs, a plugin
 * host with no allocator callback.  This entry point takes the arguments of
 * m3_scan_fwd minus the workspace and computes the same result, using a fixed
 * scratch array of M3_NOALLOC_SCRATCH_BYTES that is part of the library's
 * device image (every GPU that loads the library keeps it reserved until the
 * process exits).  It allocates nothing.
 *
 *   - Sizes whose workspace (m3_scan_fwd_workspace_size) exceeds
 *     M3_NOALLOC_SCRATCH_BYTES return M3_ERR_WORKSPACE and launch nothing;
 *     other errors are those of m3_scan_fwd.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents (each call clears what must start at zero).  Calls that
 *     overlap on the GPU -- on different streams or from different host
 *     threads -- race on it: serialise them.
 *   - The tensor-core kernels record a timeout of their bounded waits in the
 *     array's first word, which the caller cannot reach: m3_device_status
 *     reports it (for the most recent call on the current device).
 *   - The address is cached per device with the unique id of the context it
 *     was looked up in, so a call after cudaDeviceReset (a new primary
 *     context) looks it up again.
 */
M3_API int m3_scan_fwd_noalloc(const void* x, const void* B, const void* C, const float* dt, const float* A,
                               const float* lambda, const float* omega, int R, int chunk,
                               void* y, float* final_state,
                               int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                               int io_dtype, void* stream);

/*
 * One decode token for every (batch, head): the recurrence above with T = 1
 * from a carried state (the single-token mode of section 3.3 / Table 6).
 *
 *   state          in/out [batch, H, N, P] fp32, physical frame
 *   x_t            [batch, H, R, P] io dtype
 *   B_t, C_t       [batch, H, R, N] io dtype
 *   B_prev_x_prev  in/out [batch, H, R*N + R*P] io dtype: the factors of the
 *                  previous token's write, B_{t-1} as [R, N] then X_{t-1} as
 *                  [R, P], unrotated; overwritten with B_t, X_t.  Zero for a
 *                  sequence's first token; after m3_scan_fwd, B[:, T-1] and
 *                  x[:, T-1].
 *   dt_t, lambda_t [batch, H] fp32;  A [H] fp32;  omega_t [batch, H, N/2] fp32
 *   y_t            out [batch, H, R, P] io dtype
 *   Sizes as for m3_scan_fwd; batch may be 0 (nothing is launched).
 * state and B_prev_x_prev must not overlap any other argument.
 */
M3_API int m3_decode_step(float* state, const void* x_t, const void* B_t, void* B_prev_x_prev,
                   const void* C_t, const float* dt_t, const float* A, const float* lambda_t,
                   const float* omega_t, void* y_t,
                   int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate, int R,
                   int io_dtype, void* stream);

/*
 * Pre-SSM options of the _prep entry points.  All pointers are device
 * pointers, nullable, 16-byte aligned; a NULL params pointer means all off.
 *
 *   dt_bias  [H] fp32: Delta_t = softplus(dt_raw_t + dt_bias[h]) (NULL = 0)
 *   bc_norm  nonzero: every (token, rank) row v of B and of C is RMS-normalised
 *            over the N channels, v / sqrt(mean(v^2) + bc_eps) * gain, before
 *            the rotation (the BC normalisation of section 3.4)
 *   bc_eps   >= 0, added to the mean square
 *   B_gain, C_gain  [N] fp32 per-channel gains of the normalisation (NULL = 1;
 *            unused without bc_norm)
 *   B_bias, C_bias  [H, R, N] fp32 head-specific channel biases added after the
 *            normalisation (or to the raw rows without it) (NULL = 0)
 *   z        y's layout and io dtype (prefill [batch, T, H, R, P], decode
 *            [batch, H, R, P]), nullable: the output gate y <- y * silu(z),
 *            silu(z) = z / (1 + e^-z), applied in the kernels' epilogues (the
 *            SSM+Gate fusion of Tables 11-12; the pages give no gate formula,
 *            this is the Mamba family's)
 */
typedef struct m3_prep_params {
    const float* dt_bias;
    int bc_norm;
    float bc_eps;
    const float* B_gain;
    const float* C_gain;
    const float* B_bias;
    const float* C_bias;
    const void* z;
} m3_prep_params;

/*
 * Per-token parameters from their pre-activations.  The time-varying
 * discretizations of Table 1 ("Mamba-3: Improved Sequence Modeling using
 * State Space Principles") take a decay generator per token, alpha_t =
 * exp(Delta_t A_t), and the default parameterisation of lambda in the
 * appendix ablation table is lambda_t = sigmoid(u_t).  These entry points take
 *
 *   dt_raw   [batch, T, H] fp32: Delta_t = softplus(dt_raw_t + dt_bias[h])
 *            (softplus(z) = log(1 + e^z); the pages leave Delta's
 *            parameterisation open, this is the Mamba family's)
 *   A        [batch, T, H] fp32: A_t <= 0, one per token
 *   u        [batch, T, H] fp32: lambda_t = sigmoid(u_t) = 1 / (1 + e^-u_t)
 *   params   the options above (dt_bias, B / C normalisation and biases)
 *
 * and otherwise behave exactly as m3_scan_fwd / m3_decode_step (same
 * layouts, sizes, errors and stream semantics).  The delayed-write cache of
 * the decode step keeps the raw B_{t-1}, X_{t-1}; both B_t and B_{t-1} are
 * normalised and biased inside the step.  The tensor-core prefill and the
 * decode kernels apply softplus, sigmoid, the normalisation and the biases to
 * the staged values inside the kernel; the CUDA-core prefill first writes
 * Delta, lambda and the inverse RMS of every B / C row to the workspace.
 * Workspace: m3_scan_fwd_prep_workspace_size bytes (at least
 * m3_scan_fwd_workspace_size; larger on the CUDA-core path).  Errors: as
 * m3_scan_fwd, and M3_ERR_INVALID_ARG for a misaligned pointer inside params or
 * bc_eps < 0.  The params struct itself is read on the host: it needs only
 * its natural alignment; the device pointers inside it must be 16-byte aligned.
 */
M3_API size_t m3_scan_fwd_prep_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                              int64_t dstate, int R, int chunk, int io_dtype);
M3_API int m3_scan_fwd_prep(const void* x, const void* B, const void* C, const float* dt_raw, const float* A,
                            const float* u, const float* omega, int R, int chunk, void* y, float* final_state,
                            int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                            int io_dtype, const m3_prep_params* params, void* workspace, size_t workspace_bytes,
                            void* stream);
/* Decode on pre-activations: dt_raw_t, A_t, u_t [batch, H] fp32. */
M3_API int m3_decode_step_prep(float* state, const void* x_t, const void* B_t, void* B_prev_x_prev,
                               const void* C_t, const float* dt_raw_t, const float* A_t, const float* u_t,
                               const float* omega_t, void* y_t, int64_t batch, int64_t nheads, int64_t headdim,
                               int64_t dstate, int R, int io_dtype, const m3_prep_params* params, void* stream);

/*
 * Backward pass of m3_scan_fwd (training): the gradients of a loss L with
 * respect to every input, given dy = dL/dy and d_final = dL/d final_state.
 * The adjoint of the recurrence runs backwards in time (dL/dh_t =
 * C_t dy_t^T + alpha_{t+1} R(phi_{t+1})^T dL/dh_{t+1}), with the chain rule
 * through Eq. 6's alpha, beta, gamma and the angle phi = Delta omega; the
 * chunked algorithm's backward is the use of section 3.3 for training.
 *
 *   x, B, C, dt, A, lambda, omega, R, sizes, io_dtype: as m3_scan_fwd
 *   dy        [batch, T, H, R, P] io dtype
 *   d_final   [batch, H, N, P] fp32, nullable (= 0)
 *   dx        out [batch, T, H, R, P] fp32;  dB, dC  out [batch, T, H, R, N] fp32
 *   ddt, dlambda  out [batch, T, H] fp32;  domega  out [batch, T, H, N/2] fp32
 *   dA        out [H] fp32 (summed over batch and tokens)
 *   workspace: m3_scan_bwd_workspace_size bytes, 256-byte aligned: the
 *            state entering every chunk of Q tokens (Q = 8 for R <= 2,
 *            4 for R >= 4; batch * H * ceil(T/Q) * N * P fp32)
 *            and per-pair-block partial sums of dx and of four per-token
 *            scalars (fp32).
 * CUDA cores, one CTA per (batch, head, block of state pairs): a forward
 * sweep stores the chunk checkpoints; the reverse sweep recomputes each
 * chunk's states from its checkpoint and runs the adjoint from the last token
 * to the first; a finishing kernel adds the pair blocks' partial sums and
 * applies the chain rule for dt, lambda and A.  dA is accumulated with
 * atomics, so its last bits may differ between runs; every other output is
 * deterministic.  Sizes: R in {1, 2, 4, 8}; P in {4, 8, 16, 32, 64, 128};
 * N even, <= 256; otherwise M3_ERR_UNSUPPORTED.  Errors as m3_scan_fwd.
 */
M3_API size_t m3_scan_bwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                         int64_t dstate, int R, int io_dtype);
M3_API int m3_scan_bwd(const void* x, const void* B, const void* C, const float* dt, const float* A,
                       const float* lambda, const float* omega, int R, const void* dy, const float* d_final,
                       float* dx, float* dB, float* dC, float* ddt, float* dA, float* dlambda, float* domega,
                       int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                       int io_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass of m3_scan_fwd_prep:
 * the gradients with respect to the pre-activations of Delta_t =
 * softplus(dt_raw_t + dt_bias_h) and lambda_t = sigmoid(u_t), and to the
 * per-token decay generators A_t (Table 1's time-varying discretisations).
 *
 *   x, B, C, omega, R, sizes, io_dtype, dy, d_final: as m3_scan_bwd
 *   dt_raw, A, u   [batch, T, H] fp32 (A one value per token, as in
 *                  m3_scan_fwd_prep)
 *   params         nullable; as m3_scan_fwd_prep (dt_bias, the B/C
 *                  normalisation with its gains and biases, the gate's z)
 *   dx, dB, dC, domega  out, as m3_scan_bwd
 *   ddt_raw, dA, du     out [batch, T, H] fp32
 *   ddt_bias       nullable out [H] fp32: sum over batch and tokens of ddt_raw
 *                  (accumulated with atomics)
 *   dz             out [batch, T, H, R, P] fp32 when params->z is set (the
 *                  output gate y = y_pre * SiLU(z)), else unused
 *   dB_gain, dC_gain  nullable out [N] fp32; dB_bias, dC_bias  nullable out
 *                  [H, R, N] fp32: the B/C normalisation's parameters (sums
 *                  over rows by atomics); dB, dC are then the raw rows'
 *                  gradients (through v -> v r gain + bias, r = rsqrt(mean(v^2)
 *                  + eps)).  With bf16 io, or together with the gate, the
 *                  adjoint runs in fp32 on fp32 copies of x, of the seed
 *                  dy * SiLU(z) and of the normalised rows, so that nothing it
 *                  reads is rounded to bf16 beyond the inputs themselves
 *   workspace: m3_scan_bwd_prep_workspace_size bytes, 256-byte aligned, an
 *            upper bound over the options params may select: m3_scan_bwd's
 *            (fp32 layout where the B/C normalisation's fp32 copies need it),
 *            Delta and lambda (2 * batch * T * H fp32), the normalised B and C
 *            rows and their inverse RMS, the fp32 copies of x and of the seed,
 *            and, where the forward entry supports the shape, the ungated
 *            output y_pre (io dtype, y's layout) and m3_scan_fwd_prep's
 *            workspace.
 * Delta and lambda are derived with the forward entry's own functions; the
 * derivative of softplus is sigmoid, that of sigmoid is lambda (1 - lambda).
 * With the gate, the seed of the recurrence is dy * SiLU(z) (fp32, inside the
 * kernel) and dz = dy * y_pre * SiLU'(z), y_pre written by m3_scan_fwd_prep
 * without the gate (chunk 64) in the io dtype; shapes that entry does not
 * take give M3_ERR_UNSUPPORTED.  Sizes and errors as m3_scan_bwd.
 */
M3_API size_t m3_scan_bwd_prep_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                              int64_t dstate, int R, int io_dtype);
M3_API int m3_scan_bwd_prep(const void* x, const void* B, const void* C, const float* dt_raw, const float* A,
                            const float* u, const float* omega, int R, const void* dy, const float* d_final,
                            float* dx, float* dB, float* dC, float* ddt_raw, float* dA, float* du, float* domega,
                            float* ddt_bias, float* dz, float* dB_gain, float* dC_gain, float* dB_bias,
                            float* dC_bias, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                            int64_t dstate, int io_dtype, const m3_prep_params* params, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Device-side error words of the calls that take no workspace, on the
 * current device: M3_OK, or M3_ERR_TIMEOUT once a bounded wait inside a
 * decode kernel (sticky across calls) or inside the most recent
 * m3_scan_fwd_noalloc call's tensor-core kernels gave up (the outputs of that
 * call are then not valid).  It first synchronises the current device
 * (cudaDeviceSynchronize), so every stream's work is finished when the words
 * are read; clear != 0 resets them to M3_OK afterwards.  Returns M3_OK,
 * M3_ERR_TIMEOUT, or M3_ERR_CUDA if the device could not be synchronised or
 * read.  m3_scan_fwd callers read the first int of their workspace instead.
 */
M3_API int m3_device_status(int clear);

/*
 * Failure injection for tests.  The paper has no counterpart: this exercises
 * the library's own error paths without faulting or hanging a GPU.
 *
 *   what = M3_TEST_LAUNCH_FAILURE: the next `count` calls of entry points
 *          that would launch work return M3_ERR_CUDA after their argument
 *          checks and launch nothing (a launch failure made on the host).
 *          Calls rejected by their checks, or with nothing to launch, do not
 *          use one up.  Returns how many were still armed before this call.
 *   what = M3_TEST_PREFILL_TIMEOUT: the next plain m3_scan_fwd (or
 *          m3_scan_fwd_noalloc) call that takes the tensor-core path with
 *          N = 128, R = 1, chunk 64 runs a test instantiation of its kernel in
 *          which every CTA's consumer warps, at their local chunk `count`, wait
 *          with a 50 us limit on an mbarrier that nothing completes.  The
 *          bounded-wait failure path then runs for real: both warp groups give
 *          up, the copies and MMAs in flight are drained (each with the
 *          normal 2 s limit), TMEM is freed and M3_ERR_TIMEOUT is written to the
 *          status word (the workspace's first int; m3_device_status for the
 *          noalloc entry).  That call's y and final_state are not valid; the
 *          next call is normal.  Returns the chunk previously armed, or -1.
 *   what = 0: disarm both; returns 0.
 * Returns M3_ERR_INVALID_ARG for another `what` or a negative count.
 */
#define M3_TEST_LAUNCH_FAILURE 1
#define M3_TEST_PREFILL_TIMEOUT 2
M3_API int m3_test_inject(int what, int count);

/*
 * Inter-chunk state passing of the chunked algorithm (the chunked parallel
 * form of "Mamba-3: Improved Sequence Modeling using State Space Principles",
 * section 3.3, applied to the recurrence of Proposition 1 / Eq. 6 with the
 * rotary form of Propositions 3-4), in place:
 *
 *   H_c = exp(l_c) R(Theta_c) H_{c-1} + U_c,   c = 0 .. nchunks-1,
 *
 * with H_{-1} = init_state (zero if NULL) and R(Theta_c) rotating state rows
 * (2j, 2j+1) by Theta_c[j].  l_c is a chunk's summed log-decay
 * (sum of dt_t A) and Theta_c its summed rotation angle per pair.
 *
 *   chunk_states    in/out [batch, H, nchunks, N, P] fp32: in = U_c (a
 *                   chunk's own contribution), out = H_{c-1} (the state
 *                   entering chunk c)
 *   chunk_logdecay  [batch, H, nchunks] fp32
 *   chunk_angle     [batch, H, nchunks, N/2] fp32
 *   init_state      nullable [batch, H, N, P] fp32
 *   final_state     nullable out [batch, H, N, P] fp32: H_{nchunks-1}
 *   Sizes: N even, 2 <= N <= 256; P a multiple of 4, 4 <= P <= 256;
 *   nchunks >= 0 (0 copies init_state, or zeros, to final_state).
 */
M3_API int m3_state_passing(float* chunk_states, const float* chunk_logdecay, const float* chunk_angle,
                     const float* init_state, float* final_state,
                     int64_t batch, int64_t nheads, int64_t nchunks, int64_t dstate, int64_t headdim,
                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* M3_H */
