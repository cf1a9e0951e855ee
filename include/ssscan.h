/*
 * ssscan.h -- C ABI of the B300 (sm_103a) selective-scan library.
 *
 * The two scans and what sits around them, all asynchronous on the caller's
 * CUDA stream:
 *
 *   ss_selective_scan_fwd        the Mamba (Mamba-1) selective scan
 *   ss_ssd_chunk_scan_fwd        the Mamba-2 SSD scan in chunked form
 *   ss_selective_scan_fwd_init,  the same, continuing from a given state
 *   ss_ssd_chunk_scan_fwd_init
 *   ss_conv_selective_scan_fwd   the causal conv1d + SiLU fused in front
 *   ss_selective_scan_bwd        the selective scan's gradients
 *   ss_selective_scan_fwd_ckpt,  a training step's forward / backward that
 *   ss_selective_scan_bwd_ckpt   share the states every 8 steps
 *   ss_selective_state_update,   one decode step of either model
 *   ss_ssd_state_update
 *   ss_selective_scan_fwd_host   the selective scan from host buffers
 *   ss_ssd_chunk_scan_fwd_host   the SSD scan from host buffers
 *   ss_selective_scan_fwd_noalloc the selective scan with no allocation
 *   ss_status_string, ss_get_device_error, ss_launch_count, ss_version,
 *   ss_selftest_timeout,         status, errors and diagnostics
 *   ss_debug_set_path, ss_probe_ex2_rate, ss_probe_scan_forms
 *
 * Every buffer is caller-owned device memory described by an ss_tensor
 * (pointer, dtype, shape, strides in elements).  The library keeps no pointer
 * after a call returns, never synchronises the stream, and allocates only the
 * stream-ordered scratch documented per call.  Optional inputs are passed as
 * NULL.  Calls return SS_OK (0) or a negative status; ss_status_string()
 * names it.  An argument error is detected on the host before anything is
 * launched.  Errors found on the device (a bounded wait that ran out) are
 * recorded in a per-device error word that ss_get_device_error() reads.
 */
#ifndef SSSCAN_H
#define SSSCAN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define SS_OK 0
#define SS_ERR_INVALID_ARG (-1)  /* NULL where required, bad flag, bad chunk  */
#define SS_ERR_SHAPE (-2)        /* shapes disagree with each other           */
#define SS_ERR_DTYPE (-3)        /* unsupported or mixed dtypes               */
#define SS_ERR_ALIGNMENT (-4)    /* pointer not aligned to its element size   */
#define SS_ERR_UNSUPPORTED (-5)  /* valid but outside what is compiled (N)    */
#define SS_ERR_ALLOC (-6)        /* stream-ordered scratch allocation failed  */
#define SS_ERR_LAUNCH (-7)       /* kernel launch failed                      */
#define SS_ERR_TIMEOUT (-8)      /* a device-side bounded wait ran out        */
#define SS_ERR_CUDA (-9)         /* other CUDA runtime error                  */

/* ---- tensors ----------------------------------------------------------- */
#define SS_F32 0
#define SS_BF16 1

typedef struct ss_tensor {
    void* data;         /* device pointer (caller-owned)                 */
    int32_t dtype;      /* SS_F32 or SS_BF16                             */
    int32_t ndim;       /* number of used entries in shape / stride       */
    int64_t shape[4];
    int64_t stride[4];  /* in elements; any non-negative values           */
} ss_tensor;

/*
 * Selective scan, forward.
 *
 * Defines (page "Mamba模型笔记", §2.2 discrete recurrence, §4.1 input-dependent
 * B, C and Delta, §4.3 gate branch, §4.4 one SSM per channel; page 0539edu
 * paper talk §2.3 discretisation Abar = exp(Delta A), Bbar = Delta B,
 * Delta > 0 through softplus), for every batch row b, channel d and step t:
 *
 *   dl        = delta[b,d,t] + delta_bias[d]        (bias optional)
 *   dl        = softplus(dl) = log(1 + e^dl)        (if softplus != 0)
 *   h[n]      = exp(dl * A[d,n]) * h[n] + dl * B[b,n,t] * u[b,d,t],  h = 0 at t = 0
 *   out       = sum_n C[b,n,t] * h[n] + D[d] * u[b,d,t]               (D optional)
 *   y[b,d,t]  = out * z * sigmoid(z),  z = z[b,d,t]                   (z optional)
 *   last_state[b,d,n] = h[n] after the last step                      (optional)
 *
 * Shapes (element strides free unless noted):
 *   u, delta, z, y : (Bsz, D, L)        dtype T (all four the same)
 *   A              : (D, N)             f32
 *   B, C           : (Bsz, N, L)        dtype T; shared by all channels of row b
 *               or   (Bsz, G, N, L)     dtype T; one B, C per group of D/G
 *                                       consecutive channels (channel d reads
 *                                       group d / (D/G)); G = D is one B, C
 *                                       per channel.  D % G must be 0.
 *   D, delta_bias  : (D)                f32
 *   last_state     : (Bsz, D, N)        f32
 * T is SS_F32 or SS_BF16.  N <= 256; the fast paths are compiled for N = 16
 * and, with B, C shared by a whole batch row, for N = 32, 64 and 128 (bf16;
 * fp32 too for 64 and 128); other N run a slower general kernel.  The fast
 * paths need unit stride in t and 16-byte aligned rows for u/delta/z/y/B/C;
 * grouped B, C (N = 16) with groups of at least 64 channels (a multiple of
 * 64) share the shared-B, C kernel, smaller groups run a kernel that streams
 * each channel's own B, C.  A call with unit t-strides whose row pitch or
 * base is not a multiple of 16 bytes (an odd L in bf16, L not a multiple of
 * 4 in fp32) is run on padded copies: u, delta, z, B, C go into
 * stream-ordered scratch with 16-byte row pitch (one copy launch), the fast
 * path scans them and y is copied back (one more launch), about twice the
 * scan's own DRAM traffic.  Other layouts, and padded copies that do not fit
 * in device memory, take the general kernel (same results up to rounding
 * order).  y may not alias an input.
 * Arithmetic: fp32 state and accumulation for both dtypes.
 *
 * Scratch: when the channel count is too small to fill the GPU, the
 * sequence is split into segments scanned in parallel (a summary pass, then
 * the main pass seeded with each segment's incoming state); the summaries
 * live in stream-ordered memory (cudaMallocAsync / cudaFreeAsync on
 * `stream`), at most 2 * Bsz * D * N * 64 floats.  The padded copies above
 * take the same kind of memory, (3 or 4) * Bsz * D + 2 * Bsz * G * N rows of
 * the padded length.
 *
 * Zero-size inputs (Bsz, D or L = 0) return SS_OK without a launch.
 * `stream` is a cudaStream_t (NULL = legacy default stream).
 */
int ss_selective_scan_fwd(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                          const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                          const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                          ss_tensor* y, ss_tensor* last_state, void* stream);

/*
 * Allocation-free selective scan.  The pages have no counterpart to this
 * call: it is a deployment variant of ss_selective_scan_fwd for callers that
 * cannot allocate device memory while a call runs -- code whose allocator is
 * owned by another runtime or arena, loops that must not enter the CUDA
 * allocator (its locks and its implicit synchronisation), or processes that
 * have handed all free device memory to a pool.
 *
 * Same arguments, checks and status codes as ss_selective_scan_fwd, and the
 * same results up to rounding, except where the segment summaries live:
 * instead of stream-ordered memory they use one fixed 4 MiB array in device
 * memory, defined in the library and held by every GPU that loads it until
 * the process exits.  The call makes no cudaMalloc / cudaMallocAsync /
 * cudaFree and no allocating library call.
 *   - The number of time segments is capped so that the summaries fit the
 *     array: where ss_selective_scan_fwd would use more (long sequences over
 *     few channels, e.g. 1 x 2048 x 262144 at N = 16 takes 17 segments here
 *     instead of 28), the segments are longer and the call can be slower, and
 *     the summation order (hence the rounding) differs.
 *   - SS_ERR_UNSUPPORTED is returned, before anything is launched, only if a
 *     request still exceeded the array.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the array and it keeps the last call's
 *     contents; the summary pass writes every entry the main pass reads, so
 *     nothing needs clearing.  Calls whose kernels overlap on the GPU (other
 *     streams, other threads) race on the array: serialise them.
 */
int ss_selective_scan_fwd_noalloc(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                                  const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                                  const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                                  ss_tensor* y, ss_tensor* last_state, void* stream);

/*
 * Mamba-2 SSD scan, forward, chunked.
 *
 * Defines (page "Mamba模型笔记" §5, SSD; state-spaces/mamba README §4.3,
 * Mamba-2 with d_state 64 or 128 and a scalar A per head; skill card, Mamba-2
 * config headdim / ngroups), for every batch row b and head h, with group
 * g = h / (H / G):
 *
 *   a         = exp(dt[b,t,h] * A_head[h])
 *   S[p][n]   = a * S[p][n] + dt[b,t,h] * x[b,t,h,p] * B[b,t,g,n],  S = 0 at t = 0
 *   y[b,t,h,p]= sum_n C[b,t,g,n] * S[p][n] + D[h] * x[b,t,h,p]       (D optional)
 *   last_state[b,h,p,n] = S[p][n] after the last step                 (optional)
 *
 * computed chunk by chunk: within a chunk of `chunk` steps through the
 * quadratic (attention-like) form (C B^T masked by the decays) times x, and
 * across chunks through the carried state.  The result does not depend on
 * `chunk` beyond rounding.
 *
 * Shapes:
 *   x, y       : (Bsz, L, H, P)    dtype T
 *   dt         : (Bsz, L, H)       dtype T, already positive (no bias, no softplus)
 *   A_head, D  : (H)               f32
 *   B, C       : (Bsz, L, G, N)    dtype T, H % G == 0
 *   last_state : (Bsz, H, P, N)    f32
 * chunk must be one of 64, 128, 256 (else SS_ERR_INVALID_ARG), but it does
 * not change the computation: the tensor-core kernels always work in blocks
 * of 128 steps (the largest diagonal block whose C B^T tile and decay matrix
 * fit one SM's tensor memory next to the state), and the CUDA-core kernel
 * steps through time one step at a time.  The chunked form's result does not
 * depend on the chunk length beyond rounding, so every accepted value gives
 * the same result.  N <= 256, P <= 256.  The tensor-core path is compiled for
 * bf16 with P = 64, N = 128, unit inner strides and 16-byte aligned rows
 * (dt's t-stride a multiple of 8 elements).  A dt whose head stride is 1 but
 * whose t-stride is not a multiple of 8 (H not a multiple of 8, contiguous)
 * is copied into stream-ordered scratch at a pitch of H rounded up to 8 (one
 * small copy launch) and takes the tensor-core path; everything else runs the
 * general CUDA-core kernel.  Zero-size inputs return SS_OK without a launch.
 */
int ss_ssd_chunk_scan_fwd(const ss_tensor* x, const ss_tensor* dt, const ss_tensor* A_head,
                          const ss_tensor* B, const ss_tensor* C, const ss_tensor* D, int chunk,
                          ss_tensor* y, ss_tensor* last_state, void* stream);

/*
 * Scans that continue from a given state (page 0539edu paper talk §5.3: split
 * a long text into chunks and pass the state across; §4.3: generation keeps
 * only the fixed-size state).  Same arguments and results as the calls above
 * plus `initial_state`, the state entering step 0 (NULL = zero):
 *   ss_selective_scan_fwd_init : initial_state (Bsz, D, N) f32
 *   ss_ssd_chunk_scan_fwd_init : initial_state (Bsz, H, P, N) f32
 * Running [0, L1) and then [L1, L) from the first call's last_state gives the
 * result of one call over [0, L) up to rounding.  initial_state and
 * last_state must not overlap.
 */
int ss_selective_scan_fwd_init(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                               const ss_tensor* initial_state, ss_tensor* y,
                               ss_tensor* last_state, void* stream);
int ss_ssd_chunk_scan_fwd_init(const ss_tensor* x, const ss_tensor* dt, const ss_tensor* A_head,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               int chunk, const ss_tensor* initial_state, ss_tensor* y,
                               ss_tensor* last_state, void* stream);

/*
 * The conv branch feeding the scan, fused: u = silu(causal_conv1d(x)) is
 * computed on chip and never written to memory, then scanned as in
 * ss_selective_scan_fwd (page "Mamba模型笔记" §4.3: the SSM branch passes a
 * local convolution first; 0539edu paper talk §3.1: causal-conv1d, width
 * d_conv = 4).  For every b, d, t:
 *   u[b,d,t] = silu(conv_bias[d] + sum_{k<W} conv_weight[d,k] * x[b,d,t-W+1+k])
 * with x = 0 before t = 0.  x (Bsz, D, L) has the dtype and layout rules of u;
 * conv_weight (D, W) f32 with 1 <= W <= 4; conv_bias (D) f32 or NULL.  The
 * other arguments are those of ss_selective_scan_fwd; the D skip and the gate
 * use u.  Starts from a zero state and zero conv history.
 */
int ss_conv_selective_scan_fwd(const ss_tensor* x, const ss_tensor* conv_weight,
                               const ss_tensor* conv_bias, const ss_tensor* delta,
                               const ss_tensor* A, const ss_tensor* B, const ss_tensor* C,
                               const ss_tensor* D, const ss_tensor* z,
                               const ss_tensor* delta_bias, int softplus, ss_tensor* y,
                               ss_tensor* last_state, void* stream);

/*
 * The selective scan of ss_selective_scan_fwd with every tensor in HOST
 * memory (no counterpart on the pages: this is the path a caller whose data
 * lives on the host takes, copies included).  Same arguments, shapes, dtypes
 * and results as ss_selective_scan_fwd, except:
 *   - every ss_tensor.data is a host pointer; page-locked (pinned) memory
 *     lets the copies run asynchronously, pageable memory works but the
 *     copies then block the calling thread;
 *   - every tensor must be contiguous (else SS_ERR_UNSUPPORTED).
 * The batch is cut into chunks of about 32 MB of inputs: whole batch rows, or,
 * when one row holds more, blocks of that row's channels (whole channel groups
 * when B, C are grouped; the row's B and C are copied once per buffer set);
 * chunks alternate between `stream` and one library-owned side stream per
 * device, so copies in, scans and copies out of neighbouring chunks overlap.  All work is joined back
 * into `stream` before the call returns (asynchronously: y and last_state
 * are valid once `stream` has completed, and the host buffers must stay
 * valid until then).  Device memory for the chunks is taken stream-ordered
 * (cudaMallocAsync / cudaFreeAsync on `stream`).  Calls on different streams
 * of one device share the side stream and so partly serialise.
 */
int ss_selective_scan_fwd_host(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                               ss_tensor* y, ss_tensor* last_state, void* stream);

/*
 * The SSD scan of ss_ssd_chunk_scan_fwd with every tensor in HOST memory (no
 * counterpart on the pages: the path of a caller whose data lives on the
 * host, copies included).  Same arguments, shapes, dtypes and results as
 * ss_ssd_chunk_scan_fwd, except:
 *   - every ss_tensor.data is a host pointer; page-locked (pinned) memory
 *     lets the copies run asynchronously, pageable memory works but the
 *     copies then block the calling thread;
 *   - every tensor must be contiguous (else SS_ERR_UNSUPPORTED).
 * The batch is cut into chunks of about 32 MB of x: whole batch rows, or,
 * when one row holds more, blocks of that row's heads (whole channel groups;
 * x and y move as 2-D copies, dt to a device pitch of a multiple of 8 heads,
 * the row's B and C once per buffer set); chunks alternate between `stream`
 * and the library-owned side stream of ss_selective_scan_fwd_host, so copies
 * in, scans and copies out of neighbouring chunks overlap.  All work is
 * joined back into `stream` before the call returns (asynchronously: y and
 * last_state are valid once `stream` has completed, and the host buffers must
 * stay valid until then).  Device memory for the chunks is taken
 * stream-ordered (cudaMallocAsync / cudaFreeAsync on `stream`).
 */
int ss_ssd_chunk_scan_fwd_host(const ss_tensor* x, const ss_tensor* dt, const ss_tensor* A_head,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               int chunk, ss_tensor* y, ss_tensor* last_state, void* stream);

/*
 * Backward of the selective scan (training): given dout, the gradient of a
 * loss with respect to the y of ss_selective_scan_fwd (same inputs, zero
 * initial state), writes the gradients with respect to every input
 * (0539edu paper talk §5.4: training recomputes the states of the scan
 * instead of keeping one per step; the forward it differentiates is that of
 * ss_selective_scan_fwd, "Mamba模型笔记" §2.2 and §4.3).
 *
 * With pre_t = sum_n C[b,n,t] h_t[n] + D[d] u_t and the adjoint state
 * g_t[n] = C[b,n,t] dpre_t + abar_{t+1}[n] g_{t+1}[n]:
 *   dz     = dout * pre * silu'(z);       dpre = dout * silu(z)  (dout if z NULL)
 *   du     = D dpre + sum_n g dl B;       dD   = sum_{b,t} dpre u
 *   dA     = sum_{b,t} g h_{t-1} abar dl
 *   dB     = sum_d g dl u;                dC   = sum_d dpre h_t
 *   ddelta = softplus'(delta + bias) * sum_n g (h_{t-1} abar A + B u)
 *   ddelta_bias = sum_{b,t} ddelta
 *
 * Inputs: as in ss_selective_scan_fwd; dout (Bsz, D, L) dtype T.
 * Outputs (all overwritten, none may overlap an input or another output):
 *   du, ddelta, dz  (Bsz, D, L) dtype T, any strides (dz iff z given)
 *   dA (D, N), dB, dC (Bsz, N, L), dD (D) iff D given,
 *   ddelta_bias (D) iff delta_bias given -- f32, contiguous (else
 *   SS_ERR_UNSUPPORTED).
 * N <= 16 (else SS_ERR_UNSUPPORTED).  With N = 16, unit t-stride and 16-byte
 * aligned rows the sums over channels, batch rows and steps are added in a
 * fixed order (bitwise reproducible).  With N = 16 and unit t-strides but rows
 * whose pitch or base is not a multiple of 16 bytes (an odd L in bf16), u,
 * delta, z, dout, B and C are copied into padded rows, the same kernel runs
 * there and du, ddelta, dz are copied back (one copy launch each way; same
 * fixed order).  Other layouts use f32 atomics, whose order, and so the last
 * bits, can differ from call to call.  Scratch is taken stream-ordered from
 * the device's default pool: the state every 8 steps (Bsz*D*ceil(L/8)*64
 * bytes) and per-block partial sums of dB, dC (ceil(D/32)*Bsz*L*128 bytes) on
 * the fast path, plus the padded copies (5 or 7 activations and B, C) where
 * taken; SS_ERR_ALLOC if the fast path's own scratch cannot be had (padded
 * copies that do not fit fall back to the atomics kernel).
 */
int ss_selective_scan_bwd(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                          const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                          const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                          const ss_tensor* dout, ss_tensor* du, ss_tensor* ddelta, ss_tensor* dA,
                          ss_tensor* dB, ss_tensor* dC, ss_tensor* dD, ss_tensor* dz,
                          ss_tensor* ddelta_bias, void* stream);

/*
 * Forward and backward of a training step that share the states (0539edu
 * paper talk §5.4 weighs keeping the scan's intermediate states for the
 * backward against recomputing them from the forward; here the forward keeps
 * the state every 8 steps, 64 bytes per channel and 8 steps, so that the
 * backward needs no forward pass of its own and recomputes only within 8
 * steps).
 *
 * ss_selective_scan_fwd_ckpt: ss_selective_scan_fwd (same arguments,
 *   checks, y and last_state) that also writes `ckpt`, f32 (Bsz, D,
 *   ceil(L/8), 16), contiguous, 16-byte aligned: ckpt[b,d,k,:] = the state
 *   h before step 8k (h after steps 0 .. 8k-1; zero at k = 0).  N = 16, B, C
 *   (Bsz, N, L) shared per batch row and unit t-strides only; else
 *   SS_ERR_UNSUPPORTED.  Rows whose pitch or base is not a multiple of 16
 *   bytes (an odd L in bf16) run on padded copies as in ss_selective_scan_fwd
 *   (the checkpoints are written in place); SS_ERR_UNSUPPORTED when those
 *   copies do not fit in device memory.
 * ss_selective_scan_bwd_ckpt: ss_selective_scan_bwd (same arguments, checks
 *   and gradients) given that checkpoint tensor from the forward of the same
 *   inputs; it reads the states from it instead of recomputing them (the
 *   scratch of the states is not taken).  Same layout limits and padded
 *   copies, else SS_ERR_UNSUPPORTED; a null ckpt is SS_ERR_INVALID_ARG.  Gradients equal
 *   ss_selective_scan_bwd's up to rounding (bit for bit when the forward did
 *   not split the sequence into segments).
 */
int ss_selective_scan_fwd_ckpt(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                               ss_tensor* y, ss_tensor* last_state, ss_tensor* ckpt,
                               void* stream);
int ss_selective_scan_bwd_ckpt(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                               const ss_tensor* dout, const ss_tensor* ckpt, ss_tensor* du,
                               ss_tensor* ddelta, ss_tensor* dA, ss_tensor* dB, ss_tensor* dC,
                               ss_tensor* dD, ss_tensor* dz, ss_tensor* ddelta_bias, void* stream);

/*
 * One recurrent step (decoding one token), updating the state in place
 * (0539edu paper talk §4.3: the step function of the recurrent form; the
 * state is the only thing carried between tokens).
 *
 * ss_selective_state_update, per batch row b and channel d:
 *   dl = softplus?(delta[b,d] + delta_bias[d]);
 *   state[b,d,n] = exp(dl A[d,n]) state[b,d,n] + dl B[b,n] u[b,d];
 *   y[b,d] = (sum_n C[b,n] state[b,d,n] + D[d] u[b,d]) * z * sigmoid(z)
 *   state (Bsz, D, N) f32 in/out; u, delta, z, y (Bsz, D) dtype T;
 *   B, C (Bsz, N) dtype T; A (D, N), D, delta_bias (D) f32.  N <= 256.
 *
 * ss_ssd_state_update, per batch row b, head h (group g = h / (H/G)), p:
 *   a = exp(dt[b,h] A_head[h]);
 *   state[b,h,p,n] = a state[b,h,p,n] + dt[b,h] x[b,h,p] B[b,g,n];
 *   y[b,h,p] = sum_n C[b,g,n] state[b,h,p,n] + D[h] x[b,h,p]
 *   state (Bsz, H, P, N) f32 in/out; x, y (Bsz, H, P) dtype T; dt (Bsz, H)
 *   dtype T (positive); B, C (Bsz, G, N) dtype T; A_head, D (H) f32.
 *
 * Applying the step to t = 0 .. L-1 in turn gives the scans' y and final state.
 */
int ss_selective_state_update(ss_tensor* state, const ss_tensor* u, const ss_tensor* delta,
                              const ss_tensor* A, const ss_tensor* B, const ss_tensor* C,
                              const ss_tensor* D, const ss_tensor* z, const ss_tensor* delta_bias,
                              int softplus, ss_tensor* y, void* stream);
int ss_ssd_state_update(ss_tensor* state, const ss_tensor* x, const ss_tensor* dt,
                        const ss_tensor* A_head, const ss_tensor* B, const ss_tensor* C,
                        const ss_tensor* D, ss_tensor* y, void* stream);

/* Name of a status code (static string, never NULL). */
const char* ss_status_string(int status);

/*
 * Device-side error word of the current device: synchronises `stream`, then
 * returns SS_OK or SS_ERR_TIMEOUT if any kernel of this library gave up on a
 * bounded wait since the last call, and clears the word.
 */
int ss_get_device_error(void* stream);

/*
 * Self-test of the failure path (no counterpart on the pages): launches a
 * kernel on `stream` whose bounded wait on an mbarrier can never complete and
 * gives up after `limit_us` microseconds (1 .. 100000, else
 * SS_ERR_INVALID_ARG), recording the same device error bit as a scan kernel
 * whose wait ran out.  The next ss_get_device_error on that stream returns
 * SS_ERR_TIMEOUT and clears it; the CUDA context stays usable.  Nothing
 * faults, traps or hangs.
 */
int ss_selftest_timeout(unsigned limit_us, void* stream);

/*
 * Diagnostic switches (no counterpart on the pages): which kernel a call
 * takes, for tests that must reach one kernel on purpose and for
 * measurements.  The library reads no environment variable; these switches
 * change only when this function is called.  The setting is process-wide (all
 * devices, all threads), read at the start of each call: change it only
 * while no call of this library is in flight on another host thread.
 * `value` -1 restores the library's own choice (the default of every switch).
 *
 *   SS_DEBUG_SCAN_PATH      selective scan: 0 the general kernel (any layout),
 *                           1 scan_fast (lanes per channel from
 *                           SS_DEBUG_SCAN_SPLIT), 2 scan_seq
 *   SS_DEBUG_SCAN_SPLIT     scan_fast lanes per channel: 1, 2, 4 or 8
 *   SS_DEBUG_SCAN_SHAPE     scan_seq launch shape 1 .. 7: lanes per channel
 *                           and channels per CTA 1/128, 1/128, 2/64, 4/32,
 *                           2/64, 1/128, 2/64 (tile rows, stages, CTAs per SM
 *                           and the helper warp differ)
 *   SS_DEBUG_SCAN_SEGMENTS  scan_seq time segments (1 .. 128)
 *   SS_DEBUG_SCAN_SEG_TILES scan_seq shortest segment of its own choice, in tiles of t
 *   SS_DEBUG_SSD_PATH       SSD scan: 0 the CUDA-core kernel, 1 the tensor-core
 *                           kernels only, 2 the one-head tensor-core kernel
 *                           only; with 1 or 2 a shape or layout those kernels
 *                           do not take returns SS_ERR_UNSUPPORTED instead of
 *                           falling back
 *   SS_DEBUG_BWD_PATH       backward: 0 the general kernel
 *   SS_DEBUG_GROUPED_PATH   B, C per small channel group: 0 the row kernel
 *                           (scan_pc) instead of the TMA kernel
 *   SS_DEBUG_SSD_LATE_CUMSUM 1: the two-head tensor-core SSD kernel forms
 *                           every next block's cumulative decay after the
 *                           state update, never early while the MMAs run
 *                           (which of the two it takes otherwise depends on
 *                           when dt lands; the results are the same)
 *   SS_DEBUG_FAULT_ALLOC    1: every stream-ordered scratch allocation fails,
 *                           so calls that need scratch return SS_ERR_ALLOC
 *                           before launching anything (host-side fault
 *                           injection)
 *
 * Returns SS_OK, or SS_ERR_INVALID_ARG for an unknown switch.
 */
#define SS_DEBUG_SCAN_PATH 0
#define SS_DEBUG_SCAN_SPLIT 1
#define SS_DEBUG_SCAN_SHAPE 2
#define SS_DEBUG_SCAN_SEGMENTS 3
#define SS_DEBUG_SSD_PATH 4
#define SS_DEBUG_BWD_PATH 5
#define SS_DEBUG_GROUPED_PATH 6
#define SS_DEBUG_FAULT_ALLOC 7
#define SS_DEBUG_SCAN_SEG_TILES 8
#define SS_DEBUG_SSD_LATE_CUMSUM 9
#define SS_DEBUG_COUNT 10
int ss_debug_set_path(int which, int value);

/*
 * Throughput probe (no counterpart on the pages): measures how many
 * ex2.approx.f32 operations (the MUFU exponential every state of the
 * selective scan needs once per step) one SM completes per clock on the
 * current device, with one 1024-thread CTA per SM running independent
 * chains, timed by the SM's own clock.  Writes the rate to
 * *ex2_per_sm_per_clock.  Synchronises `stream`; allocates nothing.
 * Returns SS_OK, SS_ERR_INVALID_ARG (NULL output), SS_ERR_LAUNCH or
 * SS_ERR_CUDA.
 */
int ss_probe_ex2_rate(double* ex2_per_sm_per_clock, void* stream);

/*
 * Throughput probe of the two forms of the recurrence (page "Mamba模型笔记"
 * §4.5: the selective scan as a parallel scan over (A_bar, B_bar u) pairs):
 * on synthetic 32-step tiles of one channel with 16 states and a shared B | C
 * table, `seq` steps one lane per channel through t with the states in
 * registers (the form the scan kernels use); `shfl` gives each lane one step
 * and composes the tile's 32 pairs with a five-level warp-shuffle scan per
 * state, then applies the previous tile's carry and takes the readout.  Writes
 * the channel-steps per second of each form.  Synchronises `stream`;
 * allocates nothing.  Returns SS_OK, SS_ERR_INVALID_ARG or SS_ERR_CUDA.
 */
int ss_probe_scan_forms(double* seq_steps_per_s, double* shfl_steps_per_s, void* stream);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t ss_launch_count(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int ss_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSSCAN_H */
