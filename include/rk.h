/*
 * rk.h -- C ABI of the GB300 recurrent-layer library (ONNX LSTM / GRU / RNN
 * forward pass on one GPU, sm_103a).
 *
 * The operation is the one defined on the web page "Recurrent layers"
 * (onegpu docs):
 *   - first paragraph: cells RNN, GRU, LSTM; directions forward, reverse,
 *     bidirectional; layouts 0 and 1; sequence_lens; initial states;
 *     peepholes; clip; input_forget; linear_before_reset; the eleven ONNX
 *     activations with alpha / beta resolved by the caller; all tensors
 *     float32 or all Half, with float32 accumulation and float32 state
 *     (bfloat16 tensors as a third type, the way the web page "Matrix
 *     multiplication (Gemm)" admits them in its first paragraph, same
 *     float32 arithmetic);
 *   - the C# example and the paragraph after it: a problem description
 *     (RecurrentProblem) and an operand list X, W, R, B, sequence_lens,
 *     initial_h, initial_c, P, Y, Y_h, Y_c, each a buffer plus an element
 *     offset (GpuTensorRef); W, R, B, P used as stored, gate order i, o, f, c
 *     (LSTM) and z, r, h (GRU); null outputs are not written;
 *   - section "How a layer runs": the input projection Xw = X . W^T for all
 *     steps and directions, the state setup, the steps, the outputs;
 *   - section "Arithmetic and determinism": pre = ((xw + rec) + Wb) + Rb,
 *     then peepholes, clip, activation, state update; runs are bit-identical;
 *   - section "Semantics": sequence_lens, Seq = 0, Batch = 0, clip, options
 *     legal per cell (anything else is an error);
 *   - the "Scratch" paragraph: XwLength / StateLength floats, kept by the
 *     library and grown on demand, or placed by the caller with element
 *     offsets (both may sit in one arena); checks in safe arithmetic before
 *     anything is launched, with an error that names the cell and argument.
 *
 * Shapes (D = 2 for bidirectional, else 1; G = 4 LSTM, 3 GRU, 1 RNN;
 * S seq, N batch, I input, H hidden), all dense row-major:
 *   X            [S, N, I] (layout 0)   or [N, S, I] (layout 1)
 *   W            [D, G*H, I]
 *   R            [D, G*H, H]
 *   B            [D, 2*G*H]   (Wb then Rb)               optional, else 0
 *   sequence_lens[N] int32                                optional, else S
 *   initial_h    [D, N, H]   (layout 0) or [N, D, H]      optional, else 0
 *   initial_c    same as initial_h, LSTM only             optional, else 0
 *   P            [D, 3*H]    (i, o, f), LSTM only         optional, else 0
 *   Y            [S, D, N, H] (layout 0) or [N, S, D, H]  optional output
 *   Y_h          [D, N, H]   (layout 0) or [N, D, H]      optional output
 *   Y_c          same as Y_h, LSTM only                   optional output
 * Every tensor other than sequence_lens has the problem's dtype (float32,
 * IEEE binary16 or bfloat16).  Inputs are widened exactly to float32;
 * outputs are rounded to nearest even when 16-bit.
 *
 * Ownership: every tensor pointer is caller-owned DEVICE memory (except in
 * rk_encode_host, which takes host memory).  The library never frees or
 * rewrites an input.  Handles are not thread-safe: one host thread at a time.
 * Errors: every function returns an rk_status; nothing is launched when a
 * check fails; rk_last_error() then names the cell and the argument.
 */
#ifndef RK_H_
#define RK_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t rk_status;
#define RK_OK 0
#define RK_ERR_SHAPE 1       /* bad size, offset, option for the cell, overflow */
#define RK_ERR_UNSUPPORTED 2 /* legal but not runnable here (residency, size)  */
#define RK_ERR_CUDA 3        /* a CUDA call failed; message has the error name  */
#define RK_ERR_TIMEOUT 4     /* a bounded device wait gave up                   */
#define RK_ERR_OOM 5         /* device scratch allocation failed                */
#define RK_ERR_ARG 6         /* null handle / problem / operand list            */

enum rk_cell { RK_LSTM = 0, RK_GRU = 1, RK_RNN = 2 };
enum rk_direction { RK_FORWARD = 0, RK_REVERSE = 1, RK_BIDIRECTIONAL = 2 };
enum rk_dtype { RK_F32 = 0, RK_F16 = 1, RK_BF16 = 2 };
enum rk_activation_kind {
  RK_ACT_SIGMOID = 0,
  RK_ACT_TANH = 1,
  RK_ACT_RELU = 2,
  RK_ACT_AFFINE = 3,           /* alpha*x + beta */
  RK_ACT_LEAKY_RELU = 4,       /* x >= 0 ? x : alpha*x */
  RK_ACT_THRESHOLDED_RELU = 5, /* x > alpha ? x : 0 */
  RK_ACT_SCALED_TANH = 6,      /* alpha*tanh(beta*x) */
  RK_ACT_HARD_SIGMOID = 7,     /* clamp(alpha*x + beta, 0, 1) */
  RK_ACT_ELU = 8,              /* x >= 0 ? x : alpha*(exp(x) - 1) */
  RK_ACT_SOFTSIGN = 9,         /* x / (1 + |x|) */
  RK_ACT_SOFTPLUS = 10         /* log(1 + exp(x)) */
};

/* rk_create flags */
#define RK_FORCE_SIMT_PROJECTION 1u /* 16-bit problems: SIMT projection, no tensor cores */
#define RK_FORCE_GRID_STEP 2u       /* use the grid-wide step kernel even where a cluster fits */
#define RK_FORCE_GENERAL_STEP 4u    /* never the one-row-per-cluster register-resident step kernel */
#define RK_FORCE_SIMT_STEP 8u       /* 16-bit problems: never the tensor-core step kernel */
#define RK_SEPARATE_PROJECTION 16u  /* never compute the projection on the SMs the tensor-core
                                       recurrence leaves idle (always a launch of its own) */
#define RK_PREFER_TENSOR_STEP 32u   /* 16-bit problems: a tensor-core step kernel wherever one applies,
                                       ahead of the register-resident SIMT kernel (which is faster
                                       wherever all its clusters fit the GPU) */

/* One activation slot (GpuRecurrentActivation): kind plus resolved alpha/beta. */
typedef struct rk_activation {
  int32_t kind;
  float alpha;
  float beta;
} rk_activation;

/* The layer (RecurrentProblem). */
typedef struct rk_problem {
  int32_t cell;                /* rk_cell */
  int32_t direction;           /* rk_direction */
  int32_t dtype;               /* rk_dtype, shared by all tensors */
  int32_t layout;              /* 0 or 1 */
  int64_t seq, batch, input, hidden;
  float clip;                  /* > 0 clamps pre-activations to [-clip, clip]; else off */
  int32_t input_forget;        /* LSTM only: f = 1 - i */
  int32_t linear_before_reset; /* GRU only */
  int32_t num_acts;            /* 0: ONNX defaults; else G' * D (G' = 3 LSTM, 2 GRU, 1 RNN) */
  rk_activation act[6];        /* slots f, g, h of direction 0, then of direction 1 */
  int64_t max_length;          /* 0: seq.  Else a promise that no sequence_lens
                                  entry exceeds it; shortens the step loop.
                                  Needs sequence_lens when < seq. */
} rk_problem;

/* A tensor (GpuTensorRef): base pointer, element offset from it, and the
 * number of elements available from the base (the buffer's length), so the
 * library can check offset + extent <= length.  ptr == NULL means absent. */
typedef struct rk_tensor {
  void* ptr;
  int64_t offset;
  int64_t length;
} rk_tensor;

/* The operand list (RecurrentOperands).  X, W, R are required. */
typedef struct rk_operands {
  rk_tensor X, W, R, B, sequence_lens, initial_h, initial_c, P, Y, Y_h, Y_c;
} rk_operands;

/* Caller-placed scratch (float32 device memory).  Either pointer may be NULL,
 * in which case the library uses its own grown-on-demand allocation.  The two
 * regions may lie in one arena buffer but must not overlap.  state + offset
 * must be 16-byte aligned (it is read as float4); xw has no alignment rule. */
typedef struct rk_scratch {
  float* xw;
  int64_t xw_offset;
  int64_t xw_length;
  float* state;
  int64_t state_offset;
  int64_t state_length;
} rk_scratch;

typedef struct rk_handle rk_handle;

/* Version of this ABI (major * 10000 + minor * 100 + patch).  No counterpart
 * on the pages (their version is a package version). */
int32_t rk_version(void);

/* Create a handle: the kernel family object of the web page "Recurrent
 * layers" (`new RecurrentKernels(device)` in its C# example), which keeps the
 * scratch it grows on demand (paragraph "Scratch").  The device is the CUDA
 * device current at the first encode; no CUDA call is made until then, so
 * this works without a GPU.  flags: the rk_create flag bits above (kernel
 * choices; the pages' GpuKernelMode has no counterpart here since every
 * kernel is deterministic, section "Arithmetic and determinism").  *out
 * receives the handle, owned by the caller until rk_destroy.  Returns
 * RK_ERR_ARG for out == NULL, RK_ERR_OOM if the host allocation fails. */
rk_status rk_create(rk_handle** out, uint32_t flags);

/* Wait for the handle's work on the streams it used, free its scratch and the
 * handle (the disposal of the C# example's `using var rnn` on the web page
 * "Recurrent layers"; the scratch is the family's own, paragraph "Scratch").
 * NULL is accepted.  Caller-owned tensors and caller-placed scratch are not
 * touched. */
rk_status rk_destroy(rk_handle* h);

/* Floats of projection scratch the problem needs: RecurrentKernels.XwLength
 * of the web page "Recurrent layers", paragraph "Scratch" (the float32 Xw of
 * section "How a layer runs", step 1): D * S * N * G * H for S, N > 0, else
 * 0.  Host only.  Returns -1 for an invalid problem (p == NULL included). */
int64_t rk_xw_length(const rk_problem* p);

/* Floats of state scratch the problem needs: StateLength of the web page
 * "Recurrent layers", paragraph "Scratch".  The pages' state holds every
 * step's output; here, where the steps run inside one kernel, it holds 256
 * counter words, the grid step kernel's team counters, 64 per direction and
 * group of up to 64 batch rows, the double-buffered hidden state
 * exchanged between blocks of the step kernel, 2 * D * N * KP, and a region
 * for r (.) h or the 16-bit copies of h used by the tensor cores,
 * D * (N + 128) * KP (KP = hidden rounded up to a multiple of 128).  Host
 * only.  Returns -1 for an invalid problem. */
int64_t rk_state_length(const rk_problem* p);

/* Host-only validation of a problem and its operands: the checks of the web
 * page "Recurrent layers", paragraph "Scratch" (sizes, offsets and shapes in
 * safe 64-bit arithmetic, an error naming LSTM / GRU / RNN and the argument)
 * and section "Semantics", last item (peepholes, input_forget, initial_c and
 * Y_c only for an LSTM, linear_before_reset only for a GRU; anything else is
 * an error).  Makes no CUDA call.  Returns RK_OK, RK_ERR_SHAPE (the pages'
 * GpuKernelShapeException), RK_ERR_UNSUPPORTED (sizes past 32-bit indexing)
 * or RK_ERR_ARG (null handle, problem or operand list), with rk_last_error
 * set. */
rk_status rk_validate(rk_handle* h, const rk_problem* p, const rk_operands* ops);

/* Host-only check of a HOST copy of sequence_lens (web page "Recurrent
 * layers", section "Semantics": the kernels read the lengths on the device
 * and do not validate them -- a negative length runs as 0 steps and one
 * above seq as seq).  lens points to n int32 values.  Returns RK_OK when
 * n == batch and every value lies in [0, seq], and also in [0, max_length]
 * when max_length > 0 (the promise that shortens the step loop); else
 * RK_ERR_SHAPE with rk_last_error naming the cell, the first offending row
 * and its value (RK_ERR_ARG for a null handle or problem, or lens == NULL
 * with n > 0).  Makes no CUDA call. */
rk_status rk_validate_lengths(rk_handle* h, const rk_problem* p, const int32_t* lens, int64_t n);

/* Enqueue the whole layer on `stream` (a cudaStream_t; NULL = legacy default
 * stream): `rnn.Encode(encoder, problem, tensors)` of the web page "Recurrent
 * layers" (C# example), computing section "How a layer runs" steps 1-4 with
 * the arithmetic of section "Arithmetic and determinism" and the rules of
 * section "Semantics": the input projection, then one persistent step kernel
 * that sets up the state, runs every step and writes Y, Y_h, Y_c.
 * Asynchronous: returns after enqueueing.  scratch may be NULL (the handle's
 * own, grown on demand) or place both regions (paragraph "Scratch").  All
 * operand pointers are caller-owned device pointers, read or written only by
 * the enqueued kernels.  Errors: the checks of rk_validate (nothing is
 * launched); RK_ERR_UNSUPPORTED when no step kernel can be resident; RK_ERR_OOM
 * when growing the scratch fails; RK_ERR_CUDA when a launch fails.  Batch = 0
 * or hidden = 0 records nothing; Seq = 0 writes only Y_h / Y_c (the initial
 * states or zeros). */
rk_status rk_encode(rk_handle* h, const rk_problem* p, const rk_operands* ops,
                    const rk_scratch* scratch, void* stream);

/* Same layer with HOST operand pointers (no counterpart on the pages, whose
 * tensors are always device buffers): encodes on `stream` and synchronises
 * the stream before returning.  X and W are always copied to device buffers
 * owned by the handle (grown on demand): W on `stream`, X on a second stream
 * owned by the handle (started after the work already on `stream`, joined
 * before the projection), so the two copies overlap.  Every other operand
 * (R, B, sequence_lens, initial states, P; the outputs Y, Y_h, Y_c) that
 * lies in page-locked host memory (cudaHostAlloc, cudaHostRegister, e.g. a
 * pinned torch tensor) is not copied: the step kernel reads or writes it in
 * place through the device's mapping of that memory, each element once.
 * Operands in other host memory are copied: inputs on the second stream,
 * joined just before the step kernel (they land while the projection
 * runs), outputs back on `stream` after it.  When it returns, success or
 * error, every copy and kernel it issued has completed (the host buffers may
 * be reused at once). */
rk_status rk_encode_host(rk_handle* h, const rk_problem* p, const rk_operands* host_ops,
                         void* stream);

/* Synchronise `stream`, read and clear the device status word of the handle
 * (and, once rk_encode_noalloc has run on the handle, the status word of its
 * fixed array): RK_OK, or RK_ERR_TIMEOUT if a bounded device wait of a step
 * kernel or of the tensor-core projection gave up during a previous encode;
 * the outputs of that encode are then undefined.  The web page "Recurrent
 * layers" has no counterpart: its design waits on nothing inside a launch
 * (one pass per step, paragraph "Why a pass per step"), while this library's
 * persistent kernels wait on the device, each wait bounded so that a launch
 * that cannot finish reports RK_ERR_TIMEOUT instead of hanging. */
rk_status rk_status_poll(rk_handle* h, void* stream);

/* (No counterpart on the pages; see rk_status_poll.)
 * Nanoseconds (measured on the GPU's global timer) a device-side wait of the
 * step kernel may spin before it gives up, sets the status word and lets the
 * kernel wind down; default 2e9 (2 s).  limit must be >= 1. */
rk_status rk_set_wait_limit(rk_handle* h, int64_t limit);

/* (No counterpart on the pages; see rk_status_poll.)
 * Run the step kernels' bounded device waits against a release counter and an
 * mbarrier that nothing completes (one CTA, no other memory touched): each
 * must give up after timeout_ns and set the handle's status word.  Returns
 * RK_OK once the check kernel is enqueued on `stream`; rk_status_poll then
 * returns RK_ERR_TIMEOUT.  Used to test the give-up path without a hang. */
rk_status rk_selftest_timeout(rk_handle* h, void* stream, int64_t timeout_ns);

/* The layer of rk_encode, for callers that cannot allocate device memory:
 * a runtime whose memory planner owns every device allocation and allows no
 * new one after start-up, a process with a fixed device-memory budget, or
 * code that must not pay the device-wide synchronisation cudaFree can imply.
 * The pages have no counterpart of this entry point.
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine.  Its scratch
 * (projection Xw plus the step kernel's exchange buffers, barrier counters
 * and status word) is a fixed 16 MiB float32 array inside the library, which
 * every GPU that loads the library holds until the process exits.  A layer
 * needing more than 4 Mi floats (rk_state_length rounded up to 64, plus
 * rk_xw_length) is rejected with RK_ERR_UNSUPPORTED and a message giving both
 * numbers; nothing is launched then.  The caller passes inputs and outputs as
 * for rk_encode (device pointers); h holds only host-side state.
 *
 * The first call on each device takes the array's device address with
 * cudaGetSymbolAddress (with that device current); make that first call
 * before any stream capture.  Every call on a device shares the one array,
 * which keeps the previous call's contents: the call clears what must start
 * at zero (barrier counters, status word).  Calls whose work overlaps on the
 * GPU (other streams, other host threads) race on the array and give
 * undefined results: order them on one stream.  Both resets are enqueued
 * before the call's first kernel, so after the call the array's status word
 * holds the give-ups of both kernels: rk_status_poll on the same handle reads
 * and clears it (RK_ERR_TIMEOUT: the outputs of that call are undefined).
 * With rk_set_profiling on, the call records its projection and step events
 * like rk_encode. */
rk_status rk_encode_noalloc(rk_handle* h, const rk_problem* p, const rk_operands* ops, void* stream);

/* (No counterpart on the pages, which time whole layers.)
 * Kernel timing for measurement: with enabled != 0 every later encode records
 * CUDA events (on its stream) around its projection launch and its step
 * launch; rk_last_timings then waits for them and returns the two durations
 * of the most recent encode in milliseconds (-1 for a launch that did not
 * happen).  Disabled by default. */
rk_status rk_set_profiling(rk_handle* h, int32_t enabled);
rk_status rk_last_timings(rk_handle* h, float* projection_ms, float* step_ms);

/* Message of the last failed call on this handle ("" if none): the text the
 * web page "Recurrent layers" gives its shape errors (paragraph "Scratch":
 * it names LSTM / GRU / RNN and the argument), e.g. "GRU: R: offset 0 +
 * extent 768 exceeds buffer length 5".  The string belongs to the handle and
 * stays valid until its next call. */
const char* rk_last_error(const rk_handle* h);

/* Number of kernels this handle has launched so far (all encodes): the
 * evidence that a layer costs a fixed number of launches whatever its
 * sequence length, where the web page "Recurrent layers" spends one pass per
 * step (section "How a layer runs", step 3; paragraph "What a step costs"). */
uint64_t rk_launch_count(const rk_handle* h);

/* (No counterpart on the pages.)
 * Describe the plan encode would use for a problem (for logs and tests): a
 * NUL-terminated text such as "proj=simt_f32 step=cluster16 nb=1 ..." written
 * into buf (at most len bytes).  Host only. */
rk_status rk_describe_plan(rk_handle* h, const rk_problem* p, char* buf, int64_t len);

#ifdef __cplusplus
}
#endif

#endif /* RK_H_ */
