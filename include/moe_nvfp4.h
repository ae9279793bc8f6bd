/*
 * moe_nvfp4.h -- C ABI of the GB300 (sm_103a) routed-experts MoE step over
 * NVFP4 expert weights.
 *
 * The operation (one MoE layer's routed experts, one step):
 *
 *   y_t = sum_{j < k, slot valid} w_tj * W_down[e_tj] ( SiLU(W_gate[e_tj] x_t) (.) (W_up[e_tj] x_t) )
 *         [ + W_down_s ( SiLU(W_gate_s x_t) (.) (W_up_s x_t) )   with a shared expert ]
 *
 * for T tokens with router ids e_tj and weights w_tj.  This is the step the
 * serving pages' "lna2" kernel computes ("LNA-CANON.md", section "lna2 とは":
 * resident expert teams pulling dynamic tickets with no grid-wide barrier, rows
 * per expert R_e, m <= 24 tokens; "dsv4-carve" README, section "house kernel
 * lna2": 104.0 us per launch against exl3_moe's 232.6 us).  The pages' EXL3
 * trellis weights are never defined there; the expert weights here are NVFP4
 * (V100 page, section 7.1: NVFP4 expands into FP16 in registers almost for
 * free): E2M1 values, one E4M3 scale per 16 elements along the reduction axis,
 * one FP32 tensor scale per (expert, projection).
 *
 * Conventions shared by every entry point:
 *  - Pointers named *_dev are CUDA device pointers on the plan's device; the
 *    caller owns them (allocates, frees, keeps them alive while work that
 *    uses them is in flight).  The library never frees caller memory and
 *    allocates no device memory.  Pointers named *_host are host pointers,
 *    also owned by the caller.
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *    stream.  Work is enqueued asynchronously; no entry point below
 *    synchronises except moe_check.
 *  - A status other than MOE_OK leaves nothing enqueued; moe_last_error()
 *    returns a message for the calling thread's last failure.
 *  - There is no CPU fallback and no other backend: a shape or argument the
 *    sm_103a kernels do not take is an error, never a silent detour.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_NVFP4_ABI_VERSION 8

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,       /* null pointer, bad size, T > T_max, ...          */
    MOE_ERR_UNSUPPORTED_SHAPE = 2, /* H, I, E or top_k outside what the kernels take  */
    MOE_ERR_NOT_FAST_PATH = 3,     /* strict mode: call would leave the named path     */
    MOE_ERR_MISALIGNED = 4,        /* a pointer is not aligned as documented          */
    MOE_ERR_CUDA = 5,              /* a CUDA runtime call failed (message has details) */
    MOE_ERR_TIMEOUT = 6,           /* device: a bounded wait gave up (see moe_check)   */
    MOE_ERR_BAD_EXPERT_ID = 7,     /* device: an id >= E was seen (slot skipped)       */
    MOE_ERR_RANGE = 8,             /* device: an intermediate (h) was not finite      */
    MOE_ERR_SCALE = 9,             /* device: a weight block scale the tensor-core     */
                                   /*   kernels cannot read (sign bit set, or NaN;    */
                                   /*   found by moe_workspace_init's scan)           */
    MOE_ERR_WORKSPACE_BUSY = 10    /* host: another thread is launching on the        */
                                   /*   workspace from another stream                 */
} moe_status_t;

/* Opaque plan: host memory owned by the library (moe_plan_destroy frees it). */
typedef struct moe_plan *moe_plan_t;

/* Plan description.  Weight layouts (row-major, C order):
 *   gate_q, up_q  uint8 [E, I, H/2]  element c of a row: low nibble of byte c/2
 *   down_q        uint8 [E, H, I/2]  if c is even, high nibble if c is odd
 *   gate_s, up_s  uint8 [E, I, H/16] E4M3 scale of elements 16b .. 16b+15
 *   down_s        uint8 [E, H, I/16]
 *   gate_ts, up_ts, down_ts  float [E]  FP32 tensor scale per (expert, projection)
 * A weight is  E2M1(nibble) * E4M3(block scale) * tensor scale.
 * Every weight pointer must be 16-byte aligned; the *_ts arrays 4-byte aligned. */
typedef struct {
    int H;      /* hidden size, multiple of 128                                  */
    int I;      /* expert intermediate size, multiple of 128                     */
    int E;      /* number of experts, 1 .. 1024                                  */
    int top_k;  /* slots per token, 1 .. 16                                      */
    int T_max;  /* largest T any call on this plan may pass (sizes workspaces)   */
    const uint8_t *gate_q_dev, *up_q_dev, *down_q_dev;
    const uint8_t *gate_s_dev, *up_s_dev, *down_s_dev;
    const float *gate_ts_dev, *up_ts_dev, *down_ts_dev;
    int device; /* CUDA device ordinal the pointers live on; -1 = current device */
    int strict; /* 1: refuse (MOE_ERR_NOT_FAST_PATH) anything but the named path; */
                /*    the environment variable MOE_STRICT=1 forces it on          */
    int pdl;    /* 1: launch with programmatic dependent launch allowed          */
    int kernel; /* which step kernel runs moe_decode / moe_prefill:               */
                /*   MOE_KERNEL_AUTO: per launch: for one token (T = 1), where H */
                /*     is a multiple of 2048 up to 16384, I a multiple of 256 up */
                /*     to 4096 and act_quant is 0, the one-token row kernel      */
                /*     (E2M1 x E4M3 dequantised in registers, fp16 mma.sync, one */
                /*     grid-wide barrier between gate/up and down; the           */
                /*     environment variable MOE_GEMV=0 at plan creation leaves   */
                /*     it out); else, where the shape allows the tensor cores    */
                /*     (H and I multiples of 256, I <= 4096): the small-launch   */
                /*     tensor-core kernel for at most 4 tokens and 32 (token,    */
                /*     slot) pairs, the tensor-core ticket kernel for more than  */
                /*     8 pairs;                                                  */
                /*     otherwise the register kernel.  The one-token row kernel   */
                /*     needs every CTA of its grid (one per SM) resident at once: */
                /*     a step that shares the device with other work may wait     */
                /*     for SMs, and past the plan's wait limit reports            */
                /*     MOE_ERR_TIMEOUT;                                           */
                /*   MOE_KERNEL_REGISTER: E2M1 x E4M3 dequantised in registers,   */
                /*     fp16 mma.sync (any shape the plan accepts);                */
                /*   MOE_KERNEL_TENSOR: tcgen05 block-scaled FP4 MMA on the        */
                /*     NVFP4 bytes, activations as four FP4 digit rows: the      */
                /*     small-launch kernel for launches it takes, else the        */
                /*     ticket kernel (the environment variable MOE_SMALL=0 at    */
                /*     plan creation leaves the small-launch kernel out) (the plan */
                /*     is refused with UNSUPPORTED_SHAPE where the shape does not */
                /*     allow it).  The tensor-core kernels need non-negative,     */
                /*     non-NaN E4M3 block scales (the MMA reads them unsigned),   */
                /*     as an NVFP4 quantiser writes them: moe_workspace_init of a */
                /*     plan that may run them scans every weight block scale and  */
                /*     a negative or NaN one makes moe_check report MOE_ERR_SCALE */
                /*     (their y would be wrong).  The register and row kernels    */
                /*     decode the sign.                                           */
    /* Shared expert (optional; NULL shared_gate_q_dev: none).  One always-on
     * SwiGLU expert in the same NVFP4 format, added to every token's y with
     * weight 1 after the routed slots, inside the same launch (the serving
     * pages run it on a second stream, which deadlocked: "dsv4-carve" README,
     * "The three traps", trap 3; "LNA-CANON.md" launches with the shared-expert
     * fusion switched off).  Layouts: gate_q, up_q [I, H/2]; down_q [H, I/2];
     * gate_s, up_s [I, H/16]; down_s [H, I/16]; ts float [3] = the gate, up
     * and down tensor scales.  Same alignment rules as the routed arrays. */
    const uint8_t *shared_gate_q_dev, *shared_up_q_dev, *shared_down_q_dev;
    const uint8_t *shared_gate_s_dev, *shared_up_s_dev, *shared_down_s_dev;
    const float *shared_ts_dev;
    /* Expert range (expert parallelism): this plan serves experts e_lo ..
     * e_hi-1 of the E the router picks from, and the routed weight arrays
     * above hold only those (expert e at index e - e_lo).  A valid id outside
     * the range belongs to another plan and counts as an empty slot here (not
     * as an error); y is then this plan's partial sum, and the partial sums of
     * plans over disjoint ranges covering [0, E) add up to the whole step (the
     * shared expert belongs in exactly one of them).  e_lo = e_hi = 0: all E. */
    int e_lo, e_hi;
    /* Activation quantisation.  0: x and h enter the MMAs as four FP4 digit
     * rows (close to their bf16 / fp32 values).  1: x and h are quantised
     * once to NVFP4 before each projection, as a checkpoint that ships
     * activation input scales expects (the V100 page, section 3.0, adds the
     * missing input_scale tensors before launch): per row one power-of-two
     * prescale (largest |v| into (1344, 2688]), per 16 elements the smallest
     * E4M3 scale >= block max / 6, each element the nearest E2M1 value (ties
     * to even) of v / scale.  Tensor-core kernels only: a plan with kernel =
     * MOE_KERNEL_REGISTER or a shape they do not take is refused with
     * UNSUPPORTED_SHAPE, and moe_decode_static refuses such a plan. */
    int act_quant;
} moe_plan_desc;

enum { MOE_KERNEL_AUTO = 0, MOE_KERNEL_REGISTER = 1, MOE_KERNEL_TENSOR = 2 };

/* Per-plan launch counters (host side; how many times each path ran). */
typedef struct {
    uint64_t decode_launches;  /* persistent ticket kernel, T <= 24             */
    uint64_t prefill_launches; /* persistent ticket kernel, prefill chunks      */
    uint64_t null_launches;    /* measurement variant (no dequant, no math)     */
    uint64_t group_launches;   /* stand-alone grouping kernel                   */
    uint64_t rejected_calls;   /* calls that returned an error status           */
    uint64_t tensor_launches;  /* of decode + prefill: tensor-core kernel       */
    uint64_t route_launches;   /* top-k routing kernel (moe_route)              */
    uint64_t small_launches;   /* of tensor_launches: the small-launch kernel   */
    uint64_t gemv_launches;    /* of decode + prefill: the one-token row kernel */
    int num_sms;               /* SMs on the plan's device (grid size)          */
    int stages;                /* shared-memory ring stages at the largest T    */
    int smem_bytes;            /* dynamic shared memory per CTA at the largest T */
} moe_stats_t;

/* Validate `desc`, record its pointers and choose tile sizes from the device's
 * SM count and shared memory.  Host only: no device allocation, no launch.
 * Errors: INVALID_ARG (null desc/out/pointer, T_max < 1), UNSUPPORTED_SHAPE
 * (H or I not a multiple of 128, E or top_k out of range, tiles do not fit in
 * shared memory, device is not sm_103), MISALIGNED, CUDA (device query failed). */
moe_status_t moe_plan_create(const moe_plan_desc *desc, moe_plan_t *out);

/* Free the plan (host memory only).  NULL is ignored. */
void moe_plan_destroy(moe_plan_t plan);

/* Bytes of device workspace a call with up to T tokens needs (1 <= T <= T_max).
 * The layout is fixed per plan (sized for min(T_max, 4096 / top_k) tokens), so
 * one workspace serves every T the plan accepts.
 * One workspace per stream that runs MoE steps concurrently: two launches
 * sharing a workspace at the same time corrupt each other's counters (the
 * pages' two-stream deadlock, "dsv4-carve" README, trap 3).  The library
 * records an event after each launch on a workspace (moe_decode, moe_prefill,
 * moe_null_step, moe_step_host, moe_group, moe_workspace_init); a launch on
 * another stream while that event is pending is ordered after it (the new
 * stream waits on the event), and a launch while another thread is launching
 * on it from another stream is refused with MOE_ERR_WORKSPACE_BUSY (nothing
 * queued).  Launches being captured into a CUDA graph are not checked: the
 * graph's replays are ordered by whoever launches them.
 * Returns 0 for an invalid plan or T. */
size_t moe_workspace_bytes(moe_plan_t plan, int T);

/* Zero a workspace of `bytes` bytes (>= moe_workspace_bytes(plan, T_max))
 * on `stream`.  Required once after allocation and after any device-side
 * error; the kernels reset their own counters after every successful launch.
 * For a plan that may run a tensor-core kernel (T_max > 1, or the one-token row
 * kernel not available) it also scans every weight block scale once (one
 * launch reading them all) and records MOE_ERR_SCALE in the workspace's error
 * word when one has its sign bit set or is NaN (see `kernel`); moe_check
 * reports it.  ws_dev must be 256-byte aligned.  Ordered after a launch
 * still in flight on the workspace from another stream (see
 * moe_workspace_bytes). */
moe_status_t moe_workspace_init(moe_plan_t plan, void *ws_dev, size_t bytes, void *stream);

/* Grouping only (bit-exact, integer): for the P = T*top_k flat pairs
 * p = t*top_k + j, counts_dev[e] = number of pairs with ids[p] == e,
 * offsets_dev[0..E] = exclusive prefix sum, perm_dev[0..P) = the pair
 * indices with a valid id sorted by (id, p) (stable), then -1 padding.
 * ids outside [0, E) are left out (>= E also sets MOE_ERR_BAD_EXPERT_ID in
 * the workspace error word).  ids_dev int32 [T, top_k]; counts int32 [E];
 * offsets int32 [E+1]; perm int32 [T*top_k].  1 <= T, T*top_k <= 4096. */
moe_status_t moe_group(moe_plan_t plan, const int32_t *ids_dev, int T, void *ws_dev,
                       int32_t *counts_dev, int32_t *offsets_dev, int32_t *perm_dev, void *stream);

/* The routed-experts step for 0 <= T <= 24 tokens (decode; T == 0 is a no-op).
 * Status: MOE_OK (queued), INVALID_ARG, MISALIGNED, NOT_FAST_PATH, CUDA, or
 * WORKSPACE_BUSY (another thread is launching on ws_dev from another stream;
 * nothing queued).  A launch still in flight on ws_dev from another stream is
 * waited for (see moe_workspace_bytes).
 * Device-side outcomes go to the workspace error word (moe_check).
 *   x_dev    bf16 [T, H] row-major, 16-byte aligned; any finite bf16 values:
 *            both kernels prescale each token's row by a power of two before
 *            narrowing it (fp16 mma.sync operands, or FP4 digit rows) and undo
 *            the prescale exactly in their fp32 epilogues
 *   ids_dev  int32 [T, top_k]: id < 0 = empty slot, id >= E = skipped + flagged
 *   w_dev    float [T, top_k] routing weights, used as given
 *   y_dev    float [T, H] row-major, 16-byte aligned; fully written
 *   ws_dev   workspace of moe_workspace_bytes(plan, T) bytes, 256-byte aligned
 * One persistent launch of the kernel the plan's `kernel` field picks for T
 * (grouping, gate/up, SiLU * up, down and the weighted combine all inside it),
 * bitwise identical run to run.  T > 24 is forwarded
 * to moe_prefill unless strict mode is on (then MOE_ERR_NOT_FAST_PATH).
 * No allocation and no synchronisation inside. */
moe_status_t moe_decode(moe_plan_t plan, const void *x_dev, const int32_t *ids_dev, const float *w_dev,
                        float *y_dev, int T, void *ws_dev, void *stream);

/* moe_decode without a caller-supplied workspace, for callers that cannot
 * allocate one: a host runtime whose device memory is fully reserved by its
 * own pool, or code being captured into a CUDA graph where cudaMalloc is not
 * allowed.  The pages have no counterpart: their kernels always take scratch
 * from the caller.
 * Same x_dev, ids_dev, w_dev, y_dev, T and stream as moe_decode
 * (0 <= T <= min(24, T_max)).  The scratch is one library-owned buffer per
 * device of 16 MiB in this library's global memory; a call needs
 * 256 + 16384 + 4*T*(H/64) + 8*T*top_k + 2*T*top_k*I + 6*T*top_k*H
 * + 32*T*top_k*(I/KB) bytes (each piece rounded up to 256; KB = 512 when I is
 * a multiple of 256, else I) and is refused with MOE_ERR_UNSUPPORTED_SHAPE
 * when that exceeds 16 MiB.  Nothing is allocated or freed: each call zeroes the
 * scratch's control block and counters (one memset on `stream`) and launches
 * the decode kernel on it.
 * The first call on each device does the set-up (it looks up the scratch's
 * device address, which may load the module); make that first call before
 * any stream capture.  Every call on a device shares the one buffer, so calls
 * that overlap in time (other streams, other threads, other plans on the
 * same device) would race: a call while the scratch is in flight on another
 * stream is ordered after that call (its stream waits), as for a workspace.
 * check == 0: asynchronous, no synchronisation.  check != 0: synchronise
 * `stream` after the launch and return the device error status (MOE_OK,
 * MOE_ERR_TIMEOUT, MOE_ERR_BAD_EXPERT_ID, MOE_ERR_SCALE or MOE_ERR_RANGE, as
 * moe_check). */
moe_status_t moe_decode_static(moe_plan_t plan, const void *x_dev, const int32_t *ids_dev, const float *w_dev,
                               float *y_dev, int T, int check, void *stream);

/* Layout of the packed input block that moe_step_host copies in one piece,
 * for T tokens: x (bf16 [T, H]) at offset 0, ids (int32 [T, top_k]) at
 * *off_ids, w (float [T, top_k]) at *off_w, each piece starting on a 256-byte
 * boundary.  Returns the block's size in bytes (a multiple of 256), or 0 for
 * a null plan or T outside [1, T_max] (the offsets are then not written).
 * off_ids and off_w may be null.  Host arithmetic only, no CUDA call.  The
 * pages have no counterpart: their step is always called on device buffers. */
size_t moe_io_bytes(moe_plan_t plan, int T, size_t *off_ids, size_t *off_w);

/* The step from host buffers to a host buffer, in one call: one host->device
 * copy of the packed input block, then the step (moe_decode for T <= 24,
 * moe_prefill above), which writes y.  For T = 1 on a plan whose single-token
 * step is the one-token row kernel, and io_host device-addressable (pinned
 * and mapped, as below), there is no copy: that kernel reads x, ids and w from
 * io_host in place with plain loads, and io_dev is not written.  With the
 * plan's pdl flag it then reads them before the previous kernel on the stream
 * has finished (its workspace writes still wait for that kernel), so io_host
 * must not be written by device work queued before the call.  If y_host is page-locked memory that
 * the device can address (cudaHostAlloc, or cudaHostRegister with mapping, on a
 * system with unified addressing), the step's kernels store y into it
 * directly and y_dev is not written.  Otherwise the step writes y_dev, and one
 * device->host copy brings it to y_host.  Everything goes on `stream`, in
 * that order.  There is no synchronisation: y_host holds the result once the
 * stream has passed the step (cudaStreamSynchronize or an event).
 *   io_host  host block of moe_io_bytes(plan, T) bytes, laid out as
 *            moe_io_bytes states.  It should be pinned (cudaHostAlloc or
 *            cudaHostRegister): the copies are then asynchronous.  From
 *            pageable memory they still work, but the runtime stages them
 *            and the call returns later.
 *   io_dev   device block of the same size, 256-byte aligned; after the call,
 *            it holds the copied x, ids and w (unless they were read in place)
 *   y_dev    device float [T, H], 16-byte aligned: the step's output when
 *            y_host is not device-addressable
 *   y_host   host float [T, H], receives y (pinned, like io_host)
 *   T        0 <= T <= T_max (T == 0 is a no-op)
 *   ws_dev   workspace, as for moe_decode
 * Both paths are named paths, so strict mode refuses neither.  The arguments
 * are checked before anything is queued.  A call rejected for its arguments
 * copies nothing and returns the status moe_decode would return.  If the
 * step cannot be launched once the input copy is queued (MOE_ERR_CUDA or
 * MOE_ERR_UNSUPPORTED_SHAPE), that copy stands and y_host is not written.
 * MOE_ERR_CUDA also means a copy could not be queued.  Device-side errors
 * (timeouts, bad ids) go to the workspace error word, as for moe_decode.
 * The caller owns every buffer.  io_host must not be rewritten, and y_host
 * must not be read, before the stream has passed the step. */
moe_status_t moe_step_host(moe_plan_t plan, const void *io_host, void *io_dev, float *y_dev, float *y_host,
                           int T, void *ws_dev, void *stream);

/* The same step for 1 <= T <= T_max (prefill chunks), same arguments.  One
 * launch of the kernel the plan chooses per chunk of at most 4096 / top_k
 * tokens (the tensor-core kernel when the shape allows it and a chunk has
 * more than 8 pairs, else the register kernel). */
moe_status_t moe_prefill(moe_plan_t plan, const void *x_dev, const int32_t *ids_dev, const float *w_dev,
                         float *y_dev, int T, void *ws_dev, void *stream);

/* Measurement variant of moe_decode/moe_prefill: streams exactly the same
 * weight bytes through the same schedule but skips dequantisation and all
 * arithmetic; y receives a checksum (register kernel) or zeros (one-token row
 * kernel), not the step's result (the pages' "null-decode" variant,
 * "LNA-CANON.md", section "lna2 とは").  A single token on a plan that takes
 * the one-token row kernel runs that kernel's schedule; every other launch the
 * register kernel's. */
moe_status_t moe_null_step(moe_plan_t plan, const void *x_dev, const int32_t *ids_dev, const float *w_dev,
                           float *y_dev, int T, void *ws_dev, void *stream);

/* Top-k routing in front of the step.  The pages do not describe the router;
 * this is the plain definition of top-k gating.  For each of the T tokens,
 * ids_dev receives the top_k experts with the largest router logits, in
 * descending order of logit.  Equal logits put the smaller expert index first,
 * and NaN counts as -infinity.  w_dev receives the softmax of those top_k
 * logits (fp32, expf); when the largest selected logit is -infinity the
 * weights are 0, and when it is +infinity the selected +infinity logits
 * share the weight equally (1/their count) and the others get 0.  These are the ids_dev / w_dev that a following moe_decode
 * or moe_prefill on the same stream takes, so routing needs no trip through
 * the host.
 *   logits_dev  float [T, E] row-major, 4-byte aligned
 *   ids_dev     int32 [T, top_k]; w_dev float [T, top_k]; 4-byte aligned
 *   T           0 <= T <= T_max (T == 0 is a no-op)
 * top_k > E is refused with MOE_ERR_UNSUPPORTED_SHAPE.  One launch, one warp
 * per token, asynchronous on `stream`.  With the plan's pdl flag it may start
 * while the previous kernel on the stream drains; it waits for that kernel
 * before it reads or writes anything.  Bitwise reproducible. */
moe_status_t moe_route(moe_plan_t plan, const float *logits_dev, int T, int32_t *ids_dev, float *w_dev,
                       void *stream);

/* Synchronise `stream`, read and clear the workspace's device error word.
 * Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_BAD_EXPERT_ID, MOE_ERR_SCALE or
 * MOE_ERR_RANGE (the first set, in that order: an unreadable scale also makes
 * h non-finite), or MOE_ERR_CUDA.  Not a
 * launch: it does not take part in the workspace's stream check. */
moe_status_t moe_check(moe_plan_t plan, void *ws_dev, void *stream);

/* Test support for the failure path: set every gate/up completion counter in
 * the workspace (of every kernel) to a value no launch reaches, so the next step's bounded
 * dependency waits expire (after the plan's wait limit, 1 s by default or
 * MOE_WAIT_TIMEOUT_MS) and it reports MOE_ERR_TIMEOUT through moe_check
 * instead of hanging.  Re-initialise the workspace afterwards. */
moe_status_t moe_debug_poison_workspace(moe_plan_t plan, void *ws_dev, void *stream);

/* Copy the plan's counters into *out. */
moe_status_t moe_stats(moe_plan_t plan, moe_stats_t *out);

/* Message for the calling thread's last error ("" if none). */
const char *moe_last_error(void);

/* Static name of a status code. */
const char *moe_status_string(moe_status_t s);

/* ABI version the library was built with (MOE_NVFP4_ABI_VERSION). */
int moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
