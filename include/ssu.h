/*
 * ssu.h - C ABI of the GB300 (sm_103a) Mamba2 decode-step selective state update.
 *
 * The operation (operands as in sglang PR #41223, Summary and Details / Kernel measurement:
 * every decode step loads and stores the fp32 SSM state of every request; state pool
 * [pool, H, 64, 128] fp32 with random state_batch_indices; x [bs, H, 64] and B/C [bs, 1, 128]
 * as views into one shared bf16 tensor; dt, A, D and dt_bias broadcast with stride 0).  The pages
 * never print the arithmetic; this library computes the standard Mamba2 decode step:
 *
 *   for each request b (slot s = state_batch_indices[b]) and head h (group g = h / (H/G)):
 *     dtv      = softplus(dt[b,h] + dt_bias[h])            fp32
 *     dA       = exp(dtv * A[h])                           fp32
 *     S[p,n]   = S[p,n] * dA + (dtv * x[b,h,p]) * B[b,g,n]  in place in state_pool[s,h]
 *     out[b,h,p] = bf16_rne( sum_n S[p,n] * C[b,g,n] + D[h] * x[b,h,p] )
 *
 * Types.  The state pool is fp32 or bf16 (ssu_shape_t.state_dtype; either way the update runs
 * in fp32 and a bf16 state is rounded to nearest even when stored).  x, dt, B, C and out are
 * bfloat16, passed as uint16_t pointers to their bit patterns.  dt_bias, A and D are fp32.
 * state_batch_indices is int32 or int64 (ssu_shape_t.index_dtype).  All data pointers are
 * DEVICE pointers on the handle's device (ssu_update_from_host alone takes its per-step
 * operands and readout in page-locked host memory); the caller owns every buffer.  Sizes and
 * strides are in ELEMENTS (not bytes).
 *
 * Streams and asynchrony.  ssu_update validates on the host, then enqueues one kernel on
 * `stream` and returns.  It allocates nothing, copies nothing and never synchronises, so it
 * may be captured in a CUDA graph.  ssu_get_error is the only call that synchronises.
 *
 * Errors.  Every entry point returns an ssu_status_t.  Argument errors are detected on the
 * host before anything is enqueued; ssu_last_error() then holds a one-line explanation
 * (thread-local).  A request whose slot lies outside [0, pool_size) is skipped on the device
 * (its slot and its out rows are not touched) and counted; ssu_get_error reports the count.
 * Duplicate slots within one call are a precondition violation (two requests would update
 * the same state concurrently); they are not detected.  So is any overlap between what a
 * call writes (the named state slots, out, intermediate states) and what it only reads.
 *
 * Threading.  A handle may be used from one host thread at a time.  Calls on different
 * handles are independent.
 */
#ifndef SSU_H
#define SSU_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSU_ABI_VERSION 2

/* Opaque per-device context: holds the device error counters and the launch-shape choice. */
typedef struct ssu_handle_s *ssu_handle_t;

/* The same type as cudaStream_t.  NULL means the legacy default stream. */
typedef struct CUstream_st *ssu_stream_t;

typedef enum {
    SSU_OK = 0,
    SSU_ERR_INVALID_ARG = 1, /* NULL pointer or handle, negative size, H % G != 0, bad stride */
    SSU_ERR_UNSUPPORTED = 2, /* a size or stride form this build does not implement */
    SSU_ERR_MISALIGNED = 3,  /* state_pool base or a state stride not a multiple of 16 bytes */
    SSU_ERR_CUDA = 4,        /* a CUDA runtime call failed; ssu_last_error() names it */
    SSU_ERR_INDEX_OOB = 5    /* ssu_get_error: at least one request was skipped */
} ssu_status_t;

typedef enum { SSU_INDEX_I32 = 0, SSU_INDEX_I64 = 1 } ssu_index_dtype_t;

/* Element type of the state pool (and of the multi-token intermediate states). */
typedef enum { SSU_STATE_F32 = 0, SSU_STATE_BF16 = 1 } ssu_state_dtype_t;

/* Problem sizes of one call. */
typedef struct {
    int64_t batch;       /* bs: requests in this step; 0 is valid and enqueues nothing */
    int64_t nheads;      /* H: 1..65535 */
    int64_t headdim;     /* P >= 1 */
    int64_t dstate;      /* N: 64, 128 or 256 */
    int64_t ngroups;     /* G >= 1 with H % G == 0; head h reads group h / (H / G) */
    int64_t pool_size;   /* slots in state_pool; valid slot ids are [0, pool_size) */
    int32_t index_dtype; /* ssu_index_dtype_t of state_batch_indices */
    int32_t state_dtype; /* ssu_state_dtype_t of state_pool (0 = fp32) */
} ssu_shape_t;

/*
 * Element strides of every operand, outermost dimension first.  Broadcast operands carry the
 * expanded shapes that the model uses (one value per head), with stride 0 over the expanded
 * dimensions; any non-negative outer stride is accepted.
 */
typedef struct {
    int64_t state[4];   /* state_pool [pool, H, P, N]: N-stride must be 1; the other three
                           must be multiples of 16 bytes (4 fp32 or 8 bf16 elements) */
    int64_t x[3];       /* x   [bs, H, P]: P-stride must be 1 */
    int64_t out[3];     /* out [bs, H, P]: P-stride must be 1 */
    int64_t dt[3];      /* dt  [bs, H, P]: P-stride must be 0 (one value per head) */
    int64_t B[3];       /* B   [bs, G, N]: N-stride must be 1 */
    int64_t C[3];       /* C   [bs, G, N]: N-stride must be 1 */
    int64_t dt_bias[2]; /* dt_bias [H, P]: P-stride must be 0 */
    int64_t D[2];       /* D       [H, P]: P-stride must be 0 */
    int64_t A[3];       /* A       [H, P, N]: P- and N-strides must be 0 */
    int64_t idx;        /* state_batch_indices [bs] */
} ssu_strides_t;

/* Launch shapes of the streaming kernel. */
typedef enum {
    SSU_MODE_AUTO = 0,   /* use the built-in table (the default) */
    SSU_MODE_VEC = 1     /* one CTA per tile; 16-byte vector loads/stores through registers */
} ssu_mode_t;

/* A tile is rows_per_warp * warps_per_cta consecutive state rows of one (request, head). */
typedef struct {
    int32_t mode;          /* ssu_mode_t */
    int32_t rows_per_warp; /* rows each warp updates per tile: 1, 2, 4 or 8 (16 for an fp32
                              state of dstate 128) */
    int32_t warps_per_cta; /* 1..16 warps */
    int32_t stages;        /* reserved: ignored (write 0) */
} ssu_launch_t;

/* ABI version this library was built with (SSU_ABI_VERSION). */
int32_t ssu_abi_version(void);

/* Human-readable name of a status code.  Never NULL. */
const char *ssu_status_string(ssu_status_t status);

/* One-line explanation of the last error returned on this host thread ("" if none). */
const char *ssu_last_error(void);

/*
 * Create a handle on CUDA device `device`.  Allocates 16 bytes of device memory for the
 * skipped-request counters and queries the SM count.  Returns SSU_ERR_CUDA without a
 * usable device.  *out is set only on success.
 */
ssu_status_t ssu_create(ssu_handle_t *out, int32_t device);

/* Release the handle and its device memory.  NULL is accepted.  Work enqueued earlier on
 * its streams must have finished (the counters are freed). */
ssu_status_t ssu_destroy(ssu_handle_t handle);

/*
 * Host-side validation of one call, exactly as ssu_update performs it, without a handle or a
 * device: pointers are checked for NULL and alignment only, never dereferenced.
 */
ssu_status_t ssu_validate(const void *state_pool, const void *state_batch_indices,
                          const uint16_t *x, const uint16_t *dt, const float *dt_bias,
                          const float *A, const uint16_t *B, const uint16_t *C, const float *D,
                          const uint16_t *out, const ssu_shape_t *shape,
                          const ssu_strides_t *strides);

/*
 * One decode step.  Reads x, dt, dt_bias, A, B, C, D and the state of every slot in
 * state_batch_indices; writes the updated state back to the same slot and the readout to
 * out.  Enqueued on `stream`; returns once enqueued.  Slots that no request names are never
 * read or written.  See the file header for the arithmetic and the error behaviour.
 */
ssu_status_t ssu_update(ssu_handle_t handle, void *state_pool, const void *state_batch_indices,
                        const uint16_t *x, const uint16_t *dt, const float *dt_bias,
                        const float *A, const uint16_t *B, const uint16_t *C, const float *D,
                        uint16_t *out, const ssu_shape_t *shape, const ssu_strides_t *strides,
                        ssu_stream_t stream);

/*
 * Bytes of device workspace that ssu_update_from_host needs for `shape` (a multiple of 256):
 * dense copies of the call's indices, x, dt, B and C, each section 256-byte aligned.
 * Returns SSU_ERR_INVALID_ARG for a NULL argument or a shape with a negative batch or a
 * dimension below 1.
 */
ssu_status_t ssu_host_workspace_bytes(const ssu_shape_t *shape, int64_t *bytes);

/*
 * One decode step whose per-step operands live in HOST memory: the same step, the same
 * arithmetic and bit-identical results as ssu_update on the same values (sglang PR #41223,
 * Details / Kernel measurement, names the operands; a serving loop produces the indices and
 * activations of each step on the host side of the CPU-GPU link).
 *
 *   state_batch_indices, x, dt, B, C   read from page-locked host memory (cudaHostAlloc or
 *                                      cudaHostRegister), with the layouts and strides of
 *                                      ssu_update; device or managed memory is accepted too
 *   out                                written in page-locked host (or device) memory
 *   state_pool, dt_bias, A, D          device memory, as for ssu_update
 *   workspace                          caller-owned DEVICE buffer, 256-byte aligned, of at
 *                                      least ssu_host_workspace_bytes(shape) bytes
 *
 * The call enqueues two kernels on `stream` and returns: the first reads the step's indices,
 * x, dt, B and C across the link in one pass (every thread one 16-byte vector where the
 * alignment allows) into the workspace; the second is the decode-step kernel of ssu_update,
 * launched as a programmatic dependent of the first, reading the workspace and writing the
 * readout straight into `out`.  No copy-engine transfer is involved.  The readout in host
 * memory is complete once the stream reaches a point after the call (an event or a
 * synchronisation).  The host buffers must stay unchanged, and the workspace unused by other
 * work, until then.  Pageable host memory that is not registered is rejected with
 * SSU_ERR_INVALID_ARG, as is device memory of another device.  Every other argument error
 * and the run-time behaviour (skipped requests counted in the handle) are those of
 * ssu_update.  The launch shape is the handle's forced VEC shape, else the built-in table.
 */
ssu_status_t ssu_update_from_host(ssu_handle_t handle, void *state_pool,
                                  const void *state_batch_indices, const uint16_t *x,
                                  const uint16_t *dt, const float *dt_bias, const float *A,
                                  const uint16_t *B, const uint16_t *C, const float *D,
                                  uint16_t *out, const ssu_shape_t *shape,
                                  const ssu_strides_t *strides, void *workspace,
                                  int64_t workspace_bytes, ssu_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the handle's device counters.
 * *skipped receives the number of requests skipped since the last read (may be NULL);
 * *first_bad receives the smallest skipped request index b, or -1 (may be NULL).
 * Returns SSU_ERR_INDEX_OOB when *skipped > 0, SSU_OK otherwise.
 */
ssu_status_t ssu_get_error(ssu_handle_t handle, ssu_stream_t stream, uint32_t *skipped,
                           int64_t *first_bad);

/*
 * Debug check of a HOST copy of state_batch_indices (it is never read from the device):
 * every id must lie in [0, pool_size) and no id may repeat (two requests naming one slot
 * would update it concurrently, a data race ssu_update does not detect).  Returns SSU_OK, or
 * SSU_ERR_INVALID_ARG with *first_bad (may be NULL) set to the index i of the first entry
 * that is out of range or repeats an earlier one.  Allocates host memory only.
 */
ssu_status_t ssu_check_indices(const void *host_indices, int64_t n, int32_t index_dtype,
                               int64_t pool_size, int64_t *first_bad);

/*
 * Force a launch shape for later ssu_update calls on this handle (for sweeps and tests).
 * NULL, or mode SSU_MODE_AUTO, restores the built-in table.  Every accepted shape computes
 * bit-identical results: each row's readout is summed in one fixed order.
 */
ssu_status_t ssu_set_launch(ssu_handle_t handle, const ssu_launch_t *launch);

/*
 * The same override written as text, for a configuration file or the environment:
 * "rows_per_warp,warps_per_cta" (for example "8,4"), optionally prefixed by the mode name
 * ("vec,8,4").  NULL, "" or "auto" restores the built-in table.  A spec that does not parse,
 * or names a shape ssu_set_launch would refuse, returns SSU_ERR_INVALID_ARG /
 * SSU_ERR_UNSUPPORTED and leaves the handle's choice unchanged.  ssu_create applies the
 * environment variable SSU_LAUNCH, when set, in the same way (and fails if it does not parse).
 */
ssu_status_t ssu_set_launch_override(ssu_handle_t handle, const char *spec);

/* The launch shape ssu_update would use for `shape` on this handle (table or override). */
ssu_status_t ssu_get_launch(ssu_handle_t handle, const ssu_shape_t *shape,
                            ssu_launch_t *launch);

/*
 * Programmatic dependent launch for this handle's VEC and multi-token launches: on
 * (enable != 0, the default for a new handle) or off.  When on, a launch may be scheduled
 * while the previous kernel in the stream is finishing; the kernel's first instruction waits
 * for that kernel to complete and its memory to be visible, so results are unchanged, and
 * each CTA releases its own dependents once its stores are issued.  This hides part of the
 * launch gap between back-to-back kernels (batch 8: 3.75 -> 3.38 us per call).  Work other
 * than a kernel (a copy, an event wait) still completes before the launch starts, as in any
 * stream.  The block copy (ssu_copy_blocks) follows the same setting; the allocation-free
 * entry point never uses it.
 */
ssu_status_t ssu_set_pdl(ssu_handle_t handle, int32_t enable);

/* ---------------------------------------------------------------------------------------
 * Multi-token step: T consecutive tokens of every request in one call, as multi-token
 * speculation verifies them (vLLM PR #48110, Test Plan: speculative decoding with two draft
 * tokens per step).  Token t applies the decode step above to the state left by token t - 1:
 *
 *   for t = 0 .. T-1:
 *     dtv = softplus(dt[b,t,h] + dt_bias[h]);   dA = exp(dtv * A[h])
 *     S[p,n] = S[p,n] * dA + (dtv * x[b,t,h,p]) * B[b,t,g,n]
 *     out[b,t,h,p] = bf16_rne( sum_n S[p,n] * C[b,t,g,n] + D[h] * x[b,t,h,p] )
 *     if intermediate: intermediate[b,t,h,p,n] = S[p,n]        (the state's dtype)
 *   state_pool[s,h] = S
 *
 * The state is read once and written once per call, whatever T; with T = 1 and no
 * intermediate buffer the result is bit-identical to ssu_update.
 */

/* Token strides (elements) of the per-token operands, and the optional intermediate buffer. */
typedef struct {
    int64_t x, out, dt, B, C;  /* stride of the token index t in x, out, dt, B and C; the
                                  other strides come from ssu_strides_t */
    int64_t intermediate[5];   /* [bs, T, H, P, N]: N-stride 1, the others multiples of 16
                                  bytes */
} ssu_token_strides_t;

#define SSU_MAX_TOKENS 64

/*
 * T consecutive decode steps (1 <= T <= SSU_MAX_TOKENS).  Pointers, shape and ssu_strides_t as
 * for ssu_update (describing token 0), plus `tokens` = T, the token strides, and
 * `intermediate` (device buffer of the state's dtype, 16-byte aligned, or NULL for none).
 * Within a call the running state stays in fp32; a bf16 state is rounded only when written.
 * Same error behaviour as ssu_update; enqueued on `stream`; allocates and synchronises
 * nothing.  B and C are read as whole 4- or 8-byte column groups when their base and strides
 * allow it, element by element otherwise (same results either way).  T = 1 without an
 * intermediate buffer runs as ssu_update.
 *
 * Two forms compute the step.  With an intermediate buffer, with a forced launch shape, and
 * for short runs, the tokens are applied one after another as written above.  Without an
 * intermediate buffer, runs of 5 tokens or more on an fp32 state (16 or more on a bf16 state
 * at dstate 128) with dstate 64 or 128, headdim a multiple of 8, and B, C and x 16-byte aligned
 * with strides in multiples of 8 elements take the chunked matrix form: the same
 * recurrence rewritten per chunk of up to 8 tokens through the running product of dA, on
 * tensor-core MMAs with fp32 operands split into two tf32 parts.  Its values are the same real
 * numbers rounded in another order: within the same tolerance of an exact evaluation, but not
 * bit-identical to the token-by-token form.  Each form gives the same bits for the same
 * inputs whatever the launch shape.
 */
ssu_status_t ssu_update_tokens(ssu_handle_t handle, void *state_pool,
                               const void *state_batch_indices, const uint16_t *x,
                               const uint16_t *dt, const float *dt_bias, const float *A,
                               const uint16_t *B, const uint16_t *C, const float *D,
                               uint16_t *out, void *intermediate, const ssu_shape_t *shape,
                               const ssu_strides_t *strides, int64_t tokens,
                               const ssu_token_strides_t *token_strides, ssu_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * State-block copy (vLLM PR #48110, Purpose and Test Plan / Microbenchmark): under prefix
 * caching and multi-token speculation a request's recurrent states are copied from one cache
 * block to another, for every state tensor of the model (one temporal fp32 state and one conv
 * state per hybrid layer).  One call copies, for every request i and every described tensor,
 * block src_idx[i] to block dst_idx[i] of that tensor.  Bytes are copied verbatim.
 */

/* One state tensor viewed as blocks: block k is block_bytes bytes at base + k * stride. */
typedef struct {
    void *base;                 /* device pointer, 16-byte aligned */
    int64_t block_bytes;        /* bytes copied per block: > 0, a multiple of 16 */
    int64_t block_stride_bytes; /* distance between blocks: a multiple of 16, >= block_bytes */
    int64_t num_blocks;         /* valid block ids are [0, num_blocks) */
} ssu_block_tensor_t;

#define SSU_COPY_MAX_TENSORS 64

typedef enum {
    SSU_COPY_AUTO = 0,  /* built-in choice */
    SSU_COPY_VEC = 1    /* 16-byte vector loads and stores through registers */
} ssu_copy_mode_t;

typedef struct {
    int32_t mode;        /* ssu_copy_mode_t */
    int32_t chunk_kib;   /* bytes per work item, KiB: 4, 8, 16, 32 or 64 */
    int32_t stages;      /* 16-byte vectors per thread per pass: 1, 2, 4, 8 or 16 */
    int32_t threads;     /* threads per CTA, 32..256 (multiple of 32) */
} ssu_copy_launch_t;

/*
 * Copy block src_idx[i] -> block dst_idx[i] of each of the `num_tensors` tensors (host array,
 * at most SSU_COPY_MAX_TENSORS), for i in [0, n).  src_idx and dst_idx are device int32 or
 * int64 arrays (index_dtype) of n entries.  A request whose src or dst id is out of a tensor's
 * range is skipped for every tensor and counted (ssu_get_error).  Preconditions (not checked):
 * the dst ids are distinct and no dst id equals a src id of the same call (the copies run
 * concurrently).  Enqueued on `stream`; allocates and synchronises nothing.  Errors: NULL or
 * misaligned pointers, sizes or strides that are not multiples of 16 -> SSU_ERR_MISALIGNED /
 * SSU_ERR_INVALID_ARG before anything is enqueued.
 */
ssu_status_t ssu_copy_blocks(ssu_handle_t handle, const ssu_block_tensor_t *tensors,
                             int32_t num_tensors, const void *src_idx, const void *dst_idx,
                             int64_t n, int32_t index_dtype, ssu_stream_t stream);

/* Force a launch shape for later ssu_copy_blocks calls on this handle (NULL or mode AUTO
 * restores the built-in choice).  All shapes copy the same bytes. */
ssu_status_t ssu_copy_set_launch(ssu_handle_t handle, const ssu_copy_launch_t *launch);

/*
 * Allocation-free variant of ssu_update.  No counterpart exists in the paper: it serves
 * callers that cannot call cudaMalloc, such as code running under an allocator that must not
 * be re-entered, or a runtime that hands out only memory it owns, and so cannot create a
 * handle (ssu_create allocates the device counters).  It takes no handle and allocates
 * nothing: the skipped-request counters the kernel needs live in a fixed 256-byte array in
 * the library's device memory (SSU_STATIC_SCRATCH_BYTES, held by every GPU that loads the
 * library until the process exits).
 *
 * Arguments are those of ssu_update, on the CURRENT CUDA device, plus:
 *   counters_out  optional caller-owned DEVICE buffer of 3 uint32: after the kernel the call
 *                 enqueues a copy of [skipped requests, smallest skipped request index
 *                 (0xFFFFFFFF if none), 0 (reserved)]; NULL skips the copy.
 * Each call clears the shared counters, launches the VEC kernel of the built-in table and
 * copies the counters out, all on `stream`.  Every call looks up the array's device address
 * on the current device (cudaGetSymbolAddress, with that device current) and fails with
 * SSU_ERR_CUDA if the lookup does; nothing is cached, so the address stays right after a
 * device reset.  The first call on a device also loads the library's device code there: make
 * that first call before any stream capture.  Every call on a device shares the one array:
 * calls that overlap on the GPU (different streams, no ordering) race on the counters, so
 * order them.
 * Batches above SSU_STATIC_MAX_BATCH requests are rejected with SSU_ERR_UNSUPPORTED (the
 * smallest skipped index is kept in one 32-bit word of the array).  Never calls cudaMalloc,
 * cudaFree or any allocating routine.
 */
#define SSU_STATIC_SCRATCH_BYTES 256
#define SSU_STATIC_MAX_BATCH 2147483647LL
ssu_status_t ssu_update_static(void *state_pool, const void *state_batch_indices,
                               const uint16_t *x, const uint16_t *dt, const float *dt_bias,
                               const float *A, const uint16_t *B, const uint16_t *C,
                               const float *D, uint16_t *out, const ssu_shape_t *shape,
                               const ssu_strides_t *strides, uint32_t *counters_out,
                               ssu_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSU_H */
