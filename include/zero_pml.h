/*
 * zero_pml.h -- C ABI of the ZeRO partitioned mixed-precision optimizer step
 * for NVIDIA GB300 (sm_103a).
 *
 * The library does the per-rank part of a ZeRO data-parallel training step:
 * the model states are flattened and partitioned over Nd ranks, and for one
 * rank's shard hand-written CUDA kernels run the mixed-precision AdamW update
 * with dynamic loss scaling and global gradient-norm clipping.
 *
 * Sources (web pages on ZeRO / DeepSpeed):
 *   [ZeRO card] "ZeRO: Memory Optimizations Toward Training Trillion
 *               Parameter Models - 中文验证版" (ai-papers.xuzou.cn/zh/papers/zero_2019/),
 *               sections 瓶颈 (bottleneck), 方法适配 (method), 证据 (evidence).
 *   [DS news]   DeepSpeed release news (lxsoso.com/blog/19320.html).
 *   [ZeRO-2]    "探秘微软大规模人工智能的新框架 ZeRO-2" (infoq.cn).
 * The update equations, which the pages do not print, are Adam (Kingma & Ba
 * 2015) with decoupled weight decay (Loshchilov & Hutter 2019) and dynamic
 * loss scaling (Micikevicius et al. 2018).
 *
 * Conventions for every entry point:
 *   - Returns ZERO_OK (0) or a negative ZERO_E* code; zero_strerror() names
 *     it.  Arguments are checked on the host before anything is enqueued: a
 *     call that returns an argument error has launched nothing and changed
 *     nothing.  No C++ exception crosses the ABI.
 *   - The caller owns all memory.  The library never allocates device
 *     memory; it works in caller-provided device buffers and a caller-provided
 *     device workspace (see zero_workspace_bytes).  Calls that copy a table
 *     into the workspace (lists of arrays, the parameter gather, the 1-bit
 *     server) stage it through two pinned host buffers per device that the
 *     library allocates on first use and keeps until the process exits.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Device work is enqueued asynchronously on it, on the calling
 *     thread's current CUDA device; no call synchronises the host (a table
 *     copy may wait for the copy two table copies earlier to have finished)
 *     except zero_workspace_stalls, whose job is to read a device count.
 *   - Device arrays must start on a 16-byte boundary (ZERO_EALIGN otherwise);
 *     any element count is accepted, including 0 and counts of 2^31 and more.
 *   - Element types: ZERO_F16 (IEEE binary16), ZERO_BF16 (bfloat16),
 *     ZERO_F32 (IEEE binary32).
 *   - CUDA graphs.  A call whose device work is kernels alone may be issued
 *     while `stream` is being captured; the graph then holds the pointers,
 *     sizes and hyperparameters of the captured call, while the device state
 *     (loss scale, step count, the norm) moves on at every replay exactly as
 *     it would over the same calls issued one by one.  These are: zero_step,
 *     zero_adam_step and zero_grad_norm_overflow on one array per list (a
 *     flat shard), zero_step_prepared (any list), zero_accumulate_grads,
 *     zero_accumulate_grads_norm, zero_reduce_grads,
 *     zero_grad_norm_overflow_static (after a first call outside capture),
 *     zero_gather_params / zero_scatter_params with at most 64 tensors and
 *     256 shards, zero_onebit_worker, zero_onebit_server with at most 256
 *     workers, and zero_onebit_update.  A call that would copy a host-built
 *     table (a list of several arrays, a larger gather or server) returns
 *     ZERO_ECAPTURE under capture, having enqueued nothing: a captured copy
 *     would read the staging buffer when the graph is replayed, after later
 *     calls have reused it.  Issue those calls outside capture (for a list
 *     step: prepare it outside, then capture zero_step_prepared).
 */
#ifndef ZERO_PML_H
#define ZERO_PML_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ codes */

#define ZERO_OK 0
#define ZERO_EINVAL (-1)     /* a required pointer is NULL, or a bad flag/count */
#define ZERO_EALIGN (-2)     /* a device array does not start on 16 bytes */
#define ZERO_EDTYPE (-3)     /* an element type that this argument does not take */
#define ZERO_ESIZE (-4)      /* element counts that do not match across lists */
#define ZERO_EWORKSPACE (-5) /* workspace NULL or smaller than required */
#define ZERO_ECAPACITY (-6)  /* an output array is too small (see *n_frags) */
#define ZERO_ECUDA (-7)      /* the CUDA runtime reported an error */
#define ZERO_ELAYOUT (-8)    /* nd < 1, align < 1 or not a power of two */
#define ZERO_ECAPTURE (-9)   /* a table copy asked for while the stream is captured */

#define ZERO_F16 0
#define ZERO_BF16 1
#define ZERO_F32 2

/* Pointer checks: every device pointer of a call is checked to be memory
 * the kernels may reach (cudaPointerGetAttributes), except in lists of more
 * than 64 arrays, where the first and the last array are checked (so that
 * the host cost of a call does not grow with the list). */

/* Text of a ZERO_* code; for ZERO_ECUDA, the last CUDA error seen by this
 * library on the calling thread is appended.  Never NULL.  The string stays
 * valid until the next call on the same thread. */
const char *zero_strerror(int code);

/* ------------------------------------------------------------------ layout */

/* One piece of a tensor inside one rank's shard. */
typedef struct zero_frag {
    int64_t tensor;        /* index in the tensor list */
    int64_t tensor_offset; /* first element of the piece, within the tensor */
    int64_t rank;          /* owning rank, 0 .. nd-1 */
    int64_t shard_offset;  /* first element of the piece, within that rank's shard */
    int64_t length;        /* elements in the piece (> 0) */
} zero_frag_t;

/* The flat partition of the model states over nd data-parallel ranks
 * ([ZeRO card §方法适配]: states are split across DP ranks, not replicated).
 *
 * The tensors (numel[0..n_tensors-1] elements each) are concatenated in list
 * order into one flat buffer; its length is padded at the tail up to a
 * multiple of nd*align; rank r owns the contiguous shard [r*S, (r+1)*S) with
 *     S = ceil(total / (nd*align)) * align.
 * A tensor that straddles a shard boundary is cut there.  The same layout
 * serves every state (fp16 params/grads, fp32 master/momentum/variance), so
 * one rank's shard of each is one contiguous array of S elements.
 *
 * Host only (no device work).  Outputs: *shard_numel = S, *padded_total =
 * nd*S, tensor_offset[i] = flat offset of tensor i (array of n_tensors, may
 * be NULL), frags[0..] the pieces in flat order (may be NULL when frag_cap is
 * 0).  *n_frags always receives the number of pieces; if it exceeds frag_cap,
 * the first frag_cap are written and ZERO_ECAPACITY is returned.
 * Errors: ZERO_EINVAL (numel NULL with n_tensors > 0, negative numel or
 * n_tensors, NULL outputs), ZERO_ELAYOUT (nd < 1, align < 1 or not a power of
 * two, or a padded total past 2^62). */
int zero_partition_layout(const int64_t *numel, int64_t n_tensors, int32_t nd, int64_t align,
                          int64_t *shard_numel, int64_t *padded_total, int64_t *tensor_offset,
                          zero_frag_t *frags, int64_t frag_cap, int64_t *n_frags);

/* ------------------------------------------------------------------ state */

/* Per-rank optimizer state that lives in device memory (64 bytes, 8-byte
 * aligned).  The first two fields are the step's partial reduction: on a
 * multi-rank run they are the 16 bytes to sum over the ranks between
 * zero_grad_norm_overflow and zero_adam_step. */
typedef struct zero_state {
    double sumsq;         /* sum of squares of the unscaled gradient, this step */
    double found_inf;     /* > 0 if any gradient element was +-inf or NaN */
    double loss_scale;    /* S: gradients arrive multiplied by S (a power of two) */
    int64_t step;         /* t: steps applied so far (skipped steps excluded) */
    int64_t good_steps;   /* clean steps since the scale last changed */
    int64_t skipped;      /* total skipped steps */
    double last_norm;     /* global L2 norm of the unscaled gradient, last step */
    float last_clip;      /* clip coefficient applied by the last step (1 = none) */
    int32_t last_skipped; /* 1 if the last step was skipped */
} zero_state_t;

/* Fills a HOST zero_state_t for a fresh optimizer: zero moments counters,
 * the given initial loss scale (a power of two, >= 1).  Copy it to the
 * device state buffer before the first step.  Errors: ZERO_EINVAL. */
int zero_state_init(zero_state_t *host_state, double initial_loss_scale);

/* AdamW and loss-scaler settings, read on the host at each zero_adam_step. */
typedef struct zero_hparams {
    double lr, beta1, beta2, eps, weight_decay;
    double max_norm;      /* global-norm clip threshold; <= 0 turns clipping off */
    double min_scale;     /* floor of the loss scale on overflow (a power of two >= 1) */
    int64_t scale_window; /* clean steps in a row before the scale doubles (>= 1) */
} zero_hparams_t;

/* ------------------------------------------------------------------ lists */

/* A list of n device arrays of one element type: ptrs[i] holds numel[i]
 * elements.  ptrs and numel are HOST arrays; ptrs[i] are device pointers.
 * A flat shard is a list of one array. */
typedef struct zero_tlist {
    void *const *ptrs;
    const int64_t *numel;
    int64_t n;
    int32_t dtype;
} zero_tlist_t;

/* Bytes of device workspace that zero_grad_norm_overflow, zero_adam_step,
 * zero_step and zero_list_prepare need for lists of up to max_tensors arrays
 * holding up to max_total_numel elements in all -- one rank's partition of
 * the model states ([ZeRO card §方法适配]), flat or as its tensors -- and
 * that zero_accumulate_grads_norm and zero_reduce_grads need for one array
 * of n elements (the 1-bit Adam calls: zero_workspace_bytes(Nd, Nd * S)).
 * It holds the reduction ticket and partials, the step's binary32 scalars
 * and a list's tables.  The workspace must start on a 256-byte boundary (as
 * cudaMalloc and PyTorch allocations do) and be zero-filled before its first
 * use; each call leaves its reduction counter at zero again.  One workspace
 * must not be used by two calls that may run at the same time (two streams).
 * Device pointers passed to the library must be device (or managed) memory
 * (ZERO_EINVAL otherwise; see "Pointer checks" above). */
size_t zero_workspace_bytes(int64_t max_tensors, int64_t max_total_numel);

/* Waits that gave up.  Pass 1 over a large flat shard stages the gradient
 * through shared memory with bulk copies and waits for each to land; a wait
 * that has not ended after 1 s gives up rather than hang the GPU: that call
 * then reports the gradient as non-finite (found_inf > 0, so the step is
 * skipped) and adds one to a count kept in the workspace.  This call copies
 * that count (every wait that gave up since the workspace was zero-filled)
 * into *stalls.  It is the one call that waits for the GPU: it returns once
 * `stream` has reached the copy (so it cannot be issued while `stream` is
 * being captured into a graph: ZERO_ECUDA).  ws: a device workspace as
 * above; stalls: host.  Errors: ZERO_EINVAL (NULL argument, ws not device
 * memory), ZERO_EALIGN (ws not on a 256-byte boundary), ZERO_ECUDA. */
int zero_workspace_stalls(const void *ws, uint32_t *stalls, void *stream);

/* ------------------------------------------------------------------ calls */

/* Gradient accumulation over micro-batches ([DS news]: the engine manages
 * gradient accumulation):
 *     acc[i] = (overwrite ? 0 : acc[i]) + g_0[i] + g_1[i] + ... + g_{n_bufs-1}[i]
 * summed in binary32 in micro-batch order (with overwrite the sum starts
 * from g_0[i]).  acc: device fp32[n]; g: HOST array of n_bufs device
 * pointers to arrays of `dtype` (F16, BF16 or F32) with n elements;
 * 1 <= n_bufs <= 8.  Errors: ZERO_EINVAL, ZERO_EDTYPE, ZERO_EALIGN,
 * ZERO_ECUDA. */
int zero_accumulate_grads(float *acc, const void *const *g, int32_t n_bufs, int32_t dtype,
                          int64_t n, int32_t overwrite, void *stream);

/* zero_accumulate_grads followed by zero_grad_norm_overflow on acc, in one
 * pass: the same accumulated sums (stored in acc), and the squared norm and
 * overflow of the stored sums folded into d_state as pass 1 over acc would
 * (loss scale from d_state; accumulate as there).  The sums are not read
 * back, so the step moves 4 bytes per element less (12 + 0 instead of
 * 12 + 4 with four 16-bit micro-batches).  d_state: device zero_state_t; ws
 * as for zero_grad_norm_overflow (one array of n elements).  Errors: as
 * zero_accumulate_grads, plus ZERO_EWORKSPACE. */
int zero_accumulate_grads_norm(float *acc, const void *const *g, int32_t n_bufs, int32_t dtype, int64_t n,
                               int32_t overwrite, zero_state_t *d_state, int32_t accumulate, void *ws,
                               size_t ws_bytes, void *stream);

/* Pass 1: unscale + overflow detection + squared norm.
 * [ZeRO card §瓶颈]: mixed-precision training keeps an fp16 gradient beside
 * the fp32 optimizer state; [DS news]: the engine manages mixed precision.
 * The pages print no arithmetic for it; the reading is dynamic loss scaling
 * (Micikevicius et al. 2018, section 3.2: the gradient arrives multiplied by
 * the loss scale S; any inf/NaN in it skips the step) and global
 * gradient-norm clipping, whose norm is taken here.
 * For g = float(grad) / S over every element of `grads` (F16, BF16 or F32),
 * computes sum g^2 and whether any element is +-inf or NaN.  The squares are
 * summed in binary32 over at most 32 elements, then in binary64, in a fixed
 * order (the result is the same bit for bit on every run); for BF16 and F32
 * data a group of 8 whose binary32 square sum would overflow or fall below
 * binary32's normal range is summed in binary64 instead, so every finite
 * gradient gives a finite norm within 1e-6 of the exact one.
 * S is read from d_state: the call takes no loss-scale argument, because the
 * scale lives on the device and changes there (halved on an overflow,
 * doubled after a clean run) without the host ever reading it back.  With
 * accumulate = 0 the results are written to d_state->sumsq / found_inf; with
 * accumulate = 1 they are added, so that several calls (e.g. the Nd shards
 * of a layout on one GPU) fold into one global norm and overflow flag.
 * d_state: device zero_state_t.
 * ws: device workspace of ws_bytes >= zero_workspace_bytes(grads->n, total).
 * Errors: ZERO_EINVAL, ZERO_EDTYPE, ZERO_EALIGN, ZERO_EWORKSPACE, ZERO_ECUDA. */
int zero_grad_norm_overflow(const zero_tlist_t *grads, zero_state_t *d_state,
                            int32_t accumulate, void *ws, size_t ws_bytes, void *stream);

/* ZeRO stage 2 on one rank ([ZeRO card §方法适配]: stage 2 partitions the
 * gradients; each rank keeps only the reduced gradient of its shard, which
 * the data-parallel reduce-scatter delivers): the reduction of the Nd
 * replicas' slices of this rank's shard fused with pass 1.
 *     out[i] = round( (replica_0[i] + ... + replica_{Nd-1}[i]) / Nd )
 * summed in binary32 in rank order, one IEEE division, rounded to nearest
 * even into out_dtype (F32 output stored as is); then pass 1 over the stored
 * out, exactly as zero_grad_norm_overflow would compute it (loss scale from
 * d_state; accumulate as there).  On one GPU this is the arithmetic of the
 * reduce-scatter with the replicas in local memory.  replicas: HOST array of
 * n_replicas (1..64) device pointers, n elements of `dtype` each; out: device,
 * n elements of out_dtype.  ws as for zero_grad_norm_overflow (one array).
 * Errors: ZERO_EINVAL, ZERO_EDTYPE, ZERO_EALIGN, ZERO_EWORKSPACE, ZERO_ECUDA. */
int zero_reduce_grads(const void *const *replicas, int32_t n_replicas, int32_t dtype, int64_t n, void *out,
                      int32_t out_dtype, zero_state_t *d_state, int32_t accumulate, void *ws, size_t ws_bytes,
                      void *stream);

/* Pass 1 without a workspace: the same computation and results as
 * zero_grad_norm_overflow, for callers that cannot allocate device memory
 * and so cannot provide the workspace -- code running where another
 * component owns all device memory (a training framework whose caching
 * allocator has reserved the GPU, a plugin host that hands its plugins only
 * their input and output buffers) or code that must keep the step's memory
 * footprint fixed.  The ZeRO pages have no counterpart of this call: it is
 * an interface convenience of this library.
 *
 * The scratch (a reduction ticket and per-block partials, 16,640 bytes) is a
 * static device array inside the library; every GPU on which the library is
 * loaded holds it until the process exits.  The first call on a device looks
 * up that array's device address (with the device current) and caches it
 * with the identity of the current context; make that first call before any
 * stream capture.  A device reset replaces the context, and the next call
 * after one looks the address up again (so make that call outside capture
 * too).  Every pointer of the list is checked to be device memory.  Each call
 * resets the ticket on `stream` before its kernel.  All calls share the one array and
 * it keeps the last call's contents, so calls that can overlap on the GPU
 * (different streams, or several host threads) race and must not be issued.
 * Limit: at most 32 arrays in `grads` (any lengths); a longer list returns
 * ZERO_ECAPACITY.  Allocates nothing (no cudaMalloc / cudaFree).
 * Errors: as zero_grad_norm_overflow, plus ZERO_ECAPACITY. */
int zero_grad_norm_overflow_static(const zero_tlist_t *grads, zero_state_t *d_state,
                                   int32_t accumulate, void *stream);

/* Pass 2 (preceded by a decision kernel of one small block): the step.
 * [ZeRO card §瓶颈]: mixed-precision Adam keeps an fp16 parameter and
 * gradient plus an fp32 parameter copy, momentum and variance (16 bytes per
 * parameter); [ZeRO card §方法适配]: each data-parallel rank updates only its
 * own partition of that state.  The update itself, which the pages do not
 * print, is read as Adam (Kingma & Ba 2015) with decoupled weight decay
 * (Loshchilov & Hutter 2019), dynamic loss scaling (Micikevicius et al.
 * 2018, section 3.2) and global gradient-norm clipping.
 * From d_state's global sumsq / found_inf (left there by
 * zero_grad_norm_overflow, summed over ranks if there are several):
 *   - found_inf > 0: the step is skipped -- no state array, p_lp or t is
 *     touched -- and loss_scale = max(loss_scale / 2, min_scale);
 *   - otherwise t += 1, the scale doubles after scale_window clean steps in a
 *     row, and every element is updated in binary32 (no FMA contraction):
 *         g  = float(grad) * (1/S);  g = g * clip   (clip = max_norm / (norm + 1e-6) when < 1)
 *         m  = b1*m + (1-b1)*g;      v = b2*v + (1-b2)*(g*g)
 *         p  = p - (lr/(1-b1^t) * m / (sqrt(v) * (1/sqrt(1-b2^t)) + eps) + lr*wd*p)
 *         p_lp = p rounded to nearest even
 *     with every scalar computed in binary64 and rounded once to binary32.
 * sumsq and found_inf are reset to 0; last_norm, last_clip, last_skipped are
 * set.  grads: F16, BF16 or F32; master, m, v: F32; p_lp: F16 or BF16, or
 * NULL for no low-precision copy.  master, m and v may be pinned HOST memory
 * (cudaHostAlloc / cudaHostRegister) instead of device memory: the GPU then
 * streams the optimizer state over the host link (NVLink-C2C on GB300) while
 * the gradient and the fp16 parameters stay in HBM -- the ZeRO-Offload
 * memory split with the update still computed by the GPU.  All lists must have the same n and the
 * same numel per entry.  hp: host.  ws as for zero_grad_norm_overflow.
 * Errors: ZERO_EINVAL, ZERO_EDTYPE, ZERO_EALIGN, ZERO_ESIZE, ZERO_EWORKSPACE,
 * ZERO_ECUDA. */
int zero_adam_step(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                   const zero_tlist_t *v, const zero_tlist_t *p_lp, const zero_hparams_t *hp,
                   zero_state_t *d_state, void *ws, size_t ws_bytes, void *stream);

/* One whole step of a single-rank shard in one call: zero_grad_norm_overflow
 * (accumulate = 0) followed by zero_adam_step on the same lists, with the
 * same results bit for bit.  Use it when no cross-rank sum has to happen
 * between the passes ([ZeRO card §方法适配]: each rank updates its own
 * partition; with one rank, or when the norm and overflow of this shard
 * alone decide the step).  For a non-empty list the last block of pass 1
 * takes the decision (no decision kernel) and pass 2 is scheduled while
 * pass 1 drains.  Arguments and errors as zero_adam_step. */
int zero_step(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
              const zero_tlist_t *v, const zero_tlist_t *p_lp, const zero_hparams_t *hp,
              zero_state_t *d_state, void *ws, size_t ws_bytes, void *stream);

/* A prepared step: the tables of a list of arrays built and copied into the
 * workspace once, for steps that then copy nothing from the host.
 *
 * zero_list_prepare checks the lists as zero_adam_step does, copies the list's
 * table into `ws` (stream-ordered on `stream`) and fills *plan (a HOST struct
 * the caller keeps; its fields are the library's).  zero_step_prepared then
 * runs zero_step over those lists from the resident table: pass 1, the
 * decision and pass 2, with the results of zero_step bit for bit.  It copies
 * nothing from the host, so it can be captured into a CUDA graph (the plan
 * itself cannot be prepared under capture: ZERO_ECAPTURE), and its host cost
 * does not grow with the number of arrays.  The arrays, their sizes and
 * their element types are fixed at preparation; their contents change
 * between steps as usual.  While a plan is in use its workspace serves that
 * plan alone: a call that copies another table into it, or keeps block
 * partials in its table region (zero_reduce_grads, the gather and the 1-bit
 * server), overwrites the plan's table.  `ws` must be the workspace the plan
 * was prepared in (ZERO_EINVAL otherwise).  A one-array list is accepted
 * (the plan then holds its five pointers).  Errors: as zero_adam_step, plus
 * ZERO_ECAPTURE from zero_list_prepare. */
typedef struct zero_list_plan {
    const void *ws;                         /* the workspace holding the table */
    const void *ents, *tiles, *chunks;      /* the table's parts in ws (device) */
    void *one[5];                           /* a one-array list: grad, master, m, v, p_lp */
    int64_t n, total, n_tiles, n_chunks;    /* arrays, elements, work items of pass 2 and pass 1 */
    int32_t gdtype, pdtype;                 /* element types; pdtype -1: no low-precision copy */
    int32_t aligned32, reserved;
} zero_list_plan_t;

int zero_list_prepare(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                      const zero_tlist_t *v, const zero_tlist_t *p_lp, void *ws, size_t ws_bytes,
                      zero_list_plan_t *plan, void *stream);
int zero_step_prepared(const zero_list_plan_t *plan, const zero_hparams_t *hp, zero_state_t *d_state, void *ws,
                       size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ offload */

/* ZeRO-Offload with the update on the host cores (DeepSpeed release news,
 * lxsoso.com/blog/19320.html: ZeRO-Offload extends ZeRO-2 with CPU memory, so
 * that one GPU trains a model about ten times larger).  (On GB300 the faster
 * split keeps the state in pinned host memory and lets zero_step /
 * zero_adam_step stream it over NVLink-C2C; these calls serve hosts whose
 * link is too slow for that.)  The fp32 master, momentum and variance live in
 * HOST memory and the host cores update them;
 * the GPU computes pass 1 (zero_grad_norm_overflow) on its fp16 gradient and
 * keeps the fp16 parameters.  A step: pass 1 on the GPU; copy the gradient
 * and the zero_state_t to the host; zero_offload_decide on the host state;
 * zero_offload_apply (whole arrays or chunk by chunk, as the gradient
 * arrives); copy the low-precision parameters and the state back.  The
 * results are those of zero_adam_step bit for bit (same binary32 expression,
 * same binary64 step scalars). */

/* The binary32 scalars of one step's element update (host). */
typedef struct zero_offload_scalars {
    float inv_scale, clip;
    float beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
    float step_size;    /* lr / (1 - beta1^t) */
    float inv_sqrt_bc2; /* 1 / sqrt(1 - beta2^t) */
    float lr_wd;        /* lr * weight_decay */
    int32_t skip;       /* 1: the step is skipped, apply does nothing */
    int32_t reserved;
} zero_offload_scalars_t;

/* The step decision of zero_adam_step on a HOST zero_state_t whose sumsq and
 * found_inf hold the step's global values: skip or apply, loss scale, step
 * count, last norm / clip / skip, and the element scalars in *out.  Resets
 * sumsq and found_inf.  Errors: ZERO_EINVAL. */
int zero_offload_decide(zero_state_t *host_state, const zero_hparams_t *hp, zero_offload_scalars_t *out);

/* The element update of zero_adam_step on HOST arrays of n elements, on
 * n_threads host threads (a persistent pool; the calling thread is one of
 * them): grad (F16, BF16 or F32), master, m, v (fp32, updated in place),
 * p_lp (F16 or BF16, or NULL).  Any alignment; chunks of one step may be
 * applied by separate calls.  Does nothing when sc->skip is set.
 * Errors: ZERO_EINVAL, ZERO_EDTYPE. */
int zero_offload_apply(const void *grad, int32_t gdtype, float *master, float *m, float *v, void *p_lp,
                       int32_t pdtype, int64_t n, const zero_offload_scalars_t *sc, int32_t n_threads);

/* memcpy of `bytes` host bytes on n_threads threads of the same pool, for
 * staging and for measuring the host-memory bandwidth the apply runs
 * against.  Errors: ZERO_EINVAL. */
int zero_offload_copy(void *dst, const void *src, size_t bytes, int32_t n_threads);

/* ------------------------------------------------------------------ stage 3: parameter gather */

/* ZeRO stage 3 partitions the parameters as well ("ZeRO: Memory Optimizations
 * Toward Training Trillion Parameter Models - 中文验证版", section 方法适配):
 * a rank keeps only its shard of the flat parameter buffer and assembles a
 * tensor -- or a whole layer, one at a time, as the ZeRO-Infinity page's
 * memory-centric tiling does -- from the ranks' shards before using it.
 * These calls are the data movement of that gather and of its inverse on one
 * GPU, where the Nd shards are Nd device arrays; with several GPUs it is the
 * all-gather of a collective library.
 *
 * The flat buffer is the concatenation of the Nd shards in rank order
 * (nd * shard_numel elements, the layout of zero_partition_layout), and a
 * tensor i covers its flat elements [tensor_offset[i], tensor_offset[i] +
 * numel[i]).  Elements are copied bit for bit (no conversion); the element
 * type is the list's (F16, BF16 or F32) and the shards hold the same type.
 *
 *   shards         HOST array of nd DEVICE pointers, shard r holding
 *                  shard_numel elements; each 16-byte aligned.
 *   tensors        the tensors (zero_tlist_t; device arrays, 16-byte
 *                  aligned; any element counts).
 *   tensor_offset  HOST array of tensors->n flat offsets.
 *   ws             device workspace of at least
 *                  zero_gather_workspace_bytes(tensors->n, nd) bytes,
 *                  256-byte aligned; the call copies its tables there in
 *                  stream order, so one workspace must not serve two calls
 *                  that can run at the same time.
 * Tensors must not overlap one another or a shard in memory.  Work is
 * enqueued on `stream`; nothing is synchronised.
 * Errors: ZERO_EINVAL (NULL or negative arguments, memory that is not device
 * memory), ZERO_EALIGN, ZERO_EDTYPE, ZERO_ELAYOUT (a tensor's range outside
 * [0, nd * shard_numel), or nd * shard_numel past 2^62; for the scatter also
 * two tensors whose ranges overlap), ZERO_EWORKSPACE, ZERO_ECUDA. */
size_t zero_gather_workspace_bytes(int64_t n_tensors, int32_t nd);

/* Shards -> tensors (the all-gather). */
int zero_gather_params(const void *const *shards, int32_t nd, int64_t shard_numel, const zero_tlist_t *tensors,
                       const int64_t *tensor_offset, void *ws, size_t ws_bytes, void *stream);

/* Tensors -> shards (partitioning a model's tensors into the flat shards).
 * Flat elements outside every tensor's range (the tail padding) are not
 * written. */
int zero_scatter_params(const zero_tlist_t *tensors, const int64_t *tensor_offset, void *const *shards,
                        int32_t nd, int64_t shard_numel, void *ws, size_t ws_bytes, void *stream);

/* One rank's part of one layer's gather. */
typedef struct zero_gather_piece {
    int64_t layer;        /* layer index */
    int64_t rank;         /* the rank that holds the piece */
    int64_t shard_offset; /* its first element within that rank's shard */
    int64_t length;       /* elements (> 0) */
    int64_t layer_offset; /* where it lands, counted from the layer's first element */
} zero_gather_piece_t;

/* The per-layer gather schedule of stage 3 (host only).  A layer is a run of
 * consecutive tensors: layer L holds tensors [layer_first[L],
 * layer_first[L+1]) (layer_first: n_layers + 1 non-decreasing entries in
 * [0, n_tensors]).  Its parameters are then one flat range, written to
 * layer_flat[L] .. layer_flat[L+1] (layer_flat: n_layers + 1 entries, may be
 * NULL), and each rank whose shard meets that range contributes exactly one
 * contiguous piece; pieces are listed by layer, then rank.  The layout is
 * zero_partition_layout's for (numel, n_tensors, nd, align).  *n_pieces
 * always receives the count; past `cap` only the first cap are written and
 * ZERO_ECAPACITY is returned.  *max_layer_numel (may be NULL) receives the
 * largest layer, the size of the buffer one gathered layer needs.
 * Errors: ZERO_EINVAL, ZERO_ELAYOUT (as zero_partition_layout, or a bad
 * layer_first), ZERO_ECAPACITY. */
int zero_gather_plan(const int64_t *numel, int64_t n_tensors, const int64_t *layer_first, int64_t n_layers,
                     int32_t nd, int64_t align, int64_t *layer_flat, zero_gather_piece_t *pieces, int64_t cap,
                     int64_t *n_pieces, int64_t *max_layer_numel);

/* ------------------------------------------------------------------ 1-bit Adam */

/* 1-bit Adam (DeepSpeed release news, lxsoso.com/blog/19320.html: Adam with
 * up to 5x less communication and Adam's convergence).  The page gives no
 * algorithm; these calls follow the outline of the published method (Tang et
 * al. 2021): after a warm-up of T_w plain steps (zero_adam_step), the
 * variance is frozen and the workers average their MOMENTUM, not their
 * gradient, through an all-reduce compressed to one bit per element with
 * error feedback at both ends.  One compression-stage step of rank r of Nd
 * (n = Nd * S elements, the padded flat layout; rank r serves chunk r,
 * elements [r*S, (r+1)*S)):
 *
 *   zero_grad_norm_overflow(g)         overflow flag (and norm) of the local
 *                                      gradient, summed over the ranks
 *   zero_onebit_worker                 x = b1*m + (1-b1)*g + e_w;
 *                                      e_w <- x - C(x); signs, scale of C(x)
 *   (exchange: chunk j of every worker's signs and its scale to rank j)
 *   zero_onebit_server                 y = mean over workers of C(x_i) on
 *                                      chunk r, + e_s; e_s <- y - C(y)
 *   (the errors e_w and e_s are held in deferred form, see below)
 *   (exchange: every rank's server signs and scale to every worker)
 *   zero_onebit_update                 m <- the servers' C(y_j), all chunks;
 *                                      p <- p - (lr/(1-b1^t) * m /
 *                                      (sqrt(v) * isb2(T_w) + eps) + lr*wd*p)
 *
 * The compressor: C(x) = scale * sign(x) with scale = ||x||_2 / sqrt(len)
 * (binary64 sum, rounded once to binary32) and sign(0) = +1.  Signs travel
 * as 32-bit words, bit k of word w holding element 32w + k, 1 for +.  The
 * server's mean is the binary32 sum over workers in rank order followed by
 * one division by Nd.  Element arithmetic is binary32, each operation
 * rounded on its own.  The three calls of one step use the same state and
 * workspace (zero_workspace_bytes(Nd, n)) in stream order; the worker call's
 * decision (skip on overflow, loss scale, step count) holds for the other
 * two, and a skipped step changes nothing.  n and S must be multiples of 32
 * (ZERO_ESIZE); arrays 16-byte aligned.  Errors otherwise as
 * zero_adam_step.
 *
 * The errors in deferred form.  Each error is x - C(x) for the input x of
 * the compression that left it, so the calls keep x itself (x_w, x_s) and
 * its scale (the call's own `scale`, read on entry and replaced on return)
 * and form the error x - scale*sign(x) -- one binary32 subtraction, the
 * same bits as forming it at once -- when the next step reads x.  A
 * compression is then one pass over its input instead of two (8 bytes per
 * element less).  Start the compression stage with x_w (x_s) zero and
 * *scale zero: the error is then zero.  More generally, with *scale zero
 * the array itself is the error (x - 0*sign(x) = x exactly), which is how to
 * resume from an explicit error; the error of a pair (x, s) is
 * x - s where x >= 0 or x is -0, x + s elsewhere. */

/* Worker side.  grad: n elements (F16, BF16 or F32).  The synchronised
 * momentum comes either dense, m (fp32, n elements, read), or -- with m
 * NULL -- compressed, as the previous step's servers left it: m_bits (n/32
 * words) and m_scales (n/S floats), element i being +-m_scales[i / S] (S a
 * multiple of 32 dividing n; ignored when m is given).  After the first
 * compression step the compressed form is exact and saves the 4 bytes per
 * element of a dense momentum on both the update's write and this read.
 * x_w: the worker's error in deferred form (fp32, n elements: the input of
 * this worker's previous compression on entry, this one's on return);
 * bits: n/32 words (written); scale: one device float (the previous
 * compression's scale on entry, this one's on return).  freeze_step: T_w,
 * the count of the last warm-up step (>= 1). */
int zero_onebit_worker(const void *grad, int32_t gdtype, const float *m, const uint32_t *m_bits,
                       const float *m_scales, int64_t S, float *x_w, int64_t n, uint32_t *bits, float *scale,
                       const zero_hparams_t *hp, int64_t freeze_step, zero_state_t *d_state, void *ws,
                       size_t ws_bytes, void *stream);

/* Server side for this rank's chunk of S elements.  worker_bits: HOST array
 * of nd device pointers, each to S/32 words (the chunk's signs from worker
 * i); worker_scales: device array of nd floats; x_s: the server's error in
 * deferred form (S fp32: the input of this rank's previous server
 * compression on entry, this one's on return); bits: S/32 words (written);
 * scale: one device float (the previous server compression's scale on
 * entry, this one's on return).
 * At most 4096 workers (ZERO_ECAPACITY).  Up to 256 workers the pointers
 * travel as a launch argument; beyond, as a table copied into the
 * workspace (not capturable: ZERO_ECAPTURE under stream capture).  The
 * result is the rank-order sum itself: each block tabulates the sums of the
 * first min(nd, 14) workers' terms for every sign pattern, with the same
 * additions in the same order, and adds the remaining workers' terms to the
 * entry an element's signs select. */
int zero_onebit_server(const uint32_t *const *worker_bits, const float *worker_scales, int32_t nd, int64_t S,
                       float *x_s, uint32_t *bits, float *scale, void *ws, size_t ws_bytes, void *stream);

/* Update.  bits: nd*S/32 words, the servers' signs in rank order;
 * server_scales: device array of nd floats; m: the dense momentum, nd*S
 * fp32 elements (the whole padded buffer, which the compressed all-reduce
 * covers), written if not NULL; p, v: fp32 arrays of at least `numel`
 * elements (p written, v read); p_lp: F16 or BF16 copy of p (or NULL).
 * Parameters from `numel` to nd*S (padding) are not touched. */
int zero_onebit_update(const uint32_t *bits, const float *server_scales, int32_t nd, int64_t S, int64_t numel,
                       float *p, float *m, const float *v, void *p_lp, int32_t pdtype, void *ws, size_t ws_bytes,
                       void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_PML_H */
