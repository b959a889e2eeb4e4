/*
 * mfsdp.h -- C ABI of the owner-local optimizer step of MatrixFSDP on one GPU.
 *
 * Source: "MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3
 * Parameter Sharding" (Gao, Xu, Zhang; arXiv 2607.05895).  Abstract: for each
 * 2D weight one data-parallel rank owns the whole matrix and the other ranks
 * hold empty shards; non-matrix tensors are packed into tail owners and stay
 * on AdamW; the reduced gradient lands whole on its owner, so Muon's momentum
 * and Newton-Schulz run locally; the runtime carries the plan in MatrixShard
 * metadata produced by a balance-aware owner planner.  FAQ (docshare page):
 * MatrixShard metadata carries the owner plan through optimizer routing and
 * resharding; owner segments replace equal-size shard assumptions.
 *
 * Conventions for every entry point:
 *   - Return value: MFSDP_OK (0) or a negative mfsdp_status.  The library never
 *     aborts, never prints and never allocates device memory; it keeps no state
 *     between calls.
 *   - Device pointers are plain CUDA device addresses owned by the caller and
 *     must stay valid until the work queued on `stream` has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All device work is asynchronous on it; all argument checks happen on the
 *     host before anything is queued, so an error return means nothing ran.
 *   - A matrix is stored row-major, `rows` x `cols`, in a flat buffer at an
 *     element `offset`.  s = min(rows, cols), l = max(rows, cols).
 */
#ifndef MFSDP_H
#define MFSDP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MFSDP_OK = 0,
  MFSDP_ERR_INVALID_ARG = -1,        /* null pointer, negative count, bad enum, bad hyper-parameter */
  MFSDP_ERR_MISALIGNED = -2,         /* base pointer not 16-byte aligned, workspace not 256-byte aligned */
  MFSDP_ERR_OVERLAP = -3,            /* two segments, or two distinct buffers, share elements */
  MFSDP_ERR_OUT_OF_BOUNDS = -4,      /* a segment extends past its buffer */
  MFSDP_ERR_UNSUPPORTED_DTYPE = -5,  /* dtype code other than MFSDP_DTYPE_F32 / _BF16 where allowed */
  MFSDP_ERR_UNSUPPORTED_SHAPE = -6,  /* dimension < 1, s > MFSDP_MAX_SHORT_SIDE, or l > MFSDP_MAX_LONG_SIDE */
  MFSDP_ERR_WORKSPACE_TOO_SMALL = -7,
  MFSDP_ERR_CUDA = -8,               /* a CUDA runtime call failed (no device, launch failure, ...) */
  MFSDP_ERR_DEVICE_TIMEOUT = -9,     /* a kernel's bounded wait expired (reported by mfsdp_muon_device_status) */
  MFSDP_ERR_IO = -10,                /* a checkpoint file could not be opened, written or read */
  MFSDP_ERR_FORMAT = -11             /* not a checkpoint of this format, or a damaged or truncated one */
} mfsdp_status;

typedef enum { MFSDP_DTYPE_F32 = 0, MFSDP_DTYPE_BF16 = 1 } mfsdp_dtype;
typedef enum { MFSDP_KIND_MATRIX = 0, MFSDP_KIND_TAIL = 1 } mfsdp_kind;

#define MFSDP_MAX_SHORT_SIDE 32768
#define MFSDP_MAX_LONG_SIDE (1 << 24)

/* One parameter of the model, in declaration order (its index is its param id).
 * kind MATRIX: a 2D weight updated by Muon.  kind TAIL: any tensor updated by
 * AdamW; numel = rows * cols (a 1D tensor of n elements is rows = n, cols = 1). */
typedef struct {
  int64_t rows;
  int64_t cols;
  int32_t kind;
  int32_t reserved;
} mfsdp_param;

/* MatrixShard: one whole matrix inside its owner's flat matrix buffer.
 * The owner's gradient, fp32 momentum and update buffers all use this offset.
 * transposed = rows > cols: Newton-Schulz then runs on the transpose, so the
 * Gram matrix is always s x s.  cost = ns_steps * (4 s^2 l + 2 s^3), the dense
 * Newton-Schulz FLOP count the planner balances. */
typedef struct {
  int32_t param_id;
  int32_t owner;
  int64_t offset;
  int64_t rows;
  int64_t cols;
  int32_t transposed;
  int32_t reserved;
  uint64_t cost;
} mfsdp_matrix_shard;

/* One tail tensor inside its owner's flat fp32 tail buffer. */
typedef struct {
  int32_t param_id;
  int32_t owner;
  int64_t offset;
  int64_t numel;
} mfsdp_tail_shard;

/* Balance-aware owner planner (Abstract: "a balance-aware owner planner";
 * every 2D weight wholly on one rank, tail tensors on tail owners).  Host only.
 *
 * The pages give no algorithm; this one is:
 *   matrices sorted by (cost desc, param id asc), each to the rank with the
 *   smallest (matrix load, rank id) -- longest-processing-time first;
 *   tail tensors sorted by (numel desc, param id asc), each to the rank with the
 *   smallest (tail load, matrix load, rank id);
 *   per rank, segments in ascending param id, each offset rounded up to
 *   align_elems, matrix and tail buffers separate.
 *
 * params[n_params]     in: the model's parameters.
 * world                in: number of data-parallel ranks (>= 1).
 * ns_steps             in: Newton-Schulz steps (>= 0; scales every cost).
 * align_elems          in: segment alignment in elements (>= 1; 128 keeps
 *                      every segment 256-byte aligned in bf16).
 * out_m                out: capacity >= number of MATRIX params; filled in
 *                      (owner, offset) order.  *n_m receives the count.
 * out_t                out: capacity >= number of TAIL params; same order.
 * rank_matrix_elems    out[world]: each rank's matrix-buffer extent, the end of
 *                      its last segment rounded up to align_elems (0 if empty).
 * rank_tail_elems      out[world]: the same for the tail buffer.
 * Any out pointer except out_m/out_t/n_m/n_t may be NULL.  Errors:
 * INVALID_ARG, UNSUPPORTED_SHAPE (dimension < 1 or a cost above 2^64). */
int mfsdp_plan_owners(const mfsdp_param* params, int32_t n_params, int32_t world,
                      int32_t ns_steps, int64_t align_elems,
                      mfsdp_matrix_shard* out_m, int32_t* n_m,
                      mfsdp_tail_shard* out_t, int32_t* n_t,
                      int64_t* rank_matrix_elems, int64_t* rank_tail_elems);

/* Bytes of device workspace mfsdp_muon_owner_step needs for these shards
 * (0 on invalid input).  Holds, per matrix, X (two bf16 ping-pong copies of
 * the s x l iterate, the second at least three s x s matrices long when the
 * shape may run the Gram-space form, whose C and Q it holds) and the s x s
 * bf16 matrices A = X X^T and B = bA + cA^2 (Gram space: P), each padded to
 * multiples of 128 (the short side to 256), plus norm partials, the
 * Newton-Schulz tile and completion counters and a status word. */
size_t mfsdp_muon_workspace_bytes(const mfsdp_matrix_shard* shards, int32_t n_shards);

/* Owner-local Muon step over one rank's owned matrices (Abstract: the reduced
 * gradient lands whole on its owner; "Newton-Schulz runs locally with no
 * optimizer-step matrix collective"; the update matches full-matrix Muon).
 *
 * For every shard (offset, rows, cols):
 *   M <- beta*M + G                         (fp32, in place in `momentum`)
 *   U  = M  (nesterov = 0)  or  G + beta*M  (nesterov = 1)
 *   X  = U / (||U||_F + eps), transposed to s x l when rows > cols
 *   ns_steps times:  A = X X^T,  B = b*A + c*A*A,  X <- a*X + B*X
 *   update[offset ..] = X, transposed back to rows x cols.
 * A matrix with l >= 2 s, l >= s + 384 and s >= 128, for 1 <= ns_steps <= 5,
 * evaluates the same iteration in Gram space: with P_k = a I + b A_k + c A_k A_k,
 * X_{k+1} = P_k X_k, so A_{k+1} = P_k A_k P_k and the update is
 * P_{T-1} ... P_0 X: it iterates the s x s matrices A (as C = P A, A <- C P)
 * and Q = P_k Q_{k-1}, and multiplies X by Q once (about half the tensor
 * FLOPs of the direct form for such shapes, and the long K = l only in the
 * first Gram product; equal in exact arithmetic, and within the same error of
 * the fp64 definition in bf16).  mfsdp_muon_gram_space_layout says which
 * matrices do.
 * The Newton-Schulz products run on tensor cores with bf16 operands and fp32
 * accumulation; A, B and X (Gram space: A, P, C, Q) are held in bf16 between
 * products, and the hyper-parameters are applied as fp32 values rounded from
 * the doubles given.
 * A matrix whose momentum is exactly zero gets an all-zero update.  The fp32
 * Gram product needs ||U||_F < 1e18 and the entries of U above ~1e-18 in
 * magnitude (outside that range the result may be Inf/NaN or lose the small
 * entries).
 *
 * shards[n_shards]  host array; segments must not overlap.  owner is ignored.
 * grad              device, `numel` elements of grad_dtype (F32 or BF16).
 * momentum          device, `numel` fp32; read and written.
 * update            device, `numel` elements of update_dtype (F32 or BF16);
 *                   only the shards' elements are written.  update may equal
 *                   grad when both dtypes match (in-place); otherwise the three
 *                   buffers must not overlap.
 * numel             length of each buffer in elements.
 * ns_steps          0..64; 0 returns the normalised momentum.
 * workspace         device, >= mfsdp_muon_workspace_bytes(), 256-byte aligned;
 *                   scratch only, contents undefined after the call.
 * Errors: INVALID_ARG, MISALIGNED, OVERLAP, OUT_OF_BOUNDS, UNSUPPORTED_DTYPE,
 * UNSUPPORTED_SHAPE, WORKSPACE_TOO_SMALL, CUDA_ERROR. */
int mfsdp_muon_owner_step(const mfsdp_matrix_shard* shards, int32_t n_shards,
                          const void* grad, int32_t grad_dtype,
                          float* momentum,
                          void* update, int32_t update_dtype,
                          int64_t numel,
                          double beta, int32_t nesterov, int32_t ns_steps,
                          double a, double b, double c, double eps,
                          void* workspace, size_t workspace_bytes, void* stream);

/* The same step split in two, for callers that interleave other work or time
 * the phases separately: `phases` is a bit set of
 *   MFSDP_PHASE_MOMENTUM        momentum, segment view and norm (writes
 *                               momentum and the workspace; clears its status word)
 *   MFSDP_PHASE_NEWTON_SCHULZ   the Newton-Schulz products and the update
 *                               (reads what the momentum phase left in the workspace)
 * Calling MOMENTUM then NEWTON_SCHULZ with identical arguments on one stream
 * gives bit-identical results to mfsdp_muon_owner_step (phases = both).
 * Same arguments and errors as mfsdp_muon_owner_step, plus INVALID_ARG for an
 * empty or unknown phase set. */
#define MFSDP_PHASE_MOMENTUM 1
#define MFSDP_PHASE_NEWTON_SCHULZ 2
int mfsdp_muon_owner_step_phases(const mfsdp_matrix_shard* shards, int32_t n_shards,
                                 const void* grad, int32_t grad_dtype,
                                 float* momentum,
                                 void* update, int32_t update_dtype,
                                 int64_t numel,
                                 double beta, int32_t nesterov, int32_t ns_steps,
                                 double a, double b, double c, double eps,
                                 void* workspace, size_t workspace_bytes, void* stream,
                                 int32_t phases);

/* The owner step followed by applying the update to the weights, fused into
 * the last Newton-Schulz epilogue.  The pages stop at the orthogonalised
 * update; applying it is the step right after, in Muon's decoupled form:
 *   W <- W * (1 - lr * weight_decay) - lr * scale * O
 * with scale_mode 0: scale = 1; 1: sqrt(max(1, rows/cols)); 2:
 * 0.2 * sqrt(max(rows, cols)).  The products run in fp32 from the same fp32
 * accumulator the update comes from (bf16 weights are rounded once).
 *   weights  device, numel elements of weight_dtype (F32 or BF16), the same
 *            offsets as the gradient; read and written.  Must not overlap the
 *            other buffers.
 *   update   may be NULL (O is then not stored); otherwise as for
 *            mfsdp_muon_owner_step, and the O it receives is bit-identical.
 *   ns_steps >= 1.  A matrix with all-zero momentum has O = 0, so its
 *            weights only decay.
 * Errors: as mfsdp_muon_owner_step, plus INVALID_ARG (NULL weights, bad
 * scale_mode, non-finite lr/weight_decay, ns_steps < 1). */
int mfsdp_muon_owner_step_apply(const mfsdp_matrix_shard* shards, int32_t n_shards,
                                const void* grad, int32_t grad_dtype,
                                float* momentum,
                                void* update, int32_t update_dtype,
                                void* weights, int32_t weight_dtype,
                                int64_t numel,
                                double beta, int32_t nesterov, int32_t ns_steps,
                                double a, double b, double c, double eps,
                                double lr, double weight_decay, int32_t scale_mode,
                                void* workspace, size_t workspace_bytes, void* stream);

/* The owner step with the gradient coming from, and the update going to,
 * pinned host memory.  The shards are cut into groups (mfsdp_host_step_groups);
 * group g's gradient ranges are copied host->device on an internal stream
 * while the groups before it compute on `stream`, and its update ranges are
 * copied device->host on another internal stream while later groups compute.  Each group runs the same kernels as
 * mfsdp_muon_owner_step on its own shards (results are bit-identical).
 *   grad_host / update_host  pinned host buffers (cudaHostAlloc / registered),
 *                            numel elements of grad_dtype / update_dtype.
 *   grad_dev / update_dev    device staging buffers of numel elements; every
 *                            other argument as for mfsdp_muon_owner_step.
 *   groups >= 1 (1 = no overlap), or 0: the library's choice; both as
 *                            mfsdp_host_step_groups describes.
 * The call returns once everything is queued; work queued on `stream` later
 * runs after the last copy.  The two copy streams and their events belong to
 * the library: created on a device's first call and kept until the process
 * exits.  Calls on one device enqueue one at a time (a lock held while
 * queuing, not while the GPU works) and their copies run in call order.
 * Errors: as mfsdp_muon_owner_step, plus INVALID_ARG for a NULL host buffer
 * or groups < 0, and CUDA when the current device's index is 64 or more. */
int mfsdp_muon_owner_step_host(const mfsdp_matrix_shard* shards, int32_t n_shards,
                               const void* grad_host, void* grad_dev, int32_t grad_dtype,
                               float* momentum,
                               void* update_dev, void* update_host, int32_t update_dtype,
                               int64_t numel,
                               double beta, int32_t nesterov, int32_t ns_steps,
                               double a, double b, double c, double eps,
                               void* workspace, size_t workspace_bytes, int32_t groups, void* stream);

/* The shard groups of the host-buffer step (no counterpart in the paper: a
 * property of this library's copy pipeline).  Returns the number of groups
 * mfsdp_muon_owner_step_host runs for these arguments and, when group_of is
 * not NULL, writes each shard's group (0 = first to run) to group_of[0..n).
 *   groups >= 1  shards in offset order, cut into min(groups, n) ranges of
 *                balanced Newton-Schulz cost 4 s^2 l + 2 s^3 + s l (empty
 *                ranges dropped).
 *   groups == 0  chosen from the copy volume B = sum of rows * cols * (grad +
 *                update element size).  Copies stay exposed only at the two
 *                ends; each group past the first costs some compute (up to
 *                one latency-bound Newton-Schulz chain, ~0.25 ms, when a group
 *                is too small to fill the GPU).  With g = round(sqrt(B / 50 MB)):
 *                g <= 1 one group; g == 2 or fewer than 5 shards: min(g, n)
 *                balanced ranges; g >= 6: min(g, 16) balanced ranges between a
 *                head and a tail group, each up to two of the smallest shards
 *                with the largest short side (most work per byte) holding at
 *                most 1 / (2 min(g, 16)) of the elements -- without such
 *                shards for both ends, only the balanced ranges;
 *                3 <= g <= 5: a ramp -- shards ordered small -> large -> small
 *                by size and cut at 4 %, 28 %, 72 % and 96 % of B (a shard
 *                goes where the midpoint of its bytes falls).  Both make the
 *                first copy in and the last copy out small.
 * A group's copies are the runs of its shards that neighbour each other in
 * offset order.  Host only: no device is touched.  Returns 0 for NULL shards,
 * n_shards <= 0, groups < 0 or a dtype other than F32 / BF16. */
int32_t mfsdp_host_step_groups(const mfsdp_matrix_shard* shards, int32_t n_shards, int32_t grad_dtype,
                               int32_t update_dtype, int32_t groups, int32_t* group_of);

/* mfsdp_muon_owner_step for callers that cannot allocate device memory (no
 * counterpart in the paper: an addition of this library).  Some callers have
 * no allocator to provide the workspace from -- a plug-in inside a framework
 * that owns all device memory through its own pool, a callback that must not
 * allocate, a C program linking only this library.  This entry point takes no
 * workspace: its scratch is a file-scope device array of
 * MFSDP_STATIC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits.  It calls no cudaMalloc/cudaFree and nothing that
 * allocates.
 *   - Same arguments, semantics and errors as mfsdp_muon_owner_step without
 *     workspace/workspace_bytes; an owner set whose
 *     mfsdp_muon_workspace_bytes() exceeds MFSDP_STATIC_SCRATCH_BYTES is
 *     rejected with MFSDP_ERR_WORKSPACE_TOO_SMALL before anything runs.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for the
 *     device's current CUDA context; a call in another context of the device
 *     (a new primary context after cudaDeviceReset, or a context the caller
 *     made current) looks it up again.  Make the first call on a device, in
 *     each context, before any stream capture on it.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents (the step clears what must start at zero itself).  Calls whose
 *     work overlaps on the GPU (different streams, or different host threads
 *     without ordering) race on it: serialise them.
 *   - Its device status word (a bounded wait that gave up, see
 *     mfsdp_muon_device_status) sits at the start of the array, out of the
 *     caller's reach: read it with mfsdp_muon_static_scratch_status. */
#define MFSDP_STATIC_SCRATCH_BYTES (64u << 20)
int mfsdp_muon_owner_step_static_scratch(const mfsdp_matrix_shard* shards, int32_t n_shards,
                                         const void* grad, int32_t grad_dtype,
                                         float* momentum,
                                         void* update, int32_t update_dtype,
                                         int64_t numel,
                                         double beta, int32_t nesterov, int32_t ns_steps,
                                         double a, double b, double c, double eps,
                                         void* stream);

/* The device status word of the last mfsdp_muon_owner_step_static_scratch
 * call on the current device (no counterpart in the paper).  Like
 * mfsdp_muon_device_status -- same return values and *detail encoding, and it
 * synchronises `stream` -- but it reads the library's scratch array, so queue
 * it on the stream of the call it reports on, after that call.  Returns
 * MFSDP_OK when no static-scratch call ran yet on the device (the array starts
 * zeroed), and CUDA when the array's address cannot be looked up. */
int mfsdp_muon_static_scratch_status(void* stream, int32_t* detail);

/* FLOP counts of mfsdp_muon_owner_step for these shards, host only:
 * *dense = sum over matrices of ns_steps * (4 s^2 l + 2 s^3) (the algorithmic
 * count); *executed = the tensor-core FLOPs the kernels issue (outputs
 * padded to multiples of 128, the short side to 256, and a contraction over
 * the short side to s rounded up to 128; the symmetric products
 * computed on their 256 x 256 blocks on or above the diagonal only; a matrix
 * that runs the Gram-space form counted with its own products: A_0, then per
 * iteration P_k, C_k, A_{k+1} and Q_k where they exist, all symmetric, and
 * the final Q X0; matrices whose momentum turns out to be zero, which skip
 * all products, still counted).
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE. */
int mfsdp_muon_step_flops(const mfsdp_matrix_shard* shards, int32_t n_shards, int32_t ns_steps,
                          uint64_t* dense, uint64_t* executed);

/* Reads the device status word a previous mfsdp_muon_owner_step left in
 * `workspace` (synchronising `stream`): MFSDP_OK, or MFSDP_ERR_DEVICE_TIMEOUT
 * if one of its kernels gave up on a bounded wait (its outputs are then
 * undefined).  Every wait of a Newton-Schulz launch gives up after its limit:
 * 2 s, or, for launches whose largest product (Gram, polynomial or update,
 * summed over the launch's matrices) would take longer than 2 s / 8 with
 * every CTA pair at a quarter of its bf16 tensor peak at 1 GHz, 8x that time
 * (at most an hour).  The first wait to give up records the word and every
 * other CTA then stops too.
 * *detail (may be NULL) receives the raw word: bits 0-7 the waiting role
 * (1 producer: a free pipeline stage; 2 MMA issuer: a stage's operands;
 * 3 MMA issuer: a drained accumulator; 4 epilogue: a finished accumulator;
 * 5 producer, or a role waiting behind it: the earlier products of a tile's
 * matrix; 7 scheduler: a free slot of a tile ring; 8 any role: the next
 * tile), bits 8-31 the
 * Newton-Schulz product index (3 * iteration + 0 Gram / 1 polynomial /
 * 2 update; in the Gram-space form 0 A_k, 1 P_k, 2 C_k and Q_k, and
 * 3 * ns_steps the final Q X0) where the role knows it, else 0.  The status word is cleared by
 * every call that runs the momentum phase. */
int mfsdp_muon_device_status(const void* workspace, void* stream, int32_t* detail);

/* Testing only: the next Newton-Schulz launch of this process (one launch; the
 * hook then clears itself) gives tile `tile` of its tile list a dependency
 * that is never satisfied, so the wait for it runs out after 2 s.  The kernel
 * then ends in bounded time, and mfsdp_muon_device_status reports
 * MFSDP_ERR_DEVICE_TIMEOUT with role 5 (a producer's dependency wait, or a
 * role waiting behind it) or 8 (a role waiting to be handed a tile).
 * The context stays usable.  This exercises the bounded-wait path without
 * faulting or hanging the GPU.  Returns INVALID_ARG for tile < 0. */
int mfsdp_test_inject_stall(int32_t tile);

/* Layout of the workspace, for inspection: for shard i, out[8*i + 0..7] =
 * { byte offset of X0, of X1, of A, of B, s_pad, l_pad, s, l }.  X0/X1 are
 * s_pad x l_pad, A/B s_pad x s_pad, bf16, stored as 1024-byte atoms of
 * 8 rows x 64 columns; atom (row/8, col/64) sits at
 * ((col/64) * (rows_pad/8) + row/8) * 1024, and inside it element (r, c) at
 * (r%8)*128 + ((((c%64)/8) ^ (r%8)) * 16) + (c%8)*2.  A and B (symmetric)
 * hold only their 256 x 256 blocks on or above the diagonal (col/256 >=
 * row/256); the others are never written.  Returns the status. */
int mfsdp_muon_workspace_layout(const mfsdp_matrix_shard* shards, int32_t n_shards, int64_t* out);

/* Which form of the iteration each matrix runs for ns_steps, and where the
 * Gram-space form keeps its matrices, for inspection: for shard i,
 * out[4*i + 0..3] = { 1 if Gram space else 0, byte offset of C, of Q_even,
 * of Q_odd } (s_pad x s_pad, the blocked layout above, inside X1's region;
 * P_0 = Q_0 is written to Q_even, P_k (k >= 1) to B; after a step the
 * workspace holds A_{T-1}, P_{T-1}, C_{T-2} and Q_{T-1} (in Q_even for odd T),
 * the symmetric ones as their 256 x 256 blocks on or above the diagonal).
 * Returns INVALID_ARG for ns_steps outside 0..64 or a NULL out, else as
 * mfsdp_muon_workspace_layout. */
int mfsdp_muon_gram_space_layout(const mfsdp_matrix_shard* shards, int32_t n_shards, int32_t ns_steps,
                                 int64_t* out);

/* AdamW over a packed fp32 tail buffer (Abstract: non-matrix tensors "stay on
 * AdamW"), decoupled weight decay, step counted from 1:
 *   p <- p*(1 - lr*wd); m <- b1*m + (1-b1)*g; v <- b2*v + (1-b2)*g^2;
 *   p <- p - lr/(1-b1^step) * m / (sqrt(v)/sqrt(1-b2^step) + eps)
 * p, m, v read and written in place; g read.  All device, n fp32 elements,
 * 16-byte aligned, not overlapping (n == 0 is a no-op).  The kernel computes
 * in fp32 with 1-b1, 1-b2, 1-lr*wd, lr/(1-b1^step) and 1/sqrt(1-b2^step)
 * formed in double on the host.  Errors: INVALID_ARG
 * (null pointer, n < 0, step < 1, beta outside [0, 1)), MISALIGNED, OVERLAP,
 * CUDA_ERROR. */
int mfsdp_adamw_tail_step(float* p, const float* g, float* m, float* v, int64_t n,
                          double lr, double beta1, double beta2, double eps, double wd,
                          int64_t step, void* stream);

/* ------------------------------------------------------------------------
 * Owner segments: the reduce that lands each whole matrix on its owner, and
 * owner-shard resharding (Abstract: "the ordinary backward reduction then
 * lands the full Muon input on the owner"; "deterministic owner-segment P2P
 * collectives"; "owner-shard checkpoint resharding").  On one GPU the
 * data-parallel ranks' buffers are separate flat device buffers.
 * ------------------------------------------------------------------------ */

/* Where one parameter sits: owner (rank or source-buffer index), element
 * offset and length in that owner's flat buffer.  A matrix shard maps to
 * (param_id, owner, offset, rows*cols), a tail shard to itself. */
typedef struct {
  int32_t param_id;
  int32_t owner;
  int64_t offset;
  int64_t numel;
} mfsdp_placement;

/* One contiguous run of elements to move. */
typedef struct {
  int64_t src_offset;
  int64_t dst_offset;
  int64_t numel;
  int32_t src_index;   /* GATHER: which source buffer; ignored by REDUCE */
  int32_t reserved;
} mfsdp_segment;

#define MFSDP_SEGMENT_REDUCE 0
#define MFSDP_SEGMENT_GATHER 1

/* Unsharded flat layout of a model's parameters (each rank's local gradient
 * before the reduce): declaration order, each offset rounded up to
 * align_elems.  offsets[n_params] out; *total = end rounded up to align_elems.
 * Host only.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE. */
int mfsdp_model_layout(const mfsdp_param* params, int32_t n_params, int64_t align_elems,
                       int64_t* offsets, int64_t* total);

/* Segments that fill dst_owner's buffer of placement `dst` from placement
 * `src`: for every entry of dst with owner == dst_owner (in dst-offset
 * order), the entry of src with the same param_id gives src_index (= its
 * owner) and src_offset.  out has capacity n_dst; *n_out receives the count.
 * Host only.  Errors: INVALID_ARG (a param missing from src, a param twice in
 * src, or different lengths). */
int mfsdp_placement_segments(const mfsdp_placement* src, int32_t n_src, const mfsdp_placement* dst,
                             int32_t n_dst, int32_t dst_owner, mfsdp_segment* out, int32_t* n_out);

/* Moves the segments into `dst`.
 *   mode REDUCE: dst[dst_offset+i] = sum over k = 0..n_src-1, in that order,
 *     of srcs[k][src_offset+i], accumulated in fp32 and rounded once to
 *     dst_dtype (bitwise reproducible).
 *   mode GATHER: dst[dst_offset+i] = srcs[src_index][src_offset+i] (converted).
 * srcs[n_src] (1..64) device buffers of src_numel[k] elements of src_dtype;
 * dst device, dst_numel elements of dst_dtype; dtypes F32 or BF16; every base
 * pointer 16-byte aligned.  Segments must stay inside their buffers, must not
 * overlap each other in dst, and dst must not overlap any source.  Elements of
 * dst outside the segments are left alone.  Errors: INVALID_ARG, MISALIGNED,
 * OUT_OF_BOUNDS, OVERLAP, UNSUPPORTED_DTYPE, CUDA_ERROR. */
int mfsdp_segment_copy(const void* const* srcs, const int64_t* src_numel, int32_t n_src, int32_t src_dtype,
                       const mfsdp_segment* segs, int32_t n_segs, int32_t mode,
                       void* dst, int32_t dst_dtype, int64_t dst_numel, void* stream);

/* ------------------------------------------------------------------------
 * Owner-shard checkpoints (Abstract: "owner-shard checkpoint resharding";
 * FAQ: MatrixShard metadata carries the owner plan through optimizer routing
 * and resharding).  One file holds one rank's optimizer state -- its fp32
 * momentum buffer and its packed AdamW tail (p, m, v) -- together with the
 * rank's MatrixShard and tail tables, which say where every parameter sits.
 * Reloading under another world size: read every old rank's file, plan the
 * new world with mfsdp_plan_owners, and for each new rank let
 * mfsdp_placement_segments match every parameter's old (rank, offset) to its
 * new one; mfsdp_segment_copy (GATHER) then moves the state, one buffer kind
 * at a time, from the old ranks' buffers into the new rank's.
 *
 * The file is little-endian and independent of the host (every field is
 * written byte by byte): the 8 bytes "MFSDPCK1", a u32 format version (1), the
 * header fields in the order below (i32 world, rank, ns_steps, n_matrix,
 * n_tail; i64 align_elems, matrix_elems, tail_elems, adam_step), the matrix
 * shards (48 bytes each: i32 param_id, i32 owner, i64 offset, rows, cols,
 * i32 transposed, i32 reserved, u64 cost), the tail shards (24 bytes each:
 * i32 param_id, i32 owner, i64 offset, numel), matrix_elems binary32 values of
 * momentum, tail_elems values each of tail p, m and v, and a u64 FNV-1a-64
 * digest of every byte before it.  Host only: the buffers are host memory
 * (copy device buffers out and in around these calls).
 * ------------------------------------------------------------------------ */
typedef struct {
  int32_t world;         /* ranks of the plan the file belongs to (>= 1) */
  int32_t rank;          /* this file's rank, 0 <= rank < world */
  int32_t ns_steps;      /* Newton-Schulz steps the plan's costs were computed with */
  int32_t n_matrix;      /* matrix shards of the rank */
  int32_t n_tail;        /* tail shards of the rank */
  int32_t reserved;
  int64_t align_elems;   /* segment alignment of the plan */
  int64_t matrix_elems;  /* momentum buffer length (the rank's matrix-buffer extent) */
  int64_t tail_elems;    /* tail buffer length (the rank's tail-buffer extent) */
  int64_t adam_step;     /* AdamW steps the tail state has taken */
} mfsdp_checkpoint_header;

/* Size in bytes of the file mfsdp_checkpoint_write makes for this header (0
 * for an invalid header). */
size_t mfsdp_checkpoint_bytes(const mfsdp_checkpoint_header* header);

/* Writes one rank's checkpoint to `path` (created or truncated).
 * matrix_shards[n_matrix] / tail_shards[n_tail]: the rank's tables (every
 * shard's owner must be header->rank and lie inside its buffer); momentum
 * [matrix_elems], tail_p / tail_m / tail_v [tail_elems]: host buffers.
 * Errors: INVALID_ARG (null pointer, invalid header), OUT_OF_BOUNDS (a shard
 * outside its buffer or owned by another rank), IO. */
int mfsdp_checkpoint_write(const char* path, const mfsdp_checkpoint_header* header,
                           const mfsdp_matrix_shard* matrix_shards, const mfsdp_tail_shard* tail_shards,
                           const float* momentum, const float* tail_p, const float* tail_m,
                           const float* tail_v);

/* Reads only the header of a checkpoint file (to size the buffers of
 * mfsdp_checkpoint_read).  Errors: INVALID_ARG, IO, FORMAT. */
int mfsdp_checkpoint_read_header(const char* path, mfsdp_checkpoint_header* header);

/* Reads a whole checkpoint into caller-provided host buffers of the given
 * capacities (shards, momentum elements, tail elements); the digest and the
 * tables are checked before anything is reported.  *header is written only on
 * success.  Errors: INVALID_ARG, IO, FORMAT (wrong magic or version, a
 * damaged, truncated or over-long file, tables outside the buffers),
 * WORKSPACE_TOO_SMALL (a capacity below the file's counts). */
int mfsdp_checkpoint_read(const char* path, mfsdp_checkpoint_header* header,
                          mfsdp_matrix_shard* matrix_shards, int32_t matrix_capacity,
                          mfsdp_tail_shard* tail_shards, int32_t tail_capacity,
                          float* momentum, int64_t momentum_capacity,
                          float* tail_p, float* tail_m, float* tail_v, int64_t tail_capacity_elems);

/* Static description of a status code (never NULL). */
const char* mfsdp_status_string(int status);

/* Library version as "major.minor.patch". */
const char* mfsdp_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MFSDP_H */
