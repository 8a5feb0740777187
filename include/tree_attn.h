/*
 * tree_attn.h -- C ABI of libtreeattn: causal softmax attention over a packed
 * rollout prefix tree, forward and backward, on one GB300 (sm_103a).
 *
 * What it computes.  RL rollouts share long prefixes and form a tree, often an
 * irregular one (AReaL-DTA abstract; HARTS abstract).  Each shared prefix is
 * stored once: the compact token sequence
 * lists the node segments in depth-first pre-order (roots, then children, in
 * ascending node id).  Query token i attends to key token j exactly when j
 * lies on i's root-to-node path and, inside i's own segment, j <= i.  So every
 * token gets the output and the gradients that training its root-to-leaf
 * trajectory on its own would give -- the equivalence both abstracts ask for --
 * while each shared prefix is computed once instead of once per trajectory.
 *
 *   S_ij = softmax_scale * q_i . k_j            (attended pairs only)
 *   LSE_i = ln sum_j exp(S_ij),   P_ij = exp(S_ij - LSE_i),   O_i = sum_j P_ij v_j
 *   backward: dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dO * O)),
 *             dQ = scale dS K, dK = scale dS^T Q
 *
 * Grouped-query attention: q-head h uses kv-head h / (hq / hkv); dK and dV sum
 * over the q-heads of a group.
 *
 * Conventions for every call:
 *  - Status: 0 = success, negative = error (TREE_ATTN_ERR_*); no call exits
 *    or throws across this boundary.  tree_attn_strerror() names a code.
 *  - Host pointers are read during the call only.  Device pointers and the
 *    workspace belong to the caller and must stay valid until the work queued
 *    on `stream` has finished.  The plan belongs to the library.
 *  - Device tensors are contiguous, token-major, in packed order:
 *      Q, O, dO, dQ  [N, hq, d] bf16;  K, V, dK, dV  [N, hkv, d] bf16;
 *      LSE [hq, N] fp32 (natural log).
 *    Every device pointer must be 16-byte aligned.
 *  - fwd/bwd are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream).  Launch errors are returned; faults
 *    inside a kernel surface at the caller's next synchronising call.
 *  - A plan is immutable once made and may be used from several host threads
 *    and streams at once.  Its device copy is uploaded on the first fwd/bwd on
 *    each device (or by tree_attn_plan_upload); that first call allocates
 *    device memory and synchronises, so make it outside stream capture.
 *    After it, tree_attn_fwd, tree_attn_bwd and tree_attn_bwd_stages allocate
 *    nothing and do not synchronise, so a whole step can be captured in a CUDA
 *    graph and replayed (what launch-bound small trees want).
 *  - The attention kernels are launched with programmatic stream
 *    serialization: each one's set-up may overlap the end of the kernel before
 *    it on the stream, and waits (griddepcontrol.wait) for that kernel to
 *    complete before it reads or writes any tensor; each one then allows the
 *    next kernel to start early.  A caller's own kernel launched after ours
 *    with the same attribute must likewise wait before it reads our outputs
 *    (kernels launched without it simply run after ours, as usual).
 */
#ifndef TREE_ATTN_H
#define TREE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define TREE_ATTN_OK                   0
#define TREE_ATTN_ERR_INVALID_ARG     -1  /* null pointer, bad size or count      */
#define TREE_ATTN_ERR_INVALID_TREE    -2  /* parent out of range, self-parent,
                                             cycle, no root, seg_len <= 0         */
#define TREE_ATTN_ERR_TOO_LARGE       -3  /* token count or plan size overflows   */
#define TREE_ATTN_ERR_UNSUPPORTED     -4  /* head_dim not 64/128, hq % hkv != 0,
                                             plan block size not 128 for kernels  */
#define TREE_ATTN_ERR_ALIGNMENT       -5  /* device pointer not 16-byte aligned   */
#define TREE_ATTN_ERR_WORKSPACE       -6  /* workspace null or too small          */
#define TREE_ATTN_ERR_CUDA            -7  /* CUDA runtime / driver call failed    */
#define TREE_ATTN_ERR_NO_DEVICE       -8  /* no usable sm_103 device              */
#define TREE_ATTN_ERR_OUT_OF_MEMORY   -9  /* host or device allocation failed     */
#define TREE_ATTN_ERR_DEVICE_TIMEOUT -10  /* a bounded device wait ran out        */
#define TREE_ATTN_ERR_SCRATCH_TOO_SMALL -11 /* tree_attn_bwd_noalloc: the problem
                                             needs more than its fixed scratch    */
#define TREE_ATTN_ERR_INVALID_DECAY  -12  /* device status only: a linear-attention
                                             decay outside (0, 1]                 */
#define TREE_ATTN_ERR_DEVICE_BOUNDS  -13  /* device status only, debug builds: an
                                             index failed its bounds check        */

/* ---- tile classes (tree_attn_plan_export) ------------------------------- */
#define TREE_ATTN_TILE_FULL     1   /* every valid (query, key) pair attended  */
#define TREE_ATTN_TILE_PARTIAL  2   /* some pairs attended; mask per element   */
/* empty blocks are never listed, never loaded and never computed            */

typedef struct tree_attn_plan_s* tree_attn_plan_t;

typedef struct {
    int32_t block;            /* tile edge for queries and keys; 0 = 128.  The
                                 kernels run 128 only; other sizes (1..1024)
                                 are accepted for inspecting the plan.        */
    int32_t bwd_chunk_qtiles; /* max q-tiles per backward work item; 0 = auto:
                                 24 for fewer than 64 q-tiles, 48 for fewer
                                 than 256, else 64; doubled while the kv-tiles
                                 split over several items would need more than
                                 max(2048, 8 * n_qtiles) partial slots        */
    int32_t bwd_cta_order;    /* order of the backward's CTAs inside a chunk:
                                 0 = auto (head-major when a chunk's fp32 dQ
                                 rows, chunk * 128 * hq * d * 4 bytes, exceed
                                 192 MB), 1 = item-major (the kv-heads of an
                                 item side by side), 2 = head-major (every item
                                 of kv-head 0, then of kv-head 1, ...).  The
                                 order changes no result bit of dK and dV.    */
} tree_attn_plan_opts_t;

typedef struct {
    int64_t n_tokens;         /* N, compact tokens                            */
    int32_t n_nodes;
    int32_t block;
    int32_t n_qtiles;         /* T = ceil(N / block); also the kv-tile count  */
    int32_t n_bwd_items;      /* backward work items (kv-tile, q-tile chunk)  */
    int64_t n_pairs;          /* attended (query, key) pairs                  */
    int64_t n_intervals;      /* key intervals summed over q-tiles            */
    int64_t n_tile_entries;   /* non-empty (q-tile, kv-tile) blocks           */
    int64_t n_full_tiles;     /* of which full                                */
    int32_t n_split_kv_tiles; /* kv-tiles whose q-range spans >1 work item    */
    int32_t bwd_chunk_qtiles; /* chunk size in force                          */
    int64_t n_partial_slots;  /* dK/dV partial buffers the backward needs     */
} tree_attn_plan_info_t;

/* Caller-allocated destinations for tree_attn_plan_export; any may be NULL.  */
typedef struct {
    int32_t* node_order;  /* [n_nodes]     node id at each packed position      */
    int32_t* node_off;    /* [n_nodes]     first packed token of node v (by id) */
    int32_t* subend;      /* [n_tokens]    one past the last query attending
                                           key j = end of j's subtree           */
    int32_t* qi_ptr;      /* [n_qtiles+1]  CSR offsets into qi_lo / qi_hi       */
    int32_t* qi_lo;       /* [n_intervals] maximal key intervals [lo, hi) of    */
    int32_t* qi_hi;       /*               each q-tile, ascending               */
    int32_t* qt_ptr;      /* [n_qtiles+1]  CSR offsets into qt_kv / qt_cls      */
    int32_t* qt_kv;       /* [n_tile_entries] non-empty kv-tiles, ascending     */
    uint8_t* qt_cls;      /* [n_tile_entries] TREE_ATTN_TILE_FULL / _PARTIAL    */
    int32_t* kv_qlo;      /* [n_qtiles]    q-tiles [kv_qlo, kv_qhi) use kv-tile */
    int32_t* kv_qhi;      /* [n_qtiles]                                         */
    int32_t* fwd_order;   /* [n_qtiles]    q-tiles, heaviest first              */
    int32_t* bwd_items;   /* [4*n_bwd_items] {kv-tile, q-tile begin, end,
                                           partial slot or -1}: q-ranges cut at
                                           multiples of bwd_chunk_qtiles, run
                                           chunk by chunk, longest first within */
} tree_attn_plan_arrays_t;

/* Build a plan from a rollout tree or forest (host only, no GPU needed).
 * parent[v]: parent node id, -1 for a root.  seg_len[v] > 0: tokens of node v.
 * n_nodes >= 1 (an empty tree is TREE_ATTN_ERR_INVALID_ARG; the smallest
 * input is one node of one token).
 * Section: AReaL-DTA abstract (DFS traversal of the rollout prefix tree);
 * HARTS abstract (arbitrary rollout trees; prefix compression to compact
 * tokens).  opts may be NULL.  *out receives a new plan on success. */
int tree_attn_plan(const int32_t* parent, const int32_t* seg_len, int32_t n_nodes,
                   const tree_attn_plan_opts_t* opts, tree_attn_plan_t* out);

int tree_attn_plan_info(tree_attn_plan_t plan, tree_attn_plan_info_t* info);

/* Copy plan arrays into caller buffers sized per tree_attn_plan_info(). */
int tree_attn_plan_export(tree_attn_plan_t plan, const tree_attn_plan_arrays_t* dst);

/* Upload the plan's device tables to the current device now (optional; the
 * first fwd/bwd on a device does it otherwise).  Allocates and synchronises. */
int tree_attn_plan_upload(tree_attn_plan_t plan);

/* Bytes of device workspace fwd and bwd need for these head sizes. */
int tree_attn_workspace_size(tree_attn_plan_t plan, int32_t hq, int32_t hkv, int32_t d,
                             size_t* fwd_bytes, size_t* bwd_bytes);

/* Forward: O and LSE (see the formulas above).  softmax_scale (> 0, finite)
 * is applied to the logits (pass 1/sqrt(d) for standard attention).  d in {64, 128}.  The
 * forward needs no workspace (pass NULL, 0).  Work is queued on `stream`.
 * Section: AReaL-DTA abstract (each shared prefix computed once in the forward
 * pass, with every trajectory's result unchanged); HARTS abstract (attention
 * over compact tokens of an arbitrary rollout tree, equal to per-trajectory
 * training).  Only the kv-tiles on a q-tile's ancestor list are loaded.
 * Errors: INVALID_ARG (null pointer, scale not finite or <= 0), UNSUPPORTED
 * (head layout), TOO_LARGE, ALIGNMENT, NO_DEVICE, OUT_OF_MEMORY (the plan's
 * first upload), CUDA (launch). */
int tree_attn_fwd(tree_attn_plan_t plan, const void* q, const void* k, const void* v,
                  void* o, float* lse, int32_t hq, int32_t hkv, int32_t d,
                  float softmax_scale, void* workspace, size_t ws_bytes, void* stream);

/* Backward: dQ, dK, dV from Q, K, V, the forward's O and LSE, and dO.  Needs
 * the workspace tree_attn_workspace_size reports (device memory, 256-byte
 * aligned, contents on entry ignored).  dK and dV are reduced over a kv-tile's
 * descendant q-tiles in a fixed order, so they are bitwise reproducible; dQ is
 * accumulated with fp32 atomics, so its last bits may vary run to run.
 * Section: AReaL-DTA abstract and HARTS abstract (the backward pass too
 * computes each shared prefix once, and every trajectory gets the gradients
 * training it alone would give).  dout is the compact gradient of one scalar
 * loss (per-trajectory weights already folded in, e.g. tree_attn_scale_rows).
 * Errors as tree_attn_fwd, plus WORKSPACE (missing or smaller than reported;
 * ALIGNMENT when not 256-byte aligned). */
int tree_attn_bwd(tree_attn_plan_t plan, const void* q, const void* k, const void* v,
                  const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, int32_t hq, int32_t hkv, int32_t d,
                  float softmax_scale, void* workspace, size_t ws_bytes, void* stream);

/* The backward in stages (the same arguments as tree_attn_bwd, plus a mask):
 *   TREE_ATTN_BWD_PRE  -- Delta = rowsum(dO * O), LSE in log2 units, zero the
 *                         fp32 dQ accumulator (memory-bound)
 *   TREE_ATTN_BWD_MAIN -- the tensor-core pass over (kv-tile, q-tile) blocks
 *   TREE_ATTN_BWD_POST -- dQ to bf16; fixed-order sum of split dK/dV partials
 * Stages must run in this order, on one stream, with one workspace;
 * tree_attn_bwd is all three.  Lets a caller time or overlap each stage. */
#define TREE_ATTN_BWD_PRE  1
#define TREE_ATTN_BWD_MAIN 2
#define TREE_ATTN_BWD_POST 4
int tree_attn_bwd_stages(tree_attn_plan_t plan, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout,
                         void* dq, void* dk, void* dv, int32_t hq, int32_t hkv, int32_t d,
                         float softmax_scale, void* workspace, size_t ws_bytes, void* stream,
                         int32_t stages);

/* Backward that allocates nothing.  (The pages have no counterpart: this is a
 * convenience of this library.)  Some callers cannot call cudaMalloc or
 * cudaFree at the point where they run the backward: code whose device memory
 * is owned by another allocator (a framework's caching pool that has claimed
 * the memory), code that must not synchronise the device (cudaMalloc and
 * cudaFree can), or code held to a fixed memory budget.  This entry point takes
 * the same tensors as tree_attn_bwd but no workspace: the plan's tables and the
 * workspace go into one fixed array in device memory that the library declares
 * at file scope, tree_attn_noalloc_scratch_bytes() bytes (32 MiB), held by every
 * device that loads the library until the process exits.
 *  - Problems whose tables plus workspace exceed that size are rejected with
 *    TREE_ATTN_ERR_SCRATCH_TOO_SMALL (use tree_attn_bwd with a workspace).
 *  - Every call uses the same array.  Calls that run at the same time on the
 *    GPU (different streams, or different host threads) race on it; serialise
 *    them, e.g. on one stream.  Each call overwrites the array before reading
 *    it, so nothing from an earlier call leaks into the result.
 *  - The first call on a device looks up the array's device address.  Each
 *    call copies the plan tables into the array from pageable host memory:
 *    4 bytes per token (rounded up to a multiple of 128 tokens), 4 per q-tile
 *    and 16 per backward work item, e.g. 45 KB for an 11k-token tree.  A copy
 *    from pageable memory is staged through the driver before the call returns,
 *    so the host waits for it, and such a copy is not allowed during stream
 *    capture: this call cannot be captured in a CUDA graph (capture
 *    tree_attn_bwd with a workspace instead).  The call makes no cudaMalloc,
 *    cudaFree or other allocating call.
 * Arguments, layouts, stream semantics and the other status codes are those of
 * tree_attn_bwd. */
int tree_attn_bwd_noalloc(tree_attn_plan_t plan, const void* q, const void* k, const void* v,
                          const void* o, const float* lse, const void* dout,
                          void* dq, void* dk, void* dv, int32_t hq, int32_t hkv, int32_t d,
                          float softmax_scale, void* stream);

/* Size in bytes of the fixed scratch tree_attn_bwd_noalloc uses. */
size_t tree_attn_noalloc_scratch_bytes(void);

/* Synchronise `stream`, then read and clear the device status word of the
 * current device: 0 when every kernel's bounded waits finished in time,
 * otherwise TREE_ATTN_ERR_DEVICE_TIMEOUT - 1000 * (site of the wait),
 * TREE_ATTN_ERR_ALIGNMENT (shared memory misaligned) or
 * TREE_ATTN_ERR_INVALID_DECAY (tree_linear.h: a decay outside (0, 1]), or in
 * a debug build TREE_ATTN_ERR_DEVICE_BOUNDS - 1000 * (site of the check).  The
 * first error recorded wins.  Kernels that hit a failed wait return early and
 * leave their outputs incomplete. */
int tree_attn_get_device_status(void* stream);

/* Self-test of the kernels' failure path: launches one thread that waits on a
 * barrier nothing completes, bounded by limit_ms (1..2000), so the wait runs
 * out, records TREE_ATTN_ERR_DEVICE_TIMEOUT - 1000 * 99 in the device status
 * word and the kernel returns -- the same path every bounded wait of the
 * attention kernels takes, with no fault and the context still usable.  Read
 * the result with tree_attn_get_device_status. */
int tree_attn_selftest_wait_timeout(int32_t limit_ms, void* stream);

/* Debug builds.  The library built with -DTREE_ATTN_DEBUG (libtreeattn_debug.so,
 * made beside libtreeattn.so by the package's build) checks, in every attention
 * kernel, the indices that come from the plan's tables and the tree's shape --
 * work items, q-tile kv-tile lists, subtree ends of partial and ragged tiles,
 * partial dK/dV slots, LSE / Delta rows, head numbers -- before they address
 * global memory.  A failed check records TREE_ATTN_ERR_DEVICE_BOUNDS - 1000 *
 * site in the device status word and the access is skipped or clamped to an
 * in-range index, so nothing is read or written out of bounds; the results are
 * then wrong, and the status says where.  (It stands in for a memory checker
 * that cannot run on every machine.)  Release builds carry no checks.
 * tree_attn_debug_checks() is 1 in a debug build, 0 otherwise. */
int tree_attn_debug_checks(void);

/* Self-test of the debug checks: one thread checks an index that is out of
 * range on purpose, so a debug build records TREE_ATTN_ERR_DEVICE_BOUNDS -
 * 1000 * 98 in the device status word (read it with
 * tree_attn_get_device_status) and skips the access.  Release builds return
 * TREE_ATTN_ERR_UNSUPPORTED and launch nothing. */
int tree_attn_selftest_bounds(void* stream);

/* Free the plan and its device copies (call after work using it finished). */
void tree_attn_plan_destroy(tree_attn_plan_t plan);

const char* tree_attn_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif /* TREE_ATTN_H */
