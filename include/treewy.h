/*
 * treewy.h -- C ABI of the TreeWY speculative-verification library for Gated
 * DeltaNet (GDN) layers on sm_103a (GB300).
 *
 * Method: "TreeWY: Speculative Verification for Gated DeltaNet Hybrids".
 * For one GDN layer, a batch of R requests, H value heads and one draft tree
 * per request, verification computes every draft node's output from the
 * committed state S0 without materialising a per-node state, and commit
 * rebuilds the one accepted state.
 *
 *   gated delta rule (paper §1 Eq. (1)):
 *       S_n = alpha_n S_par (I - beta_n k_n k_n^T) + beta_n v_n k_n^T,  o_n = S_n q_n
 *   pseudo-values U (paper §3 "Key rewrite" and Eq. (2)):
 *       (I + A) U = diag(beta) (V - diag(gamma) (S0 K^T)^T),
 *       A[n,i] = beta_n (gamma_n / gamma_i) (k_i . k_n) for i a strict ancestor of n,
 *       gamma_n = product of alpha over the root-to-n path, n included
 *   outputs (technical review §3.1 Eq. (5), restricted to ancestors as in §3.2):
 *       o_n = gamma_n S0 q_n + sum_{i ancestor of n or n} (gamma_n/gamma_i) (k_i . q_n) u_i
 *   commit (paper §3 "Reconstruct on commit", review Eq. (6)):
 *       S_a = gamma_a S0 + sum_{i on the root-to-a path} (gamma_a/gamma_i) u_i k_i^T
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All pointers in treewy_batch are DEVICE pointers to memory the caller
 *   owns; the library allocates no device memory and keeps no pointer after
 *   a call returns.  Calls are asynchronous on `stream` (0 = legacy default
 *   stream) and never synchronise the host.
 * - Errors the host can see (null pointers, unsupported sizes, misaligned
 *   buffers, launch failures) return a non-zero treewy_status before or at
 *   launch; treewy_last_error() then describes the problem.  Errors in the
 *   contents of device arrays (a parent index out of range, a tree larger
 *   than max_nodes, an accepted index outside the tree, a node range past T)
 *   cannot be seen by the host: the kernels set bits in status[r] for the
 *   request and skip it, leaving its outputs (or its state) untouched.
 * - Node rows: request r owns rows t = node_offset[r] .. node_offset[r+1]-1
 *   of every per-node array, node n of the request being row node_offset[r]+n.
 *   Nodes are in a topological order (every parent precedes its children;
 *   the pages use DFS pre-order, which is one such order).
 */
#ifndef TREEWY_H
#define TREEWY_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum treewy_status {
  TREEWY_OK = 0,
  TREEWY_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misalignment */
  TREEWY_ERR_UNSUPPORTED = 3,   /* sizes outside what the kernels implement */
  TREEWY_ERR_CUDA = 4           /* a CUDA runtime/driver call failed */
} treewy_status;

/* Bits of the per-request device status word.  Kernels only OR bits into
   status[r]; the caller zeroes the array before a round of calls. */
enum {
  TREEWY_STATUS_BAD_TREE = 1,       /* parent[n] outside [-1, n), or node range past T */
  TREEWY_STATUS_TOO_MANY_NODES = 2, /* N_r > max_nodes (or N_r < 0) */
  TREEWY_STATUS_BAD_ACCEPTED = 4,   /* accepted[r] outside [-1, N_r) (commit only) */
  TREEWY_STATUS_BAD_SLOT = 8,       /* state_slot[r] outside [0, num_slots) */
  TREEWY_STATUS_TIMEOUT = 16,       /* an internal wait gave up after ~1 s; that
                                       (request, head) was skipped */
  TREEWY_STATUS_COMMIT_REFUSED = 32 /* treewy_commit_verify only: the previous
                                       round's commit of this request was refused
                                       (its state is unchanged); the bits beside
                                       it say why */
};

/* Element type of q, k and v. */
enum {
  TREEWY_DTYPE_BF16 = 0,
  TREEWY_DTYPE_F32 = 1
};

/* Flags. */
enum {
  /* Use the portable kernels (CUDA cores, no bulk tensor copies) even where
     the tensor-core verification (dk = dv = 128, bf16 q/k/v: warp-level
     MMAs for batches of trees of at most 32 nodes, tcgen05 above) or the
     bulk-copy commit (dk = dv = 128) applies.  Same results within rounding. */
  TREEWY_FLAG_FORCE_GENERIC = 1u,
  /* The state pool holds bf16 instead of f32: the dtype in which the GDN
     state is kept when serving (paper §2 "The memory problem": dv x dk x 2 B
     per head), half the bytes of every state read and write.  Verification
     takes the bf16 S0 as exact values; commit forms S_a in f32 and stores it
     rounded to nearest (ties to even) bf16, so each committed element is
     within 2^-8 of its relative value.  The storeall comparator entry points
     reject this flag with TREEWY_ERR_UNSUPPORTED. */
  TREEWY_FLAG_STATE_BF16 = 2u
};

/* Largest draft tree per request. */
#define TREEWY_MAX_NODES 64

/*
 * One GDN layer's worth of draft-tree data.
 *
 * Sizes: R >= 0 requests, H >= 1 value heads, key/value head sizes
 * 1 <= dk, dv <= 128 (the tensor-core path needs dk = dv = 128 and bf16
 * q/k/v; every other size runs the CUDA-core path), 1 <= max_nodes <= 64,
 * T >= node_offset[R] rows in every per-node array, num_slots >= 1 blocks in
 * the state pool, R * H < 2^31 (request, head) pairs.
 *
 * Layouts (row-major, innermost index last; all device memory):
 *   node_offset  int32 [R+1], non-decreasing
 *   parent       int32 [T]        request-local parent index, -1 = hangs off S0
 *   q, k         bf16|f32 [T][H][dk]   (16-byte aligned base)
 *   v            bf16|f32 [T][H][dv]   (16-byte aligned base)
 *   alpha, beta  f32 [T][H]       decay gate and write strength, in (0,1)
 *   state        f32 [num_slots][H][dv][dk]  committed states S0 (row d of a
 *                                 head's state holds S0[d][0..dk-1]); 16-byte aligned;
 *                                 bf16, same shape, with TREEWY_FLAG_STATE_BF16
 *   state_slot   int32 [R]        pool slot of each request, in [0, num_slots)
 *   o            f32 [T][H][dv]   verify output o_n (16-byte aligned base)
 *   U            f32 [T][H][dv]   verify output u_n, commit input (16-byte
 *                                 aligned base; keep it
 *                                 alive from verify to commit: it replaces
 *                                 the per-node snapshots)
 *   gamma        f32 [T][H]       optional verify output gamma_n (may be NULL)
 *   status       int32 [R]        per-request error bits, OR-ed (see above)
 * The per-node arrays (parent, q, k, v, alpha, beta, o, U, gamma) may be
 * NULL when T = 0, a batch whose trees are all empty.
 */
typedef struct treewy_batch {
  int32_t R;
  int32_t H;
  int32_t dk;
  int32_t dv;
  int32_t max_nodes;
  int32_t qkv_dtype;
  int64_t T;
  int64_t num_slots;
  const int32_t* node_offset;
  const int32_t* parent;
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  void* state;                    /* f32, or bf16 with TREEWY_FLAG_STATE_BF16 */
  const int32_t* state_slot;
  float* o;
  float* U;
  float* gamma;
  int32_t* status;
  uint32_t flags;
  uint32_t reserved;
} treewy_batch;

/*
 * treewy_verify -- TreeWY verification of every draft node
 * (paper §3 "Verifying a draft", Eq. (2); review §3.2 Algorithm, steps 1-5).
 *
 * Reads node_offset, parent, q, k, v, alpha, beta, state (through
 * state_slot); writes o, U, gamma (if non-NULL) and ORs error bits into
 * status[r].  The outputs of a request with an error bit are left untouched.
 * The state is not modified.
 */
treewy_status treewy_verify(const treewy_batch* batch, cudaStream_t stream);

/*
 * treewy_commit -- reconstruct the accepted state in place
 * (paper §3 "Reconstruct on commit", Eq. (3); review §3.3, Eq. (6)).
 *
 * accepted: device int32 [R], request-local index of the accepted node, or -1
 * when no draft node is accepted (the state is then left untouched and not
 * read).  Reads node_offset, parent, alpha, k, U (from treewy_verify on the
 * same inputs) and state; overwrites state[state_slot[r]] with S_a.  q, v and
 * o are not read.  Requests with a bad tree or accepted index get status bits
 * OR-ed into status[r] and keep their state.  Requests must map to distinct
 * slots (two requests committing into one slot race).
 */
treewy_status treewy_commit(const treewy_batch* batch, const int32_t* accepted,
                            cudaStream_t stream);

/*
 * treewy_commit_verify -- the previous round's commit fused into this round's
 * verification (the deferred state write that the paper's §6 and the review's
 * §7(c)(3) point to: write the accepted state once, inside the next pass that
 * reads it).
 *
 * For every request r, state[state_slot[r]] holds S0 of the previous round;
 * `prev` describes that round (node_offset, parent, alpha, k and U from its
 * treewy_verify; q, v, o, beta are not read) and prev_accepted its accepted
 * nodes (device int32 [R], -1 = nothing accepted).  The kernel rebuilds
 * S_a = gamma_a S0 + sum_{i on path(a)} (gamma_a/gamma_i) u_i k_i^T on chip,
 * writes it back to the state block once, and verifies `next` from it: the
 * results equal treewy_commit(prev, prev_accepted) followed by
 * treewy_verify(next), with one state read per head instead of two.  (Shapes
 * other than dk = dv = 128 with bf16 q/k/v in both rounds, and a bf16 pool
 * whose next trees have at most 8 nodes while the previous ones have more
 * than 8, or 9 to 32 nodes while the previous ones have more than 16,
 * run as those two calls back to back on `stream`.)  A request with no node
 * in `next` still gets its commit.  prev and next must have the
 * same R, H, dk, dv, state pool pointer, num_slots, state_slot pointer and
 * TREEWY_FLAG_STATE_BF16.
 * Errors, as for the two calls made one after the other, with every status
 * bit going to next->status:
 *   - an error in the previous round (its tree, node range or accepted index)
 *     refuses that request's commit: its state is left unchanged, the bits of
 *     the reason are set together with TREEWY_STATUS_COMMIT_REFUSED, and `next`
 *     is still verified, from the unchanged state;
 *   - an error in `next` (its tree or node range) skips that request's
 *     verification (outputs untouched) but not its commit: S_a is written;
 *   - a state slot outside the pool refuses both (TREEWY_STATUS_BAD_SLOT |
 *     TREEWY_STATUS_COMMIT_REFUSED when a node was accepted).
 * So S_a was written for request r exactly when prev_accepted[r] >= 0 and
 * TREEWY_STATUS_COMMIT_REFUSED is clear in next->status[r].
 */
treewy_status treewy_commit_verify(const treewy_batch* prev, const int32_t* prev_accepted,
                                   const treewy_batch* next, cudaStream_t stream);

/*
 * treewy_storeall_verify -- the snapshot-per-node comparator ("storeall", the
 * full-state snapshotting of paper §2, approach (i)).
 *
 * Applies the gated delta rule node by node and writes every node's state to
 * snapshots, plus o (and U is not written).  snapshots: device f32
 * [T'][H][dv][dk] where T' = node_offset[R] - node_offset[0]: snapshot rows
 * are indexed relative to the batch's first node, so a caller can verify a
 * large batch in request chunks (pass node_offset + r0 and R_chunk) with
 * snapshot memory for one chunk only.  16-byte aligned.  status as in
 * treewy_verify.
 */
treewy_status treewy_storeall_verify(const treewy_batch* batch, float* snapshots,
                                     cudaStream_t stream);

/*
 * treewy_storeall_commit -- storeall rollback: copy the accepted node's
 * snapshot into state[state_slot[r]] (nothing for accepted = -1).
 * snapshots indexed as in treewy_storeall_verify for the same batch.
 */
treewy_status treewy_storeall_commit(const treewy_batch* batch, const float* snapshots,
                                     const int32_t* accepted, cudaStream_t stream);

/*
 * treewy_selftest_wait_timeout -- diagnostic of the kernels' bounded waits.
 *
 * Launches one thread that waits, with the same bounded wait every kernel
 * uses on its barriers, for a barrier phase that nothing completes, giving
 * up after limit_us microseconds (1 .. 10,000,000).  It then ORs
 * TREEWY_STATUS_TIMEOUT into status[0] and writes the measured wait in
 * nanoseconds to the two int32 words status[1] (low) and status[2] (high).
 * status: device int32 [3], caller-owned; the caller zeroes status[0].
 * Shows that a wait which never completes returns control, reports through
 * the status word and leaves the CUDA context usable.
 */
treewy_status treewy_selftest_wait_timeout(int32_t* status, uint32_t limit_us,
                                           cudaStream_t stream);

/* Message for the last non-OK return on the calling host thread ("" if none). */
const char* treewy_last_error(void);

/* Library version string. */
const char* treewy_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TREEWY_H */
