// treewy_api.cu -- the C ABI entry points: argument validation, tensor-map
// construction for the tensor-core path, kernel dispatch and error reporting.
// No device memory is allocated here and the host never synchronises.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "treewy_internal.h"

namespace {

thread_local std::string g_last_error;

treewy_status fail(treewy_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

treewy_status cuda_fail(cudaError_t err, const char* what) {
  return fail(TREEWY_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-visible checks common to every entry point.
treewy_status validate(const treewy_batch* b, bool need_qv, bool need_outputs, bool need_k,
                       bool need_tree = true) {
  if (b == nullptr) return fail(TREEWY_ERR_INVALID_ARG, "batch is NULL");
  if (b->R < 0) return fail(TREEWY_ERR_INVALID_ARG, "R = %d is negative", b->R);
  if (b->H < 1) return fail(TREEWY_ERR_INVALID_ARG, "H = %d must be >= 1", b->H);
  if (b->dk < 1 || b->dv < 1)
    return fail(TREEWY_ERR_INVALID_ARG, "dk = %d, dv = %d must be >= 1", b->dk, b->dv);
  if (b->dk > 128 || b->dv > 128)
    return fail(TREEWY_ERR_UNSUPPORTED, "dk = %d, dv = %d: head sizes above 128 are not supported",
                b->dk, b->dv);
  if (b->max_nodes < 1 || b->max_nodes > TREEWY_MAX_NODES)
    return fail(TREEWY_ERR_UNSUPPORTED, "max_nodes = %d outside [1, %d]", b->max_nodes,
                TREEWY_MAX_NODES);
  if (b->qkv_dtype != TREEWY_DTYPE_BF16 && b->qkv_dtype != TREEWY_DTYPE_F32)
    return fail(TREEWY_ERR_INVALID_ARG, "qkv_dtype = %d is not TREEWY_DTYPE_BF16/F32", b->qkv_dtype);
  if (b->flags & ~(TREEWY_FLAG_FORCE_GENERIC | TREEWY_FLAG_STATE_BF16))
    return fail(TREEWY_ERR_INVALID_ARG, "flags = 0x%x has unknown bits", b->flags);
  if (b->T < 0 || b->T > (int64_t(1) << 31) - 1)
    return fail(TREEWY_ERR_INVALID_ARG, "T = %lld outside [0, 2^31)", (long long)b->T);
  if (int64_t(b->R) * b->H > (int64_t(1) << 31) - 1)
    return fail(TREEWY_ERR_UNSUPPORTED, "R * H = %lld (request, head) pairs exceed 2^31 - 1",
                (long long)(int64_t(b->R) * b->H));
  if (b->num_slots < 1) return fail(TREEWY_ERR_INVALID_ARG, "num_slots = %lld must be >= 1",
                                    (long long)b->num_slots);
  if (b->num_slots * b->H * int64_t(b->dv) > (int64_t(1) << 31) - 1)
    return fail(TREEWY_ERR_UNSUPPORTED, "state pool rows num_slots*H*dv exceed 2^31");
  if (b->T * b->H * int64_t(b->dv > b->dk ? b->dv : b->dk) > (int64_t(1) << 40))
    return fail(TREEWY_ERR_UNSUPPORTED, "per-node arrays too large");
  if (b->R == 0) return TREEWY_OK;
  if (!b->node_offset || !b->state || !b->state_slot || !b->status)
    return fail(TREEWY_ERR_INVALID_ARG,
                "node_offset, state, state_slot and status must be non-NULL");
  // per-node arrays have T rows; with T = 0 (every tree empty) they may be NULL
  const bool rows = b->T > 0;
  if (rows && need_tree && (!b->parent || !b->alpha))
    return fail(TREEWY_ERR_INVALID_ARG, "parent and alpha must be non-NULL");
  if (rows && need_k && !b->k) return fail(TREEWY_ERR_INVALID_ARG, "k is NULL");
  if (rows && need_qv && (!b->q || !b->v || !b->beta))
    return fail(TREEWY_ERR_INVALID_ARG, "q, v and beta must be non-NULL");
  if (rows && need_outputs && (!b->o || !b->U))
    return fail(TREEWY_ERR_INVALID_ARG, "o and U must be non-NULL");
  if (!aligned16(b->state)) return fail(TREEWY_ERR_INVALID_ARG, "state must be 16-byte aligned");
  if (need_k && !aligned16(b->k)) return fail(TREEWY_ERR_INVALID_ARG, "k must be 16-byte aligned");
  if (need_qv && (!aligned16(b->q) || !aligned16(b->v)))
    return fail(TREEWY_ERR_INVALID_ARG, "q and v must be 16-byte aligned");
  if (need_outputs && (!aligned16(b->o) || !aligned16(b->U)))
    return fail(TREEWY_ERR_INVALID_ARG, "o and U must be 16-byte aligned");
  return TREEWY_OK;
}

bool use_tensor_cores(const treewy_batch* b) {
  return b->dk == 128 && b->dv == 128 && b->qkv_dtype == TREEWY_DTYPE_BF16 &&
         (b->flags & TREEWY_FLAG_FORCE_GENERIC) == 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

// State pool of a dk = dv = 128 batch as rows [slots*H*128][128]; one box =
// box_rows state rows x 128 bytes (32 f32 or 64 bf16 columns), 128-byte swizzle.
treewy_status make_state_map(const treewy_batch* b, CUtensorMap* map, uint32_t box_rows = 128) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return fail(TREEWY_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint32_t ones[2] = {1, 1};
  const bool sb = (b->flags & TREEWY_FLAG_STATE_BF16) != 0;
  const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(b->num_slots) * b->H * 128};
  const cuuint64_t strides[1] = {128 * (sb ? 2u : 4u)};
  const cuuint32_t box[2] = {sb ? 64u : 32u, box_rows};
  CUresult rc = enc(map, sb ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                    b->state, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (rc != CUDA_SUCCESS) return fail(TREEWY_ERR_CUDA, "tensor map for state failed (%d)", (int)rc);
  return TREEWY_OK;
}

treewy_status make_maps(const treewy_batch* b, treewy::VerifyMaps* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return fail(TREEWY_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint32_t ones[3] = {1, 1, 1};
  treewy_status st = make_state_map(b, &m->s0);
  if (st != TREEWY_OK) return st;
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(b->H), static_cast<cuuint64_t>(b->T)};
  const cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(b->H) * 128 * 2};
  // boxes of 32 and 16 rows: a tree's rows, rounded up to 16, take at most
  // two boxes per tensor and 64-column chunk
  const cuuint32_t box16[3] = {64, 1, 16};
  const cuuint32_t box32[3] = {64, 1, 32};
  const void* ptrs[4] = {b->k, b->q, b->k, b->q};
  CUtensorMap* maps[4] = {&m->k, &m->q, &m->k32, &m->q32};
  for (int i = 0; i < 4; ++i) {
    CUresult rc = enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptrs[i]), dims,
                      strides, i < 2 ? box16 : box32, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rc != CUDA_SUCCESS)
      return fail(TREEWY_ERR_CUDA, "tensor map for %s failed (%d)", (i & 1) ? "q" : "k", (int)rc);
  }
  return TREEWY_OK;
}

// Commit with the bulk-copy kernel for dk = dv = 128 (unless the portable
// kernels are forced), with the register-streaming kernel otherwise.
treewy_status launch_commit_any(const treewy_batch* b, const int32_t* accepted, int refused_bit,
                                cudaStream_t stream, const char* what) {
  cudaError_t err;
  if (b->dk == 128 && b->dv == 128 && (b->flags & TREEWY_FLAG_FORCE_GENERIC) == 0) {
    // tiles of 64 rows for an f32 pool (two CTAs per head), 128 rows for bf16
    CUtensorMap map;
    treewy_status st = make_state_map(b, &map, (b->flags & TREEWY_FLAG_STATE_BF16) ? 128u : 64u);
    if (st != TREEWY_OK) return st;
    err = treewy::launch_commit_tma(*b, map, accepted, refused_bit, stream);
  } else {
    err = treewy::launch_commit(*b, accepted, refused_bit, stream);
  }
  return err == cudaSuccess ? TREEWY_OK : cuda_fail(err, what);
}

}  // namespace

extern "C" {

const char* treewy_last_error(void) { return g_last_error.c_str(); }

const char* treewy_version(void) { return "treewy-gb300 0.1 (sm_103a)"; }

treewy_status treewy_selftest_wait_timeout(int32_t* status, uint32_t limit_us, cudaStream_t stream) {
  g_last_error.clear();
  if (status == nullptr) return fail(TREEWY_ERR_INVALID_ARG, "status is NULL");
  if ((reinterpret_cast<uintptr_t>(status) & 3u) != 0)
    return fail(TREEWY_ERR_INVALID_ARG, "status is not 4-byte aligned");
  if (limit_us < 1u || limit_us > 10000000u)
    return fail(TREEWY_ERR_INVALID_ARG, "limit_us %u outside 1 .. 10,000,000", limit_us);
  const cudaError_t err = treewy::launch_wait_selftest(status, limit_us, stream);
  return err == cudaSuccess ? TREEWY_OK : cuda_fail(err, "treewy_selftest_wait_timeout launch");
}

treewy_status treewy_verify(const treewy_batch* batch, cudaStream_t stream) {
  g_last_error.clear();
  treewy_status st = validate(batch, true, true, true);
  if (st != TREEWY_OK || batch->R == 0) return st;
  cudaError_t err;
  // Trees of at most kSmallTreeNodes nodes are verified by the small-tree
  // kernel, of at most kWarpTreeNodes by the warp-MMA kernel (both multiply
  // straight from the state tile), larger ones by the tcgen05 kernel.  (A
  // batch of empty trees, T = 0, goes to the portable kernel: there are no
  // rows to map, and it still checks node_offset and the slots.)
  if (use_tensor_cores(batch) && batch->T > 0 && batch->max_nodes <= treewy::kWarpTreeNodes) {
    CUtensorMap map;
    st = make_state_map(batch, &map);
    if (st != TREEWY_OK) return st;
    err = batch->max_nodes <= treewy::kSmallTreeNodes
              ? treewy::launch_verify_small(*batch, map, nullptr, stream)
              : treewy::launch_verify_warp(*batch, map, nullptr, stream);
  } else if (use_tensor_cores(batch) && batch->T > 0) {
    treewy::VerifyMaps maps;
    st = make_maps(batch, &maps);
    if (st != TREEWY_OK) return st;
    err = treewy::launch_verify_tc(*batch, maps, batch->max_nodes, stream);
  } else {
    err = treewy::launch_verify_generic(*batch, stream);
  }
  return err == cudaSuccess ? TREEWY_OK : cuda_fail(err, "treewy_verify launch");
}

treewy_status treewy_commit(const treewy_batch* batch, const int32_t* accepted, cudaStream_t stream) {
  g_last_error.clear();
  treewy_status st = validate(batch, false, false, true);
  if (st != TREEWY_OK || batch->R == 0) return st;
  if (!batch->U && batch->T > 0) return fail(TREEWY_ERR_INVALID_ARG, "U is NULL");
  if (!aligned16(batch->U)) return fail(TREEWY_ERR_INVALID_ARG, "U must be 16-byte aligned");
  if (!accepted) return fail(TREEWY_ERR_INVALID_ARG, "accepted is NULL");
  return launch_commit_any(batch, accepted, 0, stream, "treewy_commit launch");
}

treewy_status treewy_commit_verify(const treewy_batch* prev, const int32_t* prev_accepted,
                                   const treewy_batch* next, cudaStream_t stream) {
  g_last_error.clear();
  treewy_status st = validate(next, true, true, true);
  if (st != TREEWY_OK) return st;
  st = validate(prev, false, false, true);
  if (st != TREEWY_OK) return st;
  if (prev->R != next->R || prev->H != next->H || prev->dk != next->dk || prev->dv != next->dv)
    return fail(TREEWY_ERR_INVALID_ARG, "prev and next must have the same R, H, dk and dv");
  if (prev->state != next->state || prev->state_slot != next->state_slot ||
      prev->num_slots != next->num_slots)
    return fail(TREEWY_ERR_INVALID_ARG, "prev and next must share the state pool and state_slot");
  if ((prev->flags ^ next->flags) & TREEWY_FLAG_STATE_BF16)
    return fail(TREEWY_ERR_INVALID_ARG, "prev and next must agree on TREEWY_FLAG_STATE_BF16");
  if (next->R == 0) return TREEWY_OK;
  if (!prev->U && prev->T > 0) return fail(TREEWY_ERR_INVALID_ARG, "prev->U is NULL");
  if (!aligned16(prev->U)) return fail(TREEWY_ERR_INVALID_ARG, "prev->U must be 16-byte aligned");
  if (!prev_accepted) return fail(TREEWY_ERR_INVALID_ARG, "prev_accepted is NULL");
  cudaError_t err;
  // Kernel for the next round: the small-tree kernel up to 8 nodes, the
  // warp-MMA kernel up to 16 (up to 32 for a bf16 pool, whose fused or
  // two-call form there beats the tcgen05 kernel's), the tcgen05 kernel
  // above.  The warp-MMA kernels apply an accepted path 8 or 16 entries per
  // pass over the state tile; a bf16 pool is rounded at the end of each pass,
  // so it takes their fused form only while every path fits one pass (S_a
  // rounded once, as the separate commit does), and otherwise the commit and
  // the verification run as two calls.
  const bool bf16_pool = (next->flags & TREEWY_FLAG_STATE_BF16) != 0;
  const bool small = next->max_nodes <= treewy::kFusedWarpNodes ||
                     (bf16_pool && next->max_nodes <= treewy::kWarpTreeNodes);
  const int seg = next->max_nodes <= treewy::kSmallTreeNodes ? treewy::kSmallTreeNodes
                                                              : treewy::kWarpSegEntries;
  const bool small_fused_ok = !bf16_pool || prev->max_nodes <= seg;
  if (use_tensor_cores(next) && next->T > 0 && prev->qkv_dtype == TREEWY_DTYPE_BF16 &&
      (!small || small_fused_ok)) {
    treewy::PrevRound pr;
    pr.node_offset = prev->node_offset;
    pr.parent = prev->parent;
    pr.alpha = prev->alpha;
    pr.k = prev->k;
    pr.U = prev->U;
    pr.accepted = prev_accepted;
    pr.T = prev->T;
    pr.max_nodes = prev->max_nodes;
    pr.active = 1;
    if (small) {
      CUtensorMap map;
      st = make_state_map(next, &map);
      if (st != TREEWY_OK) return st;
      err = next->max_nodes <= treewy::kSmallTreeNodes
                ? treewy::launch_verify_small(*next, map, &pr, stream)
                : treewy::launch_verify_warp(*next, map, &pr, stream);
    } else {
      treewy::VerifyMaps maps;
      st = make_maps(next, &maps);
      if (st != TREEWY_OK) return st;
      err = treewy::launch_commit_verify_tc(*next, pr, maps, next->max_nodes, stream);
    }
    return err == cudaSuccess ? TREEWY_OK : cuda_fail(err, "treewy_commit_verify launch");
  }
  // other shapes: the two kernels back to back on the same stream, the
  // commit's status bits going to next->status as on the fused path
  treewy_batch pc = *prev;
  pc.status = next->status;
  st = launch_commit_any(&pc, prev_accepted, TREEWY_STATUS_COMMIT_REFUSED, stream,
                         "treewy_commit_verify (commit) launch");
  if (st != TREEWY_OK) return st;
  return treewy_verify(next, stream);
}

treewy_status treewy_storeall_verify(const treewy_batch* batch, float* snapshots, cudaStream_t stream) {
  g_last_error.clear();
  treewy_status st = validate(batch, true, false, true);
  if (st != TREEWY_OK) return st;
  if (batch->flags & TREEWY_FLAG_STATE_BF16)
    return fail(TREEWY_ERR_UNSUPPORTED, "the storeall comparator keeps f32 states only");
  if (batch->R == 0) return st;
  if (batch->T > 0 && !batch->o) return fail(TREEWY_ERR_INVALID_ARG, "o is NULL");
  if ((batch->T > 0 && !snapshots) || !aligned16(snapshots))
    return fail(TREEWY_ERR_INVALID_ARG, "snapshots must be non-NULL and 16-byte aligned");
  cudaError_t err = treewy::launch_storeall_verify(*batch, snapshots, stream);
  return err == cudaSuccess ? TREEWY_OK : cuda_fail(err, "treewy_storeall_verify launch");
}

treewy_status treewy_storeall_commit(const treewy_batch* batch, const float* snapshots,
                                     const int32_t* accepted, cudaStream_t stream) {
  g_last_error.clear();
  treewy_status st = validate(batch, false, false, false, false);
  if (st == TREEWY_OK && (batch->flags & TREEWY_FLAG_STATE_BF16))
    return fail(TREEWY_ERR_UNSUPPORTED, "the storeall comparator keeps f32 states only");
  if (st == TREEWY_OK && batch->R > 0 && batch->T > 0 && !batch->parent)
    return fail(TREEWY_ERR_INVALID_ARG, "parent is NULL");
  if (st != TREEWY_OK || batch->R == 0) return st;
  if ((batch->T > 0 && !snapshots) || !aligned16(snapshots))
    return fail(TREEWY_ERR_INVALID_ARG, "snapshots must be non-NULL and 16-byte aligned");
  if (!accepted) return fail(TREEWY_ERR_INVALID_ARG, "accepted is NULL");
  cudaError_t err = treewy::launch_storeall_commit(*batch, snapshots, accepted, stream);
  return err == cudaSuccess ? TREEWY_OK : cuda_fail(err, "treewy_storeall_commit launch");
}

}  // extern "C"
