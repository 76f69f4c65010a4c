// treewy_internal.h -- host-side declarations shared by the library's
// translation units (launchers); not part of the public C ABI.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "treewy.h"

namespace treewy {

// Runs `set` (a cudaFuncSetAttribute call) once per device: the attributes
// are per device and function, so a process driving several GPUs needs them
// on each.  `done` is a per-call-site bit mask of the devices already set
// (ordinals >= 64 are set on every call).
template <typename F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = set();
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Tensor maps the tensor-core verify kernel reads through (built on the host
// per call; passed by value as kernel parameters).
struct VerifyMaps {
  CUtensorMap s0;  // state pool [rows = slots*H*128][128], box 128 rows x 128 bytes
                   // (32 fp32 or 64 bf16 columns), 128B swizzle
  CUtensorMap k;    // keys, bf16 [T][H][128], box 64 x 1 x 16, 128B swizzle
  CUtensorMap q;    // queries, same layout as keys
  CUtensorMap k32;  // keys, box 64 x 1 x 32
  CUtensorMap q32;  // queries, box 64 x 1 x 32
};

size_t verify_generic_smem(int dk, int dv, int npm);
cudaError_t launch_verify_generic(const treewy_batch& b, cudaStream_t stream);

// The previous round whose commit is applied inside the next verification:
// its trees, gates, keys and pseudo-values U, and the accepted nodes.
struct PrevRound {
  const int32_t* node_offset;
  const int32_t* parent;
  const float* alpha;
  const void* k;  // bf16 [T][H][128]
  const float* U;
  const int32_t* accepted;
  int64_t T;
  int32_t max_nodes;
  int32_t active;  // 0: plain verification
};

// Batches whose trees have at most this many nodes (max_nodes) are verified
// by the small-tree kernel (verify_small.cu: warp-level MMAs straight from
// the state tile) when dk = dv = 128 and q/k/v are bf16; larger ones by the
// tcgen05 kernel.
constexpr int kSmallTreeNodes = 8;
// state_map: the state pool as VerifyMaps::s0; prev != nullptr fuses the
// previous round's commit in front (PrevRound below).
struct PrevRound;
cudaError_t launch_verify_small(const treewy_batch& b, const CUtensorMap& state_map,
                                const PrevRound* prev, cudaStream_t stream);

// Batches of at most kWarpTreeNodes nodes per tree (and more than
// kSmallTreeNodes) are verified by warp-level MMAs over the whole method
// (verify_warp.cu), with the previous round's commit fused in front up to
// kFusedWarpNodes (fp32 pool) or kWarpTreeNodes (bf16 pool); larger trees by
// the tcgen05 kernel, whose state products run at several times the rate of
// warp-level MMAs.
constexpr int kWarpTreeNodes = 32;
constexpr int kFusedWarpNodes = 16;
// Path entries the warp-MMA kernel applies per update pass of its fused
// commit (a bf16 pool takes the fused form when every path fits one pass).
constexpr int kWarpSegEntries = 16;
cudaError_t launch_verify_warp(const treewy_batch& b, const CUtensorMap& state_map,
                               const PrevRound* prev, cudaStream_t stream);

// npm: tree capacity bucket (32 or 64 nodes; launched for max_nodes > 16).
cudaError_t launch_verify_tc(const treewy_batch& b, const VerifyMaps& maps, int npm,
                             cudaStream_t stream);
cudaError_t launch_commit_verify_tc(const treewy_batch& next, const PrevRound& prev,
                                    const VerifyMaps& maps, int npm, cudaStream_t stream);
// The same kernel for a bf16 state pool; prev == nullptr for plain verification.
cudaError_t launch_verify_tc_bf16state(const treewy_batch& b, const VerifyMaps& maps,
                                       const PrevRound* prev, int npm, cudaStream_t stream);

// refused_bit: extra status bit OR-ed in, beside the reason, when a request's
// commit is refused (TREEWY_STATUS_COMMIT_REFUSED inside treewy_commit_verify,
// 0 for treewy_commit).
cudaError_t launch_commit(const treewy_batch& b, const int32_t* accepted, int refused_bit,
                          cudaStream_t stream);
// dk = dv = 128: the state tile moved by bulk tensor copies (state_map as VerifyMaps::s0).
cudaError_t launch_commit_tma(const treewy_batch& b, const CUtensorMap& state_map,
                              const int32_t* accepted, int refused_bit, cudaStream_t stream);

cudaError_t launch_storeall_verify(const treewy_batch& b, float* snapshots, cudaStream_t stream);
cudaError_t launch_storeall_commit(const treewy_batch& b, const float* snapshots,
                                   const int32_t* accepted, cudaStream_t stream);

// One thread waiting for a barrier phase nothing completes (bounded).
cudaError_t launch_wait_selftest(int32_t* status, uint32_t limit_us, cudaStream_t stream);

}  // namespace treewy
