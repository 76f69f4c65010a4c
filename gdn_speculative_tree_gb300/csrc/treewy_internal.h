// treewy_internal.h -- host-side declarations shared by the library's
// translation units (launchers); not part of the public C ABI.
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

#include "treewy.h"

namespace treewy {

// Tensor maps the tensor-core verify kernel reads through (built on the host
// per call; passed by value as kernel parameters).
struct VerifyMaps {
  CUtensorMap s0;  // state pool, fp32 [rows = slots*H*128][128], box 32 x 128, 128B swizzle
  CUtensorMap k;   // keys, bf16 [T][H][128], box 64 x 1 x 8, 128B swizzle
  CUtensorMap q;   // queries, same layout as keys
};

size_t verify_generic_smem(int dk, int dv, int npm);
cudaError_t launch_verify_generic(const treewy_batch& b, cudaStream_t stream);

// npm: padded tree capacity (16, 32 or 64).
size_t verify_tc_smem(int npm);
cudaError_t launch_verify_tc(const treewy_batch& b, const VerifyMaps& maps, int npm,
                             cudaStream_t stream);

cudaError_t launch_commit(const treewy_batch& b, const int32_t* accepted, cudaStream_t stream);

cudaError_t launch_storeall_verify(const treewy_batch& b, float* snapshots, cudaStream_t stream);
cudaError_t launch_storeall_commit(const treewy_batch& b, const float* snapshots,
                                   const int32_t* accepted, cudaStream_t stream);

}  // namespace treewy
