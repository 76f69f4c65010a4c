// commit.cu -- reconstruct-on-commit (TreeWY paper §3 "Reconstruct on commit",
// Eq. (3); technical review §3.3, Eq. (6)):
//
//   S_a = gamma_a S0 + sum_{i on the root-to-a path} (gamma_a / gamma_i) u_i k_i^T,
//
// written in place over S0 in the state pool.  The update has rank
// |path(a)| <= depth, so the kernel is a streaming pass over the 64 KB state
// (read once, written once) with the path's u and k rows staged in shared
// memory; ratios gamma_a / gamma_i are products of alpha over the path segment.
//
// One CTA of 256 threads per (request, head).  The state loads are issued
// before the path walk so their latency overlaps it.
#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

constexpr int kThreads = 256;
constexpr int kSeg = 16;             // path nodes staged per pass
constexpr int kMaxVec = 16;          // float4 per thread for a 128 x 128 state

// Streaming (evict-first) access: every state byte is touched exactly once.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

// Two resident blocks per SM: the 16 float4 state registers per thread stay
// in registers (a three-block cap spills them and was measured slower).
__global__ void __launch_bounds__(kThreads, 2)
    commit_kernel(const treewy_batch b, const int32_t* __restrict__ accepted) {
  __shared__ int s_parent[kMaxNodes];
  __shared__ float s_alpha[kMaxNodes];
  __shared__ int s_path[kMaxNodes];
  __shared__ float s_c[kMaxNodes];
  __shared__ int s_info[6];  // tok0, N, slot, a, flags, path length
  __shared__ float s_gamma_a;
  __shared__ __align__(16) float cu[kSeg][128];  // c_j * u_{path j}[d]
  __shared__ __align__(16) float kf[kSeg][128];  // k_{path j}[e]

  const int H = b.H, dk = b.dk, dv = b.dv;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const bool bf16 = b.qkv_dtype == TREEWY_DTYPE_BF16;

  if (t == 0) {
    const int a = accepted[r];
    const int lo = b.node_offset[r], hi = b.node_offset[r + 1];
    const int slot = b.state_slot[r];
    const int N = hi - lo;
    int flags = 0;
    if (a != -1) {
      if (N < 0 || N > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
      else if (lo < 0 || static_cast<int64_t>(hi) > b.T) flags |= TREEWY_STATUS_BAD_TREE;
      if (a < -1 || a >= N) flags |= TREEWY_STATUS_BAD_ACCEPTED;
      if (slot < 0 || static_cast<int64_t>(slot) >= b.num_slots) flags |= TREEWY_STATUS_BAD_SLOT;
    }
    s_info[0] = lo;
    s_info[1] = N;
    s_info[2] = slot;
    s_info[3] = a;
    s_info[4] = flags;
  }
  __syncthreads();
  const int a = s_info[3];
  if (a == -1) return;  // nothing accepted: the state is neither read nor written
  if (s_info[4]) {
    if (t == 0 && h == 0) atomicOr(b.status + r, s_info[4]);
    return;
  }
  const int64_t tok0 = s_info[0];
  const int N = s_info[1];
  float* S = b.state + (static_cast<int64_t>(s_info[2]) * H + h) * dv * dk;
  const int nelem = dv * dk;
  const bool vec = (dk & 3) == 0;
  const int nvec = nelem >> 2;

  // 1. state loads in flight
  float4 acc[kMaxVec];
  if (vec) {
#pragma unroll
    for (int m = 0; m < kMaxVec; ++m) {
      const int f = t + m * kThreads;
      acc[m] = (f < nvec) ? ld_stream(reinterpret_cast<const float4*>(S) + f)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  // 2. the path root..a, with c = gamma_a / gamma_i as alpha products; the
  //    whole tree is validated (U of an invalid tree was never written)
  bool bad_parent = false;
  if (t < N) {
    const int p = __ldg(b.parent + tok0 + t);
    bad_parent = !(p >= -1 && p < t);
    s_parent[t] = p;
    s_alpha[t] = __ldg(b.alpha + (tok0 + t) * H + h);
  }
  if (__syncthreads_or(bad_parent)) {
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE);
    return;
  }
  if (t == 0) {
    int cur = a, len = 0, bad = 0;
    float c = 1.0f;
    while (true) {
      s_path[len] = cur;
      s_c[len] = c;
      ++len;
      c *= s_alpha[cur];
      const int p = s_parent[cur];
      if (p < -1 || p >= cur) {
        bad = 1;
        break;
      }
      if (p == -1) break;
      cur = p;
    }
    s_info[5] = bad ? -1 : len;
    s_gamma_a = c;
  }
  __syncthreads();
  const int len = s_info[5];
  if (len < 0) {
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE);
    return;
  }
  const float ga = s_gamma_a;

  if (vec) {
    // 3. rank-|path| update, kSeg path nodes per pass.  The path rows are
    //    requested before the state registers are touched, so their round
    //    trip overlaps the state loads still in flight.
    for (int seg = 0; seg < len; seg += kSeg) {
      const int ns = min(kSeg, len - seg);
      for (int e = t; e < ns * 128; e += kThreads) {
        const int j = e >> 7, x = e & 127;
        const int64_t row = (tok0 + s_path[seg + j]) * H + h;
        cu[j][x] = (x < dv) ? s_c[seg + j] * __ldg(b.U + row * dv + x) : 0.f;
        kf[j][x] = (x < dk) ? load_qkv(b.k, row * dk + x, bf16) : 0.f;
      }
      __syncthreads();
      if (seg == 0) {
#pragma unroll
        for (int m = 0; m < kMaxVec; ++m) {
          acc[m].x *= ga;
          acc[m].y *= ga;
          acc[m].z *= ga;
          acc[m].w *= ga;
        }
      }
      if (dk == 128) {
        // float4 f = t + 256 m covers row d = t/32 + 8m, columns x..x+3 with
        // x = 4 (t % 32): the k chunk of a path node is loaded once per node
        const int x = (t & 31) << 2;
        const int d0 = t >> 5;
        for (int j = 0; j < ns; ++j) {
          const float4 kk = *reinterpret_cast<const float4*>(&kf[j][x]);
#pragma unroll
          for (int m = 0; m < kMaxVec; ++m) {
            const int d = d0 + 8 * m;
            if (d < dv) {
              const float u = cu[j][d];
              acc[m].x = fmaf(u, kk.x, acc[m].x);
              acc[m].y = fmaf(u, kk.y, acc[m].y);
              acc[m].z = fmaf(u, kk.z, acc[m].z);
              acc[m].w = fmaf(u, kk.w, acc[m].w);
            }
          }
        }
      } else {
#pragma unroll
        for (int m = 0; m < kMaxVec; ++m) {
          const int f = t + m * kThreads;
          if (f < nvec) {
            const int e = f << 2;
            const int d = e / dk, x = e - d * dk;
            for (int j = 0; j < ns; ++j) {
              const float u = cu[j][d];
              const float4 kk = *reinterpret_cast<const float4*>(&kf[j][x]);
              acc[m].x = fmaf(u, kk.x, acc[m].x);
              acc[m].y = fmaf(u, kk.y, acc[m].y);
              acc[m].z = fmaf(u, kk.z, acc[m].z);
              acc[m].w = fmaf(u, kk.w, acc[m].w);
            }
          }
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int m = 0; m < kMaxVec; ++m) {
      const int f = t + m * kThreads;
      if (f < nvec) st_stream(reinterpret_cast<float4*>(S) + f, acc[m]);
    }
  } else {
    // scalar path for head sizes that are not a multiple of 4
    for (int seg = 0; seg < len; seg += kSeg) {
      const int ns = min(kSeg, len - seg);
      for (int e = t; e < ns * 128; e += kThreads) {
        const int j = e >> 7, x = e & 127;
        const int64_t row = (tok0 + s_path[seg + j]) * H + h;
        cu[j][x] = (x < dv) ? s_c[seg + j] * __ldg(b.U + row * dv + x) : 0.f;
        kf[j][x] = (x < dk) ? load_qkv(b.k, row * dk + x, bf16) : 0.f;
      }
      __syncthreads();
      for (int e = t; e < nelem; e += kThreads) {
        const int d = e / dk, x = e - d * dk;
        float s = (seg == 0) ? ga * S[e] : S[e];
        for (int j = 0; j < ns; ++j) s = fmaf(cu[j][d], kf[j][x], s);
        S[e] = s;
      }
      __syncthreads();
    }
  }
}

}  // namespace

cudaError_t launch_commit(const treewy_batch& b, const int32_t* accepted, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  commit_kernel<<<grid, kThreads, 0, stream>>>(b, accepted);
  return cudaGetLastError();
}

}  // namespace treewy
