// commit.cu -- reconstruct-on-commit (TreeWY paper §3 "Reconstruct on commit",
// Eq. (3); technical review §3.3, Eq. (6)):
//
//   S_a = gamma_a S0 + sum_{i on the root-to-a path} (gamma_a / gamma_i) u_i k_i^T,
//
// written in place over S0 in the state pool (f32, or bf16 rounded to nearest
// even from the f32 result).  The update has rank |path(a)| <= depth, so the
// kernel is a streaming pass over the state (64 KB f32 / 32 KB bf16, read once,
// written once) with the path's u and k rows staged in shared
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

// State elements per 16-byte vector and the f32 <-> storage conversions: f32
// state (4 per vector) or bf16 state (8 per vector, rounded to nearest even).
template <bool SB>
struct StateVec {
  static constexpr int E = SB ? 8 : 4;
  // Streaming (evict-first) access: every state byte is touched exactly once.
  __device__ static __forceinline__ void load(const void* base, int f, float (&x)[E]) {
    const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(base) + f);
    if constexpr (SB) {
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
      x[0] = __uint_as_float(raw.x);
      x[1] = __uint_as_float(raw.y);
      x[2] = __uint_as_float(raw.z);
      x[3] = __uint_as_float(raw.w);
    }
  }
  __device__ static __forceinline__ void store(void* base, int f, const float (&x)[E]) {
    uint4 raw;
    if constexpr (SB) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&p);
      }
      raw = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      raw = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                       __float_as_uint(x[3]));
    }
    __stcs(reinterpret_cast<uint4*>(base) + f, raw);
  }
};

// Two resident blocks per SM: the 64 state values per thread stay in
// registers (a three-block cap spills them and was measured slower).
template <bool SB>
__global__ void __launch_bounds__(kThreads, 2)
    commit_kernel(const treewy_batch b, const int32_t* __restrict__ accepted, int refused_bit) {
  using SV = StateVec<SB>;
  constexpr int E = SV::E;
  constexpr int kNV = 128 * 128 / (E * kThreads);  // vectors per thread for a 128 x 128 state
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
    if (t == 0 && h == 0) atomicOr(b.status + r, s_info[4] | refused_bit);
    return;
  }
  const int64_t tok0 = s_info[0];
  const int N = s_info[1];
  const int64_t head0 = (static_cast<int64_t>(s_info[2]) * H + h) * dv * dk;
  void* S = SB ? static_cast<void*>(static_cast<__nv_bfloat16*>(b.state) + head0)
               : static_cast<void*>(static_cast<float*>(b.state) + head0);
  const int nelem = dv * dk;
  const bool vec = (dk % E) == 0;
  const int nvec = nelem / E;

  // 1. state loads in flight
  float acc[kNV][E];
  if (vec) {
#pragma unroll
    for (int m = 0; m < kNV; ++m) {
      const int f = t + m * kThreads;
      if (f < nvec) {
        SV::load(S, f, acc[m]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) acc[m][e] = 0.f;
      }
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
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE | refused_bit);
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
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE | refused_bit);
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
        for (int m = 0; m < kNV; ++m)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[m][e] *= ga;
      }
      if (dk == 128) {
        // vector f = t + 256 m covers row d = t / V + (256 / V) m, columns
        // x..x+E-1 with x = E (t % V), V = 128 / E vectors per row: the k
        // chunk of a path node is loaded once per node
        constexpr int V = 128 / E;
        const int x = (t % V) * E;
        const int d0 = t / V;
        for (int j = 0; j < ns; ++j) {
          float kk[E];
#pragma unroll
          for (int e = 0; e < E; e += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(&kf[j][x + e]);
            kk[e] = k4.x;
            kk[e + 1] = k4.y;
            kk[e + 2] = k4.z;
            kk[e + 3] = k4.w;
          }
#pragma unroll
          for (int m = 0; m < kNV; ++m) {
            const int d = d0 + (kThreads / V) * m;
            if (d < dv) {
              const float u = cu[j][d];
#pragma unroll
              for (int e = 0; e < E; ++e) acc[m][e] = fmaf(u, kk[e], acc[m][e]);
            }
          }
        }
      } else {
#pragma unroll
        for (int m = 0; m < kNV; ++m) {
          const int f = t + m * kThreads;
          if (f < nvec) {
            const int e0 = f * E;
            const int d = e0 / dk, x = e0 - d * dk;
            for (int j = 0; j < ns; ++j) {
              const float u = cu[j][d];
#pragma unroll
              for (int e = 0; e < E; ++e) acc[m][e] = fmaf(u, kf[j][x + e], acc[m][e]);
            }
          }
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int m = 0; m < kNV; ++m) {
      const int f = t + m * kThreads;
      if (f < nvec) SV::store(S, f, acc[m]);
    }
  } else {
    // scalar path for head sizes that are not a multiple of the vector
    // width: blocks of kThreads x kSc elements stay in f32 registers across
    // every pass and are stored (rounded once, for a bf16 state) at the end
    constexpr int kSc = 16;
    for (int e0 = 0; e0 < nelem; e0 += kThreads * kSc) {
      float sreg[kSc];
#pragma unroll
      for (int i = 0; i < kSc; ++i) {
        const int e = e0 + t + i * kThreads;
        sreg[i] = (e < nelem) ? ga * load_qkv(S, e, SB) : 0.f;
      }
      for (int seg = 0; seg < len; seg += kSeg) {
        const int ns = min(kSeg, len - seg);
        __syncthreads();  // the previous pass is done with cu / kf
        for (int e = t; e < ns * 128; e += kThreads) {
          const int j = e >> 7, x = e & 127;
          const int64_t row = (tok0 + s_path[seg + j]) * H + h;
          cu[j][x] = (x < dv) ? s_c[seg + j] * __ldg(b.U + row * dv + x) : 0.f;
          kf[j][x] = (x < dk) ? load_qkv(b.k, row * dk + x, bf16) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kSc; ++i) {
          const int e = e0 + t + i * kThreads;
          if (e < nelem) {
            const int d = e / dk, x = e - d * dk;
            for (int j = 0; j < ns; ++j) sreg[i] = fmaf(cu[j][d], kf[j][x], sreg[i]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kSc; ++i) {
        const int e = e0 + t + i * kThreads;
        if (e < nelem) {
          if constexpr (SB) static_cast<__nv_bfloat16*>(S)[e] = __float2bfloat16_rn(sreg[i]);
          else static_cast<float*>(S)[e] = sreg[i];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_commit(const treewy_batch& b, const int32_t* accepted, int refused_bit,
                          cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  if (b.flags & TREEWY_FLAG_STATE_BF16)
    commit_kernel<true><<<grid, kThreads, 0, stream>>>(b, accepted, refused_bit);
  else
    commit_kernel<false><<<grid, kThreads, 0, stream>>>(b, accepted, refused_bit);
  return cudaGetLastError();
}

}  // namespace treewy
