// storeall.cu -- the snapshot-per-node comparator: full-state snapshotting
// ("storeall", TreeWY paper §2 "The memory problem", approach (i)).
//
// Verify applies the gated delta rule (paper §1 Eq. (1)) node by node,
//   S_n = alpha_n (S_par - beta_n (S_par k_n) k_n^T) + beta_n v_n k_n^T,  o_n = S_n q_n,
// writing every S_n to a caller-owned snapshot buffer; rollback copies the
// accepted node's snapshot over the committed state.  This is the memory
// behaviour TreeWY removes; it is kept as an in-library baseline.
//
// One CTA of 256 threads per (request, head), the state held in registers.  For
// dk = dv = 128 each warp owns whole 512-byte rows (coalesced snapshot stores);
// other head sizes use a half-row-per-thread layout.  A node whose parent is
// not the previous node reloads the parent's snapshot (which the same thread
// wrote) from global memory.
#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

constexpr int kThreads = 256;
constexpr int kCols = 64;

struct StoreallSmemLayout {
  size_t ks, qs, vs, total;
};

__host__ __device__ inline StoreallSmemLayout storeall_layout(int dk, int dv, int npm) {
  StoreallSmemLayout L;
  size_t off = 0;
  L.ks = off; off += sizeof(float) * npm * dk;
  L.qs = off; off += sizeof(float) * npm * dk;
  L.vs = off; off += sizeof(float) * npm * dv;
  L.total = (off + 15) & ~size_t(15);
  return L;
}

__global__ void __launch_bounds__(kThreads)
    storeall_verify_kernel(const treewy_batch b, float* __restrict__ snapshots, int npm) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_parent[kMaxNodes];
  __shared__ float s_alpha[kMaxNodes], s_beta[kMaxNodes];
  __shared__ int s_info[5];  // tok0, N, slot, flags, base row

  const int H = b.H, dk = b.dk, dv = b.dv;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const bool bf16 = b.qkv_dtype == TREEWY_DTYPE_BF16;
  const StoreallSmemLayout L = storeall_layout(dk, dv, npm);
  float* Ks = reinterpret_cast<float*>(smem + L.ks);
  float* Qs = reinterpret_cast<float*>(smem + L.qs);
  float* Vs = reinterpret_cast<float*>(smem + L.vs);

  if (t == 0) {
    const int lo = b.node_offset[r], hi = b.node_offset[r + 1];
    const int slot = b.state_slot[r];
    const int N = hi - lo;
    int flags = 0;
    if (N < 0 || N > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
    else if (lo < b.node_offset[0] || static_cast<int64_t>(hi) > b.T || hi > b.node_offset[b.R])
      flags |= TREEWY_STATUS_BAD_TREE;  // snapshot rows must lie in [node_offset[0], node_offset[R])
    if (slot < 0 || static_cast<int64_t>(slot) >= b.num_slots) flags |= TREEWY_STATUS_BAD_SLOT;
    s_info[0] = lo;
    s_info[1] = flags ? 0 : N;
    s_info[2] = slot;
    s_info[3] = flags;
    s_info[4] = b.node_offset[0];
  }
  __syncthreads();
  if (s_info[3]) {
    if (t == 0 && h == 0) atomicOr(b.status + r, s_info[3]);
    return;
  }
  const int N = s_info[1];
  if (N == 0) return;
  const int64_t tok0 = s_info[0];
  const int64_t rel0 = tok0 - s_info[4];

  bool bad = false;
  if (t < N) {
    const int p = __ldg(b.parent + tok0 + t);
    bad = !(p >= -1 && p < t);
    s_parent[t] = p;
    s_alpha[t] = __ldg(b.alpha + (tok0 + t) * H + h);
    s_beta[t] = __ldg(b.beta + (tok0 + t) * H + h);
  }
  for (int e = t; e < N * dk; e += kThreads) {
    const int n = e / dk, j = e - n * dk;
    const int64_t g = ((tok0 + n) * H + h) * dk + j;
    Ks[e] = load_qkv(b.k, g, bf16);
    Qs[e] = load_qkv(b.q, g, bf16);
  }
  for (int e = t; e < N * dv; e += kThreads) {
    const int n = e / dv, j = e - n * dv;
    Vs[e] = load_qkv(b.v, ((tok0 + n) * H + h) * dv + j, bf16);
  }
  if (__syncthreads_or(bad)) {
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE);
    return;
  }

  const int d = t >> 1;
  const int c0 = (t & 1) * kCols;
  const bool row_ok = d < dv;
  const int64_t head_elems = static_cast<int64_t>(dv) * dk;
  const float* S0 = static_cast<const float*>(b.state) + (static_cast<int64_t>(s_info[2]) * H + h) * head_elems;
  auto snap = [&](int n) { return snapshots + ((rel0 + n) * H + h) * head_elems; };

  float s[kCols];
  auto load_state = [&](const float* src) {
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      const int x = c0 + j;
      s[j] = (row_ok && x < dk) ? src[d * dk + x] : 0.f;
    }
  };
  load_state(S0);
  int cur = -1;  // node whose state the registers hold (-1: S0)
  for (int n = 0; n < N; ++n) {
    const int p = s_parent[n];
    if (p != cur) load_state(p < 0 ? S0 : snap(p));
    const float* kn = Ks + n * dk;
    const float* qn = Qs + n * dk;
    float sk = 0.f;
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      const int x = c0 + j;
      if (x < dk) sk = fmaf(s[j], kn[x], sk);
    }
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    const float a = s_alpha[n], be = s_beta[n];
    const float vd = row_ok ? Vs[n * dv + d] : 0.f;
    const float bsk = be * sk, bv = be * vd;
    float so = 0.f;
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      const int x = c0 + j;
      if (x < dk) {
        s[j] = fmaf(a, fmaf(-bsk, kn[x], s[j]), bv * kn[x]);
        so = fmaf(s[j], qn[x], so);
      }
    }
    so += __shfl_xor_sync(0xffffffffu, so, 1);
    if (row_ok) {
      float* dst = snap(n) + d * dk;
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        const int x = c0 + j;
        if (x < dk) dst[x] = s[j];
      }
      if ((t & 1) == 0) b.o[((tok0 + n) * H + h) * dv + d] = so;
    }
    cur = n;
  }
}

// Fast layout for dk = dv = 128: thread t owns rows d = t/32 + 8m (m < 16)
// at columns 4(t%32)..4(t%32)+3, so every warp-wide snapshot store writes one
// full 512-byte row; S k and S q are warp all-reductions per row.
constexpr int kRowsPerThread = 16;

__global__ void __launch_bounds__(kThreads)
    storeall_verify_rows_kernel(const treewy_batch b, float* __restrict__ snapshots) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_parent[kMaxNodes];
  __shared__ float s_alpha[kMaxNodes], s_beta[kMaxNodes];
  __shared__ int s_info[5];  // tok0, N, slot, flags, base row
  constexpr int kD = 128;
  float* Ks = reinterpret_cast<float*>(smem);              // [N][128]
  float* Qs = Ks + kMaxNodes * kD;
  float* Vs = Qs + kMaxNodes * kD;

  const int H = b.H;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const bool bf16 = b.qkv_dtype == TREEWY_DTYPE_BF16;

  if (t == 0) {
    const int lo = b.node_offset[r], hi = b.node_offset[r + 1];
    const int slot = b.state_slot[r];
    const int N = hi - lo;
    int flags = 0;
    if (N < 0 || N > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
    else if (lo < b.node_offset[0] || static_cast<int64_t>(hi) > b.T || hi > b.node_offset[b.R])
      flags |= TREEWY_STATUS_BAD_TREE;  // snapshot rows must lie in [node_offset[0], node_offset[R])
    if (slot < 0 || static_cast<int64_t>(slot) >= b.num_slots) flags |= TREEWY_STATUS_BAD_SLOT;
    s_info[0] = lo;
    s_info[1] = flags ? 0 : N;
    s_info[2] = slot;
    s_info[3] = flags;
    s_info[4] = b.node_offset[0];
  }
  __syncthreads();
  if (s_info[3]) {
    if (t == 0 && h == 0) atomicOr(b.status + r, s_info[3]);
    return;
  }
  const int N = s_info[1];
  if (N == 0) return;
  const int64_t tok0 = s_info[0];
  const int64_t rel0 = tok0 - s_info[4];

  bool bad = false;
  if (t < N) {
    const int p = __ldg(b.parent + tok0 + t);
    bad = !(p >= -1 && p < t);
    s_parent[t] = p;
    s_alpha[t] = __ldg(b.alpha + (tok0 + t) * H + h);
    s_beta[t] = __ldg(b.beta + (tok0 + t) * H + h);
  }
  for (int e = t; e < N * kD; e += kThreads) {
    const int n = e >> 7, j = e & 127;
    const int64_t g = ((tok0 + n) * H + h) * kD + j;
    Ks[e] = load_qkv(b.k, g, bf16);
    Qs[e] = load_qkv(b.q, g, bf16);
    Vs[e] = load_qkv(b.v, g, bf16);
  }
  if (__syncthreads_or(bad)) {
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE);
    return;
  }

  const int x = (t & 31) << 2;
  const int d0 = t >> 5;
  constexpr int64_t kHead = kD * kD;
  const float* S0 = static_cast<const float*>(b.state) + (static_cast<int64_t>(s_info[2]) * H + h) * kHead;
  auto snap = [&](int n) { return snapshots + ((rel0 + n) * H + h) * kHead; };
  float4 S[kRowsPerThread];
  auto load_state = [&](const float* src) {
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m)
      S[m] = *reinterpret_cast<const float4*>(src + (d0 + 8 * m) * kD + x);
  };
  load_state(S0);
  int cur = -1;  // node whose state the registers hold (-1: S0)
  for (int n = 0; n < N; ++n) {
    const int p = s_parent[n];
    if (p != cur) load_state(p < 0 ? S0 : snap(p));
    const float4 kk = *reinterpret_cast<const float4*>(Ks + n * kD + x);
    const float4 qq = *reinterpret_cast<const float4*>(Qs + n * kD + x);
    const float a = s_alpha[n], be = s_beta[n];
    float sk[kRowsPerThread];
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m)
      sk[m] = S[m].x * kk.x + S[m].y * kk.y + S[m].z * kk.z + S[m].w * kk.w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int m = 0; m < kRowsPerThread; ++m) sk[m] += __shfl_xor_sync(0xffffffffu, sk[m], o);
    }
    float* dst = snap(n);
    float so[kRowsPerThread];
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m) {
      const int d = d0 + 8 * m;
      const float bsk = be * sk[m], bv = be * Vs[n * kD + d];
      S[m].x = fmaf(a, fmaf(-bsk, kk.x, S[m].x), bv * kk.x);
      S[m].y = fmaf(a, fmaf(-bsk, kk.y, S[m].y), bv * kk.y);
      S[m].z = fmaf(a, fmaf(-bsk, kk.z, S[m].z), bv * kk.z);
      S[m].w = fmaf(a, fmaf(-bsk, kk.w, S[m].w), bv * kk.w);
      so[m] = S[m].x * qq.x + S[m].y * qq.y + S[m].z * qq.z + S[m].w * qq.w;
      *reinterpret_cast<float4*>(dst + d * kD + x) = S[m];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int m = 0; m < kRowsPerThread; ++m) so[m] += __shfl_xor_sync(0xffffffffu, so[m], o);
    }
    if ((t & 31) < kRowsPerThread) {
      // lane m of each warp writes row d0 + 8m (static register index by unrolled select)
      float v = 0.f;
#pragma unroll
      for (int m = 0; m < kRowsPerThread; ++m)
        if ((t & 31) == m) v = so[m];
      b.o[((tok0 + n) * H + h) * kD + d0 + 8 * (t & 31)] = v;
    }
    cur = n;
  }
}

__global__ void __launch_bounds__(kThreads)
    storeall_commit_kernel(const treewy_batch b, const float* __restrict__ snapshots,
                           const int32_t* __restrict__ accepted) {
  const int H = b.H;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const int a = accepted[r];
  if (a == -1) return;
  const int lo = b.node_offset[r], hi = b.node_offset[r + 1];
  const int slot = b.state_slot[r];
  const int N = hi - lo;
  int flags = 0;
  if (N < 0 || N > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
  else if (lo < b.node_offset[0] || static_cast<int64_t>(hi) > b.T || hi > b.node_offset[b.R])
    flags |= TREEWY_STATUS_BAD_TREE;
  if (a < -1 || a >= N) flags |= TREEWY_STATUS_BAD_ACCEPTED;
  if (slot < 0 || static_cast<int64_t>(slot) >= b.num_slots) flags |= TREEWY_STATUS_BAD_SLOT;
  if (flags) {
    if (t == 0 && h == 0) atomicOr(b.status + r, flags);
    return;
  }
  // the snapshots of an invalid tree were never written
  bool bad = false;
  if (t < N) {
    const int p = __ldg(b.parent + lo + t);
    bad = !(p >= -1 && p < t);
  }
  if (__syncthreads_or(bad)) {
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE);
    return;
  }
  const int64_t head_elems = static_cast<int64_t>(b.dv) * b.dk;
  const int64_t rel = static_cast<int64_t>(lo) - b.node_offset[0] + a;
  const float* src = snapshots + (rel * H + h) * head_elems;
  float* dst = static_cast<float*>(b.state) + (static_cast<int64_t>(slot) * H + h) * head_elems;
  if ((head_elems & 3) == 0) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* d4 = reinterpret_cast<float4*>(dst);
    for (int64_t f = t; f < head_elems / 4; f += kThreads) d4[f] = s4[f];
  } else {
    for (int64_t f = t; f < head_elems; f += kThreads) dst[f] = src[f];
  }
}

}  // namespace

cudaError_t launch_storeall_verify(const treewy_batch& b, float* snapshots, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  if (b.dk == 128 && b.dv == 128) {
    const size_t smem = sizeof(float) * 3 * kMaxNodes * 128;
    static std::atomic<uint64_t> attr_done{0};
    const cudaError_t attr = once_per_device(attr_done, [smem] {
      return cudaFuncSetAttribute(storeall_verify_rows_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    });
    if (attr != cudaSuccess) return attr;
    storeall_verify_rows_kernel<<<grid, kThreads, smem, stream>>>(b, snapshots);
    return cudaGetLastError();
  }
  const int npm = b.max_nodes;
  const size_t smem = storeall_layout(b.dk, b.dv, npm).total;
  cudaError_t err = cudaFuncSetAttribute(storeall_verify_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  storeall_verify_kernel<<<grid, kThreads, smem, stream>>>(b, snapshots, npm);
  return cudaGetLastError();
}

cudaError_t launch_storeall_commit(const treewy_batch& b, const float* snapshots,
                                   const int32_t* accepted, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  storeall_commit_kernel<<<grid, kThreads, 0, stream>>>(b, snapshots, accepted);
  return cudaGetLastError();
}

}  // namespace treewy
