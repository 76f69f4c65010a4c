// verify_generic.cu -- TreeWY verification on CUDA cores, for any head size
// dk, dv <= 128 and bf16 or fp32 q/k/v (the tensor-core kernel covers
// dk = dv = 128 with bf16 q/k/v).
//
// One CTA per (request, head), 128 threads.  Steps (TreeWY paper §3 Eq. (2);
// technical review §3.2 Algorithm):
//   1. path decays gamma and strict-ancestor lists (tree_prepare);
//   2. S0 k_n, S0 q_n by dot products from shared memory;
//   3. ancestor-masked Gram entries A[n,i] = beta_n (gamma_n/gamma_i) k_i.k_n and
//      M[n,i] = (gamma_n/gamma_i) k_i.q_n, only for i an ancestor of n;
//   4. right-hand side W = beta (v - gamma S0 k), forward substitution for U,
//      read-out of o (review Eq. (5) restricted to ancestors).
#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

constexpr int kThreads = 128;

struct GenericLayout {
  int dk, dv, npm, E;
  size_t s0, kq, us, idx, coefA, coefM, qks, total;
};

__host__ __device__ inline GenericLayout generic_layout(int dk, int dv, int npm) {
  GenericLayout L;
  L.dk = dk;
  L.dv = dv;
  L.npm = npm;
  L.E = max_anc_entries(npm);
  size_t off = 0;
  L.s0 = off;    off += sizeof(float) * dv * (dk + 1);
  L.kq = off;    off += sizeof(float) * 2 * npm * (dk + 1);
  L.us = off;    off += sizeof(float) * npm * dv;
  L.coefA = off; off += sizeof(float) * L.E;
  L.coefM = off; off += sizeof(float) * L.E;
  L.qks = off;   off += sizeof(float) * npm;
  L.idx = off;   off += L.E;
  L.total = (off + 15) & ~size_t(15);
  return L;
}

__global__ void __launch_bounds__(kThreads)
    verify_generic_kernel(const treewy_batch b, int npm) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ TreeSmem ts;
  const GenericLayout L = generic_layout(b.dk, b.dv, npm);
  float* S0s = reinterpret_cast<float*>(smem + L.s0);
  float* Ks = reinterpret_cast<float*>(smem + L.kq);
  float* Qs = Ks + npm * (b.dk + 1);
  float* Us = reinterpret_cast<float*>(smem + L.us);
  float* coefA = reinterpret_cast<float*>(smem + L.coefA);
  float* coefM = reinterpret_cast<float*>(smem + L.coefM);
  float* qks = reinterpret_cast<float*>(smem + L.qks);
  uint8_t* idx = smem + L.idx;

  const int H = b.H, dk = b.dk, dv = b.dv;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const bool bf16 = b.qkv_dtype == TREEWY_DTYPE_BF16;

  if (t == 0) {
    const int lo = b.node_offset[r], hi = b.node_offset[r + 1];
    const int slot = b.state_slot[r];
    int flags = 0;
    const int N = hi - lo;
    if (N < 0 || N > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
    else if (lo < 0 || static_cast<int64_t>(hi) > b.T) flags |= TREEWY_STATUS_BAD_TREE;
    if (slot < 0 || static_cast<int64_t>(slot) >= b.num_slots) flags |= TREEWY_STATUS_BAD_SLOT;
    ts.tok0 = lo;
    ts.N = flags ? 0 : N;
    ts.slot = slot;
    ts.flags = flags;
  }
  __syncthreads();
  if (ts.flags) {
    if (t == 0 && h == 0) atomicOr(b.status + r, ts.flags);
    return;
  }
  const int N = ts.N;
  if (N == 0) return;
  if (!tree_prepare(ts, b.parent, b.alpha, b.beta, H, h)) {
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE);
    return;
  }
  const int64_t tok0 = ts.tok0;

  // stage S0 (row pitch dk+1 keeps column reads conflict-free), K, Q, V
  const bool state_bf16 = (b.flags & TREEWY_FLAG_STATE_BF16) != 0;
  const int64_t s0_base = (static_cast<int64_t>(ts.slot) * H + h) * dv * dk;
  for (int e = t; e < dv * dk; e += kThreads) {
    const int d = e / dk, j = e - d * dk;
    S0s[d * (dk + 1) + j] = load_qkv(b.state, s0_base + e, state_bf16);
  }
  for (int e = t; e < N * dk; e += kThreads) {
    const int n = e / dk, j = e - n * dk;
    const int64_t g = ((tok0 + n) * H + h) * dk + j;
    Ks[n * (dk + 1) + j] = load_qkv(b.k, g, bf16);
    Qs[n * (dk + 1) + j] = load_qkv(b.q, g, bf16);
  }
  for (int e = t; e < N * dv; e += kThreads) {
    const int n = e / dv, j = e - n * dv;
    Us[n * dv + j] = load_qkv(b.v, ((tok0 + n) * H + h) * dv + j, bf16);
  }
  __syncthreads();

  auto dot = [&](const float* x, const float* y) {
    float s = 0.f;
    for (int j = 0; j < dk; ++j) s = fmaf(x[j], y[j], s);
    return s;
  };

  // ancestor-masked Gram coefficients: threads 0..63 build node t's A entries,
  // threads 64..127 node (t-64)'s M entries (and the self term q_n.k_n)
  if (t < N) {
    const int n = t;
    const float bn = ts.beta[n];
    for_each_ancestor(ts, n, [&](int j, int i, float c) {
      const int e = ts.aoff[n] + j;
      idx[e] = static_cast<uint8_t>(i);
      coefA[e] = bn * c * dot(Ks + n * (dk + 1), Ks + i * (dk + 1));
    });
  } else if (t >= 64 && t - 64 < N) {
    const int n = t - 64;
    for_each_ancestor(ts, n, [&](int j, int i, float c) {
      coefM[ts.aoff[n] + j] = c * dot(Qs + n * (dk + 1), Ks + i * (dk + 1));
    });
    qks[n] = dot(Qs + n * (dk + 1), Ks + n * (dk + 1));
  }

  // right-hand side W[n][d] = beta_n (v_n[d] - gamma_n (S0 k_n)[d]), in place of V
  const int d = t;
  if (d < dv) {
    for (int n = 0; n < N; ++n) {
      const float pk = dot(S0s + d * (dk + 1), Ks + n * (dk + 1));
      Us[n * dv + d] = ts.beta[n] * (Us[n * dv + d] - ts.gamma[n] * pk);
    }
  }
  __syncthreads();

  if (d < dv) {
    solve_inplace(ts, Us, dv, d, idx, coefA);
    for (int n = 0; n < N; ++n) {
      const float pq = dot(S0s + d * (dk + 1), Qs + n * (dk + 1));
      const float o = readout_node(ts, n, pq, Us, dv, d, idx, coefM, qks);
      const int64_t g = ((tok0 + n) * H + h) * dv + d;
      b.o[g] = o;
      b.U[g] = Us[n * dv + d];
    }
  }
  if (b.gamma != nullptr && t < N) b.gamma[(tok0 + t) * H + h] = ts.gamma[t];
}

}  // namespace

size_t verify_generic_smem(int dk, int dv, int npm) { return generic_layout(dk, dv, npm).total; }

cudaError_t launch_verify_generic(const treewy_batch& b, cudaStream_t stream) {
  const int npm = b.max_nodes;
  const size_t smem = verify_generic_smem(b.dk, b.dv, npm);
  cudaError_t err = cudaFuncSetAttribute(verify_generic_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  verify_generic_kernel<<<grid, kThreads, smem, stream>>>(b, npm);
  return cudaGetLastError();
}

}  // namespace treewy
