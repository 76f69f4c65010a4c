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
// dk = dv = 128 (storeall_verify_rows_kernel) each thread owns 4 rows x 16
// columns, the nodes are walked in depth-first pre-order and a parent's
// snapshot is read back only after a branch point; other head sizes
// (storeall_verify_kernel) use a half-row-per-thread layout in index order,
// where a node whose parent is not the previous node reloads the parent's
// snapshot (which the same thread wrote) from global memory.
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

// Fast path for dk = dv = 128.  Thread layout: warp w, lane l = 8 rg + lr
// owns rows d_i = 16 w + 4 rg + i (i < 4) at columns c_j = 32 j + 4 lr .. +3
// (j < 4), so the eight lanes of a row group hold a whole row: S k and S q
// are three-step shuffle reductions over those lanes, and for each (i, j) the
// lanes lr = 0..7 store 128 contiguous bytes of a snapshot row.  Nodes are
// walked in DFS pre-order (children in index order), so the registers already
// hold the parent's state except after a branch point, where the parent's
// snapshot is read back; the next node's k, q and v are requested while the
// current node is computed.
constexpr int kRowsT = 4;       // rows per thread
constexpr int kColChunks = 4;   // 4-column chunks per thread

// k, q (columns c_j) and v (rows d_i) of one node as stored: bf16 pairs
// (18 words) or f32 (36 words); element e of chunk j is kv(j, e).
template <bool BF16>
struct NodeVecs;

template <>
struct NodeVecs<true> {
  uint2 k[kColChunks], q[kColChunks], v;
  __device__ __forceinline__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
  __device__ __forceinline__ static float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
  __device__ __forceinline__ float kv(int j, int e) const {
    return e == 0 ? lo(k[j].x) : e == 1 ? hi(k[j].x) : e == 2 ? lo(k[j].y) : hi(k[j].y);
  }
  __device__ __forceinline__ float qv(int j, int e) const {
    return e == 0 ? lo(q[j].x) : e == 1 ? hi(q[j].x) : e == 2 ? lo(q[j].y) : hi(q[j].y);
  }
  __device__ __forceinline__ float vv(int i) const {
    return i == 0 ? lo(v.x) : i == 1 ? hi(v.x) : i == 2 ? lo(v.y) : hi(v.y);
  }
  __device__ __forceinline__ void load(const treewy_batch& b, int64_t row, int lr, int d0) {
    const uint2* kg = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(b.k) + row * 128);
    const uint2* qg = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(b.q) + row * 128);
#pragma unroll
    for (int j = 0; j < kColChunks; ++j) {
      k[j] = __ldg(kg + 8 * j + lr);
      q[j] = __ldg(qg + 8 * j + lr);
    }
    v = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(b.v) + row * 128 + d0));
  }
};

template <>
struct NodeVecs<false> {
  float4 k[kColChunks], q[kColChunks], v;
  __device__ __forceinline__ static float el(const float4& x, int e) {
    return e == 0 ? x.x : e == 1 ? x.y : e == 2 ? x.z : x.w;
  }
  __device__ __forceinline__ float kv(int j, int e) const { return el(k[j], e); }
  __device__ __forceinline__ float qv(int j, int e) const { return el(q[j], e); }
  __device__ __forceinline__ float vv(int i) const { return el(v, i); }
  __device__ __forceinline__ void load(const treewy_batch& b, int64_t row, int lr, int d0) {
    const float4* kg = reinterpret_cast<const float4*>(static_cast<const float*>(b.k) + row * 128);
    const float4* qg = reinterpret_cast<const float4*>(static_cast<const float*>(b.q) + row * 128);
#pragma unroll
    for (int j = 0; j < kColChunks; ++j) {
      k[j] = __ldg(kg + 8 * j + lr);
      q[j] = __ldg(qg + 8 * j + lr);
    }
    v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(b.v) + row * 128 + d0));
  }
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
    storeall_verify_rows_kernel(const treewy_batch b, float* __restrict__ snapshots) {
  __shared__ int s_parent[kMaxNodes];
  __shared__ int s_size[kMaxNodes];     // subtree sizes
  __shared__ int s_depth[kMaxNodes];
  __shared__ int s_pre[kMaxNodes];      // DFS pre-order position
  __shared__ int s_order[kMaxNodes];    // node at each position
  __shared__ float s_alpha[kMaxNodes], s_beta[kMaxNodes];
  __shared__ int s_info[6];             // tok0, N, slot, flags, base row, max depth
  constexpr int kD = 128;

  const int H = b.H;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;

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
    s_info[5] = 0;
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
    s_parent[t] = bad ? -1 : p;
    s_alpha[t] = __ldg(b.alpha + (tok0 + t) * H + h);
    s_beta[t] = __ldg(b.beta + (tok0 + t) * H + h);
    s_size[t] = 1;
  }
  if (__syncthreads_or(bad)) {
    if (t == 0 && h == 0) atomicOr(b.status + r, TREEWY_STATUS_BAD_TREE);
    return;
  }
  // ---- DFS pre-order: depths, subtree sizes (deepest level first), then
  //      positions (shallowest level first): a node comes right after its
  //      parent plus the subtrees of its earlier siblings
  if (t < N) {
    int dep = 1;
    for (int c = s_parent[t]; c >= 0; c = s_parent[c]) ++dep;
    s_depth[t] = dep;
    atomicMax(&s_info[5], dep);
  }
  __syncthreads();
  const int maxd = s_info[5];
  for (int lev = maxd; lev >= 2; --lev) {
    if (t < N && s_depth[t] == lev) atomicAdd(&s_size[s_parent[t]], s_size[t]);
    __syncthreads();
  }
  for (int lev = 1; lev <= maxd; ++lev) {
    if (t < N && s_depth[t] == lev) {
      const int p = s_parent[t];
      int pos = (p < 0) ? 0 : s_pre[p] + 1;
      for (int m = 0; m < t; ++m)
        if (s_parent[m] == p) pos += s_size[m];
      s_pre[t] = pos;
      s_order[pos] = t;
    }
    __syncthreads();
  }

  const int w = t >> 5, l = t & 31, rg = l >> 3, lr = l & 7;
  const int d0 = 16 * w + 4 * rg;  // rows d0 .. d0+3
  constexpr int64_t kHead = kD * kD;
  const float* S0 = static_cast<const float*>(b.state) + (static_cast<int64_t>(s_info[2]) * H + h) * kHead;
  auto snap = [&](int n) { return snapshots + ((rel0 + n) * H + h) * kHead; };
  float4 S[kRowsT][kColChunks];
  auto load_state = [&](const float* src) {
#pragma unroll
    for (int i = 0; i < kRowsT; ++i)
#pragma unroll
      for (int j = 0; j < kColChunks; ++j)
        S[i][j] = *reinterpret_cast<const float4*>(src + (d0 + i) * kD + 32 * j + 4 * lr);
  };
  load_state(S0);
  // an f32 batch reloads its vectors per node (no registers for a second set)
  NodeVecs<BF16> cur, nxt;
  cur.load(b, (tok0 + s_order[0]) * H + h, lr, d0);
  int prev = -1;  // node whose state the registers hold (-1: S0)
  for (int pos = 0; pos < N; ++pos) {
    const int n = s_order[pos];
    if (BF16 && pos + 1 < N) nxt.load(b, (tok0 + s_order[pos + 1]) * H + h, lr, d0);
    if (!BF16 && pos > 0) cur.load(b, (tok0 + n) * H + h, lr, d0);
    const int p = s_parent[n];
    if (p != prev) load_state(p < 0 ? S0 : snap(p));  // after a branch point: the parent's snapshot
    // S k over the row's 128 columns: 16 products here, the rest in the row group
    float sk[kRowsT];
#pragma unroll
    for (int i = 0; i < kRowsT; ++i) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < kColChunks; ++j) {
        a = fmaf(S[i][j].x, cur.kv(j, 0), a);
        a = fmaf(S[i][j].y, cur.kv(j, 1), a);
        a = fmaf(S[i][j].z, cur.kv(j, 2), a);
        a = fmaf(S[i][j].w, cur.kv(j, 3), a);
      }
      sk[i] = a;
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
      for (int i = 0; i < kRowsT; ++i) sk[i] += __shfl_xor_sync(0xffffffffu, sk[i], o);
    // gated delta rule: S = alpha (S - beta (S k) k^T) + beta v k^T; o = S q
    const float a = s_alpha[n], be = s_beta[n];
    float* dst = snap(n);
    float so[kRowsT];
#pragma unroll
    for (int i = 0; i < kRowsT; ++i) {
      const float bsk = be * sk[i], bv = be * cur.vv(i);
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < kColChunks; ++j) {
        S[i][j].x = fmaf(a, fmaf(-bsk, cur.kv(j, 0), S[i][j].x), bv * cur.kv(j, 0));
        S[i][j].y = fmaf(a, fmaf(-bsk, cur.kv(j, 1), S[i][j].y), bv * cur.kv(j, 1));
        S[i][j].z = fmaf(a, fmaf(-bsk, cur.kv(j, 2), S[i][j].z), bv * cur.kv(j, 2));
        S[i][j].w = fmaf(a, fmaf(-bsk, cur.kv(j, 3), S[i][j].w), bv * cur.kv(j, 3));
        acc = fmaf(S[i][j].x, cur.qv(j, 0), acc);
        acc = fmaf(S[i][j].y, cur.qv(j, 1), acc);
        acc = fmaf(S[i][j].z, cur.qv(j, 2), acc);
        acc = fmaf(S[i][j].w, cur.qv(j, 3), acc);
        *reinterpret_cast<float4*>(dst + (d0 + i) * kD + 32 * j + 4 * lr) = S[i][j];
      }
      so[i] = acc;
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
      for (int i = 0; i < kRowsT; ++i) so[i] += __shfl_xor_sync(0xffffffffu, so[i], o);
    if (lr < kRowsT) {
      // lane lr of the row group writes row d0 + lr (static indices by select)
      float v = so[0];
#pragma unroll
      for (int i = 1; i < kRowsT; ++i)
        if (lr == i) v = so[i];
      b.o[((tok0 + n) * H + h) * kD + d0 + lr] = v;
    }
    prev = n;
    if (BF16) cur = nxt;
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
    if (b.qkv_dtype == TREEWY_DTYPE_BF16)
      storeall_verify_rows_kernel<true><<<grid, kThreads, 0, stream>>>(b, snapshots);
    else
      storeall_verify_rows_kernel<false><<<grid, kThreads, 0, stream>>>(b, snapshots);
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
