// verify_tc.cuh -- TreeWY verification on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators, TMA staging) for dk = dv = 128, bf16 q/k/v,
// fp32 committed state.
//
// One CTA (256 threads, two warpgroups; thread t owns TMEM lane t % 128 =
// value row d) per (request, head).  With Np = N rounded up to 16:
//
//  TMA      S0 (fp32 state: 64 KB as 4 boxes of 128 rows x 32 columns; bf16
//           state: 32 KB as 2 boxes of 128 rows x 64 columns; 128B swizzle)
//           and the tree's K and Q rows (bf16, boxes of 32 and 16 rows).
//  tree     warps 0-1, while thread 64 issues MMA 1: gamma_n and each node's
//           root path with the decay ratios gamma_n / gamma_{p_k}.
//  split    fp32 state: each thread turns its own 128-byte S0 row segments in
//           place into [hi | lo] bf16 halves, S0 ~= hi + lo (16 significant
//           bits).  A bf16 state arrives in the operand layout as it is.
//  MMA 1    D1 = S0 [K;Q]^T   (M = 128, N = 2Np, K = 128; hi and lo accumulate
//           into one fp32 accumulator): column n = S0 k_n, column Np+n = S0 q_n
//           (TreeWY paper §3 Eq. (2), R term; review §3.2 Algorithm steps 3, 5).
//           D2 = [K;Q] K^T    (M = 128, N = Np): Gram rows k_m.k_i and q_m.k_i
//           (paper Eq. (2) G; review Algorithm step 2).
//  coeffs   per node n with root-to-n path p_0 = n, p_1 = parent(n), ...:
//             A[n, p_k] = beta_n (gamma_n/gamma_{p_k}) k_{p_k}.k_n  (k >= 1)
//             M[n, p_k] = (gamma_n/gamma_{p_k}) k_{p_k}.q_n         (k >= 0)
//           then the rows of T = (I + A)^-1 and B = M T restricted to the path,
//           each by its own O(depth^2) recurrence, since T (I + A) = I and
//           B (I + A) = M: row n solves x_q = r_q - sum_{a<q} x_a A[p_a, p_q]
//           with r = e_0 for T and r_q = M[n, p_q] for B.
//  MMA 2    U = T W and O = B W with W = diag(beta)(V - diag(gamma)(S0 K^T)^T),
//           as one product [U | O] = W^T [T;B]^T (M = 128, N = 2Np, K = Np;
//           bf16 hi/lo splits of W, T and B, three accumulating terms), so the
//           triangular solve of paper Eq. (2) needs no per-column recurrence.
//  store    U[n] and o_n = gamma_n S0 q_n + O[n] (review Eq. (5) restricted to
//           ancestors), coalesced, thread d writing column d.
//
// Nothing per node is kept beyond U (N x dv), the object that replaces the
// per-node snapshots (paper §3 "Reconstruct on commit").
#pragma once

#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

constexpr int kThreads = 256;
constexpr int kDim = 128;
constexpr uint32_t kS0ChunkBytes = 128u * 128u;     // 128 rows x 128 bytes (32 fp32 / 64 bf16)
constexpr uint32_t kS0Bytes = 4u * kS0ChunkBytes;   // 64 KB: S0, then W^T and [T;B]
// Operands of the second MMA, placed in the S0 region once the first is done:
// each is 128 rows x 128 bytes (K-major, 128B swizzle, K <= 64 bf16).
constexpr uint32_t kWhiOff = 0, kWloOff = 16384, kThiOff = 32768, kTloOff = 49152;
constexpr int kRegPath = 8;  // paths up to this length keep T/B rows in registers

template <int NPM>
struct TcCfg {
  // D1 = [S0k | S0q] in columns [0, 2NPM); the Gram, then [U | O], from 2NPM
  static constexpr uint32_t kCols = 4u * NPM;
  static_assert(NPM == 32 || NPM == 64, "tree capacity bucket (smaller trees have their own kernels)");
  static constexpr int kE = NPM * (NPM + 1) / 2;              // path-list entries, worst case
  static constexpr uint32_t kListBytes = 4u * kE;
  static constexpr uint32_t kPidxBytes = (kE + 15u) & ~15u;
  static constexpr uint32_t kR2Bytes = kPidxBytes + kListBytes;  // pidx + (pc | B scratch)
  // K/Q: two 64-column chunks of 128 rows (the Gram's M = 128 operand), after
  // the S0 tile.
  static constexpr uint32_t kKQRows = 128u;
  static constexpr uint32_t kKQChunk = kKQRows * 128u;
  static constexpr uint32_t kKQ = 2u * kKQChunk;
  static constexpr uint32_t kKQOff = kS0Bytes;
  static constexpr uint32_t kS0Off = 0u;
  static constexpr uint32_t kR2Off = kS0Bytes + kKQ;
  static constexpr uint32_t kDynSmem = kR2Off + kR2Bytes + 1024u;
  static_assert(3u * kListBytes <= kKQ, "A, M and T-scratch lists must fit the K/Q region");
};

// Dynamic shared memory of one kernel instance (the fused commit's update
// operands use the K/Q region of an fp32 instance, the free half of the state
// region of a bf16 one).
template <int NPM, bool FUSED, bool SB>
struct TcSmem {
  static constexpr uint32_t kBytes = TcCfg<NPM>::kDynSmem;
};

// Per-CTA tree data for one (request, head), sized by the capacity bucket.
template <int NPM>
struct __align__(16) TreeTC {
  int parent[NPM];
  float alpha[NPM];
  float gamma[NPM];
  float2 bbg[NPM];                      // (beta_n, beta_n * gamma_n)
  int D[NPM];                           // path length root..n, n included
  int off[NPM + 1];                     // CSR offsets of the path lists
  int tok0, N, slot;
  int flags;   // this round's request errors (node range, slot): verification skipped
  int cflags;  // fused commit refused: the previous round's errors | COMMIT_REFUSED
};

// Tree preparation by the 64 threads of warps 0 and 1 (thread n = node n;
// a batch holds at most 64 nodes per tree), synchronised on hardware barrier
// 3 so that the rest of the CTA is free meanwhile.  Validates the parents
// (p, alpha, beta: this thread's node as loaded by the caller), then walks
// each node's path once: gamma_n, the path length D_n, and the path list
// p_0 = n, p_1, ... with the decay products c_k = gamma_n / gamma_{p_k}
// formed as products of alpha along the path (no division); the first
// kRegPath entries wait in registers for the CSR offsets.  Returns false
// (uniformly over the 64 threads) when a parent index is out of range.
template <int NPM>
__device__ __forceinline__ bool prepare_tree(TreeTC<NPM>& ts, uint8_t* pidx, float* pc, int p,
                                             float alpha, float beta) {
  const int t = threadIdx.x;
  const int N = ts.N;
  bool bad = false;
  if (t < N) {
    bad = !(p >= -1 && p < t);
    ts.parent[t] = bad ? -1 : p;
    ts.alpha[t] = alpha;
  }
  if (named_bar_or<3, 64>(bad)) return false;
  int anc[kRegPath];
  float cc[kRegPath];
  int D = 0;
  if (t < N) {
    float c = 1.0f;
    int cur = t;
#pragma unroll
    for (int k = 0; k < kRegPath; ++k) {
      anc[k] = 0;
      cc[k] = 0.f;
      if (cur >= 0) {
        anc[k] = cur;
        cc[k] = c;
        const float a = k == 0 ? alpha : ts.alpha[cur];
        cur = k == 0 ? p : ts.parent[cur];
        c *= a;
        ++D;
      }
    }
    for (; cur >= 0; cur = ts.parent[cur]) {
      c *= ts.alpha[cur];
      ++D;
    }
    ts.gamma[t] = c;
    ts.bbg[t] = make_float2(beta, beta * c);
    ts.D[t] = D;
  }
  named_bar_sync<3, 64>();
  if (t < 32) {
    const int i0 = 2 * t, i1 = 2 * t + 1;
    const int a0 = i0 < N ? ts.D[i0] : 0;
    const int a1 = i1 < N ? ts.D[i1] : 0;
    int s = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (t >= o) s += y;
    }
    const int excl = s - a0 - a1;
    if (i0 < NPM) ts.off[i0] = excl;
    if (i1 < NPM) ts.off[i1] = excl + a0;
    if (t == 31) ts.off[NPM] = s;
  }
  named_bar_sync<3, 64>();
  if (t < N) {
    const int o = ts.off[t];
#pragma unroll
    for (int k = 0; k < kRegPath; ++k) {
      if (k < D) {
        pidx[o + k] = static_cast<uint8_t>(anc[k]);
        pc[o + k] = cc[k];
      }
    }
    if (D > kRegPath) {
      const int last = anc[kRegPath - 1];
      float c = cc[kRegPath - 1] * ts.alpha[last];
      int k = kRegPath;
      for (int cur = ts.parent[last]; cur >= 0; cur = ts.parent[cur], ++k) {
        pidx[o + k] = static_cast<uint8_t>(cur);
        pc[o + k] = c;
        c *= ts.alpha[cur];
      }
    }
  }
  return true;
}

// Thread-private in-place conversion of one 128-byte swizzled row segment:
// 32 fp32 values become 64 bf16 values [hi(32) | lo(32)] with
// hi = rn(x), lo = rn(x - hi), in the same 128B-swizzle layout.
__device__ __forceinline__ void convert_row_hilo(unsigned char* row, int sw) {
  float f[32];
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const float4 x = *reinterpret_cast<const float4*>(row + ((g ^ sw) << 4));
    f[4 * g + 0] = x.x;
    f[4 * g + 1] = x.y;
    f[4 * g + 2] = x.z;
    f[4 * g + 3] = x.w;
  }
  uint32_t hi[16], lo[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) split_pair(f[2 * j], f[2 * j + 1], hi[j], lo[j]);
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint32_t* src = (g < 4) ? (hi + 4 * g) : (lo + 4 * (g - 4));
    *reinterpret_cast<uint4*>(row + ((g ^ sw) << 4)) = make_uint4(src[0], src[1], src[2], src[3]);
  }
}

// Zero row `row` of the hi and lo halves of a K-major 128B-swizzled operand.
__device__ __forceinline__ void zero_operand_row(unsigned char* hi, unsigned char* lo, int row) {
  unsigned char* rh = hi + row * 128;
  unsigned char* rl = lo + row * 128;
#pragma unroll
  for (int g = 0; g < 8; ++g) {  // swizzled order: conflict-free across rows
    *reinterpret_cast<uint4*>(rh + ((g ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(rl + ((g ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Store x (hi/lo bf16) at column `col` of row `row` of a K-major 128B-swizzled operand.
__device__ __forceinline__ void put_operand(unsigned char* hi, unsigned char* lo, int row, int col,
                                            float x) {
  const __nv_bfloat16 xh = __float2bfloat16_rn(x);
  const __nv_bfloat16 xl = __float2bfloat16_rn(x - __bfloat162float(xh));
  const int byte = row * 128 + (((col >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1);
  *reinterpret_cast<__nv_bfloat16*>(hi + byte) = xh;
  *reinterpret_cast<__nv_bfloat16*>(lo + byte) = xl;
}

// Row of T = (I + A)^-1 (rhs = nullptr: r = e_0) or of B = M T (rhs = node n's
// M coefficients along its path) on node n's path p_0 = n, p_1, ...: solves
// x_q = r_q - sum_{a<q} x_a A[p_a, p_q], where A[p_a, p_q] is the entry of
// p_a's strict-ancestor list at position q - a, and writes x_q (hi/lo bf16) at
// column p_q of operand row `row`, which the caller has cleared.  `scratch`
// holds x for paths longer than kRegPath (registers otherwise).
template <int NPM>
__device__ __forceinline__ void build_path_row(const TreeTC<NPM>& ts, int n, int row,
                                               const uint8_t* pidx, const float* aco,
                                               const float* rhs, float* scratch,
                                               unsigned char* thi, unsigned char* tlo) {
  const int Dn = ts.D[n], o = ts.off[n];
  if (Dn <= kRegPath) {
    int col[kRegPath], opa[kRegPath];
    float x[kRegPath];
#pragma unroll
    for (int a = 0; a < kRegPath; ++a) {
      const int c = (a < Dn) ? pidx[o + a] : 0;
      col[a] = c;
      opa[a] = ts.off[c];
      x[a] = rhs ? ((a < Dn) ? rhs[o + a] : 0.f) : (a == 0 ? 1.0f : 0.f);
    }
#pragma unroll
    for (int q = 1; q < kRegPath; ++q) {
#pragma unroll
      for (int a = 0; a < q; ++a) {
        const float A = (q < Dn) ? aco[opa[a] + (q - a)] : 0.f;
        x[q] = fmaf(-x[a], A, x[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < kRegPath; ++q)
      if (q < Dn) put_operand(thi, tlo, row, col[q], x[q]);
  } else {
    for (int q = 0; q < Dn; ++q) scratch[o + q] = rhs ? rhs[o + q] : (q == 0 ? 1.0f : 0.f);
    for (int a = 0; a + 1 < Dn; ++a) {
      const float xa = scratch[o + a];
      const int opa = ts.off[pidx[o + a]];
      for (int q = a + 1; q < Dn; ++q) scratch[o + q] = fmaf(-xa, aco[opa + (q - a)], scratch[o + q]);
    }
    for (int q = 0; q < Dn; ++q) put_operand(thi, tlo, row, pidx[o + q], scratch[o + q]);
  }
}

// Previous-round data for the fused commit (shared memory; empty when the
// kernel is not fused).
constexpr int kPrevSeg = 8;  // path entries a warpgroup stages per 16-entry update segment
template <bool FUSED>
struct PrevSmem {
  int a;
};
template <>
struct PrevSmem<true> {
  int parent[kMaxNodes];
  float alpha[kMaxNodes];
  float c[kMaxNodes];                // gamma_a / gamma_{path j} (alpha products)
  uint8_t path[kMaxNodes];           // accepted node, its parent, ... (root last)
  int tok0, N, a, len;
  float gamma_a;
};

// SB: the state pool holds bf16 (2 chunks of 64 columns) instead of fp32
// (4 chunks of 32 columns).  Two CTAs share an SM either way (shared memory
// and TMEM); the instances other than the plain fp32 one for 64-node trees
// state it so the register allocation avoids spills, that one (0: no
// minimum) was measured faster with the default allocation.
template <int NPM, bool FUSED, bool SB>
__global__ void __launch_bounds__(kThreads, (SB || FUSED || NPM < 64) ? 2 : 0)
    verify_tc_kernel(const __grid_constant__ CUtensorMap map_s0,
                     const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_k32,
                     const __grid_constant__ CUtensorMap map_q32, const treewy_batch b,
                     const PrevRound prev) {
  using C = TcCfg<NPM>;
  constexpr int kChunks = SB ? 2 : 4;      // S0 boxes of 16 KB
  constexpr int kChunkCols = SB ? 64 : 32;
  // The fused commit forms its rank-|path| update on the tensor cores into
  // TMEM columns 0..127 (before the first products need them), with its
  // operands in a 16 KB tile: the free upper half of the state region for a
  // bf16 state; for an fp32 one the K/Q region (whose K/Q boxes are then
  // requested once the update has read it).
  constexpr bool kDeferKQ = FUSED && !SB;
  constexpr uint32_t kTmemCols = C::kCols;
  extern __shared__ unsigned char smem_raw[];
  __shared__ TreeTC<NPM> ts;
  __shared__ PrevSmem<FUSED> pv;
  // 0-3: S0 chunks, 4: K/Q, 5: S0 [K;Q]^T done, 6: second MMA done, 7: Gram
  // done, 8: the fused commit's update products done
  __shared__ __align__(8) uint64_t bars[9];
  __shared__ int s_kq_issued;   // the K/Q boxes have been requested
  __shared__ uint32_t tmem_holder;
  __shared__ int s_fail;
  __shared__ int s_bad_tree;    // written by thread 0 after the tree preparation
  __shared__ int s_mma_issued;  // written by the issuer of the first products

  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
  unsigned char* s0 = base + C::kS0Off;
  unsigned char* kq = base + C::kKQOff;
  uint8_t* pidx = base + C::kR2Off;
  float* pc = reinterpret_cast<float*>(pidx + C::kPidxBytes);
  float* xB = pc;  // long-path B rows reuse the decay products once consumed
  float* aco = reinterpret_cast<float*>(kq);
  float* mco = aco + C::kE;
  float* xT = mco + C::kE;
  unsigned char* thi = s0 + kThiOff;
  unsigned char* tlo = s0 + kTloOff;

  const int H = b.H;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const int lane = t & 127;  // TMEM lane = value row d
  const int wg = t >> 7;
  const int warp = t >> 5;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  bool mma2_issued = false;

  // Every thread reads the request's metadata itself, so that its node of
  // the tree and (warpgroup 1) its V columns are requested straight after
  // the first memory round trip rather than after thread 0 has published
  // it.  Nothing loaded here is used unless the request's checks
  // below pass; the range test only keeps the loads inside the batch.
  const int lo_s = __ldg(b.node_offset + r), hi_s = __ldg(b.node_offset + r + 1);
  const int slot_s = __ldg(b.state_slot + r);
  int pa_s = -1, plo_s = 0, phi_s = 0;
  if constexpr (FUSED) {
    pa_s = __ldg(prev.accepted + r);
    plo_s = __ldg(prev.node_offset + r);
    phi_s = __ldg(prev.node_offset + r + 1);
  }
  const int n_s = hi_s - lo_s;
  const bool range_ok = n_s > 0 && n_s <= b.max_nodes && lo_s >= 0 && static_cast<int64_t>(hi_s) <= b.T;
  int tree_p = -1;
  float tree_alpha = 0.f, tree_beta = 0.f;
  if (range_ok && t < n_s) {
    const int64_t row = static_cast<int64_t>(lo_s) + t;
    tree_p = __ldg(b.parent + row);
    tree_alpha = __ldg(b.alpha + row * H + h);
    tree_beta = __ldg(b.beta + row * H + h);
  }
  // Column `lane` of V for the warpgroup that builds W.  Each thread loads the
  // bf16 pair of columns (lane & ~1, lane | 1) of every other node (half the
  // load requests of one 2-byte load per node), and neighbouring lanes swap
  // halves after the tree is prepared.
  uint32_t vpk[NPM / 2];
#pragma unroll
  for (int i = 0; i < NPM / 2; ++i) vpk[i] = 0u;
  if (range_ok && wg == 1) {
    const uint32_t* vg = reinterpret_cast<const uint32_t*>(b.v);
    const int par = lane & 1;
#pragma unroll
    for (int i = 0; i < NPM / 2; ++i) {
      const int n = 2 * i + par;
      if (n < n_s && n < NPM)
        vpk[i] = __ldg(vg + (((static_cast<int64_t>(lo_s) + n) * H + h) * kDim + (lane & ~1)) / 2);
    }
  }

  // Fused commit: this thread's node of the previous tree, requested the
  // same way (used only when the previous request's checks pass).
  int prev_p = -1;
  float prev_al = 0.f;
  if constexpr (FUSED) {
    const int pn_s = phi_s - plo_s;
    const bool prange_ok = pa_s >= 0 && pn_s > 0 && pn_s <= prev.max_nodes && plo_s >= 0 &&
                           static_cast<int64_t>(phi_s) <= prev.T;
    if (prange_ok && t < pn_s) {
      const int64_t row = static_cast<int64_t>(plo_s) + t;
      prev_p = __ldg(prev.parent + row);
      prev_al = __ldg(prev.alpha + row * H + h);
    }
  }

  if (t == 0) {
#pragma unroll
    for (int i = 0; i < 9; ++i) mbar_init(&bars[i], 1);
    s_kq_issued = 0;
    fence_mbarrier_init();
    s_fail = 0;
    s_bad_tree = 0;
    s_mma_issued = 0;
    // every further metadata load of this CTA is independent: one round trip
    const int lo = lo_s, hi = hi_s;
    const int slot = slot_s;
    int pa = -1, plo = 0, phi = 0;
    if constexpr (FUSED) {
      pa = pa_s;
      plo = plo_s;
      phi = phi_s;
    }
    // errors of this round's request (they skip its verification) and of the
    // previous round (they refuse the fused commit) are kept apart, so that
    // either half runs exactly when the corresponding separate call would
    int flags = 0;
    const int N = hi - lo;
    if (N < 0 || N > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
    else if (lo < 0 || static_cast<int64_t>(hi) > b.T) flags |= TREEWY_STATUS_BAD_TREE;
    const bool bad_slot = slot < 0 || static_cast<int64_t>(slot) >= b.num_slots;
    if (bad_slot) flags |= TREEWY_STATUS_BAD_SLOT;
    int cflags = 0;
    if constexpr (FUSED) {
      // the previous round's accepted node and tree range for this request
      if (pa != -1) {
        const int pn = phi - plo;
        if (pn < 0 || pn > prev.max_nodes) cflags |= TREEWY_STATUS_TOO_MANY_NODES;
        else if (plo < 0 || static_cast<int64_t>(phi) > prev.T) cflags |= TREEWY_STATUS_BAD_TREE;
        if (pa < -1 || pa >= pn) cflags |= TREEWY_STATUS_BAD_ACCEPTED;
        if (cflags || bad_slot) cflags |= TREEWY_STATUS_COMMIT_REFUSED;
        pv.tok0 = plo;
        pv.N = pn;
      }
      pv.a = cflags ? -1 : pa;
    }
    ts.tok0 = lo;
    ts.N = flags ? 0 : N;
    ts.slot = slot;
    ts.flags = flags;
    ts.cflags = cflags;
    if (!bad_slot && ((flags == 0 && N > 0) || (FUSED && cflags == 0 && pa >= 0))) {
      const int y = (slot * H + h) * kDim;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        mbar_arrive_expect_tx(&bars[c], kS0ChunkBytes);
        tma_load_2d(s0 + c * kS0ChunkBytes, &map_s0, &bars[c], kChunkCols * c, y);
      }
    }
    if (flags == 0 && N > 0) {
      // 2 tensors x 2 column chunks x Np rows x 128 bytes (boxes past T are
      // zero-filled and count in full)
      mbar_arrive_expect_tx(&bars[4], static_cast<uint32_t>((N + 15) & ~15) * 512u);
    }
  }
  // The K and Q boxes, issued by the lanes of warp 0 in parallel (thread 0
  // has set up the barrier and the expected bytes).  Each issue costs the
  // issuing warp tens of cycles, so the Np = N rounded up to 16 rows of a
  // (tensor, column chunk) come as 32-row boxes and at most one 16-row box:
  // 4 boxes for N <= 32, 8 above, against 4 * N/8 boxes of 8 rows.  Rows
  // N..Np-1 (the next request's, or zero fill past T) are never used.
  auto issue_kq = [&]() {
    const int N = ts.N;
    if (ts.flags == 0 && N > 0) {
      const int Np = (N + 15) & ~15;
      const int n32 = Np >> 5;
      const int per = n32 + ((Np >> 4) & 1);  // boxes per (tensor, column chunk)
      for (int i = t; i < 4 * per; i += 32) {
        const int c2 = (i >> 1) & 1, j = i >> 2, rb = 32 * j;
        const bool big = j < n32;
        unsigned char* chunk = kq + c2 * C::kKQChunk;
        if (i & 1)
          tma_load_3d(chunk + (Np + rb) * 128, big ? &map_q32 : &map_q, &bars[4], 64 * c2, h,
                      ts.tok0 + rb);
        else
          tma_load_3d(chunk + rb * 128, big ? &map_k32 : &map_k, &bars[4], 64 * c2, h, ts.tok0 + rb);
      }
      if (t == 0) s_kq_issued = 1;
    }
  };
  // an fp32 fused commit that will run keeps the K/Q region for its update
  bool kq_deferred = false;
  if (warp == 0) {
    __syncwarp();
    if constexpr (kDeferKQ) kq_deferred = pv.a >= 0;
    if (!kq_deferred) issue_kq();
  } else if (warp == 1) {
    // TMEM is allocated by a warp that does not wait on the metadata loads
    tmem_alloc(&tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_holder;
  const int N = ts.N;
  const int Np = (N + 15) & ~15;
  const int nch = Np / 16;
  const bool issued = (ts.flags == 0 && N > 0);
  int commit_a = -1;  // accepted node of the previous round still to be applied
  if constexpr (FUSED) commit_a = pv.a;
  const bool have_s0 = issued || commit_a >= 0;
  const int64_t tok0 = ts.tok0;


  // Fused commit: validate the previous tree, walk the accepted node's path and
  // stage its first segment (c_j u_j[lane] and k_j[lane] in registers).
  bool bad_prev = false;
  float cu[kPrevSeg];
  uint32_t kb[kPrevSeg / 2];  // k_j[lane] of this thread's path entries, in pairs
#pragma unroll
  for (int j = 0; j < kPrevSeg; ++j) cu[j] = 0.f;
#pragma unroll
  for (int j = 0; j < kPrevSeg / 2; ++j) kb[j] = 0u;
  // The fused commit: this thread's part of a 16-entry path segment starting at
  // seg, entries seg + 8wg .. seg + 8wg + 7: c_j u_j[lane] (row `lane` of the
  // update's left operand) and k_j[lane] (row `lane` of its right operand),
  // zero past the path's end; all loads issued before any result is used.
  auto stage_tc = [&](int seg) {
    if constexpr (FUSED) {
      const unsigned short* kg = reinterpret_cast<const unsigned short*>(prev.k);
      uint32_t kh[kPrevSeg];
      float uv[kPrevSeg];
#pragma unroll
      for (int j = 0; j < kPrevSeg; ++j) {
        const int pos = seg + kPrevSeg * wg + j;
        kh[j] = 0u;
        uv[j] = 0.f;
        if (pos < pv.len) {
          const int64_t row = (static_cast<int64_t>(pv.tok0) + pv.path[pos]) * H + h;
          kh[j] = __ldg(kg + row * kDim + lane);
          uv[j] = __ldg(prev.U + row * kDim + lane);
        }
      }
#pragma unroll
      for (int j = 0; j < kPrevSeg; ++j) {
        const int pos = seg + kPrevSeg * wg + j;
        cu[j] = (pos < pv.len) ? pv.c[pos] * uv[j] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kPrevSeg / 2; ++j) kb[j] = kh[2 * j] | (kh[2 * j + 1] << 16);
    }
  };
  if constexpr (FUSED) {
    if (commit_a >= 0) {
      bool bad = false;
      if (t < pv.N) {
        bad = !(prev_p >= -1 && prev_p < t);
        pv.parent[t] = prev_p;
        pv.alpha[t] = prev_al;
      }
      bad_prev = __syncthreads_or(bad);
      if (!bad_prev && t == 0) {
        int len = 0;
        float c = 1.0f;
        for (int cur = commit_a; cur >= 0; cur = pv.parent[cur]) {
          pv.path[len] = static_cast<uint8_t>(cur);
          pv.c[len] = c;
          c *= pv.alpha[cur];
          ++len;
        }
        pv.len = len;
        pv.gamma_a = c;
      }
      __syncthreads();
      if (!bad_prev) stage_tc(0);
      __syncthreads();
    }
  }
  const bool commit_now = commit_a >= 0 && !bad_prev;
  if constexpr (kDeferKQ) {
    // a refused commit does not need the K/Q region: its boxes go now
    if (warp == 0 && kq_deferred && !commit_now) issue_kq();
  }
  if (wg == 1) {
    const int par = lane & 1;
#pragma unroll
    for (int i = 0; i < NPM / 2; ++i) {
      // this lane holds a column pair of node 2i+par, its neighbour of node 2i+1-par
      const uint32_t mine2 = vpk[i];
      const uint32_t other = __shfl_xor_sync(0xffffffffu, mine2, 1);
      // node 2i: from the even lane's load; node 2i+1: from the odd lane's load
      const uint32_t n0 = par ? other : mine2;   // node 2i columns pair
      const uint32_t n1 = par ? mine2 : other;   // node 2i+1 columns pair
      const uint32_t v0 = par ? (n0 >> 16) : (n0 & 0xFFFFu);
      const uint32_t v1 = par ? (n1 >> 16) : (n1 & 0xFFFFu);
      vpk[i] = v0 | (v1 << 16);
    }
  }

  // S0 chunks -> [hi | lo] bf16: warpgroup wg converts chunks 2wg, 2wg+1 of row
  // `lane` (fp32 state; a bf16 state's chunk wg is already an operand).
  // Waits on an mbarrier are done by one thread per warpgroup; the others
  // sleep at a hardware barrier instead of spinning.
  int fail = 0;
  if (have_s0) {
    if (lane == 0) {
      if constexpr (SB) fail = !mbar_wait(&bars[wg], 0);
      else fail = !(mbar_wait(&bars[2 * wg], 0) && mbar_wait(&bars[2 * wg + 1], 0));
    }
    fail = wg ? named_bar_or<2, 128>(fail) : named_bar_or<1, 128>(fail);
  }
  bool stored = false;  // the fused commit has stored S_a (uniform)
  int reb_pending = -1;  // thread 0: parity of an update product not yet waited for
  if constexpr (FUSED) {
    // S_a = gamma_a S0 + sum_j c_j u_j k_j^T on this thread's own part of row
    // `lane` (columns 64wg .. 64wg+63: chunks 2wg, 2wg+1 of an fp32 tile,
    // chunk wg of a bf16 one), written back once (rounded once for a bf16
    // state).
    if (commit_now && !__syncthreads_or(fail)) {
      const float ga = pv.gamma_a;
      const int len = pv.len;
      {
        // The update sum_j c_j u_j k_j^T on the tensor cores: per 16-entry
        // path segment, D += [c u]_hi K_p^T + [c u]_lo K_p^T (M = N = 128,
        // K = 16) into TMEM columns 0..127, both operands in one 128-row tile
        // (K-major, 128-byte swizzle): k-slot 0 holds (c_j u_j[d])_hi, slot 1
        // the _lo parts, slot 2 k_j[c]; thread (wg, lane) writes entries
        // 8wg..8wg+7 of row `lane` of each.  Then S_a = gamma_a S0 + D row by
        // row (rounded once for a bf16 state).
        unsigned char* opt = SB ? s0 + 2 * kS0ChunkBytes : kq;
        unsigned char* orow = opt + lane * 128;
        const int r7 = lane & 7;
        const int nseg = (len + 2 * kPrevSeg - 1) / (2 * kPrevSeg);
        for (int sg = 0; sg < nseg; ++sg) {
          uint32_t hi[kPrevSeg / 2], lo[kPrevSeg / 2];
#pragma unroll
          for (int j = 0; j < kPrevSeg / 2; ++j) split_pair(cu[2 * j], cu[2 * j + 1], hi[j], lo[j]);
          *reinterpret_cast<uint4*>(orow + (((0 + wg) ^ r7) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(orow + (((2 + wg) ^ r7) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint4*>(orow + (((4 + wg) ^ r7) << 4)) = make_uint4(kb[0], kb[1], kb[2], kb[3]);
          fence_proxy_async_smem();
          __syncthreads();
          if (t == 0) {
            tc_fence_after_sync();
            const uint64_t dt = smem_desc_sw128(smem_addr(opt), 1024);
            const uint32_t idr = idesc_bf16_f32(128, 128);
            mma_bf16(tmem, dt, dt + (64 >> 4), idr, sg ? 1u : 0u);
            mma_bf16(tmem, dt + (32 >> 4), dt + (64 >> 4), idr, 1u);
            mma_commit(&bars[8]);
            reb_pending = sg & 1;
          }
          // the next segment's values are requested while the products run
          if (sg + 1 < nseg) stage_tc(2 * kPrevSeg * (sg + 1));
          // the tile is rewritten (or D read) only once the products are done
          bool ok = true;
          if (t == 0) {
            ok = mbar_wait(&bars[8], sg & 1);
            if (ok) reb_pending = -1;
          }
          fail = __syncthreads_or(!ok);
          if (fail) break;
        }
        if constexpr (kDeferKQ) {
          // the update has read its tile: the K/Q boxes may land there now
          if (!fail && warp == 0) issue_kq();
        }
        if (!fail) {
          tc_fence_after_sync();
          if constexpr (SB) {
            unsigned char* row = s0 + wg * kS0ChunkBytes + lane * 128;
            for (int hb = 0; hb < 2; ++hb) {
              uint32_t d0[16], d1[16];
              tmem_ld16_async(tmem + lane_base + 64 * wg + 32 * hb, d0);
              tmem_ld16_async(tmem + lane_base + 64 * wg + 32 * hb + 16, d1);
              tmem_wait16(d0);
              tmem_wait16(d1);
#pragma unroll
              for (int g4 = 0; g4 < 4; ++g4) {
                unsigned char* gp = row + (((4 * hb + g4) ^ r7) << 4);
                const uint4 raw = *reinterpret_cast<const uint4*>(gp);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int j = 8 * g4 + 2 * i;  // column 64wg + 32hb + j
                  const float u0 = __uint_as_float(j < 16 ? d0[j] : d1[j - 16]);
                  const float u1 = __uint_as_float(j < 16 ? d0[j + 1] : d1[j - 15]);
                  const __nv_bfloat162 p = __floats2bfloat162_rn(fmaf(ga, __uint_as_float(w[i] << 16), u0),
                                                                 fmaf(ga, __uint_as_float(w[i] & 0xFFFF0000u), u1));
                  o[i] = *reinterpret_cast<const uint32_t*>(&p);
                }
                *reinterpret_cast<uint4*>(gp) = make_uint4(o[0], o[1], o[2], o[3]);
              }
            }
            // the bf16 chunk holds both column blocks: stored once both are
            // done.  The products only read the tile, so they are issued while
            // the store is still reading it; the store's read is waited for
            // further down, before anything overwrites the region.
            fence_proxy_async_smem();
            if (wg) named_bar_sync<2, 128>(); else named_bar_sync<1, 128>();
            if (lane == 0) {
              tma_store_2d(&map_s0, s0 + wg * kS0ChunkBytes, 64 * wg, (ts.slot * H + h) * kDim);
              bulk_commit_group();
            }
          } else {
            // fp32: chunk 2wg + hb of row `lane` = columns 64wg + 32hb ..; each
            // chunk goes back to the pool by a bulk tensor store while the
            // next one is formed
            for (int hb = 0; hb < 2; ++hb) {
              uint32_t d0[16], d1[16];
              tmem_ld16_async(tmem + lane_base + 64 * wg + 32 * hb, d0);
              tmem_ld16_async(tmem + lane_base + 64 * wg + 32 * hb + 16, d1);
              tmem_wait16(d0);
              tmem_wait16(d1);
              unsigned char* row = s0 + (2 * wg + hb) * kS0ChunkBytes + lane * 128;
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                float4* gp = reinterpret_cast<float4*>(row + ((g ^ r7) << 4));
                const float4 v = *gp;
                const int j = 4 * g;  // column 64wg + 32hb + j
                const float a0 = __uint_as_float(j < 16 ? d0[j] : d1[j - 16]);
                const float a1 = __uint_as_float(j < 16 ? d0[j + 1] : d1[j - 15]);
                const float a2 = __uint_as_float(j < 16 ? d0[j + 2] : d1[j - 14]);
                const float a3 = __uint_as_float(j < 16 ? d0[j + 3] : d1[j - 13]);
                *gp = make_float4(fmaf(ga, v.x, a0), fmaf(ga, v.y, a1), fmaf(ga, v.z, a2),
                                  fmaf(ga, v.w, a3));
              }
              fence_proxy_async_smem();
              if (wg) named_bar_sync<2, 128>(); else named_bar_sync<1, 128>();
              if (lane == 0) {
                tma_store_2d(&map_s0, s0 + (2 * wg + hb) * kS0ChunkBytes, 32 * (2 * wg + hb),
                             (ts.slot * H + h) * kDim);
                bulk_commit_group();
              }
            }
            if (!issued) {
              // nothing to convert: the stores still finish reading before the CTA ends
              if (lane == 0) bulk_wait_group_read0();
              if (wg) named_bar_sync<2, 128>(); else named_bar_sync<1, 128>();
            }
          }
          stored = true;
        }
      }
    }
  }
  if constexpr (!SB) {
    if (issued && !fail) {
      // a chunk is converted in place only after the fused commit's store has
      // read it: the first store is waited for while the second may still run
      if (FUSED && stored) {
        if (lane == 0) bulk_wait_group_read1();
        if (wg) named_bar_sync<2, 128>(); else named_bar_sync<1, 128>();
      }
      convert_row_hilo(s0 + (2 * wg) * kS0ChunkBytes + lane * 128, lane & 7);
      if (FUSED && stored) {
        if (lane == 0) bulk_wait_group_read0();
        if (wg) named_bar_sync<2, 128>(); else named_bar_sync<1, 128>();
      }
      convert_row_hilo(s0 + (2 * wg + 1) * kS0ChunkBytes + lane * 128, lane & 7);
    }
  }
  fence_proxy_async_smem();
  fail = __syncthreads_or(fail);

  // The first products need only S0 and K/Q, not the tree: thread 64 issues
  // them while warps 0 and 1 prepare the tree, so the walks run during the
  // products.  (A tree found invalid leaves the products unused; they are
  // waited for before the CTA ends.)
  const bool go = issued && !fail;
  if (go && t < 64) {
    const bool bad = !prepare_tree(ts, pidx, pc, tree_p, tree_alpha, tree_beta);
    if (t == 0) s_bad_tree = bad;
  } else if (go && t == 64) {
    if (!mbar_wait(&bars[4], 0)) {
      s_fail = 1;
    } else {
      tc_fence_after_sync();
      const uint64_t da = smem_desc_sw128(smem_addr(s0), 1024);
      const uint64_t db = smem_desc_sw128(smem_addr(kq), 1024);
      // S0 [K;Q]^T first: its completion frees the S0 region for W^T while the
      // Gram still runs; the Gram's commit covers both products, after which
      // the K/Q region and the rest of the S0 region are free.
      const uint32_t id1 = idesc_bf16_f32(128, 2 * Np);
      if constexpr (SB) {
        // chunk c = S0 columns 64c..64c+63 = the K/Q chunk c; one product per k-step
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint64_t bd = db + ((c * C::kKQChunk + s * 32) >> 4);
            const uint64_t a = da + ((c * kS0ChunkBytes + s * 32) >> 4);
            mma_bf16(tmem, a, bd, id1, (c | s) ? 1u : 0u);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint64_t bd = db + (((c >> 1) * C::kKQChunk + (c & 1) * 64 + s * 32) >> 4);
            const uint64_t ahi = da + ((c * kS0ChunkBytes + s * 32) >> 4);
            const uint64_t alo = da + ((c * kS0ChunkBytes + 64 + s * 32) >> 4);
            mma_bf16(tmem, ahi, bd, id1, (c | s) ? 1u : 0u);
            mma_bf16(tmem, alo, bd, id1, 1u);
          }
        }
      }
      mma_commit(&bars[5]);
      const uint32_t id2 = idesc_bf16_f32(128, Np);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t dsc = db + (((s >> 2) * C::kKQChunk + (s & 3) * 32) >> 4);
        mma_bf16(tmem + 2 * NPM, dsc, dsc, id2, s ? 1u : 0u);
      }
      mma_commit(&bars[7]);
      s_mma_issued = 1;
    }
  }
  if constexpr (FUSED && SB) {
    // a bf16 pool's S_a tile went out by bulk stores issued by lane 0 of each
    // warpgroup: they finish reading it here, while the products run and
    // before the second product's operands overwrite the region (and before
    // the CTA can end)
    if (lane == 0) bulk_wait_group_read0();
  }
  __syncthreads();
  fail |= s_fail;
  const bool bad_tree = go && s_bad_tree;
  const bool work = issued && !bad_tree;

  // Thread 0's last duties: the request's status bits, and (waits = true) a
  // check that no copy or product still targets this CTA's memory.  On the
  // full path every barrier has already been waited for by the thread that
  // consumed it, so only the status is written, before the stores of U and o
  // (which would otherwise hold it, and the CTA's exit, back); on every other
  // path both run at the end.
  bool finished = false;
  auto finish = [&](bool waits) {
    int bits = (fail ? kStatusTimeout : 0);
    if (h == 0) bits |= ts.flags | ts.cflags | (bad_tree ? TREEWY_STATUS_BAD_TREE : 0);
    // the previous round's tree failed its checks, or a wait gave up before
    // S_a was stored: that request's commit did not happen
    if (bad_prev && h == 0) bits |= TREEWY_STATUS_BAD_TREE | TREEWY_STATUS_COMMIT_REFUSED;
    if (fail && commit_now && !stored) bits |= TREEWY_STATUS_COMMIT_REFUSED;
    if (bits) atomicOr(b.status + r, bits);
    finished = true;
    if (!waits) return;
    // No async copy or MMA may still target this CTA's memory at exit.
    if constexpr (FUSED) {
      if (reb_pending >= 0) mbar_wait(&bars[8], reb_pending);
    }
    if (have_s0)
      for (int i = 0; i < kChunks; ++i) mbar_wait(&bars[i], 0);
    if (issued) {
      if (s_kq_issued) mbar_wait(&bars[4], 0);
      if (s_mma_issued) {
        mbar_wait(&bars[5], 0);
        mbar_wait(&bars[7], 0);
      }
      if (mma2_issued) mbar_wait(&bars[6], 0);
    }
  };

  if (work && !fail) {
    // warpgroup 1 (W^T) waits for S0 [K;Q]^T, warpgroup 0 for the Gram (both products)
    if (lane == 0 && !mbar_wait(&bars[wg ? 5 : 7], 0)) fail = 1;
    fail = wg ? named_bar_or<2, 128>(fail) : named_bar_or<1, 128>(fail);
    tc_fence_after_sync();
    if (fail) {
      // skip this warpgroup's work; the join below reports the failure
    } else if (wg == 0) {
      // ---- ancestor coefficients from this lane's Gram row.  The row is
      //      dumped to shared memory where this lane's own row of [T;B] will
      //      go (columns 0-31 in the hi operand row, 32-63 in the lo row, as
      //      16-byte groups of four columns, group g of a half at position
      //      g ^ (lane & 7): conflict-free across each eight lanes), then each
      //      lane walks its own node's path: A entries for lanes < N, M
      //      entries for lanes Np..Np+N-1.  No other lane reads the dump, so
      //      each lane clears its operand row as soon as its own walk is done.
      float* dhi = reinterpret_cast<float*>(thi + lane * 128);
      float* dlo = reinterpret_cast<float*>(tlo + lane * 128);
      const int gsw = lane & 7;
#pragma unroll
      for (int c = 0; c < NPM / 16; ++c) {
        if (c < nch) {
          // load and wait back to back: the load targets are written
          // asynchronously, so no other code may run in between
          uint32_t cur[16];
          tmem_ld16_async(tmem + lane_base + 2 * NPM + 16 * c, cur);
          tmem_wait16(cur);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int g = 4 * c + q;  // column group 0..15
            *reinterpret_cast<uint4*>((g < 8 ? dhi : dlo) + (((g & 7) ^ gsw) << 2)) =
                make_uint4(cur[4 * q], cur[4 * q + 1], cur[4 * q + 2], cur[4 * q + 3]);
          }
        }
      }
      // column i of the dumped row
      auto gram = [&](int i) {
        return ((i & 32) ? dlo : dhi)[((((i >> 2) & 7) ^ gsw) << 2) | (i & 3)];
      };
      const bool isA = lane < N;
      const int myn = isA ? lane : ((lane >= Np && lane < Np + N) ? lane - Np : -1);
      if (myn >= 0) {
        const int Dn = ts.D[myn], offn = ts.off[myn];
        const float scale = isA ? ts.bbg[myn].x : 1.0f;
        float* dst = isA ? aco : mco;
        const int k0 = isA ? 1 : 0;  // A has strict ancestors only
        if (Dn <= kRegPath) {
#pragma unroll
          for (int k = 0; k < kRegPath; ++k) {
            if (k >= k0 && k < Dn) {
              dst[offn + k] = scale * pc[offn + k] * gram(pidx[offn + k]);
            }
          }
        } else {
          for (int k = k0; k < Dn; ++k) dst[offn + k] = scale * pc[offn + k] * gram(pidx[offn + k]);
        }
      }
      if (lane < 2 * Np) zero_operand_row(thi, tlo, lane);
    } else {
      // ---- row `lane` of W^T: W[n][d] = beta_n v_n[d] - beta_n gamma_n (S0 k_n)[d]
      unsigned char* whi = s0 + kWhiOff + lane * 128;
      unsigned char* wlo = s0 + kWloOff + lane * 128;
      const int sw = lane & 7;
#pragma unroll
      for (int c = 0; c < NPM / 16; ++c) {
        if (c < nch) {
          uint32_t cur[16];
          tmem_ld16_async(tmem + lane_base + 16 * c, cur);
          tmem_wait16(cur);
          float w[16];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            // (beta, beta gamma) of nodes n and n + 1 in one 16-byte broadcast
            const int n = 16 * c + j;
            const uint32_t pair = vpk[n >> 1];
            const float4 bb = *reinterpret_cast<const float4*>(&ts.bbg[n]);
            const float v0 = __uint_as_float(pair << 16), v1 = __uint_as_float(pair & 0xFFFF0000u);
            w[j] = (n < N) ? fmaf(-bb.y, __uint_as_float(cur[j]), bb.x * v0) : 0.f;
            w[j + 1] = (n + 1 < N) ? fmaf(-bb.w, __uint_as_float(cur[j + 1]), bb.z * v1) : 0.f;
          }
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) split_pair(w[2 * j], w[2 * j + 1], hi[j], lo[j]);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int gg = 2 * c + g;
            *reinterpret_cast<uint4*>(whi + ((gg ^ sw) << 4)) =
                make_uint4(hi[4 * g], hi[4 * g + 1], hi[4 * g + 2], hi[4 * g + 3]);
            *reinterpret_cast<uint4*>(wlo + ((gg ^ sw) << 4)) =
                make_uint4(lo[4 * g], lo[4 * g + 1], lo[4 * g + 2], lo[4 * g + 3]);
          }
        }
      }
    }
    if (wg == 0 && !fail) {
      named_bar_sync<1, 128>();
      // ---- row t of [T;B] by thread t (the lane whose walk produced that
      //      node's coefficients): T rows for t < N, B rows for Np <= t < Np+N
      const bool isT = t < N, isB = t >= Np && t < Np + N;
      if (isT || isB)
        build_path_row(ts, isT ? t : t - Np, t, pidx, aco, isB ? mco : nullptr, isB ? xB : xT, thi, tlo);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    fail = __syncthreads_or(fail);
    if (!fail && t == 0) {
      tc_fence_after_sync();
      // [U | O] = W^T [T;B]^T as one N = 2Np product into the columns after the
      // (consumed) Gram; S0 q_n stays in columns Np..2Np-1.
      const uint64_t da = smem_desc_sw128(smem_addr(s0), 1024);
      const uint32_t id = idesc_bf16_f32(128, 2 * Np);
#pragma unroll
      for (int s = 0; s < NPM / 16; ++s) {
        if (s < nch) {
          const uint32_t ko = s * 32;
          const uint64_t whi = da + ((kWhiOff + ko) >> 4);
          const uint64_t wlo = da + ((kWloOff + ko) >> 4);
          const uint64_t thd = da + ((kThiOff + ko) >> 4);
          const uint64_t tld = da + ((kTloOff + ko) >> 4);
          mma_bf16(tmem + 2 * NPM, whi, thd, id, s ? 1u : 0u);
          mma_bf16(tmem + 2 * NPM, wlo, thd, id, 1u);
          mma_bf16(tmem + 2 * NPM, whi, tld, id, 1u);
        }
      }
      mma_commit(&bars[6]);
      mma2_issued = true;
    }
    if (!fail && t == 0 && !mbar_wait(&bars[6], 0)) fail = 1;
    fail = __syncthreads_or(fail);
    if (!fail) {
      tc_fence_after_sync();
      if (t == 0) finish(false);
      // ---- U[n] and o_n = gamma_n S0 q_n + O[n], column d = lane; warpgroup
      //      wg stores nodes 16c + 8wg .. 16c + 8wg + 7 of every 16-node chunk,
      //      reading only those 8 columns of U, O and S0 q, two chunks per
      //      wait (no code runs between the loads and their wait: the load
      //      targets are written asynchronously)
      float* og = b.o + (tok0 * H + h) * kDim + lane;
      float* ug = b.U + (tok0 * H + h) * kDim + lane;
      const int64_t stride = static_cast<int64_t>(H) * kDim;
      const int half = 8 * wg;
      constexpr int kPairs = (NPM / 16 + 1) / 2;
#pragma unroll
      for (int cp = 0; cp < kPairs; ++cp) {
        const int c0 = 2 * cp;
        if (c0 < nch) {
          uint32_t ua[8], oa[8], qa[8], ub[8], ob[8], qb[8];
          const bool two = (c0 + 1 < nch) && (c0 + 1 < NPM / 16);
          tmem_ld8_async(tmem + lane_base + 2 * NPM + 16 * c0 + half, ua);
          tmem_ld8_async(tmem + lane_base + 2 * NPM + Np + 16 * c0 + half, oa);
          tmem_ld8_async(tmem + lane_base + Np + 16 * c0 + half, qa);
          if (two) {
            tmem_ld8_async(tmem + lane_base + 2 * NPM + 16 * (c0 + 1) + half, ub);
            tmem_ld8_async(tmem + lane_base + 2 * NPM + Np + 16 * (c0 + 1) + half, ob);
            tmem_ld8_async(tmem + lane_base + Np + 16 * (c0 + 1) + half, qb);
          }
          tmem_wait8(ua, oa, qa);
          tmem_wait8(ub, ob, qb);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t(&u)[8] = k ? ub : ua;
            uint32_t(&oo)[8] = k ? ob : oa;
            uint32_t(&pq)[8] = k ? qb : qa;
            if (k == 0 || two) {
              // gamma of the eight nodes in two 16-byte broadcasts
              const int n0 = 16 * (c0 + k) + half;
              const float4 g0 = *reinterpret_cast<const float4*>(&ts.gamma[n0]);
              const float4 g1 = *reinterpret_cast<const float4*>(&ts.gamma[n0 + 4]);
              const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int n = n0 + j;
                if (n < N) {
                  ug[n * stride] = __uint_as_float(u[j]);
                  og[n * stride] = fmaf(gm[j], __uint_as_float(pq[j]), __uint_as_float(oo[j]));
                }
              }
            }
          }
        }
      }
      if (b.gamma != nullptr && t < N) b.gamma[(tok0 + t) * H + h] = ts.gamma[t];
    }
  }

  if (t == 0 && !finished) finish(true);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NPM, bool FUSED, bool SB>
cudaError_t launch_npm(const treewy_batch& b, const VerifyMaps& m, const PrevRound& prev,
                       cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t attr = once_per_device(attr_done, [] {
    cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel<NPM, FUSED, SB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(TcSmem<NPM, FUSED, SB>::kBytes));
    // the whole unified L1/shared array as shared memory, so that two
    // resident CTAs fit
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(verify_tc_kernel<NPM, FUSED, SB>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
    return e;
  });
  if (attr != cudaSuccess) return attr;
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  verify_tc_kernel<NPM, FUSED, SB><<<grid, kThreads, TcSmem<NPM, FUSED, SB>::kBytes, stream>>>(
      m.s0, m.k, m.q, m.k32, m.q32, b, prev);
  return cudaGetLastError();
}

// Plain verification (prev == nullptr) or with the previous round's commit
// fused in, for the tree-capacity bucket that covers npm.
template <bool SB>
cudaError_t launch_tc(const treewy_batch& b, const VerifyMaps& m, const PrevRound* prev, int npm,
                      cudaStream_t stream) {
  // plain verification of trees of more than 32 nodes; the fused form above
  // 16 nodes for an fp32 pool, above 32 for a bf16 one (smaller trees go to
  // the small-tree and warp-MMA kernels)
  if (prev == nullptr) return launch_npm<64, false, SB>(b, m, PrevRound{}, stream);
  if constexpr (!SB) {
    if (npm <= 32) return launch_npm<32, true, false>(b, m, *prev, stream);
  }
  return launch_npm<64, true, SB>(b, m, *prev, stream);
}

}  // namespace
}  // namespace treewy
