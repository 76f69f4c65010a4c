// verify_small.cu -- TreeWY verification of small draft trees (at most 8
// nodes, e.g. multi-token-prediction chains) for dk = dv = 128, bf16 q/k/v,
// fp32 or bf16 committed state.
//
// With N <= 8 the first products S0 [K;Q]^T multiply the 128 x 128 state by
// at most 16 vectors, so the call is bound by reading S0 (64 KB per head),
// and the fixed costs of the tensor-core kernel (TMEM allocation and round
// trips, ~80-cycle tcgen05 issues for M = 128 products, the path lists and
// rows built for 64 nodes) dominate it.  Here the state tile lands in shared
// memory by bulk tensor copies and each warp multiplies its own 16 state rows
// with warp-level bf16 MMAs (m16n8k16, fp32 accumulation) whose operands come
// straight from registers: each state element is read from shared memory
// once and split into hi + lo bf16 halves on the way (16 significant bits),
// with no cross-warp reduction.  The rest of the method (TreeWY paper §3
// Eq. (2); review §3.2 Algorithm) is O(N^2) per value row:
//
//  Gram     warp 0: [K;Q] K^T as one more MMA per k-step (bf16 rows exact):
//           k_i.k_n and k_i.q_n.
//  tree     warp 0, lane n = node n: parent check, gamma_n, and the decay
//           ratios gamma_n / gamma_i along the root path as products of alpha,
//           giving the ancestor-masked
//             A[n, i] = beta_n (gamma_n/gamma_i) k_i.k_n   (i strict ancestor)
//             M[n, i] = (gamma_n/gamma_i) k_i.q_n          (i ancestor or n)
//  MMA 1    warp w: rows 16w..16w+15 of S0 k_n and S0 q_n.
//  solve    lane (row d, role): W_n = beta_n v_n - beta_n gamma_n (S0 k_n),
//           u_n = W_n - sum_{i anc n} A[n, i] u_i in node order (parents come
//           first): the unit-lower-triangular system (I + A) U = W.
//  read-out o_n = gamma_n (S0 q_n) + sum_{i anc-or-self n} M[n, i] u_i
//           (review Eq. (5) restricted to ancestors).
//  store    of each row d, one lane writes U[n][d], another o_n[d].
#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

constexpr int kSThreads = 256;
constexpr int kSDim = 128;
constexpr uint32_t kSChunk = 128u * 128u;  // one 16 KB box: 128 rows x 128 bytes
constexpr uint32_t kKQStride = 288u;       // bf16 K/Q row: 256 bytes + 32 (bank offset)
constexpr uint32_t kPathStride = 272u;     // bf16 key row of the accepted path: 256 + 16

// Per-tree data after the K/Q rows in dynamic shared memory.
struct SmallTree {
  uint64_t bar;         // state tile landed
  int par[8];
  float alpha[8];
  float bbg[8][2];      // (beta_n, beta_n gamma_n)
  float gamma[8];
  float gram[16][8];    // gram[m][n] = slot_m . slot_n for the vector slots below
  float A[8][8];        // A[n][i], zero unless i is a strict ancestor of n
  float M[8][8];        // M[n][i], zero unless i is n or an ancestor of n
};

// The previous round's tree and the accepted node's root path, for the
// commit fused in front of the verification.
struct SmallPrev {
  int parent[kMaxNodes];
  float alpha[kMaxNodes];
  float c[kMaxNodes];        // gamma_a / gamma_{path j} as products of alpha
  uint8_t path[kMaxNodes];   // accepted node, its parent, ... (root last)
  float w[8];                // previous trees of at most 8 nodes: c_j by node
  int onpath;                // ... and the nodes on the accepted path (bit j)
  int len;
  float gamma_a;
};
constexpr int kSeg = 8;      // path entries applied per pass over the tile
static_assert(kSeg == kSmallTreeNodes, "a bf16 pool's fused commit needs one pass per path");

// NT n8-tiles of vectors: NT = 1 holds keys 0..3 in slots 0..3 and queries
// 0..3 in slots 4..7 (trees of up to 4 nodes); NT = 2 holds keys 0..7 in
// slots 0..7 and queries in 8..15.  The K/Q region always has 16 rows (the
// Gram's M = 16 operand), unused ones zero.  Dynamic shared memory: alignment
// slack, the state tile (4 boxes of 32 fp32 or 2 of 64 bf16 columns, 128B
// swizzle), the 16 K/Q rows, the per-tree data; with the commit fused in,
// the previous tree and kSeg bf16 key rows of the accepted path.
template <bool SB, int NT, bool FUSED>
struct SmallCfg {
  static constexpr int kMaxN = 4 * NT;  // node capacity
  static constexpr int kQ0 = kMaxN;     // slot of query 0
  static constexpr uint32_t kS0Bytes = SB ? 2u * kSChunk : 4u * kSChunk;
  static constexpr uint32_t kKQOff = kS0Bytes;
  static constexpr uint32_t kTreeOff = kKQOff + 16u * kKQStride;
  static constexpr uint32_t kPrevOff = (kTreeOff + static_cast<uint32_t>(sizeof(SmallTree)) + 15u) & ~15u;
  static constexpr uint32_t kPathKOff = (kPrevOff + static_cast<uint32_t>(sizeof(SmallPrev)) + 15u) & ~15u;
  static constexpr uint32_t kEnd = FUSED ? kPathKOff + kSeg * kPathStride
                                         : kTreeOff + static_cast<uint32_t>(sizeof(SmallTree));
  static constexpr uint32_t kDynSmem = 1024u + kEnd;
  // three CTAs per SM: 228 KB of shared memory, 1 KB of it reserved per CTA
  static_assert(3u * (kDynSmem + 1024u) <= 228u * 1024u, "three CTAs per SM");
};

// Warp-level MMAs: mma16816_bf16 (treewy_device.cuh).
//
// The products only need A and B to agree on which state column each k
// stands for, so within a k-step of 16 columns k = 2q, 2q+1, 2q+8, 2q+9
// stand for columns 4q .. 4q+3: a lane reads one 16-byte granule of a state
// row (8 bytes of a bf16 one, or of a key row) per fragment row.  And the
// fragment rows g stand for state rows perm(g) (below), so that the lanes
// of each shared-memory load phase meet rows of different 128B-swizzle
// phases: every load of the state tile and of the key rows is free of bank
// conflicts.
__device__ __forceinline__ uint2 lds64(const unsigned char* p) {
  return *reinterpret_cast<const uint2*>(p);
}

// State row of fragment row g (0..7) of a warp's 16 rows.  fp32 tile: 16-byte
// loads run in phases of 8 lanes (fragment rows 2i, 2i+1), which take rows i
// and i+4, whose swizzles place the row's four granules in opposite halves
// of the 128-byte line.  bf16 tile: 8-byte loads run in phases of 16 lanes
// (rows 4i .. 4i+3), which take rows of distinct swizzle pairs 0, 2, 4, 6
// (or 1, 3, 5, 7).
template <bool SB>
__device__ __forceinline__ int frag_row(int g) {
  return SB ? ((g & 3) << 1) | (g >> 2) : (g >> 1) | ((g & 1) << 2);
}

// One CTA per (request, head), 256 threads.  Warp w owns state rows
// 16w..16w+15; lane (g, q) = (lane / 4, lane % 4) holds fragment rows g and
// g+8 of the MMA tiles, which stand for state rows r0 = 16w + frag_row(g) and
// r0 + 8, and for the solve takes row r0 (q < 2) or r0 + 8 (q >= 2), writing
// U (q even) or o (q odd).
//
// FUSED: the previous round's commit first, S_a = gamma_a S0 +
// sum_{j in path(a)} c_j u_j k_j^T with c_j = gamma_a / gamma_j (TreeWY
// paper §3 "Reconstruct on commit"), applied to the tile rows as the first
// products read them and written back to the pool once; the verification
// then runs from S_a.  Each half runs exactly when its separate call would:
// a refused commit leaves the state alone, a bad next tree still commits.
//
// Residency: three CTAs per SM for an fp32 pool (shared memory); a bf16 pool's
// 4-node instances fit more (40-43 KB), and are held to the registers of five
// (plain: 48) or four (fused: 64) CTAs per SM.
template <bool SB, int NT, bool FUSED>
__global__ void __launch_bounds__(kSThreads, (SB && NT == 1) ? (FUSED ? 4 : 5) : 3)
    verify_small_kernel(const __grid_constant__ CUtensorMap map_s0, const treewy_batch b,
                        const PrevRound prev) {
  using C = SmallCfg<SB, NT, FUSED>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
  unsigned char* s0 = base;
  unsigned char* kqs = base + C::kKQOff;
  SmallTree& ts = *reinterpret_cast<SmallTree*>(base + C::kTreeOff);
  SmallPrev& pv = *reinterpret_cast<SmallPrev*>(base + C::kPrevOff);  // FUSED only
  unsigned char* pathk = base + C::kPathKOff;                          // FUSED only

  const int H = b.H;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int g = lane >> 2, q = lane & 3;
  const int r0 = 16 * warp + frag_row<SB>(g);  // this lane's state rows r0 and r0 + 8
  const int row = r0 + ((q & 2) ? 8 : 0);       // and its row in the solve
  const bool is_o = (q & 1) != 0;

  // Every thread reads the request's metadata and checks it (the same
  // outcome everywhere), so that its own loads follow one round trip later.
  const int lo = __ldg(b.node_offset + r), hi = __ldg(b.node_offset + r + 1);
  const int slot = __ldg(b.state_slot + r);
  int flags = 0;
  if (hi - lo < 0 || hi - lo > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
  else if (lo < 0 || static_cast<int64_t>(hi) > b.T) flags |= TREEWY_STATUS_BAD_TREE;
  const bool bad_slot = slot < 0 || static_cast<int64_t>(slot) >= b.num_slots;
  if (bad_slot) flags |= TREEWY_STATUS_BAD_SLOT;
  const int N = flags ? 0 : hi - lo;  // at most C::kMaxN (the launcher's max_nodes bound)
  const bool issued = N > 0;
  // the previous round's request: its errors refuse the commit only
  int cflags = 0, commit_a = -1, plo = 0, pn = 0;
  if constexpr (FUSED) {
    const int pa = __ldg(prev.accepted + r);
    plo = __ldg(prev.node_offset + r);
    const int phi = __ldg(prev.node_offset + r + 1);
    pn = phi - plo;
    if (pa != -1) {
      if (pn < 0 || pn > prev.max_nodes) cflags |= TREEWY_STATUS_TOO_MANY_NODES;
      else if (plo < 0 || static_cast<int64_t>(phi) > prev.T) cflags |= TREEWY_STATUS_BAD_TREE;
      if (pa < -1 || pa >= pn) cflags |= TREEWY_STATUS_BAD_ACCEPTED;
      if (cflags || bad_slot) cflags |= TREEWY_STATUS_COMMIT_REFUSED;
    }
    commit_a = cflags ? -1 : pa;
  }
  const bool have_s0 = issued || commit_a >= 0;

  // this thread's 16 bytes of the K/Q rows: slot v = t / 16 (keys from slot
  // 0, queries from slot kQ0), zero where the slot holds no node
  const int kv = t >> 4;
  const int kn = kv < C::kQ0 ? kv : kv - C::kQ0;
  const bool kval = kv < 2 * C::kQ0 && kn < N;
  uint4 kraw = make_uint4(0u, 0u, 0u, 0u);
  if (kval) {
    const uint4* src = reinterpret_cast<const uint4*>(kv < C::kQ0 ? b.k : b.q);
    kraw = __ldg(src + ((static_cast<int64_t>(lo) + kn) * H + h) * (kSDim / 8) + (t & 15));
  }
  // node t of the tree
  int p = -1;
  float al = 0.f, be = 0.f;
  if (t < N) {
    const int64_t rw = static_cast<int64_t>(lo) + t;
    p = __ldg(b.parent + rw);
    al = __ldg(b.alpha + rw * H + h);
    be = __ldg(b.beta + rw * H + h);
  }
  // node t of the previous tree
  int pp = -1;
  float pal = 0.f;
  if (FUSED && commit_a >= 0 && t < pn) {
    const int64_t rw = static_cast<int64_t>(plo) + t;
    pp = __ldg(prev.parent + rw);
    pal = __ldg(prev.alpha + rw * H + h);
  }
  // A previous tree of at most kSeg nodes: every node's U values in this
  // lane's two state rows and (threads < 128) its key row are requested in
  // the same round trip as the tree; the path walk then only weights them
  // (c_j on the accepted path; nodes off it are skipped), so S_a waits for
  // no further memory round trip.
  const bool spec = FUSED && commit_a >= 0 && prev.max_nodes <= kSeg;
  // The update's left operand for this lane: u_j of entries j = 2q, 2q+1 in
  // rows r0 (cu[0], cu[1]) and r0 + 8 (cu[2], cu[3]), later times c_j.
  float cu[4] = {0.f, 0.f, 0.f, 0.f};
  uint4 pkr = make_uint4(0u, 0u, 0u, 0u);
  if (spec) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = 2 * q + e;
      if (j < pn) {
        const float* ur = prev.U + ((static_cast<int64_t>(plo) + j) * H + h) * kSDim;
        cu[e] = __ldg(ur + r0);
        cu[2 + e] = __ldg(ur + r0 + 8);
      }
    }
    if (t < kSeg * 16 && (t >> 4) < pn) {
      const uint4* kg4 = reinterpret_cast<const uint4*>(prev.k);
      pkr = __ldg(kg4 + ((static_cast<int64_t>(plo) + (t >> 4)) * H + h) * (kSDim / 8) + (t & 15));
    }
  }
  // column `row` of every node's v, as bf16 pairs until the solve
  uint32_t vpk[C::kMaxN / 2];
  const unsigned short* vg = reinterpret_cast<const unsigned short*>(b.v);
#pragma unroll
  for (int i = 0; i < C::kMaxN / 2; ++i) {
    uint32_t v0 = 0u, v1 = 0u;
    if (2 * i < N) v0 = __ldg(vg + ((static_cast<int64_t>(lo) + 2 * i) * H + h) * kSDim + row);
    if (2 * i + 1 < N) v1 = __ldg(vg + ((static_cast<int64_t>(lo) + 2 * i + 1) * H + h) * kSDim + row);
    vpk[i] = v0 | (v1 << 16);
  }
  // the state tile, requested once this thread's own loads are on their way
  if (t == 0) {
    mbar_init(&ts.bar, 1);
    fence_mbarrier_init();
    if (have_s0) {
      const int y = (slot * H + h) * kSDim;
      mbar_arrive_expect_tx(&ts.bar, C::kS0Bytes);
#pragma unroll
      for (int c = 0; c < (SB ? 2 : 4); ++c)
        tma_load_2d(s0 + c * kSChunk, &map_s0, &ts.bar, (SB ? 64 : 32) * c, y);
    }
  }

  *reinterpret_cast<uint4*>(kqs + kv * kKQStride + (t & 15) * 16) = kraw;
  if (spec && t < kSeg * 16) *reinterpret_cast<uint4*>(pathk + (t >> 4) * kPathStride + (t & 15) * 16) = pkr;
  if (t < 128) (t < 64 ? &ts.A[0][0] : &ts.M[0][0])[t & 63] = 0.f;
  bool bad = false;
  if (t < N) {
    bad = !(p >= -1 && p < t);
    ts.par[t] = bad ? -1 : p;
    ts.alpha[t] = al;
  }
  const bool bad_tree = __syncthreads_or(bad);
  const bool work = issued && !bad_tree;

  // ---- the previous tree: parents checked, then (thread 0) the accepted
  //      node's root path with the decay ratios c_j = gamma_a / gamma_j as
  //      products of alpha (no division), published by the barrier after the
  //      state tile's wait
  bool bad_prev = false;
  if constexpr (FUSED) {
    if (commit_a >= 0) {
      bool badp = false;
      if (t < pn) {
        badp = !(pp >= -1 && pp < t);
        pv.parent[t] = pp;
        pv.alpha[t] = pal;
      }
      bad_prev = __syncthreads_or(badp);
      if (!bad_prev && t == 0) {
        int len = 0, onpath = 0;
        float c = 1.f;
        for (int cur = commit_a; cur >= 0; cur = pv.parent[cur]) {
          pv.path[len] = static_cast<uint8_t>(cur);
          pv.c[len] = c;
          if (spec) {
            pv.w[cur] = c;
            onpath |= 1 << cur;
          }
          c *= pv.alpha[cur];
          ++len;
        }
        pv.len = len;
        pv.onpath = onpath;
        pv.gamma_a = c;
      }
    }
  }
  const bool commit_now = commit_a >= 0 && !bad_prev;

  if (work && warp == 0) {
    // ---- Gram: slot_m . slot_n for the 16 slots m and the 8 slots n of the
    //      first tile (the B fragment of a slot row is its A fragment)
    float gd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint2 x0 = lds64(kqs + g * kKQStride + (16 * ks + 4 * q) * 2);
      const uint2 x1 = lds64(kqs + (g + 8) * kKQStride + (16 * ks + 4 * q) * 2);
      mma16816_bf16(gd, x0.x, x1.x, x0.y, x1.y, x0.x, x0.y);
    }
    ts.gram[g][2 * q] = gd[0];
    ts.gram[g][2 * q + 1] = gd[1];
    ts.gram[g + 8][2 * q] = gd[2];
    ts.gram[g + 8][2 * q + 1] = gd[3];
    __syncwarp();
    // ---- decays and the masked coefficients, lane n = node n
    if (lane < N) {
      const int n = lane;
      // k_i.k_n, and k_i.q_n (slot kQ0 + n in the first tile for NT = 1;
      // query slot 8 + n against key i for NT = 2)
      auto kk = [&](int i) { return ts.gram[i][n]; };
      auto kq = [&](int i) { return NT == 1 ? ts.gram[i][C::kQ0 + n] : ts.gram[C::kQ0 + n][i]; };
      float c = 1.f;  // gamma_n / gamma_i as the product of alpha over (i, n]
      ts.M[n][n] = kq(n);
      int cur = n;
      for (int i = ts.par[n]; i >= 0; i = ts.par[i]) {
        c *= ts.alpha[cur];
        ts.A[n][i] = be * c * kk(i);
        ts.M[n][i] = c * kq(i);
        cur = i;
      }
      const float gm = c * ts.alpha[cur];  // times alpha of the root: gamma_n
      ts.gamma[n] = gm;
      ts.bbg[n][0] = be;
      ts.bbg[n][1] = be * gm;
    }
  }
  int fail = 0;
  if (have_s0 && t == 0 && !mbar_wait(&ts.bar, 0)) fail = 1;
  fail = __syncthreads_or(fail);
  const bool go = work && !fail;
  const bool commit_go = commit_now && !fail;

  // ---- passes over this warp's 16 tile rows, per k-step of 16 state
  //      columns: the fused commit's update applied to the A fragment's
  //      elements and written back to the tile, then the first products
  //      S0 [K;Q]^T with the fragment split into hi + lo (fp32 state) or used
  //      as it is (bf16 state), one MMA per part and tile.  A path longer
  //      than kSeg entries takes one update-only pass per further kSeg.
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const int len = (FUSED && commit_go) ? pv.len : 0;
  const int nseg = spec ? (commit_go ? 1 : 0) : (len + kSeg - 1) / kSeg;
  const int npass = nseg > 0 ? nseg : (go ? 1 : 0);
  const int sw = r0 & 7;  // rows r0 and r0 + 8: the same swizzle phase
  for (int ps = 0; ps < npass; ++ps) {
    const bool upd = ps < nseg;
    const bool mma_pass = go && ps == npass - 1;
    const int j0 = kSeg * ps;
    float ga = 1.f;
    // the update's A fragment (rows r0, r0 + 8; entries 2q, 2q+1 as k), split
    // into hi + lo bf16 halves
    uint32_t uh0 = 0u, uh1 = 0u, ul0 = 0u, ul1 = 0u;
    if constexpr (FUSED) {
      if (upd && spec) {
        // entries = the previous tree's nodes: those on the accepted path
        // weighted by c_j, the others zero (their key rows cleared as well)
        const int use = pv.onpath;
        if (t < kSeg * 16 && !((use >> (t >> 4)) & 1))
          *reinterpret_cast<uint4*>(pathk + (t >> 4) * kPathStride + (t & 15) * 16) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = 2 * q + e;
          const float w = ((use >> j) & 1) ? pv.w[j] : 0.f;
          cu[e] = ((use >> j) & 1) ? cu[e] * w : 0.f;
          cu[2 + e] = ((use >> j) & 1) ? cu[2 + e] * w : 0.f;
        }
        ga = pv.gamma_a;
        __syncthreads();  // the cleared key rows
      } else if (upd) {
        // c_j u_j of this lane's two rows for path entries j0 + 2q, j0 + 2q + 1,
        // and (shared) the key rows k_j of entries j0 .. j0 + kSeg - 1 (zero
        // past the path)
        if (ps > 0) __syncthreads();  // the previous pass has read the key rows
        if (t < kSeg * 16) {
          const int j = t >> 4;
          uint4 kr = make_uint4(0u, 0u, 0u, 0u);
          if (j0 + j < len) {
            const uint4* kg4 = reinterpret_cast<const uint4*>(prev.k);
            kr = __ldg(kg4 + ((static_cast<int64_t>(plo) + pv.path[j0 + j]) * H + h) * (kSDim / 8) +
                       (t & 15));
          }
          *reinterpret_cast<uint4*>(pathk + j * kPathStride + (t & 15) * 16) = kr;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + 2 * q + e;
          cu[e] = cu[2 + e] = 0.f;
          if (j < len) {
            const float* ur = prev.U + ((static_cast<int64_t>(plo) + pv.path[j]) * H + h) * kSDim;
            cu[e] = pv.c[j] * __ldg(ur + r0);
            cu[2 + e] = pv.c[j] * __ldg(ur + r0 + 8);
          }
        }
        if (ps == 0) ga = pv.gamma_a;
        __syncthreads();
      }
      if (upd) {
        split_pair(cu[0], cu[1], uh0, ul0);
        split_pair(cu[2], cu[3], uh1, ul1);
      }
    }
#pragma unroll(FUSED ? 1 : 2)
    for (int ks = 0; ks < 8; ++ks) {
      // a[hr], a[2 + hr]: row r0 + 8hr, state columns c0, c0+1 and c0+2, c0+3
      uint32_t ah[4], al4[4];
      const int c0 = 16 * ks + 4 * q;
      // the fused commit's update sum_j c_j u_j k_j^T on these elements, as
      // two tiles of warp MMAs: A = [c u] (rows; path entries as k), B = the
      // path's key rows, with D column n of tile tt standing for state column
      // 16 ks + 4 (n / 2) + 2 tt + n % 2, so that du[tt] lands on this lane's
      // columns c0 + 2 tt, c0 + 2 tt + 1 (rows r0: du[tt][0..1], r0 + 8: [2..3])
      float du[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if constexpr (FUSED) {
        if (upd) {
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
            const int pc = 16 * ks + 4 * (g >> 1) + 2 * tt + (g & 1);
            const uint32_t k0 = *reinterpret_cast<const unsigned short*>(pathk + (2 * q) * kPathStride + pc * 2);
            const uint32_t k1 = *reinterpret_cast<const unsigned short*>(pathk + (2 * q + 1) * kPathStride + pc * 2);
            const uint32_t bk = k0 | (k1 << 16);
            mma16816_bf16(du[tt], uh0, uh1, 0u, 0u, bk, 0u);
            mma16816_bf16(du[tt], ul0, ul1, 0u, 0u, bk, 0u);
          }
        }
      }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int rr = r0 + 8 * hr;
        // box c0 / 32 (fp32) or c0 / 64 (bf16), 16-byte granule in the row
        unsigned char* ep = SB ? s0 + (c0 >> 6) * kSChunk + rr * 128 +
                                     ((((c0 & 63) >> 3) ^ sw) << 4) + (c0 & 7) * 2
                               : s0 + (c0 >> 5) * kSChunk + rr * 128 + ((((c0 & 31) >> 2) ^ sw) << 4);
        float x[4];
        uint2 raw = make_uint2(0u, 0u);
        if constexpr (SB) {
          raw = lds64(ep);
          x[0] = __uint_as_float(raw.x << 16);
          x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
          x[2] = __uint_as_float(raw.y << 16);
          x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
        } else {
          const float4 v = *reinterpret_cast<const float4*>(ep);
          x[0] = v.x;
          x[1] = v.y;
          x[2] = v.z;
          x[3] = v.w;
        }
        if constexpr (FUSED) {
          if (upd) {
            // S_a = gamma_a S0 + sum_j c_j u_j k_j^T on these four elements
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = fmaf(ga, x[i], du[i >> 1][2 * hr + (i & 1)]);
            if constexpr (SB) {
              const __nv_bfloat162 p0 = __floats2bfloat162_rn(x[0], x[1]);  // rounded once
              const __nv_bfloat162 p1 = __floats2bfloat162_rn(x[2], x[3]);
              raw = make_uint2(*reinterpret_cast<const uint32_t*>(&p0),
                               *reinterpret_cast<const uint32_t*>(&p1));
              *reinterpret_cast<uint2*>(ep) = raw;
            } else {
              *reinterpret_cast<float4*>(ep) = make_float4(x[0], x[1], x[2], x[3]);
            }
          }
        }
        if constexpr (SB) {
          ah[hr] = raw.x;
          ah[2 + hr] = raw.y;
        } else {
          split_pair(x[0], x[1], ah[hr], al4[hr]);
          split_pair(x[2], x[3], ah[2 + hr], al4[2 + hr]);
        }
      }
      if (mma_pass) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 bk = lds64(kqs + (8 * nt + g) * kKQStride + c0 * 2);
          mma16816_bf16(acc[nt], ah[0], ah[1], ah[2], ah[3], bk.x, bk.y);
          if constexpr (!SB) mma16816_bf16(acc[nt], al4[0], al4[1], al4[2], al4[3], bk.x, bk.y);
        }
      }
    }
  }
  // the committed state goes back to the pool once every row is updated
  bool stored = false;
  if constexpr (FUSED) {
    if (commit_go) {
      fence_proxy_async_smem();
      __syncthreads();
      if (t == 0) {
#pragma unroll
        for (int c = 0; c < (SB ? 2 : 4); ++c)
          tma_store_2d(&map_s0, s0 + c * kSChunk, (SB ? 64 : 32) * c, (slot * H + h) * kSDim);
        bulk_commit_group();
      }
      stored = true;
    }
  }

  // ---- row `row`: gather its products from the quad, then W, the solve
  //      for U and (odd lanes) the read-out, and the stores
  if (go) {
    const int qb = lane & ~3;
    const bool upper = (q & 2) != 0;  // row g + 8 of the tile
    float s0v[2 * C::kMaxN];          // slot v of this row: keys, then queries
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int nn = 0; nn < 8; ++nn) {
        const float lo_v = __shfl_sync(0xffffffffu, acc[nt][nn & 1], qb + (nn >> 1));
        const float hi_v = __shfl_sync(0xffffffffu, acc[nt][2 + (nn & 1)], qb + (nn >> 1));
        s0v[8 * nt + nn] = upper ? hi_v : lo_v;
      }
    }
    float* dst = (is_o ? b.o : b.U) + (static_cast<int64_t>(lo) * H + h) * kSDim + row;
    const int64_t stride = static_cast<int64_t>(H) * kSDim;
    float u[C::kMaxN];
#pragma unroll
    for (int n = 0; n < C::kMaxN; ++n) {
      u[n] = 0.f;
      if (n < N) {
        const uint32_t pr = vpk[n >> 1];
        const float vn = __uint_as_float((n & 1) ? (pr & 0xFFFF0000u) : (pr << 16));
        float w = fmaf(-ts.bbg[n][1], s0v[n], ts.bbg[n][0] * vn);
#pragma unroll
        for (int i = 0; i < n; ++i) w = fmaf(-ts.A[n][i], u[i], w);
        u[n] = w;
        float val = w;
        if (is_o) {
          val = ts.gamma[n] * s0v[C::kQ0 + n];
#pragma unroll
          for (int i = 0; i <= n; ++i) val = fmaf(ts.M[n][i], u[i], val);
        }
        dst[n * stride] = val;
      }
    }
    if (b.gamma != nullptr && t < N) b.gamma[(static_cast<int64_t>(lo) + t) * H + h] = ts.gamma[t];
  }

  if (t == 0) {
    int bits = fail ? kStatusTimeout : 0;
    if (h == 0) bits |= flags | cflags | (issued && bad_tree ? TREEWY_STATUS_BAD_TREE : 0);
    // the previous tree failed its checks, or a wait gave up before S_a was
    // stored: that request's commit did not happen
    if (bad_prev && h == 0) bits |= TREEWY_STATUS_BAD_TREE | TREEWY_STATUS_COMMIT_REFUSED;
    if (fail && commit_now && !stored) bits |= TREEWY_STATUS_COMMIT_REFUSED;
    if (bits) atomicOr(b.status + r, bits);
    // no copy may still target this CTA's memory at exit
    if (fail) mbar_wait(&ts.bar, 0);
    if (stored) bulk_wait_group_read0();
  }
}

template <bool SB, int NT, bool FUSED>
cudaError_t launch_small(const treewy_batch& b, const CUtensorMap& map_s0, const PrevRound& prev,
                         cudaStream_t stream) {
  using C = SmallCfg<SB, NT, FUSED>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t attr = once_per_device(attr_done, [] {
    cudaError_t e = cudaFuncSetAttribute(verify_small_kernel<SB, NT, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kDynSmem));
    // the whole unified L1/shared array as shared memory: three or more CTAs per SM
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(verify_small_kernel<SB, NT, FUSED>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
    return e;
  });
  if (attr != cudaSuccess) return attr;
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  verify_small_kernel<SB, NT, FUSED><<<grid, kSThreads, C::kDynSmem, stream>>>(map_s0, b, prev);
  return cudaGetLastError();
}

template <bool FUSED>
cudaError_t launch_small_any(const treewy_batch& b, const CUtensorMap& map_s0, const PrevRound& prev,
                             cudaStream_t stream) {
  const bool sb = (b.flags & TREEWY_FLAG_STATE_BF16) != 0;
  if (b.max_nodes <= 4)
    return sb ? launch_small<true, 1, FUSED>(b, map_s0, prev, stream)
              : launch_small<false, 1, FUSED>(b, map_s0, prev, stream);
  return sb ? launch_small<true, 2, FUSED>(b, map_s0, prev, stream)
            : launch_small<false, 2, FUSED>(b, map_s0, prev, stream);
}

}  // namespace

cudaError_t launch_verify_small(const treewy_batch& b, const CUtensorMap& map_s0, const PrevRound* prev,
                                cudaStream_t stream) {
  if (prev == nullptr) return launch_small_any<false>(b, map_s0, PrevRound{}, stream);
  return launch_small_any<true>(b, map_s0, *prev, stream);
}

}  // namespace treewy
