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
constexpr uint32_t kKQStride = 272u;       // bf16 K/Q row: 256 bytes + 16 (bank offset)

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

// NT n8-tiles of vectors: NT = 1 holds keys 0..3 in slots 0..3 and queries
// 0..3 in slots 4..7 (trees of up to 4 nodes); NT = 2 holds keys 0..7 in
// slots 0..7 and queries in 8..15.  The K/Q region always has 16 rows (the
// Gram's M = 16 operand), unused ones zero.  Dynamic shared memory: alignment
// slack, the state tile (4 boxes of 32 fp32 or 2 of 64 bf16 columns, 128B
// swizzle), the 16 K/Q rows, the per-tree data.
template <bool SB, int NT>
struct SmallCfg {
  static constexpr int kMaxN = 4 * NT;  // node capacity
  static constexpr int kQ0 = kMaxN;     // slot of query 0
  static constexpr uint32_t kS0Bytes = SB ? 2u * kSChunk : 4u * kSChunk;
  static constexpr uint32_t kKQOff = kS0Bytes;
  static constexpr uint32_t kTreeOff = kKQOff + 16u * kKQStride;
  static constexpr uint32_t kDynSmem = 1024u + kTreeOff + static_cast<uint32_t>(sizeof(SmallTree));
};

// D += A B for one m16n8k16 bf16 tile with fp32 accumulation.  Fragments
// (g = lane / 4, q = lane % 4): a0 row g, columns 2q, 2q+1; a1 row g+8;
// a2 row g, columns 2q+8, 2q+9; a3 row g+8, those columns; b0 column g,
// rows 2q, 2q+1; b1 rows 2q+8, 2q+9; d[0..1] row g, columns 2q, 2q+1;
// d[2..3] row g+8.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds32(const unsigned char* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// One CTA per (request, head), 256 threads.  Warp w owns state rows
// 16w..16w+15; lane (g, q) = (lane / 4, lane % 4) holds rows 16w+g and
// 16w+g+8 of the MMA tiles, and for the solve takes row 16w+g (q < 2) or
// 16w+g+8 (q >= 2), writing U (q even) or o (q odd).
template <bool SB, int NT>
__global__ void __launch_bounds__(kSThreads, 3)
    verify_small_kernel(const __grid_constant__ CUtensorMap map_s0, const treewy_batch b) {
  using C = SmallCfg<SB, NT>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
  unsigned char* s0 = base;
  unsigned char* kqs = base + C::kKQOff;
  SmallTree& ts = *reinterpret_cast<SmallTree*>(base + C::kTreeOff);

  const int H = b.H;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int g = lane >> 2, q = lane & 3;
  const int row = 16 * warp + g + ((q & 2) ? 8 : 0);  // this lane's row in the solve
  const bool is_o = (q & 1) != 0;

  // Every thread reads the request's metadata and checks it (the same
  // outcome everywhere), so that its own loads follow one round trip later.
  const int lo = __ldg(b.node_offset + r), hi = __ldg(b.node_offset + r + 1);
  const int slot = __ldg(b.state_slot + r);
  int flags = 0;
  if (hi - lo < 0 || hi - lo > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
  else if (lo < 0 || static_cast<int64_t>(hi) > b.T) flags |= TREEWY_STATUS_BAD_TREE;
  if (slot < 0 || static_cast<int64_t>(slot) >= b.num_slots) flags |= TREEWY_STATUS_BAD_SLOT;
  const int N = flags ? 0 : hi - lo;  // at most C::kMaxN (the launcher's max_nodes bound)
  const bool issued = N > 0;

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
    if (issued) {
      const int y = (slot * H + h) * kSDim;
      mbar_arrive_expect_tx(&ts.bar, C::kS0Bytes);
#pragma unroll
      for (int c = 0; c < (SB ? 2 : 4); ++c)
        tma_load_2d(s0 + c * kSChunk, &map_s0, &ts.bar, (SB ? 64 : 32) * c, y);
    }
  }

  *reinterpret_cast<uint4*>(kqs + kv * kKQStride + (t & 15) * 16) = kraw;
  if (t < 128) (t < 64 ? &ts.A[0][0] : &ts.M[0][0])[t & 63] = 0.f;
  bool bad = false;
  if (t < N) {
    bad = !(p >= -1 && p < t);
    ts.par[t] = bad ? -1 : p;
    ts.alpha[t] = al;
  }
  const bool bad_tree = __syncthreads_or(bad);
  const bool work = issued && !bad_tree;

  if (work && warp == 0) {
    // ---- Gram: slot_m . slot_n for the 16 slots m and the 8 slots n of the
    //      first tile (the B fragment of a slot row is its A fragment)
    float gd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const unsigned char* r0 = kqs + g * kKQStride + (16 * ks + 2 * q) * 2;
      const unsigned char* r1 = r0 + 8 * kKQStride;
      const uint32_t a0 = lds32(r0), a1 = lds32(r1), a2 = lds32(r0 + 16), a3 = lds32(r1 + 16);
      mma16816(gd, a0, a1, a2, a3, a0, a2);
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
  if (issued && t == 0 && !mbar_wait(&ts.bar, 0)) fail = 1;
  fail = __syncthreads_or(fail);
  const bool go = work && !fail;

  // ---- S0 [K;Q]^T, rows 16w..16w+15: per k-step of 16 state columns the A
  //      fragment is read from the swizzled tile and split into hi + lo (fp32
  //      state) or read as it is (bf16 state); one MMA per part and tile
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  if (go) {
    const int r0 = 16 * warp + g;  // and r0 + 8: the same swizzle phase
    const int sw = r0 & 7;
#pragma unroll 2
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t ah[4], al4[4];
      if constexpr (!SB) {
        // box ks / 2 holds columns 32 (ks / 2) .. + 31, four per 16-byte granule
        const unsigned char* box = s0 + (ks >> 1) * kSChunk;
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const int col = 16 * (ks & 1) + 2 * q + ((f & 2) ? 8 : 0);
          const int rr = r0 + ((f & 1) ? 8 : 0);
          const float2 x = *reinterpret_cast<const float2*>(box + rr * 128 + (((col >> 2) ^ sw) << 4) +
                                                            (col & 3) * 4);
          split_pair(x.x, x.y, ah[f], al4[f]);
        }
      } else {
        // box ks / 4 holds columns 64 (ks / 4) .. + 63, eight per granule
        const unsigned char* box = s0 + (ks >> 2) * kSChunk;
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const int col = 16 * (ks & 3) + 2 * q + ((f & 2) ? 8 : 0);
          const int rr = r0 + ((f & 1) ? 8 : 0);
          ah[f] = lds32(box + rr * 128 + (((col >> 3) ^ sw) << 4) + (col & 7) * 2);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const unsigned char* bp = kqs + (8 * nt + g) * kKQStride + (16 * ks + 2 * q) * 2;
        const uint32_t b0 = lds32(bp), b1 = lds32(bp + 16);
        mma16816(acc[nt], ah[0], ah[1], ah[2], ah[3], b0, b1);
        if constexpr (!SB) mma16816(acc[nt], al4[0], al4[1], al4[2], al4[3], b0, b1);
      }
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
    if (h == 0) bits |= flags | (issued && bad_tree ? TREEWY_STATUS_BAD_TREE : 0);
    if (bits) atomicOr(b.status + r, bits);
    // no copy may still target this CTA's memory at exit
    if (fail) mbar_wait(&ts.bar, 0);
  }
}

template <bool SB, int NT>
cudaError_t launch_small(const treewy_batch& b, const CUtensorMap& map_s0, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t attr = once_per_device(attr_done, [] {
    cudaError_t e = cudaFuncSetAttribute(verify_small_kernel<SB, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SmallCfg<SB, NT>::kDynSmem));
    // the whole unified L1/shared array as shared memory: three CTAs per SM
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(verify_small_kernel<SB, NT>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
    return e;
  });
  if (attr != cudaSuccess) return attr;
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  verify_small_kernel<SB, NT><<<grid, kSThreads, SmallCfg<SB, NT>::kDynSmem, stream>>>(map_s0, b);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify_small(const treewy_batch& b, const CUtensorMap& map_s0, cudaStream_t stream) {
  const bool sb = (b.flags & TREEWY_FLAG_STATE_BF16) != 0;
  if (b.max_nodes <= 4) return sb ? launch_small<true, 1>(b, map_s0, stream)
                                  : launch_small<false, 1>(b, map_s0, stream);
  return sb ? launch_small<true, 2>(b, map_s0, stream) : launch_small<false, 2>(b, map_s0, stream);
}

}  // namespace treewy
