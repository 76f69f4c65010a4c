// verify_warp.cu -- TreeWY verification of trees of 9 to 32 nodes with
// warp-level MMAs, dk = dv = 128, bf16 q/k/v, fp32 or bf16 committed state.
//
// One CTA of 256 threads per (request, head).  The state tile lands in
// shared memory by bulk tensor copies; warp w owns 16 of its rows (value
// dimensions) and carries them through every product of the method (TreeWY
// paper §3 Eq. (2); review §3.2) with m16n8k16 bf16 MMAs (fp32 accumulation)
// whose operands come straight from registers or shared memory:
//
//  MMA 1    S0 [K;Q]^T for the warp's rows: each state element is read once
//           and split into hi + lo bf16 halves on the way (fp32 state: two
//           MMAs per tile, 16 significant bits; a bf16 state needs one).
//  W        in the accumulator registers: W[d][n] = beta_n v_n[d] -
//           beta_n gamma_n (S0 k_n)[d], and the read-out's first term
//           gamma_n (S0 q_n)[d]; the accumulator layout of MMA 1 is already
//           the A-operand layout of MMA 2.
//  Gram     slots 16m..16m+15 of [K;Q] times K^T, the key columns split in
//           halves between warps m and m + NPM/8, each half written over its
//           warp's own (already read) rows of the state tile.
//  rows     thread t builds operand row t of [T;B], T = (I + A)^-1 and
//           B = M T restricted to node n's root path (both non-zero only
//           there), by the recurrence x_q = r_q - sum_{a<q} x_a A[p_a, p_q]
//           with A[m, j] = beta_m (gamma_m / gamma_j) k_j.k_m and
//           r = e_0 (T) or M[n, p_q] = (gamma_n / gamma_{p_q}) k_{p_q}.q_n (B);
//           the decay ratios are products of alpha along the path.
//  MMA 2    [U | O] = W [T;B]^T (W and [T;B] in hi + lo bf16, three terms),
//           O accumulated onto gamma_n S0 q_n; only the blocks of input nodes
//           that can be ancestors of a tile's nodes (parents precede their
//           children) are multiplied.
//  store    each lane writes its two adjacent value rows of U[n] and o_n.
//
// The kernel is written for a capacity NPM of up to 32 nodes, and launched
// for NPM = 16 (plain and fused) and 32 (plain; fused on a bf16 pool): three
// CTAs per SM fit (76 KB of shared memory at 16 nodes, 68 KB at 32 with the
// fp32 state streamed through a ring of three of its four boxes, 80
// registers; a bf16 pool's 16-node instances four CTAs, 44 KB and 64
// registers: its 32 KB tile region also holds the Gram rows and the [T;B]
// halves).  A 64-node version measured
// ~35 % slower than the tcgen05 kernel: the first products take two warp
// MMAs per 8-node tile and state element pair (hi and lo), and warp MMAs run
// at ~0.47 m16n8k16 per cycle per SM, about a quarter of the tcgen05 rate,
// so two resident 64-node CTAs keep the MMA pipe saturated.
#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

constexpr int kWThreads = 256;
constexpr int kWDim = 128;
constexpr uint32_t kWBox = 128u * 128u;  // one 16 KB box: 128 rows x 128 bytes
constexpr uint32_t kWKQStride = 288u;    // bf16 K/Q row: 256 bytes + 32 (bank offset)
constexpr int kWRegPath = 8;             // root paths up to this long stay in registers

template <int NPM>
struct WarpTree {
  uint64_t bar;   // state tile landed (ring: boxes 0-2)
  uint64_t bar3;  // ring: box 3 landed in box 0's slot
  int par[NPM];
  float alpha[NPM];
  float beta[NPM];
  float4 coef[NPM];  // (beta_n, beta_n gamma_n, gamma_n, 0)
};

// The previous round's tree and the accepted node's root path, for the
// commit fused in front of the verification; with kWSeg bf16 key rows of the
// path, they sit in the K/Q region until the update is applied (the K/Q rows
// wait in registers meanwhile).
struct WarpPrev {
  int parent[kMaxNodes];
  float alpha[kMaxNodes];
  float c[kMaxNodes];        // gamma_a / gamma_{path j} as products of alpha
  uint8_t path[kMaxNodes];   // accepted node, its parent, ... (root last)
  float w[16];               // previous trees of at most 16 nodes: c_j by node
  int onpath;                // ... and the nodes on the accepted path (bit j)
  int len;
  float gamma_a;
};
constexpr int kWSeg = 16;             // path entries applied per pass over the tile (the MMA's k)
constexpr uint32_t kWPathStride = 272u;  // bf16 key row of the path: 256 + 16
constexpr uint32_t kWPathOff = 1024u;    // key rows after WarpPrev in the K/Q region
static_assert(sizeof(WarpPrev) <= kWPathOff, "previous tree before the key rows");

// Dynamic shared memory: alignment slack, a 64 KB region that first holds
// the state tile (4 boxes of 32 fp32 or 2 of 64 bf16 columns, 128B swizzle)
// and later the Gram rows (box 0: each warp over its own state rows) and
// the hi and lo halves of the [T;B] operand (boxes 2 and 3), the 2 NPM K/Q
// slot rows (later the x scratch of root paths longer than kWRegPath), the
// tree.
template <int NPM, bool SB, bool FUSED>
struct WarpCfg {
  static constexpr int kSlots = 2 * NPM;  // keys 0..NPM-1, queries NPM..2NPM-1
  static constexpr int kKT = NPM / 8;     // n8-tiles of keys (and of queries)
  // A bf16 pool's instances: the 32 KB tile region also holds the Gram rows
  // (box 0) and the [T;B] halves (box 1).  32-node instances on an fp32 pool
  // keep three of the four 16 KB state boxes at a time: box 3 lands in box
  // 0's slot once every warp has multiplied box 0 (a ring of 48 KB), the
  // Gram rows go over slot 0, the [T;B] halves into slots 1 and 2.  Both
  // leave room for three CTAs per SM.
  static constexpr bool kCompact = SB;
  static constexpr bool kRing = !SB && NPM == 32 && !FUSED;
  static constexpr uint32_t kKQOff = (kCompact ? 2u : (kRing ? 3u : 4u)) * kWBox;
  static constexpr uint32_t kKQBytes = kSlots * kWKQStride;
  static constexpr uint32_t kTreeOff = kKQOff + kKQBytes;
  static constexpr uint32_t kEnd = kTreeOff + static_cast<uint32_t>(sizeof(WarpTree<NPM>));
  static constexpr uint32_t kDynSmem = 1024u + kEnd;
  // CTAs per SM (a fused fp32 32-node instance keeps the whole tile: two)
  static constexpr int kBlocks = (SB && NPM == 16) ? 4 : ((NPM == 16 || SB || kRing) ? 3 : 2);
  static_assert(kBlocks * (kDynSmem + 1024u) <= 228u * 1024u, "CTAs per SM");
  static_assert(8u * NPM * NPM <= kKQBytes, "x scratch of 2 NPM long paths");
  static_assert(2 * NPM <= kWThreads && NPM <= 32, "one operand row per thread; Gram halves in box 0");
  static_assert(kWPathOff + kWSeg * kWPathStride <= kKQBytes, "fused commit staging");
  static_assert(kWSeg == kWarpSegEntries, "entries per update pass");
};

// Fragment row g of a warp's tiles stands for state rows 16 w + 2 f(g) (row
// g) and 16 w + 2 f(g) + 1 (row g + 8): a lane's two rows are adjacent, so
// its v loads and U / o stores take both at once.  f pairs the fragment rows
// that share a shared-memory load phase (2i and 2i + 1 for 16-byte loads of
// an fp32 tile, 4i .. 4i + 3 for 8-byte loads of a bf16 tile) with rows of
// distinct 128B-swizzle phases, so no tile load has a bank conflict.
__device__ __forceinline__ int wfrag(int g) { return (g & 4) | ((g & 1) << 1) | ((g >> 1) & 1); }

__device__ __forceinline__ uint2 wlds64(const unsigned char* p) {
  return *reinterpret_cast<const uint2*>(p);
}

// Gram entry slot_m . key_i (fp32) in the Gram region of box 0.  The key
// columns come in two halves computed by different warps (warp w: slots of
// tile w mod KT, half w / KT); half h of slot m sits at state row m + 2 NPM h,
// i.e. over the computing warp's own rows, its words XOR-ed by (m mod 4) * 8
// so that the dump's 8-byte stores meet distinct banks.
template <int NPM>
__device__ __forceinline__ uint32_t gram_off(int m, int i) {
  const int hh = i / (NPM / 2);
  return static_cast<uint32_t>((m + 2 * NPM * hh) * 128 + (((i & 31) ^ ((m & 3) << 3)) << 2));
}

// [T;B] operand halves: row o = output column (T rows 0..NPM-1, B rows
// NPM..2NPM-1), column i = input node, in the 128-byte swizzled layout
// (sw128_off).
__device__ __forceinline__ void put_op(unsigned char* oph, unsigned char* opl, int o, int i, float x) {
  const __nv_bfloat16 xh = __float2bfloat16_rn(x);
  const __nv_bfloat16 xl = __float2bfloat16_rn(x - __bfloat162float(xh));
  const uint32_t off = sw128_off(o, i);
  *reinterpret_cast<__nv_bfloat16*>(oph + off) = xh;
  *reinterpret_cast<__nv_bfloat16*>(opl + off) = xl;
}

// FUSED: the previous round's commit first, S_a = gamma_a S0 +
// sum_{j in path(a)} c_j u_j k_j^T with c_j = gamma_a / gamma_j (TreeWY paper
// §3 "Reconstruct on commit"), applied to the state tile by update passes
// (two warp MMAs per 8-column tile and 8 path entries: A = c_j u_j of the
// warp's rows split into hi + lo bf16, B = the entries' key rows, the D
// columns ordered so that each lane's update lands on the elements it holds),
// written back to the pool once; the verification then runs from S_a.  Each
// half runs exactly when its separate call would: a refused commit leaves the
// state alone, a bad next tree still commits.
template <int NPM, bool SB, bool FUSED>
__global__ void __launch_bounds__(kWThreads, WarpCfg<NPM, SB, FUSED>::kBlocks)
    verify_warp_kernel(const __grid_constant__ CUtensorMap map_s0, const treewy_batch b,
                       const PrevRound prev) {
  using C = WarpCfg<NPM, SB, FUSED>;
  constexpr int KT = C::kKT;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
  unsigned char* s0 = base;
  unsigned char* kqs = base + C::kKQOff;
  WarpTree<NPM>& ts = *reinterpret_cast<WarpTree<NPM>*>(base + C::kTreeOff);
  WarpPrev& pv = *reinterpret_cast<WarpPrev*>(kqs);  // FUSED only
  unsigned char* pathk = kqs + kWPathOff;             // FUSED only

  const int H = b.H;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int g = lane >> 2, q = lane & 3;
  const int sr0 = 16 * warp + 2 * wfrag(g);  // this lane's state rows sr0, sr0 + 1

  // Every thread reads the request's metadata and checks it (the same
  // outcome everywhere), so that its own loads follow one round trip later.
  const int lo = __ldg(b.node_offset + r), hi = __ldg(b.node_offset + r + 1);
  const int slot = __ldg(b.state_slot + r);
  int flags = 0;
  if (hi - lo < 0 || hi - lo > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
  else if (lo < 0 || static_cast<int64_t>(hi) > b.T) flags |= TREEWY_STATUS_BAD_TREE;
  if (slot < 0 || static_cast<int64_t>(slot) >= b.num_slots) flags |= TREEWY_STATUS_BAD_SLOT;
  const int N = flags ? 0 : hi - lo;  // at most NPM (the launcher's max_nodes bound)
  const bool issued = N > 0;
  const bool bad_slot = (flags & TREEWY_STATUS_BAD_SLOT) != 0;
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
  // a commit to apply keeps the K/Q region for its staging: the K/Q rows
  // are stored there once the update is done
  const bool kq_late = FUSED && commit_a >= 0;
  const int64_t rowstride = static_cast<int64_t>(H) * kWDim;
  const int64_t node0 = static_cast<int64_t>(lo) * H + h;  // (node 0, head h) row

  // the K/Q slot rows this thread copies: 16 bytes of slot 16 p + t / 16 per
  // group p of 16 slots (two n8-tiles); groups of dead tiles are skipped
  constexpr int kGroups = C::kSlots / 16;
  uint4 kraw[kGroups];
#pragma unroll
  for (int p = 0; p < kGroups; ++p) {
    kraw[p] = make_uint4(0u, 0u, 0u, 0u);
    const int s = 16 * p + (t >> 4);
    const int n = s < NPM ? s : s - NPM;
    if (issued && n < N) {
      const uint4* src = reinterpret_cast<const uint4*>(s < NPM ? b.k : b.q);
      kraw[p] = __ldg(src + (node0 + static_cast<int64_t>(n) * H) * (kWDim / 8) + (t & 15));
    }
  }
  // node t of the tree
  int p_t = -1;
  float al_t = 0.f, be_t = 0.f;
  if (t < N) {
    const int64_t rw = static_cast<int64_t>(lo) + t;
    p_t = __ldg(b.parent + rw);
    al_t = __ldg(b.alpha + rw * H + h);
    be_t = __ldg(b.beta + rw * H + h);
  }
  // node t of the previous tree
  int pp = -1;
  float pal = 0.f;
  if (FUSED && commit_a >= 0 && t < pn) {
    const int64_t rw = static_cast<int64_t>(plo) + t;
    pp = __ldg(prev.parent + rw);
    pal = __ldg(prev.alpha + rw * H + h);
  }
  // A previous tree of at most kWSeg nodes: every node's U values in this
  // lane's two rows and (threads < 128) its key row are requested in the same
  // round trip as the tree; the path walk then only weights them (c_j on the
  // accepted path; nodes off it are skipped), so S_a waits for no further
  // memory round trip.  cu = the update's A operand (the m16n8k16 fragment,
  // path entries as k): u_j of entries j = 2q + e (cu[e], row sr0; cu[2 + e],
  // row sr0 + 1) and j = 2q + 8 + e (cu[4 + e], cu[6 + e]).
  const bool spec = FUSED && commit_a >= 0 && prev.max_nodes <= kWSeg;
  float cu[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  uint4 pkr = make_uint4(0u, 0u, 0u, 0u);
  if (spec) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = 2 * q + 8 * hh + e;
        if (j < pn) {
          const float2 u2 = __ldg(reinterpret_cast<const float2*>(
              prev.U + ((static_cast<int64_t>(plo) + j) * H + h) * kWDim + sr0));
          cu[4 * hh + e] = u2.x;
          cu[4 * hh + 2 + e] = u2.y;
        }
      }
    }
    if (t < kWSeg * 16 && (t >> 4) < pn) {
      const uint4* kg4 = reinterpret_cast<const uint4*>(prev.k);
      pkr = __ldg(kg4 + ((static_cast<int64_t>(plo) + (t >> 4)) * H + h) * (kWDim / 8) + (t & 15));
    }
  }
  // v_n at this lane's rows sr0, sr0 + 1 for the nodes n = 8 j + 2 q + e of
  // its accumulator columns, as bf16 pairs
  uint32_t vv[KT][2];
  const unsigned short* vg = reinterpret_cast<const unsigned short*>(b.v);
#pragma unroll
  for (int j = 0; j < KT; ++j) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 8 * j + 2 * q + e;
      vv[j][e] = 0u;
      if (n < N)
        vv[j][e] = __ldg(reinterpret_cast<const uint32_t*>(vg + (node0 + static_cast<int64_t>(n) * H) * kWDim + sr0));
    }
  }
  // the state tile, requested once this thread's own loads are on their way
  if (t == 0) {
    mbar_init(&ts.bar, 1);
    if constexpr (C::kRing) mbar_init(&ts.bar3, 1);
    fence_mbarrier_init();
    if (have_s0) {
      const int y = (slot * H + h) * kWDim;
      constexpr int kFirst = SB ? 2 : (C::kRing ? 3 : 4);  // boxes requested now
      mbar_arrive_expect_tx(&ts.bar, kFirst * kWBox);
#pragma unroll
      for (int c = 0; c < kFirst; ++c)
        tma_load_2d(s0 + c * kWBox, &map_s0, &ts.bar, (SB ? 64 : 32) * c, y);
    }
  }
  const int live_tiles = (N + 7) >> 3;  // n8-tiles of keys holding a node
  auto store_kq = [&]() {
#pragma unroll
    for (int p = 0; p < kGroups; ++p) {
      const int tile0 = 2 * p < KT ? 2 * p : 2 * p - KT;
      if (tile0 < live_tiles)
        *reinterpret_cast<uint4*>(kqs + (16 * p + (t >> 4)) * kWKQStride + (t & 15) * 16) = kraw[p];
    }
  };
  if (!kq_late) store_kq();
  if (spec && t < kWSeg * 16) *reinterpret_cast<uint4*>(pathk + (t >> 4) * kWPathStride + (t & 15) * 16) = pkr;
  bool bad = false;
  if (t < N) {
    bad = !(p_t >= -1 && p_t < t);
    ts.par[t] = bad ? -1 : p_t;
    ts.alpha[t] = al_t;
    ts.beta[t] = be_t;
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

  // gamma_n: the product of alpha over node n's root path
  if (work && t < N) {
    float c = 1.f;
    for (int cur = t; cur >= 0; cur = ts.par[cur]) c *= ts.alpha[cur];
    ts.coef[t] = make_float4(be_t, be_t * c, c, 0.f);
  }
  int fail = 0;
  if (have_s0 && t == 0 && !mbar_wait(&ts.bar, 0)) fail = 1;
  fail = __syncthreads_or(fail);
  const bool go = work && !fail;
  const bool commit_go = commit_now && !fail;

  // ---- the fused commit: update passes over this warp's rows of the tile,
  //      per k-step of 16 state columns, then S_a back to the pool
  bool stored = false;
  if constexpr (FUSED) {
    if (commit_go) {
      const int len = pv.len;
      const int nseg = spec ? 1 : (len + kWSeg - 1) / kWSeg;
      const int swz = sr0 & 7;
      for (int ps = 0; ps < nseg; ++ps) {
        const int j0 = kWSeg * ps;
        float ga = 1.f;
        if (spec) {
          // entries = the previous tree's nodes: those on the accepted path
          // weighted by c_j, the others zero (their key rows cleared as well)
          const int use = pv.onpath;
          if (t < kWSeg * 16 && !((use >> (t >> 4)) & 1))
            *reinterpret_cast<uint4*>(pathk + (t >> 4) * kWPathStride + (t & 15) * 16) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int j = 2 * q + 8 * hh + e;
              const bool on = (use >> j) & 1;
              const float wj = on ? pv.w[j] : 0.f;
              cu[4 * hh + e] = on ? cu[4 * hh + e] * wj : 0.f;
              cu[4 * hh + 2 + e] = on ? cu[4 * hh + 2 + e] * wj : 0.f;
            }
          }
          ga = pv.gamma_a;
          __syncthreads();  // the cleared key rows
        } else {
          // c_j u_j of this lane's two rows for path entries j0 + 2q + e and
          // j0 + 2q + 8 + e, and (shared) the key rows of entries j0 ..
          // j0 + kWSeg - 1 (zero past the path)
          if (ps > 0) __syncthreads();  // the previous pass has read the key rows
          if (t < kWSeg * 16) {
            const int j = t >> 4;
            uint4 kr = make_uint4(0u, 0u, 0u, 0u);
            if (j0 + j < len) {
              const uint4* kg4 = reinterpret_cast<const uint4*>(prev.k);
              kr = __ldg(kg4 + ((static_cast<int64_t>(plo) + pv.path[j0 + j]) * H + h) * (kWDim / 8) +
                         (t & 15));
            }
            *reinterpret_cast<uint4*>(pathk + j * kWPathStride + (t & 15) * 16) = kr;
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int j = j0 + 2 * q + 8 * hh + e;
              cu[4 * hh + e] = cu[4 * hh + 2 + e] = 0.f;
              if (j < len) {
                const float2 u2 = __ldg(reinterpret_cast<const float2*>(
                    prev.U + ((static_cast<int64_t>(plo) + pv.path[j]) * H + h) * kWDim + sr0));
                cu[4 * hh + e] = pv.c[j] * u2.x;
                cu[4 * hh + 2 + e] = pv.c[j] * u2.y;
              }
            }
          }
          if (ps == 0) ga = pv.gamma_a;
          __syncthreads();
        }
        uint32_t uh[4], ul[4];  // A fragment a0..a3, hi and lo halves
#pragma unroll
        for (int i = 0; i < 4; ++i) split_pair(cu[2 * i], cu[2 * i + 1], uh[i], ul[i]);
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
          const int c0 = 16 * ks + 4 * q;
          // D column n of tile tt stands for state column 16 ks + 4 (n / 2) +
          // 2 tt + n % 2, so du[tt] lands on this lane's columns c0 + 2 tt,
          // c0 + 2 tt + 1 (rows sr0: du[tt][0..1], sr0 + 1: du[tt][2..3])
          float du[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
            const int pc = 16 * ks + 4 * (g >> 1) + 2 * tt + (g & 1);
            // b0: key rows of entries 2q, 2q+1; b1: of entries 2q+8, 2q+9
            const unsigned char* kc = pathk + pc * 2;
            const uint32_t b0 = static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(kc + (2 * q) * kWPathStride)) |
                                (static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(kc + (2 * q + 1) * kWPathStride)) << 16);
            const uint32_t b1 = static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(kc + (2 * q + 8) * kWPathStride)) |
                                (static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(kc + (2 * q + 9) * kWPathStride)) << 16);
            mma16816_bf16_nv(du[tt], uh[0], uh[1], uh[2], uh[3], b0, b1);
            mma16816_bf16_nv(du[tt], ul[0], ul[1], ul[2], ul[3], b0, b1);
          }
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int rr = sr0 + hr;
            const int sr = swz ^ hr;
            if constexpr (SB) {
              unsigned char* ep = s0 + (c0 >> 6) * kWBox + rr * 128 + ((((c0 & 63) >> 3) ^ sr) << 4) + (c0 & 7) * 2;
              const uint2 raw = wlds64(ep);
              float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                            __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
#pragma unroll
              for (int i = 0; i < 4; ++i) x[i] = fmaf(ga, x[i], du[i >> 1][2 * hr + (i & 1)]);
              const __nv_bfloat162 p0 = __floats2bfloat162_rn(x[0], x[1]);  // rounded once
              const __nv_bfloat162 p1 = __floats2bfloat162_rn(x[2], x[3]);
              *reinterpret_cast<uint2*>(ep) = make_uint2(*reinterpret_cast<const uint32_t*>(&p0),
                                                         *reinterpret_cast<const uint32_t*>(&p1));
            } else {
              float4* ep = reinterpret_cast<float4*>(s0 + (c0 >> 5) * kWBox + rr * 128 +
                                                     ((((c0 & 31) >> 2) ^ sr) << 4));
              const float4 x = *ep;
              *ep = make_float4(fmaf(ga, x.x, du[0][2 * hr]), fmaf(ga, x.y, du[0][2 * hr + 1]),
                                fmaf(ga, x.z, du[1][2 * hr]), fmaf(ga, x.w, du[1][2 * hr + 1]));
            }
          }
        }
      }
      // the committed state goes back to the pool once every row is updated
      fence_proxy_async_smem();
      __syncthreads();
      if (t == 0) {
#pragma unroll
        for (int c = 0; c < (SB ? 2 : 4); ++c)
          tma_store_2d(&map_s0, s0 + c * kWBox, (SB ? 64 : 32) * c, (slot * H + h) * kWDim);
        bulk_commit_group();
      }
      stored = true;
    }
    if (kq_late) {
      // every read of the staging area is done (the barriers above): the K/Q
      // rows go to their region now
      if (go) store_kq();
      __syncthreads();
    }
  }

  int ring_fail = 0;  // ring: the wait for box 3 gave up (uniform)
  if (go) {
    // ---- MMA 1: acc[nt] = S0 [K;Q]^T, tile nt of slots 8 nt .. 8 nt + 7
    //      (keys: nt < KT; queries: nt >= KT).  Within a k-step of 16 state
    //      columns, k = 2q, 2q+1, 2q+8, 2q+9 stand for columns 4q .. 4q+3: a
    //      lane reads one 16-byte granule (8 bytes of a bf16 state) per row.
    float acc[2 * KT][4];
#pragma unroll
    for (int nt = 0; nt < 2 * KT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int sw = sr0 & 7;  // sr0 + 1: sw ^ 1
#pragma unroll 2
    for (int ks = 0; ks < 8; ++ks) {
      const int c0 = 16 * ks + 4 * q;
      if constexpr (C::kRing) {
        if (ks == 2) {
          // every warp is done with box 0: box 3 into its slot
          __syncthreads();
          if (t == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&ts.bar3, kWBox);
            tma_load_2d(s0, &map_s0, &ts.bar3, 96, (slot * H + h) * kWDim);
          }
        } else if (ks == 6) {
          int f3 = 0;
          if (t == 0 && !mbar_wait(&ts.bar3, 0)) f3 = 1;
          ring_fail = __syncthreads_or(f3);
        }
      }
      uint32_t ah[4], al4[4];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int rr = sr0 + hr;
        const int sr = sw ^ hr;
        if constexpr (SB) {
          const uint2 raw = wlds64(s0 + (c0 >> 6) * kWBox + rr * 128 + ((((c0 & 63) >> 3) ^ sr) << 4) +
                                   (c0 & 7) * 2);
          ah[hr] = raw.x;
          ah[2 + hr] = raw.y;
        } else {
          const int box = c0 >> 5;  // its slot: box 3 reuses box 0's (ring)
          const float4 x = *reinterpret_cast<const float4*>(s0 + ((C::kRing && box == 3) ? 0 : box) * kWBox +
                                                            rr * 128 + ((((c0 & 31) >> 2) ^ sr) << 4));
          split_pair(x.x, x.y, ah[hr], al4[hr]);
          split_pair(x.z, x.w, ah[2 + hr], al4[2 + hr]);
        }
      }
      // groups of 4 tiles: their hi products, then their lo products, so
      // that no MMA waits for the one before it
#pragma unroll
      for (int nt0 = 0; nt0 < 2 * KT; nt0 += 4) {
        uint2 bk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int nt = nt0 + i;
          bk[i] = make_uint2(0u, 0u);
          if ((nt < KT ? nt : nt - KT) < live_tiles) bk[i] = wlds64(kqs + (8 * nt + g) * kWKQStride + c0 * 2);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int nt = nt0 + i;
          if ((nt < KT ? nt : nt - KT) < live_tiles)
            mma16816_bf16_nv(acc[nt], ah[0], ah[1], ah[2], ah[3], bk[i].x, bk[i].y);
        }
        if constexpr (!SB) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int nt = nt0 + i;
            if ((nt < KT ? nt : nt - KT) < live_tiles)
              mma16816_bf16_nv(acc[nt], al4[0], al4[1], al4[2], al4[3], bk[i].x, bk[i].y);
          }
        }
      }
    }
    if (!ring_fail) {

    // ---- W in the key tiles, gamma_n S0 q_n in the query tiles (zero for
    //      nodes past N), then W as MMA 2's A fragments in hi + lo bf16:
    //      k-step s of input nodes 16 s .. 16 s + 15 is key tiles 2s, 2s+1
#pragma unroll
    for (int j = 0; j < KT; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int n = 8 * j + 2 * q + e;
        float be = 0.f, bg = 0.f, gm = 0.f;
        if (n < N) {
          const float4 cf = ts.coef[n];
          be = cf.x;
          bg = cf.y;
          gm = cf.z;
        }
        const float v0 = __uint_as_float(vv[j][e] << 16), v1 = __uint_as_float(vv[j][e] & 0xFFFF0000u);
        acc[j][e] = fmaf(-bg, acc[j][e], be * v0);
        acc[j][2 + e] = fmaf(-bg, acc[j][2 + e], be * v1);
        acc[KT + j][e] *= gm;
        acc[KT + j][2 + e] *= gm;
      }
    }
    uint32_t wh[KT / 2][4], wl[KT / 2][4];
#pragma unroll
    for (int s = 0; s < KT / 2; ++s) {
      split_pair(acc[2 * s][0], acc[2 * s][1], wh[s][0], wl[s][0]);
      split_pair(acc[2 * s][2], acc[2 * s][3], wh[s][1], wl[s][1]);
      split_pair(acc[2 * s + 1][0], acc[2 * s + 1][1], wh[s][2], wl[s][2]);
      split_pair(acc[2 * s + 1][2], acc[2 * s + 1][3], wh[s][3], wl[s][3]);
    }
    float oi[KT][4];
#pragma unroll
    for (int j = 0; j < KT; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) oi[j][i] = acc[KT + j][i];

    // ---- Gram: warps w and w + KT take the two halves of the live key
    //      tiles against slots 16 (w mod KT) .. + 15 (fragment rows g, g + 8)
    //      and write them over their own rows of the state tile (all read
    //      above; a fused commit's store of S_a must have read the tile first)
    if (stored) {
      if (t == 0) bulk_wait_group_read0();
      __syncthreads();
    }
    __syncwarp();
    if (warp < 2 * KT) {
      const int gmt = warp % KT, hh = warp / KT;
      const int mtp = gmt < KT / 2 ? gmt : gmt - KT / 2;  // key tile pair of these slots
      constexpr int kNH = KT / 2;                         // key tiles per half
      const int nt0 = hh * kNH;
      if (2 * mtp < live_tiles && nt0 < live_tiles) {
        float gd[kNH][4];
#pragma unroll
        for (int i = 0; i < kNH; ++i) gd[i][0] = gd[i][1] = gd[i][2] = gd[i][3] = 0.f;
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
          const int cb = (16 * ks + 4 * q) * 2;
          const uint2 x0 = wlds64(kqs + (16 * gmt + g) * kWKQStride + cb);
          const uint2 x1 = wlds64(kqs + (16 * gmt + g + 8) * kWKQStride + cb);
#pragma unroll
          for (int i = 0; i < kNH; ++i) {
            if (nt0 + i < live_tiles) {
              const uint2 bk = wlds64(kqs + (8 * (nt0 + i) + g) * kWKQStride + cb);
              mma16816_bf16_nv(gd[i], x0.x, x1.x, x0.y, x1.y, bk.x, bk.y);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < kNH; ++i) {
          const int col = 8 * (nt0 + i) + 2 * q;
          const int m0 = 16 * gmt + g;
          *reinterpret_cast<float2*>(s0 + gram_off<NPM>(m0, col)) = make_float2(gd[i][0], gd[i][1]);
          *reinterpret_cast<float2*>(s0 + gram_off<NPM>(m0 + 8, col)) = make_float2(gd[i][2], gd[i][3]);
        }
      }
    }
    __syncthreads();

    // ---- operand rows of [T;B]: thread t < NPM the T row of node t, thread
    //      NPM + n the B row of node n, over boxes 2 (hi) and 3 (lo)
    unsigned char* oph = s0 + (C::kCompact || C::kRing ? kWBox : 2 * kWBox);
    unsigned char* opl = C::kCompact ? oph + 2 * NPM * 128 : s0 + (C::kRing ? 2 : 3) * kWBox;
    if (t < 2 * NPM) {
      const bool isB = t >= NPM;
      const int n = isB ? t - NPM : t;
      if (n < N) {
#pragma unroll
        for (int c = 0; c < NPM / 8; ++c) {
          const uint32_t off = static_cast<uint32_t>(t * 128 + ((c ^ (t & 7)) << 4));
          *reinterpret_cast<uint4*>(oph + off) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(opl + off) = make_uint4(0u, 0u, 0u, 0u);
        }
        const unsigned char* gq = s0;  // Gram rows: key slot m = node m, query slot NPM + n
        auto G = [&](int m, int i) { return *reinterpret_cast<const float*>(gq + gram_off<NPM>(m, i)); };
        int pn[kWRegPath];
        float al[kWRegPath], be[kWRegPath], x[kWRegPath];
        int L = 0, cur = n;
#pragma unroll
        for (int s = 0; s < kWRegPath; ++s) {
          pn[s] = 0;
          al[s] = 0.f;
          be[s] = 0.f;
          if (cur >= 0) {
            pn[s] = cur;
            al[s] = ts.alpha[cur];
            be[s] = ts.beta[cur];
            cur = ts.par[cur];
            ++L;
          }
        }
        if (cur < 0) {
          // root path of at most kWRegPath nodes: x in registers
          float c = 1.f;
#pragma unroll
          for (int s = 0; s < kWRegPath; ++s) {
            x[s] = isB ? ((s < L) ? c * G(NPM + n, pn[s]) : 0.f) : (s == 0 ? 1.f : 0.f);
            c *= al[s];
          }
#pragma unroll
          for (int qq = 1; qq < kWRegPath; ++qq) {
            if (qq < L) {
              float rt = 1.f;  // gamma_{p_a} / gamma_{p_qq}
#pragma unroll
              for (int a = qq - 1; a >= 0; --a) {
                rt *= al[a];
                x[qq] = fmaf(-x[a] * be[a] * rt, G(pn[a], pn[qq]), x[qq]);
              }
            }
          }
#pragma unroll
          for (int s = 0; s < kWRegPath; ++s)
            if (s < L) put_op(oph, opl, t, pn[s], x[s]);
        } else {
          // longer root path: x in this thread's scratch row (the K/Q region
          // is free: every product that reads it is complete), each settled
          // x_a pushed into the later entries
          float* xs = reinterpret_cast<float*>(kqs) + t * NPM;
          float c = 1.f;
          L = 0;
          for (int cu = n; cu >= 0; cu = ts.par[cu]) {
            xs[L] = isB ? c * G(NPM + n, cu) : (L == 0 ? 1.f : 0.f);
            c *= ts.alpha[cu];
            ++L;
          }
          int pa = n;
          for (int a = 0; a + 1 < L; ++a) {
            const float ba = ts.beta[pa] * xs[a];
            float rt = 1.f;
            int node = pa;
            for (int qq = a + 1; qq < L; ++qq) {
              rt *= ts.alpha[node];
              node = ts.par[node];
              xs[qq] = fmaf(-ba * rt, G(pa, node), xs[qq]);
            }
            pa = ts.par[pa];
          }
          int node = n;
          for (int s = 0; s < L; ++s, node = ts.par[node]) put_op(oph, opl, t, node, xs[s]);
        }
      }
    }
    if (b.gamma != nullptr && t < N) b.gamma[node0 + static_cast<int64_t>(t) * H] = ts.coef[t].z;
    __syncthreads();

    // ---- MMA 2 and the stores, per pair of output tiles (16 nodes): O onto
    //      gamma S0 q, then U; input k-steps up to the pair's own (a node's
    //      ancestors have smaller indices)
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const bool isO = part == 0;
      float* dstb = (isO ? b.o : b.U) + node0 * kWDim + sr0;
#pragma unroll
      for (int jp = 0; jp < KT / 2; ++jp) {
        if (16 * jp < N) {
          float d[2][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            d[0][i] = isO ? oi[2 * jp][i] : 0.f;
            d[1][i] = isO ? oi[2 * jp + 1][i] : 0.f;
          }
          const int orow = (isO ? NPM : 0) + 16 * jp + ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
          for (int s = 0; s <= jp; ++s) {
            uint32_t bh[4], bl[4];
            const uint32_t off = sw128_off(orow, 16 * s + ((lane >> 3) & 1) * 8);
            ldsm_x4(bh, oph + off);
            ldsm_x4(bl, opl + off);
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
              mma16816_bf16_nv(d[tt], wh[s][0], wh[s][1], wh[s][2], wh[s][3], bh[2 * tt], bh[2 * tt + 1]);
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
              mma16816_bf16_nv(d[tt], wl[s][0], wl[s][1], wl[s][2], wl[s][3], bh[2 * tt], bh[2 * tt + 1]);
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
              mma16816_bf16_nv(d[tt], wh[s][0], wh[s][1], wh[s][2], wh[s][3], bl[2 * tt], bl[2 * tt + 1]);
          }
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int n = 16 * jp + 8 * tt + 2 * q + e;
              if (n < N)
                *reinterpret_cast<float2*>(dstb + static_cast<int64_t>(n) * rowstride) =
                    make_float2(d[tt][e], d[tt][2 + e]);
            }
          }
        }
      }
    }
    }  // !ring_fail
  }

  if (t == 0) {
    int bits = (fail || ring_fail) ? kStatusTimeout : 0;
    if (h == 0) bits |= flags | cflags | (issued && bad_tree ? TREEWY_STATUS_BAD_TREE : 0);
    // the previous tree failed its checks, or a wait gave up before S_a was
    // stored: that request's commit did not happen
    if (bad_prev && h == 0) bits |= TREEWY_STATUS_BAD_TREE | TREEWY_STATUS_COMMIT_REFUSED;
    if (fail && commit_now && !stored) bits |= TREEWY_STATUS_COMMIT_REFUSED;
    if (bits) atomicOr(b.status + r, bits);
    // no copy may still target this CTA's memory at exit
    if (fail) mbar_wait(&ts.bar, 0);
    if (C::kRing && ring_fail) mbar_wait(&ts.bar3, 0);
    if (stored) bulk_wait_group_read0();
  }
}

template <int NPM, bool SB, bool FUSED>
cudaError_t launch_warp(const treewy_batch& b, const CUtensorMap& map_s0, const PrevRound& prev,
                        cudaStream_t stream) {
  using C = WarpCfg<NPM, SB, FUSED>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t attr = once_per_device(attr_done, [] {
    cudaError_t e = cudaFuncSetAttribute(verify_warp_kernel<NPM, SB, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kDynSmem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(verify_warp_kernel<NPM, SB, FUSED>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
    return e;
  });
  if (attr != cudaSuccess) return attr;
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  verify_warp_kernel<NPM, SB, FUSED><<<grid, kWThreads, C::kDynSmem, stream>>>(map_s0, b, prev);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify_warp(const treewy_batch& b, const CUtensorMap& map_s0, const PrevRound* prev,
                               cudaStream_t stream) {
  static_assert(kWarpTreeNodes == 32 && kFusedWarpNodes == 16, "launched capacities");
  const bool sb = (b.flags & TREEWY_FLAG_STATE_BF16) != 0;
  if (prev == nullptr) {
    const PrevRound none{};
    if (b.max_nodes > 16)
      return sb ? launch_warp<32, true, false>(b, map_s0, none, stream)
                : launch_warp<32, false, false>(b, map_s0, none, stream);
    return sb ? launch_warp<16, true, false>(b, map_s0, none, stream)
              : launch_warp<16, false, false>(b, map_s0, none, stream);
  }
  // the fused 32-node form is launched for a bf16 pool only (an fp32 pool's
  // runs on the tcgen05 kernel)
  if (b.max_nodes > 16)
    return sb ? launch_warp<32, true, true>(b, map_s0, *prev, stream) : cudaErrorInvalidValue;
  return sb ? launch_warp<16, true, true>(b, map_s0, *prev, stream)
            : launch_warp<16, false, true>(b, map_s0, *prev, stream);
}

}  // namespace treewy
