// verify_tc.cu -- TreeWY verification on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators, TMA staging) for dk = dv = 128, bf16 q/k/v,
// fp32 committed state.
//
// One CTA (128 threads, one per value row d = TMEM lane) per (request, head):
//
//  TMA     S0 (64 KB fp32, 4 boxes of 128 rows x 32 columns, 128B swizzle) and
//          the K and Q rows of the tree (bf16, 8-row boxes) into shared memory.
//  convert each thread turns its own 128-byte S0 row segment in place into
//          [hi | lo] bf16 halves, S0 ~= hi + lo (16 significant bits), so the
//          fp32 state goes through bf16 MMAs without tf32-level rounding.
//  MMA     D1 = S0 [K;Q]^T  (M = dv = 128, N = 2*Np, K = dk = 128; hi and lo
//          accumulate into the same fp32 TMEM columns): column n holds
//          S0 k_n, column Np + n holds S0 q_n  (TreeWY paper §3 Eq. (2) R term,
//          review §3.2 Algorithm step 3 and the read-out of step 5);
//          D2 = [K;Q] K^T  (M = 128, N = Np): the Gram rows k_m.k_i, q_m.k_i
//          (Eq. (2) G, review Algorithm step 2).
//  solve   thread d: W = beta (v - gamma S0 k), forward substitution over the
//          ancestor lists, read-out o_n (review Eq. (5) restricted to
//          ancestors), coalesced stores of o and U.
//
// Nothing per node is kept beyond U (N x dv), the object that replaces the
// per-node snapshots (paper §3 "Reconstruct on commit").
#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

constexpr int kThreads = 128;
constexpr int kDim = 128;
constexpr uint32_t kS0ChunkBytes = 128u * 128u;          // 128 rows x 32 fp32
constexpr uint32_t kS0Bytes = 4u * kS0ChunkBytes;        // 64 KB
constexpr uint32_t kKQChunkBytes = 128u * 128u;          // 128 rows x 64 bf16
constexpr uint32_t kKQBytes = 2u * kKQChunkBytes;        // 32 KB
constexpr uint32_t kDynSmem = kS0Bytes + kKQBytes + 1024u;  // + alignment slack

template <int NPM>
struct TcCfg {
  static constexpr uint32_t kCols = (3 * NPM <= 64) ? 64u : (3 * NPM <= 128 ? 128u : 256u);
  static constexpr int kGramPitch = NPM + 1;
  static constexpr int kE = max_anc_entries(NPM);
  static constexpr uint32_t kGramBytes = 128u * kGramPitch * 4u;
  static constexpr uint32_t kIdxOff = kGramBytes;
  static constexpr uint32_t kCoefAOff = kIdxOff + ((kE + 15u) & ~15u);
  static constexpr uint32_t kCoefMOff = kCoefAOff + 4u * kE;
  static constexpr uint32_t kQksOff = kCoefMOff + 4u * kE;
  static_assert(kQksOff + 4u * NPM <= kS0Bytes, "post-MMA scratch must fit the S0 region");
  static_assert(NPM * kDim * 4u <= kKQBytes, "U staging must fit the K/Q region");
};

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
  for (int j = 0; j < 16; ++j) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(f[2 * j]);
    const __nv_bfloat16 h1 = __float2bfloat16_rn(f[2 * j + 1]);
    const __nv_bfloat16 l0 = __float2bfloat16_rn(f[2 * j] - __bfloat162float(h0));
    const __nv_bfloat16 l1 = __float2bfloat16_rn(f[2 * j + 1] - __bfloat162float(h1));
    hi[j] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
            (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
    lo[j] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
            (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
  }
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint32_t* src = (g < 4) ? (hi + 4 * g) : (lo + 4 * (g - 4));
    *reinterpret_cast<uint4*>(row + ((g ^ sw) << 4)) = make_uint4(src[0], src[1], src[2], src[3]);
  }
}

template <int NPM>
__global__ void __launch_bounds__(kThreads)
    verify_tc_kernel(const __grid_constant__ CUtensorMap map_s0,
                     const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_q, const treewy_batch b) {
  using C = TcCfg<NPM>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ TreeSmem ts;
  __shared__ __align__(8) uint64_t bars[6];  // 0-3: S0 chunks, 4: K/Q, 5: MMA done
  __shared__ uint32_t tmem_holder;
  __shared__ int s_fail;

  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
  unsigned char* s0 = base;
  unsigned char* kq = base + kS0Bytes;

  const int H = b.H;
  const int r = blockIdx.x / H;
  const int h = blockIdx.x - r * H;
  const int t = threadIdx.x;
  const int warp = t >> 5;
  bool mma_issued = false;

  if (t == 0) {
#pragma unroll
    for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
    fence_mbarrier_init();
    s_fail = 0;
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
    if (flags == 0 && N > 0) {
      const int y = (slot * H + h) * kDim;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        mbar_arrive_expect_tx(&bars[c], kS0ChunkBytes);
        tma_load_2d(s0 + c * kS0ChunkBytes, &map_s0, &bars[c], 32 * c, y);
      }
      const int N8 = (N + 7) & ~7;
      const int Np = (N + 15) & ~15;
      // 2 tensors x 2 column chunks x N8 rows x 128 bytes
      mbar_arrive_expect_tx(&bars[4], static_cast<uint32_t>(N8) * 512u);
      for (int c2 = 0; c2 < 2; ++c2) {
        unsigned char* chunk = kq + c2 * kKQChunkBytes;
        for (int rb = 0; rb < N8; rb += 8) {
          tma_load_3d(chunk + rb * 128, &map_k, &bars[4], 64 * c2, h, lo + rb);
          tma_load_3d(chunk + (Np + rb) * 128, &map_q, &bars[4], 64 * c2, h, lo + rb);
        }
      }
    }
  }
  if (warp == 0) {
    tmem_alloc(&tmem_holder, C::kCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_holder;
  const int N = ts.N;
  const bool issued = (ts.flags == 0 && N > 0);
  const int64_t tok0 = ts.tok0;

  // Prefetch this thread's column of V (one bf16 per node) into registers;
  // consumed after the MMA.
  uint32_t vpk[NPM / 2];
  {
    const unsigned short* vg = reinterpret_cast<const unsigned short*>(b.v);
#pragma unroll
    for (int i = 0; i < NPM / 2; ++i) {
      uint32_t v0 = 0, v1 = 0;
      if (issued && 2 * i < N) v0 = __ldg(vg + ((tok0 + 2 * i) * H + h) * kDim + t);
      if (issued && 2 * i + 1 < N) v1 = __ldg(vg + ((tok0 + 2 * i + 1) * H + h) * kDim + t);
      vpk[i] = v0 | (v1 << 16);
    }
  }

  bool bad_tree = false;
  if (issued) bad_tree = !tree_prepare(ts, b.parent, b.alpha, b.beta, H, h);

  // S0 chunks -> [hi | lo] bf16, each thread converting its own row d = t.
  int fail = 0;
  if (issued) {
    for (int c = 0; c < 4; ++c) {
      if (!mbar_wait(&bars[c], 0)) {
        fail = 1;
        break;
      }
      if (!bad_tree) convert_row_hilo(s0 + c * kS0ChunkBytes + t * 128, t & 7);
    }
    fence_proxy_async_smem();
  }
  fail = __syncthreads_or(fail);

  const int Np = (N + 15) & ~15;
  if (issued && !bad_tree && !fail && t == 0) {
    if (!mbar_wait(&bars[4], 0)) {
      s_fail = 1;
    } else {
      tc_fence_after_sync();
      const uint32_t a0 = smem_addr(s0);
      const uint32_t b0 = smem_addr(kq);
      const uint32_t id1 = idesc_bf16_f32(128, 2 * Np);
      const uint32_t id2 = idesc_bf16_f32(128, Np);
      // D1 = S0 [K;Q]^T over dk in 8 steps of 16, hi then lo part of S0.
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const uint64_t bd = smem_desc_sw128(b0 + (c >> 1) * kKQChunkBytes + (c & 1) * 64 + s * 32, 1024);
          const uint64_t ahi = smem_desc_sw128(a0 + c * kS0ChunkBytes + s * 32, 1024);
          const uint64_t alo = smem_desc_sw128(a0 + c * kS0ChunkBytes + 64 + s * 32, 1024);
          mma_bf16(tmem, ahi, bd, id1, (c | s) ? 1u : 0u);
          mma_bf16(tmem, alo, bd, id1, 1u);
        }
      }
      // D2 = [K;Q] K^T (rows past 2*Np are don't-care lanes).
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t dsc = smem_desc_sw128(b0 + (s >> 2) * kKQChunkBytes + (s & 3) * 32, 1024);
        mma_bf16(tmem + 2 * NPM, dsc, dsc, id2, s ? 1u : 0u);
      }
      mma_commit(&bars[5]);
      mma_issued = true;
    }
  }
  __syncthreads();
  fail |= s_fail;
  if (issued && !bad_tree && !fail) {
    if (!mbar_wait(&bars[5], 0)) fail = 1;
  }
  fail = __syncthreads_or(fail);

  if (issued && !bad_tree && !fail) {
    tc_fence_after_sync();
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float* gram = reinterpret_cast<float*>(s0);
    uint8_t* idx = s0 + C::kIdxOff;
    float* coefA = reinterpret_cast<float*>(s0 + C::kCoefAOff);
    float* coefM = reinterpret_cast<float*>(s0 + C::kCoefMOff);
    float* qks = reinterpret_cast<float*>(s0 + C::kQksOff);
    float* Us = reinterpret_cast<float*>(kq);

    // Gram row of this lane: k_t.k_i (t < Np) or q_{t-Np}.k_i (t >= Np).
    for (int c = 0; c < Np / 16; ++c) {
      float g[16];
      tmem_ld16(tmem + lane_base + 2 * NPM + 16 * c, g);
#pragma unroll
      for (int j = 0; j < 16; ++j) gram[t * C::kGramPitch + 16 * c + j] = g[j];
    }
    // ancestor-masked coefficients from the thread's own Gram row
    if (t < N) {
      const int n = t;
      const float bn = ts.beta[n];
      for_each_ancestor(ts, n, [&](int j, int i, float c) {
        const int e = ts.aoff[n] + j;
        idx[e] = static_cast<uint8_t>(i);
        coefA[e] = bn * c * gram[t * C::kGramPitch + i];
      });
    }
    if (t >= Np && t < Np + N) {
      const int n = t - Np;
      for_each_ancestor(ts, n, [&](int j, int i, float c) {
        coefM[ts.aoff[n] + j] = c * gram[t * C::kGramPitch + i];
      });
      qks[n] = gram[t * C::kGramPitch + n];
    }
    // W[n][d] = beta_n (v_n[d] - gamma_n (S0 k_n)[d])
#pragma unroll
    for (int c = 0; c < NPM / 16; ++c) {
      if (16 * c < N) {
        float p[16];
        tmem_ld16(tmem + lane_base + 16 * c, p);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = 16 * c + j;
          if (n < N) {
            const uint32_t pair = vpk[n >> 1];
            const float vv = bf16_bits_to_float(static_cast<uint16_t>((n & 1) ? (pair >> 16) : pair));
            Us[n * kDim + t] = ts.beta[n] * (vv - ts.gamma[n] * p[j]);
          }
        }
      }
    }
    __syncthreads();

    solve_inplace(ts, Us, kDim, t, idx, coefA);
#pragma unroll
    for (int c = 0; c < NPM / 16; ++c) {
      if (16 * c < N) {
        float pq[16];
        tmem_ld16(tmem + lane_base + Np + 16 * c, pq);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = 16 * c + j;
          if (n < N) {
            const float o = readout_node(ts, n, pq[j], Us, kDim, t, idx, coefM, qks);
            b.o[((tok0 + n) * H + h) * kDim + t] = o;
          }
        }
      }
    }
    for (int n = 0; n < N; ++n) b.U[((tok0 + n) * H + h) * kDim + t] = Us[n * kDim + t];
    if (b.gamma != nullptr && t < N) b.gamma[(tok0 + t) * H + h] = ts.gamma[t];
  }

  if (t == 0) {
    int bits = (fail ? kStatusTimeout : 0);
    if (h == 0) bits |= ts.flags | (bad_tree ? TREEWY_STATUS_BAD_TREE : 0);
    if (bits) atomicOr(b.status + r, bits);
    if (issued) {
      // No async copy or MMA may still target this CTA's memory at exit.
      for (int i = 0; i < 5; ++i) mbar_wait(&bars[i], 0);
      if (mma_issued) mbar_wait(&bars[5], 0);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kCols);
  }
}

template <int NPM>
cudaError_t launch_npm(const treewy_batch& b, const VerifyMaps& m, cudaStream_t stream) {
  static cudaError_t attr = cudaFuncSetAttribute(
      verify_tc_kernel<NPM>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kDynSmem));
  if (attr != cudaSuccess) return attr;
  const unsigned grid = static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H);
  verify_tc_kernel<NPM><<<grid, kThreads, kDynSmem, stream>>>(m.s0, m.k, m.q, b);
  return cudaGetLastError();
}

}  // namespace

size_t verify_tc_smem(int) { return kDynSmem; }

cudaError_t launch_verify_tc(const treewy_batch& b, const VerifyMaps& maps, int npm,
                             cudaStream_t stream) {
  if (npm <= 16) return launch_npm<16>(b, maps, stream);
  if (npm <= 32) return launch_npm<32>(b, maps, stream);
  return launch_npm<64>(b, maps, stream);
}

}  // namespace treewy
