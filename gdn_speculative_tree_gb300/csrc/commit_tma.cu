// commit_tma.cu -- reconstruct-on-commit for dk = dv = 128 with the state
// tile moved by TMA (TreeWY paper §3 "Reconstruct on commit", Eq. (3);
// technical review §3.3, Eq. (6)):
//
//   S_a = gamma_a S0 + sum_{i on the root-to-a path} (gamma_a / gamma_i) u_i k_i^T.
//
// One CTA of 128 threads owns a 32 KB tile of one (request, head): half of
// an f32 state (64 rows, two CTAs per head) or all of a bf16 state (128
// rows).  The tile is requested by bulk tensor loads as soon as the request's
// slot is known, lands in shared memory in the 128-byte-swizzled layout, is
// updated there row by row while the path's u and k rows are staged, and
// leaves by bulk tensor stores.  Nothing of the state passes through
// registers while in flight, and six CTAs per SM (192 KB of tiles) keep
// enough independent load chains in flight to stream HBM.
#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

constexpr int kThreads = 128;
constexpr int kSeg = 8;                             // path nodes staged per pass
constexpr uint32_t kTileBytes = 32768u;

// Tile geometry: f32 state -> 64 rows x 4 chunks of 32 columns (8 KB each),
// two CTAs per head; bf16 state -> 128 rows x 2 chunks of 64 columns (16 KB).
template <bool SB>
struct CommitCfg {
  static constexpr int kRows = SB ? 128 : 64;
  static constexpr int kChunks = SB ? 2 : 4;
  static constexpr int kChunkCols = SB ? 64 : 32;
  static constexpr uint32_t kChunkBytes = kRows * 128u;
  static constexpr int kSplit = 128 / kRows;        // CTAs per head
  static constexpr int kBlocksPerThread = 4 * kRows / kThreads;  // 32-column blocks
};

struct CommitSmem {
  int8_t parent[kMaxNodes];
  float alpha[kMaxNodes];
  float c[kMaxNodes];                 // gamma_a / gamma_{path j} (alpha products)
  uint8_t path[kMaxNodes];            // a, parent(a), ..., root
  float k[kSeg][128];                 // staged k rows of one pass
  int tok0, N, slot, a, flags, len;
  float gamma_a;
};

// Columns 32 blk .. 32 blk + 31 of tile row d, as f32.
template <bool SB>
__device__ __forceinline__ void load_block(const unsigned char* tile, int d, int blk, float (&x)[32]) {
  constexpr uint32_t kChunkBytes = CommitCfg<SB>::kChunkBytes;
  if constexpr (SB) {
    const unsigned char* row = tile + (blk >> 1) * kChunkBytes + d * 128;
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4) {
      const int g = 4 * (blk & 1) + g4;
      const uint4 raw = *reinterpret_cast<const uint4*>(row + ((g ^ (d & 7)) << 4));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * g4 + 2 * i] = __uint_as_float(w[i] << 16);
        x[8 * g4 + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  } else {
    const unsigned char* row = tile + blk * kChunkBytes + d * 128;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float4 v = *reinterpret_cast<const float4*>(row + ((g ^ (d & 7)) << 4));
      x[4 * g] = v.x;
      x[4 * g + 1] = v.y;
      x[4 * g + 2] = v.z;
      x[4 * g + 3] = v.w;
    }
  }
}

template <bool SB>
__device__ __forceinline__ void store_block(unsigned char* tile, int d, int blk, const float (&x)[32]) {
  constexpr uint32_t kChunkBytes = CommitCfg<SB>::kChunkBytes;
  if constexpr (SB) {
    unsigned char* row = tile + (blk >> 1) * kChunkBytes + d * 128;
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4) {
      const int g = 4 * (blk & 1) + g4;
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(x[8 * g4 + 2 * i], x[8 * g4 + 2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&p);
      }
      *reinterpret_cast<uint4*>(row + ((g ^ (d & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    unsigned char* row = tile + blk * kChunkBytes + d * 128;
#pragma unroll
    for (int g = 0; g < 8; ++g)
      *reinterpret_cast<float4*>(row + ((g ^ (d & 7)) << 4)) =
          make_float4(x[4 * g], x[4 * g + 1], x[4 * g + 2], x[4 * g + 3]);
  }
}

template <bool SB>
__global__ void __launch_bounds__(kThreads)
    commit_tma_kernel(const __grid_constant__ CUtensorMap map_s, const treewy_batch b,
                      const int32_t* __restrict__ accepted, int refused_bit) {
  using C = CommitCfg<SB>;
  __shared__ __align__(1024) unsigned char tile[kTileBytes];
  __shared__ CommitSmem cs;
  __shared__ __align__(8) uint64_t bar;

  const int H = b.H;
  const int head = blockIdx.x / C::kSplit;
  const int part = blockIdx.x - head * C::kSplit;   // which rows of the head
  const int r = head / H;
  const int h = head - r * H;
  const int t = threadIdx.x;
  const int dl = t % C::kRows;                       // tile row of this thread
  const int d = part * C::kRows + dl;                // state row (value index)
  const int blk0 = (t / C::kRows) * C::kBlocksPerThread;
  const bool kbf16 = b.qkv_dtype == TREEWY_DTYPE_BF16;
  const bool lead = (h == 0 && part == 0);           // reports request-level flags

  // Every thread reads the request's metadata itself (one round trip), so
  // that threads < N request their node's parent and gate straight after it
  // rather than after thread 0 has published it; the loads stay inside the
  // batch and are used only when thread 0's checks pass.
  const int a_s = __ldg(accepted + r);
  const int lo_s = __ldg(b.node_offset + r), hi_s = __ldg(b.node_offset + r + 1);
  const int slot_s = __ldg(b.state_slot + r);
  const int n_s = hi_s - lo_s;
  const bool range_ok =
      a_s >= 0 && n_s > 0 && n_s <= b.max_nodes && lo_s >= 0 && static_cast<int64_t>(hi_s) <= b.T;
  int node_p = -1;
  float node_alpha = 0.f;
  if (range_ok && t < n_s) {
    node_p = __ldg(b.parent + lo_s + t);
    node_alpha = __ldg(b.alpha + (static_cast<int64_t>(lo_s) + t) * H + h);
  }

  if (t == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    const int a = a_s;
    const int lo = lo_s, hi = hi_s;
    const int slot = slot_s;
    const int N = hi - lo;
    int flags = 0;
    if (a != -1) {
      if (N < 0 || N > b.max_nodes) flags |= TREEWY_STATUS_TOO_MANY_NODES;
      else if (lo < 0 || static_cast<int64_t>(hi) > b.T) flags |= TREEWY_STATUS_BAD_TREE;
      if (a < -1 || a >= N) flags |= TREEWY_STATUS_BAD_ACCEPTED;
      if (slot < 0 || static_cast<int64_t>(slot) >= b.num_slots) flags |= TREEWY_STATUS_BAD_SLOT;
    }
    cs.tok0 = lo;
    cs.N = N;
    cs.slot = slot;
    cs.flags = flags;
    cs.a = flags ? -1 : a;
    if (a != -1 && flags == 0) {
      const int y = (slot * H + h) * 128 + part * C::kRows;
      mbar_arrive_expect_tx(&bar, kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_2d(tile + c * C::kChunkBytes, &map_s, &bar, C::kChunkCols * c, y);
    }
  }
  __syncthreads();
  const int a = cs.a;
  if (a < 0) {
    // nothing accepted (state neither read nor written) or a bad request
    if (t == 0 && lead && cs.flags) atomicOr(b.status + r, cs.flags | refused_bit);
    return;
  }
  const int64_t tok0 = cs.tok0;
  const int N = cs.N;

  // the whole tree is validated (U of an invalid tree was never written)
  bool bad = false;
  if (t < N) {
    bad = !(node_p >= -1 && node_p < t);
    cs.parent[t] = static_cast<int8_t>(bad ? -1 : node_p);
    cs.alpha[t] = node_alpha;
  }
  bad = __syncthreads_or(bad);
  if (!bad && t == 0) {
    int len = 0;
    float c = 1.0f;
    for (int cur = a; cur >= 0; cur = cs.parent[cur]) {
      cs.path[len] = static_cast<uint8_t>(cur);
      cs.c[len] = c;
      c *= cs.alpha[cur];
      ++len;
    }
    cs.len = len;
    cs.gamma_a = c;
  }
  __syncthreads();

  // stage pass `s`: k rows in shared memory, c_j u_j[d] in registers.  Every
  // load is issued before any result is used (a shared-memory store of a
  // loaded value would hold back the loads behind it by a round trip).
  float cu[kSeg];
  auto stage = [&](int s) {
    const int ns = min(kSeg, cs.len - s * kSeg);
    float kv[kSeg];                     // element x = t of path node j
#pragma unroll
    for (int j = 0; j < kSeg; ++j) {
      kv[j] = 0.f;
      cu[j] = 0.f;
      if (j < ns) {
        const int64_t row = (tok0 + cs.path[s * kSeg + j]) * H + h;
        kv[j] = load_qkv(b.k, row * 128 + t, kbf16);
        cu[j] = __ldg(b.U + row * 128 + d);
      }
    }
#pragma unroll
    for (int j = 0; j < kSeg; ++j) {
      if (j < ns) {
        cs.k[j][t] = kv[j];
        cu[j] *= cs.c[s * kSeg + j];
      }
    }
  };
  if (!bad) stage(0);

  int fail = 0;
  if (t == 0) fail = !mbar_wait(&bar, 0);
  fail = __syncthreads_or(fail);
  if (bad || fail) {
    if (t == 0) {
      if (fail) mbar_wait(&bar, 0);  // nothing may still target this CTA's memory
      int bits = (fail ? kStatusTimeout : 0) | ((bad && lead) ? TREEWY_STATUS_BAD_TREE : 0);
      if (bits) bits |= refused_bit;
      if (bits) atomicOr(b.status + r, bits);
    }
    return;
  }

  // tile row dl, 32 columns at a time, f32 across every pass, stored once
  const int len = cs.len;
  const int nseg = (len + kSeg - 1) / kSeg;
  const float ga = cs.gamma_a;
  int staged = 0;
  for (int blk = blk0; blk < blk0 + C::kBlocksPerThread; ++blk) {
    float x[32];
    load_block<SB>(tile, dl, blk, x);
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] *= ga;
    for (int s = 0; s < nseg; ++s) {
      if (s != staged) {
        __syncthreads();
        stage(s);
        __syncthreads();
        staged = s;
      }
      const int ns = min(kSeg, len - s * kSeg);
#pragma unroll
      for (int j = 0; j < kSeg; ++j) {
        if (j < ns) {
          const float u = cu[j];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 kk = *reinterpret_cast<const float4*>(&cs.k[j][32 * blk + e]);
            x[e] = fmaf(u, kk.x, x[e]);
            x[e + 1] = fmaf(u, kk.y, x[e + 1]);
            x[e + 2] = fmaf(u, kk.z, x[e + 2]);
            x[e + 3] = fmaf(u, kk.w, x[e + 3]);
          }
        }
      }
    }
    store_block<SB>(tile, dl, blk, x);
  }

  // S_a back to the pool; the tile must stay until the stores have read it
  fence_proxy_async_smem();
  __syncthreads();
  if (t == 0) {
    const int y = (cs.slot * H + h) * 128 + part * C::kRows;
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c)
      tma_store_2d(&map_s, tile + c * C::kChunkBytes, C::kChunkCols * c, y);
    bulk_commit_group();
    bulk_wait_group_read0();
  }
}

template <bool SB>
cudaError_t launch(const treewy_batch& b, const CUtensorMap& map, const int32_t* accepted,
                   int refused_bit, cudaStream_t stream) {
  // the whole unified L1/shared array as shared memory: six 38 KB CTAs per SM
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t attr = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(commit_tma_kernel<SB>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                static_cast<int>(cudaSharedmemCarveoutMaxShared));
  });
  if (attr != cudaSuccess) return attr;
  const unsigned grid =
      static_cast<unsigned>(b.R) * static_cast<unsigned>(b.H) * CommitCfg<SB>::kSplit;
  commit_tma_kernel<SB><<<grid, kThreads, 0, stream>>>(map, b, accepted, refused_bit);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_commit_tma(const treewy_batch& b, const CUtensorMap& state_map,
                              const int32_t* accepted, int refused_bit, cudaStream_t stream) {
  if (b.flags & TREEWY_FLAG_STATE_BF16) return launch<true>(b, state_map, accepted, refused_bit, stream);
  return launch<false>(b, state_map, accepted, refused_bit, stream);
}

}  // namespace treewy
