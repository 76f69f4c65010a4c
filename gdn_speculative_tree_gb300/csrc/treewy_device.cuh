// treewy_device.cuh -- device-side helpers shared by the TreeWY kernels:
// inline-PTX wrappers for mbarrier, TMA and tcgen05 (sm_103a), bounded waits,
// and the per-(request, head) draft-tree preparation (decays, ancestor lists).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "treewy.h"

namespace treewy {

constexpr int kMaxNodes = TREEWY_MAX_NODES;
// Status bits beyond the public ones: an internal wait gave up (outputs of
// that request/head were not written).  Public in treewy.h as well.
constexpr int kStatusTimeout = 16;
constexpr int kStatusBadSlot = 8;
// Longest a kernel waits on an mbarrier before it gives up (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ---------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two-term bf16 split of two fp32 values: hi = rn(x), lo = rn(x - hi), each
// pair packed as bf16x2 (first value in the low half).  hi + lo carries 16
// significant bits, so products on the bf16 tensor cores keep near-fp32
// accuracy.
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Load element i of a q/k/v row (or of a state block) as float (bf16 or fp32 storage).
__device__ __forceinline__ float load_qkv(const void* base, int64_t idx, bool is_bf16) {
  if (is_bf16) {
    return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(base) + idx));
  }
  return __ldg(reinterpret_cast<const float*>(base) + idx);
}

// Barrier among NTHREADS threads (whole warps) on hardware barrier ID (0 is
// __syncthreads); returns the OR of `pred` over those threads.
template <int ID, int NTHREADS>
__device__ __forceinline__ bool named_bar_or(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "n"(ID), "n"(NTHREADS)
      : "memory");
  return out != 0;
}

template <int ID, int NTHREADS>
__device__ __forceinline__ void named_bar_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(NTHREADS) : "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete; false after
// limit_ns without completion (the caller records a timeout and skips).
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 31u) {
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        return false;
      }
    }
  }
}

// The kernels' wait: gives up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Tile store shared -> global through the same tensor map (swizzle undone on
// the way out); completion is tracked per issuing thread by bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store of this thread has finished reading
// its shared-memory source (the writes to global memory may still be in flight).
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until all but the most recently committed bulk group of this thread
// have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(holder)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc)^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread
// have completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// D += A B for one m16n8k16 warp-level tile, bf16 x bf16 -> fp32: the
// register-operand tensor path, for products too small to pay for tcgen05's
// TMEM round trip.  Fragments (g = lane / 4, q = lane % 4): a0 row g, k 2q,
// 2q+1; a1 row g+8; a2 row g, k 2q+8, 2q+9; a3 row g+8, those k; b0 column g,
// k 2q, 2q+1; b1 k 2q+8, 2q+9; d[0..1] row g, columns 2q, 2q+1; d[2..3] row
// g+8.
__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA without `volatile`: the compiler may interleave independent
// products with the loads around them.
__device__ __forceinline__ void mma16816_bf16_nv(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                 uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8 x 8 b16 matrices from shared memory (ldmatrix): lanes 8i .. 8i+7
// give the row addresses of matrix i (16-byte aligned), and lane (g, q) =
// (lane / 4, lane % 4) receives elements 2q, 2q+1 of row g of matrix i in
// r[i]: the B fragments of a warp MMA for two n8-tiles when the matrices are
// (tile 0, k 0-7), (tile 0, k 8-15), (tile 1, k 0-7), (tile 1, k 8-15).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

// Byte of entry (row o, column i) of a K-major bf16 operand with 128-byte
// rows and 128-byte swizzle (16-byte chunk i / 8 of row o at position
// (i / 8) XOR (o mod 8)), which ldmatrix reads without bank conflicts (eight
// rows of one chunk column).
__device__ __forceinline__ uint32_t sw128_off(int o, int i) {
  return static_cast<uint32_t>(o * 128 + ((((i >> 3) ^ (o & 7))) << 4) + ((i & 7) << 1));
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.  The hardware
// writes the target registers asynchronously, until tcgen05.wait::ld; the
// compiler sees them as written here, so the matching wait (tmem_wait16 /
// tmem_wait8 on the same arrays) must follow with no other code in between.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Eight consecutive 32-bit TMEM columns of this thread's lane (same rule).
__device__ __forceinline__ void tmem_ld8_async(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_wait8(uint32_t (&a)[8], uint32_t (&b)[8], uint32_t (&c)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]),
                 "+r"(a[7]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]),
                 "+r"(b[6]), "+r"(b[7]), "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3]), "+r"(c[4]),
                 "+r"(c[5]), "+r"(c[6]), "+r"(c[7])
               :
               : "memory");
}

// Wait for all of this thread's outstanding TMEM loads; the register array is
// passed through so no use of it is scheduled before the wait.
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand with a
// 128-byte swizzle, rows 128 bytes apart, 8-row groups `sbo` bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);        // start address
  d |= static_cast<uint64_t>(1u) << 16;                       // leading byte offset (unused)
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;     // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                       // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                       // swizzle: 128B
  return d;
}

// Instruction descriptor: kind::f16, A and B bf16 K-major, D fp32, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
  return (1u << 4)             // D format: f32
         | (1u << 7)           // A format: bf16
         | (1u << 10)          // B format: bf16
         | ((N >> 3) << 17)    // N / 8
         | ((M >> 4) << 24);   // M / 16
}

// ---------------------------------------------------------------- tree prep

// Per-CTA draft-tree data in shared memory for one (request, head).
struct TreeSmem {
  int parent[kMaxNodes];
  float alpha[kMaxNodes];
  float beta[kMaxNodes];
  float gamma[kMaxNodes];
  int nanc[kMaxNodes];        // number of strict ancestors
  int aoff[kMaxNodes + 1];    // CSR offsets of the strict-ancestor lists
  int tok0, N, slot, flags;   // broadcast request data
};

// Maximum number of strict-ancestor entries of a tree with n nodes.
__host__ __device__ constexpr int max_anc_entries(int n) { return n * (n - 1) / 2; }

// Load parents and gates of nodes 0..N-1 of this request/head, validate the
// parents (every parent in [-1, n)), and form the path decays
// gamma_n = prod of alpha over root..n (the review's Algorithm step 1) and
// the strict-ancestor counts.  Must be called by all threads; returns false
// (uniformly) when the tree is invalid.  Requires blockDim.x >= 64.
__device__ __forceinline__ bool tree_prepare(TreeSmem& ts, const int32_t* __restrict__ parent_g,
                                             const float* __restrict__ alpha_g,
                                             const float* __restrict__ beta_g, int H, int h) {
  const int t = threadIdx.x;
  const int N = ts.N;
  bool bad = false;
  if (t < N) {
    const int64_t row = static_cast<int64_t>(ts.tok0) + t;
    const int p = __ldg(parent_g + row);
    bad = !(p >= -1 && p < t);
    ts.parent[t] = bad ? -1 : p;
    ts.alpha[t] = __ldg(alpha_g + row * H + h);
    ts.beta[t] = __ldg(beta_g + row * H + h);
  }
  if (__syncthreads_or(bad)) return false;
  if (t < N) {
    // walk towards the root: gamma_t = alpha_t * alpha_p * ...
    float g = ts.alpha[t];
    int cnt = 0;
    int p = ts.parent[t];
    while (p >= 0) {
      g *= ts.alpha[p];
      ++cnt;
      p = ts.parent[p];
    }
    ts.gamma[t] = g;
    ts.nanc[t] = cnt;
  }
  __syncthreads();
  if (t < 32) {
    // exclusive scan of nanc over up to 64 nodes, two per lane
    const int i0 = 2 * t, i1 = 2 * t + 1;
    const int a0 = i0 < N ? ts.nanc[i0] : 0;
    const int a1 = i1 < N ? ts.nanc[i1] : 0;
    int s = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (t >= o) s += y;
    }
    const int excl = s - a0 - a1;
    ts.aoff[i0] = excl;
    ts.aoff[i1] = excl + a0;
    if (t == 31) ts.aoff[kMaxNodes] = s;
  }
  __syncthreads();
  return true;
}

// Walk node n's strict ancestors, nearest first, calling f(j, i, c) for the
// j-th ancestor i with decay ratio c = gamma_n / gamma_i formed as the
// product of alpha over the path segment (i, n] (no division).
template <typename F>
__device__ __forceinline__ void for_each_ancestor(const TreeSmem& ts, int n, F&& f) {
  float c = 1.0f;
  int cur = n;
  int j = 0;
  int p = ts.parent[n];
  while (p >= 0) {
    c *= ts.alpha[cur];
    f(j, p, c);
    ++j;
    cur = p;
    p = ts.parent[p];
  }
}

// Column-parallel forward substitution of (I + A) U = W for the thread's
// column d (one unit-lower-triangular solve, TreeWY paper §3 Eq. (2)): Us
// holds W on entry (row pitch `pitch` floats) and U on exit.  Row n only
// subtracts its strict ancestors' rows, A[n, idx[e]] = coefA[e].
__device__ __forceinline__ void solve_inplace(const TreeSmem& ts, float* Us, int pitch, int d,
                                              const uint8_t* idx, const float* coefA) {
  const int N = ts.N;
  for (int n = 0; n < N; ++n) {
    float acc = Us[n * pitch + d];
    const int e0 = ts.aoff[n], e1 = ts.aoff[n + 1];
    for (int e = e0; e < e1; ++e) acc = fmaf(-coefA[e], Us[idx[e] * pitch + d], acc);
    Us[n * pitch + d] = acc;
  }
}

// Output of node n in column d (review §3.1 Eq. (5) restricted to ancestors):
// o_n = gamma_n (S0 q_n) + (k_n.q_n) u_n + sum_{strict ancestors i} M[n,i] u_i.
__device__ __forceinline__ float readout_node(const TreeSmem& ts, int n, float s0q,
                                              const float* Us, int pitch, int d,
                                              const uint8_t* idx, const float* coefM,
                                              const float* qk_self) {
  float acc = ts.gamma[n] * s0q;
  acc = fmaf(qk_self[n], Us[n * pitch + d], acc);
  const int e0 = ts.aoff[n], e1 = ts.aoff[n + 1];
  for (int e = e0; e < e1; ++e) acc = fmaf(coefM[e], Us[idx[e] * pitch + d], acc);
  return acc;
}

}  // namespace treewy
