// Device helpers for the verification kernels (sm_103a).
//
// Nothing here is shared with the CPU oracle; the Philox block function below
// is written from its published definition (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11).
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

namespace sv {

constexpr int kThreads = 256;          // threads per CTA of every kernel
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------- Philox ---
// Ten rounds of Philox4x32: counter words 0 and 2 are multiplied by two fixed
// odd constants; the high halves are xored with the other counter words and
// the key; the key takes a Weyl increment between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 key) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      key.x += 0x9E3779B9u;
      key.y += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ key.x, lo1, hi0 ^ c.w ^ key.y, lo0);
  }
  return c;
}

__device__ __forceinline__ uint2 philox_key(uint64_t seed) {
  return make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
}

// U(w) = ((w >> 9) + 0.5) * 2^-23: every step is exact in fp32.
__device__ __forceinline__ float uniform_of(uint32_t w) {
  return ((float)(w >> 9) + 0.5f) * 0x1p-23f;
}

// Standard Gumbel noise from a uniform, with the accurate logf (the inner
// logarithm of a uniform near 1 must keep its relative accuracy).
__device__ __forceinline__ float gumbel_of(float u) { return -logf(-logf(u)); }

// Uniform deciding draft position i of sequence b.
__device__ __forceinline__ float accept_uniform(uint2 key, uint32_t b, int i) {
  return uniform_of(philox4x32_10(make_uint4(0u, (uint32_t)i, b, 0u), key).x);
}

// The four Gumbel uniforms of ids 4g .. 4g+3 on row j of sequence b.
__device__ __forceinline__ uint4 gumbel_words(uint2 key, uint32_t b, int j, uint32_t g) {
  return philox4x32_10(make_uint4(g, (uint32_t)j, b, 1u), key);
}

// ------------------------------------------------------------ arithmetic ---
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that returns NaN if either operand is NaN.
__device__ __forceinline__ float nanmax(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Packed bf16x2 max that propagates NaN.
__device__ __forceinline__ uint32_t bf16x2_nanmax(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Packed bf16x2 min (operands are never NaN where it is used).
__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16 -> fp32 is exact: the 16 bits become the top half of the fp32 word.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_at(const uint16_t* p, size_t i) {
  return __uint_as_float(((uint32_t)__ldg(p + i)) << 16);
}

// Streaming 16-byte load: read once, do not keep in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Order-preserving map from float to unsigned (a < b  <=>  bits(a) < bits(b) for
// non-NaN floats), so an atomicMax on the bits is a max on the floats; the
// encoding 0 lies below every float and stands for "none yet".
__device__ __forceinline__ unsigned ordered_bits(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered(unsigned o) {
  if (o == 0u) return -CUDART_INF_F;
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// ---------------------------------------------------- (value, index) order ---
// a beats b: larger value, then lower index.  Index INT_MAX stands for "none".
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// -------------------------------------------------------- block reductions ---
// All threads of the CTA must call these; results are returned to every thread.
struct BlockScratch {
  float f[kWarps];
  float g[kWarps];
  int i[kWarps];
  int flag;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (beats(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Scale of a partial sum kept relative to max m when the common max is M >= m.
__device__ __forceinline__ float rescale(float s, float m, float M, float c) {
  return (m == M) ? s : s * ex2_approx((m - M) * c);
}

// Combine per-thread (max, sum of exp2((x - max) c)) pairs over the CTA.
__device__ __forceinline__ void block_lse(float& m, float& s, float c, BlockScratch& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float M = warp_max(m);
  s = warp_sum(rescale(s, m, M, c));
  if (lane == 0) { sh.f[w] = M; sh.g[w] = s; }
  __syncthreads();
  float bm = (lane < kWarps) ? sh.f[lane] : -CUDART_INF_F;
  float bs = (lane < kWarps) ? sh.g[lane] : 0.f;
  const float BM = warp_max(bm);
  bs = warp_sum(rescale(bs, bm, BM, c));
  __syncthreads();
  m = BM;
  s = bs;
}

__device__ __forceinline__ void block_argmax(float& v, int& i, BlockScratch& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  warp_argmax(v, i);
  if (lane == 0) { sh.f[w] = v; sh.i[w] = i; }
  __syncthreads();
  float bv = (lane < kWarps) ? sh.f[lane] : -CUDART_INF_F;
  int bi = (lane < kWarps) ? sh.i[lane] : 0x7fffffff;
  warp_argmax(bv, bi);
  __syncthreads();
  v = bv;
  i = bi;
}

// Barrier over the reducing threads: the whole CTA, or (kNamed) named barrier
// 1 over the first kThreads threads, for kernels whose extra warps do not
// take part.
template <bool kNamed>
__device__ __forceinline__ void reducers_sync() {
  if constexpr (kNamed) asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
  else __syncthreads();
}

// (max, sum, bad-flag) over the CTA in one pass: two barriers.
template <bool kNamed = false>
__device__ __forceinline__ void block_lse_flag(float& m, float& s, int& bad, float c, BlockScratch& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const float M = warp_max(m);
  s = warp_sum(rescale(s, m, M, c));
  const int wb = __any_sync(0xffffffffu, bad);
  if (lane == 0) { sh.f[w] = M; sh.g[w] = s; sh.i[w] = wb; }
  reducers_sync<kNamed>();
  const float bm = (lane < kWarps) ? sh.f[lane] : -CUDART_INF_F;
  float bs = (lane < kWarps) ? sh.g[lane] : 0.f;
  bad = __any_sync(0xffffffffu, lane < kWarps && sh.i[lane]);
  const float BM = warp_max(bm);
  bs = warp_sum(rescale(bs, bm, BM, c));
  reducers_sync<kNamed>();
  m = BM;
  s = bs;
}

// (value, lowest index, bad-flag) over the CTA in one pass: two barriers.
template <bool kNamed = false>
__device__ __forceinline__ void block_argmax_flag(float& v, int& i, int& bad, BlockScratch& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  warp_argmax(v, i);
  const int wb = __any_sync(0xffffffffu, bad);
  if (lane == 0) { sh.f[w] = v; sh.i[w] = i; sh.g[w] = __int_as_float(wb); }
  reducers_sync<kNamed>();
  float bv = (lane < kWarps) ? sh.f[lane] : -CUDART_INF_F;
  int bi = (lane < kWarps) ? sh.i[lane] : 0x7fffffff;
  bad = __any_sync(0xffffffffu, lane < kWarps && __float_as_int(sh.g[lane]));
  warp_argmax(bv, bi);
  reducers_sync<kNamed>();
  v = bv;
  i = bi;
}

// ------------------------------------------- bulk copies, barriers, flags ---
__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make the initialised barriers visible to the bulk-copy engine.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
               : "memory");
}

// Arrive and announce `bytes` of bulk-copy data that will complete this phase.
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr long long kWaitLimitNs = 1000000000LL;   // 1 s: a bulk copy that has not landed by then never will

__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait that lets the hardware suspend the thread until the phase completes
// or about `hint_ns` nanoseconds pass, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, unsigned parity, unsigned hint_ns) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`; false if it did not complete within the limit.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = global_ns();
  while (!mbar_try_wait_suspend(bar, parity, 100000u))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// As mbar_wait_bounded, for one warp waiting on behalf of a CTA whose other
// warps sleep at a barrier: between polls the warp sleeps (32 ns, doubling up
// to 512 ns), so that it takes no issue slots from warps that compute.
__device__ __forceinline__ bool mbar_wait_sleepy(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = global_ns();
  unsigned ns = 32;
  while (!mbar_try_wait(bar, parity)) {
    __nanosleep(ns);
    ns = ns < 512 ? 2 * ns : 512;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// As mbar_wait_bounded, but also gives up (false) once *stop is nonzero.
__device__ __forceinline__ bool mbar_wait_bounded_unless(uint64_t* bar, unsigned parity, const int* stop) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = global_ns();
  while (!mbar_try_wait_suspend(bar, parity, 20000u)) {
    if (*(const volatile int*)stop) return false;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// One bulk copy global -> this CTA's shared memory; completion is counted on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Order this CTA's earlier shared-memory accesses before later bulk-copy writes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------------ thread-block clusters ---
// A launch without a cluster attribute is a cluster of one CTA.
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_ctas() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_index() {
  unsigned r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// The cluster barrier: a hardware barrier over every thread of the cluster's
// CTAs, which the hardware runs at the same time (no spinning in software).
// Every thread calls arrive, then wait, in the same order.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// The shared-memory address of `p`'s counterpart in the cluster's CTA `rank`.
__device__ __forceinline__ unsigned cluster_map(const void* p, unsigned rank) {
  unsigned a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void cluster_red_add(unsigned a, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t cluster_atom_add(unsigned a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void cluster_store(unsigned a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ int block_or(int x, BlockScratch& sh) {
  if (threadIdx.x == 0) sh.flag = 0;
  __syncthreads();
  if (x) atomicOr(&sh.flag, 1);
  __syncthreads();
  const int r = sh.flag;
  __syncthreads();
  return r;
}

}  // namespace sv
