// Batched speculative-decoding verification for GB300 (sm_103a): kernels and C ABI.
//
// The rule ("Speculative Decoding: Faster Generation Without Changing the
// Model", section "The acceptance rule"; restated as the review step in
// "Cascade Speculative Drafting for Even Faster LLM Inference"): drafts are
// scanned left to right, x_i is accepted iff q_i(x_i) <= p_i(x_i) or
// u_i < p_i(x_i)/q_i(x_i); the first rejection is replaced by a draw from
// max(0, p_i - q_i) and ends the scan; if all k pass, a bonus token is drawn
// from target row k.  Greedy: accept iff x_i is the argmax of target row i.
// Tree ("Ouroboros: Generating Longer Drafts Phrase by Phrase for Faster
// Speculative Decoding", 3.4.3 "Selecting the accepted tokens"): the longest
// accepted branch plus the target's next token.
//
// The work is a stream over the vocabulary rows, bound by HBM bandwidth:
//
//   row pass     one persistent launch over all rows that need statistics.
//                Every CTA owns a contiguous range of fixed-size vocabulary
//                tiles of the (virtual) row list, streams it with 16-byte
//                no-L1 loads and keeps per-thread running (max, sum of
//                exp2((x - max) log2e / T)) -- or (max, first index) in greedy
//                mode -- in registers; a row piece ends in one CTA reduction
//                and one 8-byte partial.  The CTA that completes a row (atomic
//                tile count) merges its partials into (max, ln S) or the
//                argmax; the CTA that completes a sequence runs the per-
//                sequence step: the accept scan (one warp, one position per
//                lane, first rejection by ballot), the greedy match, or the
//                tree walk.  No CTA ever waits for another.
//   sample pass  stochastic mode only: grid (vocabulary tiles x B).  Each CTA
//                takes one tile of the row the sequence needs (the rejected
//                position's target and draft rows, or the bonus row), scores
//                ln(max(0, p - q)) + Gumbel (or z + Gumbel) with Philox noise
//                and keeps the best (score, lowest id); the last CTA of a
//                sequence merges and writes the committed tokens.
//
// Workspace counters return to zero at the end of every call, so the
// workspace needs zero-filling only once.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "spec_device.cuh"
#include "spec_verify.h"

namespace sv {

enum Mode { kStochastic = 0, kGreedy = 1, kTree = 2 };

struct RowStat {
  float m;      // max raw logit (stochastic) or the max value (greedy)
  float lnS;    // ln sum_v exp((x_v - m) / T)
  int arg;      // argmax, lowest index (greedy / tree)
  int status;   // SPEC_OK or SPEC_ERR_NONFINITE
};

struct Partial {
  float a;      // piece max (NaN = bad data seen)
  float b;      // stochastic: sum relative to a; greedy: index bits
};

struct SeqState {
  int n;
  int status;
};

struct Workspace {
  Partial* row_partial;    // [R][nt]
  unsigned* row_cnt;       // [R]
  RowStat* row_stat;       // [R]
  unsigned* seq_cnt;       // [B]
  SeqState* seq;           // [B]
  Partial* samp_partial;   // [B][nt2]
  unsigned* samp_cnt;      // [B]
};

struct Params {
  const void* target;
  const void* draft;
  const int32_t* tokens;       // [B][k] (tree: node tokens [B][N])
  const int32_t* parents;      // tree only
  int B, k, V;                 // tree: k = N
  int nt;                      // row-pass tiles per row
  int nt2;                     // sample-pass tiles per row
  int rows_per_seq;            // rows with statistics per sequence
  long long R;                 // rows with statistics
  float invT;                  // 1 / T (stochastic)
  float c;                     // log2(e) / T (stochastic)
  uint2 key;
  uint32_t b0;                 // global index of sequence 0 (Philox counter word 2)
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* out_leaf;
  int32_t* status;
  float* p_draft;
  float* q_draft;
  float* lse;
  Workspace ws;
};

// ------------------------------------------------------------------ rows ---
template <typename T>
__device__ __forceinline__ float load_elem(const T* p, size_t i);
template <>
__device__ __forceinline__ float load_elem<uint16_t>(const uint16_t* p, size_t i) { return bf16_at(p, i); }
template <>
__device__ __forceinline__ float load_elem<float>(const float* p, size_t i) { return __ldg(p + i); }

// Virtual row r of the row pass -> its address and its sequence.
// Stochastic: per sequence, target rows 0..k-1 then draft rows 0..k-1 (the
// bonus row k needs no normaliser).  Greedy / tree: the sequence's target rows.
template <typename T, int kMode>
__device__ __forceinline__ const T* row_ptr(const Params& P, long long r, int& b) {
  if constexpr (kMode == kStochastic) {
    const int twok = 2 * P.k;
    b = (int)(r / twok);
    const int w = (int)(r % twok);
    if (w < P.k) return (const T*)P.target + ((size_t)b * (P.k + 1) + w) * P.V;
    return (const T*)P.draft + ((size_t)b * P.k + (w - P.k)) * P.V;
  }
  b = (int)(r / P.rows_per_seq);
  const int j = (int)(r % P.rows_per_seq);
  return (const T*)P.target + ((size_t)b * P.rows_per_seq + j) * P.V;
}

// ------------------------------------------------- per-thread accumulators ---
// Elements of a 16-byte vector: 8 bf16 or 4 fp32.
template <typename T>
struct Vec;
template <>
struct Vec<uint16_t> {
  static constexpr int n = 8;
  __device__ static float at(const uint4& v, int e) {
    const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
  template <int U>
  __device__ static float nanmax_all(const uint4 (&v)[U]) {
    uint32_t m = bf16x2_nanmax(v[0].x, v[0].y);
    m = bf16x2_nanmax(m, bf16x2_nanmax(v[0].z, v[0].w));
#pragma unroll
    for (int u = 1; u < U; ++u)
      m = bf16x2_nanmax(m, bf16x2_nanmax(bf16x2_nanmax(v[u].x, v[u].y), bf16x2_nanmax(v[u].z, v[u].w)));
    return nanmax(bf16_lo(m), bf16_hi(m));
  }
};
template <>
struct Vec<float> {
  static constexpr int n = 4;
  __device__ static float at(const uint4& v, int e) {
    const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
  template <int U>
  __device__ static float nanmax_all(const uint4 (&v)[U]) {
    float m = nanmax(nanmax(__uint_as_float(v[0].x), __uint_as_float(v[0].y)),
                     nanmax(__uint_as_float(v[0].z), __uint_as_float(v[0].w)));
#pragma unroll
    for (int u = 1; u < U; ++u)
      m = nanmax(m, nanmax(nanmax(__uint_as_float(v[u].x), __uint_as_float(v[u].y)),
                           nanmax(__uint_as_float(v[u].z), __uint_as_float(v[u].w))));
    return m;
  }
};

// Running max m of the raw logits and sums s_j = sum exp2((x - m) c), c = log2(e)/T.
// The max of each chunk is found first (packed max on the raw data), so each
// element costs one FFMA, one MUFU ex2 and one add; the sums are rescaled only
// when the running max rises.
struct LseAcc {
  float c, m, mc;
  float s[8];
  int bad;  // NaN seen
  __device__ void init(float c_) {
    c = c_;
    m = -CUDART_INF_F;
    mc = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = 0.f;
    bad = 0;
  }
  __device__ __forceinline__ bool raise(float cm) {
    if (cm != cm) { bad = 1; return false; }
    if (cm > m) {
      const float f = ex2_approx((m - cm) * c);
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j] *= f;
      m = cm;
      mc = m * c;
    }
    return m != -CUDART_INF_F;
  }
  template <typename T, int U>
  __device__ __forceinline__ void vec(const uint4 (&v)[U], const int (&)[U]) {
    if (!raise(Vec<T>::template nanmax_all<U>(v))) return;
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int e = 0; e < Vec<T>::n; ++e) s[e] += ex2_approx(fmaf(Vec<T>::at(v[u], e), c, -mc));
  }
  __device__ __forceinline__ void scalar(float x, int) {
    if (raise(x)) s[0] += ex2_approx(fmaf(x, c, -mc));
  }
  __device__ float sum() const {
    return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
  }
};

// Running (max, lowest index of the max) over the raw logits.  Each thread sees
// its elements in increasing index order, so a strictly greater chunk max is
// the only event that moves the index.
struct ArgmaxAcc {
  float bv;
  int bi;
  int bad;
  __device__ void init() {
    bv = -CUDART_INF_F;
    bi = INT_MAX;
    bad = 0;
  }
  template <typename T, int U>
  __device__ __forceinline__ void vec(const uint4 (&v)[U], const int (&idx)[U]) {
    const float cm = Vec<T>::template nanmax_all<U>(v);
    if (cm != cm) { bad = 1; return; }
    if (cm > bv || bi == INT_MAX) {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < Vec<T>::n; ++e)
          if (Vec<T>::at(v[u], e) == cm) {
            bv = cm;
            bi = idx[u] + e;
            return;
          }
    }
  }
  __device__ __forceinline__ void scalar(float x, int i) {
    if (x != x) { bad = 1; return; }
    if (x > bv || bi == INT_MAX) { bv = x; bi = i; }
  }
};

// Stream elements [e0, e1) of one row through `acc`: scalar head up to the
// first 16-byte boundary, 16-byte vectors kUnroll at a time (each load
// coalesced across the warp), then the vector remainder and a scalar tail.
template <typename T, class Acc>
__device__ __forceinline__ void scan_segment(const T* row, int e0, int e1, Acc& acc) {
  constexpr int kVec = Vec<T>::n;
  const int tid = threadIdx.x;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row + e0);
  int head = (int)(((16u - (unsigned)(addr & 15u)) & 15u) / sizeof(T));
  head = min(head, e1 - e0);
  if (tid < head) acc.scalar(load_elem<T>(row, e0 + tid), e0 + tid);
  const int vb = e0 + head;
  const int nvec = (e1 - vb) / kVec;
  const uint4* vp = reinterpret_cast<const uint4*>(row + vb);
  int j = tid;
  for (; j + (kUnroll - 1) * kThreads < nvec; j += kUnroll * kThreads) {
    uint4 v[kUnroll];
    int idx[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream16(vp + j + u * kThreads);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) idx[u] = vb + (j + u * kThreads) * kVec;
    acc.template vec<T, kUnroll>(v, idx);
  }
  for (; j < nvec; j += kThreads) {
    uint4 v[1] = {ld_stream16(vp + j)};
    int idx[1] = {vb + j * kVec};
    acc.template vec<T, 1>(v, idx);
  }
  const int tb = vb + nvec * kVec;
  if (tid < e1 - tb) acc.scalar(load_elem<T>(row, tb + tid), tb + tid);
}

__device__ __forceinline__ RowStat ldcg_stat(const RowStat* p) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  return RowStat{v.x, v.y, __float_as_int(v.z), __float_as_int(v.w)};
}

__device__ __forceinline__ void stcg_stat(RowStat* p, const RowStat& s) {
  __stcg(reinterpret_cast<float4*>(p), make_float4(s.m, s.lnS, __int_as_float(s.arg), __int_as_float(s.status)));
}

// --------------------------------------------------- per-sequence steps ---

// Accept scan of one sequence (warp 0): lane i evaluates position i of each
// 32-position chunk; the first rejection is the lowest set bit of the ballot.
template <typename T>
__device__ void accept_scan(const Params& P, int b) {
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const long long rbase = (long long)b * 2 * k;
  int n = k;
  unsigned tok_bad = 0, nf_bad = 0;
  for (int base = 0; base < k; base += 32) {
    const int i = base + lane;
    const bool valid = i < k;
    bool acc = true;
    bool tbad = false, fbad = false;
    if (valid) {
      const int x = P.tokens[(size_t)b * k + i];
      const RowStat rt = ldcg_stat(P.ws.row_stat + rbase + i);
      const RowStat rd = ldcg_stat(P.ws.row_stat + rbase + k + i);
      fbad = rt.status != SPEC_OK || rd.status != SPEC_OK;
      tbad = x < 0 || x >= P.V;
      if (!tbad) {
        const float xt = load_elem<T>((const T*)P.target, ((size_t)b * (k + 1) + i) * P.V + x);
        const float xd = load_elem<T>((const T*)P.draft, ((size_t)b * k + i) * P.V + x);
        const float lp = (xt - rt.m) * P.invT - rt.lnS;   // ln p_i(x_i)
        const float lq = (xd - rd.m) * P.invT - rd.lnS;   // ln q_i(x_i)
        const float u = accept_uniform(P.key, P.b0 + (uint32_t)b, i);
        acc = (lq <= lp) || (u < expf(lp - lq));
        if (P.p_draft) P.p_draft[(size_t)b * k + i] = expf(lp);
        if (P.q_draft) P.q_draft[(size_t)b * k + i] = expf(lq);
      }
      if (P.lse) {
        P.lse[rbase + i] = rt.m * P.invT + rt.lnS;
        P.lse[rbase + k + i] = rd.m * P.invT + rd.lnS;
      }
    }
    tok_bad |= __ballot_sync(0xffffffffu, tbad);
    nf_bad |= __ballot_sync(0xffffffffu, fbad);
    const unsigned rej = __ballot_sync(0xffffffffu, valid && !acc);
    if (n == k && rej) n = base + __ffs(rej) - 1;
  }
  if (lane == 0) {
    const int st = tok_bad ? SPEC_ERR_TOKEN : nf_bad ? SPEC_ERR_NONFINITE : SPEC_OK;
    P.ws.seq[b] = SeqState{n, st};
  }
}

// Greedy match of one sequence (warp 0): n = first i with x_i != argmax_i.
__device__ void greedy_match(const Params& P, int b) {
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const long long rbase = (long long)b * (k + 1);
  int n = k;
  unsigned tok_bad = 0, nf_bad = 0;
  for (int base = 0; base <= k; base += 32) {
    const int i = base + lane;
    bool mism = false, tbad = false, fbad = false;
    if (i <= k) {
      const RowStat rs = ldcg_stat(P.ws.row_stat + rbase + i);
      fbad = rs.status != SPEC_OK;
      if (i < k) {
        const int x = P.tokens[(size_t)b * k + i];
        tbad = x < 0 || x >= P.V;
        mism = x != rs.arg;
      }
    }
    tok_bad |= __ballot_sync(0xffffffffu, tbad);
    nf_bad |= __ballot_sync(0xffffffffu, fbad);
    const unsigned mm = __ballot_sync(0xffffffffu, mism);
    if (n == k && mm) n = base + __ffs(mm) - 1;
  }
  const int st = tok_bad ? SPEC_ERR_TOKEN : nf_bad ? SPEC_ERR_NONFINITE : SPEC_OK;
  const int an = ldcg_stat(P.ws.row_stat + rbase + n).arg;
  for (int i = lane; i <= k; i += 32) {
    int v = -1;
    if (st == SPEC_OK) v = i < n ? P.tokens[(size_t)b * k + i] : (i == n ? an : -1);
    P.out_tokens[(size_t)b * (k + 1) + i] = v;
  }
  if (lane == 0) {
    P.out_n[b] = st == SPEC_OK ? n : -1;
    if (P.status) P.status[b] = st;
  }
}

// Greedy tree verification of one sequence (whole CTA).  Node m is accepted iff
// its parent is (the context is) and its token is the argmax of the parent's
// row; the deepest accepted node wins, the lowest index among equals.
__device__ void tree_walk(const Params& P, int b) {
  __shared__ short s_par[SPEC_MAX_TREE_N];
  __shared__ short s_dep[SPEC_MAX_TREE_N];  // depth if accepted, 0 if not; ok flag before the walk
  __shared__ int s_best, s_bad;
  const int N = P.k;
  const long long rbase = (long long)b * (N + 1);
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int tbad = 0, fbad = 0;
  for (int m = threadIdx.x; m < N; m += kThreads) {
    const int par = P.parents[(size_t)b * N + m];
    const int tok = P.tokens[(size_t)b * N + m];
    const bool ok_shape = par >= -1 && par < m && tok >= 0 && tok < P.V;
    tbad |= !ok_shape;
    int ok = 0;
    if (ok_shape) ok = tok == ldcg_stat(P.ws.row_stat + rbase + (par < 0 ? 0 : par + 1)).arg;
    s_par[m] = (short)(ok_shape ? par : -1);
    s_dep[m] = (short)ok;
  }
  for (int r = threadIdx.x; r <= N; r += kThreads) fbad |= ldcg_stat(P.ws.row_stat + rbase + r).status != SPEC_OK;
  if (tbad) atomicOr(&s_bad, 2);
  if (fbad) atomicOr(&s_bad, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = -1, best_d = 0;
    for (int m = 0; m < N; ++m) {
      const int par = s_par[m];
      int d = 0;
      if (s_dep[m]) d = par < 0 ? 1 : (s_dep[par] > 0 ? s_dep[par] + 1 : 0);
      s_dep[m] = (short)d;
      if (d > best_d) { best_d = d; best = m; }
    }
    s_best = best;
  }
  __syncthreads();
  const int st = (s_bad & 2) ? SPEC_ERR_TOKEN : (s_bad & 1) ? SPEC_ERR_NONFINITE : SPEC_OK;
  const int best = s_best;
  const int depth = best < 0 ? 0 : s_dep[best];
  int32_t* out = P.out_tokens + (size_t)b * (N + 1);
  for (int i = threadIdx.x; i <= N; i += kThreads)
    if (st != SPEC_OK || i > depth) out[i] = -1;
  if (threadIdx.x == 0 && st == SPEC_OK) {
    out[depth] = ldcg_stat(P.ws.row_stat + rbase + (best < 0 ? 0 : best + 1)).arg;
    for (int m = best, d = depth - 1; m >= 0; m = s_par[m], --d) out[d] = P.tokens[(size_t)b * N + m];
  }
  if (threadIdx.x == 0) {
    P.out_n[b] = st == SPEC_OK ? depth : -1;
    if (P.out_leaf) P.out_leaf[b] = st == SPEC_OK ? best : -1;
    if (P.status) P.status[b] = st;
  }
}

// --------------------------------------------------------------- row pass ---

template <typename T, int kMode>
__device__ void finish_row(const Params& P, long long r, int b, BlockScratch& sh, int& s_last) {
  __threadfence();
  const Partial* src = P.ws.row_partial + r * P.nt;
  RowStat st;
  if constexpr (kMode == kStochastic) {
    float m = -CUDART_INF_F, s = 0.f;
    int bad = 0;
    for (int t = threadIdx.x; t < P.nt; t += kThreads) {
      const float2 p = __ldcg(reinterpret_cast<const float2*>(src + t));
      if (p.x != p.x) { bad = 1; continue; }
      const float M = fmaxf(m, p.x);
      s = rescale(s, m, M, P.c) + rescale(p.y, p.x, M, P.c);
      m = M;
    }
    bad = block_or(bad, sh);
    block_lse(m, s, P.c, sh);
    const bool finite = m > -CUDART_INF_F && m < CUDART_INF_F && s > 0.f && s < CUDART_INF_F;
    st = RowStat{m, logf(s), 0, (bad || !finite) ? SPEC_ERR_NONFINITE : SPEC_OK};
  } else {
    float v = -CUDART_INF_F;
    int ix = INT_MAX, bad = 0;
    for (int t = threadIdx.x; t < P.nt; t += kThreads) {
      const float2 p = __ldcg(reinterpret_cast<const float2*>(src + t));
      if (p.x != p.x) { bad = 1; continue; }
      const int pi = __float_as_int(p.y);
      if (beats(p.x, pi, v, ix)) { v = p.x; ix = pi; }
    }
    bad = block_or(bad, sh);
    block_argmax(v, ix, sh);
    st = RowStat{v, 0.f, ix, bad ? SPEC_ERR_NONFINITE : SPEC_OK};
  }
  if (threadIdx.x == 0) {
    stcg_stat(P.ws.row_stat + r, st);
    P.ws.row_cnt[r] = 0;  // ready for the next call
    __threadfence();
    const unsigned old = atomicAdd(P.ws.seq_cnt + b, 1u);
    s_last = old + 1 == (unsigned)P.rows_per_seq;
    if (s_last) P.ws.seq_cnt[b] = 0;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    if constexpr (kMode == kTree) {
      tree_walk(P, b);
    } else if (threadIdx.x < 32) {
      if constexpr (kMode == kStochastic) accept_scan<T>(P, b);
      else greedy_match(P, b);
    }
  }
}

template <typename T, int kMode>
__global__ void __launch_bounds__(kThreads) row_pass_kernel(const Params P) {
  __shared__ BlockScratch sh;
  __shared__ int s_last;
  const long long I = P.R * P.nt;
  const long long i0 = I * blockIdx.x / gridDim.x;
  const long long i1 = I * (blockIdx.x + 1) / gridDim.x;
  for (long long i = i0; i < i1;) {
    const long long r = i / P.nt;
    const int t0 = (int)(i % P.nt);
    const int t1 = (int)min((long long)P.nt, (long long)t0 + (i1 - i));
    int b;
    const T* row = row_ptr<T, kMode>(P, r, b);
    const int e0 = t0 * kTile, e1 = min(P.V, t1 * kTile);
    float2 part;
    if constexpr (kMode == kStochastic) {
      LseAcc acc;
      acc.init(P.c);
      scan_segment<T>(row, e0, e1, acc);
      float m = acc.m, s = acc.sum();
      const int bad = block_or(acc.bad, sh);
      block_lse(m, s, P.c, sh);
      part = make_float2(bad ? CUDART_NAN_F : m, s);
    } else {
      ArgmaxAcc acc;
      acc.init();
      scan_segment<T>(row, e0, e1, acc);
      float v = acc.bv;
      int ix = acc.bi;
      const int bad = block_or(acc.bad, sh);
      block_argmax(v, ix, sh);
      part = make_float2(bad ? CUDART_NAN_F : v, __int_as_float(ix));
    }
    if (threadIdx.x == 0) {
      float2* dst = reinterpret_cast<float2*>(P.ws.row_partial + r * P.nt);
      __stcg(dst + t0, part);
      const float2 neutral = make_float2(-CUDART_INF_F, kMode == kStochastic ? 0.f : __int_as_float(INT_MAX));
      for (int t = t0 + 1; t < t1; ++t) __stcg(dst + t, neutral);
      __threadfence();
      const unsigned add = (unsigned)(t1 - t0);
      const unsigned old = atomicAdd(P.ws.row_cnt + r, add);
      s_last = old + add == (unsigned)P.nt;
    }
    __syncthreads();
    if (s_last) finish_row<T, kMode>(P, r, b, sh, s_last);
    __syncthreads();
    i += t1 - t0;
  }
}

// ------------------------------------------------------------ sample pass ---

template <typename T>
__global__ void __launch_bounds__(kThreads) sample_pass_kernel(const Params P) {
  __shared__ BlockScratch sh;
  __shared__ int s_last;
  const int b = blockIdx.x / P.nt2;
  const int t = blockIdx.x % P.nt2;
  const int k = P.k;
  const SeqState ss = P.ws.seq[b];
  const int n = ss.n;
  float best = -CUDART_INF_F;
  int bidx = INT_MAX, bad = 0;
  const int v0 = t * kSampleTile, v1 = min(P.V, v0 + kSampleTile);
  if (ss.status == SPEC_OK) {
    if (n < k) {
      // residual: ln(p - q) = ln p + ln(1 - exp(ln q - ln p)) where p > q
      const RowStat rt = ldcg_stat(P.ws.row_stat + (long long)b * 2 * k + n);
      const RowStat rd = ldcg_stat(P.ws.row_stat + (long long)b * 2 * k + k + n);
      const T* trow = (const T*)P.target + ((size_t)b * (k + 1) + n) * P.V;
      const T* drow = (const T*)P.draft + ((size_t)b * k + n) * P.V;
      for (int g = (v0 >> 2) + threadIdx.x; 4 * g < v1; g += kThreads) {
        const uint4 w = gumbel_words(P.key, P.b0 + (uint32_t)b, n, (uint32_t)g);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = 4 * g + e;
          if (v >= v1) break;
          const float lp = (load_elem<T>(trow, v) - rt.m) * P.invT - rt.lnS;
          const float lq = (load_elem<T>(drow, v) - rd.m) * P.invT - rd.lnS;
          if (lp > lq) {
            const float sc = lp + logf(-expm1f(lq - lp)) + gumbel_of(uniform_of(ws[e]));
            if (beats(sc, v, best, bidx)) { best = sc; bidx = v; }
          }
        }
      }
    } else {
      // bonus: argmax of x/T + Gumbel over target row k
      const T* trow = (const T*)P.target + ((size_t)b * (k + 1) + k) * P.V;
      for (int g = (v0 >> 2) + threadIdx.x; 4 * g < v1; g += kThreads) {
        const uint4 w = gumbel_words(P.key, P.b0 + (uint32_t)b, k, (uint32_t)g);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = 4 * g + e;
          if (v >= v1) break;
          const float x = load_elem<T>(trow, v);
          if (x != x || x == CUDART_INF_F) bad = 1;
          const float sc = x * P.invT + gumbel_of(uniform_of(ws[e]));
          if (beats(sc, v, best, bidx)) { best = sc; bidx = v; }
        }
      }
    }
  }
  bad = block_or(bad, sh);
  block_argmax(best, bidx, sh);
  if (threadIdx.x == 0) {
    __stcg(reinterpret_cast<float2*>(P.ws.samp_partial) + (size_t)b * P.nt2 + t,
           make_float2(bad ? CUDART_NAN_F : best, __int_as_float(bidx)));
    __threadfence();
    const unsigned old = atomicAdd(P.ws.samp_cnt + b, 1u);
    s_last = old + 1 == (unsigned)P.nt2;
    if (s_last) P.ws.samp_cnt[b] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  best = -CUDART_INF_F;
  bidx = INT_MAX;
  bad = 0;
  for (int tt = threadIdx.x; tt < P.nt2; tt += kThreads) {
    const float2 p = __ldcg(reinterpret_cast<const float2*>(P.ws.samp_partial) + (size_t)b * P.nt2 + tt);
    if (p.x != p.x) { bad = 1; continue; }
    const int pi = __float_as_int(p.y);
    if (beats(p.x, pi, best, bidx)) { best = p.x; bidx = pi; }
  }
  bad = block_or(bad, sh);
  block_argmax(best, bidx, sh);
  int st = ss.status;
  if (st == SPEC_OK && n == k && (bad || !(best > -CUDART_INF_F))) st = SPEC_ERR_NONFINITE;
  if (st == SPEC_OK && n < k && bidx == INT_MAX) {
    // empty residual in fp32: draw from p_n itself with the same noise
    const T* trow = (const T*)P.target + ((size_t)b * (k + 1) + n) * P.V;
    best = -CUDART_INF_F;
    for (int g = threadIdx.x; 4 * g < P.V; g += kThreads) {
      const uint4 w = gumbel_words(P.key, P.b0 + (uint32_t)b, n, (uint32_t)g);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      for (int e = 0; e < 4 && 4 * g + e < P.V; ++e) {
        const int v = 4 * g + e;
        const float sc = load_elem<T>(trow, v) * P.invT + gumbel_of(uniform_of(ws[e]));
        if (beats(sc, v, best, bidx)) { best = sc; bidx = v; }
      }
    }
    block_argmax(best, bidx, sh);
  }
  int32_t* out = P.out_tokens + (size_t)b * (k + 1);
  for (int i = threadIdx.x; i <= k; i += kThreads) {
    int v = -1;
    if (st == SPEC_OK) v = i < n ? P.tokens[(size_t)b * k + i] : (i == n ? bidx : -1);
    out[i] = v;
  }
  if (threadIdx.x == 0) {
    P.out_n[b] = st == SPEC_OK ? n : -1;
    if (P.status) P.status[b] = st;
  }
}

// -------------------------------------------------------------- randomness ---
__global__ void random_kernel(uint2 key, int b, int j, int V, float* gu, float* gg, float* au) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g == 0 && au) au[0] = accept_uniform(key, b, j);
  if (4 * g >= V) return;
  const uint4 w = gumbel_words(key, b, j, (uint32_t)g);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  for (int e = 0; e < 4 && 4 * g + e < V; ++e) {
    const float u = uniform_of(ws[e]);
    if (gu) gu[4 * g + e] = u;
    if (gg) gg[4 * g + e] = gumbel_of(u);
  }
}

// --------------------------------------------------------------- host side ---

struct Layout {
  size_t row_partial, row_cnt, row_stat, seq_cnt, seq, samp_partial, samp_cnt, total;
  int nt, nt2;
  long long rmax;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static bool make_layout(int B, int k, int V, Layout& L) {
  if (B <= 0 || k <= 0 || V <= 0) return false;
  L.nt = (V + kTile - 1) / kTile;
  L.nt2 = (V + kSampleTile - 1) / kSampleTile;
  L.rmax = (long long)B * (long long)(2 * k > k + 1 ? 2 * k : k + 1);
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = align_up(off + bytes, 256); return o; };
  L.row_partial = take((size_t)L.rmax * L.nt * sizeof(Partial));
  L.row_cnt = take((size_t)L.rmax * sizeof(unsigned));
  L.row_stat = take((size_t)L.rmax * sizeof(RowStat));
  L.seq_cnt = take((size_t)B * sizeof(unsigned));
  L.seq = take((size_t)B * sizeof(SeqState));
  L.samp_partial = take((size_t)B * L.nt2 * sizeof(Partial));
  L.samp_cnt = take((size_t)B * sizeof(unsigned));
  L.total = off;
  return true;
}

static Workspace bind(void* base, const Layout& L) {
  char* p = static_cast<char*>(base);
  return Workspace{reinterpret_cast<Partial*>(p + L.row_partial), reinterpret_cast<unsigned*>(p + L.row_cnt),
                   reinterpret_cast<RowStat*>(p + L.row_stat),    reinterpret_cast<unsigned*>(p + L.seq_cnt),
                   reinterpret_cast<SeqState*>(p + L.seq),        reinterpret_cast<Partial*>(p + L.samp_partial),
                   reinterpret_cast<unsigned*>(p + L.samp_cnt)};
}

// Resident CTAs of a kernel on the current device, cached per (device, kernel).
static int resident_ctas(const void* fn) {
  static std::mutex mu;
  static struct Entry { int dev; const void* fn; int ctas; } cache[64];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].fn == fn) return cache[i].ctas;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0) != cudaSuccess) return 0;
  const int ctas = sms * (per_sm > 0 ? per_sm : 1);
  if (used < 64) cache[used++] = Entry{dev, fn, ctas};
  return ctas;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The completion counters sit at layout-dependent offsets, and a call returns
// only them to zero.  A workspace used with new sizes is therefore cleared
// first; the library remembers the sizes each workspace last served.
static int prepare_workspace(void* ws, const Layout& L, int B, int k, int V, cudaStream_t stream) {
  static std::mutex mu;
  static std::unordered_map<uintptr_t, uint64_t> last;
  const uint64_t sig = ((uint64_t)(uint32_t)V << 32) ^ ((uint64_t)(uint32_t)B << 12) ^ (uint64_t)(uint32_t)k ^
                       ((uint64_t)(uint32_t)k << 44);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = last.find(reinterpret_cast<uintptr_t>(ws));
    if (it != last.end() && it->second == sig) return SPEC_OK;
    last[reinterpret_cast<uintptr_t>(ws)] = sig;
  }
  if (cudaMemsetAsync(ws, 0, L.total, stream) != cudaSuccess) {
    std::lock_guard<std::mutex> lock(mu);
    last.erase(reinterpret_cast<uintptr_t>(ws));
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

template <typename T, int kMode>
static int launch_row_pass(const Params& P, cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(&row_pass_kernel<T, kMode>);
  const int ctas = resident_ctas(fn);
  if (ctas <= 0) return SPEC_ERR_CUDA;
  const long long items = P.R * P.nt;
  const int grid = (int)(items < ctas ? items : ctas);
  row_pass_kernel<T, kMode><<<grid, kThreads, 0, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

template <typename T>
static int launch_stochastic(const Params& P, cudaStream_t stream, const spec_verify_aux* aux) {
  auto rec = [&](int i) {
    return (aux && aux->events[i]) ? cudaEventRecord(static_cast<cudaEvent_t>(aux->events[i]), stream) : cudaSuccess;
  };
  if (rec(0) != cudaSuccess) return SPEC_ERR_CUDA;
  int rc = launch_row_pass<T, kStochastic>(P, stream);
  if (rc != SPEC_OK) return rc;
  if (rec(1) != cudaSuccess || rec(2) != cudaSuccess) return SPEC_ERR_CUDA;
  sample_pass_kernel<T><<<P.B * P.nt2, kThreads, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  return rec(3) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_workspace_size(int B, int k, int V, int dtype) {
  if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return 0;
  Layout L;
  if (!make_layout(B, k, V, L)) return 0;
  return L.total;
}

int spec_workspace_init(void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!workspace || workspace_bytes == 0) return SPEC_ERR_ARG;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

static int check_common(const void* target, int B, int V, int dtype, void* workspace, const Layout& L,
                        size_t workspace_bytes) {
  if (!target || B <= 0 || V <= 0) return SPEC_ERR_ARG;
  if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return SPEC_ERR_ARG;
  if (!aligned(target, dtype == SPEC_BF16 ? 2 : 4)) return SPEC_ERR_ALIGN;
  if (!workspace || !aligned(workspace, 16) || workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

int spec_verify_ex(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens, int B, int k,
                   int V, int dtype, float temperature, uint64_t seed, int32_t* out_tokens, int32_t* out_n_accepted,
                   void* workspace, size_t workspace_bytes, void* cuda_stream, const spec_verify_aux* aux) {
  if (k <= 0 || B <= 0 || V <= 0) return SPEC_ERR_ARG;
  if (k > SPEC_MAX_K) return SPEC_ERR_UNSUPPORTED;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SPEC_ERR_ARG;
  const bool greedy = temperature == 0.f;
  if (!draft_tokens || !out_tokens || !out_n_accepted || (!greedy && !draft_logits)) return SPEC_ERR_ARG;
  if ((size_t)B * (size_t)(k + 1) > (size_t)INT_MAX) return SPEC_ERR_UNSUPPORTED;
  Layout L;
  make_layout(B, k, V, L);
  int rc = check_common(target_logits, B, V, dtype, workspace, L, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  if (!greedy && !aligned(draft_logits, dtype == SPEC_BF16 ? 2 : 4)) return SPEC_ERR_ALIGN;
  if (!aligned(draft_tokens, 4) || !aligned(out_tokens, 4) || !aligned(out_n_accepted, 4)) return SPEC_ERR_ALIGN;
  if ((long long)B * L.nt2 > INT_MAX) return SPEC_ERR_UNSUPPORTED;

  Params P;
  std::memset(&P, 0, sizeof(P));
  P.target = target_logits;
  P.draft = draft_logits;
  P.tokens = draft_tokens;
  P.B = B;
  P.k = k;
  P.V = V;
  P.nt = L.nt;
  P.nt2 = L.nt2;
  P.key = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
  P.out_tokens = out_tokens;
  P.out_n = out_n_accepted;
  P.ws = bind(workspace, L);
  if (aux) {
    P.status = aux->status;
    P.p_draft = aux->p_draft;
    P.q_draft = aux->q_draft;
    P.lse = aux->lse;
    P.b0 = aux->sequence_offset;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if ((rc = prepare_workspace(workspace, L, B, k, V, stream)) != SPEC_OK) return rc;
  if (greedy) {
    P.rows_per_seq = k + 1;
    P.R = (long long)B * (k + 1);
    auto rec = [&](int i) {
      return (aux && aux->events[i]) ? cudaEventRecord(static_cast<cudaEvent_t>(aux->events[i]), stream)
                                     : cudaSuccess;
    };
    if (rec(0) != cudaSuccess) return SPEC_ERR_CUDA;
    rc = dtype == SPEC_BF16 ? launch_row_pass<uint16_t, kGreedy>(P, stream) : launch_row_pass<float, kGreedy>(P, stream);
    if (rc != SPEC_OK) return rc;
    return rec(1) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  P.rows_per_seq = 2 * k;
  P.R = (long long)B * 2 * k;
  P.invT = 1.0f / temperature;
  P.c = (float)(1.4426950408889634 / (double)temperature);
  return dtype == SPEC_BF16 ? launch_stochastic<uint16_t>(P, stream, aux) : launch_stochastic<float>(P, stream, aux);
}

int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens, int B, int k, int V,
                int dtype, float temperature, uint64_t seed, int32_t* out_tokens, int32_t* out_n_accepted,
                void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return spec_verify_ex(target_logits, draft_logits, draft_tokens, B, k, V, dtype, temperature, seed, out_tokens,
                        out_n_accepted, workspace, workspace_bytes, cuda_stream, nullptr);
}

int spec_verify_tree(const void* target_logits, const int32_t* node_tokens, const int32_t* parents, int B, int N,
                     int V, int dtype, float temperature, int32_t* out_tokens, int32_t* out_n_accepted,
                     int32_t* out_leaf, int32_t* status, void* workspace, size_t workspace_bytes,
                     void* cuda_stream) {
  if (B <= 0 || N <= 0 || V <= 0) return SPEC_ERR_ARG;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SPEC_ERR_ARG;
  if (temperature != 0.f || N > SPEC_MAX_TREE_N) return SPEC_ERR_UNSUPPORTED;
  if (!node_tokens || !parents || !out_tokens || !out_n_accepted) return SPEC_ERR_ARG;
  if ((size_t)B * (size_t)(N + 1) > (size_t)INT_MAX) return SPEC_ERR_UNSUPPORTED;
  Layout L;
  make_layout(B, N, V, L);
  const int rc = check_common(target_logits, B, V, dtype, workspace, L, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  if (!aligned(node_tokens, 4) || !aligned(parents, 4) || !aligned(out_tokens, 4) || !aligned(out_n_accepted, 4))
    return SPEC_ERR_ALIGN;
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.target = target_logits;
  P.tokens = node_tokens;
  P.parents = parents;
  P.B = B;
  P.k = N;
  P.V = V;
  P.nt = L.nt;
  P.nt2 = L.nt2;
  P.rows_per_seq = N + 1;
  P.R = (long long)B * (N + 1);
  P.out_tokens = out_tokens;
  P.out_n = out_n_accepted;
  P.out_leaf = out_leaf;
  P.status = status;
  P.ws = bind(workspace, L);
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  const int prc = prepare_workspace(workspace, L, B, N, V, stream);
  if (prc != SPEC_OK) return prc;
  return dtype == SPEC_BF16 ? launch_row_pass<uint16_t, kTree>(P, stream) : launch_row_pass<float, kTree>(P, stream);
}

int spec_random(uint64_t seed, int b, int j, int V, float* gumbel_u, float* gumbel_g, float* accept_u,
                void* cuda_stream) {
  if (V <= 0 || b < 0 || j < 0) return SPEC_ERR_ARG;
  const int groups = (V + 3) / 4;
  random_kernel<<<(groups + kThreads - 1) / kThreads, kThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)), b, j, V, gumbel_u, gumbel_g, accept_u);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

const char* spec_strerror(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_ARG: return "invalid argument";
    case SPEC_ERR_ALIGN: return "misaligned pointer";
    case SPEC_ERR_TOKEN: return "token id or tree parent out of range";
    case SPEC_ERR_NONFINITE: return "NaN or +inf logit, or a row with no finite logit";
    case SPEC_ERR_UNSUPPORTED: return "unsupported configuration";
    case SPEC_ERR_TIMEOUT: return "device wait timed out";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int spec_abi_version(void) { return (1 << 16) | 0; }

}  // extern "C"

// ------------------------------------------------- allocation-free variant ---
// spec_verify_noalloc runs the same kernels as spec_verify, with the kernels'
// scratch (partials, counters, per-row and per-sequence state) in a
// fixed-size array that is part of this library's device image, so the
// caller passes no workspace and nothing is allocated at call time.  Every
// GPU that loads the library holds this array until the process exits.
namespace sv {

constexpr size_t kNoAllocScratchBytes = SPEC_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array on the current device.  The host-side name
// g_noalloc_scratch is only a stand-in for the symbol, never a device
// pointer, so the address is looked up once per device, with that device
// current, and cached.
static int noalloc_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kNoAllocMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return SPEC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return SPEC_OK;
}

}  // namespace sv

extern "C" int spec_verify_noalloc(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                                   int B, int k, int V, int dtype, float temperature, uint64_t seed,
                                   int32_t* out_tokens, int32_t* out_n_accepted, void* cuda_stream) {
  const size_t need = spec_workspace_size(B, k, V, dtype);
  if (need > sv::kNoAllocScratchBytes) return SPEC_ERR_WORKSPACE;  // sizes beyond the built-in scratch
  void* scratch = nullptr;
  const int rc = sv::noalloc_scratch_address(&scratch);
  if (rc != SPEC_OK) return rc;
  // The scratch keeps whatever the previous call left in it.  The counters
  // that must start at zero are returned to zero by every call, and
  // spec_verify_ex clears the region first whenever the sizes differ from
  // those of the previous call on this scratch.
  return spec_verify_ex(target_logits, draft_logits, draft_tokens, B, k, V, dtype, temperature, seed, out_tokens,
                        out_n_accepted, scratch, sv::kNoAllocScratchBytes, cuda_stream, nullptr);
}
