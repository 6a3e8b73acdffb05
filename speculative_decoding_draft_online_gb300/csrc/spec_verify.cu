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
// The work is a stream over the vocabulary rows, bound by HBM bandwidth.
//
//   row pass    one persistent launch.  Each CTA owns a contiguous range of
//               4096-element row tiles of the virtual row list (balanced to
//               one tile) and streams it with 16-byte no-L1 loads, four
//               vectors per thread in flight at a time.  Threads keep running
//               (max, sum of exp2((x - max) log2e / T)) -- or (max, first
//               index) in greedy mode -- across the tiles of a row, one MUFU
//               ex2 per element;
//               a row piece ends in one CTA reduction and one 16-byte partial.
//               The CTA that completes a row (atomic tile count) merges its
//               partials in one warp; the one that completes a sequence runs
//               its per-sequence step in that warp: the accept scan (one
//               position per lane, first rejection by ballot), the greedy
//               match, or the tree walk.  Greedy and tree batches of aligned
//               rows larger than L2 stream through a ring of bulk copies into
//               shared memory instead, fed by a producer warp.
//   sampling    stochastic mode, a second launch that starts while the row
//               pass drains (programmatic dependent launch): for each sequence,
//               as many CTAs as fill the GPU once share the 4096-id tiles of the
//               rows it needs (the rejected position's target and draft rows,
//               or the bonus row), staged by bulk copies, scoring
//               ln max(0, p - q) + Gumbel, or z + Gumbel, with Philox noise,
//               pruned exactly against the best score reached so far; the
//               last CTA of a sequence merges and writes the committed tokens.
//
// No kernel waits on a flag another CTA sets (the bulk-copy waits are on the
// CTA's own barriers, bounded); completion is detected with atomic counters by
// whichever CTA finishes last.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstddef>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "spec_device.cuh"
#include "spec_verify.h"

namespace sv {

enum Mode { kStochastic = 0, kGreedy = 1, kTree = 2 };

constexpr int kPartTile = 4096;            // row pass: partition granularity, elements
constexpr int kUnroll = 4;                 // row pass: 16-byte vectors per thread per batch
constexpr int kGroups = kPartTile / 4 / kThreads;   // sampling: 4-id groups per thread per tile

struct RowStat {
  float m;      // max raw logit
  float lnS;    // ln sum_v exp((x_v - m) / T) (stochastic)
  int arg;      // index of the max, lowest among equals (greedy and tree)
  int status;   // SPEC_OK or SPEC_ERR_NONFINITE
};

// One row piece: (max or NaN for bad data, sum relative to the max, index of
// the max in greedy and tree mode).
struct Partial {
  float m;
  float s;
  int idx;
  int pad;
};

// A sequence's state after its accept scan, and what the sampling pass needs
// of its sampled row, in one 32-byte record: a sampling CTA has all of it
// after one load and issues its copies at once.
struct SeqState {
  int n;
  int status;
  int pad;               // (keeps the record two 16-byte words)
  float tau_d;           // residual, filtering: the draft's kept set is x_d >= tau_d (-inf: all)
  float mt, lnSt;        // residual: target row max and ln of its (kept) mass relative to the max
  float cdelta;          // residual: delta_v = fma(x_d - x_t, 1/T, cdelta)
  float tau_t;           // filtering: the sampled row's kept set is x_t >= tau_t (-inf: all)
};
static_assert(sizeof(SeqState) == 32, "one 32-byte record a sequence");

struct Workspace {
  Partial* row_partial;    // [R][nt]
  unsigned* row_cnt;       // [R]
  RowStat* row_stat;       // [R]
  float2* row_filter;      // [R] filtering mode: (threshold value, ln of the kept mass relative to the max)
  unsigned* seq_cnt;       // [B]
  SeqState* seq;           // [B]
  float2* samp_partial;    // [B][ns] (best score or NaN, index bits)
  unsigned* samp_cnt;      // [B]
  unsigned* samp_floor;    // [B] best score reached so far, order-preserving encoding (0 = none)
};

struct Params {
  const void* target;
  const void* draft;
  const int32_t* tokens;       // [B][k] (tree: node tokens [B][N])
  const int32_t* parents;      // tree only
  int B, k, V;                 // tree: k = N
  int nt;                      // row-pass tiles per row
  int ns;                      // sampling CTAs per sequence (1 <= ns <= nt)
  int rows_per_seq;            // rows with statistics per sequence
  long long R;                 // rows with statistics
  float invT;                  // 1 / T (stochastic)
  float T;                     // temperature (stochastic)
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
  int out_w;                   // out_tokens row width
  float lenience;              // l >= 1 (stochastic); 1 is the exact rule
  float ln_lenience;           // ln l
  const int32_t* stop_ids;     // [n_stop]: the committed tokens end at the first one
  int n_stop;
  int32_t* n_committed;        // [B] or null
  uint8_t* match_mask;         // greedy: [B][k] or null
  int32_t* n_match;            // greedy: [B] or null
  int32_t* tail_runs;          // greedy: [B] or null
  const int32_t* guide;        // guided greedy: [B][L] or null
  int L;
  int filtering;               // stochastic rows go through top-k / top-p
  int top_k;                   // 0: off
  float top_p;                 // 0 or 1: off
  int force_timeout;           // test hook: every bulk-copy stage wait gives up at once
  Workspace ws;
};

// ------------------------------------------------------------------ rows ---
template <typename T>
__device__ __forceinline__ float load_elem(const T* p, size_t i);
template <>
__device__ __forceinline__ float load_elem<uint16_t>(const uint16_t* p, size_t i) { return bf16_at(p, i); }
template <>
__device__ __forceinline__ float load_elem<float>(const float* p, size_t i) { return __ldg(p + i); }

// Virtual row r -> its address and its sequence.  Stochastic: per sequence,
// target rows 0..k-1 then draft rows 0..k-1 (the bonus row k needs no
// normaliser), then, when filtering, target row k (its filter needs one).
// Greedy / tree: the sequence's target rows.
template <typename T, int kMode>
__device__ __forceinline__ const T* row_ptr(const Params& P, long long r, int& b) {
  if constexpr (kMode == kStochastic) {
    b = (int)(r / P.rows_per_seq);
    const int w = (int)(r % P.rows_per_seq);
    if (w < P.k) return (const T*)P.target + ((size_t)b * (P.k + 1) + w) * P.V;
    if (w < 2 * P.k) return (const T*)P.draft + ((size_t)b * P.k + (w - P.k)) * P.V;
    return (const T*)P.target + ((size_t)b * (P.k + 1) + P.k) * P.V;   // filtering: the bonus row
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

// First index of value cm among the vectors' elements (it is there).
template <typename T, int U>
__device__ __forceinline__ int first_index_of(const uint4 (&v)[U], const int (&idx)[U], float cm) {
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int e = 0; e < Vec<T>::n; ++e)
      if (Vec<T>::at(v[u], e) == cm) return idx[u] + e;
  return INT_MAX;
}

// Running max m of the raw logits and sums s_j = sum exp2((x - m) c),
// c = log2(e)/T.  The max of each chunk is found first (packed max on the raw
// data), so each element costs one FFMA, one MUFU ex2 and one add; the sums
// are rescaled only when the running max rises.  (The index of the max is not
// tracked: searching for it whenever some lane's max rises costs more than
// the rest of the fold.)
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
  __device__ __forceinline__ void rise(float cm) {
    const float f = ex2_approx((m - cm) * c);
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] *= f;
    m = cm;
    mc = m * c;
  }
  template <typename T, int U>
  __device__ __forceinline__ void vec(const uint4 (&v)[U], const int (&)[U]) {
    const float cm = Vec<T>::template nanmax_all<U>(v);
    if (cm != cm) { bad = 1; return; }
    if (cm > m) rise(cm);
    if (m == -CUDART_INF_F) return;
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int e = 0; e < Vec<T>::n; ++e) s[e] += ex2_approx(fmaf(Vec<T>::at(v[u], e), c, -mc));
  }
  __device__ __forceinline__ void scalar(float x, int) {
    if (x != x) { bad = 1; return; }
    if (x > m) rise(x);
    if (m != -CUDART_INF_F) s[0] += ex2_approx(fmaf(x, c, -mc));
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
      bv = cm;
      bi = first_index_of<T, U>(v, idx, cm);
    }
  }
  __device__ __forceinline__ void scalar(float x, int i) {
    if (x != x) { bad = 1; return; }
    if (x > bv || bi == INT_MAX) { bv = x; bi = i; }
  }
};

// Stream elements [e0, e1) of one row through `acc`: a scalar head up to the
// first 16-byte boundary, then 16-byte vectors kUnroll per thread per batch
// (each load coalesced across the warp; all of a batch's loads are issued
// before it is folded), then the vector remainder and a scalar tail.  Four
// CTAs of 64 registers per SM keep enough loads in flight; a software
// pipeline that requests the next batch early needs more registers, and the
// occupancy it costs loses more than it gains.
// Each thread sees its elements in increasing index order.
template <typename T, class Acc>
__device__ __forceinline__ void scan_segment(const T* row, int e0, int e1, Acc& acc) {
  constexpr int kVec = Vec<T>::n;
  constexpr int kBatch = kUnroll * kThreads;   // vectors per CTA per batch
  const int tid = threadIdx.x;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row + e0);
  const int head = min((int)(((16u - (unsigned)(addr & 15u)) & 15u) / sizeof(T)), e1 - e0);
  if (tid < head) acc.scalar(load_elem<T>(row, e0 + tid), e0 + tid);
  const int vb = e0 + head;
  const int nvec = (e1 - vb) / kVec;
  const uint4* vp = reinterpret_cast<const uint4*>(row + vb);
  const int nfull = nvec / kBatch;
  for (int bt = 0; bt < nfull; ++bt) {
    const int base = bt * kBatch + tid;
    uint4 v[kUnroll];
    int idx[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream16(vp + base + u * kThreads);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) idx[u] = vb + (base + u * kThreads) * kVec;
    acc.template vec<T, kUnroll>(v, idx);
  }
  for (int j = nfull * kBatch + tid; j < nvec; j += kThreads) {
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
// All of these run in warp 0 of the CTA that completed the sequence.

// Accept scan: lane i evaluates position i of each 32-position chunk; the
// first rejection is the lowest set bit of the ballot.
template <typename T>
__device__ void accept_scan(const Params& P, int b) {
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const long long rbase = (long long)b * P.rows_per_seq;
  const long long obase = (long long)b * 2 * k;   // [B][2k] lse output
  int n = k;
  unsigned tok_bad = 0, nf_bad = 0, to_bad = 0;
  // the sampled row's record: the rejected position's rows (set below), or the bonus row's filter
  SeqState rec{0, 0, 0, -CUDART_INF_F, 0.f, 0.f, 0.f, -CUDART_INF_F};
  for (int base = 0; base < k; base += 32) {
    const int i = base + lane;
    const bool valid = i < k;
    bool acc = true;
    bool tbad = false, fbad = false, tmo = false;
    SeqState mine{0, 0, 0, -CUDART_INF_F, 0.f, 0.f, 0.f, -CUDART_INF_F};   // this lane's position as the sampled one
    if (valid) {
      const int x = P.tokens[(size_t)b * k + i];
      const RowStat rt = ldcg_stat(P.ws.row_stat + rbase + i);
      const RowStat rd = ldcg_stat(P.ws.row_stat + rbase + k + i);
      float2 ft = make_float2(-CUDART_INF_F, rt.lnS), fd = make_float2(-CUDART_INF_F, rd.lnS);
      if (P.filtering) {
        ft = __ldcg(P.ws.row_filter + rbase + i);
        fd = __ldcg(P.ws.row_filter + rbase + k + i);
      }
      fbad = rt.status != SPEC_OK || rd.status != SPEC_OK;
      tmo = rt.status == SPEC_ERR_TIMEOUT || rd.status == SPEC_ERR_TIMEOUT;
      tbad = x < 0 || x >= P.V;
      mine.tau_d = fd.x;
      mine.mt = rt.m;
      mine.lnSt = ft.y;
      mine.cdelta = -(rd.m - rt.m) * P.invT - (fd.y - ft.y);
      mine.tau_t = ft.x;
      if (!tbad) {
        const float xt = load_elem<T>((const T*)P.target, ((size_t)b * (k + 1) + i) * P.V + x);
        const float xd = load_elem<T>((const T*)P.draft, ((size_t)b * k + i) * P.V + x);
        float lp = (xt - rt.m) * P.invT - rt.lnS;          // ln p_i(x_i)
        float lq = (xd - rd.m) * P.invT - rd.lnS;          // ln q_i(x_i)
        if (P.filtering) {
          // the filtered, renormalised rows: 0 outside the kept set
          lp = xt >= ft.x ? (xt - rt.m) * P.invT - ft.y : -CUDART_INF_F;
          lq = xd >= fd.x ? (xd - rd.m) * P.invT - fd.y : -CUDART_INF_F;
        }
        const float u = accept_uniform(P.key, P.b0 + (uint32_t)b, i);
        // "Asymmetric lenience": keep when q <= l p, else with probability l p / q
        acc = (lq <= lp + P.ln_lenience) || (u < P.lenience * expf(lp - lq));
        if (P.p_draft) P.p_draft[(size_t)b * k + i] = expf(lp);
        if (P.q_draft) P.q_draft[(size_t)b * k + i] = expf(lq);
      }
      if (P.lse) {
        P.lse[obase + i] = rt.m * P.invT + rt.lnS;
        P.lse[obase + k + i] = rd.m * P.invT + rd.lnS;
      }
    }
    tok_bad |= __ballot_sync(0xffffffffu, tbad);
    nf_bad |= __ballot_sync(0xffffffffu, fbad);
    to_bad |= __ballot_sync(0xffffffffu, tmo);
    const unsigned rej = __ballot_sync(0xffffffffu, valid && !acc);
    if (n == k && rej) {
      n = base + __ffs(rej) - 1;
      const int src = n - base;
      rec.tau_d = __shfl_sync(0xffffffffu, mine.tau_d, src);
      rec.mt = __shfl_sync(0xffffffffu, mine.mt, src);
      rec.lnSt = __shfl_sync(0xffffffffu, mine.lnSt, src);
      rec.cdelta = __shfl_sync(0xffffffffu, mine.cdelta, src);
      rec.tau_t = __shfl_sync(0xffffffffu, mine.tau_t, src);
    }
  }
  // filtering runs over every row of the sequence, the bonus row included
  if (P.filtering) {
    const int bs = ldcg_stat(P.ws.row_stat + rbase + 2 * k).status;
    if (bs != SPEC_OK) nf_bad = 1;
    if (bs == SPEC_ERR_TIMEOUT) to_bad = 1;
    if (n == k) rec.tau_t = __ldcg(P.ws.row_filter + rbase + 2 * k).x;   // the bonus row's filter
  }
  if (lane == 0) {
    rec.n = n;
    rec.status = tok_bad ? SPEC_ERR_TOKEN : to_bad ? SPEC_ERR_TIMEOUT : nf_bad ? SPEC_ERR_NONFINITE : SPEC_OK;
    int4* dst = reinterpret_cast<int4*>(P.ws.seq + b);
    __stcg(dst, make_int4(rec.n, rec.status, 0, __float_as_int(rec.tau_d)));
    __stcg(reinterpret_cast<float4*>(dst + 1), make_float4(rec.mt, rec.lnSt, rec.cdelta, rec.tau_t));
  }
}

// Write one sequence's committed tokens with one warp.  token(i) is the i-th
// committed token, or -1 past the last; the row ends after the first token
// that is a stop id ("Speculative Decoding: ...", "Constraints must be
// applied consistently": nothing after an end-of-sequence token is kept).
// Returns the committed count.
template <class F>
__device__ int write_committed(const Params& P, int32_t* out, int width, F token) {
  const int lane = threadIdx.x & 31;
  int cut = INT_MAX;                                 // position of the first stop token
  if (P.n_stop > 0) {
    for (int base = 0; base < width && cut == INT_MAX; base += 32) {
      const int i = base + lane;
      bool stop = false;
      if (i < width) {
        const int v = token(i);
        if (v >= 0)
          for (int s = 0; s < P.n_stop; ++s) stop |= v == __ldg(P.stop_ids + s);
      }
      const unsigned m = __ballot_sync(0xffffffffu, stop);
      if (m) cut = base + __ffs(m) - 1;
    }
  }
  int count = 0;
  for (int base = 0; base < width; base += 32) {
    const int i = base + lane;
    int v = -1;
    if (i < width && i <= cut) v = token(i);
    if (i < width) out[i] = v;
    count += __popc(__ballot_sync(0xffffffffu, v >= 0));
  }
  return count;
}

// Greedy match: n = first i with x_i != argmax_i.  With a guide ("Double: ...",
// "Multi-token Pre-verify"), the correction is followed by the guide's tokens
// when the guide agrees with it.  Optionally the per-position matches
// ("Ouroboros: ...", Equation (10)), their count and the runs of matches after
// the first mismatch.
__device__ void greedy_match(const Params& P, int b) {
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const long long rbase = (long long)b * (k + 1);
  int n = k;
  unsigned tok_bad = 0, nf_bad = 0, to_bad = 0;
  for (int base = 0; base <= k; base += 32) {
    const int i = base + lane;
    bool mism = false, tbad = false, fbad = false, tmo = false;
    if (i <= k) {
      const RowStat rs = ldcg_stat(P.ws.row_stat + rbase + i);
      fbad = rs.status != SPEC_OK;
      tmo = rs.status == SPEC_ERR_TIMEOUT;
      if (i < k) {
        const int x = P.tokens[(size_t)b * k + i];
        tbad = x < 0 || x >= P.V;
        mism = x != rs.arg;
      }
    }
    tok_bad |= __ballot_sync(0xffffffffu, tbad);
    nf_bad |= __ballot_sync(0xffffffffu, fbad);
    to_bad |= __ballot_sync(0xffffffffu, tmo);
    const unsigned mm = __ballot_sync(0xffffffffu, mism);
    if (n == k && mm) n = base + __ffs(mm) - 1;
  }
  // the guide: ids must be in range; it continues the corrected path only if
  // it agrees with the correction, and it ends at its first negative entry
  const int an = ldcg_stat(P.ws.row_stat + rbase + n).arg;
  const int32_t* g = P.guide ? P.guide + (size_t)b * P.L : nullptr;
  int gend = n + 1;
  if (g) {
    unsigned gbad = 0;
    int first_neg = P.L;
    for (int base = 0; base < P.L; base += 32) {
      const int i = base + lane;
      const int v = i < P.L ? g[i] : 0;
      gbad |= __ballot_sync(0xffffffffu, v >= P.V);
      const unsigned neg = __ballot_sync(0xffffffffu, i < P.L && i > n && v < 0);
      if (neg && first_neg == P.L) first_neg = base + __ffs(neg) - 1;
    }
    tok_bad |= gbad;
    if (n < P.L && g[n] == an) gend = first_neg;
  }
  const int st = tok_bad ? SPEC_ERR_TOKEN : to_bad ? SPEC_ERR_TIMEOUT : nf_bad ? SPEC_ERR_NONFINITE : SPEC_OK;
  int32_t* out = P.out_tokens + (size_t)b * P.out_w;
  const int32_t* x = P.tokens + (size_t)b * k;
  const int committed = write_committed(P, out, P.out_w, [&](int i) -> int {
    if (st != SPEC_OK) return -1;
    if (i < n) return x[i];
    if (i == n) return an;
    return i < gend ? g[i] : -1;
  });
  if (P.match_mask || P.n_match || P.tail_runs) {
    int n_match = 0, runs = 0;
    unsigned carry = 1;                              // position -1 counts as a match
    for (int base = 0; base < k; base += 32) {
      const int i = base + lane;
      bool hit = false;
      if (i < k && st == SPEC_OK) hit = x[i] == ldcg_stat(P.ws.row_stat + rbase + i).arg;
      if (i < k && P.match_mask) P.match_mask[(size_t)b * k + i] = hit ? 1 : 0;
      const unsigned hits = __ballot_sync(0xffffffffu, hit);
      const unsigned starts = hits & ~((hits << 1) | carry);
      const unsigned after = __ballot_sync(0xffffffffu, i > n);
      n_match += __popc(hits);
      runs += __popc(starts & after);
      carry = hits >> 31;
    }
    if (lane == 0) {
      if (P.n_match) P.n_match[b] = st == SPEC_OK ? n_match : -1;
      if (P.tail_runs) P.tail_runs[b] = st == SPEC_OK ? runs : -1;
    }
  }
  if (lane == 0) {
    P.out_n[b] = st == SPEC_OK ? n : -1;
    if (P.n_committed) P.n_committed[b] = st == SPEC_OK ? committed : -1;
    if (P.status) P.status[b] = st;
  }
  __syncwarp();
  for (int i = lane; i <= k; i += 32) stcg_stat(P.ws.row_stat + rbase + i, RowStat{0.f, 0.f, 0, 0});
}

// Greedy tree verification.  Node m is accepted iff its parent is (the context
// is) and its token is the argmax of the parent's row; the deepest accepted
// node wins, the lowest index among equals.
__device__ void tree_walk(const Params& P, int b) {
  __shared__ short s_par[SPEC_MAX_TREE_N];
  __shared__ short s_dep[SPEC_MAX_TREE_N];  // ok flag, then depth if accepted (0 if not)
  const int lane = threadIdx.x & 31;
  const int N = P.k;
  const long long rbase = (long long)b * (N + 1);
  int tbad = 0, fbad = 0;
  for (int m = lane; m < N; m += 32) {
    const int par = P.parents[(size_t)b * N + m];
    const int tok = P.tokens[(size_t)b * N + m];
    const bool ok_shape = par >= -1 && par < m && tok >= 0 && tok < P.V;
    tbad |= !ok_shape;
    int ok = 0;
    if (ok_shape) ok = tok == ldcg_stat(P.ws.row_stat + rbase + (par < 0 ? 0 : par + 1)).arg;
    s_par[m] = (short)(ok_shape ? par : -1);
    s_dep[m] = (short)ok;
  }
  int tmo = 0;
  for (int r = lane; r <= N; r += 32) {
    const int rs = ldcg_stat(P.ws.row_stat + rbase + r).status;
    fbad |= rs != SPEC_OK;
    tmo |= rs == SPEC_ERR_TIMEOUT;
  }
  tbad = __any_sync(0xffffffffu, tbad);
  fbad = __any_sync(0xffffffffu, fbad);
  tmo = __any_sync(0xffffffffu, tmo);
  __syncwarp();
  int best = -1, best_d = 0;
  if (lane == 0) {
    for (int m = 0; m < N; ++m) {
      const int par = s_par[m];
      int d = 0;
      if (s_dep[m]) d = par < 0 ? 1 : (s_dep[par] > 0 ? s_dep[par] + 1 : 0);
      s_dep[m] = (short)d;
      if (d > best_d) { best_d = d; best = m; }
    }
  }
  best = __shfl_sync(0xffffffffu, best, 0);
  best_d = __shfl_sync(0xffffffffu, best_d, 0);
  __syncwarp();
  const int st = tbad ? SPEC_ERR_TOKEN : tmo ? SPEC_ERR_TIMEOUT : fbad ? SPEC_ERR_NONFINITE : SPEC_OK;
  int32_t* out = P.out_tokens + (size_t)b * (N + 1);
  for (int i = lane; i <= N; i += 32)
    if (st != SPEC_OK || i > best_d) out[i] = -1;
  if (lane == 0) {
    if (st == SPEC_OK) {
      out[best_d] = ldcg_stat(P.ws.row_stat + rbase + (best < 0 ? 0 : best + 1)).arg;
      for (int m = best, d = best_d - 1; m >= 0; m = s_par[m], --d) out[d] = P.tokens[(size_t)b * N + m];
    }
    P.out_n[b] = st == SPEC_OK ? best_d : -1;
    if (P.out_leaf) P.out_leaf[b] = st == SPEC_OK ? best : -1;
    if (P.status) P.status[b] = st;
  }
  __syncwarp();
  for (int r = lane; r <= N; r += 32) stcg_stat(P.ws.row_stat + rbase + r, RowStat{0.f, 0.f, 0, 0});
}

// A row's last piece has landed: merge its partials into the row statistics
// (warp 0); if that completes the sequence, run its per-sequence step.
template <typename T, int kMode>
__device__ void finish_row(const Params& P, long long r, int b) {
  const int lane = threadIdx.x & 31;
  __threadfence();
  float4* src = reinterpret_cast<float4*>(P.ws.row_partial + r * P.nt);
  float m = -CUDART_INF_F, s = 0.f;
  int ix = INT_MAX, bad = 0, tmo = 0;
  for (int t = lane; t < P.nt; t += 32) {
    const float4 p = __ldcg(src + t);
    __stcg(src + t, make_float4(0.f, 0.f, 0.f, 0.f));  // read for the last time: the workspace is left zeroed
    if (p.w != 0.f) { tmo = 1; continue; }          // a piece whose data never arrived
    if (p.x != p.x) { bad = 1; continue; }
    if constexpr (kMode == kStochastic) {
      const float M = fmaxf(m, p.x);
      s = rescale(s, m, M, P.c) + rescale(p.y, p.x, M, P.c);
    } else {
      const int pi = __float_as_int(p.z);
      if (beats(p.x, pi, m, ix)) ix = pi;
    }
    m = fmaxf(m, p.x);
  }
  RowStat st;
  if constexpr (kMode == kStochastic) {
    const float M = warp_max(m);
    s = warp_sum(rescale(s, m, M, P.c));
    bad = __any_sync(0xffffffffu, bad);
    tmo = __any_sync(0xffffffffu, tmo);
    const bool finite = M > -CUDART_INF_F && M < CUDART_INF_F && s > 0.f && s < CUDART_INF_F;
    // (stochastic rows need no argmax)
    st = RowStat{M, logf(s), 0, tmo ? SPEC_ERR_TIMEOUT : (bad || !finite) ? SPEC_ERR_NONFINITE : SPEC_OK};
  } else {
    warp_argmax(m, ix);
    bad = __any_sync(0xffffffffu, bad);
    tmo = __any_sync(0xffffffffu, tmo);
    st = RowStat{m, 0.f, ix, tmo ? SPEC_ERR_TIMEOUT : bad ? SPEC_ERR_NONFINITE : SPEC_OK};
  }
  if (kMode == kStochastic && P.filtering) {
    // the filter pass takes the row from here and runs the accept scan
    if (lane == 0) {
      stcg_stat(P.ws.row_stat + r, st);
      P.ws.row_cnt[r] = 0;
    }
    return;
  }
  int last = 0;
  if (lane == 0) {
    stcg_stat(P.ws.row_stat + r, st);
    P.ws.row_cnt[r] = 0;  // ready for the next call
    __threadfence();
    const unsigned old = atomicAdd(P.ws.seq_cnt + b, 1u);
    last = old + 1 == (unsigned)P.rows_per_seq;
    if (last) P.ws.seq_cnt[b] = 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  if constexpr (kMode == kTree) tree_walk(P, b);
  else if constexpr (kMode == kStochastic) accept_scan<T>(P, b);
  else greedy_match(P, b);
}

// --------------------------------------------------------------- row pass ---

// A CTA has finished its piece [t0, t1) of row r with partial `part`: store it
// (the piece's other tiles get a neutral partial) and, if that completes the
// row, merge the row in warp 0.
template <typename T, int kMode>
__device__ __forceinline__ void end_piece(const Params& P, long long r, int b, int t0, int t1, const float4& part) {
  if (threadIdx.x >= 32) return;
  int last = 0;
  if (threadIdx.x == 0) {
    float4* dst = reinterpret_cast<float4*>(P.ws.row_partial + r * P.nt);
    __stcg(dst + t0, part);
    // the piece's other tiles: nothing to add to the sums or the argmax
    const float4 neutral = make_float4(-CUDART_INF_F, 0.f, __int_as_float(INT_MAX), 0.f);
    for (int u = t0 + 1; u < t1; ++u) __stcg(dst + u, neutral);
    __threadfence();
    const unsigned add = (unsigned)(t1 - t0);
    last = atomicAdd(P.ws.row_cnt + r, add) + add == (unsigned)P.nt;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) finish_row<T, kMode>(P, r, b);
}

// Resident CTAs per SM the row pass is compiled for. Six 256-thread CTAs of
// 16-bit rows (40 registers a thread, no spills) keep more loads in flight than
// the four the default register budget allows; fp32 rows keep four, since their
// argmax modes would spill at six.
template <typename T>
constexpr int kRowPassMinCtas = sizeof(T) == 2 ? 6 : 4;

template <typename T, int kMode>
__global__ void __launch_bounds__(kThreads, kRowPassMinCtas<T>) row_pass_kernel(const Params P) {
  __shared__ BlockScratch sh;
  // the sampling launch may be scheduled as this grid's CTAs retire; it waits
  // for this grid's results before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) sh.flag = 0;
  __syncthreads();
  const long long I = P.R * P.nt;
  const long long i0 = I * blockIdx.x / gridDim.x;
  const long long i1 = I * (blockIdx.x + 1) / gridDim.x;
  for (long long i = i0; i < i1;) {
    const long long r = i / P.nt;
    const int t0 = (int)(i % P.nt);
    const int t1 = (int)min((long long)P.nt, (long long)t0 + (i1 - i));
    int b;
    const T* row = row_ptr<T, kMode>(P, r, b);
    const int e0 = t0 * kPartTile, e1 = min(P.V, t1 * kPartTile);
    float4 part;
    if constexpr (kMode == kStochastic) {
      LseAcc acc;
      acc.init(P.c);
      scan_segment<T>(row, e0, e1, acc);
      float m = acc.m, s = acc.sum();
      int bad = acc.bad;
      block_lse_flag(m, s, bad, P.c, sh);
      part = make_float4(bad ? CUDART_NAN_F : m, s, __int_as_float(INT_MAX), 0.f);
    } else {
      ArgmaxAcc acc;
      acc.init();
      scan_segment<T>(row, e0, e1, acc);
      float v = acc.bv;
      int ix = acc.bi, bad = acc.bad;
      block_argmax_flag(v, ix, bad, sh);
      part = make_float4(bad ? CUDART_NAN_F : v, 0.f, __int_as_float(ix), 0.f);
    }
    end_piece<T, kMode>(P, r, b, t0, t1, part);
    __syncthreads();
    i += t1 - t0;
  }
}

// ------------------------------------------------ row pass, bulk-copy ring ---
//
// For greedy and tree verification, when every row starts on a 16-byte
// boundary, the row pass stages its data in shared memory with bulk copies.
// A producer warp keeps kRingStages copies of up to kRingBytes of the CTA's
// range in flight, each completing on its stage's "full" barrier; the eight
// consumer warps fold a stage from shared memory and release it on its
// "empty" barrier.  The bytes in flight per SM are then set by the ring, not
// by how many loads a thread can hold in registers.  Ranges, pieces, partials
// and the completion steps are those of the register row pass above.  Every
// wait is bounded: a wait that runs out stops the producer, marks the CTA's
// remaining pieces as timed out (their rows and sequences get
// SPEC_ERR_TIMEOUT) and, before the CTA leaves, the producer waits (bounded)
// for the copies it has in flight.
constexpr int kRingStages = 3;
constexpr int kRingBytes = 16384;
constexpr int kRingThreads = kThreads + 32;   // eight consumer warps, one producer warp
constexpr int kRingMinCtas = 4;
constexpr double kRingMinBytes = 134217728.0;   // 128 MiB of rows

struct RingSmem {
  alignas(128) unsigned char buf[kRingStages][kRingBytes];
  uint64_t full[kRingStages];
  uint64_t empty[kRingStages];
  int abort;   // a wait ran out: the rest of the range is marked as timed out
};

// Piece walk shared by the producer and the consumers: the CTA's tiles
// [i, i1) of the virtual row list, cut at row ends.
struct PieceWalk {
  long long i, i1;
  __device__ PieceWalk(const Params& P) {
    const long long I = P.R * P.nt;
    i = I * blockIdx.x / gridDim.x;
    i1 = I * (blockIdx.x + 1) / gridDim.x;
  }
};

template <typename T, int kMode>
__global__ void __launch_bounds__(kRingThreads, kRingMinCtas) row_pass_ring(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  RingSmem& S = *reinterpret_cast<RingSmem*>(dyn_smem);
  __shared__ BlockScratch sh;
  // the sampling launch may be scheduled as this grid's CTAs retire; it waits
  // for this grid's results before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRingStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kWarps);
    }
    fence_mbar_init();
    S.abort = 0;
  }
  __syncthreads();

  if (warp == kWarps) {
    // producer: one lane issues the copies, kRingStages ahead of the consumers
    if (lane != 0) return;
    long long q = 0;
    PieceWalk w(P);
    while (w.i < w.i1 && !*(volatile int*)&S.abort) {
      const long long r = w.i / P.nt;
      const int t0 = (int)(w.i % P.nt);
      const int t1 = (int)min((long long)P.nt, (long long)t0 + (w.i1 - w.i));
      int b;
      const unsigned char* row = reinterpret_cast<const unsigned char*>(row_ptr<T, kMode>(P, r, b));
      const size_t x0 = (size_t)t0 * kPartTile * sizeof(T);
      const size_t x1 = (size_t)min(P.V, t1 * kPartTile) * sizeof(T);
      for (size_t x = x0; x < x1 && !S.abort; x += kRingBytes, ++q) {
        const int s = (int)(q % kRingStages);
        // a consumer that gave up releases no stage: stop waiting when it says so
        if (q >= kRingStages &&
            !mbar_wait_bounded_unless(&S.empty[s], (unsigned)((q / kRingStages) - 1) & 1u, &S.abort)) {
          S.abort = 1;
          break;
        }
        fence_proxy_async_smem();
        const unsigned nb = (unsigned)min((size_t)kRingBytes, x1 - x);
        mbar_arrive_tx(&S.full[s], nb);
        bulk_copy_g2s(S.buf[s], row + x, nb, &S.full[s]);
      }
      w.i += t1 - t0;
    }
    if (*(volatile int*)&S.abort) {
      // leave no copy in flight into this CTA's shared memory (bounded)
      for (long long x = q - 1; x >= 0 && x >= q - kRingStages; --x)
        mbar_wait_bounded(&S.full[x % kRingStages], (unsigned)(x / kRingStages) & 1u);
    }
    return;
  }

  // consumers: fold each stage, release it, and end each piece as the register
  // row pass does
  constexpr int kVec = Vec<T>::n;
  constexpr int kPer = kRingBytes / 16 / kThreads;   // 16-byte vectors per thread per full stage
  long long q = 0;
  PieceWalk w(P);
  while (w.i < w.i1) {
    const long long r = w.i / P.nt;
    const int t0 = (int)(w.i % P.nt);
    const int t1 = (int)min((long long)P.nt, (long long)t0 + (w.i1 - w.i));
    int b;
    row_ptr<T, kMode>(P, r, b);
    const int e0 = t0 * kPartTile, e1 = min(P.V, t1 * kPartTile);
    constexpr int kStageElems = kRingBytes / (int)sizeof(T);
    LseAcc lacc;
    ArgmaxAcc aacc;
    if constexpr (kMode == kStochastic) lacc.init(P.c);
    else aacc.init();
    for (int ex = e0; ex < e1; ex += kStageElems, ++q) {
      const int s = (int)(q % kRingStages);
      if (!*(volatile int*)&S.abort &&
          (P.force_timeout || !mbar_wait_bounded(&S.full[s], (unsigned)(q / kRingStages) & 1u)))
        S.abort = 1;
      // one decision per warp, so that every lane reaches the same __syncwarp
      if (__any_sync(0xffffffffu, *(volatile int*)&S.abort != 0)) continue;
      const uint4* sv = reinterpret_cast<const uint4*>(S.buf[s]);
      const int nvec = min(kStageElems, e1 - ex) / kVec;
      if (nvec == kPer * kThreads) {
        uint4 v[kPer];
        int idx[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          v[u] = sv[u * kThreads + threadIdx.x];
          idx[u] = ex + (u * kThreads + threadIdx.x) * kVec;
        }
        if constexpr (kMode == kStochastic) lacc.template vec<T, kPer>(v, idx);
        else aacc.template vec<T, kPer>(v, idx);
      } else {
        for (int j = threadIdx.x; j < nvec; j += kThreads) {
          uint4 v[1] = {sv[j]};
          int idx[1] = {ex + j * kVec};
          if constexpr (kMode == kStochastic) lacc.template vec<T, 1>(v, idx);
          else aacc.template vec<T, 1>(v, idx);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
    }
    // after the reduction's barriers every skipped stage has set the flag: a
    // piece that lost data is marked timed out
    float4 part;
    if constexpr (kMode == kStochastic) {
      float m = lacc.m, sum = lacc.sum();
      int bad = lacc.bad;
      block_lse_flag<true>(m, sum, bad, P.c, sh);
      part = make_float4(bad ? CUDART_NAN_F : m, sum, __int_as_float(INT_MAX), 0.f);
    } else {
      float v = aacc.bv;
      int ix = aacc.bi, bad = aacc.bad;
      block_argmax_flag<true>(v, ix, bad, sh);
      part = make_float4(bad ? CUDART_NAN_F : v, 0.f, __int_as_float(ix), 0.f);
    }
    if (*(volatile int*)&S.abort) part.w = 1.f;
    // warp 0 stores the partial (and merges a completed row) while the other
    // consumer warps go on: the next reduction's barriers order the scratch
    end_piece<T, kMode>(P, r, b, t0, t1, part);
    w.i += t1 - t0;
  }
}

// ------------------------------------------------------------- filtering ---
// Consistent top-k / top-p ("Speculative Decoding: ...", "Logit-processor
// gaps" and "Constraints must be applied consistently"; the Ouroboros page
// samples with top-p 0.8): every target and draft row of a sequence goes
// through the same filter before the rule.  Order: temperature, top-k, then
// top-p on the top-k distribution.  Both are value thresholds, so ties at a
// threshold are kept.  One CTA per row -- or a cluster of CTAs, each scanning
// one segment of the row, their histograms summed at the cluster's first CTA
// through distributed shared memory (filter_cluster_ctas says when) -- finds
// each threshold in two steps:
//   1. histograms of count and mass exp((x - m) / T) by distance below the row
//      max (m from the row pass) pick the bin where the count (top-k) or the
//      mass (top-p) summed from the top first reaches its target.  The bins
//      are 1/170 nat wide over the first 12 nats, where nearly all the mass
//      lies; ids further down are only counted, in registers, and a target that
//      lies further down is found in a second or third window of coarser bins.
//      Only the ids near the top take shared-memory atomics, spread over many
//      bins.
//   2. the bin holds a contiguous range of order-preserving keys of the raw
//      logits, found by a parallel search; when it spans fewer than 2048 keys
//      (always for bf16 near the top) one pass histograms key - smallest,
//      otherwise radix rounds over the key bits (11 a round) decide the exact
//      value.
// Every pass tests each 16-byte vector first, from its largest and smallest
// logit, and only vectors that straddle a boundary take the per-id test.
// Masses are summed as 64-bit fixed point (2^-40 units) with 32-bit integer
// atomics, exactly and in any order.  Top-p after top-k reuses the top-k
// pass's window-0 histogram when the top-k key was found there.

constexpr int kHistBits = 11;
constexpr int kHistBins = 1 << kHistBits;

template <typename T>
struct Keys;
template <>
struct Keys<uint16_t> {
  static constexpr int kBits = 16;
  __device__ static uint32_t of(float x) {
    const uint32_t h = __float_as_uint(x) >> 16;
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
  }
  __device__ static float value(uint32_t k) {
    return __uint_as_float(((k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu)) << 16);
  }
};
template <>
struct Keys<float> {
  static constexpr int kBits = 32;
  __device__ static uint32_t of(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  __device__ static float value(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k); }
};

constexpr int kDistBins = 2048;            // step 1: bin 0 = the window's tail, bins 1..2047 (2047 = the top)
constexpr int kWindows = 3;
static_assert(kDistBins <= kHistBins, "the distance histogram shares the radix histogram's storage");

// Step 1 looks at the scaled distance d = (m - x) / T >= 0 below the row max in
// windows: window 0 has bins of 1/170 nat over its first 2047/170 (12) nats,
// window 1 bins of 1/8 nat over the next 2047/8, window 2 bins of 2 nats beyond.
__device__ __forceinline__ float win_scale(int w) { return w == 0 ? 170.f : (w == 1 ? 8.f : 0.5f); }
__device__ __forceinline__ float win_start(int w) {
  return w == 0 ? 0.f : (w == 1 ? 2047.f / 170.f : 2047.f / 170.f + 2047.f / 8.f);
}

// Window w of a row as an affine map of the logit: its scaled position of x is
// s_w(x) = fma(-x, a, b) = ((m - x) / T - start_w) * scale_w, rounded once and
// non-increasing in x.  Window w begins where window w - 1's tail begins, so an
// id outside window w - 1's tail lies above window w (and every earlier
// window's tail holds window w - 1's).
struct WinMap {
  float ap, bp;       // window w - 1 (w > 0)
  float a, b;         // window w
  bool first;         // w == 0
  __device__ WinMap(float m, float invT, int w) : first(w == 0) {
    const int p = w > 0 ? w - 1 : 0;
    a = invT * win_scale(w);
    b = (m * invT - win_start(w)) * win_scale(w);
    ap = invT * win_scale(p);
    bp = (m * invT - win_start(p)) * win_scale(p);
  }
  __device__ __forceinline__ bool above(float x) const {
    return !first && !(fmaf(-x, ap, bp) >= (float)(kDistBins - 1));
  }
  // kDistBins above the window, 0 in its tail, else its bin 1..2047.
  // Non-decreasing in x.
  __device__ __forceinline__ int bin(float x) const {
    if (above(x)) return kDistBins;
    const float s = fmaxf(fmaf(-x, a, b), 0.f);
    return s < (float)(kDistBins - 1) ? (kDistBins - 1) - (int)s : 0;
  }
};

// Largest and smallest logit of a 16-byte vector (the rows the filter sees
// hold no NaN: a row with one reports an error and is not filtered).
template <typename T>
__device__ __forceinline__ void vec_range(const uint4& v, float& hi, float& lo) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t mx = bf16x2_nanmax(bf16x2_nanmax(v.x, v.y), bf16x2_nanmax(v.z, v.w));
    const uint32_t mn = bf16x2_min(bf16x2_min(v.x, v.y), bf16x2_min(v.z, v.w));
    hi = fmaxf(bf16_lo(mx), bf16_hi(mx));
    lo = fminf(bf16_lo(mn), bf16_hi(mn));
  } else {
    hi = fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    lo = fminf(fminf(__uint_as_float(v.x), __uint_as_float(v.y)), fminf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
}

// The histogram passes test each 16-byte vector first (from its largest and
// smallest logit): most vectors take no part or are counted whole.  The rest
// of a batch go into the warp's queue, and then the warp's lanes share their
// ids out, so the per-id test runs with every lane busy, one queue run (two
// warp syncs) per batch.  Only scan_segment's full batches come here: every
// thread of the CTA takes part in them, as the warp-wide ballot and syncs
// need; its remainder loop, where a warp may be partly idle, tests every id.
// The queues (a batch's vectors for each warp, 32 KB) leave room for four CTAs
// per SM, at up to 64 registers; a queue run per vector (4 KB of queues, six
// CTAs of 40 registers) took 94.9 us for top-p 0.8 on 64 x 17 rows of 128256
// bf16 logits, against 86.0 us now.
// Queue one vector of a batch (slow: it needs the per-id test); `fill` counts
// the warp's queued vectors.
__device__ __forceinline__ void warp_queue_put(uint4* q, int& fill, const uint4& v, bool slow) {
  const int lane = threadIdx.x & 31;
  const unsigned m = __ballot_sync(0xffffffffu, slow);
  if (slow) q[fill + __popc(m & ((1u << lane) - 1u))] = v;
  fill += __popc(m);
}
// Run the per-id test on the batch's queued vectors, the lanes sharing the ids.
template <typename T, class Acc>
__device__ __forceinline__ void warp_queue_run(Acc& acc, const uint4* q, int fill) {
  if (!fill) return;
  const int lane = threadIdx.x & 31;
  __syncwarp();
  const int n = fill * Vec<T>::n;
  for (int i = lane; i < n; i += 32) acc.elem(Vec<T>::at(q[i / Vec<T>::n], i % Vec<T>::n));
  __syncwarp();                          // the queue is refilled by the next batch
}

constexpr float kMassUnit = 1099511627776.0f;   // 2^40: fixed-point scale of a mass in (0, 1]

struct FilterScratch {
  uint32_t cnt[kHistBins];
  float mass[kHistBins];
  // fixed-point sums of the masses (2^-40 units, exact and independent of the
  // order of the adds) as 32-bit halves, turned into `mass` after a pass
  uint32_t mlo[kHistBins], mhi[kHistBins];
  uint32_t wc[kWarps];
  float wm[kWarps];
  uint4 vq[kWarps][kUnroll * 32];        // per warp: a batch's 16-byte vectors that need the per-id test
  // select_bin's result (six words, sent to the cluster's other CTAs as such)
  int sel_bin;
  uint32_t sel_cnt_above, sel_cnt_bin, total_cnt;
  float sel_mass_above, sel_mass_bin;
};
constexpr int kPickWords = 6;
static_assert(offsetof(FilterScratch, sel_mass_bin) - offsetof(FilterScratch, sel_bin) == (kPickWords - 1) * 4,
              "the pick is six consecutive words");

// The filter's scratch, named at file scope so that the out-of-line threshold
// search addresses it as shared memory (32-bit addresses, shared-memory
// atomics) rather than through a generic pointer.
__shared__ FilterScratch filter_scratch;

__device__ __forceinline__ void clear_hist(FilterScratch& S, int nbins) {
  for (int i = threadIdx.x; i < nbins; i += kThreads) {
    S.cnt[i] = 0u;
    S.mlo[i] = 0u;
    S.mhi[i] = 0u;
    S.mass[i] = 0.f;
  }
}

__device__ __forceinline__ void fix_masses(FilterScratch& S, int nbins) {
  for (int i = threadIdx.x; i < nbins; i += kThreads)
    if (S.mlo[i] | S.mhi[i])
      S.mass[i] = (float)(((unsigned long long)S.mhi[i] << 32) | S.mlo[i]) * (1.0f / kMassUnit);
}

// Add one id's mass (in (0, 1]) to a bin: the 32-bit low half with an atomic
// that returns the old value, so the one add that wraps it carries into the
// high half.  Native 32-bit atomics; a 64-bit shared-memory add loses far more
// under contention (a pass where every id of a row lands in the window).
__device__ __forceinline__ void add_mass(FilterScratch& S, int bin, float mass) {
  const unsigned long long q = (unsigned long long)(mass * kMassUnit);
  const uint32_t ql = (uint32_t)q, qh = (uint32_t)(q >> 32);
  uint32_t carry = 0u;
  if (ql) {
    const uint32_t old = atomicAdd(&S.mlo[bin], ql);
    carry = old + ql < old;
  }
  if (qh + carry) atomicAdd(&S.mhi[bin], qh + carry);
}

// A row is cut into `nrank` consecutive segments, one per CTA of a cluster,
// and each CTA scans its segment into its own histogram.  Then:
//   hist_merge   once every CTA has finished its scan (so rank 0's own
//                shared-memory atomics are done), adds this CTA's non-empty
//                bins into rank 0's histogram through distributed shared
//                memory, and waits until every CTA has added;
//   pick_share   after rank 0 has picked the bin: rank 0 writes the pick into
//                the other CTAs' scratch, and all wait for it.
// Every CTA of a cluster makes the same calls in the same order: the control
// flow depends only on the row's statistics and on the picks, which all of the
// cluster's CTAs hold alike.  With one CTA the calls do nothing.
__device__ __forceinline__ void hist_merge(FilterScratch& S, int nbins, unsigned rank, unsigned nrank) {
  if (nrank == 1) return;
  cluster_arrive();
  cluster_wait();                                   // every scan is done
  if (rank != 0) {
    for (int i = threadIdx.x; i < nbins; i += kThreads) {
      const uint32_t c = S.cnt[i];
      if (!c) continue;
      cluster_red_add(cluster_map(&S.cnt[i], 0), c);
      const uint32_t ql = S.mlo[i], qh = S.mhi[i];
      uint32_t carry = 0u;
      if (ql) {
        const uint32_t old = cluster_atom_add(cluster_map(&S.mlo[i], 0), ql);
        carry = old + ql < old;
      }
      if (qh + carry) cluster_red_add(cluster_map(&S.mhi[i], 0), qh + carry);
    }
  }
  cluster_arrive();
  cluster_wait();                                   // every CTA's bins are in
}

__device__ __forceinline__ void pick_share(FilterScratch& S, unsigned rank, unsigned nrank) {
  if (nrank == 1) return;
  const int t = threadIdx.x;
  if (rank == 0 && t < (int)(nrank - 1) * kPickWords) {
    const uint32_t* words = reinterpret_cast<const uint32_t*>(&S.sel_bin);
    cluster_store(cluster_map(&words[t % kPickWords], 1 + t / kPickWords), words[t % kPickWords]);
  }
  cluster_arrive();
  cluster_wait();
}

// Step 2's histogram over the ids with keys in [klo, khi], fed by scan_segment:
// one round over key - klo when the range is under kHistBins keys, otherwise
// radix rounds over the key bits from the top.
template <typename T>
struct HistAcc {
  FilterScratch* S;
  uint32_t klo, khi;  // the ids taking part
  bool one_round;
  uint32_t prefix;    // radix rounds: the key bits decided so far
  int shift_hi;       //   at key bits [shift_hi, kBits); kBits: none yet
  int shift_lo;       //   this round's bits are [shift_lo, shift_hi)
  float c, mc;        // mass = exp2(x c - mc) = exp((x - m) / T)
  __device__ __forceinline__ void elem(float x) {
    if (!(x > -CUDART_INF_F)) return;                  // -inf ids are never kept
    const uint32_t key = Keys<T>::of(x);
    if (key < klo || key > khi) return;
    uint32_t bin;
    if (one_round) {
      bin = key - klo;
    } else {
      if (shift_hi < Keys<T>::kBits && (key >> shift_hi) != prefix) return;
      bin = (key >> shift_lo) & ((1u << (shift_hi - shift_lo)) - 1u);
    }
    atomicAdd(&S->cnt[bin], 1u);
    add_mass(*S, bin, ex2_approx(fmaf(x, c, -mc)));
  }
  template <typename TT, int U>
  __device__ __forceinline__ void vec(const uint4 (&v)[U], const int (&)[U]) {
    if constexpr (U == kUnroll) {
      uint4* q = S->vq[threadIdx.x >> 5];
      int fill = 0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        // keys are ordered like the logits: a vector whose largest key lies
        // below the range, or whose smallest lies above it, takes no part
        float hi, lo;
        vec_range<T>(v[u], hi, lo);
        warp_queue_put(q, fill, v[u], !(Keys<T>::of(hi) < klo || Keys<T>::of(lo) > khi));
      }
      warp_queue_run<T>(*this, q, fill);
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < Vec<T>::n; ++e) elem(Vec<T>::at(v[u], e));
    }
  }
  __device__ __forceinline__ void scalar(float x, int) { elem(x); }
};

// The bin where the count (by_mass false) or the mass, summed from the top
// bin down, first reaches `need` (clamped to the total), with the count and
// mass of the bins above it and of the bin itself.  With `tail_unsummed`,
// bin 0 is the window's tail, counted but without its mass: a mass target
// above the other bins' total lies in the tail, and bin 0 is the pick.  All
// threads call it.
__device__ void select_bin(FilterScratch& S, int nbins, bool by_mass, bool tail_unsummed, uint32_t need_cnt,
                           float need_mass) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int per = nbins >= kThreads ? nbins / kThreads : 1;
  const int owners = nbins / per;
  const int t = threadIdx.x;
  uint32_t lc = 0;
  float lm = 0.f;
  if (t < owners)
    for (int j = 0; j < per; ++j) {
      const int bin = nbins - 1 - (t * per + j);
      lc += S.cnt[bin];
      lm += S.mass[bin];
    }
  // inclusive scan in thread order (thread 0 holds the top bins)
  uint32_t ic = lc;
  float im = lm;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t c2 = __shfl_up_sync(0xffffffffu, ic, o);
    const float m2 = __shfl_up_sync(0xffffffffu, im, o);
    if (lane >= o) { ic += c2; im += m2; }
  }
  if (lane == 31) { S.wc[w] = ic; S.wm[w] = im; }
  __syncthreads();
  uint32_t oc = 0;
  float om = 0.f;
  for (int q = 0; q < w; ++q) { oc += S.wc[q]; om += S.wm[q]; }
  ic += oc;
  im += om;
  const uint32_t ec = ic - lc;                         // exact for counts
  float em = __shfl_up_sync(0xffffffffu, im, 1);
  if (lane == 0) em = om;
  // totals as the last owner's inclusive values, so the comparisons below agree with them
  __syncthreads();
  if (t == owners - 1) { S.wc[0] = ic; S.wm[0] = im; }
  __syncthreads();
  const uint32_t tc = S.wc[0];
  const float tm = S.wm[0];
  bool mine;
  if (by_mass && tail_unsummed && need_mass > tm && S.cnt[0] > 0u) {
    mine = false;
    if (t == 0) {
      S.sel_bin = 0;
      S.sel_cnt_above = tc - S.cnt[0];
      S.sel_mass_above = tm;
      S.sel_cnt_bin = S.cnt[0];
      S.sel_mass_bin = 0.f;
    }
  } else if (by_mass) {
    const float need = fminf(need_mass, tm);
    mine = t < owners && lc > 0 && em < need && need <= im;
    if (!(tm > 0.f)) mine = t < owners && lc > 0 && ec + lc == tc;   // no mass seen: the lowest non-empty bin
  } else {
    const uint32_t need = min(need_cnt, tc);
    mine = t < owners && lc > 0 && ec < need && need <= ic;
  }
  if (mine) {
    uint32_t c = ec;
    float mm = em;
    int pick = -1, last_nonzero = -1;
    uint32_t pc = 0;
    float pm = 0.f;
    for (int j = 0; j < per; ++j) {
      const int bin = nbins - 1 - (t * per + j);
      const uint32_t bc = S.cnt[bin];
      const float bm = S.mass[bin];
      if (bc) { last_nonzero = bin; pc = c; pm = mm; }
      if (bc && (by_mass ? (tm > 0.f && mm + bm >= fminf(need_mass, tm)) : (c + bc >= min(need_cnt, tc)))) {
        pick = bin;
        break;
      }
      c += bc;
      mm += bm;
    }
    if (pick < 0) pick = last_nonzero;                // rounding left the target a hair above: the last bin
    else { pc = c; pm = mm; }
    S.sel_bin = pick;
    S.sel_cnt_above = pc;
    S.sel_mass_above = pm;
    S.sel_cnt_bin = S.cnt[pick];
    S.sel_mass_bin = S.mass[pick];
  }
  if (t == 0) S.total_cnt = tc;
  __syncthreads();
}

// Step 1's histogram for one window, fed by scan_segment (kFirst: window 0,
// which has no earlier window above it).
template <typename T, bool kFirst>
struct DistAcc {
  FilterScratch* S;
  uint32_t key_min;   // ids with smaller keys take no part (0: every id)
  float c, mc;        // mass = exp2(x c - mc) = exp((x - m) / T)
  WinMap W;
  uint32_t tail_cnt;
  // Above the window: nothing (an earlier window has it); in its tail:
  // counted; else its bin takes the id's count and mass.
  __device__ __forceinline__ void elem(float x) {
    if (!(x > -CUDART_INF_F)) return;                  // -inf ids are never kept
    if (key_min != 0u && Keys<T>::of(x) < key_min) return;
    if (!kFirst && W.above(x)) return;
    const float s = fmaf(-x, W.a, W.b);
    if (!(s < (float)(kDistBins - 1))) {
      ++tail_cnt;
      return;
    }
    const int bin = (kDistBins - 1) - (int)fmaxf(s, 0.f);
    atomicAdd(&S->cnt[bin], 1u);
    add_mass(*S, bin, ex2_approx(fmaf(x, c, -mc)));
  }
  template <typename TT, int U>
  __device__ __forceinline__ void vec(const uint4 (&v)[U], const int (&)[U]) {
    if constexpr (U == kUnroll) {
      uint4* q = S->vq[threadIdx.x >> 5];
      int fill = 0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        // the window's position and the key are monotone in the logit, so the
        // largest and smallest logit decide for the whole vector when: every
        // id lies below key_min or above the window (nothing to do), or every
        // id takes part and lies in the window's tail (counted at once)
        float hi, lo;
        vec_range<T>(v[u], hi, lo);
        const bool none = (key_min != 0u && Keys<T>::of(hi) < key_min) || (!kFirst && W.above(lo));
        const bool tail = lo > -CUDART_INF_F && (key_min == 0u || Keys<T>::of(lo) >= key_min) &&
                          !(fmaf(-hi, W.a, W.b) < (float)(kDistBins - 1));
        if (!none && tail) tail_cnt += Vec<T>::n;
        warp_queue_put(q, fill, v[u], !none && !tail);
      }
      warp_queue_run<T>(*this, q, fill);
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < Vec<T>::n; ++e) elem(Vec<T>::at(v[u], e));
    }
  }
  __device__ __forceinline__ void scalar(float x, int) { elem(x); }
};

// The smallest k in [l, h) with pred(k), else h, for a predicate that is
// false and then true over the range.  All threads call it: each round tests
// kThreads evenly spaced keys at once and keeps the one gap that holds the
// change (two rounds for 16-bit keys, four or five for 32-bit ones).
template <class Pred>
__device__ uint32_t first_true(uint32_t l, uint32_t h, Pred pred) {
  while (l < h) {
    const uint64_t step = ((uint64_t)(h - l) + kThreads - 1) / kThreads;
    const uint64_t q = (uint64_t)l + (uint64_t)threadIdx.x * step;
    const int f = __syncthreads_count(q < h && !pred((uint32_t)q));
    if (f == 0) return l;
    // tests 0..f-1 false, test f (where it lies below h) true
    const uint64_t nh = (uint64_t)l + (uint64_t)f * step;
    l = (uint32_t)((uint64_t)l + (uint64_t)(f - 1) * step + 1);
    if (nh < h) h = (uint32_t)nh;
  }
  return h;
}

// The largest key whose count (by_mass false) or mass of ids at or above it,
// among the ids with key >= key_min, reaches the target.  Returns false when
// the count target is at least the number of those ids (no threshold).
// `reuse_w0`: the scratch already holds window 0's histogram of every id of
// the row (a previous call left it, `left_w0`); ids with keys below key_min
// then sit in bins below the target's, so the first pass is not repeated.
// Kept out of line: the filter calls it twice (top-k, then top-p), and one
// copy of its histogram loops instead of two cut the filter's
// instruction-fetch stalls (measured 118.4 -> 94.5 us on C3 with top-p 0.8).
template <typename T>
__device__ __noinline__ bool find_threshold(const T* row, int e0, int e1, unsigned rank, unsigned nrank, const Params& P,
                                            const RowStat& rs, bool by_mass, uint32_t need_cnt, float need_mass,
                                            uint32_t key_min, bool reuse_w0, uint32_t& key, float& mass_ge,
                                            bool& left_w0) {
  FilterScratch& S = filter_scratch;
  left_w0 = false;
  // step 1: the distance bin, window by window until the target falls in a bin
  uint32_t cnt_above = 0;
  float mass_above = 0.f, bin_mass = 0.f;
  int win = 0, dbin = 0;
  for (; win < kWindows; ++win) {
    if (win > 0 || !reuse_w0) {
      clear_hist(S, kDistBins);
      __syncthreads();
      uint32_t tail = 0;
      if (win == 0) {
        DistAcc<T, true> da{&S, key_min, P.c, rs.m * P.c, WinMap(rs.m, P.invT, 0), 0u};
        scan_segment<T>(row, e0, e1, da);
        tail = da.tail_cnt;
      } else {
        DistAcc<T, false> da{&S, key_min, P.c, rs.m * P.c, WinMap(rs.m, P.invT, win), 0u};
        scan_segment<T>(row, e0, e1, da);
        tail = da.tail_cnt;
      }
      const uint32_t tc = __reduce_add_sync(0xffffffffu, tail);
      if ((threadIdx.x & 31) == 0 && tc) atomicAdd(&S.cnt[0], tc);
      __syncthreads();
      hist_merge(S, kDistBins, rank, nrank);
      if (rank == 0) {
        fix_masses(S, kDistBins);
        __syncthreads();
      }
    }
    if (rank == 0) {
      // the tail's mass is not summed: a mass target beyond the other bins'
      // total lands on the tail, and the next window takes it up
      select_bin(S, kDistBins, by_mass, true, need_cnt - cnt_above, need_mass - mass_above);
    }
    pick_share(S, rank, nrank);
    if (win == 0 && !by_mass && S.total_cnt <= need_cnt) {
      left_w0 = key_min == 0u;
      return false;
    }
    dbin = S.sel_bin;
    cnt_above += S.sel_cnt_above;
    mass_above += S.sel_mass_above;
    bin_mass = S.sel_mass_bin;
    __syncthreads();
    if (dbin > 0) break;
  }
  if (win == kWindows) win = kWindows - 1;
  // the bin's key range: its position is non-decreasing in the key over the
  // finite values up to the max (whose key + 1 does not overflow)
  const WinMap W(rs.m, P.invT, win);
  const uint32_t z = Keys<T>::of(rs.m);
  const uint32_t a = max(Keys<T>::of(-CUDART_INF_F) + 1, key_min);
  const uint32_t lo = first_true(a, z, [&](uint32_t k) { return W.bin(Keys<T>::value(k)) >= dbin; });
  const uint32_t hi = first_true(lo + 1, z + 1, [&](uint32_t k) { return W.bin(Keys<T>::value(k)) > dbin; }) - 1;
  if (dbin > 0 && lo == hi) {
    // one key in the bin (the usual case near the top): step 1 has it all
    key = lo;
    mass_ge = mass_above + bin_mass;
    left_w0 = win == 0 && key_min == 0u;
    return true;
  }
  // step 2: the exact key among the ids of that bin
  HistAcc<T> acc{&S, lo, hi, hi - lo < (uint32_t)kHistBins, 0u, Keys<T>::kBits, 0, P.c, rs.m * P.c};
  constexpr int kBits = Keys<T>::kBits;
  uint32_t prefix = 0;
  int decided = acc.one_round ? kBits : 0;
  float mb = 0.f;
  do {
    const int w = acc.one_round ? kHistBits : min(kHistBits, kBits - decided);
    const int nbins = 1 << w;
    clear_hist(S, nbins);
    __syncthreads();
    acc.prefix = prefix;
    acc.shift_hi = kBits - decided;
    acc.shift_lo = kBits - decided - w;
    scan_segment<T>(row, e0, e1, acc);
    __syncthreads();
    hist_merge(S, nbins, rank, nrank);
    if (rank == 0) {
      fix_masses(S, nbins);
      __syncthreads();
      select_bin(S, nbins, by_mass, false, need_cnt - cnt_above, need_mass - mass_above);
    }
    pick_share(S, rank, nrank);
    if (acc.one_round) {
      prefix = lo + (uint32_t)S.sel_bin;
    } else {
      prefix = (prefix << w) | (uint32_t)S.sel_bin;
      decided += w;
    }
    cnt_above += S.sel_cnt_above;
    mass_above += S.sel_mass_above;
    mb = S.sel_mass_bin;
    __syncthreads();
  } while (decided < kBits);
  key = prefix;
  mass_ge = mass_above + mb;
  return true;
}

// One cluster per row (filter_cluster_ctas CTAs, each scanning one segment
// of the row into its own histograms, merged at rank 0): the row's threshold
// and kept mass; the cluster that filters a sequence's last row runs the
// sequence's accept scan on the filtered rows.
template <typename T>
__global__ void __launch_bounds__(kThreads, 4) filter_kernel(const Params P) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the row pass's statistics must be visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const unsigned rank = cluster_rank(), nrank = cluster_ctas();
  const long long r = blockIdx.x / nrank;
  // segments of whole batches of 16-byte vectors (the last one shorter)
  constexpr int kBatchElems = kUnroll * kThreads * Vec<T>::n;
  const int per = (int)(((P.V + kBatchElems - 1) / kBatchElems + nrank - 1) / nrank) * kBatchElems;
  const int e0 = min(P.V, (int)rank * per), e1 = min(P.V, e0 + per);
  int b;
  const T* row = row_ptr<T, kStochastic>(P, r, b);
  const RowStat rs = ldcg_stat(P.ws.row_stat + r);
  float tau = -CUDART_INF_F, lnM = rs.lnS;
  if (rs.status == SPEC_OK) {
    float mass = __expf(rs.lnS);                       // the row's mass relative to its max
    uint32_t key = 0, key_min = 0;
    bool thr = false, w0 = false;
    if (P.top_k > 0) {
      float mk;
      if (find_threshold<T>(row, e0, e1, rank, nrank, P, rs, false, (uint32_t)P.top_k, 0.f, 0u, false, key, mk, w0)) {
        thr = true;
        mass = mk;
        key_min = key;
      }
    }
    if (P.top_p > 0.f && P.top_p < 1.f) {
      // top-p on the top-k ids: when the top-k pass ended on window 0's
      // histogram, the kept ids are that histogram's bins from the top down to
      // the top-k key's, and the top-p target lies among them
      float mp;
      bool unused;
      find_threshold<T>(row, e0, e1, rank, nrank, P, rs, true, 0u, P.top_p * mass, key_min, w0, key, mp, unused);
      thr = true;
      mass = mp;
    }
    if (thr) {
      tau = Keys<T>::value(key);
      lnM = logf(mass);
    }
  }
  if (rank == 0 && threadIdx.x < 32) {
    int last = 0;
    if (threadIdx.x == 0) {
      __stcg(P.ws.row_filter + r, make_float2(tau, lnM));
      __threadfence();
      last = atomicAdd(P.ws.seq_cnt + b, 1u) + 1 == (unsigned)P.rows_per_seq;
      if (last) P.ws.seq_cnt[b] = 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence();
      accept_scan<T>(P, b);
    }
  }
}

// ------------------------------------------------------------ sampling ---
//
// Gumbel noise is bounded above: U <= 1 - 2^-24 gives G < 16.64.  An id whose
// score bound -- ln p_v for the residual (ln(p - q) <= ln p), z_v = x_v / T for
// the bonus -- plus that bound stays below a score some id reaches cannot win,
// so its noise is never drawn.  Each thread scores the candidate with its own
// best bound; the CTA's floor is the best of those scores and of what the
// sequence's other tiles had published when this one started (atomic max,
// nothing waits for it).  An id that passes the bound meets a cheap
// conservative test on its uniform before the accurate logarithms.  The result
// is the unpruned argmax, ties included.
//
// For the residual the kernel works with delta_v = ln q_v - ln p_v =
// ((x_d - x_t) - (m_d - m_t)) / T - (lnS_d - lnS_t): an id is a candidate iff
// delta_v < 0, and ln(p - q) = ln p + ln(-expm1(delta)).
constexpr float kGumbelMax = 16.7f;      // > -ln(-ln(1 - 2^-24)) = 16.6355
constexpr float kPruneSlack = 1e-3f;     // covers the fp32 error of the fast test

// May a draw from uniform u lift a score bound h to `floor`?  G(u) >= need holds
// iff u >= exp(-exp(-need)); the fast exponentials are off by far less than the
// slack and the 3e-5 relative allowance, so every id that can reach is kept.
__device__ __forceinline__ bool may_reach(float u, float h, float floor) {
  const float need = floor - h - kPruneSlack;
  return u >= __expf(-__expf(-need)) * (1.0f - 3e-5f);
}

// The smallest value of w >> 9 for a Philox word w whose uniform may lift bound
// h to `floor`: the integer form of may_reach's test (U(w) = ((w >> 9) + 0.5)
// 2^-23 >= umin iff w >> 9 >= ceil(umin 2^23 - 0.5), exact in fp32).  A group's
// ids share the threshold of its largest bound, so a test of each word against
// it keeps every id may_reach keeps; it is independent of the Philox chain, and
// the words that pass it meet may_reach itself before the exact score.
__device__ __forceinline__ uint32_t reach_word(float h, float floor) {
  const float need = floor - h - kPruneSlack;
  const float umin = __expf(-__expf(-need)) * (1.0f - 3e-5f);
  const float t = ceilf(umin * 8388608.0f - 0.5f);
  return t <= 0.f ? 0u : (t >= 8388608.f ? 0x800000u : (uint32_t)t);
}

// Four consecutive logits: 8 bytes of bf16 or 16 bytes of fp32.
template <typename T>
struct Raw4 {
  uint32_t w[sizeof(T)];
};

template <typename T>
__device__ __forceinline__ Raw4<T> lds_raw4(const T* p) {
  Raw4<T> r;
  if constexpr (sizeof(T) == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    r.w[0] = w.x;
    r.w[1] = w.y;
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    r.w[0] = w.x; r.w[1] = w.y; r.w[2] = w.z; r.w[3] = w.w;
  }
  return r;
}

template <typename T>
__device__ __forceinline__ float raw_at(const Raw4<T>& r, int e) {
  if constexpr (sizeof(T) == 2) return (e & 1) ? bf16_hi(r.w[e >> 1]) : bf16_lo(r.w[e >> 1]);
  else return __uint_as_float(r.w[e]);
}

// NaN-propagating max of the first `cnt` (1..4) logits of a group (bf16, all
// four: one packed max).
template <typename T>
__device__ __forceinline__ float group_max(const Raw4<T>& r, int cnt) {
  if (cnt >= 4) {
    if constexpr (sizeof(T) == 2) {
      const uint32_t m = bf16x2_nanmax(r.w[0], r.w[1]);
      return nanmax(bf16_lo(m), bf16_hi(m));
    } else {
      return nanmax(nanmax(__uint_as_float(r.w[0]), __uint_as_float(r.w[1])),
                    nanmax(__uint_as_float(r.w[2]), __uint_as_float(r.w[3])));
    }
  }
  float m = raw_at<T>(r, 0);
  for (int e = 1; e < cnt; ++e) m = nanmax(m, raw_at<T>(r, e));
  return m;
}

// What a sampling CTA knows about its sequence's row.
struct SampleRow {
  bool resid;
  float mt, lnSt;       // target row statistics (residual; lnSt of the kept mass when filtering)
  float cdelta;         // delta_v = fma(x_d - x_t, 1/T, cdelta)
  float tau_t, tau_d;   // filtering: the kept sets are x_t >= tau_t (sampled row) and x_d >= tau_d;
                        // -inf without filtering
};

// Exact score of id v (or -inf if it is no candidate) from its logits and noise uniform.
__device__ __forceinline__ float exact_score(float invT, const SampleRow& R, float xt, float xd, float u) {
  if (!(xt >= R.tau_t)) return -CUDART_INF_F;
  if (R.resid) {
    // q = 0 outside the draft's kept set: delta = -inf, ln(1 - e^delta) = 0
    const float delta = xd >= R.tau_d ? fmaf(xd - xt, invT, R.cdelta) : -CUDART_INF_F;
    if (!(delta < 0.f)) return -CUDART_INF_F;
    const float lp = (xt - R.mt) * invT - R.lnSt;
    return lp + logf(-expm1f(delta)) + gumbel_of(u);
  }
  if (!(xt > -CUDART_INF_F)) return -CUDART_INF_F;
  return xt * invT + gumbel_of(u);
}

__device__ __forceinline__ float uniform_at(uint2 key, uint32_t b, int j, int v) {
  const uint4 w = gumbel_words(key, b, j, (uint32_t)(v >> 2));
  const int e = v & 3;
  return uniform_of(e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w);
}

// What a sampling thread knows about its sequence's draw.
struct Draw {
  float invT, T;
  SampleRow R;
  uint2 key;
  uint32_t gb;            // Philox counter word 2: the sequence's global index
  int j;                  // Philox counter word 1: the row whose noise is drawn
};

// Candidate test and score bound of one id: ln p for the residual, z for the bonus.
__device__ __forceinline__ bool bound_of(const Draw& D, float x, float xdv, float& h) {
  if (D.R.resid) {
    h = (x - D.R.mt) * D.invT - D.R.lnSt;
    return x >= D.R.tau_t && (xdv < D.R.tau_d || fmaf(xdv - x, D.invT, D.R.cdelta) < 0.f);
  }
  h = x * D.invT;
  return x > -CUDART_INF_F && x >= D.R.tau_t;
}

// The lowest target logit that can still reach score fl: bound + G_max >= fl.
__device__ __forceinline__ float threshold_of(const Draw& D, float fl) {
  if (!(fl > -CUDART_INF_F)) return -CUDART_INF_F;
  return D.R.resid ? D.R.mt + (fl - kGumbelMax + D.R.lnSt) * D.T : (fl - kGumbelMax) * D.T;
}

// Shared memory of a sampling CTA: a ring of tiles (target and draft logits
// of 4096 ids each), filled by bulk copies, and each warp's queue of groups
// whose noise is to be drawn.
template <typename T>
struct SampleSmem {
  static constexpr int kStages = sizeof(T) == 2 ? 3 : 2;
  T tile[kStages][2][kPartTile];
  uint64_t bar[kStages];
  uint32_t queue[kWarps][kGroups * 32];
};

// Score the ids of tile [v0, v1) (staged at st / sd) that can reach the
// floor.  Thread g owns groups g, g + kThreads, ...; a group whose largest
// target logit reaches the threshold goes into the warp's queue, and the
// warp's lanes share the queued groups out: the id-by-id bound and candidate
// tests, and the noise draw of a group with an id that passes them, run only
// there, one group per lane, so no lane waits on another's groups.
template <typename T>
__device__ __forceinline__ void score_tile(const Draw& D, int v0, int v1, const T* st, const T* sd,
                                           uint32_t* queue, float& floor, float& best, int& bidx, int& bad) {
  const int lane = threadIdx.x & 31;
  const float xthr = threshold_of(D, floor);
  const int nv = v1 - v0;
  int cnt = 0;
#pragma unroll
  for (int q = 0; q < kGroups; ++q) {
    const int o = 4 * (q * kThreads + threadIdx.x);
    bool hit = false;
    if (o < nv) {
      const float gm = group_max<T>(lds_raw4<T>(st + o), min(4, nv - o));
      if (!D.R.resid && !(gm < CUDART_INF_F)) bad = 1;     // NaN or +inf in the bonus row
      hit = gm >= xthr;
    }
    const unsigned need = __ballot_sync(0xffffffffu, hit);
    if (hit) queue[cnt + __popc(need & ((1u << lane) - 1u))] = (uint32_t)o;
    cnt += __popc(need);
  }
  __syncwarp();
  for (int it = lane; it < cnt; it += 32) {
    const int o = (int)queue[it];
    const int v = v0 + o;
    const int ne = min(4, nv - o);
    const Raw4<T> gt = lds_raw4<T>(st + o);
    Raw4<T> gd;
    if (D.R.resid) gd = lds_raw4<T>(sd + o);
    unsigned pass = 0;
    float hmax = -CUDART_INF_F;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = raw_at<T>(gt, e);
      float h;
      if (e < ne && x >= xthr && bound_of(D, x, D.R.resid ? raw_at<T>(gd, e) : 0.f, h)) {
        pass |= 1u << e;
        hmax = fmaxf(hmax, h);
      }
    }
    if (!pass) continue;
    const uint32_t wmin = reach_word(hmax, floor);
    const uint4 w = gumbel_words(D.key, D.gb, D.j, (uint32_t)(v >> 2));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!((pass >> e) & 1u) || (ws[e] >> 9) < wmin) continue;
      const float x = raw_at<T>(gt, e);
      const float xdv = D.R.resid ? raw_at<T>(gd, e) : 0.f;
      float h;
      bound_of(D, x, xdv, h);
      const float u = uniform_of(ws[e]);
      if (!may_reach(u, h, floor)) continue;
      const float sc = exact_score(D.invT, D.R, x, xdv, u);
      if (beats(sc, v + e, best, bidx)) {
        best = sc;
        bidx = v + e;
        floor = fmaxf(floor, sc);
      }
    }
  }
  __syncwarp();   // the queue is refilled by the next tile
}


// One sequence's draw runs on ns CTAs over the row pass's 4096-id tiles.
//
//   1. floor: in the first tile a CTA scores (its own first tile), each
//      thread scores the candidate with its best bound, and the CTA takes the
//      best of those scores and of what the sequence's other CTAs have
//      published; before each later tile it takes up what they have
//      published since.  None waits for another.
//   2. CTA c scores tiles c, c + ns, ...  Tiles reach shared memory through
//      bulk copies kStages ahead of use, so the loads of a CTA's tiles are in
//      flight together (rows whose tiles do not meet the bulk copy's 16-byte
//      rules are loaded by the threads, one tile at a time).
//   3. per-CTA (best, index) partials; the sequence's last CTA merges them and
//      writes the committed tokens.
template <typename T>
__global__ void __launch_bounds__(kThreads) sample_kernel(const Params P) {
  using Smem = SampleSmem<T>;
  constexpr int kStages = Smem::kStages;
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  Smem& S = *reinterpret_cast<Smem*>(dyn_smem);
  __shared__ BlockScratch sh;
  __shared__ float s_floor[kWarps];
  __shared__ float s_fresh;
  __shared__ int s_last, s_timeout;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&S.bar[i], 1);
    fence_mbar_init();
    s_timeout = 0;
  }
  // the row pass's statistics and sequence states must be visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x / P.ns;
  const int c = blockIdx.x % P.ns;
  const int k = P.k;
  // the sequence's record: n, status and the sampled row's statistics at once
  const int4 q0 = __ldcg(reinterpret_cast<const int4*>(P.ws.seq + b));
  const float4 q1 = __ldcg(reinterpret_cast<const float4*>(P.ws.seq + b) + 1);
  const int n = q0.x, status = q0.y;
  const bool active = status == SPEC_OK;            // uniform over the CTA
  Draw D;
  D.invT = P.invT;
  D.T = P.T;
  D.key = P.key;
  D.gb = P.b0 + (uint32_t)b;
  D.j = n < k ? n : k;
  D.R.resid = n < k;
  D.R.mt = D.R.lnSt = D.R.cdelta = 0.f;
  D.R.tau_t = D.R.tau_d = -CUDART_INF_F;
  const T* trow = (const T*)P.target + ((size_t)b * (k + 1) + (active ? D.j : 0)) * P.V;
  const T* drow = D.R.resid ? (const T*)P.draft + ((size_t)b * k + (active ? n : 0)) * P.V : nullptr;
  // bulk copies need 16-byte aligned rows and tiles of whole 16-byte units
  const bool bulk = (reinterpret_cast<uintptr_t>(trow) % 16 == 0) &&
                    (!drow || reinterpret_cast<uintptr_t>(drow) % 16 == 0) &&
                    ((size_t)P.V * sizeof(T)) % 16 == 0;
  // the CTA's tiles c, c + ns, ... in that order; the first one also gives
  // the CTA's floor.  (A separate floor tile, the one holding the row's max,
  // read and scored by every CTA, gave a better floor but cost more than it
  // saved: 76.8 against 74.8 us a step on 64 sequences of 8 drafts over
  // 128256 bf16 logits.)
  const int n_own = (P.nt - c + P.ns - 1) / P.ns;
  const int m = active ? n_own : 0;
  auto tile_of = [&](int i) { return c + i * P.ns; };
  int issued = 0;                                   // thread 0: tiles whose copies are issued
  auto issue = [&](int i) {      // thread 0: bulk copies of the i-th tile into its stage
    issued = i + 1 > issued ? i + 1 : issued;
    const int t = tile_of(i), s = i % kStages;
    const int v0 = t * kPartTile;
    const unsigned bytes = (unsigned)((min(P.V, v0 + kPartTile) - v0) * sizeof(T));
    mbar_arrive_tx(&S.bar[s], drow ? 2 * bytes : bytes);
    bulk_copy_g2s(S.tile[s][0], trow + v0, bytes, &S.bar[s]);
    if (drow) bulk_copy_g2s(S.tile[s][1], drow + v0, bytes, &S.bar[s]);
  };
  if (active) {
    D.R.tau_t = q1.w;                                // filtering: the sampled row's kept set
    if (D.R.resid) {
      D.R.mt = q1.x;
      D.R.lnSt = q1.y;
      D.R.cdelta = q1.z;
      D.R.tau_d = __int_as_float(q0.w);
    }
  }
  __syncthreads();                                   // barriers initialised
  if (bulk && threadIdx.x == 0)
    for (int i = 0; i < min(m, kStages); ++i) issue(i);
  uint32_t* queue = S.queue[threadIdx.x >> 5];

  float floor = -CUDART_INF_F, best = -CUDART_INF_F;
  int bidx = INT_MAX, bad = 0;
  int i = 0;
  for (; i < m; ++i) {
    const int s = i % kStages;
    const int t = tile_of(i);
    const int v0 = t * kPartTile, v1 = min(P.V, v0 + kPartTile);
    const unsigned pub = __ldcg(P.ws.samp_floor + b);
    bool ok = true;
    if (bulk) {
      // warp 0 waits for the stage (sleeping between polls) while the other
      // warps sleep at the barrier; then every warp observes the completed phase
      const unsigned par = (unsigned)(i / kStages) & 1u;
      if (threadIdx.x < 32) ok = !P.force_timeout && mbar_wait_sleepy(&S.bar[s], par);
      ok = __syncthreads_and(ok);
      if (ok && threadIdx.x >= 32) ok = mbar_try_wait(&S.bar[s], par) || mbar_wait_bounded(&S.bar[s], par);
      if (!ok) s_timeout = 1;
    } else {
      for (int o = threadIdx.x; o < v1 - v0; o += kThreads) {
        S.tile[s][0][o] = trow[v0 + o];
        if (drow) S.tile[s][1][o] = drow[v0 + o];
      }
      __syncthreads();
    }
    const T* st = S.tile[s][0];
    const T* sd = S.tile[s][1];
    if (i == 0) {
      // 1. the floor: each thread's candidate with the largest target logit
      float ub = -CUDART_INF_F, ub_xd = 0.f;
      int ub_i = INT_MAX;
      if (ok) {
#pragma unroll
        for (int q = 0; q < kGroups; ++q) {
          const int o = 4 * (q * kThreads + threadIdx.x);
          if (o >= v1 - v0) continue;
          const Raw4<T> gt = lds_raw4<T>(st + o);
          Raw4<T> gd;
          if (D.R.resid) gd = lds_raw4<T>(sd + o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (o + e >= v1 - v0) continue;
            const float x = raw_at<T>(gt, e);
            const float xdv = D.R.resid ? raw_at<T>(gd, e) : 0.f;
            float h;
            if (bound_of(D, x, xdv, h) && x > ub) { ub = x; ub_i = v0 + o + e; ub_xd = xdv; }
          }
        }
      }
      float f = ub > -CUDART_INF_F ? exact_score(D.invT, D.R, ub, ub_xd, uniform_at(D.key, D.gb, D.j, ub_i))
                                   : -CUDART_INF_F;
      f = warp_max(f);
      if ((threadIdx.x & 31) == 0) s_floor[threadIdx.x >> 5] = f;
      __syncthreads();
      floor = from_ordered(pub);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) floor = fmaxf(floor, s_floor[w]);
      // publish this CTA's floor and take up the sequence's best so far in the
      // same atomic: the other CTAs computed theirs at about the same time, and
      // the first tile is scored against the best of them (a round trip that
      // measured 1.2 us a step faster than scoring against the CTA's own floor)
      if (threadIdx.x == 0) {
        const unsigned prev = atomicMax(P.ws.samp_floor + b, floor > -CUDART_INF_F ? ordered_bits(floor) : 0u);
        s_fresh = fmaxf(floor, from_ordered(prev));
      }
      __syncthreads();
      floor = s_fresh;
    } else {
      floor = fmaxf(floor, from_ordered(pub));
    }
    // 2. score the tile
    if (ok) {
      const float floor_in = floor;
      score_tile<T>(D, v0, v1, st, sd, queue, floor, best, bidx, bad);
      if (floor > floor_in) atomicMax(P.ws.samp_floor + b, ordered_bits(floor));
    }
    __syncthreads();                                 // the stage is free again
    if (s_timeout) break;
    if (bulk && threadIdx.x == 0 && i + kStages < m) {
      fence_proxy_async_smem();
      issue(i + kStages);
    }
  }
  if (s_timeout && bulk) {
    // leave no bulk copy in flight into this CTA's shared memory: wait (bounded)
    // for every tile issued but not consumed, oldest first
    if (threadIdx.x == 0)
      for (int x = i; x < issued; ++x) mbar_wait_bounded(&S.bar[x % kStages], (unsigned)(x / kStages) & 1u);
    __syncthreads();
  }

  // 3. partials and the merge
  block_argmax_flag(best, bidx, bad, sh);
  if (threadIdx.x == 0) {
    // index -2 marks a tile that timed out
    P.ws.samp_partial[(size_t)b * P.ns + c] =
        make_float2(bad ? CUDART_NAN_F : best, __int_as_float(s_timeout ? -2 : bidx));
    __threadfence();
    s_last = atomicAdd(P.ws.samp_cnt + b, 1u) + 1 == (unsigned)P.ns;
    if (s_last) {
      P.ws.samp_cnt[b] = 0;
      P.ws.samp_floor[b] = 0;
    }
  }
  __syncthreads();
  if (!s_last) return;

  __threadfence();
  best = -CUDART_INF_F;
  bidx = INT_MAX;
  bad = 0;
  int timed_out = 0;
  for (int q = threadIdx.x; q < P.ns; q += kThreads) {
    const float2 p = __ldcg(P.ws.samp_partial + (size_t)b * P.ns + q);
    __stcg(P.ws.samp_partial + (size_t)b * P.ns + q, make_float2(0.f, 0.f));   // the workspace is left zeroed
    const int pi = __float_as_int(p.y);
    if (pi == -2) { timed_out = 1; continue; }
    if (p.x != p.x) { bad = 1; continue; }
    if (beats(p.x, pi, best, bidx)) { best = p.x; bidx = pi; }
  }
  block_argmax_flag(best, bidx, bad, sh);
  timed_out = __syncthreads_or(timed_out);
  int st = status;
  if (st == SPEC_OK && timed_out) st = SPEC_ERR_TIMEOUT;
  if (st == SPEC_OK && !D.R.resid && (bad || !(best > -CUDART_INF_F))) st = SPEC_ERR_NONFINITE;
  if (st == SPEC_OK && D.R.resid && bidx == INT_MAX) {
    // empty residual in fp32: draw from p_n itself with the same noise
    const T* row = (const T*)P.target + ((size_t)b * (k + 1) + n) * P.V;
    best = -CUDART_INF_F;
    for (int g = threadIdx.x; 4 * g < P.V; g += kThreads) {
      const uint4 w = gumbel_words(P.key, D.gb, n, (uint32_t)g);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      for (int e = 0; e < 4 && 4 * g + e < P.V; ++e) {
        const int v = 4 * g + e;
        const float x = load_elem<T>(row, v);
        if (!(x >= D.R.tau_t)) continue;             // filtering: only the kept ids of p_n
        const float sc = x * P.invT + gumbel_of(uniform_of(ws[e]));
        if (beats(sc, v, best, bidx)) { best = sc; bidx = v; }
      }
    }
    block_argmax(best, bidx, sh);
  }
  // every CTA of the sequence has read its statistics and state: the
  // workspace is left zeroed
  {
    const long long rb = (long long)b * P.rows_per_seq;
    for (int r = threadIdx.x; r < P.rows_per_seq; r += kThreads) {
      stcg_stat(P.ws.row_stat + rb + r, RowStat{0.f, 0.f, 0, 0});
      if (P.filtering) __stcg(P.ws.row_filter + rb + r, make_float2(0.f, 0.f));
    }
    if (threadIdx.x == 0) {
      __stcg(reinterpret_cast<int4*>(P.ws.seq + b), make_int4(0, 0, 0, 0));
      __stcg(reinterpret_cast<int4*>(P.ws.seq + b) + 1, make_int4(0, 0, 0, 0));
    }
  }
  if (threadIdx.x >= 32) return;
  int32_t* out = P.out_tokens + (size_t)b * P.out_w;
  const int32_t* x = P.tokens + (size_t)b * k;
  const int committed = write_committed(P, out, P.out_w, [&](int i) -> int {
    if (st != SPEC_OK) return -1;
    return i < n ? x[i] : (i == n ? bidx : -1);
  });
  if (threadIdx.x == 0) {
    P.out_n[b] = st == SPEC_OK ? n : -1;
    if (P.n_committed) P.n_committed[b] = st == SPEC_OK ? committed : -1;
    if (P.status) P.status[b] = st;
  }
}

// -------------------------------------------------------------- randomness ---
__global__ void random_kernel(uint2 key, int b, int j, int V, float* gu, float* gg, float* au) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g == 0 && au) au[0] = accept_uniform(key, (uint32_t)b, j);
  if (4 * g >= V) return;
  const uint4 w = gumbel_words(key, (uint32_t)b, j, (uint32_t)g);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  for (int e = 0; e < 4 && 4 * g + e < V; ++e) {
    const float u = uniform_of(ws[e]);
    if (gu) gu[4 * g + e] = u;
    if (gg) gg[4 * g + e] = gumbel_of(u);
  }
}

// ------------------------------------------------------------ read probe ---
// The row pass's load pattern with nothing else: a persistent grid of
// contiguous ranges, 16-byte no-L1 loads, kUnroll per thread in flight, the
// words folded by xor so that no load is dead.  Its rate is the read ceiling
// the row pass streams against.
__global__ void __launch_bounds__(kThreads, 6) probe_read_kernel(const uint4* data, long long nvec, unsigned* sink) {
  const long long v0 = nvec * blockIdx.x / gridDim.x, v1 = nvec * (blockIdx.x + 1) / gridDim.x;
  constexpr int kBatch = kUnroll * kThreads;
  unsigned acc = 0;
  long long i = v0 + threadIdx.x;
  for (; i + (kUnroll - 1) * kThreads < v1; i += kBatch) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream16(data + i + u * kThreads);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < v1; i += kThreads) {
    const uint4 v = ld_stream16(data + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if ((threadIdx.x & 31) == 0) atomicXor(sink + blockIdx.x, acc);
}

// --------------------------------------------------------------- host side ---

// The workspace: the completion counters, then the records every call writes
// before it reads them.  A call leaves all of it zeroed (see below).
struct Layout {
  size_t row_cnt, seq_cnt, samp_cnt, samp_floor, counters_end;
  size_t row_partial, row_stat, row_filter, seq, samp_partial, total;
  int nt;
  long long rmax;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static bool make_layout(int B, int k, int V, Layout& L) {
  if (B <= 0 || k <= 0 || V <= 0) return false;
  L.nt = (V + kPartTile - 1) / kPartTile;
  L.rmax = (long long)B * (long long)(2 * k + 1);   // the most rows any mode takes statistics of
  size_t off = 0;
  auto take = [&](size_t bytes, size_t a) { off = align_up(off, a); const size_t o = off; off += bytes; return o; };
  L.row_cnt = take((size_t)L.rmax * sizeof(unsigned), 4);
  L.seq_cnt = take((size_t)B * sizeof(unsigned), 4);
  L.samp_cnt = take((size_t)B * sizeof(unsigned), 4);
  L.samp_floor = take((size_t)B * sizeof(unsigned), 4);
  L.counters_end = off;
  L.row_partial = take((size_t)L.rmax * L.nt * sizeof(Partial), 256);
  L.row_stat = take((size_t)L.rmax * sizeof(RowStat), 256);
  L.row_filter = take((size_t)L.rmax * sizeof(float2), 256);
  L.seq = take((size_t)B * sizeof(SeqState), 256);
  L.samp_partial = take((size_t)B * L.nt * sizeof(float2), 256);
  L.total = align_up(off, 256);
  return true;
}

static Workspace bind(void* base, const Layout& L) {
  char* p = static_cast<char*>(base);
  Workspace w;
  w.row_partial = reinterpret_cast<Partial*>(p + L.row_partial);
  w.row_cnt = reinterpret_cast<unsigned*>(p + L.row_cnt);
  w.row_stat = reinterpret_cast<RowStat*>(p + L.row_stat);
  w.row_filter = reinterpret_cast<float2*>(p + L.row_filter);
  w.seq_cnt = reinterpret_cast<unsigned*>(p + L.seq_cnt);
  w.seq = reinterpret_cast<SeqState*>(p + L.seq);
  w.samp_partial = reinterpret_cast<float2*>(p + L.samp_partial);
  w.samp_cnt = reinterpret_cast<unsigned*>(p + L.samp_cnt);
  w.samp_floor = reinterpret_cast<unsigned*>(p + L.samp_floor);
  return w;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The workspace between calls.  Every call leaves zeroed everything it wrote
// there: its counters, and each record once its last reader has read it (a
// row's partials when the row is merged, the rows' statistics and filters,
// the sequence state and the draw partials when the sequence's output is
// written).  So whatever sizes the calls use, and whether they run eagerly or
// as replays of a captured graph, a call finds the workspace all zero -- as
// it was first handed over -- and needs no clearing.

// CTAs per row in the filter (a cluster; the kernel takes any size up to the
// portable 8).  Measured on 64 x 17 rows of 128256 bf16 logits: a row's first
// pass streams at the same rate cut or whole, and every CTA of a cut row pays
// the merge and waits for the pick, so top-p alone is fastest whole (98.8 us;
// 2 CTAs 107, 4 CTAs 137).  A top-k target below window 0 (rows whose max
// stands far above the rest) takes two more passes over its row, at the end
// of the launch; two CTAs halve those (top-k 50: 222 -> 179 us; with top-p
// 0.8: 245 -> 203 us).  So rows of 128 KB or more take two CTAs when a top-k
// stage runs.
static int filter_cluster_ctas(int V, size_t esize, int top_k) {
  return top_k > 0 && (long long)V * (long long)esize >= 131072 ? 2 : 1;
}

// Resident CTAs of a kernel with `threads` threads and `smem` bytes of dynamic
// shared memory on the current device, cached per (device, kernel).
static int resident_ctas(const void* fn, size_t smem = 0, int threads = kThreads) {
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
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess) return 0;
  const int ctas = sms * (per_sm > 0 ? per_sm : 1);
  if (used < 64) cache[used++] = Entry{dev, fn, ctas};
  return ctas;
}

// Test hook: when set, every bulk-copy stage wait of the next launches gives up
// at once, as if its copy had not landed within the limit.
static std::atomic<int> g_force_timeout{0};

template <typename T, int kMode>
static int launch(Params& P, cudaStream_t stream, const spec_verify_aux* aux) {
  P.force_timeout = g_force_timeout.load(std::memory_order_relaxed);
  auto rec = [&](int i) {
    return (aux && aux->events[i]) ? cudaEventRecord(static_cast<cudaEvent_t>(aux->events[i]), stream)
                                   : cudaSuccess;
  };
  const long long items = P.R * P.nt;
  // greedy and tree rows on 16-byte boundaries, over more than L2 holds, are
  // staged by bulk copies (measured: 30.6 vs 33.2 us on 64 x 9 rows of 128256
  // bf16; on 66 MB of rows 22.0 vs 21.1 us, so smaller batches keep the
  // register path); the stochastic pass, with an exponential per element,
  // keeps more warps per SM with the register path (51.0 vs 55.0 us on 64 x 16
  // rows), as do unaligned rows
  const bool ring = kMode != kStochastic && aligned(P.target, 16) && ((size_t)P.V * sizeof(T)) % 16 == 0 &&
                    (double)P.R * (double)P.V * sizeof(T) >= kRingMinBytes;
  const void* rp = ring ? reinterpret_cast<const void*>(&row_pass_ring<T, kMode>)
                        : reinterpret_cast<const void*>(&row_pass_kernel<T, kMode>);
  const size_t rsmem = ring ? sizeof(RingSmem) : 0;
  const int ctas = resident_ctas(rp, rsmem, ring ? kRingThreads : kThreads);
  if (ctas <= 0) return SPEC_ERR_CUDA;
  const int grid = (int)(items < ctas ? items : ctas);
  if (rec(0) != cudaSuccess) return SPEC_ERR_CUDA;
  if (ring) row_pass_ring<T, kMode><<<grid, kRingThreads, rsmem, stream>>>(P);
  else row_pass_kernel<T, kMode><<<grid, kThreads, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (rec(1) != cudaSuccess) return SPEC_ERR_CUDA;
  if constexpr (kMode == kStochastic) {
    // as many CTAs per sequence as fill the GPU once, at most one per tile
    const size_t smem = sizeof(SampleSmem<T>);
    const int slots = resident_ctas(reinterpret_cast<const void*>(&sample_kernel<T>), smem);
    if (slots <= 0) return SPEC_ERR_CUDA;
    P.ns = slots / P.B;
    P.ns = P.ns < 1 ? 1 : (P.ns > P.nt ? P.nt : P.ns);
    // launched as programmatic dependents of the kernel before them: their CTAs
    // may start while it drains and wait for its results in griddepcontrol.wait
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (P.filtering) {
      const int fc = filter_cluster_ctas(P.V, sizeof(T), P.top_k);
      if (P.R * fc > (long long)INT_MAX) return SPEC_ERR_UNSUPPORTED;
      cudaLaunchAttribute fattr[2];
      fattr[0] = attr[0];
      fattr[1].id = cudaLaunchAttributeClusterDimension;
      fattr[1].val.clusterDim.x = (unsigned)fc;
      fattr[1].val.clusterDim.y = 1;
      fattr[1].val.clusterDim.z = 1;
      cudaLaunchConfig_t fcfg = {};
      fcfg.gridDim = dim3((unsigned)(P.R * fc));
      fcfg.blockDim = dim3(kThreads);
      fcfg.stream = stream;
      fcfg.attrs = fattr;
      fcfg.numAttrs = fc > 1 ? 2 : 1;
      if (cudaLaunchKernelEx(&fcfg, filter_kernel<T>, P) != cudaSuccess) return SPEC_ERR_CUDA;
    }
    if (rec(2) != cudaSuccess) return SPEC_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(P.B * P.ns));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, sample_kernel<T>, P) != cudaSuccess) return SPEC_ERR_CUDA;
  } else {
    if (rec(2) != cudaSuccess) return SPEC_ERR_CUDA;
  }
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

  float lenience = 1.f;
  int top_k = 0;
  float top_p = 0.f;
  if (aux) {
    if (aux->top_k < 0 || !(aux->top_p >= 0.f && aux->top_p <= 1.f)) return SPEC_ERR_ARG;
    top_k = aux->top_k < V ? aux->top_k : 0;          // k >= V keeps every id
    top_p = aux->top_p < 1.f ? aux->top_p : 0.f;      // 1 keeps every id
    if (aux->lenience != 0.f) {
      if (!(aux->lenience >= 1.f) || !std::isfinite(aux->lenience)) return SPEC_ERR_ARG;
      lenience = aux->lenience;
    }
    if (aux->n_stop < 0 || (aux->n_stop > 0 && !aux->stop_ids)) return SPEC_ERR_ARG;
    if (aux->n_stop > SPEC_MAX_STOP) return SPEC_ERR_UNSUPPORTED;
    if (!greedy && (aux->match_mask || aux->n_match || aux->tail_runs)) return SPEC_ERR_ARG;
    if ((aux->stop_ids && !aligned(aux->stop_ids, 4)) || (aux->n_committed && !aligned(aux->n_committed, 4)) ||
        (aux->n_match && !aligned(aux->n_match, 4)) || (aux->tail_runs && !aligned(aux->tail_runs, 4)))
      return SPEC_ERR_ALIGN;
  }

  Params P;
  std::memset(&P, 0, sizeof(P));
  P.target = target_logits;
  P.draft = draft_logits;
  P.tokens = draft_tokens;
  P.B = B;
  P.k = k;
  P.V = V;
  P.nt = L.nt;
  P.key = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
  P.out_tokens = out_tokens;
  P.out_n = out_n_accepted;
  P.out_w = k + 1;
  P.lenience = lenience;
  P.ln_lenience = (float)std::log((double)lenience);
  P.ws = bind(workspace, L);
  if (aux) {
    P.status = aux->status;
    P.p_draft = aux->p_draft;
    P.q_draft = aux->q_draft;
    P.lse = aux->lse;
    P.b0 = aux->sequence_offset;
    P.stop_ids = aux->n_stop > 0 ? aux->stop_ids : nullptr;
    P.n_stop = aux->n_stop > 0 ? aux->n_stop : 0;
    P.n_committed = aux->n_committed;
    P.match_mask = aux->match_mask;
    P.n_match = aux->n_match;
    P.tail_runs = aux->tail_runs;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if (greedy) {
    P.rows_per_seq = k + 1;
    P.R = (long long)B * (k + 1);
    return dtype == SPEC_BF16 ? launch<uint16_t, kGreedy>(P, stream, aux) : launch<float, kGreedy>(P, stream, aux);
  }
  // filtering (stochastic only: it leaves every argmax where it is) also needs
  // the bonus row's statistics
  P.filtering = (top_k > 0 || top_p > 0.f) ? 1 : 0;
  P.top_k = top_k;
  P.top_p = top_p;
  P.rows_per_seq = 2 * k + P.filtering;
  P.R = (long long)B * P.rows_per_seq;
  P.invT = 1.0f / temperature;
  P.T = temperature;
  P.c = (float)(1.4426950408889634 / (double)temperature);
  return dtype == SPEC_BF16 ? launch<uint16_t, kStochastic>(P, stream, aux) : launch<float, kStochastic>(P, stream, aux);
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
  int rc = check_common(target_logits, B, V, dtype, workspace, L, workspace_bytes);
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
  P.rows_per_seq = N + 1;
  P.R = (long long)B * (N + 1);
  P.out_w = N + 1;
  P.lenience = 1.f;
  P.out_tokens = out_tokens;
  P.out_n = out_n_accepted;
  P.out_leaf = out_leaf;
  P.status = status;
  P.ws = bind(workspace, L);
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  return dtype == SPEC_BF16 ? launch<uint16_t, kTree>(P, stream, nullptr) : launch<float, kTree>(P, stream, nullptr);
}

int spec_verify_guided(const void* target_logits, const int32_t* draft_tokens, const int32_t* guide, int B, int k,
                       int L, int V, int dtype, int32_t* out_tokens, int32_t* out_n_accepted,
                       int32_t* out_n_committed, int32_t* status, void* workspace, size_t workspace_bytes,
                       void* cuda_stream) {
  if (k <= 0 || B <= 0 || V <= 0 || L < 0) return SPEC_ERR_ARG;
  if (k > SPEC_MAX_K) return SPEC_ERR_UNSUPPORTED;
  if (!draft_tokens || !out_tokens || !out_n_accepted || !out_n_committed || (L > 0 && !guide)) return SPEC_ERR_ARG;
  const int W = L > k + 1 ? L : k + 1;
  if ((size_t)B * (size_t)W > (size_t)INT_MAX) return SPEC_ERR_UNSUPPORTED;
  Layout Lw;
  make_layout(B, k, V, Lw);
  int rc = check_common(target_logits, B, V, dtype, workspace, Lw, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  if (!aligned(draft_tokens, 4) || !aligned(out_tokens, 4) || !aligned(out_n_accepted, 4) ||
      !aligned(out_n_committed, 4) || (guide && !aligned(guide, 4)) || (status && !aligned(status, 4)))
    return SPEC_ERR_ALIGN;
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.target = target_logits;
  P.tokens = draft_tokens;
  P.B = B;
  P.k = k;
  P.V = V;
  P.nt = Lw.nt;
  P.out_tokens = out_tokens;
  P.out_n = out_n_accepted;
  P.n_committed = out_n_committed;
  P.status = status;
  P.out_w = W;
  P.lenience = 1.f;
  P.guide = L > 0 ? guide : nullptr;
  P.L = L;
  P.ws = bind(workspace, Lw);
  P.rows_per_seq = k + 1;
  P.R = (long long)B * (k + 1);
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  return dtype == SPEC_BF16 ? launch<uint16_t, kGreedy>(P, stream, nullptr) : launch<float, kGreedy>(P, stream, nullptr);
}

int spec_random(uint64_t seed, int b, int j, int V, float* gumbel_u, float* gumbel_g, float* accept_u,
                void* cuda_stream) {
  if (V <= 0 || b < 0 || j < 0) return SPEC_ERR_ARG;
  const int groups = (V + 3) / 4;
  random_kernel<<<(groups + kThreads - 1) / kThreads, kThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)), b, j, V, gumbel_u, gumbel_g, accept_u);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_probe_read(const void* data, size_t bytes, unsigned* sink, int ctas, void* cuda_stream) {
  if (!data || !sink || bytes < 16 || !aligned(data, 16) || ctas < 0) return SPEC_ERR_ARG;
  int grid = ctas;
  if (grid == 0) grid = resident_ctas(reinterpret_cast<const void*>(&probe_read_kernel));
  if (grid <= 0) return SPEC_ERR_CUDA;
  probe_read_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      static_cast<const uint4*>(data), (long long)(bytes / 16), sink);
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

int spec_abi_version(void) { return (1 << 16) | 3; }

int spec_test_force_stage_timeouts(int on) { return g_force_timeout.exchange(on ? 1 : 0); }

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
  // The scratch starts zeroed (a static device array) and every call leaves
  // it zeroed, whatever its sizes: no call needs to clear it.
  return spec_verify_ex(target_logits, draft_logits, draft_tokens, B, k, V, dtype, temperature, seed, out_tokens,
                        out_n_accepted, scratch, sv::kNoAllocScratchBytes, cuda_stream, nullptr);
}
