/*
 * spec_verify.h -- batched speculative-decoding verification on GB300 (sm_103a).
 *
 * C ABI of libspecverify.so.  Plain pointers and sizes only; every buffer is
 * owned by the caller and every call is asynchronous on the caller's CUDA
 * stream.  The library never allocates or frees device memory.
 *
 * What is computed.  For each of B sequences the target model gives k+1 logit
 * rows and the draft model k logit rows over a vocabulary of V ids, plus the k
 * drafted ids.  "Speculative Decoding: Faster Generation Without Changing the
 * Model" (section "The acceptance rule") states the rule: drafts are examined
 * left to right, x_i is accepted with probability min(1, p_i(x_i)/q_i(x_i));
 * the first rejection is replaced by a draw from the residual distribution
 * proportional to max(0, p_i - q_i) and ends the round; if every draft passes,
 * one bonus token is drawn from the target row k.  Under greedy decoding a
 * draft is accepted iff it equals the target argmax and the first mismatch is
 * replaced by that argmax.  "Cascade Speculative Drafting for Even Faster LLM
 * Inference" restates the review step as: accept when q <= p, otherwise reject
 * with probability 1 - p/q (lenience 1 at the target).  Tree verification
 * follows "Ouroboros: Generating Longer Drafts Phrase by Phrase for Faster
 * Speculative Decoding", 3.4.3 "Selecting the accepted tokens": keep the
 * longest accepted branch and append the target's own next token.
 *
 * Conventions shared by every call.
 *   p_j = softmax(target_row_j / T), q_i = softmax(draft_row_i / T).
 *   Randomness is Philox4x32-10 (Salmon et al., SC'11) keyed by
 *   (seed mod 2^32, seed >> 32):
 *     accept uniform of (b, i)         word 0 of counter (0, i, b, 0)
 *     Gumbel uniform of (b, j, v)      word v%4 of counter (v>>2, j, b, 1)
 *     U(w) = ((w >> 9) + 0.5) * 2^-23;  G = -ln(-ln U)
 *   accept_i  <=>  q_i(x_i) <= p_i(x_i)  or  U(b, i) < p_i(x_i)/q_i(x_i)
 *   draws     =    argmax over the support of ln(w_v) + G(b, j, v),
 *                  lowest id on ties (Gumbel-max; exact in law)
 *   An empty residual (p <= q everywhere in fp32) falls back to a draw from p_i.
 *   All arithmetic is fp32; argmax and token comparisons are exact.
 *
 * Logit layout: row-major and contiguous, element type by `dtype`
 * (SPEC_BF16: 16-bit bfloat16; SPEC_FP32: IEEE float).  Any alignment of the
 * element type is accepted; 16-byte aligned rows take the vector path.
 *
 * Workspace: a caller-owned device buffer of spec_workspace_size() bytes.  It
 * must be zero-filled once before its first use (spec_workspace_init or any
 * memset).  Every call that completes leaves all of it zeroed again (its
 * counters, and each record once its last reader has read it), so one
 * workspace serves calls of any sizes and modes in any order -- eager calls
 * and replays of captured graphs alike -- with no clearing in between and no
 * state kept on the host.  Two calls that may overlap in time must not share
 * a workspace.  After a call that returned SPEC_ERR_CUDA, zero-fill it again.
 *
 * Errors: argument errors are detected on the host and returned before any
 * launch (nothing is written).  Conditions only visible in the data -- a NaN
 * or +inf logit, a row with no finite logit in stochastic mode, a token id
 * outside [0, V), a bad tree parent -- are reported per sequence through the
 * optional device `status` array (SPEC_ERR_TOKEN / SPEC_ERR_NONFINITE); such a
 * sequence gets n_accepted = -1 and an all -1 token row.  No kernel traps,
 * asserts or waits without bound.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum spec_dtype { SPEC_BF16 = 0, SPEC_FP32 = 1 };

enum spec_status {
  SPEC_OK = 0,
  SPEC_ERR_ARG = -1,          /* NULL pointer, non-positive size, bad dtype, T < 0 or not finite */
  SPEC_ERR_ALIGN = -2,        /* pointer not aligned to its element type                      */
  SPEC_ERR_TOKEN = -3,        /* (device) token id outside [0, V) or bad tree parent          */
  SPEC_ERR_NONFINITE = -4,    /* (device) NaN / +inf logit, or a row with no finite logit     */
  SPEC_ERR_UNSUPPORTED = -5,  /* e.g. stochastic tree verification, k or N above the limit    */
  SPEC_ERR_TIMEOUT = -6,      /* (device) a bounded wait on a bulk copy gave up (1 s); the    */
                              /*   sequences whose rows it held get -1 outputs                 */
  SPEC_ERR_CUDA = -7,         /* a CUDA runtime call failed (launch, event record)           */
  SPEC_ERR_WORKSPACE = -8     /* workspace NULL, misaligned or smaller than required          */
};

/* Limits of this build. */
#define SPEC_MAX_K 1024        /* drafts per sequence (spec_verify)              */
#define SPEC_MAX_TREE_N 4096   /* nodes per sequence (spec_verify_tree)          */
#define SPEC_MAX_STOP 64       /* stop ids per call (spec_verify_aux.stop_ids)   */

/* Bytes of device workspace for B sequences of k drafts (or N tree nodes) over
 * V ids.  Enough for spec_verify, spec_verify_ex and spec_verify_tree with the
 * same (B, k or N, V).  Returns 0 for invalid sizes. */
size_t spec_workspace_size(int B, int k, int V, int dtype);

/* Zero-fill a workspace on `cuda_stream` (cudaMemsetAsync).  Needed once
 * before first use.  Returns SPEC_OK or SPEC_ERR_ARG / SPEC_ERR_CUDA. */
int spec_workspace_init(void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * spec_verify -- verify B sequences of k drafted tokens.
 *
 *   target_logits  device, [B][k+1][V] of dtype (row k is the bonus row)
 *   draft_logits   device, [B][k][V] of dtype; may be NULL iff temperature == 0
 *   draft_tokens   device, [B][k] int32
 *   B, k, V        1 <= B, 1 <= k <= SPEC_MAX_K, 2 <= V < 2^31
 *   dtype          SPEC_BF16 or SPEC_FP32
 *   temperature    > 0: stochastic verification at that temperature;
 *                  == 0: greedy verification (draft_logits unused, seed unused)
 *   seed           64-bit Philox key
 *   out_tokens     device, [B][k+1] int32: the n+1 committed ids, then -1
 *   out_n_accepted device, [B] int32: n = accepted drafts in [0, k]
 *   workspace      device, >= spec_workspace_size(B, k, V, dtype) bytes, 16-byte aligned
 *   cuda_stream    cudaStream_t to launch on (NULL = legacy default stream)
 *
 * Returns SPEC_OK once the work is enqueued (the results are valid after the
 * stream reaches them), or a negative host-side error code.
 */
int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                int B, int k, int V, int dtype, float temperature, uint64_t seed,
                int32_t* out_tokens, int32_t* out_n_accepted,
                void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Optional extra outputs and timing hooks of spec_verify_ex; any field may be NULL. */
typedef struct spec_verify_aux {
  float* p_draft;      /* device [B][k]: p_i(x_i) (stochastic mode)                         */
  float* q_draft;      /* device [B][k]: q_i(x_i) (stochastic mode)                         */
  float* lse;          /* device [B][2k]: ln sum_v exp(x_v/T) of target rows 0..k-1, then   */
                       /*   of draft rows 0..k-1 (stochastic mode)                          */
  int32_t* status;     /* device [B]: SPEC_OK or the sequence's device-detected error       */
  void* events[4];     /* cudaEvent_t recorded on cuda_stream: before / after the row pass, */
                       /*   before / after the sampling pass (stochastic) -- for timing     */
  uint32_t sequence_offset; /* global index of sequence 0 in the Philox counters: a batch  */
                       /*   split across devices draws the same numbers as the whole batch  */
                       /*   when each shard passes the index of its first sequence          */

  /* ---- since ABI 1.1 (zero-initialise the struct: zero keeps each off) ---- */

  float lenience;      /* stochastic: l >= 1 ("Cascade Speculative Drafting for Even Faster */
                       /*   LLM Inference", "Asymmetric lenience"): accept when q <= l p,    */
                       /*   otherwise keep with probability l p / q; the residual stays      */
                       /*   norm(max(0, p - q)).  0 or 1 = the exact rule; any other value   */
                       /*   below 1, or not finite, is SPEC_ERR_ARG.  l > 1 changes the      */
                       /*   output law: the pages apply it only when a draft model reviews.  */
  const int32_t* stop_ids; /* device [n_stop] or NULL: the committed tokens end at the first */
                       /*   one that is a stop id ("Speculative Decoding: ...", "Constraints */
                       /*   must be applied consistently"); the later ones become -1         */
  int32_t n_stop;      /* 0..SPEC_MAX_STOP (n_stop > 0 with stop_ids NULL: SPEC_ERR_ARG)     */
  int32_t* n_committed; /* device [B] or NULL: committed tokens per sequence after the stop  */
                       /*   truncation (n_accepted + 1 without one); -1 for a bad sequence   */
  uint8_t* match_mask; /* greedy (temperature 0) only, device [B][k] or NULL: 1 iff x_i is   */
                       /*   the argmax of target row i ("Ouroboros: ...", Equation (10))     */
  int32_t* n_match;    /* greedy only, device [B] or NULL: #Match = the mask's sum           */
  int32_t* tail_runs;  /* greedy only, device [B] or NULL: maximal runs of matches after the */
                       /*   first mismatch (the segments a phrase harvester keeps)           */
                       /* Any of the three in stochastic mode: SPEC_ERR_ARG.                 */

  /* ---- since ABI 1.2 ---- */

  int32_t top_k;       /* stochastic: consistent top-k on every target and draft row ("Speculative */
                       /*   Decoding: ...", "Logit-processor gaps"): keep the ids whose logit is   */
                       /*   at least the k-th largest (ties kept); 0, or >= V, keeps every id      */
  float top_p;         /* stochastic: then consistent top-p on the top-k distribution: keep the    */
                       /*   ids at or above the largest logit whose mass at or above it reaches    */
                       /*   top_p (ties kept); 0 or 1 keeps every id.  Both are applied after the  */
                       /*   temperature, to target rows 0..k and draft rows 0..k-1 alike, and the  */
                       /*   rule runs on the renormalised rows; p_draft / q_draft report the       */
                       /*   filtered values, lse the unfiltered normalisers.  top_k < 0 or top_p   */
                       /*   outside [0, 1]: SPEC_ERR_ARG.  Greedy mode ignores both (they never    */
                       /*   move an argmax).  A NaN or +inf in the bonus row is SPEC_ERR_NONFINITE */
                       /*   for the sequence when filtering, whatever n is.                        */
} spec_verify_aux;

/* spec_verify plus the auxiliary outputs in `aux` (which may be NULL). */
int spec_verify_ex(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                   int B, int k, int V, int dtype, float temperature, uint64_t seed,
                   int32_t* out_tokens, int32_t* out_n_accepted,
                   void* workspace, size_t workspace_bytes, void* cuda_stream,
                   const spec_verify_aux* aux);

/*
 * spec_verify_tree -- greedy verification of a candidate tree per sequence.
 *
 *   target_logits  device, [B][N+1][V] of dtype; row 0 is the target's output at
 *                  the context, row 1+m its output at node m (a leaf's row is
 *                  its bonus row)
 *   node_tokens    device, [B][N] int32: the drafted id at each node
 *   parents        device, [B][N] int32: -1 = child of the context, else the
 *                  parent node, which must precede the node (parents[m] < m)
 *   temperature    must be 0 (no stochastic tree rule is defined); else
 *                  SPEC_ERR_UNSUPPORTED
 *   out_tokens     device, [B][N+1] int32: path ids from the root level down to
 *                  the chosen node, then the argmax of that node's row, then -1
 *   out_n_accepted device, [B]: depth of the chosen node (0 = none accepted)
 *   out_leaf       device, [B] or NULL: the chosen node, -1 = none
 *   status         device, [B] or NULL: per-sequence device-detected errors
 *
 * Node m is accepted iff its parent is (the context always is) and its id is
 * the argmax of its parent's row.  The deepest accepted node is chosen, the
 * lowest node index among equally deep ones.
 */
int spec_verify_tree(const void* target_logits, const int32_t* node_tokens, const int32_t* parents,
                     int B, int N, int V, int dtype, float temperature,
                     int32_t* out_tokens, int32_t* out_n_accepted, int32_t* out_leaf, int32_t* status,
                     void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * spec_random -- the randomness the rule draws, for checking (not on the hot path).
 *   Writes U(b, j, v) and G(b, j, v) for v in [0, V) (device fp32 arrays of V,
 *   either may be NULL) and, when accept_u is not NULL, U(b, i) of the accept
 *   decision i = j into accept_u[0].
 */
int spec_random(uint64_t seed, int b, int j, int V, float* gumbel_u, float* gumbel_g,
                float* accept_u, void* cuda_stream);

/*
 * spec_verify_noalloc -- spec_verify for callers that cannot allocate device
 * memory.  (The pages describe no such call: this is an interface addition of
 * this library, not part of the method.)
 *
 * Some callers have no device allocator they may use: a plugin inside a host
 * program that owns all device memory, a runtime whose memory is carved up
 * before it starts, or a latency-critical path where cudaMalloc's implicit
 * device synchronisation is not acceptable.  They cannot provide the workspace
 * spec_verify needs.  This entry point takes no workspace: the kernels use a
 * fixed array of SPEC_NOALLOC_SCRATCH_BYTES that belongs to the library's
 * device image, which every GPU that loads the library holds until exit.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   Arguments and results are those of spec_verify (inputs and outputs are
 *   still the caller's device buffers).
 *   Sizes whose spec_workspace_size(B, k, V, dtype) exceeds
 *   SPEC_NOALLOC_SCRATCH_BYTES are rejected with SPEC_ERR_WORKSPACE before any
 *   launch; use spec_verify with a workspace for those.
 *   The first call on each device looks up the array's device address (once,
 *   with that device current); make that first call before any stream capture.
 *   All calls share the one array per device.  It starts zeroed and, as a
 *   workspace, every call leaves it zeroed, so calls of any sizes, eager or
 *   replayed from a graph, can follow one another; but calls whose work may
 *   overlap on the GPU -- other streams, other host threads, a graph replay
 *   next to an eager call -- race with each other: order them on one stream.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int spec_verify_noalloc(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                        int B, int k, int V, int dtype, float temperature, uint64_t seed,
                        int32_t* out_tokens, int32_t* out_n_accepted, void* cuda_stream);

/*
 * spec_verify_guided -- greedy verification followed by a target-side guide
 * ("Double: Breaking the Acceleration Limit via Double Retrieval Speculative
 * Parallelism", "Multi-token Pre-verify" and D.2 "Proof of Lossless
 * Acceleration", greedy decoding).
 *
 *   target_logits   device, [B][k+1][V] of dtype (as spec_verify, greedy)
 *   draft_tokens    device, [B][k] int32
 *   guide           device, [B][L] int32: the target-side token for each
 *                   position 0..L-1; a negative entry ends the guide (may be
 *                   NULL when L == 0)
 *   out_tokens      device, [B][max(k+1, L)] int32
 *   out_n_accepted  device, [B]: accepted drafts n
 *   out_n_committed device, [B]: committed tokens
 *   status          device, [B] or NULL
 *
 * Committed: x_0..x_{n-1} (the drafts that equal the target argmax of their
 * row), the correction a*_n (the argmax of row n; the bonus when n = k), and,
 * when guide[n] == a*_n, the guide's tokens guide[n+1], guide[n+2], ... up to
 * its end: they follow the corrected target path.  Then -1.  A guide id >= V
 * is SPEC_ERR_TOKEN for the sequence.  Workspace: spec_workspace_size(B, k,
 * V, dtype).  Host errors as spec_verify (L < 0: SPEC_ERR_ARG).
 */
int spec_verify_guided(const void* target_logits, const int32_t* draft_tokens, const int32_t* guide,
                       int B, int k, int L, int V, int dtype,
                       int32_t* out_tokens, int32_t* out_n_accepted, int32_t* out_n_committed,
                       int32_t* status, void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * spec_probe_read -- measurement helper (not on the hot path): reads `bytes`
 * (rounded down to 16) of device memory at `data` (16-byte aligned) with the
 * row pass's load pattern and nothing else -- a persistent grid of `ctas` CTAs
 * (0 = as many as fit on the GPU at once) over contiguous ranges, 16-byte
 * loads that bypass L1, four per thread in flight -- and xors the words into
 * sink[0 .. ctas-1] (device; the caller zero-fills it).  Time it with events on
 * `cuda_stream`: bytes / time is the read ceiling the row pass streams against.
 * Returns SPEC_OK or SPEC_ERR_ARG / SPEC_ERR_CUDA.
 */
int spec_probe_read(const void* data, size_t bytes, unsigned* sink, int ctas, void* cuda_stream);

/*
 * spec_test_force_stage_timeouts -- test hook (since ABI 1.3), off by default.
 *   on != 0: from the next call on, every wait of a bulk-copy stage (the ring
 *   row pass of large greedy and tree batches, and the sampling pass of
 *   stochastic calls on 16-byte aligned rows) gives up at once, as a wait does
 *   when a copy has not landed within its 1 s limit: the affected sequences get
 *   SPEC_ERR_TIMEOUT and -1 outputs, and before a CTA exits it still waits
 *   (bounded) for the copies it has in flight.  on == 0 restores normal waits.
 *   The setting is process-wide and read when a call is queued; it is meant
 *   for tests of the timeout path, never for production calls.  Returns the
 *   previous setting.
 */
int spec_test_force_stage_timeouts(int on);

/* Human-readable name of a status code (static storage). */
const char* spec_strerror(int status);

/* ABI version of this library: (major << 16) | minor. */
int spec_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
