/*
 * specverify — the batched draft-verify step of speculative decoding on one
 * GB300 (sm_103a), behind a plain C ABI.
 *
 * What it computes.  For each of B independent sequences the target scored the
 * prefix plus k drafted tokens in one pass, giving k+1 rows of logits l_0..l_k
 * over a vocabulary of V tokens; row i judges draft x_i and row k is the bonus
 * row ("Decodificação especulativa explicada: rascunhe barato, verifique numa
 * passada", §"O ciclo de rascunho e verificação"; "Speculative decoding: el
 * secretario que adelanta lo que va a decir el jefe", §"El mecanismo desnudo",
 * paso 2).
 *
 *   p_i = softmax(l_i / T).
 *   Sampled mode: judge x_0, x_1, ... left to right and accept x_i when
 *     p_i(x_i) >= q_i(x_i) or u_accept[i] < p_i(x_i) / q_i(x_i), i.e. with
 *     probability min(1, p/q); stop at the first rejection n and draw the
 *     replacement from norm(max(0, p_n - q_n)); if all k survive, draw a bonus
 *     token from p_k ("Decodificação especulativa explicada", §"A regra de
 *     amostragem por rejeição", rules 1-3; "Speculative Decoding" (ch15, LLM
 *     serving from scratch), §"Why the result is exactly the target model").
 *   Greedy mode: accept while x_i == argmax p_i; emit argmax p_n at the first
 *     mismatch, or argmax p_k as the bonus (same sections, greedy case).
 *   A draw from weights w takes the first j whose running sum C_j exceeds
 *     u_resample * C_{V-1} ("Decodificação especulativa explicada",
 *     §"Amostragem especulativa em numpy, com prova", the sampler), so a
 *     zero-weight token is never drawn.
 *   num_accepted[b] = n is also the number of drafted positions whose KV-cache
 *     entries the caller keeps (§"O ciclo de rascunho e verificação",
 *     bookkeeping paragraph); the round emits n + 1 tokens.
 *
 * Readings where the pages are silent: a tie u == p/q rejects; p >= q always
 * accepts (so q(x) == 0 accepts); one uniform per sequence serves the single
 * draw that happens; argmax ties go to the lowest token id; a rejection whose
 * residual has zero mass (possible only through rounding or an unnormalised q)
 * draws from p instead and is counted; output positions after the drawn token
 * are -1.
 *
 * Conventions shared by every entry point.
 *  - All tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *    row-major, 16-byte aligned.  Any V >= 1 is accepted.
 *  - The library allocates nothing.  Scratch lives in the caller's workspace
 *    (ws, ws_bytes >= spec_verify_workspace_size(...)), 16-byte aligned; it
 *    needs no initialisation and may be reused by later calls on the same
 *    stream.  Calls sharing one workspace must not overlap in time.
 *  - Launches are asynchronous on `stream`; nothing synchronises except
 *    spec_verify_read_status and spec_verify_row_stats.
 *  - Argument errors return an error code synchronously and launch nothing.
 *  - Bad data found on the device (a NaN or +inf logit, an all -inf row, a draft
 *    token outside [0,V), a uniform outside [0,1), a NaN or negative q(x)) on a
 *    row or token that the scan reaches marks that sequence invalid: its
 *    num_accepted is -1 and its out_tokens row is all -1, and a bit is set in
 *    the workspace status word (spec_verify_read_status).
 *  - Limits: 1 <= k <= 64, 1 <= V <= 2^21, B >= 0, B*(k+1)*V < 2^40,
 *    B*(k+1) < 2^27.  B == 0 launches nothing (the workspace is left as it was).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad T, misaligned pointer */
    SV_ERR_WORKSPACE = 2,    /* workspace missing or smaller than required */
    SV_ERR_UNSUPPORTED = 3,  /* sizes beyond the limits above, or no sm_103a device */
    SV_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, copy) */
    SV_ERR_DATA = 5,         /* device-detected bad data (spec_verify_read_status) */
    SV_ERR_TIMEOUT = 6       /* reserved: no device-side wait exists in this version */
} sv_status;

typedef enum { SV_BF16 = 0, SV_F32 = 1 } sv_dtype;

typedef enum { SV_MODE_SAMPLE = 0, SV_MODE_GREEDY = 1 } sv_mode;

/* Bits of the device status word. */
#define SV_DEV_BAD_ROW 0x1u      /* a reached row held a NaN / +inf, or was all -inf */
#define SV_DEV_BAD_TOKEN 0x2u    /* a reached draft token outside [0, V) */
#define SV_DEV_BAD_UNIFORM 0x4u  /* a used uniform outside [0, 1) (or NaN) */
#define SV_DEV_BAD_Q 0x8u        /* q_i(x_i) NaN or negative at a reached position */
#define SV_DEV_DEGENERATE 0x10u  /* informational: a zero-mass residual drew from p */
#define SV_DEV_PRECISE 0x20u     /* informational: a draw needed the float-float pass */
#define SV_DEV_BAD_TREE 0x40u    /* spec_verify_tree: a parent index outside [0, j) at node j */

/* Bytes of workspace the calls below need for these sizes (0 for invalid sizes). */
size_t spec_verify_workspace_size(int B, int k, int V, sv_dtype dtype);

/* Greedy verify.
 *   logits       [B, k+1, V] bf16 or fp32 (dtype), the target's logits.
 *   draft_tokens [B, k] int32.
 *   out_tokens   [B, k+1] int32 (written): argmax-accepted drafts 0..n-1, the
 *                argmax token at n, -1 after.
 *   num_accepted [B] int32 (written): n in [0, k], or -1 for an invalid sequence.
 * Temperature plays no part in greedy verify. */
sv_status spec_verify_greedy(const void* logits, sv_dtype dtype,
                             const int32_t* draft_tokens, int B, int k, int V,
                             int32_t* out_tokens, int32_t* num_accepted,
                             void* ws, size_t ws_bytes, cudaStream_t stream);

/* Sampled verify (rejection sampling).
 *   logits       [B, k+1, V] bf16 or fp32, the target's logits; p = softmax(l/T).
 *   draft_probs  [B, k, V] fp32, the draft's distributions q recorded while
 *                drafting (used as given, no temperature applied).
 *   draft_tokens [B, k] int32.
 *   u_accept     [B, k] fp32 in [0, 1): uniform for the accept test at i.
 *   u_resample   [B] fp32 in [0, 1): uniform for the one draw per sequence.
 *   T            temperature, finite and > 0.
 *   out_tokens   [B, k+1] int32 (written): accepted drafts 0..n-1, the drawn
 *                token at n, -1 after.
 *   num_accepted [B] int32 (written): n in [0, k], or -1 for an invalid sequence.
 * The acceptance ratios are formed from fp32 row statistics (relative error
 * ~1e-7..1e-6).  The draw is exact up to ~1e-12: a first fp32 pass with exact
 * integer prefix sums carries a rigorous error bound D and keeps its token when
 * u_resample * C lies farther than 2D from both edges of the chosen bin;
 * otherwise (a few percent of draws, flagged SV_DEV_PRECISE) a second pass
 * recomputes the row in float-float (~48 bits), so the token matches an
 * exact-arithmetic draw except when u_resample lies within ~1e-12 of a bin
 * boundary. */
sv_status spec_verify_sample(const void* logits, sv_dtype dtype, const float* draft_probs,
                             const int32_t* draft_tokens, const float* u_accept,
                             const float* u_resample, float T, int B, int k, int V,
                             int32_t* out_tokens, int32_t* num_accepted,
                             void* ws, size_t ws_bytes, cudaStream_t stream);

/* Sample-and-match verify ("Decodificação especulativa explicada", §"A regra de
 * amostragem por rejeição", the simpler exact scheme some engines use): a
 * target token y_i is drawn from p_i = softmax(l_i / T) at every position, the
 * draft token kept while y_i == x_i; the first position i < k where they
 * differ, or position k, emits y_i.  Every emitted token is a draw from p, so
 * the output is exact, but a draft survives position i only with probability
 * sum_v p_i(v) q_i(v), never more than spec_verify_sample's acceptance.  The
 * draft's q is not needed.
 *   u_draw  [B, k] fp32 in [0, 1): the uniform of the draw at position i < k.
 *   u_bonus [B] fp32 in [0, 1): the uniform of the draw at position k.
 *   out_tokens [B, k+1]: y_0..y_n (= the accepted drafts, then the emitted
 *   draw), -1 after; num_accepted [B] = n, or -1 for an invalid sequence (a bad
 *   row, draft token or uniform at a position the scan reaches).
 * The draws are those of spec_verify_sample (certified fp32 pass, float-float
 * fallback, exact integer prefix sums).  Workspace as for the other calls. */
sv_status spec_verify_match(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                            const float* u_draw, const float* u_bonus, float T, int B, int k,
                            int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                            size_t ws_bytes, cudaStream_t stream);

/* Tree verification: several drafted continuations checked at once
 * ("Decodificação especulativa explicada", §"A família de rascunhos": Medusa
 * verifies candidate continuations with tree attention; "Speculative decoding:
 * el secretario...", §"Tree attention").  The pages name the technique but give
 * no acceptance rule; this is the plainest exact one, and with one child per
 * node it is spec_verify_greedy / spec_verify_sample.
 *   Each sequence drafts a tree of N nodes (2 <= N <= 65): node 0 is the root
 *   (the last committed token), node j >= 1 a drafted token whose parent
 *   precedes it.
 *   logits [B, N, V] bf16/fp32: the target's logits at each node (row j: the
 *     distribution of the token after node j), e.g. from one tree-attention pass;
 *   tree_tokens [B, N] int32: node j's token (entry 0 unused);
 *   tree_parents [B, N] int32: node j's parent, 0 <= parent < j (entry 0 unused);
 *   draft_probs [B, N, V] fp32 (sampled): the draft distribution at each node,
 *     from which that node's children were drawn, independently;
 *   u_accept [B, N] fp32 (sampled): the uniform of child j's test (entry 0 unused);
 *   u_resample [B] fp32 (sampled): the uniform of the final draw.
 * The walk starts at the root.  Greedy: the first child (in index order) whose
 * token is the node's argmax is accepted and the walk moves on to it; when none
 * is, the argmax is emitted.  Sampled: the node's current distribution r starts
 * as p = softmax(logits/T); child j (token x) is accepted iff r(x) >= q(x) or
 * u_accept[j] < r(x)/q(x); a rejection replaces r by the normalised residual
 * max(0, r - q) (by p again when that has no mass: SV_DEV_DEGENERATE); an
 * accepted child continues the walk with its own p; when no child of the node
 * is accepted the token is drawn from r with u_resample (the categorical rule
 * of spec_verify_sample, in fp32 weights with float64 sums).
 *   out_tokens [B, N]: the accepted tokens, then the emitted one, -1 after;
 *   out_nodes [B, N]: the accepted node indices (to keep their KV entries), -1
 *     after;
 *   num_accepted [B]: the accepted count, or -1 for an invalid sequence (a
 *     parent outside [0, j): SV_DEV_BAD_TREE; or a row, token, uniform or q(x)
 *     the walk reaches that is bad, as for the chain).
 * Workspace: spec_verify_workspace_size(B, N - 1, V, dtype) bytes; status and
 * row statistics as for the chain calls (row_stats with k = N - 1). */
sv_status spec_verify_tree(sv_mode mode, const void* logits, sv_dtype dtype,
                           const float* draft_probs, const int32_t* tree_tokens,
                           const int32_t* tree_parents, const float* u_accept,
                           const float* u_resample, float T, int B, int N, int V,
                           int32_t* out_tokens, int32_t* out_nodes, int32_t* num_accepted,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/* N-gram (prompt-lookup) drafter: proposals that need no draft model
 * ("Decodificação especulativa explicada", §"A família de rascunhos";
 * "Speculative Decoding" (ch15), §"What proposes the tokens", NgramDrafter).
 *   history [B, Lmax] int32 DEVICE: each sequence's tokens so far, row-major;
 *   lengths [B] int32 DEVICE: tokens in each row (clamped to [0, Lmax]).
 * For n = n_max down to n_min, the last n tokens of a sequence are looked for
 * earlier in its history; the first n that occurs wins, and of its occurrences
 * the most recent; the draft is the up to k tokens that followed it.
 *   draft_tokens [B, k] int32 (written): the proposal, -1 after num_drafted;
 *   num_drafted [B] int32 (written): 0 when nothing occurs earlier.
 * Such a proposal is a point mass: sampled verification takes q = one-hot at
 * each proposed token.  Limits: 1 <= k <= 64, 1 <= n_min <= n_max <= 32.
 * Asynchronous on `stream`; argument errors return before any launch. */
sv_status spec_ngram_draft(const int32_t* history, const int32_t* lengths, int B, int Lmax,
                           int k, int n_min, int n_max, int32_t* draft_tokens,
                           int32_t* num_drafted, cudaStream_t stream);

/* Counters a verify can add to (spec_verify_*_kv), for generation loops that
 * keep speculation statistics on the device ("Speculative Decoding" (ch15, LLM
 * serving from scratch), the stats argument of speculative_generate; the
 * tokens-per-target-pass figure of "Decodificação especulativa explicada",
 * §"Quanto mais rápido: a matemática" is emitted / rounds). */
typedef struct {
    unsigned long long rounds;    /* valid sequences verified: one target pass each */
    unsigned long long proposed;  /* drafted tokens judged: k per valid sequence */
    unsigned long long accepted;  /* accepted drafts: the sum of num_accepted */
    unsigned long long emitted;   /* tokens emitted: the sum of num_accepted + 1 */
    unsigned long long invalid;   /* sequences marked invalid (num_accepted = -1) */
} sv_spec_stats;

/* spec_verify_sample / spec_verify_greedy with the bookkeeping of a generation
 * loop fused into the kernel that writes num_accepted ("Decodificação
 * especulativa explicada", §"O ciclo de rascunho e verificação", bookkeeping
 * paragraph: the entries after the first rejection are dropped):
 *   kv_len [B] int32 DEVICE (may be NULL): kv_len[b] += num_accepted[b] + 1 for
 *          every valid sequence (the n accepted drafts and the drawn token);
 *          unchanged for an invalid one.
 *   stats  DEVICE sv_spec_stats (may be NULL): counters added atomically; the
 *          caller zeroes them when it wants a fresh count.
 * Both 16-byte aligned.  All other arguments, results and errors as for the
 * calls without _kv. */
sv_status spec_verify_sample_kv(const void* logits, sv_dtype dtype, const float* draft_probs,
                                const int32_t* draft_tokens, const float* u_accept,
                                const float* u_resample, float T, int B, int k, int V,
                                int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                                cudaStream_t stream);
sv_status spec_verify_greedy_kv(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                                int B, int k, int V, int32_t* out_tokens, int32_t* num_accepted,
                                void* ws, size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                                cudaStream_t stream);

/* The work of spec_verify_greedy / spec_verify_sample, split at its one internal dependency so
 * that each half can be timed or overlapped separately.  spec_verify_rows
 * streams every logits row once and leaves per-row statistics (max, normaliser,
 * argmax, gathered l(x), q(x), p(x)) in ws; for greedy batches that take the
 * flat stream (the whole tensor cut into one range per resident CTA) it leaves
 * each range's partial argmax keys instead, which spec_verify_finish merges
 * into the row statistics.  spec_verify_finish then runs the accept scan and
 * the draws from ws and writes the outputs.  Calling rows then
 * finish on one stream with the same arguments is exactly spec_verify_greedy
 * (mode SV_MODE_GREEDY; draft_probs, u_accept, u_resample may be NULL, T is
 * ignored) or spec_verify_sample (mode SV_MODE_SAMPLE). */
sv_status spec_verify_rows(sv_mode mode, const void* logits, sv_dtype dtype,
                           const float* draft_probs, const int32_t* draft_tokens,
                           float T, int B, int k, int V, void* ws, size_t ws_bytes,
                           cudaStream_t stream);
sv_status spec_verify_finish(sv_mode mode, const void* logits, sv_dtype dtype,
                             const float* draft_probs, const int32_t* draft_tokens,
                             const float* u_accept, const float* u_resample, float T,
                             int B, int k, int V, int32_t* out_tokens,
                             int32_t* num_accepted, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* Sampled verify for callers that cannot allocate device memory.  Some callers
 * are handed only their input and output tensors and have no way to allocate a
 * workspace: operator plug-ins inside an inference engine that owns all device
 * memory, or serving loops that forbid device allocation once they have started
 * (an allocation can synchronise the device and stall every stream).  This entry
 * point takes the same arguments as spec_verify_sample minus the workspace, and
 * keeps its scratch in a fixed array inside this library instead.  (The pages
 * describe no such variant; it is an interface convenience.)
 *   - Limit: B*(k+1) <= SV_NOALLOC_MAX_ROWS rows; larger batches return
 *     SV_ERR_WORKSPACE and launch nothing.  The array is SV_NOALLOC_SCRATCH_BYTES
 *     of device memory, held by every GPU that loads the library until exit.
 *   - The first call made with a given device current looks up the array's
 *     device address (cudaGetSymbolAddress) and caches it; make that first call
 *     before any stream capture begins on that device.
 *   - Every call shares the one array and leaves its contents behind; nothing in
 *     it needs to start at zero: each call writes every header field and row
 *     record before reading it, and clears the counters that must start at zero
 *     itself (cudaMemsetAsync on the call's stream).  Calls that overlap on the
 *     GPU (for example on two streams at once) race on the array and must be
 *     avoided.
 *   - It allocates nothing and calls no allocating routine; the result and the
 *     device-detected data errors (num_accepted = -1) are as for
 *     spec_verify_sample. */
#define SV_NOALLOC_SCRATCH_BYTES 1048576
#define SV_NOALLOC_MAX_ROWS 27000
sv_status spec_verify_sample_noalloc(const void* logits, sv_dtype dtype,
                                     const float* draft_probs, const int32_t* draft_tokens,
                                     const float* u_accept, const float* u_resample, float T,
                                     int B, int k, int V, int32_t* out_tokens,
                                     int32_t* num_accepted, cudaStream_t stream);

/* Synchronises `stream`, then ORs the per-sequence status words of the last
 * call that used `ws` into *device_status (SV_DEV_* bits).  Returns SV_ERR_DATA
 * if any error bit (all but SV_DEV_DEGENERATE and SV_DEV_PRECISE) is set, else
 * SV_OK.  *n_degenerate (may be NULL) receives the number of zero-mass residual
 * draws. */
sv_status spec_verify_read_status(const void* ws, cudaStream_t stream,
                                  uint32_t* device_status, uint32_t* n_degenerate);

/* Debug / test: synchronises `stream` and copies the per-row statistics of the
 * last call that used `ws` to HOST arrays of B*(k+1) entries each (any may be
 * NULL): m = max_j l_j (the largest raw logit; max_j l_j/T = m/T),
 * S = sum_j exp((l_j - m)/T), argmax (lowest index of the largest raw logit),
 * px = p_i(x_i) and qx = q_i(x_i) (NaN on row k; px and S are 0 in greedy
 * mode, which does not form them). */
sv_status spec_verify_row_stats(const void* ws, cudaStream_t stream, int B, int k,
                                float* m, float* S, int32_t* argmax, float* px,
                                float* qx);

/* Static description of a status code. */
const char* spec_verify_status_string(sv_status status);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
