/*
 * spec_verify.h -- C ABI of libspecverify.so: the verification step of
 * speculative decoding on one NVIDIA GB300 (sm_103a).
 *
 * What the calls compute is stated on these pages (cited by title and
 * section):
 *   [EIN]  Edge Inference Notes, post on speculative decoding and EAGLE-3:
 *          "The core idea: draft, then check" (step 3, accept or correct),
 *          "Why it changes nothing about the output" (temperature, top-k and
 *          nucleus adjust both distributions before the test) and
 *          "One decode round, end to end" (greedy token tree, longest agreed
 *          path plus one correction).
 *   [TGTG] "Towards Green Text Generation: Memory-Based Speculative
 *          Decoding", section 2.4 "Verifier and Acceptance" (greedy chain
 *          verification of k drafts from k+1 target rows) and section 5.1
 *          "The Verifier Cost Model" (equation 1).
 *   [SDSC] "Speculative Decoding Speedup Calculator", steps 1-3.
 *
 * Conventions shared by every entry point:
 *   - Array arguments are DEVICE pointers owned by the caller, contiguous,
 *     row-major, row stride V, aligned to their element size.  Rows whose
 *     start is 16-byte aligned (V * element size a multiple of 16 and the
 *     base 16-byte aligned) take the bulk-copy fast path; others are read
 *     with plain loads and give the same results.
 *   - Every call is asynchronous on `cuda_stream` (a cudaStream_t, NULL for
 *     the legacy default stream), allocates nothing and does not synchronise.
 *   - `workspace` is caller-owned device memory of at least
 *     spec_verify_workspace_size(...) bytes, 256-byte aligned, ZEROED ONCE
 *     when it is created.  Every kernel leaves it zeroed again (apart from
 *     the status word), so it can be reused by later calls on the same
 *     stream.  Two calls that may run concurrently need separate workspaces.
 *   - Return codes are SPEC_OK or a negative SPEC_ERR_* value; argument
 *     errors are detected on the host before anything is launched.  Errors
 *     found in the data on the device (out-of-range tokens, NaN/+inf rows,
 *     malformed parent arrays) never trap: they set bits of the status word
 *     in the workspace, read with spec_get_status().
 *   - Ties are broken to the lowest token index (argmax, top-k cut) and to
 *     the lowest node index (deepest agreed tree node).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Return codes. */
#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG (-1)  /* null pointer, bad size, bad parameter     */
#define SPEC_ERR_DTYPE (-2)        /* dtype is not SPEC_F32 / SPEC_BF16         */
#define SPEC_ERR_WORKSPACE (-3)    /* workspace too small or misaligned         */
#define SPEC_ERR_LAUNCH (-4)       /* a CUDA launch or copy failed              */
#define SPEC_ERR_DEVICE_DATA (-5)  /* spec_get_status found a status bit set    */
#define SPEC_ERR_TIMEOUT (-6)      /* a bounded device wait gave up             */
#define SPEC_ERR_UNSUPPORTED (-7)  /* shape beyond the library's limits         */
#define SPEC_ERR_SCRATCH_LIMIT (-8) /* B or B*(k+1) beyond the fixed scratch of
                                       spec_verify_sample_noalloc              */

/* Status bits written by the device (bitwise OR, sticky until read). */
#define SPEC_STATUS_BAD_TOKEN 1u   /* a draft token outside [0, V): rejected    */
#define SPEC_STATUS_BAD_ROW 2u     /* a row with NaN, +inf or no finite entry,
                                      or a per-sequence temperature <= 0        */
#define SPEC_STATUS_BAD_PARENT 4u  /* parents[0] != -1 or parents[j] not in [0, j) */
#define SPEC_STATUS_DEPTH 8u       /* an agreed tree node deeper than max_depth */
#define SPEC_STATUS_TIMEOUT 16u    /* a bounded device wait gave up             */
#define SPEC_STATUS_BAD_KV 32u     /* spec_kv_compact: a path, length or block
                                      lookup out of range (sequence left out)   */

/* Limits. */
#define SPEC_MAX_K 31              /* drafts per sequence                       */
#define SPEC_MAX_TREE_NODES 1024   /* nodes per tree                            */
#define SPEC_MAX_V (1 << 24)       /* vocabulary size                           */

/*
 * Sampling parameters ([EIN] "Why it changes nothing about the output": the
 * same temperature and filters are applied to the target row p and to the
 * draft row q before the accept test).
 *   temperature          scalar T > 0, used when temperature_per_seq is NULL
 *   temperature_per_seq  device float[B] (per sequence, or per row for
 *                        spec_transform_probs), or NULL
 *   top_k                0 = off, else keep the top_k highest-ranked tokens
 *                        (rank = value descending, index ascending)
 *   top_p                in (0, 1]; 1 = off.  Applied after top-k, on the
 *                        renormalised top-k distribution: a token is kept iff
 *                        the mass ranked strictly before it is < top_p.
 */
typedef struct {
  float temperature;
  const float* temperature_per_seq;
  int top_k;
  float top_p;
} spec_sampling_params;

/*
 * Workspace bytes needed by spec_verify_sample / spec_verify_greedy for B
 * sequences of k drafts, by spec_verify_tree_greedy and spec_verify_tree_sample
 * with k = N - 1, and by
 * spec_transform_probs with B = R rows and k = 0.  Returns 0 for sizes
 * outside the limits.
 */
size_t spec_verify_workspace_size(int B, int k, int V, spec_dtype dtype);

/*
 * Speculative-sampling verification ([EIN] "The core idea: draft, then
 * check", step 3).  For every sequence b, left to right over i = 0..k-1:
 *   p_i = filter(softmax(target[b][i] / T)), q_i = filter(softmax(draft[b][i] / T))
 *   accept x_i = draft_tokens[b][i]  iff  u_i * q_i(x_i) < p_i(x_i)
 *   (i.e. with probability min(1, p/q)); stop at the first rejection, n = i.
 *   If n < k, draw one token from max(0, p_n - q_n) / S with u_{k+1};
 *   else draw the bonus token from p_k with u_k.  Draws take the smallest
 *   index j whose running sum (ascending index order) exceeds u * S.
 *   A residual of total mass 0 (reachable only through rounding) is replaced
 *   by p_n.
 *
 *   target_logits     [B][k+1][V] dtype   target rows at the k+1 positions
 *   draft_logits      [B][k][V]   dtype   draft LOGITS (q = filtered softmax
 *                                         of draft_logits / T); a caller that
 *                                         holds probabilities passes log q
 *   draft_tokens      [B][k]      int32
 *   uniforms          [B][k+2]    float   in [0, 1): u_0..u_{k-1} accept
 *                                         tests, u_k bonus, u_{k+1} resample
 *   B >= 1, 1 <= k <= SPEC_MAX_K, 1 <= V <= SPEC_MAX_V
 *   params            HOST pointer
 *   out_tokens        [B][k+1]    int32   x_0..x_{n-1}, drawn token, then -1
 *   out_num_accepted  [B]         int32   n in [0, k]; n + 1 tokens committed
 *   out_p_draft, out_q_draft  [B][k] float or NULL: p_i(x_i), q_i(x_i) for
 *                     every i (computed for all positions, not only i <= n)
 * A draft token outside [0, V) is rejected and sets SPEC_STATUS_BAD_TOKEN;
 * a non-finite row gives drawn token -1 and sets SPEC_STATUS_BAD_ROW.
 */
int spec_verify_sample(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* uniforms, int B, int k,
                       int V, spec_dtype dtype, const spec_sampling_params* params,
                       int32_t* out_tokens, int32_t* out_num_accepted, float* out_p_draft,
                       float* out_q_draft, void* workspace, size_t workspace_bytes,
                       void* cuda_stream);

/*
 * The rejection fast path ([TGTG] section 2.4, KV-cached regime): the first
 * draft token is checked against the previous step's logits (already
 * computed), so that the k-token verification pass runs only when it is
 * accepted.  For every sequence b, a = argmax of prev_rows[b] (raw logits,
 * lowest index on ties):
 *   prev_rows   [B][V] dtype   device
 *   draft0      [B]    int32   device: each sequence's first draft token
 *   out_accept  [B]    int32   device: 1 iff draft0[b] == a, else 0
 *   out_argmax  [B]    int32   device: a (the token to commit on rejection)
 * Workspace: spec_verify_workspace_size(B, 1, V, dtype) bytes, as for
 * spec_verify_greedy (left zeroed).  Greedy only: the pages check the first
 * token by exact match.
 */
int spec_first_draft_check(const void* prev_rows, const int32_t* draft0, int B, int V,
                           spec_dtype dtype, int32_t* out_accept, int32_t* out_argmax,
                           void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Greedy chain verification ([TGTG] section 2.4): a_i = argmax of the raw
 * target row i (lowest index on ties; temperature and filters do not change
 * an argmax and are not taken); n = first i < k with x_i != a_i, else k.
 *   target_logits [B][k+1][V], draft_tokens [B][k]
 *   out_tokens [B][k+1] = x_0..x_{n-1}, a_n, then -1; out_num_accepted [B] = n
 */
int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int k,
                       int V, spec_dtype dtype, int32_t* out_tokens, int32_t* out_num_accepted,
                       void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Greedy token-tree verification ([EIN] "One decode round, end to end").
 * Node 0 of every tree is the root (the last committed token, its token is
 * ignored); row j of node_logits is the target's distribution for the token
 * after node j.  Node j (j >= 1) is agreed iff its parent is agreed and
 * node_tokens[j] == argmax(row parents[j]).  The deepest agreed node d*
 * (lowest index among equally deep ones) is committed with its path.
 *   node_logits  [B][N][V], node_tokens [B][N], parents [B][N]
 *                (parents[0] = -1, 0 <= parents[j] < j), 1 <= N <= 1024
 *   max_depth    >= 1, at least the depth of every node that can be agreed
 *   out_tokens   [B][max_depth+1]: tokens of the path root-exclusive, then
 *                argmax(row d*), then -1
 *   out_path     [B][max_depth+1]: node ids of the path (root excluded), -1 padded;
 *                for a KV cache these are the nodes to keep, node out_path[d]
 *                moving to position d + 1 after the root
 *   out_num_accepted [B] = depth(d*)
 * A malformed parent entry sets SPEC_STATUS_BAD_PARENT (that node is not
 * agreed); an agreed node deeper than max_depth is ignored and sets
 * SPEC_STATUS_DEPTH.
 */
int spec_verify_tree_greedy(const void* node_logits, const int32_t* node_tokens,
                            const int32_t* parents, int B, int N, int V, int max_depth,
                            spec_dtype dtype, int32_t* out_tokens, int32_t* out_path,
                            int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                            void* cuda_stream);

/*
 * Token-tree sampling verification ([EIN] "One decode round, end to end":
 * the accept-or-correct rule of "The core idea: draft, then check" applied
 * down the branches).  Per tree, from the root (node 0):
 *   p = softmax(node_logits[v] / T), q = softmax(draft_logits[v] / T), r = p;
 *   for each child j of v (parents[j] == v) in ascending node order:
 *     accept j iff u_j * q(x_j) < r(x_j)  -> commit x_j, v = j, start again;
 *     else r = max(0, r - q) / sum(max(0, r - q))  (r = p if that sum is 0);
 *   no child accepted: draw one token from r with u_0 (smallest index whose
 *   running sum exceeds u_0 * S) and stop.
 * The pages give the rule for a chain; the sibling rule above is the reading
 * taken for several children (each rejected child removes q from the
 * residual), which keeps the output distributed as p when the children of a
 * node are independent draws from q.  Temperature only (no top-k / top-p).
 *   node_logits   [B][N][V] dtype  target row of every node (row j: the
 *                                  distribution of the token after node j)
 *   draft_logits  [B][N][V] dtype  draft row of every node (row j: the
 *                                  distribution the children of j were drawn
 *                                  from; rows of leaves are not read)
 *   node_tokens, parents [B][N]    as for spec_verify_tree_greedy
 *   uniforms      [B][N] float     in [0, 1): u_0 the final draw, u_j (j >= 1)
 *                                  the accept test of node j
 *   temperature   T > 0, used when temperature_per_tree is NULL
 *   temperature_per_tree  device float[B] (T of every tree) or NULL; a tree whose
 *                 T is not finite and positive ends at its root with drawn
 *                 token -1 and SPEC_STATUS_BAD_ROW
 *   out_tokens    [B][max_depth+1] path tokens (root excluded), the drawn
 *                                  token, then -1
 *   out_path      [B][max_depth+1] path node ids, -1 padded (the KV keep list)
 *   out_num_accepted [B]           accepted nodes n (n + 1 tokens committed)
 * Children of a node at depth max_depth are not tested (SPEC_STATUS_DEPTH if
 * the walk stops there).  A child whose token is outside [0, V) is skipped
 * and sets SPEC_STATUS_BAD_TOKEN; a malformed parent entry detaches that node
 * and sets SPEC_STATUS_BAD_PARENT; a non-finite row on the walk ends it with
 * drawn token -1 and SPEC_STATUS_BAD_ROW.
 * Workspace: spec_verify_workspace_size(B, N - 1, V, dtype), left zeroed.
 * Returns SPEC_ERR_UNSUPPORTED when a CTA's share of the two rows, 2 *
 * ceil(V / 8) elements, exceeds 200 KiB of shared memory (V > 204800 f32 or
 * 409600 bf16).
 */
int spec_verify_tree_sample(const void* node_logits, const void* draft_logits, const int32_t* node_tokens,
                            const int32_t* parents, const float* uniforms, int B, int N, int V, int max_depth,
                            spec_dtype dtype, float temperature, const float* temperature_per_tree,
                            int32_t* out_tokens, int32_t* out_path, int32_t* out_num_accepted,
                            void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * KV-cache bookkeeping after a verification pass ([TGTG] section 2.4,
 * KV-cached regime: on rejection the cache is cut back to the accepted
 * prefix; [EIN] "One decode round, end to end": the longest agreed path is
 * committed and the other branches collapse).
 *
 * The verification pass wrote one cache entry per input position of
 * sequence b: node j of its flattened tree (node 0 the root, the last
 * committed token) at logical position kv_base[b] + j.  A chain of k drafts
 * is the tree whose node j (1 <= j <= k) is draft j - 1; pass path = NULL.
 * With n accepted nodes the cache keeps the root's entry and those of the
 * path's nodes, in path order, at logical positions kv_base[b] + d,
 * d = 0..n, and ends there: every other entry of the pass is dropped.  The
 * committed correction token has no entry yet (the next pass writes it).
 *
 *   path          [B][path_stride] int32 device: node ids of the accepted
 *                 path, root excluded (out_path of spec_verify_tree_greedy /
 *                 spec_verify_tree_sample), or NULL for a chain
 *   num_accepted  [B] int32 device: n
 *   kv_base       [B] int32 device: logical position of node 0's entry
 *   block_table   [B][max_blocks] int32 device: physical block of every
 *                 logical block of the sequence (paged cache, block_size
 *                 entries per block), or NULL: slots are logical positions
 *   out_src, out_dst  [B][max_keep] int32 device: slot of the d-th kept
 *                 entry now (src) and after the cut (dst), d = 0..n; -1 after
 *   out_new_len   [B] int32 device: kv_base + n + 1 (logical length)
 *   out_num_moves [B] int32 device or NULL: kept entries with src != dst.
 *                 Path node ids increase along a path and are >= their
 *                 depth, so the moves are a suffix of the list and each
 *                 dst is below its src: copying entry by entry in
 *                 ascending d overwrites no source still to be read.
 *   out_status    [1] uint32 device or NULL: SPEC_STATUS_BAD_KV is OR-ed
 *                 in (the caller clears it) when a sequence's n is
 *                 negative, n + 1 > max_keep, a path entry is not above the
 *                 one before it (or below 1), kv_base is negative, a
 *                 position exceeds INT32_MAX, or a block lookup falls
 *                 outside [0, max_blocks) or reads a negative block; that
 *                 sequence gets -1 everywhere and 0 moves.
 * B >= 1, max_keep >= 1, path_stride >= 1 when path is set, block_size >= 1
 * and max_blocks >= 1 when block_table is set.  No workspace; one launch.
 */
int spec_kv_compact(const int32_t* path, int path_stride, const int32_t* num_accepted, const int32_t* kv_base,
                    const int32_t* block_table, int max_blocks, int block_size, int B, int max_keep,
                    int32_t* out_src, int32_t* out_dst, int32_t* out_new_len, int32_t* out_num_moves,
                    uint32_t* out_status, void* cuda_stream);

/*
 * The filtered, normalised distribution the accept test uses, written out
 * for R independent rows ([EIN] "Why it changes nothing about the output").
 *   logits [R][V] dtype -> out_probs [R][V] float (0 outside the kept set).
 * params->temperature_per_seq, if set, is indexed by row.
 */
int spec_transform_probs(const void* logits, int R, int V, spec_dtype dtype,
                         const spec_sampling_params* params, float* out_probs, void* workspace,
                         size_t workspace_bytes, void* cuda_stream);

/*
 * Copies the status word of `workspace` to *status (host), then clears it.
 * Synchronises with `cuda_stream`.  Returns SPEC_OK if no bit was set,
 * SPEC_ERR_DEVICE_DATA if one was, SPEC_ERR_LAUNCH if the copy failed.
 */
int spec_get_status(void* workspace, uint32_t* status, void* cuda_stream);

/*
 * spec_verify_sample without a workspace: allocates nothing.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot obtain device memory for a workspace.  Examples: a serving
 * process whose memory manager reserved nearly all of HBM for its KV-cache
 * pool at start-up and treats any other cudaMalloc as an error; code
 * embedded in another runtime that forbids allocating outside that
 * runtime's own allocator; a decode loop that cannot afford the implicit
 * device-wide synchronisation that cudaFree performs.
 *
 * Arguments, layouts, results and data-error behaviour are those of
 * spec_verify_sample, except that there is no workspace and:
 *   out_status  [1] uint32 device pointer or NULL: receives the status bits
 *               (SPEC_STATUS_*) of this call only.
 * Limits: B <= SPEC_NOALLOC_MAX_B and B*(k+1) <= SPEC_NOALLOC_MAX_UNITS;
 * larger shapes return SPEC_ERR_SCRATCH_LIMIT before anything is launched.
 *
 * Scratch: a fixed array of about 18 MiB in the library's device memory, held on
 * every GPU that loads the library until the process exits.  The first call
 * on a device (with that device current) looks up the array's device
 * address; make that first call before any stream capture.  Every call
 * clears the part of the array it uses (cudaMemsetAsync on cuda_stream),
 * then launches the kernels; no call allocates or frees memory.  All calls
 * on one device share the one array: two calls whose work overlaps on the
 * GPU (different streams, no ordering between them) race and give wrong
 * results.  Calls on one stream are ordered and safe.
 */
#define SPEC_NOALLOC_MAX_B 256
#define SPEC_NOALLOC_MAX_UNITS 256
int spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                               const int32_t* draft_tokens, const float* uniforms, int B,
                               int k, int V, spec_dtype dtype,
                               const spec_sampling_params* params, int32_t* out_tokens,
                               int32_t* out_num_accepted, float* out_p_draft,
                               float* out_q_draft, uint32_t* out_status, void* cuda_stream);

/*
 * How the sampling entry points launch, for the whole process (a setting,
 * not a request of the pages):
 *   SPEC_LAUNCH_ROWS      one launch with one CTA per row: the row streams
 *                         through shared memory by bulk copies; the values
 *                         within 2^-12 of the running maximum's mass are
 *                         listed as candidates, from which the filter's cut,
 *                         its ties and the draw are decided (rows whose kept
 *                         set outgrows the list are searched again from L2);
 *                         the second CTA of each (target, draft) pair takes
 *                         the accept test and draws at a rejection.  Used for
 *                         bf16 rows with or without a filter and for f32 rows
 *                         without one, up to V * element bytes = 512 KiB; other
 *                         shapes take SPEC_LAUNCH_FUSED.  Faster than the
 *                         fused launch where the kept set is wide
 *                         (top-p near 1 over flat rows) or the temperature
 *                         varies per sequence.
 *   SPEC_LAUNCH_AUTO      (the default) SPEC_LAUNCH_SPLIT for calls whose
 *                         nucleus reaches deep below the row maximum
 *                         (0.95 <= top_p < 1) or whose temperature varies per
 *                         sequence, where the split launch is the faster one;
 *                         SPEC_LAUNCH_FUSED for the others.  For
 *                         spec_verify_sample_noalloc and spec_transform_probs
 *                         it means SPEC_LAUNCH_FUSED.
 *   SPEC_LAUNCH_SPLIT     three launches: a stream kernel reads every row
 *                         once in one wave of equal ranges, keeping per row
 *                         piece its maximum, its softmax mass and exact
 *                         counts of the 512 bf16 values below its maximum;
 *                         a row kernel merges the pieces and decides each
 *                         row's kept set and p(x) or q(x) (searching the row
 *                         again when the cut lies below those 512 values);
 *                         a draw kernel (one 8-CTA cluster per sequence)
 *                         finds n and draws at n from the two rows.  Used
 *                         for rows that start on 16-byte boundaries and hold
 *                         whole 16-byte vectors, bf16 with or without a
 *                         filter and f32 without one; other calls take
 *                         SPEC_LAUNCH_FUSED.
 *   SPEC_LAUNCH_FUSED     one cooperative launch whose CTAs
 *                         take every row's stream part, then every row's
 *                         tail part (the separate launches stand in when the
 *                         GPU refuses it)
 *   SPEC_LAUNCH_SEPARATE  a stream launch, then a tail launch
 *   SPEC_LAUNCH_FUSED_WAIT_TEST  failure detection without a fault: the
 *                         SPEC_LAUNCH_ROWS launch with its bulk copies withheld and a
 *                         short poll limit (or, for shapes it does not take,
 *                         the fused launch with its completion flags
 *                         withheld): every bounded wait runs out, every row
 *                         is treated as non-finite and SPEC_STATUS_TIMEOUT is
 *                         set; nothing is left in flight
 * spec_transform_probs always takes the stream and tail kernels.  Every mode
 * gives the same results outside decisions within rounding of their edge.
 * Returns the previous mode, or SPEC_ERR_INVALID_ARG for an unknown one.
 */
#define SPEC_LAUNCH_FUSED 1
#define SPEC_LAUNCH_SEPARATE 0
#define SPEC_LAUNCH_FUSED_WAIT_TEST 2
#define SPEC_LAUNCH_ROWS 3
#define SPEC_LAUNCH_SPLIT 4
#define SPEC_LAUNCH_AUTO 5
int spec_sample_launch_mode(int mode);

/* Static description of a return code. */
const char* spec_error_string(int code);

/* [SDSC] step 1: expected tokens per pass, 1 + a + ... + a^gamma. */
double spec_expected_tokens(double alpha, int gamma);

/* [SDSC] steps 2-3: E(alpha, gamma) / (gamma * c + 1). */
double spec_improvement_factor(double alpha, int gamma, double c);

/* [TGTG] section 5.1, equation 1: break-even acceptance k / (k + 1). */
double spec_break_even_acceptance(int k);

/*
 * [SDSC] the draft-length scan: the gamma in 1..gamma_max with the largest
 * spec_improvement_factor(alpha, gamma, c), the smallest such gamma on ties;
 * that speedup is written to *best_factor (may be NULL).  Host only.
 * Returns gamma, or SPEC_ERR_INVALID_ARG unless 0 <= alpha <= 1, c >= 0 and
 * 1 <= gamma_max <= 64.
 */
int spec_best_gamma(double alpha, double c, int gamma_max, double* best_factor);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
