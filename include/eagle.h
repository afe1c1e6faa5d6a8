/*
 * eagle.h -- C ABI of the GB300 (sm_103a) draft-tree verify-and-accept library.
 *
 * One step of EAGLE-style speculative decoding, split into the calls below:
 *   eagle2_expand        EAGLE-2 draft-tree expansion and reranking, fed by the
 *                        draft LM-head GEMM (tcgen05 tensor cores)
 *   eagle_tree_attn      tree-masked GQA attention of the tree nodes over the
 *                        committed KV cache plus their own ancestors
 *   eagle_verify_accept  temperature softmax + Leviathan rejection walk over the
 *                        tree, residual / bonus sampling, greedy mode at T = 0
 *   eagle_kv_compact     move the accepted path's K/V rows behind the committed
 *                        prefix and advance the logical length
 * plus two building blocks exposed for measurement and testing
 * (eagle_softmax_stats, eagle_lmhead_gemm), and the draft head's
 * training-time-test attention (eagle_ttt_attn).
 *
 * Pages (cited by title and section):
 *   Lesson: "推测解码与 EAGLE-3" -- "不变量：Leviathan 拒绝采样", "KV cache 回滚",
 *           "动手构建" steps 1-4.
 *   Guide:  "EAGLE-1/2/3 拆解：推测解码省的是大模型前向次数，赚不赚看草稿准确率" --
 *           "无损性的来源与它的证明位置", "EAGLE-2：草稿树的 Expansion 与 Reranking",
 *           "EAGLE-3：取消特征约束..." (the draft head's own lm_head),
 *           "一次 eagenerate 调用的完整流转".
 *   TTT:    "EAGLE-3 完全拆解：Training-Time Test ..." -- "EAGLE-3 和 EAGLE-2 动态树如何拼在一起",
 *           "训练时的 attention mask 为什么要特殊处理".
 *
 * Conventions shared by every call
 *   - Every pointer is caller-owned DEVICE memory unless stated otherwise; the
 *     library never allocates, frees, synchronises or prints.  Arrays are dense
 *     row-major in the shapes given.  bf16 data is passed as raw 16-bit words.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work; results are ready when the stream is.
 *   - Host-checkable errors (bad sizes, NULL pointers, unsupported shapes) return
 *     a non-zero eagle_status and launch nothing.
 *   - An empty batch (B == 0; rows == 0 or M == 0 for the row-wise calls;
 *     n_layers == 0 for compaction) is a no-op: once the sizes and scalars pass
 *     their checks the call returns EAGLE_OK without touching the device, and its
 *     device pointers may be NULL (host tables such as shard bounds are still
 *     checked).
 *   - Errors only visible in device data never trap: the kernel skips the
 *     affected sequence (accept_len = -1 where there is one), and ORs an
 *     EAGLE_DEV_* bit into *dev_status (an int32 in device memory the caller
 *     zeroes and reads when it synchronises).  dev_status may be NULL.
 *   - No global mutable state, except the fixed tree-state array behind
 *     eagle2_expand_static_state; other calls on different streams are
 *     independent unless they share output buffers.
 *   - Shapes: n (tree nodes, root included) <= 64; head_dim == 128;
 *     Hq % Hkv == 0; temperature == 0 selects greedy decoding.
 */
#ifndef EAGLE_GB300_H
#define EAGLE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EAGLE_OK = 0,
    EAGLE_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, T < 0 ...      */
    EAGLE_ERR_SHAPE = 2,        /* unsupported shape (n > 64, head_dim != 128) */
    EAGLE_ERR_CAPACITY = 3,     /* a buffer or workspace is too small          */
    EAGLE_ERR_CUDA = 4,         /* a CUDA launch / runtime call failed         */
    EAGLE_ERR_DEVICE_DATA = 5,  /* reserved for callers mapping dev_status     */
    EAGLE_ERR_TIMEOUT = 6       /* a bounded device wait expired               */
} eagle_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define EAGLE_DEV_BAD_TREE  0x01  /* parent[0] != -1 or parent[i] not in [0, i) */
#define EAGLE_DEV_BAD_TOKEN 0x02  /* token or draft row index out of range      */
#define EAGLE_DEV_NONFINITE 0x04  /* NaN / +inf logit, or an all -inf row        */
#define EAGLE_DEV_DEPTH     0x08  /* tree deeper than max_depth                  */
#define EAGLE_DEV_CAPACITY  0x10  /* kv_len[b] + n > Lmax                        */
#define EAGLE_DEV_TIMEOUT   0x20  /* a bounded pipeline wait gave up             */

typedef void* eagle_stream_t;

/* ---------------------------------------------------------------------------
 * eagle_tree_attn -- tree attention for one layer.
 * Lesson "KV cache 回滚" (the verifier attends with a non-causal mask that
 * follows the tree; one flash-attention call with a custom mask) and Guide
 * "EAGLE-2" (tree attention lets all tree tokens go through one forward).
 * For sequence b, node i, query head h (kv head h / (Hq/Hkv)):
 *   keys   = committed rows 0 .. L_b-1  plus tree rows L_b + j for every j that
 *            is i or an ancestor of i (L_b = kv_len[b]);
 *   out    = softmax(scale * q . k) . v, fp32 accumulation, bf16 result.
 *   q        bf16 [B, n, Hq, head_dim]
 *   k_cache  bf16 [B, Hkv, Lmax, head_dim]  (tree K already written at rows L_b + j)
 *   v_cache  bf16 [B, Hkv, Lmax, head_dim]
 *   kv_len   int32 [B]      parent int32 [B, n]  (parent[0] = -1, parent[i] < i)
 *   out      bf16 [B, n, Hq, head_dim]
 *   workspace / ws_bytes: device scratch of at least
 *            eagle_tree_attn_workspace_size(B, n, Hq, Hkv, head_dim, Lmax) bytes
 *            (may be NULL when that size is 0); contents need no initialisation.
 * Device errors: an invalid tree or kv_len[b] + n > Lmax sets a dev_status bit
 * and writes zeros for that sequence.
 * ------------------------------------------------------------------------- */
size_t eagle_tree_attn_workspace_size(int B, int n, int Hq, int Hkv, int head_dim, int Lmax);
eagle_status eagle_tree_attn(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* kv_len, const int32_t* parent, void* out,
                             int B, int n, int Hq, int Hkv, int head_dim, int Lmax, float scale,
                             void* workspace, size_t ws_bytes, int32_t* dev_status,
                             eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle_verify_accept -- the Leviathan walk over the draft tree.
 * Lesson "不变量" and steps 1-3; Guide "无损性的来源" and "EAGLE-2" (a node is
 * accepted only if all its prefixes are).  q = softmax(target/T), p =
 * softmax(draft/T).  From the root, the children of the current node v are
 * tried in increasing index; child c with token x is accepted iff p(x) <= 0
 * or u_c < q_cur(x) / p(x), u_c = Philox(seed; 0, c, b, 0) word 0 >> 8 times
 * 2^-24.  A rejected child replaces q_cur by norm(max(0, q_cur - p)) (kept if
 * that sums to 0).  An accepted child becomes v with q_cur = q(child).  When
 * no child is accepted, the final token is drawn from q_cur (residual, or the
 * bonus token from q(v)) by the exponential race argmax_t q_cur(t) / E_t,
 * E_t = -ln u'_t, u'_t = (2 (w >> 9) + 1) 2^-24 with w = word (t & 3) of
 * Philox(seed; t >> 2, 0, b, 1).  At temperature 0 a child is accepted iff
 * its token is the argmax of target row v (lowest index on ties) and the
 * final token is that argmax.
 *   target_logits f32 [B, n, V]  row i: target logits after node i.  Device
 *                 memory, or page-locked host memory the GPU addresses directly
 *                 (unified addressing): the walk then reads in place only the
 *                 rows it visits.
 *   draft_logits  f32 [B, R, V]  draft logits rows (only rows of nodes with
 *                 children are read; unused at T = 0, may then be NULL)
 *   draft_row     int32 [B, n] or NULL: row of draft_logits holding the draft
 *                 distribution after node i (NULL: row i, and R must equal n)
 *   tokens        int32 [B, n]  token of node i (node 0 ignored)
 *   parent        int32 [B, n]
 *   max_depth     D: the tree depth bound; sizes path and emit
 *   temperature   T >= 0      seed: Philox key (low word, high word)
 *   accept_len    int32 [B]       accepted drafts (root excluded), -1 on error
 *   path          int32 [B, D+1]  node ids of the accepted path, root first, -1 padded
 *   emit          int32 [B, D+1]  accepted draft tokens then the final token, -1 padded
 *   row_stats     f32 [2, B, n, 2] or NULL: (max z, sum exp(z - max)) of the
 *                 target (slot 0) and draft (slot 1) rows the walk visited;
 *                 rows it did not visit are left untouched.
 * No workspace.  Device errors: invalid tree / token / draft row, non-finite
 * rows -> accept_len[b] = -1, path/emit = -1, dev_status bit.
 * ------------------------------------------------------------------------- */
eagle_status eagle_verify_accept(const float* target_logits, const float* draft_logits,
                                 const int32_t* draft_row, const int32_t* tokens,
                                 const int32_t* parent, int B, int n, int V, int R,
                                 int max_depth, float temperature, uint64_t seed,
                                 int32_t* accept_len, int32_t* path, int32_t* emit,
                                 float* row_stats, int32_t* dev_status, eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle_verify_accept_sharded -- eagle_verify_accept with every logits row split
 * by vocabulary across S ranks, as a vocabulary-parallel LM head leaves it
 * (Lesson "不变量：Leviathan 拒绝采样": the rule the split walk must keep; Guide
 * "EAGLE-3：取消特征约束...": the draft head's own lm_head, which a tensor-parallel
 * deployment splits by vocabulary).  Rank r holds ids shard_begin[r] ..
 * shard_begin[r+1]-1 of every row in its own buffers and reads nothing else; the
 * ranks exchange only at four points: the row statistics (max, then the rescaled
 * sum, in rank order), the drafted token's q(x) and p(x) (from the rank owning x),
 * each rejection's residual normaliser (a sum in rank order) and the final
 * token's race winner (largest key, lower token on ties).  On one GPU each rank is
 * one CTA of the sequence's thread-block cluster and the exchanges go through its
 * distributed shared memory.  Results are those of eagle_verify_accept on the
 * whole rows (same uniforms, same rule), up to float summation order.
 *   target_shards  HOST array of S device pointers; shard r is f32 [B, n, Vr],
 *                  Vr = shard_begin[r+1] - shard_begin[r]
 *   draft_shards   HOST array of S device pointers, shard r f32 [B, R, Vr]; may
 *                  be NULL at T = 0
 *   shard_begin    HOST int32 [S + 1]: 0 = shard_begin[0] < ... < shard_begin[S] = V
 *   S              1 .. 8
 * Other arguments, outputs and device errors as eagle_verify_accept.  Host
 * errors: EAGLE_ERR_SHAPE for S > 8, an empty shard or bounds not 0 .. V.
 * ------------------------------------------------------------------------- */
eagle_status eagle_verify_accept_sharded(const float* const* target_shards,
                                         const float* const* draft_shards,
                                         const int32_t* shard_begin, int S,
                                         const int32_t* draft_row, const int32_t* tokens,
                                         const int32_t* parent, int B, int n, int V, int R,
                                         int max_depth, float temperature, uint64_t seed,
                                         int32_t* accept_len, int32_t* path, int32_t* emit,
                                         float* row_stats, int32_t* dev_status,
                                         eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle_verify_accept_filtered -- eagle_verify_accept with top-k / top-p
 * filtering.  Guide "一次 eagenerate 调用的完整流转": eagenerate takes
 * temperature, top_p and top_k (0 = off); the pages give no further rule.
 * Reading: at T > 0, each row's tokens are ranked by probability (logit desc,
 * lower token first on ties); top-k keeps the first top_k; top-p then keeps the
 * shortest prefix of that order whose probability, renormalised over what top-k
 * kept, reaches top_p (at least one token).  q and p are each filtered this way
 * and renormalised, and the walk, uniforms and outputs are those of
 * eagle_verify_accept on the filtered distributions (row_stats then hold the
 * filtered sums).  top_k = 0 or >= V and top_p = 0 or >= 1 switch a filter off;
 * at T = 0 (greedy) both are ignored.
 *   workspace  device, >= eagle_verify_filter_workspace_size(B, n, R) bytes,
 *              16-byte aligned; needed only when a filter is on (one 32-byte
 *              filter per target and draft row, written when the walk visits it).
 * Errors: EAGLE_ERR_INVALID_ARG for top_k < 0 or top_p < 0 / not finite;
 * EAGLE_ERR_CAPACITY for a missing or small workspace; EAGLE_ERR_SHAPE for
 * V > 4194304.  The filter decisions use the probability mass in 2^-40 fixed
 * point, so a top-p cut within ~1e-7 of top_p may fall one token apart from an
 * exact computation.
 * ------------------------------------------------------------------------- */
size_t eagle_verify_filter_workspace_size(int B, int n, int R);
eagle_status eagle_verify_accept_filtered(const float* target_logits, const float* draft_logits,
                                          const int32_t* draft_row, const int32_t* tokens,
                                          const int32_t* parent, int B, int n, int V, int R,
                                          int max_depth, float temperature, uint64_t seed,
                                          int top_k, float top_p, int32_t* accept_len,
                                          int32_t* path, int32_t* emit, float* row_stats,
                                          void* workspace, size_t ws_bytes, int32_t* dev_status,
                                          eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * Draft vocabulary (EAGLE-3).  Guide "EAGLE-3：取消特征约束…": the draft head may
 * have its own LM head over a smaller vocabulary of Vd ids, and a table d2t
 * (int32 [Vd]) returns each draft id d to the target id d + d2t[d].
 *
 * eagle_d2t_inverse -- t2d[t] = d for t = d + d2t[d], -1 for every target id no
 * draft id maps to.
 *   d2t int32 [Vd] (device, read); t2d int32 [V] (device, written; caller-owned).
 * A draft id mapped outside [0, V), or onto a target id that another draft id
 * also maps to, sets EAGLE_DEV_BAD_TOKEN and is left out of t2d.
 *
 * eagle_verify_accept_d2t -- eagle_verify_accept when the draft rows are over
 * the draft vocabulary: draft_logits f32 [B, R, Vd]; t2d int32 [V] from
 * eagle_d2t_inverse; tokens are target ids.  p over the target vocabulary is
 * softmax(draft row / T) at the ids d + d2t[d] and 0 at every other target id,
 * so a target id p never proposes keeps its full q in every residual.  The
 * walk, the uniforms, row_stats (the draft slot then over the Vd draft ids) and
 * the errors are those of eagle_verify_accept.  Vd % 4 == 0 and 16-byte aligned
 * rows take the vector path; other sizes are correct, slower.
 * ------------------------------------------------------------------------- */
eagle_status eagle_d2t_inverse(const int32_t* d2t, int Vd, int V, int32_t* t2d,
                               int32_t* dev_status, eagle_stream_t stream);
eagle_status eagle_verify_accept_d2t(const float* target_logits, const float* draft_logits,
                                     const int32_t* draft_row, const int32_t* tokens,
                                     const int32_t* parent, int B, int n, int V, int R, int Vd,
                                     const int32_t* t2d, int max_depth, float temperature,
                                     uint64_t seed, int32_t* accept_len, int32_t* path,
                                     int32_t* emit, float* row_stats, int32_t* dev_status,
                                     eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle_kv_compact -- commit the accepted path into the KV cache.
 * Lesson "KV cache 回滚" and "第 4 步" (one physical cache plus a logical
 * length).  For t = 0 .. a (a = accept_len[b]): row L_b + path[b][t] moves to
 * row L_b + t in every layer and kv head, for K and V (all source rows are read
 * before any is written); then kv_len[b] = L_b + a + 1.
 *   k_cache, v_cache bf16 [n_layers, B, Hkv, Lmax, head_dim], in place
 *   kv_len int32 [B] (read and updated)   path int32 [B, D+1]   accept_len int32 [B]
 * Sequences with accept_len < 0 are skipped.  L_b + path[a] >= Lmax or a > D
 * sets EAGLE_DEV_CAPACITY and skips the sequence.
 * ------------------------------------------------------------------------- */
eagle_status eagle_kv_compact(void* k_cache, void* v_cache, int32_t* kv_len, const int32_t* path,
                              const int32_t* accept_len, int n_layers, int B, int Hkv,
                              int head_dim, int Lmax, int max_depth, int32_t* dev_status,
                              eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle_ttt_attn -- training-time-test attention for one layer and one round.
 * TTT page, section "训练时的 attention mask 为什么要特殊处理": round 0 runs on
 * the original tokens with the causal mask; in round r >= 1 position i holds the
 * token the previous round predicted there, and it may see only its ancestors.
 * For sequence b, position i, query head h (kv head h / (Hq/Hkv)), queries of
 * round r:
 *   keys  = round-0 rows 0 .. i (the original tokens up to i) plus the rows of
 *           rounds 1 .. r at position i (its own chain, itself included);
 *   out   = softmax(scale * q . k) . v, fp32 accumulation, bf16 result.
 * Both parts run on the tensor cores: the diagonal part (at most R1 - 1 keys per
 * query) as a few more 128-key tiles, each holding up to 128 / (positions per row
 * tile) rounds of the tile's positions, with every key but a row's own masked (the
 * page suggests per-position dot products; the result is the same).
 *   q    bf16 [B, S, Hq, head_dim]        (the queries of round r)
 *   k, v bf16 [B, Hkv, R1, S, head_dim]   (round 0 = original tokens; rounds
 *        1 .. R1-1 simulated; only rounds 0 .. r are read)
 *   out  bf16 [B, S, Hq, head_dim]
 * Sizes: S >= 1, 1 <= R1 <= 16, 0 <= r < R1, head_dim == 128, Hq % Hkv == 0,
 * B * Hkv * ceil(S * Hq / Hkv / 128) < 2^31.  Every row of rounds 0 .. r must be finite
 * (rows other than a query's own keys are read and masked; a zero weight does not
 * cancel NaN).  All pointers 16-byte aligned.
 * Device errors: a wait that exceeds its limit sets EAGLE_DEV_TIMEOUT.
 * ------------------------------------------------------------------------- */
eagle_status eagle_ttt_attn(const void* q, const void* k, const void* v, void* out, int B, int S,
                            int Hq, int Hkv, int head_dim, int R1, int r, float scale,
                            int32_t* dev_status, eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle2_expand -- one level of EAGLE-2 expansion; optionally the rerank.
 * Guide "EAGLE-2：草稿树的 Expansion 与 Reranking" and TTT "EAGLE-3 和 EAGLE-2
 * 动态树如何拼在一起": node value V_i = product of draft confidences on the
 * root path; each level runs the draft forward only on the top_k nodes of the
 * previous level with the largest V; the rerank keeps the global top-n by V.
 * Confidences c = softmax(draft logits) at temperature 1; each frontier row
 * contributes its top_k tokens (larger logit first, lower token on ties);
 * products are float32.  Level 1 expands the root row into top_k candidates;
 * level l >= 2 expands the top_k frontier rows into top_k^2 candidates and keeps
 * the top_k by V (lower candidate id on ties) as the next frontier.
 * Candidate ids: root 0; level 1: 1 + j; level l: 1 + k + (l-2)k^2 + s k + j.
 * Draft rows: root 0; frontier slot s chosen at level l < depth: 1 + (l-1)k + s.
 *   level         1 .. depth (call in order; level 1 initialises tree_state)
 *   final         non-zero: after this level, rerank and write the out_* arrays
 *   hidden        bf16 [B, k_in, H] or NULL (k_in = 1 at level 1, top_k after):
 *                 the draft model's output for the current frontier rows.  When
 *                 given, logits rows of this level are computed as hidden . W^T.
 *   lm_head_w     bf16 [V, H] (needed when hidden != NULL)
 *   logits        f32 [B, R, V], R = 1 + (depth-1) top_k: draft-logit storage.
 *                 This level's rows are written (hidden != NULL) or read.
 *   tree_state    scratch of eagle2_tree_state_size(B, top_k, depth) bytes that
 *                 persists across the levels of one tree
 *   partials      NULL: the level's top_k comes from one pass over its logits
 *                 rows.  Otherwise f32 [B * k_in, ceil(V / 256), 2],
 *                 eagle2_expand_scratch_size(B, V, top_k) bytes, 8-byte aligned:
 *                 per 256-column tile of each row (row b * k_in + s) its max and
 *                 sum of exponentials, as eagle_lmhead_gemm writes them; with
 *                 hidden != NULL this call's GEMM writes them, otherwise the
 *                 caller's eagle_lmhead_gemm(..., partials, ...) for this level's
 *                 rows must have.  The row's statistics then come from the
 *                 partials, and its top_k from rescanning only the tiles whose
 *                 maximum reaches the k-th largest tile maximum (every top_k
 *                 entry lies in one), instead of a pass over the whole row.
 *   out_tokens, out_parent, out_draft_row  int32 [B, n_out] (final only):
 *                 nodes in topological order (depth asc, V desc, id asc), root
 *                 first with token -1 and draft row 0; out_draft_row = -1 for
 *                 nodes that were never expanded.
 *   frontier_tokens int32 [B, top_k] or NULL: tokens of the new frontier.
 * Constraints: 1 <= top_k <= 16, top_k <= V, 2 <= n_out <= min(64, candidates+1),
 * depth <= 16.  Device errors: non-finite logit rows set EAGLE_DEV_NONFINITE.
 * ------------------------------------------------------------------------- */
size_t eagle2_tree_state_size(int B, int top_k, int depth);
size_t eagle2_expand_scratch_size(int B, int V, int top_k);
eagle_status eagle2_expand(int level, int final, const void* hidden, const void* lm_head_w,
                           float* logits, int B, int H, int V, int top_k, int depth, int n_out,
                           void* tree_state, size_t state_bytes, float* partials, size_t partials_bytes,
                           int32_t* out_tokens, int32_t* out_parent, int32_t* out_draft_row,
                           int32_t* frontier_tokens, int32_t* dev_status, eagle_stream_t stream);

/* eagle2_tree_candidates -- read back every candidate of a tree state.
 * Same page and section as eagle2_expand: each candidate's draft confidence c
 * (the temperature-1 softmax probability of its token in its parent's draft
 * row) and path value V = V(parent) * c (float32 product, root V = 1) are the
 * numbers the per-level and global selections rank.  For each sequence b and
 * candidate id i (numbered as in eagle2_expand, C = 1 + top_k + (depth-1)
 * top_k^2 ids, root 0) writes, at [b * C + i]:
 *   value f32, conf f32, token int32 (target id), parent int32 (candidate id,
 *   root -1), cand_depth int32 (level, root 0), draft_row int32 (row of the
 *   draft logits the candidate was expanded from as a frontier node, else -1).
 * Each output may be NULL.  Only ids generated by the levels run so far hold
 * data.  tree_state / state_bytes as given to eagle2_expand.  Enqueued on
 * stream after the expansion calls; nothing is modified. */
eagle_status eagle2_tree_candidates(const void* tree_state, size_t state_bytes, int B, int top_k,
                                    int depth, float* value, float* conf, int32_t* token,
                                    int32_t* parent, int32_t* cand_depth, int32_t* draft_row,
                                    eagle_stream_t stream);

/* eagle2_expand_d2t -- eagle2_expand with a draft vocabulary: V is the draft
 * vocabulary size (the LM head's rows and the logits' width), the ranking is
 * over draft ids (ties to the lower draft id), and each chosen draft id d enters
 * the tree -- tree state, out_tokens, frontier_tokens -- as the target id
 * d + d2t[d].  d2t int32 [V] (device) must not be NULL; the caller keeps the
 * mapped ids inside the target vocabulary (eagle_d2t_inverse checks a table). */
eagle_status eagle2_expand_d2t(int level, int final, const void* hidden, const void* lm_head_w,
                               float* logits, int B, int H, int V, int top_k, int depth, int n_out,
                               void* tree_state, size_t state_bytes, float* partials,
                               size_t partials_bytes, const int32_t* d2t, int32_t* out_tokens,
                               int32_t* out_parent, int32_t* out_draft_row,
                               int32_t* frontier_tokens, int32_t* dev_status, eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * Static draft trees (EAGLE-1 / Medusa style).  Guide "EAGLE-2：草稿树的 Expansion
 * 与 Reranking": the static trees EAGLE-2 replaces add a fixed number of
 * candidates per step, whatever the context.  A static tree is a list of
 * choices, each a path of child ranks (r_1, ..., r_d) from the root: the node it
 * names takes the r_d-th best token (logit desc, lower token on ties) of its
 * parent's draft row.  The tree then feeds eagle_tree_attn and
 * eagle_verify_accept through its parent and draft_row arrays, like an EAGLE-2
 * tree.
 *
 * eagle_static_tree -- HOST planner (host pointers, no GPU work, no allocation
 * visible to the caller).  ranks int32 [n_choices, max_len] row-major, choice c
 * being ranks[c][0 .. lens[c]-1]; lens int32 [n_choices].  Writes n = n_choices
 * + 1 nodes: the root, then the choices sorted by (length, lexicographic), into
 * parent, rank (root: -1), depth and draft_row (internal nodes numbered 0, 1, ...
 * in node order; leaves -1), each int32 [n_max]; *n_nodes = n.
 * Errors: EAGLE_ERR_CAPACITY when n > n_max or n > 64; EAGLE_ERR_SHAPE for an
 * empty or too long choice, a rank outside [0, 16), a duplicate, or a choice
 * whose parent path is not itself a choice.
 *
 * eagle_static_tree_level -- one level's tokens on the GPU: for every node c at
 * depth `level`, tokens[b][c] = the rank[c]-th best token of row draft_row[parent
 * [c]] of logits f32 [B, R, V] (the draft rows of the internal nodes).  parent,
 * rank, depth, draft_row: int32 [n], device.  Other entries of tokens are left
 * as they are (the root's is the caller's).  A non-finite row sets
 * EAGLE_DEV_NONFINITE; a draft row >= R sets EAGLE_DEV_BAD_TREE.
 * ------------------------------------------------------------------------- */
eagle_status eagle_static_tree(const int32_t* ranks, const int32_t* lens, int n_choices, int max_len,
                               int n_max, int32_t* parent, int32_t* rank, int32_t* depth,
                               int32_t* draft_row, int32_t* n_nodes);
eagle_status eagle_static_tree_level(int level, const float* logits, const int32_t* parent,
                                     const int32_t* rank, const int32_t* depth,
                                     const int32_t* draft_row, int n, int B, int R, int V,
                                     int32_t* tokens, int32_t* dev_status, eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle2_expand_static_state -- eagle2_expand without caller-provided scratch.
 * No counterpart in the paper: this is a deployment convenience of this library.
 * It is for callers that cannot allocate device memory themselves: a serving
 * loop that reserves all of its device memory once at start-up and may not
 * allocate afterwards (cudaMalloc can synchronise the device and stall other
 * work), or code that sits behind an allocator owned by another framework and
 * has no way to obtain raw device memory of its own.
 * The tree state lives in a file-scope device array of 4 MiB that the library
 * holds on every device that loads it, until the process exits.  Arguments,
 * outputs and errors are those of eagle2_expand, minus tree_state/state_bytes
 * and partials/partials_bytes (none: the top-k reads the logits rows).
 *   - Returns EAGLE_ERR_CAPACITY, launching nothing, when
 *     eagle2_tree_state_size(B, top_k, depth) exceeds 4 MiB (for top_k = 10,
 *     depth = 8 that is 20,824 bytes per sequence: up to 201 sequences).
 *     Other invalid arguments return the status eagle2_expand gives them.
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream
 *     capture.  After cudaDeviceReset on a device the cached address is stale:
 *     do not call this entry point on that device again in the same process.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents: the levels of one tree must run in order, and calls that overlap
 *     on the GPU (other streams, other host threads, another tree in between)
 *     race.  Level 1 rewrites everything later levels read, so nothing needs
 *     clearing between trees.
 *   - Allocates nothing: no cudaMalloc / cudaFree, no allocating library call.
 * ------------------------------------------------------------------------- */
eagle_status eagle2_expand_static_state(int level, int final, const void* hidden,
                                        const void* lm_head_w, float* logits, int B, int H, int V,
                                        int top_k, int depth, int n_out, int32_t* out_tokens,
                                        int32_t* out_parent, int32_t* out_draft_row,
                                        int32_t* frontier_tokens, int32_t* dev_status,
                                        eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle_softmax_stats -- per-row temperature softmax statistics.
 * z = logits / T; row_max = max z; row_sum = sum exp(z - row_max) (T > 0).
 * At T = 0 only row_argmax is written (lowest index on ties).
 *   logits f32 [rows, V]; row_max, row_sum f32 [rows] (may be NULL at T = 0);
 *   row_argmax int32 [rows] or NULL.
 * Non-finite rows set EAGLE_DEV_NONFINITE.
 * ------------------------------------------------------------------------- */
eagle_status eagle_softmax_stats(const float* logits, int64_t rows, int V, float temperature,
                                 float* row_max, float* row_sum, int32_t* row_argmax,
                                 int32_t* dev_status, eagle_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle_lmhead_gemm -- the draft LM head, logits = hidden . W^T.
 * Guide "EAGLE-3" code changes: the draft head's own lm_head = Linear(hidden,
 * draft_vocab, bias=False).  bf16 inputs, fp32 accumulation and output, on the
 * tcgen05 tensor cores.
 *   hidden bf16 [M, K]   w bf16 [N, K]   (K % 64 == 0, 16-byte aligned bases)
 *   out    f32: row m of the product is stored at
 *          out + ((m / rows_per_group) * group_stride + row_offset + m % rows_per_group) * ldo
 *          (rows_per_group = M, group_stride = 0, row_offset = 0: a plain [M, ldo] matrix)
 *   partials NULL, or f32 [M, ceil(N / 256), 2] (8-byte aligned): for each row
 *          and 256-column tile, max l and sum 2^((l - max) log2 e) over the tile's
 *          columns -- the temperature-1 softmax statistics of the row, tile by
 *          tile, as eagle2_expand consumes them.
 * ------------------------------------------------------------------------- */
eagle_status eagle_lmhead_gemm(const void* hidden, const void* w, float* out, int M, int K, int N,
                               int64_t ldo, int rows_per_group, int64_t group_stride,
                               int64_t row_offset, float* partials, int32_t* dev_status,
                               eagle_stream_t stream);

/* Human-readable name of a status code (static string). */
/* ---------------------------------------------------------------------------
 * eagle_wait_selftest -- exercises the bounded-wait path of the pipelined
 * kernels.  No counterpart in the paper.  One thread waits on an mbarrier that
 * nothing completes, polling it exactly as the pipelines do, for at most
 * max_cycles SM clock cycles (1 .. 4e9), then ORs EAGLE_DEV_TIMEOUT into
 * *dev_status (required, device memory) and returns.  Lets a caller (or a test)
 * check that an expired wait reports a status and leaves the context usable.
 * ------------------------------------------------------------------------- */
eagle_status eagle_wait_selftest(int32_t* dev_status, int64_t max_cycles, eagle_stream_t stream);

const char* eagle_status_str(eagle_status s);

/* Library ABI version (major * 100 + minor). */
int eagle_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE_GB300_H */
