/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the EAGLE
 * draft-tree verify-and-accept path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library; the two are written independently from the method
 * description.
 *
 * Pages cited (by title and section):
 *   [Lesson]  "推测解码与 EAGLE-3" (aibook lesson), sections
 *             "不变量：Leviathan 拒绝采样", "什么决定加速", "KV cache 回滚",
 *             "动手构建" steps 1-5, "练习", "关键术语".
 *   [Guide]   "EAGLE-1/2/3 拆解：推测解码省的是大模型前向次数，赚不赚看草稿准确率"
 *             (txtmix.com), sections "无损性的来源与它的证明位置",
 *             "EAGLE-2：草稿树的 Expansion 与 Reranking",
 *             "一次 eagenerate 调用的完整流转", "采用顺序".
 *   [TTT]     "EAGLE-3 完全拆解：Training-Time Test 如何解除特征预测的天花板"
 *             (pinghaoyang.com.cn), section "EAGLE-3 和 EAGLE-2 动态树如何拼在一起".
 *
 * Precision: every floating-point quantity is carried in double.  Inputs
 * arrive as float32 logits or bfloat16 bit patterns and are widened exactly.
 *
 * Notation (Lesson, "不变量"): q = target (verifier) distribution,
 * p = draft distribution.  The Guide's "无损性" section uses the opposite
 * letters for the same rule.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD_TREE 1
#define ORC_BAD_TOKEN 2
#define ORC_NONFINITE 4
#define ORC_DEPTH 8
#define ORC_CAPACITY 16

/* ------------------------------------------------------------------------
 * Philox4x32-10, written from Salmon, Moraes, Dror and Shaw, "Parallel
 * Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4.2 (the Philox
 * S-box: two 32x32->64 multiplications per round, the high halves XORed
 * with the other two words and the round key, the low halves carried, the
 * words permuted) and the Weyl key schedule of the same section.
 * The method draws its uniforms from this counter-based generator
 * (accept test: Lesson "第 1 步"; residual/bonus sampling: Lesson "第 3 步").
 * ---------------------------------------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint64_t MA = 0xD2511F53u, MB = 0xCD9E8D57u;   /* round multipliers */
    const uint32_t WA = 0x9E3779B9u, WB = 0xBB67AE85u;   /* Weyl increments   */
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t pa = MA * (uint64_t)x0;
        uint64_t pb = MB * (uint64_t)x2;
        uint32_t hia = (uint32_t)(pa >> 32), loa = (uint32_t)pa;
        uint32_t hib = (uint32_t)(pb >> 32), lob = (uint32_t)pb;
        uint32_t y0 = hib ^ x1 ^ k0;
        uint32_t y1 = lob;
        uint32_t y2 = hia ^ x3 ^ k1;
        uint32_t y3 = loa;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += WA; k1 += WB;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Counter layout: (c0, c1, c2, c3) = (lane block, node or position, sequence, tag). */
#define TAG_ACCEPT 0u
#define TAG_RACE   1u
#define TAG_DRAFT  2u

static uint32_t philox_word(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2,
                            uint32_t tag, int lane)
{
    uint32_t ctr[4] = {c0, c1, c2, tag};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return out[lane];
}

/* Accept-test uniform in [0,1): top 24 bits of word 0, times 2^-24. */
double orc_u_accept(uint64_t seed, uint32_t b, uint32_t node)
{
    uint32_t w = philox_word(seed, 0u, node, b, TAG_ACCEPT, 0);
    return (double)(w >> 8) * (1.0 / 16777216.0);
}

/* Sampling uniform in (0,1): odd multiples of 2^-24, from word (t & 3) of
 * counter block t >> 2.  Used by the exponential race. */
double orc_u_race(uint64_t seed, uint32_t b, uint32_t c1, uint32_t t, uint32_t tag)
{
    uint32_t w = philox_word(seed, t >> 2, c1, b, tag, (int)(t & 3u));
    return (double)(2u * (w >> 9) + 1u) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------
 * Sampling from an unnormalised non-negative weight vector r by the
 * exponential race: y = argmax_t r_t / E_t with E_t = -ln u'_t, u'_t in
 * (0,1).  P(y = t) = r_t / sum(r) exactly (the minimum of independent
 * exponentials with rates r_t is attained at t with probability
 * r_t / sum r).  Zero weights are never chosen; ties go to the lower t.
 * Returns y, and the best and runner-up keys for near-tie accounting.
 * ---------------------------------------------------------------------- */
static int race_sample(const double* r, int V, uint64_t seed, uint32_t b, uint32_t c1,
                       uint32_t tag, double* key1, int* y2, double* key2)
{
    int best = -1, second = -1;
    double kb = -1.0, ks = -1.0;
    for (int t = 0; t < V; ++t) {
        if (!(r[t] > 0.0)) continue;
        double e = -log(orc_u_race(seed, b, c1, (uint32_t)t, tag));
        double key = r[t] / e;
        if (key > kb) { second = best; ks = kb; best = t; kb = key; }
        else if (key > ks) { second = t; ks = key; }
    }
    if (key1) *key1 = kb;
    if (y2) *y2 = second;
    if (key2) *key2 = ks;
    return best;
}

int orc_race_sample(const double* r, int V, uint64_t seed, uint32_t b, uint32_t c1, uint32_t tag)
{
    return race_sample(r, V, seed, b, c1, tag, NULL, NULL, NULL);
}

/* ------------------------------------------------------------------------
 * Tree bookkeeping.  The tree is a parent array: node 0 is the root (the
 * last emitted token, Guide "EAGLE-2" expansion stage, layer 0 = end of
 * the accepted sequence), parent[0] = -1, 0 <= parent[i] < i.  A node may
 * attend to itself and its ancestors only (Guide "EAGLE-2" on tree
 * attention; TTT page on the tree-shaped mask; Lesson "KV cache 回滚" on
 * the non-causal tree mask).  anc[i] has bit j set iff j is i or an
 * ancestor of i.
 * ---------------------------------------------------------------------- */
int orc_tree_check(const int32_t* parent, int n, uint64_t* anc, int32_t* depth)
{
    if (n < 1 || n > 64) return ORC_BAD_TREE;
    if (parent[0] != -1) return ORC_BAD_TREE;
    anc[0] = 1ull;
    depth[0] = 0;
    for (int i = 1; i < n; ++i) {
        int pa = parent[i];
        if (pa < 0 || pa >= i) return ORC_BAD_TREE;
        anc[i] = anc[pa] | (1ull << i);
        depth[i] = depth[pa] + 1;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Temperature softmax statistics of one row (Guide "一次 eagenerate 调用"
 * names the temperature argument; the plain reading is softmax(logits / T)).
 * z = l / T, m = max z, Z = sum exp(z - m), prob(t) = exp(z_t - m) / Z.
 * At T = 0 (greedy decoding) only the argmax is defined (lowest index wins
 * ties), returned through amax.
 * ---------------------------------------------------------------------- */
static int row_stats(const float* row, int V, double T, double* m_out, double* Z_out, int* amax)
{
    int arg = 0;
    double best = (double)row[0];
    for (int t = 1; t < V; ++t)
        if ((double)row[t] > best) { best = (double)row[t]; arg = t; }
    if (amax) *amax = arg;
    for (int t = 0; t < V; ++t)
        if (isnan(row[t]) || (isinf(row[t]) && row[t] > 0)) return ORC_NONFINITE;
    if (isinf(best)) return ORC_NONFINITE;          /* all -inf: no distribution */
    if (T > 0.0) {
        double m = best / T, Z = 0.0;
        for (int t = 0; t < V; ++t) Z += exp((double)row[t] / T - m);
        *m_out = m;
        *Z_out = Z;
    } else {
        *m_out = best;
        *Z_out = 1.0;
    }
    return ORC_OK;
}

void orc_softmax_rows(const float* logits, int64_t rows, int V, double T,
                      double* m, double* Z, int32_t* amax, int32_t* status)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int a = -1;
        double mm = NAN, zz = NAN;
        int st = row_stats(logits + r * (int64_t)V, V, T, &mm, &zz, &a);
        m[r] = mm; Z[r] = zz;
        if (amax) amax[r] = a;
        if (status) status[r] = st;
    }
}

/* Full probability vector of a row at temperature T > 0. */
static void row_probs(const float* row, int V, double T, double m, double Z, double* out)
{
    for (int t = 0; t < V; ++t) out[t] = exp((double)row[t] / T - m) / Z;
}

/* ------------------------------------------------------------------------
 * Verify-and-accept walk over one draft tree (per sequence).
 *
 * Chain rule (Lesson "不变量" and "第 3 步"): draft token x ~ p is accepted
 * with probability min(1, q(x)/p(x)); the first rejection stops the walk
 * and the final token is drawn from the residual norm(max(0, q - p));
 * if every draft is accepted a bonus token is drawn from the next target
 * distribution.  The accept test itself follows Lesson "第 1 步": accept
 * when p(x) <= 0, else accept iff u < q(x)/p(x).  The residual follows
 * Lesson "第 2 步": clamp at zero, normalise, and fall back to q when the
 * clamped vector sums to zero.
 *
 * Tree form (Guide "EAGLE-2": a token is accepted only if all its prefixes
 * are; the target runs once over the whole tree): starting at the root v,
 * the children of v are tried in increasing node index.  Each rejected
 * child replaces the current target distribution q_cur by the residual
 * norm(max(0, q_cur - p(v))), p(v) unchanged, before the next sibling is
 * tried.  The first accepted child c becomes the new v with q_cur = q(c).
 * When no child of v is accepted (or v is a leaf) the final token is drawn
 * from q_cur: the residual after the rejected siblings, or q(v) itself,
 * which is the bonus token.  At T = 0 (greedy) a child is accepted iff
 * its token equals argmax of the target row of v (lowest index on ties;
 * the first such child in index order), and the final token is that argmax.
 *
 * Inputs:
 *   target  f32 [B, n, V]  row i = target logits after node i
 *   draft   f32 [B, R, V]  draft logits rows; row draft_row[b,i] holds the
 *                          draft distribution after node i (only needed for
 *                          nodes with children).  draft_row NULL: row i, R = n.
 *   tokens  i32 [B, n]     token of node i (node 0 unused)
 *   parent  i32 [B, n]
 *   u_override f64 [B, n] or NULL: accept uniform for node i (tests force
 *                          outcomes with it); NULL draws Philox(seed, b, i).
 * Outputs:
 *   accept_len i32 [B]     accepted draft tokens (root excluded); -1 on error
 *   path  i32 [B, D+1]     node ids, root first, -1 padded
 *   emit  i32 [B, D+1]     accepted draft tokens then the final token
 *   trace f64 [B, n, 4]    per tested node: (u, p(x), q_cur(x), 1 accept / 2 reject)
 *   race  f64 [B, 4]       (y, best key, runner-up token, runner-up key)
 *   status i32 [B]         ORC_* flags
 * ---------------------------------------------------------------------- */
static void walk_one(const float* target, const float* draft, const int32_t* draft_row,
                     const int32_t* tokens, const int32_t* parent, int b, int n, int V, int R,
                     int D, double T, uint64_t seed, const double* u_override,
                     int32_t* accept_len, int32_t* path, int32_t* emit, double* trace,
                     double* race, int32_t* status)
{
    const int64_t Vn = V;
    const float* tgt = target + (int64_t)b * n * Vn;
    const float* drf = draft + (int64_t)b * R * Vn;
    const int32_t* tok = tokens + (int64_t)b * n;
    const int32_t* par = parent + (int64_t)b * n;
    const int32_t* drow = draft_row ? draft_row + (int64_t)b * n : NULL;
    int32_t* P = path + (int64_t)b * (D + 1);
    int32_t* E = emit + (int64_t)b * (D + 1);
    for (int i = 0; i <= D; ++i) { P[i] = -1; E[i] = -1; }
    accept_len[b] = -1;
    status[b] = ORC_OK;
    if (trace) for (int i = 0; i < 4 * n; ++i) trace[(int64_t)b * n * 4 + i] = 0.0;
    if (race) for (int i = 0; i < 4; ++i) race[b * 4 + i] = -1.0;

    uint64_t anc[64];
    int32_t depth[64];
    if (orc_tree_check(par, n, anc, depth) != ORC_OK) { status[b] = ORC_BAD_TREE; return; }
    int has_child[64] = {0};
    for (int i = 1; i < n; ++i) {
        if (tok[i] < 0 || tok[i] >= V) { status[b] = ORC_BAD_TOKEN; return; }
        if (depth[i] > D) { status[b] = ORC_DEPTH; return; }
        has_child[par[i]] = 1;
    }
    for (int i = 0; i < n; ++i) {
        int row = drow ? drow[i] : i;
        if (has_child[i] && T > 0.0 && (row < 0 || row >= R)) { status[b] = ORC_BAD_TREE; return; }
    }

    double* q = (double*)malloc(sizeof(double) * V);
    double* p = (double*)malloc(sizeof(double) * V);
    int v = 0, a = 0;
    P[0] = 0;
    for (;;) {
        const float* qrow = tgt + (int64_t)v * Vn;
        int y;
        if (T > 0.0) {
            double mq, Zq;
            if (row_stats(qrow, V, T, &mq, &Zq, NULL) != ORC_OK) { status[b] = ORC_NONFINITE; goto done; }
            row_probs(qrow, V, T, mq, Zq, q);              /* q_cur = q(v) */
            int moved = 0;
            if (has_child[v]) {
                const float* prow = drf + (int64_t)(drow ? drow[v] : v) * Vn;
                double mp, Zp;
                if (row_stats(prow, V, T, &mp, &Zp, NULL) != ORC_OK) { status[b] = ORC_NONFINITE; goto done; }
                row_probs(prow, V, T, mp, Zp, p);
                for (int c = v + 1; c < n; ++c) {
                    if (par[c] != v) continue;
                    int x = tok[c];
                    double u = u_override ? u_override[(int64_t)b * n + c]
                                          : orc_u_accept(seed, (uint32_t)b, (uint32_t)c);
                    int acc = (p[x] <= 0.0) ? 1 : (u < q[x] / p[x]);
                    if (trace) {
                        double* tr = trace + ((int64_t)b * n + c) * 4;
                        tr[0] = u; tr[1] = p[x]; tr[2] = q[x]; tr[3] = acc ? 1.0 : 2.0;
                    }
                    if (acc) {
                        ++a;
                        P[a] = c;
                        E[a - 1] = x;
                        v = c;
                        moved = 1;
                        break;
                    }
                    /* rejected: q_cur <- norm(max(0, q_cur - p)), or unchanged if that sums to 0 */
                    double s = 0.0;
                    for (int t = 0; t < V; ++t) s += fmax(0.0, q[t] - p[t]);
                    if (s > 0.0)
                        for (int t = 0; t < V; ++t) q[t] = fmax(0.0, q[t] - p[t]) / s;
                }
            }
            if (moved) continue;
            double k1, k2;
            int y2;
            y = race_sample(q, V, seed, (uint32_t)b, 0u, TAG_RACE, &k1, &y2, &k2);
            if (race) { race[b*4+0] = y; race[b*4+1] = k1; race[b*4+2] = y2; race[b*4+3] = k2; }
        } else {
            int g;
            double mq, Zq;
            if (row_stats(qrow, V, 0.0, &mq, &Zq, &g) != ORC_OK) { status[b] = ORC_NONFINITE; goto done; }
            int moved = 0;
            for (int c = v + 1; c < n; ++c) {
                if (par[c] != v) continue;
                if (tok[c] == g) {
                    if (trace) {
                        double* tr = trace + ((int64_t)b * n + c) * 4;
                        tr[3] = 1.0;
                    }
                    ++a;
                    P[a] = c;
                    E[a - 1] = tok[c];
                    v = c;
                    moved = 1;
                    break;
                }
                if (trace) trace[((int64_t)b * n + c) * 4 + 3] = 2.0;
            }
            if (moved) continue;
            y = g;
        }
        E[a] = y;
        accept_len[b] = a;
        break;
    }
done:
    if (status[b] != ORC_OK) {
        accept_len[b] = -1;
        for (int i = 0; i <= D; ++i) { P[i] = -1; E[i] = -1; }
    }
    free(q);
    free(p);
}

void orc_verify_accept(const float* target, const float* draft, const int32_t* draft_row,
                       const int32_t* tokens, const int32_t* parent, int B, int n, int V, int R,
                       int max_depth, double T, uint64_t seed, const double* u_override,
                       int32_t* accept_len, int32_t* path, int32_t* emit, double* trace,
                       double* race, int32_t* status)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        walk_one(target, draft, draft_row, tokens, parent, b, n, V, R, max_depth, T, seed,
                 u_override, accept_len, path, emit, trace, race, status);
}

/* Draw one token per row from softmax(row / T) with the exponential race
 * (tag DRAFT, c1 = row index within the sequence); T = 0 takes the argmax.
 * Test helper: it stands in for the draft model proposing a chain
 * (Lesson "第 3 步": "d ~ p"). */
void orc_sample_rows(const float* logits, int B, int rows, int V, double T, uint64_t seed,
                     int32_t* out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double* pr = (double*)malloc(sizeof(double) * V);
        for (int j = 0; j < rows; ++j) {
            const float* row = logits + ((int64_t)b * rows + j) * V;
            double m, Z;
            int g;
            if (row_stats(row, V, T, &m, &Z, &g) != ORC_OK) { out[b * rows + j] = -1; continue; }
            if (T > 0.0) {
                row_probs(row, V, T, m, Z, pr);
                out[b * rows + j] = race_sample(pr, V, seed, (uint32_t)b, (uint32_t)j, TAG_DRAFT,
                                                NULL, NULL, NULL);
            } else {
                out[b * rows + j] = g;
            }
        }
        free(pr);
    }
}

/* ------------------------------------------------------------------------
 * Tree attention (Lesson "KV cache 回滚": the verifier runs attention with
 * a non-causal mask that respects the tree; Guide "EAGLE-2": all tree
 * tokens in one forward thanks to tree attention).  For node i, query head
 * h, kv head h / (Hq / Hkv): keys are the committed rows 0..L_b-1 plus the
 * tree rows L_b + j for every j that is i or an ancestor of i.  Plain
 * softmax(scale * q.k) . v, all in double.
 *   q bf16 [B, n, Hq, d]; k, v bf16 [B, Hkv, Lmax, d]; out f64 [B, n, Hq, d]
 * ---------------------------------------------------------------------- */
static double bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int orc_tree_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const int32_t* kv_len, const int32_t* parent, int B, int n, int Hq, int Hkv,
                  int d, int Lmax, double scale, double* out)
{
    if (Hkv <= 0 || Hq % Hkv != 0) return ORC_BAD_TREE;
    const int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        uint64_t anc[64];
        int32_t depth[64];
        if (orc_tree_check(parent + (int64_t)b * n, n, anc, depth) != ORC_OK) return ORC_BAD_TREE;
        if (kv_len[b] < 0 || kv_len[b] + n > Lmax) return ORC_CAPACITY;
    }
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            uint64_t anc[64];
            int32_t depth[64];
            orc_tree_check(parent + (int64_t)b * n, n, anc, depth);
            const int L = kv_len[b];
            const int kvh = h / G;
            const uint16_t* K = k + ((int64_t)b * Hkv + kvh) * Lmax * d;
            const uint16_t* Vv = v + ((int64_t)b * Hkv + kvh) * Lmax * d;
            double* s = (double*)malloc(sizeof(double) * (L + n));
            int* key = (int*)malloc(sizeof(int) * (L + n));
            double* qd = (double*)malloc(sizeof(double) * d);
            for (int i = 0; i < n; ++i) {
                const uint16_t* Q = q + (((int64_t)b * n + i) * Hq + h) * d;
                for (int e = 0; e < d; ++e) qd[e] = bf16_to_double(Q[e]);
                int nk = 0;
                for (int j = 0; j < L; ++j) key[nk++] = j;
                for (int j = 0; j < n; ++j)
                    if (anc[i] >> j & 1ull) key[nk++] = L + j;
                double mx = -INFINITY;
                for (int t = 0; t < nk; ++t) {
                    const uint16_t* Kr = K + (int64_t)key[t] * d;
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e) acc += qd[e] * bf16_to_double(Kr[e]);
                    s[t] = acc * scale;
                    if (s[t] > mx) mx = s[t];
                }
                double den = 0.0;
                for (int t = 0; t < nk; ++t) { s[t] = exp(s[t] - mx); den += s[t]; }
                double* O = out + (((int64_t)b * n + i) * Hq + h) * d;
                for (int e = 0; e < d; ++e) O[e] = 0.0;
                for (int t = 0; t < nk; ++t) {
                    const uint16_t* Vr = Vv + (int64_t)key[t] * d;
                    double w = s[t] / den;
                    for (int e = 0; e < d; ++e) O[e] += w * bf16_to_double(Vr[e]);
                }
            }
            free(s);
            free(key);
            free(qd);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Training-time-test attention (TTT page, section
 * "训练时的 attention mask 为什么要特殊处理").  Round 0 runs on the original
 * tokens with the ordinary causal mask.  Round r >= 1 feeds back, at every
 * position i, the token the previous round
 * predicted there; a simulated token may see only its own ancestors: the
 * original tokens up to its position (0..i) and the tokens of rounds 1..r at
 * the same position (its own chain, itself included), never another
 * position's simulated tokens.  For the queries of round r, query head h,
 * kv head h / (Hq / Hkv): plain softmax(scale * q.k) . v over that key list,
 * all in double.
 *   q bf16 [B, S, Hq, d] (the queries of round r);
 *   k, v bf16 [B, Hkv, R1, S, d] (round 0 = original tokens, rounds 1..R1-1);
 *   out f64 [B, S, Hq, d]
 * ---------------------------------------------------------------------- */
int orc_ttt_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int S, int Hq,
                 int Hkv, int d, int R1, int r, double scale, double* out)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || r < 0 || r >= R1) return ORC_BAD_TREE;
    const int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            const int kvh = h / G;
            const int64_t slab = ((int64_t)b * Hkv + kvh) * R1 * S;   /* row (round, pos) */
            double* s = (double*)malloc(sizeof(double) * (S + R1));
            int64_t* key = (int64_t*)malloc(sizeof(int64_t) * (S + R1));
            double* qd = (double*)malloc(sizeof(double) * d);
            for (int i = 0; i < S; ++i) {
                const uint16_t* Q = q + (((int64_t)b * S + i) * Hq + h) * d;
                for (int e = 0; e < d; ++e) qd[e] = bf16_to_double(Q[e]);
                int nk = 0;
                for (int j = 0; j <= i; ++j) key[nk++] = slab + j;                     /* round 0 */
                for (int rr = 1; rr <= r; ++rr) key[nk++] = slab + (int64_t)rr * S + i;  /* chain */
                double mx = -INFINITY;
                for (int t = 0; t < nk; ++t) {
                    const uint16_t* Kr = k + key[t] * d;
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e) acc += qd[e] * bf16_to_double(Kr[e]);
                    s[t] = acc * scale;
                    if (s[t] > mx) mx = s[t];
                }
                double den = 0.0;
                for (int t = 0; t < nk; ++t) { s[t] = exp(s[t] - mx); den += s[t]; }
                double* O = out + (((int64_t)b * S + i) * Hq + h) * d;
                for (int e = 0; e < d; ++e) O[e] = 0.0;
                for (int t = 0; t < nk; ++t) {
                    const uint16_t* Vr = v + key[t] * d;
                    double w = s[t] / den;
                    for (int e = 0; e < d; ++e) O[e] += w * bf16_to_double(Vr[e]);
                }
            }
            free(s);
            free(key);
            free(qd);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * KV compaction and logical-length update (Lesson "KV cache 回滚" and
 * "第 4 步": keep one physical cache plus a logical length).  The tree's
 * K/V rows sit at L_b + j.  After acceptance the rows of the accepted path
 * (root first) must be contiguous behind the committed prefix: for
 * t = 0..a, row L_b + path[t] moves to row L_b + t, in every layer and kv
 * head, for K and V; then kv_len[b] += a + 1 (root plus accepted drafts;
 * the final token is the next root and has no KV yet).  Done literally:
 * every source row is copied out first, then written.
 *   k, v bf16 [n_layers, B, Hkv, Lmax, d]  (in place)
 * Sequences with accept_len < 0 are left untouched.
 * ---------------------------------------------------------------------- */
int orc_kv_compact(uint16_t* k, uint16_t* v, int32_t* kv_len, const int32_t* path,
                   const int32_t* accept_len, int n_layers, int B, int Hkv, int d, int Lmax,
                   int max_depth)
{
    int st = ORC_OK;
    uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(max_depth + 1) * d);
    for (int b = 0; b < B; ++b) {
        int a = accept_len[b];
        if (a < 0) continue;
        const int32_t* P = path + (int64_t)b * (max_depth + 1);
        const int L = kv_len[b];
        if (a > max_depth || L + P[a] >= Lmax) { st |= ORC_CAPACITY; continue; }
        for (int layer = 0; layer < n_layers; ++layer) {
            for (int kv = 0; kv < 2; ++kv) {
                uint16_t* C = kv ? v : k;
                for (int h = 0; h < Hkv; ++h) {
                    uint16_t* base = C + ((((int64_t)layer * B + b) * Hkv + h) * Lmax) * d;
                    for (int t = 0; t <= a; ++t)
                        memcpy(tmp + (size_t)t * d, base + (int64_t)(L + P[t]) * d, sizeof(uint16_t) * d);
                    for (int t = 0; t <= a; ++t)
                        memcpy(base + (int64_t)(L + t) * d, tmp + (size_t)t * d, sizeof(uint16_t) * d);
                }
            }
        }
        kv_len[b] = L + a + 1;
    }
    free(tmp);
    return st;
}

/* ------------------------------------------------------------------------
 * Draft LM head (Guide "EAGLE-3" code changes: the draft head's own
 * lm_head = Linear(hidden, draft_vocab, bias=False)): logits = hidden . W^T.
 * Only the listed rows are computed (the full product is large).
 *   hidden bf16 [M, K]; w bf16 [N, K]; out f64 [nrows, N]
 * ---------------------------------------------------------------------- */
void orc_lmhead_rows(const uint16_t* hidden, const uint16_t* w, int M, int K, int N,
                     const int32_t* rows, int nrows, double* out)
{
    (void)M;
    for (int r = 0; r < nrows; ++r) {
        const uint16_t* h = hidden + (int64_t)rows[r] * K;
        double* hd = (double*)malloc(sizeof(double) * K);
        for (int e = 0; e < K; ++e) hd[e] = bf16_to_double(h[e]);
#pragma omp parallel for schedule(static)
        for (int c = 0; c < N; ++c) {
            const uint16_t* wr = w + (int64_t)c * K;
            double acc = 0.0;
            for (int e = 0; e < K; ++e) acc += hd[e] * bf16_to_double(wr[e]);
            out[(int64_t)r * N + c] = acc;
        }
        free(hd);
    }
}

/* ------------------------------------------------------------------------
 * Draft confidence and per-row top-k (Guide "EAGLE-2", "一个可核对的经验
 * 性质": the draft model's confidence, i.e. its probability, approximates
 * the acceptance rate).  c_t = softmax(row)_t at temperature 1; the k
 * tokens with the largest c (equivalently the largest logit; lower token
 * id first on ties) are returned with their confidences, best first.
 * ---------------------------------------------------------------------- */
void orc_row_topk(const float* logits, int64_t rows, int V, int k, int32_t* tok, double* conf,
                  int32_t* status)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        const float* row = logits + r * (int64_t)V;
        double m, Z;
        int st = row_stats(row, V, 1.0, &m, &Z, NULL);
        if (status) status[r] = st;
        int32_t* T = tok + r * k;
        double* C = conf + r * k;
        for (int j = 0; j < k; ++j) { T[j] = -1; C[j] = 0.0; }
        if (st != ORC_OK) continue;
        /* Total order: larger logit first, lower token id first among equal
         * logits.  Pick j is the best token strictly after pick j-1. */
        for (int j = 0; j < k && j < V; ++j) {
            int prev = j ? T[j - 1] : -1;
            int best = -1;
            for (int t = 0; t < V; ++t) {
                if (prev >= 0 && !(row[t] < row[prev] || (row[t] == row[prev] && t > prev)))
                    continue;                       /* not after the previous pick */
                if (best < 0 || row[t] > row[best]) best = t;
            }
            T[j] = best;
            C[j] = exp((double)row[best] - m) / Z;
        }
    }
}
