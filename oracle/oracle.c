/*
 * oracle.c -- plain, slow CPU reference for one tree-verification pass.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library.  The
 * product path (the CUDA library and its Python binding) never calls it and
 * has no CPU fallback to it.  It shares no source, header, table or constant
 * generator with the CUDA path.
 *
 * Sources (cited by page title and section):
 *   [SpecInfer guide] "SpecInfer Guide: Tree-Based Speculative LLM Serving"
 *   [Inference opt.]  "Inference Optimization Techniques: Speed and Efficiency"
 *
 * Precision: attention is computed in fp64 and rounded once to the output
 * type.  The stochastic verifier takes integer decisions (accept / reject,
 * the sampled token) from floating point; there it follows the fp32
 * arithmetic contract written out above oracle_verify_stochastic, which the
 * kernels implement independently, so that both sides take each decision in
 * the same precision.  Build with -ffp-contract=off and without fast-math.
 *
 * Pins (tests that tie this file to something other than itself) are listed
 * in the header of oracle/__init__.py.  No function here is left unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Per-request status bits: the interface values of the library's device
 * status word (an interface both sides must agree on, defined here again). */
enum {
    ORC_BAD_TREE = 1,   /* parent[0] != -1, parent[i] outside [0, i), n > n_max */
    ORC_BAD_TOKEN = 2,  /* a token outside [0, V) */
    ORC_CAPACITY = 4,   /* prefix_len < 0 or prefix_len + n beyond the block table */
    ORC_BAD_BLOCK = 16, /* a block-table entry outside [0, num_blocks) */
    ORC_BAD_PATH = 32,  /* a commit path that is not a strictly increasing root path */
    ORC_BAD_TEMP = 64   /* an inverse temperature that is not finite and positive */
};
enum { ORC_F32 = 0, ORC_BF16 = 1 };

/* ------------------------------------------------------------------ */
/* Token tree                                                          */
/* ------------------------------------------------------------------ */

/* [SpecInfer guide] "Mathematical Formulation of the Token Tree": node u has
 * token t_u and parent p_u; S_u = S_{p_u} o t_u.  Flattened trees list each
 * parent before its children ("Depth-First Flattening and KV Cache Reuse"),
 * so the check is parent[0] == -1 and 0 <= parent[i] < i. */
static int tree_valid(const int32_t *parent, int n, int n_max)
{
    if (n < 0 || n > n_max) return 0;
    if (n == 0) return 1;
    if (parent[0] != -1) return 0;
    for (int i = 1; i < n; i++)
        if (parent[i] < 0 || parent[i] >= i) return 0;
    return 1;
}

/* Dense topology mask, [SpecInfer guide] "The Topology-Aware 2D Causal
 * Mask": M[u][v] = 0 if v is u or an ancestor of u, else -inf; built by
 * walking parent links from u to the root. */
static void dense_mask(const int32_t *parent, int n, double *M)
{
    for (int u = 0; u < n; u++) {
        for (int v = 0; v < n; v++) M[(size_t)u * n + v] = -INFINITY;
        M[(size_t)u * n + u] = 0.0;
        for (int c = parent[u]; c != -1; c = parent[c]) M[(size_t)u * n + c] = 0.0;
    }
}

static int node_depth(const int32_t *parent, int u)
{
    int d = 0;
    for (int c = parent[u]; c != -1; c = parent[c]) d++;
    return d;
}

/* Mask build: validate each request's tree, report depth[u] (number of
 * ancestors) and pack row u of the dense mask into 64-bit words, bit v of
 * word v/64 set iff M[u][v] == 0.  W = ceil(n_max / 64) words per node.
 * A request with a bad tree gets status ORC_BAD_TREE, all-zero mask rows and
 * depth -1.  status[] is written (not or-ed). */
int oracle_tree_mask_build(const int32_t *parent, const int32_t *tree_off, int B, int n_max,
                           uint64_t *mask, int32_t *depth, int32_t *status)
{
    int W = (n_max + 63) / 64;
    for (int b = 0; b < B; b++) {
        int off = tree_off[b], n = tree_off[b + 1] - off;
        status[b] = 0;
        if (!tree_valid(parent + off, n, n_max)) {
            status[b] = ORC_BAD_TREE;
            for (int u = 0; u < n; u++) {
                for (int w = 0; w < W; w++) mask[(size_t)(off + u) * W + w] = 0;
                depth[off + u] = -1;
            }
            continue;
        }
        double *M = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (n > 0 ? n : 1));
        dense_mask(parent + off, n, M);
        for (int u = 0; u < n; u++) {
            uint64_t *row = mask + (size_t)(off + u) * W;
            for (int w = 0; w < W; w++) row[w] = 0;
            for (int v = 0; v < n; v++)
                if (M[(size_t)u * n + v] == 0.0) row[v / 64] |= (uint64_t)1 << (v % 64);
            depth[off + u] = node_depth(parent + off, u);
        }
        free(M);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Element access                                                      */
/* ------------------------------------------------------------------ */

static double load_elem(const void *base, size_t i, int dtype)
{
    if (dtype == ORC_F32) return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* fp64 -> bfloat16, round to nearest, ties to even, in one rounding step
 * (no intermediate fp32 rounding).  bfloat16 keeps 8 significant bits, has
 * the fp32 exponent range and subnormal quantum 2^-133. */
static uint16_t f64_to_bf16(double x)
{
    if (isnan(x)) return 0x7fc0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);               /* a = m * 2^e, m in [0.5, 1) */
    int qexp = e - 8;           /* quantum of an 8-significant-bit value */
    if (qexp < -133) qexp = -133;
    double r = nearbyint(ldexp(a, -qexp)); /* exact scaling, then RNE to an integer */
    double y = ldexp(r, qexp);
    if (y > 3.3895313892515355e38) return sign | 0x7f80; /* above the largest bf16 */
    float f = (float)y;          /* exact: y has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)((bits >> 16) & 0x7fff);
}

static void store_elem(void *base, size_t i, int dtype, double v)
{
    if (dtype == ORC_F32) ((float *)base)[i] = (float)v;
    else ((uint16_t *)base)[i] = f64_to_bf16(v);
}

/* exported for the rounding pin */
uint16_t oracle_f64_to_bf16(double x) { return f64_to_bf16(x); }

/* Paged cache element (slot s of request b, kv-head h, dim d).  Layout:
 * cache[num_blocks][Hkv][block_size][D], block of slot s = block_table[b][s / block_size]. */
static size_t cache_index(const int32_t *bt_row, int block_size, int Hkv, int D, int h, int s, int d)
{
    int blk = bt_row[s / block_size];
    return (((size_t)blk * Hkv + h) * block_size + (size_t)(s % block_size)) * D + d;
}

/* ------------------------------------------------------------------ */
/* Tree attention                                                      */
/* ------------------------------------------------------------------ */

/* Shared request checks of the attention and commit steps. */
static int32_t request_checks(const int32_t *parent, int off, int n, int n_max, int P,
                              const int32_t *bt_row, int max_blocks, int block_size, int num_blocks)
{
    int32_t st = 0;
    if (!tree_valid(parent + off, n, n_max)) st |= ORC_BAD_TREE;
    if (P < 0 || (long long)P + (n > 0 ? n : 0) > (long long)max_blocks * block_size) {
        st |= ORC_CAPACITY;
        return st;
    }
    int used = (P + n + block_size - 1) / block_size;
    for (int i = 0; i < used; i++)
        if (bt_row[i] < 0 || bt_row[i] >= num_blocks) st |= ORC_BAD_BLOCK;
    return st;
}

/* [SpecInfer guide] "Generalizing Attention to Tree Topologies": node u
 * attends with weights alpha_{u,v} = softmax_v(Q_u K_v^T * scale + M_{u,v})
 * and output sum_v alpha_{u,v} V_v.  The key set is the committed prefix
 * (slots [0, P_b): every node sees the whole verified context, since S_u
 * extends the context by the root path) followed by the tree slots P_b + v
 * with M[u][v] == 0 (tree K/V appended after the prefix, "Depth-First
 * Flattening and KV Cache Reuse").  GQA: query head h reads kv-head
 * h / (Hq / Hkv).  Naive fp64: all scores, max, exponentials, weighted sum.
 *
 * q: [T][Hq][D]; out: [T][Hq][D] in dtype; out_f64 (optional): same, fp64.
 * rows (optional): list of n_rows flat indices t*Hq+h to compute; NULL = all.
 * status[b] is written: bad requests get their output rows zeroed. */
int oracle_tree_attention(const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_table, int max_blocks, int block_size, int num_blocks,
                          const int32_t *prefix_len, const int32_t *tree_off, const int32_t *parent,
                          int B, int n_max, int Hq, int Hkv, int D, int dtype, double scale,
                          const int64_t *rows, int64_t n_rows,
                          void *out, double *out_f64, int32_t *status)
{
    if (Hkv <= 0 || Hq % Hkv != 0) return 1;
    int g = Hq / Hkv;
    for (int b = 0; b < B; b++) {
        int off = tree_off[b], n = tree_off[b + 1] - off, P = prefix_len[b];
        const int32_t *bt_row = block_table + (size_t)b * max_blocks;
        status[b] = request_checks(parent, off, n, n_max, P, bt_row, max_blocks, block_size, num_blocks);
        /* which rows of this request to compute */
        int64_t lo = (int64_t)off * Hq, hi = (int64_t)(off + (n > 0 ? n : 0)) * Hq;
        if (status[b] != 0) {
            for (int64_t r = lo; r < hi; r++) {
                int want = rows == NULL;
                for (int64_t i = 0; !want && i < n_rows; i++) want = rows[i] == r;
                if (!want) continue;
                for (int d = 0; d < D; d++) {
                    store_elem(out, (size_t)r * D + d, dtype, 0.0);
                    if (out_f64) out_f64[(size_t)r * D + d] = 0.0;
                }
            }
            continue;
        }
        if (n == 0) continue;
        double *M = (double *)malloc(sizeof(double) * (size_t)n * n);
        dense_mask(parent + off, n, M);
        int maxkeys = P + n;
        int *slots = (int *)malloc(sizeof(int) * (size_t)maxkeys);
        double *s = (double *)malloc(sizeof(double) * (size_t)maxkeys);
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
        for (int u = 0; u < n; u++) {
            int nk = 0;
            for (int j = 0; j < P; j++) slots[nk++] = j;
            for (int v = 0; v < n; v++)
                if (M[(size_t)u * n + v] == 0.0) slots[nk++] = P + v;
            for (int h = 0; h < Hq; h++) {
                int64_t r = (int64_t)(off + u) * Hq + h;
                if (rows != NULL) {
                    int want = 0;
                    for (int64_t i = 0; !want && i < n_rows; i++) want = rows[i] == r;
                    if (!want) continue;
                }
                int kvh = h / g;
                double mx = -INFINITY;
                for (int k = 0; k < nk; k++) {
                    double acc = 0.0;
                    for (int d = 0; d < D; d++)
                        acc += load_elem(q, (size_t)r * D + d, dtype) *
                               load_elem(k_cache, cache_index(bt_row, block_size, Hkv, D, kvh, slots[k], d), dtype);
                    s[k] = acc * scale;
                    if (s[k] > mx) mx = s[k];
                }
                double Z = 0.0;
                for (int k = 0; k < nk; k++) {
                    s[k] = exp(s[k] - mx);
                    Z += s[k];
                }
                for (int d = 0; d < D; d++) o[d] = 0.0;
                for (int k = 0; k < nk; k++)
                    for (int d = 0; d < D; d++)
                        o[d] += s[k] * load_elem(v_cache, cache_index(bt_row, block_size, Hkv, D, kvh, slots[k], d), dtype);
                for (int d = 0; d < D; d++) {
                    double val = o[d] / Z;
                    store_elem(out, (size_t)r * D + d, dtype, val);
                    if (out_f64) out_f64[(size_t)r * D + d] = val;
                }
            }
        }
        free(o);
        free(s);
        free(slots);
        free(M);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Greedy verification                                                 */
/* ------------------------------------------------------------------ */

static int row_argmax(const float *row, int V)
{
    int best = 0;
    for (int x = 1; x < V; x++)
        if (row[x] > row[best]) best = x; /* ties keep the lowest token id */
    return best;
}

static int32_t verify_checks(const int32_t *parent, const int32_t *tokens, int off, int n, int n_max, int V)
{
    int32_t st = 0;
    if (!tree_valid(parent + off, n, n_max)) st |= ORC_BAD_TREE;
    for (int u = 0; u < n && u < n_max; u++)
        if (tokens[off + u] < 0 || tokens[off + u] >= V) {
            st |= ORC_BAD_TOKEN;
            break;
        }
    return st;
}

static void clear_outputs(int b, int n_max, int32_t *path, int32_t *accept_len, int32_t *emitted, int32_t *n_emitted)
{
    for (int i = 0; i < n_max; i++) {
        path[(size_t)b * n_max + i] = -1;
        emitted[(size_t)b * n_max + i] = -1;
    }
    accept_len[b] = 0;
    n_emitted[b] = 0;
}

/* [SpecInfer guide] "Greedy Verification Algorithm": starting at the root r,
 * take t_pred = argmax_w P(w | S_r), descend into a child whose token equals
 * t_pred, repeat; when no child matches, t_pred is emitted and verification
 * ends.  p_logits[u] is the target distribution after S_u, so child c is
 * tested against argmax of row parent(c).  Written as: ok[root] = 1,
 * ok[c] = ok[parent c] and tokens[c] == argmax(p_logits[parent c]); the
 * accepted node f is the deepest ok node (ties: lowest node index), the
 * longest root path that follows the target's argmax chain.  The root is the
 * last verified token: it is always accepted and not emitted again.  Emitted
 * tokens: the tokens of the accepted non-root nodes, then argmax(p_logits[f])
 * (the correction, or the bonus token when f is a leaf).
 * path[b][i], emitted[b][i]: [B][n_max], unused entries -1.
 * status[b] is written. */
int oracle_verify_greedy(const float *p_logits, const int32_t *tokens, const int32_t *parent,
                         const int32_t *tree_off, int B, int n_max, int V,
                         int32_t *path, int32_t *accept_len, int32_t *emitted, int32_t *n_emitted,
                         int32_t *status)
{
    for (int b = 0; b < B; b++) {
        int off = tree_off[b], n = tree_off[b + 1] - off;
        clear_outputs(b, n_max, path, accept_len, emitted, n_emitted);
        status[b] = verify_checks(parent, tokens, off, n, n_max, V);
        if (status[b] != 0 || n == 0) continue;
        const int32_t *par = parent + off;
        int *a = (int *)malloc(sizeof(int) * (size_t)n);
        int *ok = (int *)malloc(sizeof(int) * (size_t)n);
        for (int u = 0; u < n; u++) a[u] = row_argmax(p_logits + (size_t)(off + u) * V, V);
        ok[0] = 1;
        for (int c = 1; c < n; c++) ok[c] = ok[par[c]] && tokens[off + c] == a[par[c]];
        int f = 0, fd = 0;
        for (int u = 1; u < n; u++) {
            int d = node_depth(par, u);
            if (ok[u] && d > fd) {
                f = u;
                fd = d;
            }
        }
        int len = fd + 1;
        for (int i = len - 1, c = f; i >= 0; i--, c = par[c]) path[(size_t)b * n_max + i] = c;
        for (int i = 0; i + 1 < len; i++) emitted[(size_t)b * n_max + i] = tokens[off + path[(size_t)b * n_max + i + 1]];
        emitted[(size_t)b * n_max + len - 1] = a[f];
        accept_len[b] = len;
        n_emitted[b] = len;
        free(ok);
        free(a);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Stochastic verification: the fp32 arithmetic contract               */
/* ------------------------------------------------------------------ */
/*
 * The accept/reject rule is [Inference opt.] "Misconception: ..." section:
 * accept a draft token x with probability min(1, p(x)/q(x)); on rejection
 * resample from residual(x) = max(p(x) - q(x), 0) / Z.  [SpecInfer guide]
 * "Stochastic Verification Algorithm" applies it at every tree node, with
 * the residual P_residual as the new target after a rejection.  Several
 * children of a node are tried in increasing node index, each against the
 * residual left by the siblings rejected before it (multi-step speculative
 * sampling over all siblings in order); q_probs[u] is the draft distribution
 * from which every child of u was proposed.
 *
 * Contract (both the oracle and the kernels implement it, separately):
 *  C1 uniforms are raw 32-bit words: uniforms[t][0] is node t's acceptance
 *     word, uniforms[t][1] the sampling word if the walk stops at t.  The
 *     acceptance uniform is (w >> 8) * 2^-24, exact in fp32.
 *  C2 E(x), x <= 0: canon_exp below.
 *  C3 FX(v) = (uint64) trunc(v * 2^46) for v in [0, 2); sums of FX values
 *     are exact and order-free (V <= 2^17 keeps them below 2^63);
 *     Z(S) = fp32(S) * 2^-46.
 *  C4 row state of node u: m = max_x l(x); e(x) = E(l(x) - m) (fp32 sub);
 *     S_0 = sum FX(e); r_0(x) = e(x) / Z(S_0) (IEEE division).
 *  C5 after the j-th rejection: d_j(x) = r_{j-1}(x) - q(x) if that is > 0,
 *     else 0; S_j = sum FX(d_j); r_j(x) = d_j(x) / Z(S_j).  If S_j == 0
 *     (impossible in exact arithmetic after a rejection) d_j, S_j and r_j
 *     stay those of step j-1 (d_0 = e).
 *  C6 child c with token t, tested after j rejections: accept iff
 *     u_acc(c) * q(t) <= r_j(t), one fp32 multiply.
 *  C7 when no child is accepted (or the node is a leaf), sample from the
 *     weights w = e (j == 0) or d_j: W(x) = FX(w(x)), S = sum W,
 *     target = floor(U * S / 2^32) with U the raw sampling word, emit the
 *     smallest x with W(0) + ... + W(x) > target.
 * Every multiply, add, subtract and divide is a single IEEE fp32 operation;
 * the only fused multiply-adds are the explicit fmaf calls in canon_exp.
 */

static float f32_from_bits(uint32_t b)
{
    float f;
    memcpy(&f, &b, 4);
    return f;
}

/* C2.  e^x for x <= 0 from mathematics: Cody-Waite reduction x = n ln2 + r
 * (|r| <= ln2/2) with ln2 split as LN2_HI + LN2_LO, LN2_HI holding 16
 * significant bits so n * LN2_HI is exact for |n| < 256; the degree-7 Taylor
 * polynomial sum r^k / k! in Horner form; scaling by 2^n through the exponent
 * field.  Constants are the correctly rounded fp32 values (bit patterns):
 * log2(e), ln2 truncated to 16 bits, the fp32 remainder, and 1/k!. */
float oracle_canon_exp(float x)
{
    if (!(x >= -87.0f)) return 0.0f;
    const float LOG2E = f32_from_bits(0x3fb8aa3bu);
    const float LN2_HI = f32_from_bits(0x3f317200u);
    const float LN2_LO = f32_from_bits(0x35bfbe8eu);
    const float C[8] = {f32_from_bits(0x3f800000u), f32_from_bits(0x3f800000u), f32_from_bits(0x3f000000u),
                        f32_from_bits(0x3e2aaaabu), f32_from_bits(0x3d2aaaabu), f32_from_bits(0x3c088889u),
                        f32_from_bits(0x3ab60b61u), f32_from_bits(0x39500d01u)};
    float t = x * LOG2E;
    float n = rintf(t);
    float r = fmaf(-n, LN2_HI, x);
    r = fmaf(-n, LN2_LO, r);
    float p = C[7];
    for (int k = 6; k >= 0; k--) p = fmaf(p, r, C[k]);
    int ni = (int)n;
    float scale = f32_from_bits((uint32_t)(ni + 127) << 23);
    return p * scale;
}

/* C3 */
uint64_t oracle_fx(float v) { return (uint64_t)(v * 0x1p46f); }
static float z_of(uint64_t S) { return (float)S * 0x1p-46f; }

/* C7: floor(U * S / 2^32) exactly (U < 2^32, S < 2^63). */
static uint64_t sample_target(uint32_t U, uint64_t S)
{
    unsigned __int128 prod = (unsigned __int128)U * S;
    return (uint64_t)(prod >> 32);
}

/* Residual state of one node row (C4, C5) kept as full vectors. */
typedef struct {
    float *e, *d, *r, *dn;
    uint64_t S;
} row_state;

/* C4: row state of logits l (V entries) at inverse temperature tau
 * ([SpecInfer guide] "Stochastic Verification Algorithm" samples at
 * temperature T > 0: the target is softmax(l / T), here with tau = 1/T given
 * in fp32 and applied as one rounded multiply of l - m); d holds the current
 * weights (e for j == 0), r the current target distribution r_j. */
static void row_init(row_state *st, const float *l, int V, float tau)
{
    float m = l[0];
    for (int x = 1; x < V; x++)
        if (l[x] > m) m = l[x];
    uint64_t S = 0;
    for (int x = 0; x < V; x++) {
        float y = l[x] - m;
        y = y * tau;
        st->e[x] = oracle_canon_exp(y);
        S += oracle_fx(st->e[x]);
    }
    st->S = S;
    float Z = z_of(S);
    for (int x = 0; x < V; x++) {
        st->d[x] = st->e[x];
        st->r[x] = st->e[x] / Z;
    }
}

/* C5: one rejection against draft row q. */
static void row_reject(row_state *st, const float *q, int V)
{
    uint64_t S = 0;
    for (int x = 0; x < V; x++) {
        float diff = st->r[x] - q[x];
        st->dn[x] = diff > 0.0f ? diff : 0.0f;
        S += oracle_fx(st->dn[x]);
    }
    if (S == 0) return; /* keep d, S, r of the previous step */
    float Z = z_of(S);
    for (int x = 0; x < V; x++) {
        st->d[x] = st->dn[x];
        st->r[x] = st->dn[x] / Z;
    }
    st->S = S;
}

/* C7 */
static int row_sample(const row_state *st, int V, uint32_t U)
{
    uint64_t target = sample_target(U, st->S), acc = 0;
    for (int x = 0; x < V; x++) {
        acc += oracle_fx(st->d[x]);
        if (acc > target) return x;
    }
    return V - 1; /* unreachable: target < S */
}

/* Exposed for the per-token pins: the target distribution r_j of a row
 * (logits l at inverse temperature tau) after j rejections against the
 * draft rows q[0..j-1] (each V entries), and its weights d_j. */
void oracle_residual(const float *l, const float *q, int V, int j, float tau, float *r_out, float *d_out,
                     uint64_t *S_out)
{
    row_state st;
    st.e = (float *)malloc(sizeof(float) * (size_t)V * 4);
    st.d = st.e + V;
    st.r = st.d + V;
    st.dn = st.r + V;
    row_init(&st, l, V, tau);
    for (int k = 0; k < j; k++) row_reject(&st, q + (size_t)k * V, V);
    memcpy(r_out, st.r, sizeof(float) * (size_t)V);
    memcpy(d_out, st.d, sizeof(float) * (size_t)V);
    *S_out = st.S;
    free(st.e);
}

/* Stochastic tree verification: a sequential walk from the root.  At node
 * u the children are tried in increasing index (C6), a rejection moves the
 * target to the next residual (C5); the first accepted child becomes the
 * new node; if every child is rejected, or u is a leaf, a token is sampled
 * from the current weights (C7) and the walk ends.  Outputs as in
 * oracle_verify_greedy.  status[b] is written.
 *
 * inv_temp[b] (NULL: 1) is request b's inverse temperature (C4); it must be
 * finite and positive, else the request gets ORC_BAD_TEMP and is skipped.
 * Draft rows: with q_per_child == 0, q_probs row u is the distribution all
 * children of u were drawn from (one draft model expanding u).  With
 * q_per_child != 0, row c is the distribution child c itself was drawn from
 * ([SpecInfer guide] "Merge-Based Tree Construction": siblings proposed by
 * different draft models); child c is then tested against, and on rejection
 * subtracted as, its own row: accept iff u * q_c(t_c) <= r_j(t_c), and
 * r_{j+1} = norm(max(r_j - q_c, 0)). */
int oracle_verify_stochastic(const float *p_logits, const float *q_probs, const int32_t *tokens,
                             const int32_t *parent, const int32_t *tree_off, const uint32_t *uniforms,
                             int B, int n_max, int V, const float *inv_temp, int q_per_child,
                             int32_t *path, int32_t *accept_len, int32_t *emitted, int32_t *n_emitted,
                             int32_t *status)
{
    row_state st;
    st.e = (float *)malloc(sizeof(float) * (size_t)V * 4);
    st.d = st.e + V;
    st.r = st.d + V;
    st.dn = st.r + V;
    for (int b = 0; b < B; b++) {
        int off = tree_off[b], n = tree_off[b + 1] - off;
        clear_outputs(b, n_max, path, accept_len, emitted, n_emitted);
        status[b] = verify_checks(parent, tokens, off, n, n_max, V);
        const float tau = inv_temp ? inv_temp[b] : 1.0f;
        if (!(tau > 0.0f) || isinf(tau)) status[b] |= ORC_BAD_TEMP;
        if (status[b] != 0 || n == 0) continue;
        const int32_t *par = parent + off;
        int32_t *pth = path + (size_t)b * n_max, *emt = emitted + (size_t)b * n_max;
        int u = 0, len = 1;
        pth[0] = 0;
        for (;;) {
            const float *l = p_logits + (size_t)(off + u) * V;
            const float *q = q_probs + (size_t)(off + u) * V;
            row_init(&st, l, V, tau);
            int accepted = -1;
            for (int c = u + 1; c < n; c++) {
                if (par[c] != u) continue;
                int t = tokens[off + c];
                const float *qc = q_per_child ? q_probs + (size_t)(off + c) * V : q;
                float ua = (float)(uniforms[(size_t)(off + c) * 2] >> 8) * 0x1p-24f;
                if (ua * qc[t] <= st.r[t]) {
                    accepted = c;
                    break;
                }
                row_reject(&st, qc, V);
            }
            if (accepted >= 0) {
                emt[len - 1] = tokens[off + accepted];
                pth[len++] = accepted;
                u = accepted;
                continue;
            }
            emt[len - 1] = row_sample(&st, V, uniforms[(size_t)(off + u) * 2 + 1]);
            break;
        }
        accept_len[b] = len;
        n_emitted[b] = len;
    }
    free(st.e);
    return 0;
}

/* ------------------------------------------------------------------ */
/* KV commit / rollback                                                */
/* ------------------------------------------------------------------ */

/* [SpecInfer guide] "Depth-First Flattening and KV Cache Reuse": after
 * verification only the accepted path stays in the cache.  Row P_b + i of
 * every kv-head receives the old row P_b + path[b][i], i < accept_len[b],
 * read from a snapshot of the cache taken before any write; new_len[b] =
 * P_b + accept_len[b].  A request whose incoming status is non-zero, or
 * whose accept_len is 0, is left untouched (new_len = P_b).  A path that is
 * not strictly increasing from 0, or that leaves the block table, is
 * reported as ORC_BAD_PATH and left untouched.  status[b] is or-ed. */
int oracle_kv_commit(void *k_cache, void *v_cache, int64_t cache_elems,
                     const int32_t *block_table, int max_blocks, int block_size, int num_blocks,
                     const int32_t *prefix_len, const int32_t *path, int path_stride, const int32_t *accept_len,
                     int B, int Hkv, int D, int dtype, int32_t *new_len, int32_t *status)
{
    size_t es = dtype == ORC_F32 ? 4 : 2;
    unsigned char *ks = (unsigned char *)malloc((size_t)cache_elems * es);
    unsigned char *vs = (unsigned char *)malloc((size_t)cache_elems * es);
    memcpy(ks, k_cache, (size_t)cache_elems * es);
    memcpy(vs, v_cache, (size_t)cache_elems * es);
    for (int b = 0; b < B; b++) {
        int P = prefix_len[b], a = accept_len[b];
        new_len[b] = P;
        if (status[b] != 0 || a <= 0) continue;
        const int32_t *bt_row = block_table + (size_t)b * max_blocks;
        const int32_t *pth = path + (size_t)b * path_stride;
        int ok = a <= path_stride && pth[0] == 0 && P >= 0;
        for (int i = 1; ok && i < a; i++) ok = pth[i] > pth[i - 1];
        if (ok) ok = (long long)P + pth[a - 1] + 1 <= (long long)max_blocks * block_size;
        if (!ok) {
            status[b] |= ORC_BAD_PATH;
            continue;
        }
        int used = (P + pth[a - 1] + 1 + block_size - 1) / block_size;
        int bad = 0;
        for (int i = 0; i < used; i++) bad |= bt_row[i] < 0 || bt_row[i] >= num_blocks;
        if (bad) {
            status[b] |= ORC_BAD_BLOCK;
            continue;
        }
        for (int i = 0; i < a; i++)
            for (int h = 0; h < Hkv; h++) {
                size_t dst = cache_index(bt_row, block_size, Hkv, D, h, P + i, 0);
                size_t src = cache_index(bt_row, block_size, Hkv, D, h, P + pth[i], 0);
                memcpy((unsigned char *)k_cache + dst * es, ks + src * es, (size_t)D * es);
                memcpy((unsigned char *)v_cache + dst * es, vs + src * es, (size_t)D * es);
            }
        new_len[b] = P + a;
    }
    free(vs);
    free(ks);
    return 0;
}

/* [SpecInfer guide] "Depth-First Flattening and KV Cache Reuse", step 1 of
 * the verification pass: every tree token appends its computed key and
 * value to the request's active cache, in the tree's flattened node order,
 * right after the committed prefix.  Row h of node u of request b
 * (k_new[tree_off[b] + u][h][0..D-1], likewise v_new) is written to slot
 * P_b + u of kv-head h.  A request whose n_b lies outside [0, n_max] gets
 * ORC_BAD_TREE; one whose prefix is negative or whose last tree slot lies
 * beyond its block table gets ORC_CAPACITY; one whose pages covering
 * [P_b, P_b + n_b) include an id outside [0, num_blocks) gets ORC_BAD_BLOCK.
 * Such requests are left untouched.  status[b] is or-ed; nothing else of
 * the cache changes. */
int oracle_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                     const int32_t *block_table, int max_blocks, int block_size, int num_blocks,
                     const int32_t *prefix_len, const int32_t *tree_off, int B, int n_max, int Hkv, int D,
                     int dtype, int32_t *status)
{
    size_t es = dtype == ORC_F32 ? 4 : 2;
    for (int b = 0; b < B; b++) {
        int off = tree_off[b], n = tree_off[b + 1] - off, P = prefix_len[b];
        if (n < 0 || n > n_max) {
            status[b] |= ORC_BAD_TREE;
            continue;
        }
        if (P < 0 || (long long)P + n > (long long)max_blocks * block_size) {
            status[b] |= ORC_CAPACITY;
            continue;
        }
        if (n == 0) continue;
        const int32_t *bt_row = block_table + (size_t)b * max_blocks;
        int bad = 0;
        for (int s = P; s < P + n; s++) {
            int blk = bt_row[s / block_size];
            bad |= blk < 0 || blk >= num_blocks;
        }
        if (bad) {
            status[b] |= ORC_BAD_BLOCK;
            continue;
        }
        for (int u = 0; u < n; u++)
            for (int h = 0; h < Hkv; h++) {
                size_t dst = cache_index(bt_row, block_size, Hkv, D, h, P + u, 0);
                size_t src = ((size_t)(off + u) * Hkv + h) * D;
                memcpy((unsigned char *)k_cache + dst * es, (const unsigned char *)k_new + src * es, (size_t)D * es);
                memcpy((unsigned char *)v_cache + dst * es, (const unsigned char *)v_new + src * es, (size_t)D * es);
            }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Multi-layer commit and page release                                 */
/* "SpecInfer Guide", "PagedKV Allocation with Zero-Copy Pruning": the  */
/* tree's K/V rows sit in pages of the request's block table; after     */
/* verification the accepted path is compacted in every layer (the same */
/* single-layer commit per layer), then the pages lying wholly past the */
/* new length go back to the free pool in one metadata update.          */
/* Reading: the tree of request b occupies slots [P, P + n_b); pages    */
/* ceil(new_len / bs) .. ceil((P + n_b) / bs) - 1 are released, their   */
/* block-table entries set to -1 and their ids appended to the pool in  */
/* request order, then page order.  Failed requests (status != 0) keep  */
/* every page.  When the pool cannot take every page of the call, none  */
/* is released and each request that had pages to release gets          */
/* ORC_CAPACITY.                                                        */
/* ------------------------------------------------------------------ */
int oracle_kv_release(int32_t *block_table, int max_blocks, int block_size, const int32_t *prefix_len,
                      const int32_t *tree_off, const int32_t *new_len, int32_t *status, int B,
                      int32_t *free_pool, int free_cap, int32_t *free_count)
{
    int cnt = *free_count;
    long long total = 0;
    for (int b = 0; b < B; b++) {
        if (status[b] != 0) continue;
        int n = tree_off[b + 1] - tree_off[b];
        int keep = (new_len[b] + block_size - 1) / block_size;
        int span = (prefix_len[b] + n + block_size - 1) / block_size;
        if (span > max_blocks) span = max_blocks;
        if (span > keep) total += span - keep;
    }
    int fits = cnt + total <= free_cap;
    for (int b = 0; b < B; b++) {
        if (status[b] != 0) continue;
        int n = tree_off[b + 1] - tree_off[b];
        int keep = (new_len[b] + block_size - 1) / block_size;
        int span = (prefix_len[b] + n + block_size - 1) / block_size;
        if (span > max_blocks) span = max_blocks;
        if (span <= keep) continue;
        if (!fits) {
            status[b] |= ORC_CAPACITY;
            continue;
        }
        int32_t *row = block_table + (size_t)b * max_blocks;
        for (int i = keep; i < span; i++) {
            free_pool[cnt++] = row[i];
            row[i] = -1;
        }
    }
    *free_count = cnt;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Tree construction                                                   */
/* ------------------------------------------------------------------ */

/* Rank order of draft scores: a before b iff a's value is larger, or equal
 * with the lower token id.  NaN ranks below every number; -0 equals +0. */
static int score_before(float va, int ia, float vb, int ib)
{
    int na = isnan(va), nb = isnan(vb);
    if (na != nb) return nb;
    if (!na && va != vb) return va > vb;
    return ia < ib;
}

/* One level of expansion ([SpecInfer guide] "Method A: Expansion-Based Tree
 * Construction": level i expands the top-k_i tokens of every node of level
 * i-1).  Each of the B requests has the same shape: its tree occupies
 * n_total slots from b * n_total; the F frontier nodes are level_start ..
 * level_start + F - 1; frontier node i's draft scores (logits or
 * probabilities: the top-k is the same) are row b * F + i of `scores`.
 * Children are appended after the frontier, frontier node by frontier
 * node, each node's k children in rank order: child r of frontier node i
 * is node level_start + F + i * k + r.  Selection is k passes, each taking
 * the best-ranked token not yet taken. */
int oracle_tree_expand_level(const float *scores, int B, int F, int V, int k, int level_start, int n_total,
                             int32_t *parent, int32_t *tokens)
{
    if (k < 0 || k > V || level_start + F + F * k > n_total) return -1;
    char *taken = (char *)malloc((size_t)V);
    for (int b = 0; b < B; b++)
        for (int i = 0; i < F; i++) {
            const float *row = scores + ((size_t)b * F + i) * V;
            memset(taken, 0, (size_t)V);
            for (int r = 0; r < k; r++) {
                int best = -1;
                for (int x = 0; x < V; x++)
                    if (!taken[x] && (best < 0 || score_before(row[x], x, row[best], best))) best = x;
                taken[best] = 1;
                size_t c = (size_t)b * n_total + level_start + F + (size_t)i * k + r;
                parent[c] = level_start + i;
                tokens[c] = best;
            }
        }
    free(taken);
    return 0;
}

/* Merge ([SpecInfer guide] "Method B: Merge-Based Tree Construction"):
 * request b's M candidate sequences (sequence s: seqs[b][s][0 .. lens[b][s]-1],
 * row stride m) are united into one token tree in which every prefix of
 * every sequence is a node and no two nodes share a token path (for all u
 * in N_s there is v in the merged tree with S_v = S_u; identical prefixes
 * are one node).  Node 0 is the root (root_tok[b], parent -1).  Nodes are
 * numbered in insertion order: sequences in order, each from its first
 * token on, a prefix getting the next index when no earlier sequence has
 * it.  Output is packed: request b's nodes at tree_off[b] .. tree_off[b+1]-1
 * (tree_off written, tree_off[0] = 0); node_of[b][s][j] = the node of prefix
 * (s, j) (-1 past the sequence's length); src[node] = s * m + j of the
 * prefix that created it (-1 for roots).  A length outside [0, m] sets
 * ORC_BAD_TREE, a token outside [0, V) ORC_BAD_TOKEN; such a request gets
 * only its root.  Arrays parent/tokens/src hold B * (1 + M * m) entries. */
int oracle_tree_merge(const int32_t *seqs, const int32_t *lens, const int32_t *root_tok, int B, int M, int m, int V,
                      int32_t *tree_off, int32_t *parent, int32_t *tokens, int32_t *src, int32_t *node_of,
                      int32_t *status)
{
    tree_off[0] = 0;
    for (int b = 0; b < B; b++) {
        const int32_t *S = seqs + (size_t)b * M * m;
        const int32_t *len = lens + (size_t)b * M;
        int32_t *no = node_of + (size_t)b * M * m;
        int st = 0;
        for (int s = 0; s < M; s++) {
            if (len[s] < 0 || len[s] > m) st |= ORC_BAD_TREE;
            else
                for (int j = 0; j < len[s]; j++)
                    if (S[(size_t)s * m + j] < 0 || S[(size_t)s * m + j] >= V) st |= ORC_BAD_TOKEN;
        }
        if (root_tok[b] < 0 || root_tok[b] >= V) st |= ORC_BAD_TOKEN;
        status[b] = st;
        int base = tree_off[b], n = 1;
        parent[base] = -1;
        tokens[base] = root_tok[b];
        src[base] = -1;
        for (int i = 0; i < M * m; i++) no[i] = -1;
        if (st == 0) {
            for (int s = 0; s < M; s++)
                for (int j = 0; j < len[s]; j++) {
                    int par = j == 0 ? 0 : no[(size_t)s * m + j - 1];
                    int tok = S[(size_t)s * m + j];
                    /* an existing child of par with this token is the same prefix */
                    int found = -1;
                    for (int v = 1; v < n; v++)
                        if (parent[base + v] == par && tokens[base + v] == tok) {
                            found = v;
                            break;
                        }
                    if (found < 0) {
                        found = n++;
                        parent[base + found] = par;
                        tokens[base + found] = tok;
                        src[base + found] = s * m + j;
                    }
                    no[(size_t)s * m + j] = found;
                }
        }
        tree_off[b + 1] = base + n;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 uniforms                                              */
/* ------------------------------------------------------------------ */

/* Philox4x32 with 10 rounds, from Salmon, Moraes, Dror and Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3" (SC'11): each round multiplies
 * counter words 0 and 2 by 0xD2511F53 and 0xCD9E8D57 (64-bit products split
 * into hi and lo halves), outputs (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0),
 * and bumps the key by the Weyl constants 0x9E3779B9 and 0xBB67AE85. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; round++) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c[0] = n0;
        c[1] = n1;
        c[2] = n2;
        c[3] = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    for (int i = 0; i < 4; i++) out[i] = c[i];
}

/* Uniform words for one verification round: node u (local index) of
 * request b draws Philox4x32-10 at counter (u, b, round, 0) under key
 * (seed_lo, seed_hi); word 0 -> out[t][0], word 1 -> out[t][1]. */
int oracle_philox_uniforms(uint64_t seed, uint32_t round, const int32_t *tree_off, int B, uint32_t *out)
{
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    for (int b = 0; b < B; b++)
        for (int t = tree_off[b]; t < tree_off[b + 1]; t++) {
            uint32_t ctr[4] = {(uint32_t)(t - tree_off[b]), (uint32_t)b, round, 0}, w[4];
            oracle_philox4x32_10(ctr, key, w);
            out[(size_t)t * 2] = w[0];
            out[(size_t)t * 2 + 1] = w[1];
        }
    return 0;
}

/* Array helper for the exp pin. */
void oracle_canon_exp_array(const float *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; i++) y[i] = oracle_canon_exp(x[i]);
}

/* Array helpers for the contract's pins: C3's weight of every entry, and one
 * C5 residual step per entry as row_reject takes it (the previous target
 * r = d / Z, then max(r - q, 0)), with Z = Zp[i / 2]: two neighbouring
 * entries share one normaliser. */
void oracle_fx_array(const float *v, uint64_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_fx(v[i]);
}

void oracle_resid_step_array(const float *d, const float *q, const float *Zp, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) {
        float r = d[i] / Zp[i / 2];
        float diff = r - q[i];
        out[i] = diff > 0.0f ? diff : 0.0f;
    }
}


/* ------------------------------------------------------------------ */
/* Dynamic draft length (goodput tables)                               */
/* ------------------------------------------------------------------ */

/* "Hardware-aware dynamic speculative decoding": goodput = AL / ITL; the
 * offline table holds, per batch size, the K of highest goodput.  al and
 * itl are [n_bs][n_k] measurements for the draft lengths k_values[0..n_k-1];
 * a cell counts only when both are finite and itl > 0.  k_opt[b] = the K of
 * the largest goodput in row b, the earliest column on ties; -1 when no cell
 * of the row counts. */
int oracle_dsd_optimal_k(const double *al, const double *itl, int n_bs, int n_k, const int32_t *k_values,
                         int32_t *k_opt)
{
    for (int b = 0; b < n_bs; b++) {
        int best = -1;
        double best_g = 0.0;
        for (int j = 0; j < n_k; j++) {
            double a = al[(size_t)b * n_k + j], t = itl[(size_t)b * n_k + j];
            if (!isfinite(a) || !isfinite(t) || !(t > 0.0)) continue;
            double g = a / t;
            if (best < 0 || g > best_g) {
                best = j;
                best_g = g;
            }
        }
        k_opt[b] = best < 0 ? -1 : k_values[best];
    }
    return 0;
}

/* Runtime lookup: the table's entry for the largest profiled batch size not
 * above bs (bs_table ascending); below the first entry, the first. */
int oracle_dsd_select_k(const int32_t *bs_table, const int32_t *k_table, int n, int bs)
{
    if (n <= 0) return -1;
    int k = k_table[0];
    for (int i = 0; i < n; i++)
        if (bs_table[i] <= bs) k = k_table[i];
    return k;
}

/* Graph keys (same page, "Compatibility with full CUDA Graph"): every
 * <tokens, K> with 1 <= tokens <= max_tokens and 1 <= K <= max_k such that
 * tokens is divisible by K + 1 (then every request of the batch is a decode
 * request with K drafts), in increasing tokens, then K.  Returns the count;
 * at most cap pairs are stored. */
int oracle_dsd_graph_keys(int max_tokens, int max_k, int32_t *tokens_out, int32_t *k_out, int cap)
{
    int n = 0;
    for (int t = 1; t <= max_tokens; t++)
        for (int k = 1; k <= max_k; k++)
            if (t % (k + 1) == 0) {
                if (n < cap) {
                    tokens_out[n] = t;
                    k_out[n] = k;
                }
                n++;
            }
    return n;
}

/* Live statistics folded into a cell: x <- (1 - w) x + w * sample, for w in
 * (0, 1]; a cell without a finite value takes the sample. */
double oracle_dsd_blend(double cell, double sample, double w)
{
    if (!isfinite(cell)) return sample;
    return (1.0 - w) * cell + w * sample;
}
