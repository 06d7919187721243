/*
 * spectree.h -- C ABI of the GB300 (sm_103a) tree speculative verification
 * library (libspectree.so).
 *
 * One verification pass of tree-based speculative inference: the target model
 * checks a whole token tree in one forward pass, with every tree node attending
 * to the committed prefix plus its own ancestors, then a verifier picks the
 * accepted root path (greedy, or stochastic with the min(1, p/q) accept rule
 * and the norm(max(p - q, 0)) residual), and the KV cache keeps only that path.
 * Sources, by page title and section:
 *   "SpecInfer Guide: Tree-Based Speculative LLM Serving": "Mathematical
 *     Formulation of the Token Tree", "Tree-Based Parallel Decoding &
 *     Topology-Aware Causal Masking", "Depth-First Flattening and KV Cache
 *     Reuse", "Exact Output Verification: Greedy and Stochastic Sampling",
 *     "Integration with Continuous Batching", "PagedKV Allocation with
 *     Zero-Copy Pruning".
 *   "Inference Optimization Techniques: Speed and Efficiency": the accept rule
 *     and residual of the "Misconception" section, "Traced Example".
 *   Around the pass: "Token Tree Construction: Expansion vs. Merge" (SpecInfer
 *     guide) for the tree builders, and "Hardware-aware dynamic speculative
 *     decoding" (Cohere) for the goodput table and the <tokens, K> graph keys.
 *
 * Conventions shared by every call
 *   - Every pointer argument is DEVICE memory owned by the caller, except where
 *     a call says otherwise.  The library never allocates, frees or
 *     synchronises; each call enqueues kernels on `stream` (a cudaStream_t,
 *     NULL = the legacy default stream) and returns.
 *   - A batch holds B requests.  Request b owns tree nodes
 *     [tree_off[b], tree_off[b+1]) of every per-node array (ragged packing).
 *     Inside a request nodes are numbered 0..n_b-1 (local index); node 0 is
 *     the root, the last verified token, and parent[t] is the LOCAL index of
 *     the parent (-1 for the root).  Parents come before children:
 *     0 <= parent[i] < i.  n_b <= n_max <= 1024.
 *   - mask rows have W = ceil(n_max / 64) 64-bit words.
 *   - The return value reports errors visible on the host (bad scalar
 *     arguments, NULL pointers, unsupported sizes, launch failures); on such
 *     an error nothing is launched.  Errors that depend on device data are
 *     or-ed into the caller's int32 status[B] as SPEC_DEV_* bits; no kernel
 *     traps or asserts.
 *   - Paged KV cache: k_cache and v_cache are [num_blocks][Hkv][block_size][D]
 *     elements of `dtype`; slot s of request b lives in block
 *     block_table[b * max_blocks + s / block_size], row s % block_size.  Slots
 *     [0, prefix_len[b]) hold the committed prefix and slots
 *     prefix_len[b] + v hold tree node v (already written by the caller).
 */
#ifndef SPECTREE_H
#define SPECTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t spec_status;

/* Host-visible status codes (return values). */
#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG 1 /* NULL pointer, negative size, Hq not a multiple of Hkv, ... */
#define SPEC_ERR_UNSUPPORTED 2 /* D not 64/128, n_max > 1024, V > 131072, block_size not a power of two in [8, 65536] */
#define SPEC_ERR_CUDA 3        /* a CUDA launch or attribute call failed */
#define SPEC_ERR_WORKSPACE 4   /* workspace smaller than the matching *_workspace_size() */

/* Per-request device status bits, or-ed into status[b]. */
#define SPEC_DEV_BAD_TREE 1   /* parent[0] != -1, parent[i] outside [0, i), n_b < 0 or n_b > n_max */
#define SPEC_DEV_BAD_TOKEN 2  /* a node token outside [0, V) */
#define SPEC_DEV_CAPACITY 4   /* prefix_len < 0, prefix_len > max_prefix, or prefix_len + n_b beyond the block table */
#define SPEC_DEV_TIMEOUT 8    /* a bounded device wait expired (the kernel returned early) */
#define SPEC_DEV_BAD_BLOCK 16 /* a block-table entry outside [0, num_blocks) */
#define SPEC_DEV_BAD_PATH 32  /* a commit path that is not strictly increasing from node 0 */
#define SPEC_DEV_BAD_TEMP 64  /* stochastic verify: an inverse temperature that is not finite and positive */

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* spec_tree_attention flags */
/* SPEC_ATTN_AUTO: the tcgen05 tensor-core path for every bf16 call (a KV group
 * with fewer than 128 query rows runs in a zero-padded 128-row tile: the path
 * is bound by the K/V stream, and on GB300 the padded tile streams K/V at
 * 5.3 TB/s for 36-row groups where the CUDA-core kernel reaches 0.22 TB/s);
 * the CUDA-core path for fp32. */
#define SPEC_ATTN_AUTO 0u
#define SPEC_ATTN_CUDA_CORE 1u  /* force the CUDA-core path */
#define SPEC_ATTN_TCGEN05 2u    /* force the tcgen05 path (bf16 only) */

/* Library version, (major << 16) | minor. */
int spec_version(void);

/* Human-readable name of a return code (SPEC_OK, SPEC_ERR_*). */
const char* spec_status_string(spec_status s);

/* Human-readable name of one device status bit (SPEC_DEV_*); "unknown status
 * bit" for anything else (0, several bits, or an undefined bit). */
const char* spec_dev_status_string(int32_t bit);

/*
 * Topology mask build.  "SpecInfer Guide", "The Topology-Aware 2D Causal Mask":
 * M[u][v] = 0 if v is u or an ancestor of u, else -inf; here packed as bits.
 *   parent   int32 [T]     local parent index per node (-1 at the root)
 *   tree_off int32 [B+1]   request offsets into the node arrays
 *   mask     uint64 [T][W] out: bit v of word v/64 of row u set iff v is u or an ancestor of u
 *   depth    int32 [T]     out: number of ancestors of the node (root 0)
 *   status   int32 [B]     out: WRITTEN (not or-ed): 0, or SPEC_DEV_BAD_TREE; this call
 *                          starts a verification pass.  A bad request gets all-zero mask
 *                          rows and depth -1.
 */
spec_status spec_tree_mask_build(const int32_t* parent, const int32_t* tree_off, int B, int n_max,
                                 uint64_t* mask, int32_t* depth, int32_t* status, void* stream);

/* Bytes of workspace spec_tree_attention needs for this shape (T = tree_off[B],
 * max_prefix = the largest prefix_len the call may see). */
size_t spec_attention_workspace_size(int B, int T, int n_max, int max_prefix, int Hq, int Hkv, int D);

/*
 * Tree attention.  "SpecInfer Guide", "Generalizing Attention to Tree
 * Topologies" and "Depth-First Flattening and KV Cache Reuse": for request b,
 * node u and query head h, out = sum_k softmax_k(scale * q . K_k) V_k over the
 * keys k in slots [0, prefix_len[b]) (the committed prefix) and slots
 * prefix_len[b] + v for every v with mask bit v of row u set (the node and
 * its ancestors).  Query head h reads kv-head h / (Hq / Hkv).  fp32
 * accumulation; bf16 inputs give bf16 output.
 *   q        [T][Hq][D] dtype   queries (positions already applied; RoPE position = prefix + depth)
 *   k_cache, v_cache            paged cache, see the conventions above
 *   block_table int32 [B][max_blocks]
 *   prefix_len  int32 [B]       committed prefix length per request (<= max_prefix)
 *   mask        from spec_tree_mask_build
 *   out      [T][Hq][D] dtype   out
 *   workspace   device scratch of spec_attention_workspace_size() bytes
 *   status   int32 [B]          in/out: or-ed with SPEC_DEV_CAPACITY / SPEC_DEV_BAD_BLOCK.
 *                               A flagged request's output rows are unspecified (the
 *                               CUDA-core path skips requests whose status is non-zero on
 *                               entry; the tcgen05 path computes them).
 *   flags       SPEC_ATTN_*
 * The tcgen05 kernel is launched as a programmatic dependent of the previous
 * kernel in the stream: its set-up and K/V loads may overlap that kernel (the
 * mask build allows this at its start), and it reads the mask and the status
 * word, writes the status word, and loads any key tile that reaches the
 * tree's own slots (prefix_len[b] and on) only after waiting for that kernel
 * to finish; the grid does not complete before that kernel.  The tree K/V
 * rows may therefore be written by the kernel right before this call
 * (spec_kv_append).  A kernel that allows programmatic dependents and sits
 * right before this call must not write q, the prefix slots of the caches,
 * block_table, prefix_len or tree_off; kernels that do not allow it (the
 * usual case) are waited for in full, as with any launch.
 */
spec_status spec_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                                const int32_t* prefix_len, const int32_t* tree_off, const uint64_t* mask,
                                int B, int T, int n_max, int max_prefix, int Hq, int Hkv, int D,
                                spec_dtype dtype, float scale, void* out,
                                void* workspace, size_t workspace_bytes, int32_t* status,
                                uint32_t flags, void* stream);

/*
 * spec_tree_attention without a workspace argument (the pages have no
 * counterpart of this call).  Some callers cannot allocate device memory where
 * they run attention: a host framework that passes the library only the
 * tensors it owns, or a serving loop whose graphs are captured once and must
 * not pay cudaMalloc's device-wide synchronisation per shape.  When the plan
 * splits a long key range over several CTAs (long prefixes, few requests), the
 * splits' partial outputs need scratch; this call keeps it in one fixed
 * file-scope device array of SPEC_ATTN_NOALLOC_BYTES, which every GPU that
 * loads the library holds until the process exits.  It calls no allocator.
 *   Limit: the plan's scratch for this shape, dtype and flags (at most
 *   spec_attention_workspace_size()) must fit in SPEC_ATTN_NOALLOC_BYTES;
 *   otherwise SPEC_ERR_UNSUPPORTED and nothing is launched.
 *   Set-up: the first call on each device looks up the array's device address
 *   with that device current; make that first call before any stream capture.
 *   The address is cached per device together with the current context: after
 *   a reset of the device's primary context (cudaDeviceReset) the next call
 *   looks it up again, so that call too belongs before any capture.  A failed
 *   lookup returns SPEC_ERR_CUDA and leaves no pending runtime error.
 *   Sharing: every call uses the same array, which keeps the last call's
 *   contents.  Nothing in it must start at zero (a call writes every partial
 *   it reads back), but calls whose kernels overlap on the GPU race: serialise
 *   them (one stream per device).
 *   Other arguments, outputs and statuses as in spec_tree_attention.
 */
#define SPEC_ATTN_NOALLOC_BYTES (16u << 20)
spec_status spec_tree_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                                        const int32_t* prefix_len, const int32_t* tree_off, const uint64_t* mask,
                                        int B, int T, int n_max, int max_prefix, int Hq, int Hkv, int D,
                                        spec_dtype dtype, float scale, void* out, int32_t* status, uint32_t flags,
                                        void* stream);

/* Bytes of workspace the verifiers take (a small constant: the walk keeps no
 * state in global memory; the argument stays so that callers need not change
 * when a variant needs scratch). */
size_t spec_verify_workspace_size(int B, int n_max, int V);

/*
 * Greedy token-tree verification.  "SpecInfer Guide", "Greedy Verification
 * Algorithm": starting at the root, descend into the child whose token equals
 * argmax of the current node's target logits; when none matches, emit that
 * argmax and stop.  p_logits[t] is the target's next-token logits after node
 * t's sequence, so child c is tested against argmax(p_logits[parent c]).
 * The accepted node f is the deepest node whose whole root path follows the
 * argmax chain (ties between equally deep nodes: lowest node index; with
 * distinct sibling tokens this is the walk above).  argmax ties go to the
 * lowest token id.  Logits must be finite.  One thread-block cluster per
 * request walks the tree level by level; only rows of nodes on matching
 * paths are read.
 *   p_logits   float [T][V]
 *   tokens     int32 [T]       draft token of each node (the root's is not used for matching)
 *   parent, tree_off           as for spec_tree_mask_build
 *   path       int32 [B][n_max] out: accepted nodes root first (local indices), then -1
 *   accept_len int32 [B]       out: number of accepted nodes including the root
 *   emitted    int32 [B][n_max] out: tokens of path[1..] then the correction / bonus token, then -1
 *   n_emitted  int32 [B]       out: = accept_len
 *   workspace  device memory of at least spec_verify_workspace_size() bytes (not read or written)
 *   status     int32 [B]       in/out: a request whose incoming status is non-zero is skipped;
 *                              otherwise or-ed with SPEC_DEV_BAD_TREE (invalid parent array or
 *                              n_b outside [0, n_max]) and SPEC_DEV_BAD_TOKEN; a request whose
 *                              status is non-zero after the call has accept_len = n_emitted = 0
 *                              and -1 rows.
 * Both verifiers are launched as programmatic dependents of the previous
 * kernel in the stream (tree attention lets them launch once its CTAs have
 * issued their last MMA): their prologue (input checks, the root row's
 * copy) may overlap that kernel, and they read the status word only after
 * waiting for it to finish.  A kernel that allows programmatic dependents and
 * sits right before a verify call must therefore not write p_logits,
 * q_probs, tokens, parent, tree_off, uniforms or inv_temperature; kernels
 * that do not allow it are waited for in full.
 */
spec_status spec_tree_verify_greedy(const float* p_logits, const int32_t* tokens, const int32_t* parent,
                                    const int32_t* tree_off, int B, int n_max, int V,
                                    int32_t* path, int32_t* accept_len, int32_t* emitted, int32_t* n_emitted,
                                    void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Stochastic token-tree verification (multi-step speculative sampling over a
 * tree).  "SpecInfer Guide", "Stochastic Verification Algorithm" with the
 * rule of "Inference Optimization Techniques" ("Misconception" section):
 * a draft token x is accepted with probability min(1, p(x)/q(x)); after a
 * rejection the target becomes norm(max(p - q, 0)).  The children of a node
 * are tried in increasing node index, each against the residual left by the
 * siblings rejected before it; the first accepted child becomes the current
 * node.  When every child is rejected, a token is sampled from the last
 * residual; at a leaf, the bonus token is sampled from p.  The emitted tokens
 * follow the target distribution when each node's children were drawn
 * i.i.d. from q_probs of that node (SPEC_Q_PER_PARENT), or each child
 * independently from its own row (SPEC_Q_PER_CHILD: "Merge-Based Tree
 * Construction", siblings proposed by different draft models; child c is
 * tested against, and on rejection subtracted as, row c).  Sampling at
 * temperature T > 0 ("Stochastic Verification Algorithm"): the target is
 * softmax(p_logits / T), given as the inverse temperature tau = 1/T per
 * request; q_probs are the draft's probabilities as drawn (its own
 * temperature already applied).
 * Arithmetic (fixed so that every decision is reproducible bit for bit):
 * p = softmax(tau * p_logits) with e = E(fp32(fp32(l - max l) * tau)), E
 * the library's own fp32 exp (x <= 0: Cody-Waite reduction, degree-7 Taylor
 * polynomial), normalisers as exact fixed-point sums of trunc(v * 2^46);
 * accept iff u * q(t) <= r(t) with u = (word0 >> 8) * 2^-24; terminal
 * sample = smallest x whose fixed-point prefix sum exceeds
 * floor(word1 * S / 2^32).
 *   q_probs          float [T][V]  SPEC_Q_PER_PARENT: row u is the draft distribution the
 *                                  children of u were drawn from; SPEC_Q_PER_CHILD: row c is
 *                                  the distribution node c was drawn from (row 0 unused)
 *   uniforms         uint32 [T][2] raw random words: [t][0] acceptance word of node t,
 *                                  [t][1] sampling word used if the walk stops at node t
 *   inv_temperature  float [B]     tau of each request, or NULL for tau = 1 (device memory).
 *                                  A tau that is not finite and positive sets
 *                                  SPEC_DEV_BAD_TEMP; the request is skipped.
 *   q_layout         SPEC_Q_PER_PARENT or SPEC_Q_PER_CHILD (else SPEC_ERR_INVALID_ARG)
 *   other arguments as in spec_tree_verify_greedy.  One cluster per request
 *   follows the walk: a node's target row is read when the walk reaches it,
 *   a draft row when a child is rejected against it.
 */
#define SPEC_Q_PER_PARENT 0
#define SPEC_Q_PER_CHILD 1
spec_status spec_tree_verify_stochastic(const float* p_logits, const float* q_probs, const int32_t* tokens,
                                        const int32_t* parent, const int32_t* tree_off, const uint32_t* uniforms,
                                        const float* inv_temperature, int q_layout, int B, int n_max, int V,
                                        int32_t* path, int32_t* accept_len, int32_t* emitted, int32_t* n_emitted,
                                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Tree K/V append.  "SpecInfer Guide", "Depth-First Flattening and KV Cache
 * Reuse", step 1 of the verification pass: every tree token appends the key
 * and value the target model computed for it to the active cache, in the
 * tree's node order, right after the committed prefix.  Row h of node u of
 * request b, k_new[tree_off[b] + u][h][0..D-1] (likewise v_new), is written
 * to slot prefix_len[b] + u of kv-head h through the block table; no other
 * slot changes.  This is how the tree K/V reach the slots that
 * spec_tree_attention reads.
 *   k_new, v_new  [T][Hkv][D] dtype, T = tree_off[B]; 16-byte aligned, as are the caches
 *                 (else SPEC_ERR_INVALID_ARG)
 *   k_cache, v_cache, block_table, max_blocks, block_size, num_blocks  as for attention
 *   prefix_len, tree_off  int32 [B], [B+1]
 *   status   int32 [B] in/out, or-ed with SPEC_DEV_BAD_TREE (n_b outside [0, n_max]),
 *            SPEC_DEV_CAPACITY (prefix_len < 0, or prefix_len + n_b beyond the block table)
 *            or SPEC_DEV_BAD_BLOCK (an id outside [0, num_blocks) among the pages of slots
 *            [prefix_len, prefix_len + n_b)); such a request is left untouched.  The
 *            incoming status is not read: an upstream failure does not stop the append.
 * Launched as a programmatic dependent of the previous kernel (the mask build
 * allows it at its start): the copies may overlap that kernel, which must not
 * write k_new, v_new or the tree slots; the status update and the end of the
 * grid wait for it.  One launch, grid (B, parts).
 */
spec_status spec_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           const int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                           const int32_t* prefix_len, const int32_t* tree_off, int B, int n_max, int Hkv, int D,
                           spec_dtype dtype, int32_t* status, void* stream);

/*
 * KV commit / rollback.  "SpecInfer Guide", "Depth-First Flattening and KV
 * Cache Reuse" and "PagedKV Allocation with Zero-Copy Pruning": only the
 * accepted path stays.  In place, for every kv-head: slot prefix_len[b] + i
 * receives the old slot prefix_len[b] + path[b][i], i < accept_len[b] (rows
 * already in place are not copied); new_len[b] = prefix_len[b] + accept_len[b].
 * Requests with a non-zero status on entry, or accept_len 0, are untouched
 * (new_len = prefix_len).  A path that is not strictly increasing from 0 or
 * leaves the block table sets SPEC_DEV_BAD_PATH; a bad block id sets
 * SPEC_DEV_BAD_BLOCK; such requests are untouched.
 *   path        int32 [B][path_stride]  accepted local node indices, root first
 *   accept_len  int32 [B]
 *   new_len     int32 [B] out
 *   status      int32 [B] in/out (or-ed)
 */
spec_status spec_kv_commit(void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks,
                           int block_size, int num_blocks, const int32_t* prefix_len, const int32_t* path,
                           int path_stride, const int32_t* accept_len, int B, int Hkv, int D, spec_dtype dtype,
                           int32_t* new_len, int32_t* status, void* stream);

/*
 * Multi-layer KV commit and page release.  "SpecInfer Guide", "PagedKV
 * Allocation with Zero-Copy Pruning": after verification the accepted path is
 * compacted in every layer's cache (each layer exactly as spec_kv_commit
 * does, in one launch), then the tree's pages lying wholly past the new length
 * go back to the free pool in one metadata update.  The tree of request b
 * fills slots [prefix_len[b], prefix_len[b] + n_b); its pages
 * ceil(new_len / block_size) .. ceil((prefix_len + n_b) / block_size) - 1 are
 * released: their block-table entries become -1 and their ids are appended to
 * free_pool after *free_count, in request order then page order, and
 * *free_count grows by their number.  The entries are taken as the table
 * holds them (call once per pass: a second call over the same tree would
 * append the -1 entries the first left).  Requests with a non-zero status after
 * the commit keep every page.  When the pool cannot take every page of the
 * call (*free_count + released > free_cap), none is released and each request
 * that had pages to release gets SPEC_DEV_CAPACITY.
 *   k_caches, v_caches  device arrays of `layers` device pointers, each a paged
 *                       cache [num_blocks][Hkv][block_size][D] of dtype
 *   block_table int32 [B][max_blocks]  in/out (released entries become -1)
 *   tree_off    int32 [B+1]  tree sizes (as for the mask build)
 *   free_pool   int32 [free_cap], free_count int32 [1]: device memory, in/out;
 *               both NULL: commit only, no release
 *   other arguments as in spec_kv_commit.  Two kernels: the commit (grid
 *   B x Hkv x Z, each CTA moving the rows of every Z-th cache, Z chosen to
 *   fill the GPU about once), then the release (one CTA).
 */
spec_status spec_kv_commit_layers(void* const* k_caches, void* const* v_caches, int layers,
                                  int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                                  const int32_t* prefix_len, const int32_t* tree_off, const int32_t* path,
                                  int path_stride, const int32_t* accept_len, int B, int Hkv, int D,
                                  spec_dtype dtype, int32_t* new_len, int32_t* free_pool, int free_cap,
                                  int32_t* free_count, int32_t* status, void* stream);

/*
 * Philox4x32-10 random words for one verification round (Salmon et al.,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11): node u (local index)
 * of request b uses counter (u, b, round, 0) and key (seed low 32 bits, seed
 * high 32 bits); out[t][0] = output word 0, out[t][1] = output word 1.
 *   tree_off int32 [B+1]; out uint32 [T][2]; n_max bounds n_b (larger requests are skipped).
 */
spec_status spec_philox_uniforms(uint64_t seed, uint32_t round, const int32_t* tree_off, int B, int n_max,
                                 uint32_t* out, void* stream);

/*
 * Token-tree construction ("SpecInfer Guide", "Token Tree Construction:
 * Expansion vs. Merge").  The trees come out in the layout the calls above
 * take (parent before child, packed by tree_off).
 *
 * spec_tree_init: request b's tree occupies n_total slots from b * n_total;
 * node 0 gets parent -1 and token root_tok[b] (the last verified token), and
 * tree_off[b] = b * n_total for b = 0..B (tree_off may be NULL).
 *   root_tok int32 [B]; tree_off int32 [B+1] out; parent, tokens int32 [B * n_total] out.
 *   n_total in [1, 1024].
 *
 * spec_tree_expand_level: one level of "Method A: Expansion-Based Tree
 * Construction": every frontier node gets its top-k tokens as children.
 * Every request has the same shape; its F frontier nodes are level_start ..
 * level_start + F - 1 and their children are appended after them, frontier
 * node by frontier node, each node's k children in rank order: child r of
 * frontier node i is node level_start + F + i * k + r, with parent
 * level_start + i.  Rank order: larger score first, equal scores by lower
 * token id, NaN after every number, -0 equal to +0.  A whole schedule
 * <k_1, ..., k_m> is spec_tree_init, then one call per level (level_start
 * 0, 1, 1 + k_1, ...), with the draft model's rows for the new frontier in
 * between.
 *   scores   float [B * F][V]  row b * F + i: draft scores (logits or probabilities)
 *                              of frontier node i of request b
 *   parent, tokens  int32 [B * n_total]  in/out: the level's children are written
 *   k in [0, 32], k <= V; level_start + F + F * k <= n_total <= 1024, else an error
 *   code and nothing is launched.
 *
 * spec_tree_merge: "Method B: Merge-Based Tree Construction": request b's
 * M candidate sequences (one per draft model: sequence s is
 * seqs[b][s][0 .. lens[b][s]-1]) are united into one tree in which every
 * prefix of every sequence is one node and no two nodes share a token path.
 * Node 0 is the root (root_tok[b]); the others are numbered in
 * first-appearance order (sequences in order, each from its first token).
 * The output is packed: tree_off is written (tree_off[0] = 0), request b's
 * nodes are tree_off[b] .. tree_off[b+1]-1.
 *   seqs     int32 [B][M][m]   candidate tokens (entries past a length are ignored)
 *   lens     int32 [B][M]      sequence lengths in [0, m]
 *   tree_off int32 [B+1] out
 *   parent, tokens int32 [B * (1 + M * m)] out (capacity; tree_off[B] entries written)
 *   src      int32 [same]  out: s * m + j of the prefix that created each node, -1 for roots
 *   node_of  int32 [B][M][m] out: the node (request-local index) of prefix (s, j), -1 past
 *                              the length; with it per-child draft rows can be gathered
 *   status   int32 [B]     out: WRITTEN (a merge starts a pass): 0, SPEC_DEV_BAD_TREE (a
 *                              length outside [0, m]) and/or SPEC_DEV_BAD_TOKEN (a token or
 *                              root token outside [0, V)); such a request gets only its root.
 *   M * m <= 1023 and M <= 1023.  Three launches (counts, offsets, nodes).
 */
spec_status spec_tree_init(const int32_t* root_tok, int B, int n_total, int32_t* tree_off, int32_t* parent,
                           int32_t* tokens, void* stream);
spec_status spec_tree_expand_level(const float* scores, int B, int F, int V, int k, int level_start, int n_total,
                                   int32_t* parent, int32_t* tokens, void* stream);
spec_status spec_tree_merge(const int32_t* seqs, const int32_t* lens, const int32_t* root_tok, int B, int M, int m,
                            int V, int32_t* tree_off, int32_t* parent, int32_t* tokens, int32_t* src,
                            int32_t* node_of, int32_t* status, void* stream);

/*
 * Dynamic draft length ("Hardware-aware dynamic speculative decoding",
 * "Dynamic speculative decoding" and "Compatibility with full CUDA Graph"):
 * the scheduler picks, per step, the number of draft tokens K of highest
 * goodput = AL / ITL (acceptance length over inter-token latency) for the
 * current batch size, from a table profiled offline and refreshed with live
 * statistics, and replays the full CUDA graph captured for <tokens, K>.
 * HOST functions: every pointer is host memory; nothing is launched.
 *
 * spec_dsd_optimal_k: al, itl double [n_bs][n_k] (measured AL and ITL for the
 *   draft lengths k_values[0..n_k-1] at each profiled batch size); a cell
 *   counts when both are finite and itl > 0.  k_opt int32 [n_bs] out: the K
 *   of the largest goodput in each row, the earliest column on ties; -1 when
 *   no cell of the row counts.
 * spec_dsd_select_k: bs_table int32 [n] strictly ascending (else
 *   SPEC_ERR_INVALID_ARG), k_table int32 [n]; *k_out = the entry of the
 *   largest bs_table[i] <= bs, or k_table[0] when bs < bs_table[0].
 * spec_dsd_update: folds one live measurement into cell (bs_index, k_index):
 *   x <- x + weight * (sample - x), weight in (0, 1]; a cell that is not
 *   finite (unmeasured) takes the sample.  Samples must be finite.
 * spec_dsd_graph_keys: every <tokens, K> with 1 <= tokens <= max_tokens and
 *   1 <= K <= max_k such that tokens is divisible by K + 1 (every request of
 *   the batch is then a decode request with K drafts), ordered by tokens
 *   then K.  *count = their number; the first min(cap, count) are stored.
 */
spec_status spec_dsd_optimal_k(const double* al, const double* itl, int n_bs, int n_k, const int32_t* k_values,
                               int32_t* k_opt);
spec_status spec_dsd_select_k(const int32_t* bs_table, const int32_t* k_table, int n, int bs, int32_t* k_out);
spec_status spec_dsd_update(double* al, double* itl, int n_bs, int n_k, int bs_index, int k_index, double al_sample,
                            double itl_sample, double weight);
spec_status spec_dsd_graph_keys(int max_tokens, int max_k, int32_t* tokens_out, int32_t* k_out, int cap,
                                int32_t* count);

/*
 * Diagnostic of the bounded device waits (no counterpart on the pages): one
 * small kernel waits on a barrier that nothing ever completes, with a limit of
 * `polls` polls (1 .. 2^20), the same wait the tensor-core attention roles use
 * with a limit of 2^25; on expiry it or-s SPEC_DEV_TIMEOUT into status[0] and
 * returns, leaving the context usable.
 */
spec_status spec_selftest_bounded_wait(int32_t* status, uint32_t polls, void* stream);

/*
 * Diagnostics of the stochastic verifier's arithmetic contract (no
 * counterpart on the pages).  They run the very device functions the
 * verifier uses (the exp E, the fixed-point weight FX and its two
 * accumulators, the residual step) over arrays, so that a test can compare
 * them bit for bit with an independent implementation of the contract
 * described at spec_tree_verify_stochastic.  Device pointers, asynchronous on
 * `stream`; SPEC_ERR_INVALID_ARG for a negative n, a bad segment or no output.
 *
 * spec_selftest_exp: x_i is the fp32 whose bit pattern is first_bits + i
 *   (modulo 2^32), i < n.  exp_scalar[i] = E(x_i) by the scalar routine;
 *   exp_pair[i] = E(x_i) by the two-lane routine, entries 2k and 2k+1 forming
 *   one pair.  Either output may be NULL.
 * spec_selftest_fx: v float [n] (the contract's domain is [0, 2)).
 *   fx_out[i] = trunc(v[i] * 2^46); for each of the n / seg segments of seg
 *   consecutive entries (1 <= seg <= 510, n a multiple of seg), seg_scalar[s]
 *   = the fixed-point sum of the segment by the scalar accumulator and
 *   seg_pair[s] = the same by the two-lane accumulator (seg even).  Any
 *   output may be NULL (not all three).
 * spec_selftest_resid: one residual step max(d / Z - q, 0) of the contract
 *   per entry i < n, with Z = Zp[i / 2] (Zp holds ceil(n / 2) normalisers;
 *   entries 2k and 2k+1 share one, as in the verifier's paired passes):
 *   r_div by IEEE division, r_markstein by the scalar Markstein sequence the
 *   residual passes use (y = RN(1/Z)), r_pair by its two-lane form.  Any
 *   output may be NULL (not all three).
 */
spec_status spec_selftest_exp(uint32_t first_bits, long long n, float* exp_scalar, float* exp_pair, void* stream);
spec_status spec_selftest_fx(const float* v, long long n, int seg, uint64_t* fx_out, uint64_t* seg_scalar,
                             uint64_t* seg_pair, void* stream);
spec_status spec_selftest_resid(const float* d, const float* q, const float* Zp, long long n, float* r_div,
                                float* r_markstein, float* r_pair, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECTREE_H */
