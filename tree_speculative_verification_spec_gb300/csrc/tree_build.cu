// Token-tree construction on the device: one expansion level (top-k of every
// frontier node's draft row) and the merge of several drafts' candidate
// sequences into one tree ("SpecInfer Guide", "Token Tree Construction:
// Expansion vs. Merge").
#include <algorithm>

#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace spectree {

// ---------------------------------------------------------------------------
// Expansion
// ---------------------------------------------------------------------------

constexpr int kExpandThreads = 256;
constexpr int kExpandWarps = kExpandThreads / 32;

// Rank key of a draft score: larger is better.  High word: the float made
// orderable as an unsigned integer (-0 counted as +0, NaN below -inf); low
// word: the complement of the token id, so that equal scores rank the lower
// id first.  Keys of distinct tokens are distinct and all above 0.
__device__ __forceinline__ unsigned long long score_key(float v, int id) {
  uint32_t u = __float_as_uint(v);
  uint32_t k;
  if (v != v) {
    k = 0u;
  } else {
    if (u == 0x80000000u) u = 0u;
    k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  return ((unsigned long long)k << 32) | (unsigned long long)(~(uint32_t)id);
}

// The score of a key's high word: the bar below which no entry can enter a
// full list (-inf while the list has room or holds a NaN entry).
__device__ __forceinline__ float key_score(unsigned long long key) {
  const uint32_t k = (uint32_t)(key >> 32);
  if (k == 0u) return -INFINITY;
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// A warp's running top-k (k <= 32): lane r < k holds the r-th best key
// (descending), lanes >= k hold 0.  thr = the k-th best key (0 while there is
// room), bar = its score.
struct WarpTop {
  unsigned long long list = 0ull, thr = 0ull;
  float bar = -INFINITY;
  float floor = -INFINITY;  // a lower bound of the k-th best score, from a first sample

  // Lower bound for the bar from one sample per lane (its best score of a
  // first batch; NaN counted as -inf): the k-th largest of these 32 distinct
  // entries, by a bitonic sort across the warp.  No entry scored below it
  // can be among the k best.
  __device__ __forceinline__ void seed(float lane_best, int k, int lane) {
    float v = lane_best != lane_best ? -INFINITY : lane_best;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, stride);
        const bool desc = ((lane & size) == 0) == ((lane & stride) == 0);  // keep the larger in the lower lane
        v = desc ? fmaxf(v, o) : fminf(v, o);
      }
    }
    floor = __shfl_sync(0xffffffffu, v, k - 1);
    bar = fmaxf(bar, floor);
  }

  // Inserts `key` (the same value in every lane) if it beats the k-th best.
  __device__ __forceinline__ void insert(unsigned long long key, int k, int lane) {
    if (key <= thr) return;  // warp-uniform
    const int pos = __popc(__ballot_sync(0xffffffffu, list > key));  // the greater keys are lanes 0 .. pos-1
    const unsigned long long up = __shfl_up_sync(0xffffffffu, list, 1);
    if (lane > pos) list = up;
    else if (lane == pos) list = key;
    if (lane >= k) list = 0ull;
    thr = __shfl_sync(0xffffffffu, list, k - 1);
    bar = fmaxf(key_score(thr), floor);
  }

  // Every lane offers one score (valid lanes only); called by the whole warp.
  __device__ __forceinline__ void offer(float v, int x, bool valid, int k, int lane) {
    unsigned m = __ballot_sync(0xffffffffu, valid && !(v < bar));
    while (m) {
      const int l = __ffs(m) - 1;
      m &= m - 1;
      insert(score_key(__shfl_sync(0xffffffffu, v, l), __shfl_sync(0xffffffffu, x, l)), k, lane);
    }
  }

  // Every lane offers one key (0 = nothing).
  __device__ __forceinline__ void offer_key(unsigned long long key, int k, int lane) {
    unsigned m = __ballot_sync(0xffffffffu, key > thr);
    while (m) {
      const int l = __ffs(m) - 1;
      m &= m - 1;
      insert(__shfl_sync(0xffffffffu, key, l), k, lane);
    }
  }
};

// One thread-block cluster per frontier row, each CTA on a contiguous chunk
// of it (chunk: a multiple of 4 entries).  Each warp keeps a running top-k
// spread over its lanes; a batch of loads costs one compare per entry against
// the warp's bar, and only batches holding an entry at or above the bar take
// the ballot-driven inserts.  Warp 0 then takes the other warps' lists, puts
// the CTA's list into the cluster leader's shared memory, and the leader's
// warp 0 takes the cluster's lists.  The row is read once, with 16-byte loads
// when it is aligned; the cluster width is chosen so that short frontiers
// still spread over the GPU.
constexpr int kExpandMaxCluster = 8;

__global__ void __launch_bounds__(kExpandThreads) tree_expand_kernel(const float* __restrict__ scores, int F, int V,
                                                                     int k, int level_start, int n_total, int vec,
                                                                     int chunk, int32_t* __restrict__ parent,
                                                                     int32_t* __restrict__ tokens) {
  __shared__ unsigned long long wres[kExpandWarps][32];
  __shared__ unsigned long long cres[kExpandMaxCluster][32];  // leader: the CTAs' lists
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  const long long row = blockIdx.x / C;
  const int b = (int)(row / F), i = (int)(row % F);
  const int x0 = min(V, rank * chunk), x1 = min(V, x0 + chunk);
  const float* src = scores + row * (long long)V;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  WarpTop top;
  bool seeded = false;
  if (vec) {
    constexpr int kBatch = 8;  // 16-byte loads per lane issued before any is used
    const float4* s4 = reinterpret_cast<const float4*>(src + x0);
    const int n4 = (x1 - x0) >> 2;  // x0 and x1 - x0 are multiples of 4 when V is
    // warps stride over batches of kBatch * 32 consecutive float4
    for (int j0 = w * kBatch * 32; j0 < n4; j0 += kExpandWarps * kBatch * 32) {
      float4 v[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int j = j0 + q * 32 + lane;
        v[q] = j < n4 ? __ldcs(s4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      if (!seeded) {  // the first batch bounds the bar from below (32 lanes >= k entries)
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < kBatch; ++q) mx = fmaxf(mx, fmaxf(fmaxf(v[q].x, v[q].y), fmaxf(v[q].z, v[q].w)));
        top.seed(mx, k, lane);
        seeded = true;
      }
      bool any = false;
#pragma unroll
      for (int q = 0; q < kBatch; ++q)
        any |= !(v[q].x < top.bar) | !(v[q].y < top.bar) | !(v[q].z < top.bar) | !(v[q].w < top.bar);
      if (__any_sync(0xffffffffu, any)) {
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int j = j0 + q * 32 + lane;
          const bool ok = j < n4;
          const int x = x0 + 4 * j;
          top.offer(v[q].x, x, ok, k, lane);
          top.offer(v[q].y, x + 1, ok, k, lane);
          top.offer(v[q].z, x + 2, ok, k, lane);
          top.offer(v[q].w, x + 3, ok, k, lane);
        }
      }
    }
  } else {
    for (int base = x0 + w * 32; base < x1; base += kExpandThreads) {
      const int x = base + lane;
      const bool ok = x < x1;
      top.offer(ok ? __ldcs(src + x) : 0.0f, x, ok, k, lane);
    }
  }
  wres[w][lane] = top.list;
  __syncthreads();
  if (w == 0) {
    for (int w2 = 1; w2 < kExpandWarps; ++w2) top.offer_key(wres[w2][lane], k, lane);
    *cluster.map_shared_rank(&cres[rank][lane], 0) = top.list;  // the CTA's list to the leader
  }
  cluster.sync();  // the lists have landed; no CTA touches another's memory after this
  if (rank == 0 && w == 0) {
    for (int r = 1; r < C; ++r) top.offer_key(cres[r][lane], k, lane);
    if (lane < k) {
      const long long c = (long long)b * n_total + level_start + F + i * k + lane;
      parent[c] = level_start + i;
      tokens[c] = (int32_t)(~(uint32_t)(top.list & 0xffffffffull));
    }
  }
}

cudaError_t launch_expand(const float* scores, long long rows, int C, int F, int V, int k, int level_start,
                          int n_total, int vec, int chunk, int32_t* parent, int32_t* tokens, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * C), 1, 1);
  cfg.blockDim = dim3(kExpandThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_expand_kernel, scores, F, V, k, level_start, n_total, vec, chunk, parent,
                            tokens);
}

__global__ void tree_init_kernel(const int32_t* __restrict__ root_tok, int B, int n_total,
                                 int32_t* __restrict__ tree_off, int32_t* __restrict__ parent,
                                 int32_t* __restrict__ tokens) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b > B) return;
  if (tree_off) tree_off[b] = b * n_total;
  if (b < B) {
    parent[(long long)b * n_total] = -1;
    tokens[(long long)b * n_total] = root_tok[b];
  }
}

// ---------------------------------------------------------------------------
// Merge
// ---------------------------------------------------------------------------

constexpr int kMergeThreads = 1024;

struct MergeShared {
  int32_t tok[SPEC_MAX_NODES];    // the request's candidate tokens, [s][j]
  int32_t first[SPEC_MAX_NODES];  // lowest sequence sharing prefix (s, j); -1 past the length
  int32_t idx[SPEC_MAX_NODES];    // node index of (s, j) when it creates a node
  int32_t len[SPEC_MAX_NODES];
  int32_t wtot[kMergeThreads / 32];
};

// Request b's merged tree.  A prefix (s, j) is the same node as (s', j) iff
// the two sequences share the node at j - 1 and the token at j; first[s][j]
// is the lowest such s' (a canonical representative), found level by level
// with one thread per pair of sequences.
// (s, j) creates a node iff first[s][j] == s, and the nodes are numbered in
// (s, j) order after the root.  Returns the node count; with `write`, stores
// the tree at `base` and node_of.  Every thread returns the same count.
__device__ int merge_request(MergeShared& sh, int b, const int32_t* __restrict__ seqs,
                             const int32_t* __restrict__ lens, const int32_t* __restrict__ root_tok, int M, int m,
                             int V, bool write, int base, int32_t* __restrict__ parent,
                             int32_t* __restrict__ tokens, int32_t* __restrict__ src, int32_t* __restrict__ node_of,
                             int32_t* __restrict__ status) {
  const int items = M * m;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int bad = 0;
  for (int s = threadIdx.x; s < M; s += kMergeThreads) {
    const int L = lens[(long long)b * M + s];
    sh.len[s] = L;
    if (L < 0 || L > m) bad |= SPEC_DEV_BAD_TREE;
  }
  __syncthreads();
  for (int it = threadIdx.x; it < items; it += kMergeThreads) {
    const int s = it / m, j = it % m;
    const int t = seqs[(long long)b * items + it];
    sh.tok[it] = t;
    const int L = sh.len[s];
    if (L >= 0 && L <= m && j < L && (t < 0 || t >= V)) bad |= SPEC_DEV_BAD_TOKEN;
  }
  const int rt = root_tok[b];
  if (threadIdx.x == 0 && (rt < 0 || rt >= V)) bad |= SPEC_DEV_BAD_TOKEN;
  const int bad_tree = __syncthreads_or(bad & SPEC_DEV_BAD_TREE) ? SPEC_DEV_BAD_TREE : 0;
  const int bad_tok = __syncthreads_or(bad & SPEC_DEV_BAD_TOKEN) ? SPEC_DEV_BAD_TOKEN : 0;
  const int st = bad_tree | bad_tok;
  if (write) {
    if (threadIdx.x == 0) {
      status[b] = st;
      parent[base] = -1;
      tokens[base] = rt;
      src[base] = -1;
    }
  }
  if (st) {
    if (write)
      for (int it = threadIdx.x; it < items; it += kMergeThreads) node_of[(long long)b * items + it] = -1;
    return 1;
  }
  // level by level: first[s][j] = s, lowered to the lowest matching s2 < s
  // over all pairs (s2, s) in parallel
  for (int j = 0; j < m; ++j) {
    for (int s = threadIdx.x; s < M; s += kMergeThreads) sh.first[s * m + j] = j < sh.len[s] ? s : -1;
    __syncthreads();
    for (int p = threadIdx.x; p < M * M; p += kMergeThreads) {
      const int s = p / M, s2 = p - s * M;
      if (s2 >= s || j >= sh.len[s] || j >= sh.len[s2]) continue;
      const int it = s * m + j, it2 = s2 * m + j;
      if (sh.tok[it2] == sh.tok[it] && (j == 0 || sh.first[it2 - 1] == sh.first[it - 1])) atomicMin(&sh.first[it], s2);
    }
    __syncthreads();
  }
  // node numbers: exclusive scan of the creating items in (s, j) order
  // (items <= 1023 < kMergeThreads: one item per thread)
  const int it = threadIdx.x;
  const bool is_new = it < items && sh.first[it] == it / m;
  const unsigned bal = __ballot_sync(0xffffffffu, is_new);
  if (lane == 0) sh.wtot[w] = __popc(bal);
  __syncthreads();
  int before = 0, total = 0;
  for (int q = 0; q < kMergeThreads / 32; ++q) {
    const int c = sh.wtot[q];
    before += q < w ? c : 0;
    total += c;
  }
  before += __popc(bal & ((1u << lane) - 1u));
  if (is_new) sh.idx[it] = 1 + before;
  __syncthreads();
  if (write && it < items) {
    const int s = it / m, j = it % m;
    const int f = sh.first[it];
    const int node = f >= 0 ? sh.idx[f * m + j] : -1;
    node_of[(long long)b * items + it] = node;
    if (is_new) {
      const int up = j > 0 ? sh.idx[sh.first[it - 1] * m + j - 1] : 0;
      parent[base + node] = up;
      tokens[base + node] = sh.tok[it];
      src[base + node] = s * m + j;
    }
  }
  return 1 + total;
}

__global__ void __launch_bounds__(kMergeThreads) tree_merge_count_kernel(
    const int32_t* __restrict__ seqs, const int32_t* __restrict__ lens, const int32_t* __restrict__ root_tok, int M,
    int m, int V, int32_t* __restrict__ tree_off) {
  __shared__ MergeShared sh;
  const int b = blockIdx.x;
  const int n = merge_request(sh, b, seqs, lens, root_tok, M, m, V, false, 0, nullptr, nullptr, nullptr, nullptr,
                              nullptr);
  if (threadIdx.x == 0) tree_off[b + 1] = n;
}

// tree_off[1..B] hold the counts; made an inclusive prefix sum in place, with
// tree_off[0] = 0.  One CTA, rounds of kMergeThreads.
__global__ void __launch_bounds__(kMergeThreads) tree_offsets_kernel(int B, int32_t* __restrict__ tree_off) {
  __shared__ int wtot[kMergeThreads / 32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    carry = 0;
    tree_off[0] = 0;
  }
  __syncthreads();
  for (int b0 = 0; b0 < B; b0 += kMergeThreads) {
    const int b = b0 + threadIdx.x;
    const int c = b < B ? tree_off[b + 1] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wtot[w] = incl;
    __syncthreads();
    int pre = carry;
    for (int q = 0; q < w; ++q) pre += wtot[q];
    if (b < B) tree_off[b + 1] = pre + incl;
    __syncthreads();
    if (threadIdx.x == kMergeThreads - 1) carry = pre + incl;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kMergeThreads) tree_merge_write_kernel(
    const int32_t* __restrict__ seqs, const int32_t* __restrict__ lens, const int32_t* __restrict__ root_tok, int M,
    int m, int V, const int32_t* __restrict__ tree_off, int32_t* __restrict__ parent, int32_t* __restrict__ tokens,
    int32_t* __restrict__ src, int32_t* __restrict__ node_of, int32_t* __restrict__ status) {
  __shared__ MergeShared sh;
  const int b = blockIdx.x;
  merge_request(sh, b, seqs, lens, root_tok, M, m, V, true, tree_off[b], parent, tokens, src, node_of, status);
}

}  // namespace spectree

using namespace spectree;

extern "C" {

spec_status spec_tree_init(const int32_t* root_tok, int B, int n_total, int32_t* tree_off, int32_t* parent,
                           int32_t* tokens, void* stream) {
  SPEC_NVTX_RANGE("spec_tree_init");
  if (B < 0 || n_total < 1) return SPEC_ERR_INVALID_ARG;
  if (n_total > SPEC_MAX_NODES || (long long)B * n_total >= (1LL << 31)) return SPEC_ERR_UNSUPPORTED;
  if (B == 0 && !tree_off) return SPEC_OK;
  if ((B > 0 && (!root_tok || !parent || !tokens))) return SPEC_ERR_INVALID_ARG;
  const int threads = 256;
  tree_init_kernel<<<(B + 1 + threads - 1) / threads, threads, 0, (cudaStream_t)stream>>>(root_tok, B, n_total,
                                                                                         tree_off, parent, tokens);
  SPEC_LAUNCH_CHECK();
  return SPEC_OK;
}

spec_status spec_tree_expand_level(const float* scores, int B, int F, int V, int k, int level_start, int n_total,
                                   int32_t* parent, int32_t* tokens, void* stream) {
  SPEC_NVTX_RANGE("spec_tree_expand_level");
  if (B < 0 || F < 0 || V <= 0 || k < 0 || level_start < 0 || n_total < 1) return SPEC_ERR_INVALID_ARG;
  if (k > 32 || k > V || n_total > SPEC_MAX_NODES || (long long)B * n_total >= (1LL << 31))
    return SPEC_ERR_UNSUPPORTED;
  if ((long long)level_start + F + (long long)F * k > n_total) return SPEC_ERR_INVALID_ARG;
  if (B == 0 || F == 0 || k == 0) return SPEC_OK;
  if (!scores || !parent || !tokens) return SPEC_ERR_INVALID_ARG;
  const long long rows = (long long)B * F;
  if (rows >= (1LL << 31)) return SPEC_ERR_UNSUPPORTED;
  const int vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0;
  // cluster width: about two CTAs per SM over the level, chunks of at least
  // 2048 entries
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return SPEC_ERR_CUDA;
  int C = 1;
  while (C < kExpandMaxCluster && rows * C < 2LL * sms && (V + 2 * C - 1) / (2 * C) >= 2048) C *= 2;
  const int chunk = (((V + C - 1) / C) + 3) & ~3;
  if (rows * C >= (1LL << 31)) return SPEC_ERR_UNSUPPORTED;
  cudaError_t e =
      launch_expand(scores, rows, C, F, V, k, level_start, n_total, vec, chunk, parent, tokens, (cudaStream_t)stream);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  SPEC_LAUNCH_CHECK();
  return SPEC_OK;
}

spec_status spec_tree_merge(const int32_t* seqs, const int32_t* lens, const int32_t* root_tok, int B, int M, int m,
                            int V, int32_t* tree_off, int32_t* parent, int32_t* tokens, int32_t* src,
                            int32_t* node_of, int32_t* status, void* stream) {
  SPEC_NVTX_RANGE("spec_tree_merge");
  if (B < 0 || M < 0 || m < 0 || V <= 0) return SPEC_ERR_INVALID_ARG;
  if (M >= SPEC_MAX_NODES || (long long)M * m >= SPEC_MAX_NODES || V > (1 << 30) ||
      (long long)B * (1 + (long long)M * m) >= (1LL << 31) || B > (1 << 24))
    return SPEC_ERR_UNSUPPORTED;
  if (!tree_off) return SPEC_ERR_INVALID_ARG;
  if (B > 0 && (!root_tok || !parent || !tokens || !src || !status || (M > 0 && !lens) ||
                (M * m > 0 && (!seqs || !node_of))))
    return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (B > 0) {
    tree_merge_count_kernel<<<B, kMergeThreads, 0, s>>>(seqs, lens, root_tok, M, m, V, tree_off);
    SPEC_LAUNCH_CHECK();
  }
  tree_offsets_kernel<<<1, kMergeThreads, 0, s>>>(B, tree_off);
  SPEC_LAUNCH_CHECK();
  if (B > 0) {
    tree_merge_write_kernel<<<B, kMergeThreads, 0, s>>>(seqs, lens, root_tok, M, m, V, tree_off, parent, tokens,
                                                         src, node_of, status);
    SPEC_LAUNCH_CHECK();
  }
  return SPEC_OK;
}

}  // extern "C"
