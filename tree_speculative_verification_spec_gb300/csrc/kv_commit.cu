// KV commit / rollback: in-place compaction of the accepted root path.
//
// "SpecInfer Guide", "Depth-First Flattening and KV Cache Reuse": after
// verification only the accepted path stays in the cache.  The path is
// strictly increasing (parents precede children), so destination slot
// prefix + i never lies after source slot prefix + path[i]; moving rows in
// increasing i is safe provided every row of a chunk is read before any row
// of that chunk is written (a later chunk's sources are all above every
// earlier destination).  One CTA per (request, kv-head, K or V).
#include <algorithm>

#include "common.cuh"

namespace spectree {

constexpr int kCommitThreads = 256;
constexpr int kCommitChunkBytes = 32 * 1024;

// Checks shared by both commit kernels (identical in every CTA of request
// b): 0 when the accepted rows are to be moved, -1 when there is nothing to
// move (the request failed upstream or accepted nothing), else the
// SPEC_DEV_* bit that describes a bad path or block table.
__device__ __forceinline__ int commit_check(int b, const int32_t* __restrict__ bt, int max_blocks, int bs,
                                            int num_blocks, int P, int a, const int32_t* __restrict__ pth,
                                            int path_stride, const int32_t* __restrict__ status) {
  __shared__ int s_bad, s_st;
  // one read, broadcast: the request's writer CTA may set a bit meanwhile,
  // and every thread of this CTA must take the same branch
  if (threadIdx.x == 0) s_st = *(volatile const int32_t*)&status[b];
  __syncthreads();
  if (s_st != 0 || a <= 0) return -1;
  int bad = 0;
  if (a > path_stride || P < 0) bad = SPEC_DEV_BAD_PATH;
  if (!bad) {
    for (int i = threadIdx.x; i < a; i += blockDim.x) {
      const int p = pth[i];
      if (i == 0 ? p != 0 : p <= pth[i - 1]) bad = SPEC_DEV_BAD_PATH;
    }
  }
  bad = __syncthreads_or(bad) ? SPEC_DEV_BAD_PATH : 0;
  long long last = 0;
  if (!bad) {
    last = (long long)P + pth[a - 1];  // highest slot touched
    if (last + 1 > (long long)max_blocks * bs) bad = SPEC_DEV_BAD_PATH;
  }
  if (!bad) {
    const int used = (int)((last + bs) / bs);
    int bb = 0;
    for (int i = threadIdx.x; i < used; i += blockDim.x) bb |= bt[i] < 0 || bt[i] >= num_blocks;
    bad = __syncthreads_or(bb) ? SPEC_DEV_BAD_BLOCK : 0;
  }
  if (threadIdx.x == 0) s_bad = bad;
  __syncthreads();
  bad = s_bad;
  __syncthreads();  // s_bad is read by every thread before a later call may write it
  return bad;
}

// One CTA's share of a commit: kv-head h of request b in one cache (K or V
// of one layer); `writer` CTAs set new_len and the status bits.
__device__ __forceinline__ void commit_rows(char* __restrict__ cache, bool writer, int b, int h,
                                            const int32_t* __restrict__ block_table, int max_blocks, int bs,
                                            int num_blocks, const int32_t* __restrict__ prefix_len,
                                            const int32_t* __restrict__ path, int path_stride,
                                            const int32_t* __restrict__ accept_len, int Hkv, int row_bytes,
                                            int32_t* __restrict__ new_len, int32_t* __restrict__ status) {
  __shared__ uint4 buf[kCommitChunkBytes / 16];
  const int P = prefix_len[b];
  const int a = accept_len[b];
  const int32_t* bt = block_table + (size_t)b * max_blocks;
  const int32_t* pth = path + (size_t)b * path_stride;
  const int bad = commit_check(b, bt, max_blocks, bs, num_blocks, P, a, pth, path_stride, status);
  if (bad != 0) {
    if (writer && threadIdx.x == 0) {
      if (bad > 0) atomicOr(&status[b], bad);
      new_len[b] = P;
    }
    return;
  }
  const int vec_per_row = row_bytes / 16;
  const int rows_per_chunk = kCommitChunkBytes / row_bytes;
  for (int i0 = 0; i0 < a; i0 += rows_per_chunk) {
    const int i1 = min(a, i0 + rows_per_chunk);
    for (int j = threadIdx.x; j < (i1 - i0) * vec_per_row; j += blockDim.x) {
      const int i = i0 + j / vec_per_row, c = j % vec_per_row;
      const int s = P + pth[i];
      if (pth[i] == i) continue;
      const char* src = cache + ((((size_t)bt[s / bs] * Hkv + h) * bs + s % bs) * row_bytes);
      buf[j] = reinterpret_cast<const uint4*>(src)[c];
    }
    __syncthreads();
    for (int j = threadIdx.x; j < (i1 - i0) * vec_per_row; j += blockDim.x) {
      const int i = i0 + j / vec_per_row, c = j % vec_per_row;
      if (pth[i] == i) continue;
      const int d = P + i;
      char* dst = cache + ((((size_t)bt[d / bs] * Hkv + h) * bs + d % bs) * row_bytes);
      reinterpret_cast<uint4*>(dst)[c] = buf[j];
    }
    __syncthreads();
  }
  if (writer && threadIdx.x == 0) new_len[b] = P + a;
}

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(
    char* __restrict__ k_cache, char* __restrict__ v_cache, const int32_t* __restrict__ block_table, int max_blocks,
    int bs, int num_blocks, const int32_t* __restrict__ prefix_len, const int32_t* __restrict__ path, int path_stride,
    const int32_t* __restrict__ accept_len, int Hkv, int row_bytes, int32_t* __restrict__ new_len,
    int32_t* __restrict__ status) {
  commit_rows(blockIdx.z == 0 ? k_cache : v_cache, blockIdx.y == 0 && blockIdx.z == 0, blockIdx.x, blockIdx.y,
              block_table, max_blocks, bs, num_blocks, prefix_len, path, path_stride, accept_len, Hkv, row_bytes,
              new_len, status);
}

// Every layer in one launch.  The caches are numbered c = 2 * layer (K) and
// 2 * layer + 1 (V); CTA (b, h, z) moves kv-head h of request b in caches z,
// z + Z, z + 2Z, ... (Z = gridDim.z, chosen so that the grid fills the GPU
// about once).  The accepted rows that actually move (path[i] != i) are listed
// once per CTA with their source and destination offsets, which every cache
// shares; then (cache, row, 16-byte vector) is flattened and staged through
// shared memory chunk by chunk, every read of a chunk before any write of it
// (in each cache a chunk's sources lie above every earlier destination, the
// same argument as for one cache).
constexpr int kLayerRowBatch = 1024;
constexpr int kLayerBufVec = 1536;  // 24 KB staging
__global__ void __launch_bounds__(kCommitThreads) kv_commit_layers_kernel(
    char* const* __restrict__ k_caches, char* const* __restrict__ v_caches, int n_caches,
    const int32_t* __restrict__ block_table, int max_blocks, int bs, int num_blocks,
    const int32_t* __restrict__ prefix_len, const int32_t* __restrict__ path, int path_stride,
    const int32_t* __restrict__ accept_len, int Hkv, int row_bytes, int32_t* __restrict__ new_len,
    int32_t* __restrict__ status) {
  __shared__ uint4 buf[kLayerBufVec];
  __shared__ long long s_src[kLayerRowBatch], s_dst[kLayerRowBatch];
  __shared__ int s_warp[kCommitThreads / 32];
  const int b = blockIdx.x, h = blockIdx.y, z = blockIdx.z, Z = gridDim.z;
  const bool writer = h == 0 && z == 0;
  const int P = prefix_len[b];
  const int a = accept_len[b];
  const int32_t* bt = block_table + (size_t)b * max_blocks;
  const int32_t* pth = path + (size_t)b * path_stride;
  const int bad = commit_check(b, bt, max_blocks, bs, num_blocks, P, a, pth, path_stride, status);
  if (bad != 0) {
    if (writer && threadIdx.x == 0) {
      if (bad > 0) atomicOr(&status[b], bad);
      new_len[b] = P;
    }
    return;
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nq = (n_caches - z + Z - 1) / Z;  // caches of this CTA
  const int vpr = row_bytes / 16;
  auto slot = [&](int s) -> long long { return (((long long)bt[s / bs] * Hkv + h) * bs + s % bs) * row_bytes; };
  auto cache_of = [&](int q) -> char* {
    const int c = z + q * Z;
    return (c & 1) ? v_caches[c >> 1] : k_caches[c >> 1];
  };
  constexpr int kPer = kLayerRowBatch / kCommitThreads;
  for (int r0 = 0; r0 < a; r0 += kLayerRowBatch) {
    const int r1 = min(a, r0 + kLayerRowBatch);
    // list the moving rows of [r0, r1) in increasing i
    const int i0 = r0 + threadIdx.x * kPer;
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) cnt += (i0 + e < r1 && pth[i0 + e] != i0 + e);
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[w] = incl;
    __syncthreads();
    int pos = 0, m = 0;
    for (int k = 0; k < kCommitThreads / 32; ++k) {
      pos += k < w ? s_warp[k] : 0;
      m += s_warp[k];
    }
    pos += incl - cnt;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = i0 + e;
      if (i < r1 && pth[i] != i) {
        s_src[pos] = slot(P + pth[i]);
        s_dst[pos] = slot(P + i);
        ++pos;
      }
    }
    __syncthreads();
    const long long per_cache = (long long)m * vpr;
    const long long total = per_cache * nq;
    for (long long j0 = 0; j0 < total; j0 += kLayerBufVec) {
      const int n = (int)min((long long)kLayerBufVec, total - j0);
      for (int t = threadIdx.x; t < n; t += kCommitThreads) {
        const long long j = j0 + t;
        const int q = (int)(j / per_cache);
        const int r = (int)(j - q * per_cache);
        buf[t] = reinterpret_cast<const uint4*>(cache_of(q) + s_src[r / vpr])[r % vpr];
      }
      __syncthreads();
      for (int t = threadIdx.x; t < n; t += kCommitThreads) {
        const long long j = j0 + t;
        const int q = (int)(j / per_cache);
        const int r = (int)(j - q * per_cache);
        reinterpret_cast<uint4*>(cache_of(q) + s_dst[r / vpr])[r % vpr] = buf[t];
      }
      __syncthreads();
    }
    // s_warp, s_src and s_dst are rewritten by the next batch: every thread has
    // read them (also when this batch moved no row and the copy loop was empty)
    __syncthreads();
  }
  if (writer && threadIdx.x == 0) new_len[b] = P + a;
}

// "SpecInfer Guide", "PagedKV Allocation with Zero-Copy Pruning": the pages
// of request b's tree lying wholly past its new length, ceil(new_len / bs) ..
// ceil((prefix + n) / bs) - 1, go back to the pool in one metadata update:
// block-table entries -1, ids appended after *free_count in request, then
// page order.  All or nothing: when the pool cannot take every page of the
// call, none is released and each request that had pages to release is
// flagged SPEC_DEV_CAPACITY.  Failed requests keep their pages.  One CTA.
constexpr int kReleaseThreads = 1024;
__global__ void __launch_bounds__(kReleaseThreads) kv_release_kernel(
    int32_t* __restrict__ block_table, int max_blocks, int bs, const int32_t* __restrict__ prefix_len,
    const int32_t* __restrict__ tree_off, const int32_t* __restrict__ new_len, int B, int32_t* __restrict__ free_pool,
    int free_cap, int32_t* __restrict__ free_count, int32_t* __restrict__ status) {
  __shared__ long long warp_tot[kReleaseThreads / 32];
  __shared__ long long base;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  auto pages = [&](int b, int& keep) -> int {  // pages request b releases
    if (status[b] != 0) return 0;
    const int n = tree_off[b + 1] - tree_off[b];
    keep = (new_len[b] + bs - 1) / bs;
    const int span = min(max_blocks, (prefix_len[b] + n + bs - 1) / bs);
    return span > keep ? span - keep : 0;
  };
  // the call's total
  long long t = 0;
  for (int b = threadIdx.x; b < B; b += kReleaseThreads) {
    int keep;
    t += pages(b, keep);
  }
  for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if (lane == 0) warp_tot[w] = t;
  __syncthreads();
  long long total = 0;
  for (int k = 0; k < kReleaseThreads / 32; ++k) total += warp_tot[k];
  const long long start = *free_count;
  if (start + total > free_cap) {
    for (int b = threadIdx.x; b < B; b += kReleaseThreads) {
      int keep;
      if (pages(b, keep) > 0) atomicOr(&status[b], SPEC_DEV_CAPACITY);
    }
    return;
  }
  // in request order: an exclusive scan per round of kReleaseThreads requests
  if (threadIdx.x == 0) base = start;
  __syncthreads();
  for (int b0 = 0; b0 < B; b0 += kReleaseThreads) {
    const int b = b0 + threadIdx.x;
    int keep = 0;
    const int c = b < B ? pages(b, keep) : 0;
    long long incl = c;
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncthreads();  // warp_tot and base of the previous round are read
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    long long wbase = base;
    for (int k = 0; k < w; ++k) wbase += warp_tot[k];
    const long long pos = wbase + incl - c;
    if (c > 0) {
      int32_t* row = block_table + (size_t)b * max_blocks;
      for (int i = 0; i < c; ++i) {
        free_pool[pos + i] = row[keep + i];
        row[keep + i] = -1;
      }
    }
    __syncthreads();
    if (threadIdx.x == kReleaseThreads - 1) base = wbase + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) *free_count = (int32_t)base;
}

// "SpecInfer Guide", "Depth-First Flattening and KV Cache Reuse", step 1 of
// the verification pass: the tree tokens' keys and values are appended to
// the active cache in node order after the prefix.  Row h of node u of
// request b (k_new[tree_off[b] + u][h], likewise v_new) goes to slot
// prefix_len[b] + u of kv-head h.  Grid (request, part): the parts of one
// request stride over its (node, head, 16-byte vector) triples, K and V in
// the same pass.  Every CTA checks its whole request first, so a bad request
// is left untouched by all of them.  The kernel may start before the previous
// kernel of the stream ends (programmatic dependent of the mask build): its
// copies read nothing that kernel writes, and its end waits for it.
constexpr int kAppendThreads = 256;
__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, char* __restrict__ k_cache,
    char* __restrict__ v_cache, const int32_t* __restrict__ block_table, int max_blocks, int bs, int num_blocks,
    const int32_t* __restrict__ prefix_len, const int32_t* __restrict__ tree_off, int n_max, int Hkv, int row_bytes,
    int32_t* __restrict__ status) {
  const int b = blockIdx.x;
  const int off = tree_off[b];
  const int n = tree_off[b + 1] - off;
  const int P = prefix_len[b];
  int bad = 0;
  if (n < 0 || n > n_max) bad = SPEC_DEV_BAD_TREE;
  else if (P < 0 || (long long)P + n > (long long)max_blocks * bs) bad = SPEC_DEV_CAPACITY;
  const int32_t* bt = block_table + (size_t)b * max_blocks;
  if (!bad && n > 0) {
    int bb = 0;
    for (int pg = P / bs + threadIdx.x; pg <= (P + n - 1) / bs; pg += blockDim.x) bb |= bt[pg] < 0 || bt[pg] >= num_blocks;
    if (__syncthreads_or(bb)) bad = SPEC_DEV_BAD_BLOCK;
  }
  if (!bad && n > 0) {
    const int vpr = row_bytes / 16;
    const long long per = (long long)n * Hkv * vpr;  // vectors of K (and of V)
    const long long step = (long long)gridDim.y * blockDim.x;
    for (long long j = (long long)blockIdx.y * blockDim.x + threadIdx.x; j < per; j += step) {
      const int u = (int)(j / ((long long)Hkv * vpr));
      const int rem = (int)(j - (long long)u * Hkv * vpr);
      const int h = rem / vpr, c = rem - h * vpr;
      const int s = P + u;
      const long long dst = (((long long)bt[s / bs] * Hkv + h) * bs + s % bs) * row_bytes + c * 16;
      const long long src = ((long long)(off + u) * Hkv + h) * vpr + c;
      const uint4 kv = __ldg(k_new + src), vv = __ldg(v_new + src);
      *reinterpret_cast<uint4*>(k_cache + dst) = kv;
      *reinterpret_cast<uint4*>(v_cache + dst) = vv;
    }
  }
  // Every CTA waits for the previous kernel before it exits, so this grid
  // completes only after that kernel has: a kernel launched after this one
  // (tree attention, which waits for its own predecessor before it reads the
  // mask) then also finds the mask build's results.  The status update
  // follows the mask build, which writes the status word.
  if (threadIdx.x == 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (bad && blockIdx.y == 0) atomicOr(&status[b], bad);
  }
}

}  // namespace spectree

using namespace spectree;

extern "C" spec_status spec_kv_commit(void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks,
                                      int block_size, int num_blocks, const int32_t* prefix_len, const int32_t* path,
                                      int path_stride, const int32_t* accept_len, int B, int Hkv, int D,
                                      spec_dtype dtype, int32_t* new_len, int32_t* status, void* stream) {
  SPEC_NVTX_RANGE("spec_kv_commit");
  if (B < 0 || Hkv <= 0 || max_blocks <= 0 || num_blocks <= 0 || path_stride <= 0) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  if (block_size < 8 || block_size > 65536 || (block_size & (block_size - 1))) return SPEC_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!k_cache || !v_cache || !block_table || !prefix_len || !path || !accept_len || !new_len || !status)
    return SPEC_ERR_INVALID_ARG;
  const int row_bytes = D * (dtype == SPEC_F32 ? 4 : 2);
  dim3 grid(B, Hkv, 2);
  kv_commit_kernel<<<grid, kCommitThreads, 0, (cudaStream_t)stream>>>(
      (char*)k_cache, (char*)v_cache, block_table, max_blocks, block_size, num_blocks, prefix_len, path, path_stride,
      accept_len, Hkv, row_bytes, new_len, status);
  SPEC_LAUNCH_CHECK();
  return SPEC_OK;
}

extern "C" spec_status spec_kv_commit_layers(void* const* k_caches, void* const* v_caches, int layers,
                                             int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                                             const int32_t* prefix_len, const int32_t* tree_off, const int32_t* path,
                                             int path_stride, const int32_t* accept_len, int B, int Hkv, int D,
                                             spec_dtype dtype, int32_t* new_len, int32_t* free_pool, int free_cap,
                                             int32_t* free_count, int32_t* status, void* stream) {
  SPEC_NVTX_RANGE("spec_kv_commit_layers");
  if (B < 0 || layers <= 0 || Hkv <= 0 || max_blocks <= 0 || num_blocks <= 0 || path_stride <= 0 || free_cap < 0)
    return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  if (block_size < 8 || block_size > 65536 || (block_size & (block_size - 1))) return SPEC_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535 || layers > 32767) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!k_caches || !v_caches || !block_table || !prefix_len || !path || !accept_len || !new_len || !status)
    return SPEC_ERR_INVALID_ARG;
  const bool release = free_pool != nullptr || free_count != nullptr;
  if (release && (!free_pool || !free_count || !tree_off)) return SPEC_ERR_INVALID_ARG;
  const int row_bytes = D * (dtype == SPEC_F32 ? 4 : 2);
  // about one wave: Z cache groups per (request, kv-head), at least one
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return SPEC_ERR_CUDA;
  const long long pairs = (long long)B * Hkv;
  const int n_caches = 2 * layers;
  const int Z = (int)std::min<long long>(n_caches, std::max<long long>(1, (4LL * sms + pairs - 1) / pairs));
  dim3 grid(B, Hkv, Z);
  spectree::kv_commit_layers_kernel<<<grid, spectree::kCommitThreads, 0, (cudaStream_t)stream>>>(
      (char* const*)k_caches, (char* const*)v_caches, n_caches, block_table, max_blocks, block_size, num_blocks,
      prefix_len, path, path_stride, accept_len, Hkv, row_bytes, new_len, status);
  SPEC_LAUNCH_CHECK();
  if (release) {
    spectree::kv_release_kernel<<<1, spectree::kReleaseThreads, 0, (cudaStream_t)stream>>>(
        block_table, max_blocks, block_size, prefix_len, tree_off, new_len, B, free_pool, free_cap, free_count,
        status);
    SPEC_LAUNCH_CHECK();
  }
  return SPEC_OK;
}

extern "C" spec_status spec_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                      const int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                                      const int32_t* prefix_len, const int32_t* tree_off, int B, int n_max, int Hkv,
                                      int D, spec_dtype dtype, int32_t* status, void* stream) {
  SPEC_NVTX_RANGE("spec_kv_append");
  if (B < 0 || n_max < 0 || Hkv <= 0 || max_blocks <= 0 || num_blocks <= 0) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  if (block_size < 8 || block_size > 65536 || (block_size & (block_size - 1))) return SPEC_ERR_UNSUPPORTED;
  if (n_max > SPEC_MAX_NODES || B > 65535 || Hkv > 65535) return SPEC_ERR_UNSUPPORTED;
  if (B == 0 || n_max == 0) return SPEC_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !prefix_len || !tree_off || !status)
    return SPEC_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
        reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15) != 0)
    return SPEC_ERR_INVALID_ARG;
  const int row_bytes = D * (dtype == SPEC_F32 ? 4 : 2);
  // about four CTAs' worth of 16-byte vectors per thread at the largest tree
  const long long per_req = (long long)n_max * Hkv * (row_bytes / 16);
  const int parts = (int)std::max(1LL, std::min(65535LL, (per_req + 4LL * kAppendThreads - 1) / (4LL * kAppendThreads)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B, parts, 1);
  cfg.blockDim = dim3(kAppendThreads, 1, 1);
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<const uint4*>(k_new),
                                           static_cast<const uint4*>(v_new), static_cast<char*>(k_cache),
                                           static_cast<char*>(v_cache), block_table, max_blocks, block_size,
                                           num_blocks, prefix_len, tree_off, n_max, Hkv, row_bytes, status);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}
