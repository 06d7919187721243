// KV commit / rollback: in-place compaction of the accepted root path.
//
// "SpecInfer Guide", "Depth-First Flattening and KV Cache Reuse": after
// verification only the accepted path stays in the cache.  The path is
// strictly increasing (parents precede children), so destination slot
// prefix + i never lies after source slot prefix + path[i]; moving rows in
// increasing i is safe provided every row of a chunk is read before any row
// of that chunk is written (a later chunk's sources are all above every
// earlier destination).  One CTA per (request, kv-head, K or V).
#include "common.cuh"

namespace spectree {

constexpr int kCommitThreads = 256;
constexpr int kCommitChunkBytes = 32 * 1024;

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(
    char* __restrict__ k_cache, char* __restrict__ v_cache, const int32_t* __restrict__ block_table, int max_blocks,
    int bs, int num_blocks, const int32_t* __restrict__ prefix_len, const int32_t* __restrict__ path, int path_stride,
    const int32_t* __restrict__ accept_len, int Hkv, int row_bytes, int32_t* __restrict__ new_len,
    int32_t* __restrict__ status) {
  __shared__ uint4 buf[kCommitChunkBytes / 16];
  __shared__ int s_bad;
  const int b = blockIdx.x, h = blockIdx.y;
  char* cache = blockIdx.z == 0 ? k_cache : v_cache;
  const bool writer = h == 0 && blockIdx.z == 0;
  const int P = prefix_len[b];
  const int a = accept_len[b];
  const int32_t* bt = block_table + (size_t)b * max_blocks;
  const int32_t* pth = path + (size_t)b * path_stride;
  const int st = *(volatile int32_t*)&status[b];
  if (st != 0 || a <= 0) {
    if (writer && threadIdx.x == 0) new_len[b] = P;
    return;
  }
  // validation (identical in every CTA of the request)
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
  if (bad) {
    if (writer && threadIdx.x == 0) {
      atomicOr(&status[b], bad);
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

}  // namespace spectree

using namespace spectree;

extern "C" spec_status spec_kv_commit(void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks,
                                      int block_size, int num_blocks, const int32_t* prefix_len, const int32_t* path,
                                      int path_stride, const int32_t* accept_len, int B, int Hkv, int D,
                                      spec_dtype dtype, int32_t* new_len, int32_t* status, void* stream) {
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
