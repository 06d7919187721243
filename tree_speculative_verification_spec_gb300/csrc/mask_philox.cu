// Topology mask build and Philox4x32-10 random words, plus the small
// library-wide entry points (version, status strings).
#include "common.cuh"

namespace spectree {

// One CTA per request.  Validation first (so that the parent walk below is
// known to terminate), then one thread per node walks its parent chain and
// writes its ancestor-or-self bit row: bit v of word v/64 set iff v lies on
// the path from the root to u ("SpecInfer Guide", "The Topology-Aware 2D
// Causal Mask").  Ancestors are met in decreasing index order, so the words
// of a row are produced from the highest to the lowest.
__global__ void __launch_bounds__(256) mask_build_kernel(const int32_t* __restrict__ parent,
                                                         const int32_t* __restrict__ tree_off, int n_max, int W,
                                                         uint64_t* __restrict__ mask, int32_t* __restrict__ depth,
                                                         int32_t* __restrict__ status) {
  __shared__ int32_t par[SPEC_MAX_NODES];
  // the next kernel of the pass (attention) may start its set-up now; it
  // waits for this grid before it reads the mask or the status word
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  const int off = tree_off[b];
  const int n = tree_off[b + 1] - off;
  const bool size_ok = n >= 0 && n <= n_max;
  const int nn = size_ok ? n : 0;
  int bad = !size_ok;
  for (int u = threadIdx.x; u < nn; u += blockDim.x) {
    const int p = parent[off + u];
    par[u] = p;
    bad |= (u == 0) ? (p != -1) : (p < 0 || p >= u);
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) status[b] = bad ? SPEC_DEV_BAD_TREE : 0;
  if (bad) {
    // The rows of a bad request are cleared.
    for (int i = threadIdx.x; i < n * W; i += blockDim.x) mask[(size_t)off * W + i] = 0;
    for (int u = threadIdx.x; u < n; u += blockDim.x) depth[off + u] = -1;
    return;
  }
  for (int u = threadIdx.x; u < nn; u += blockDim.x) {
    uint64_t* row = mask + (size_t)(off + u) * W;
    for (int w = 0; w < W; ++w) row[w] = 0;
    int cur_w = u >> 6, d = -1;
    uint64_t acc = 0;
    for (int c = u; c != -1; c = par[c]) {
      const int w = c >> 6;
      if (w != cur_w) {
        row[cur_w] = acc;
        cur_w = w;
        acc = 0;
      }
      acc |= 1ull << (c & 63);
      ++d;
    }
    row[cur_w] = acc;
    depth[off + u] = d;
  }
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32
// multiplications by 0xD2511F53 / 0xCD9E8D57 with the key bumped by the Weyl
// increments 0x9E3779B9 / 0xBB67AE85 between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__global__ void philox_uniforms_kernel(uint32_t k0, uint32_t k1, uint32_t round, const int32_t* __restrict__ tree_off,
                                       int n_max, uint2* __restrict__ out) {
  const int b = blockIdx.y;
  const int off = tree_off[b];
  const int n = tree_off[b + 1] - off;
  if (n < 0 || n > n_max) return;
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < n; u += gridDim.x * blockDim.x) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)u, (uint32_t)b, round, 0u), k0, k1);
    out[off + u] = make_uint2(w.x, w.y);
  }
}

}  // namespace spectree

using namespace spectree;

extern "C" {

int spec_version(void) { return (0 << 16) | 1; }

const char* spec_status_string(spec_status s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported size or type";
    case SPEC_ERR_CUDA: return "CUDA launch failure";
    case SPEC_ERR_WORKSPACE: return "workspace too small";
    default: break;
  }
  return "unknown status";
}

const char* spec_dev_status_string(int32_t bit) {
  switch (bit) {
    case SPEC_DEV_BAD_TREE: return "bad tree";
    case SPEC_DEV_BAD_TOKEN: return "bad token";
    case SPEC_DEV_CAPACITY: return "prefix beyond capacity";
    case SPEC_DEV_TIMEOUT: return "device wait timed out";
    case SPEC_DEV_BAD_BLOCK: return "bad block id";
    case SPEC_DEV_BAD_PATH: return "bad commit path";
    case SPEC_DEV_BAD_TEMP: return "bad inverse temperature";
    default: break;
  }
  return "unknown status bit";
}

spec_status spec_tree_mask_build(const int32_t* parent, const int32_t* tree_off, int B, int n_max, uint64_t* mask,
                                 int32_t* depth, int32_t* status, void* stream) {
  SPEC_NVTX_RANGE("spec_tree_mask_build");
  if (B < 0 || n_max < 0) return SPEC_ERR_INVALID_ARG;
  if (n_max > SPEC_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!tree_off || !status || (n_max > 0 && (!parent || !mask || !depth))) return SPEC_ERR_INVALID_ARG;
  const int W = n_max > 0 ? (n_max + 63) / 64 : 1;
  mask_build_kernel<<<B, 256, 0, (cudaStream_t)stream>>>(parent, tree_off, n_max, W, mask, depth, status);
  SPEC_LAUNCH_CHECK();
  return SPEC_OK;
}

spec_status spec_philox_uniforms(uint64_t seed, uint32_t round, const int32_t* tree_off, int B, int n_max,
                                 uint32_t* out, void* stream) {
  SPEC_NVTX_RANGE("spec_philox_uniforms");
  if (B < 0 || n_max < 0) return SPEC_ERR_INVALID_ARG;
  if (B == 0 || n_max == 0) return SPEC_OK;
  if (!tree_off || !out) return SPEC_ERR_INVALID_ARG;
  if (B > 65535) return SPEC_ERR_UNSUPPORTED;
  const int threads = 128;
  dim3 grid((n_max + threads - 1) / threads, B);
  philox_uniforms_kernel<<<grid, threads, 0, (cudaStream_t)stream>>>((uint32_t)seed, (uint32_t)(seed >> 32), round,
                                                                     tree_off, n_max, (uint2*)out);
  SPEC_LAUNCH_CHECK();
  return SPEC_OK;
}

}  // extern "C"
