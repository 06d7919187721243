// Tree attention: CUDA-core path, split-KV combine, and the host entry point.
//
// "SpecInfer Guide", "Generalizing Attention to Tree Topologies": node u of
// request b attends to the committed prefix (slots [0, P_b)) and to the tree
// slots P_b + v of its ancestors-or-self (mask bit v of row u), with weights
// softmax(scale * q . k).  Work unit: (request, kv-head, 16-row tile, key
// split); rows of a kv-head group are (node, head-in-group) pairs, so the
// K/V tile staged in shared memory serves every query head of the group.
// Online softmax in the log2 domain; split-KV partials (unnormalised output,
// running max, running sum) are merged by attn_combine_kernel.
#include <cuda.h>

#include <mutex>

#include "attention.cuh"

#include <algorithm>

namespace spectree {

constexpr int kCcThreads = 128;
constexpr int kCcRows = 16;  // rows per CTA, 4 per warp
constexpr int kCcKeys = 32;  // keys per shared-memory tile

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T, int D>
__global__ void __launch_bounds__(kCcThreads) attn_cc_kernel(AttnArgs a) {
  constexpr int DJ = D / 32;  // output dims per lane
  __shared__ float Ks[kCcKeys][D + 1];
  __shared__ float Vs[kCcKeys][D];
  __shared__ float Qs[kCcRows][D];
  __shared__ int s_badblk;

  const int rt = blockIdx.x, split = blockIdx.y;
  const int b = blockIdx.z / a.Hkv, kvh = blockIdx.z % a.Hkv;
  const int off = a.tree_off[b];
  const int n = a.tree_off[b + 1] - off;
  const int P = a.prefix_len[b];
  const int g = a.g;
  const int rows = n * g;
  const int r0 = rt * kCcRows;
  if (n <= 0 || n > a.n_max || r0 >= rows || off < 0 || off + n > a.T) return;
  if (*(volatile int32_t*)&a.status[b] != 0) return;
  if (P < 0 || P > a.max_prefix || (long long)P + n > (long long)a.max_blocks * a.block_size) {
    if (threadIdx.x == 0 && rt == 0 && split == 0 && kvh == 0) atomicOr(&a.status[b], SPEC_DEV_CAPACITY);
    return;
  }
  const int L = P + n;
  const int k_begin = split * a.chunk;
  const int k_end = min(L, k_begin + a.chunk);
  if (k_begin >= k_end) return;

  const T* __restrict__ q = static_cast<const T*>(a.q);
  const T* __restrict__ kc = static_cast<const T*>(a.k_cache);
  const T* __restrict__ vc = static_cast<const T*>(a.v_cache);
  const int32_t* bt = a.block_table + (size_t)b * a.max_blocks;
  const int bs = a.block_size;

  // Q rows of this tile (fp32 in shared memory; rows past the group are zero)
  for (int i = threadIdx.x; i < kCcRows * D; i += blockDim.x) {
    const int lr = i / D, d = i % D, r = r0 + lr;
    float v = 0.0f;
    if (r < rows) {
      const int t = off + r / g, hh = kvh * g + r % g;
      v = to_f32(q[((size_t)t * a.Hq + hh) * D + d]);
    }
    Qs[lr][d] = v;
  }
  if (threadIdx.x == 0) s_badblk = 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m[4], l[4], o[4][DJ];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < DJ; ++j) o[i][j] = 0.0f;
  }

  constexpr int VEC = 16 / sizeof(T);  // elements per 16-byte load
  for (int k0 = k_begin; k0 < k_end; k0 += kCcKeys) {
    __syncthreads();
    for (int i = threadIdx.x; i < kCcKeys * (D / VEC); i += blockDim.x) {
      const int kk = i / (D / VEC), c = i % (D / VEC);
      const int k = k0 + kk;
      float kv[VEC], vv[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) kv[e] = vv[e] = 0.0f;
      if (k < k_end) {
        int blk = bt[k / bs];
        if (blk < 0 || blk >= a.num_blocks) {
          s_badblk = 1;
        } else {
          const size_t base = (((size_t)blk * a.Hkv + kvh) * bs + (k % bs)) * D + c * VEC;
          const uint4 kr = *reinterpret_cast<const uint4*>(kc + base);
          const uint4 vr = *reinterpret_cast<const uint4*>(vc + base);
          const T* kp = reinterpret_cast<const T*>(&kr);
          const T* vp = reinterpret_cast<const T*>(&vr);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            kv[e] = to_f32(kp[e]);
            vv[e] = to_f32(vp[e]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        Ks[kk][c * VEC + e] = kv[e];
        Vs[kk][c * VEC + e] = vv[e];
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int lr = warp * 4 + i, r = r0 + lr;
      if (r >= rows) continue;
      const int t = off + r / g;
      const int k = k0 + lane;
      bool vis = k < k_end;
      if (vis && k >= P) {
        const int v = k - P;
        vis = (a.mask[(size_t)t * a.W + (v >> 6)] >> (v & 63)) & 1ull;
      }
      float s = -INFINITY;
      if (vis) {
        float acc = 0.0f;
#pragma unroll 16
        for (int d = 0; d < D; ++d) acc = fmaf(Qs[lr][d], Ks[lane][d], acc);
        s = acc * a.scale_log2;
      }
      const float mnew = fmaxf(m[i], warp_max_f(s));
      if (mnew == -INFINITY) continue;
      const float p = fast_exp2(s - mnew);
      const float alpha = fast_exp2(m[i] - mnew);
      l[i] = l[i] * alpha + warp_sum_f(p);
#pragma unroll
      for (int j = 0; j < DJ; ++j) o[i][j] *= alpha;
#pragma unroll 8
      for (int kk = 0; kk < kCcKeys; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
        for (int j = 0; j < DJ; ++j) o[i][j] = fmaf(pk, Vs[kk][lane + 32 * j], o[i][j]);
      }
      m[i] = mnew;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_badblk) atomicOr(&a.status[b], SPEC_DEV_BAD_BLOCK);

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int lr = warp * 4 + i, r = r0 + lr;
    if (r >= rows) continue;
    const int t = off + r / g, hh = kvh * g + r % g;
    const size_t row = (size_t)t * a.Hq + hh;
    if (a.splits == 1) {
      const float inv = 1.0f / l[i];
      T* out = static_cast<T*>(a.out);
#pragma unroll
      for (int j = 0; j < DJ; ++j) out[row * D + lane + 32 * j] = from_f32<T>(o[i][j] * inv);
    } else {
      float* wo = a.ws_o + ((size_t)split * a.T * a.Hq + row) * D;
#pragma unroll
      for (int j = 0; j < DJ; ++j) wo[lane + 32 * j] = o[i][j];
      if (lane == 0) {
        float* wml = a.ws_ml + ((size_t)split * a.T * a.Hq + row) * 2;
        wml[0] = m[i];
        wml[1] = l[i];
      }
    }
  }
}

// Split-KV combine: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
// One warp per (node, query head) row.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int rowsT = a.T * a.Hq;
  if (warp_global >= rowsT) return;
  const int t = warp_global / a.Hq;
  // request of node t
  int lo = 0, hi = a.B;  // tree_off[lo] <= t < tree_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.tree_off[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int b = lo;
  const int n = a.tree_off[b + 1] - a.tree_off[b];
  if (n <= 0 || n > a.n_max || a.tree_off[b] + n > a.T || a.status[b] != 0) return;
  const int L = a.prefix_len[b] + n;
  const int ns = min(a.splits, (L + a.chunk - 1) / a.chunk);
  const size_t row = (size_t)warp_global;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, a.ws_ml[((size_t)s * rowsT + row) * 2]);
  float lsum = 0.0f, acc[D / 32];
#pragma unroll
  for (int j = 0; j < D / 32; ++j) acc[j] = 0.0f;
  for (int s = 0; s < ns; ++s) {
    const float ms = a.ws_ml[((size_t)s * rowsT + row) * 2];
    if (ms == -INFINITY) continue;
    const float w = fast_exp2(ms - M);
    lsum += w * a.ws_ml[((size_t)s * rowsT + row) * 2 + 1];
    const float* os = a.ws_o + ((size_t)s * rowsT + row) * D;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) acc[j] = fmaf(w, os[lane + 32 * j], acc[j]);
  }
  const float inv = 1.0f / lsum;
  T* out = static_cast<T*>(a.out);
#pragma unroll
  for (int j = 0; j < D / 32; ++j) out[row * D + lane + 32 * j] = from_f32<T>(acc[j] * inv);
}

template <typename T>
static cudaError_t launch_cc_t(const AttnArgs& a, cudaStream_t stream) {
  const int rows_max = a.n_max * a.g;
  dim3 grid((rows_max + kCcRows - 1) / kCcRows, a.splits, a.B * a.Hkv);
  if (a.D == 64) attn_cc_kernel<T, 64><<<grid, kCcThreads, 0, stream>>>(a);
  else attn_cc_kernel<T, 128><<<grid, kCcThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attention_cc(const AttnArgs& a, spec_dtype dt, int row_tile, cudaStream_t stream) {
  (void)row_tile;
  return dt == SPEC_F32 ? launch_cc_t<float>(a, stream) : launch_cc_t<__nv_bfloat16>(a, stream);
}

cudaError_t launch_attention_combine(const AttnArgs& a, spec_dtype dt, cudaStream_t stream) {
  const int rows = a.T * a.Hq;
  const int grid = (rows + 7) / 8;
  if (dt == SPEC_F32) {
    if (a.D == 64) attn_combine_kernel<float, 64><<<grid, 256, 0, stream>>>(a);
    else attn_combine_kernel<float, 128><<<grid, 256, 0, stream>>>(a);
  } else {
    if (a.D == 64) attn_combine_kernel<__nv_bfloat16, 64><<<grid, 256, 0, stream>>>(a);
    else attn_combine_kernel<__nv_bfloat16, 128><<<grid, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

// Split plan.  The tensor-core kernel holds a whole SM per CTA (all of TMEM),
// so the plan minimises waves x per-CTA time: a wave of the 152 SMs costs a
// fixed ~4 us (set-up, first loads, epilogue) plus ~1.3 us per 128-key tile.
// The CUDA-core kernel (several CTAs per SM) targets about two waves of CTAs.
// Key chunks are multiples of 128 keys.
AttnPlan attention_plan(int B, int n_max, int max_prefix, int Hq, int Hkv, int D, bool bf16, unsigned flags) {
  (void)D;
  AttnPlan p;
  const int g = Hq / Hkv;
  const int rows_max = n_max * g;
  p.use_tc = false;
  if (bf16 && flags != SPEC_ATTN_CUDA_CORE && attention_tc_enabled(D)) {
    // every bf16 group, padded to 128 rows when smaller: the K/V stream, not
    // the MMA, bounds small groups, and the tensor-core kernel streams it at
    // near HBM rate where the CUDA-core kernel does not
    p.use_tc = true;
  }
  p.row_tile = p.use_tc ? 128 : kCcRows;
  const long long units = (long long)B * Hkv * ((rows_max + p.row_tile - 1) / p.row_tile);
  const long long max_len = (long long)max_prefix + n_max;
  long long splits = 1;
  if (p.use_tc) {
    double best = 1e300;
    const long long smax = std::max(1LL, std::min(64LL, (max_len + 127) / 128));
    for (long long sp = 1; sp <= smax; ++sp) {
      const long long chunk = ((max_len + sp - 1) / sp + 127) / 128 * 128;
      const long long waves = (units * sp + 151) / 152;
      const double cost = (double)waves * (4.0 + 1.3 * (double)(chunk / 128));
      if (cost < best * 0.97) {  // prefer fewer splits (less partial traffic) on near-ties
        best = cost;
        splits = sp;
      }
    }
  } else {
    const long long target = 2 * 152;
    splits = units > 0 ? (target + units - 1) / units : 1;
    splits = std::max(1LL, std::min(splits, (max_len + 511) / 512));
  }
  long long chunk = (max_len + splits - 1) / splits;
  chunk = (chunk + 127) / 128 * 128;
  if (chunk < 128) chunk = 128;
  p.chunk = (int)chunk;
  p.splits = (int)((max_len + chunk - 1) / chunk);
  if (p.splits < 1) p.splits = 1;
  return p;
}

size_t attention_ws_bytes(const AttnPlan& p, int T, int Hq, int D) {
  if (p.splits <= 1) return 0;
  const size_t o = (size_t)p.splits * T * Hq * D * sizeof(float);
  const size_t ml = (size_t)p.splits * T * Hq * 2 * sizeof(float);
  return ((o + 255) & ~(size_t)255) + ml;
}

// ---------------------------------------------------------------------------
// Scratch of spec_tree_attention_noalloc: one file-scope device array (every
// GPU that loads the library holds it until the process exits).  In host code
// the symbol names a host-side stand-in, so kernels get the device address,
// looked up with the device current and cached per device together with the
// context it was looked up in: after a reset of the device's primary context
// the next call looks the address up again instead of using a stale one.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_attn_scratch[SPEC_ATTN_NOALLOC_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

static CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

static std::mutex g_attn_scratch_mutex;
static void* g_attn_scratch_ptr[128];
static CUcontext g_attn_scratch_ctx[128];

// Device address of the scratch array on the current device; NULL when the
// lookup fails (the runtime's error from the failed lookup is cleared, so a
// later cudaGetLastError() does not report it).
static void* attn_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    cudaGetLastError();
    return nullptr;
  }
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_attn_scratch_mutex);
  if (!g_attn_scratch_ptr[dev] || !ctx || g_attn_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      g_attn_scratch_ptr[dev] = nullptr;
      return nullptr;
    }
    // the runtime creates the primary context on first use: read it again
    if (!ctx && get_ctx && get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    g_attn_scratch_ptr[dev] = p;
    g_attn_scratch_ctx[dev] = ctx;
  }
  return g_attn_scratch_ptr[dev];
}

// Argument checks shared by both attention entry points, made before the
// plan is computed (the plan's row and chunk arithmetic assumes them).
// SPEC_OK when the shape and scalar arguments are acceptable.
static spec_status attention_shape_check(int B, int T, int n_max, int max_prefix, int Hq, int Hkv, int D,
                                         spec_dtype dtype, int block_size, uint32_t flags) {
  if (B < 0 || T < 0 || n_max < 0 || max_prefix < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (flags > SPEC_ATTN_TCGEN05) return SPEC_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  if (n_max > SPEC_MAX_NODES || B > 65535) return SPEC_ERR_UNSUPPORTED;
  if (block_size < 8 || block_size > 65536 || (block_size & (block_size - 1))) return SPEC_ERR_UNSUPPORTED;
  if (flags == SPEC_ATTN_TCGEN05 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if ((long long)B * Hkv > 65535 * 1024LL) return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

}  // namespace spectree

using namespace spectree;

extern "C" {

size_t spec_attention_workspace_size(int B, int T, int n_max, int max_prefix, int Hq, int Hkv, int D) {
  if (B <= 0 || T <= 0 || n_max <= 0 || Hkv <= 0 || Hq < Hkv || max_prefix < 0) return 256;
  size_t best = 256;
  for (unsigned f : {SPEC_ATTN_CUDA_CORE, SPEC_ATTN_TCGEN05, SPEC_ATTN_AUTO}) {
    const AttnPlan p = attention_plan(B, n_max, max_prefix, Hq, Hkv, D, true, f);
    best = std::max(best, attention_ws_bytes(p, T, Hq, D));
    const AttnPlan p2 = attention_plan(B, n_max, max_prefix, Hq, Hkv, D, false, f);
    best = std::max(best, attention_ws_bytes(p2, T, Hq, D));
  }
  return best;
}

spec_status spec_tree_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                int max_blocks, int block_size, int num_blocks, const int32_t* prefix_len,
                                const int32_t* tree_off, const uint64_t* mask, int B, int T, int n_max,
                                int max_prefix, int Hq, int Hkv, int D, spec_dtype dtype, float scale, void* out,
                                void* workspace, size_t workspace_bytes, int32_t* status, uint32_t flags,
                                void* stream) {
  SPEC_NVTX_RANGE("spec_tree_attention");
  const spec_status sc = attention_shape_check(B, T, n_max, max_prefix, Hq, Hkv, D, dtype, block_size, flags);
  if (sc != SPEC_OK) return sc;
  if (B == 0 || T == 0 || n_max == 0) return SPEC_OK;
  if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !tree_off || !mask || !out || !status ||
      max_blocks <= 0 || num_blocks <= 0)
    return SPEC_ERR_INVALID_ARG;

  const AttnPlan plan = attention_plan(B, n_max, max_prefix, Hq, Hkv, D, dtype == SPEC_BF16, flags);
  const size_t need = attention_ws_bytes(plan, T, Hq, D);
  if (need > 0 && (!workspace || workspace_bytes < need)) return SPEC_ERR_WORKSPACE;

  AttnArgs a = {};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.prefix_len = prefix_len;
  a.tree_off = tree_off;
  a.mask = mask;
  a.out = out;
  a.status = status;
  if (need > 0) {
    const size_t o = (size_t)plan.splits * T * Hq * D * sizeof(float);
    a.ws_o = static_cast<float*>(workspace);
    a.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o + 255) & ~(size_t)255));
  }
  a.max_blocks = max_blocks;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.B = B;
  a.T = T;
  a.n_max = n_max;
  a.max_prefix = max_prefix;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.g = Hq / Hkv;
  a.W = (n_max + 63) / 64;
  a.splits = plan.splits;
  a.chunk = plan.chunk;
  a.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t st = (cudaStream_t)stream;
  if (need > 0) spec_workspace_canary(workspace, need, st);
  cudaError_t e;
  if (plan.use_tc) e = launch_attention_tc(a, st);
  else e = launch_attention_cc(a, dtype, plan.row_tile, st);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  if (plan.splits > 1) {
    e = launch_attention_combine(a, dtype, st);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

// Attention without a workspace argument: the split-KV partials live in the
// library's fixed scratch array.  The same shape checks as spec_tree_attention
// come first (the plan assumes them), then the scratch limit; the pointers are
// checked by spec_tree_attention, which then launches.
spec_status spec_tree_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                                        const int32_t* prefix_len, const int32_t* tree_off, const uint64_t* mask,
                                        int B, int T, int n_max, int max_prefix, int Hq, int Hkv, int D,
                                        spec_dtype dtype, float scale, void* out, int32_t* status, uint32_t flags,
                                        void* stream) {
  SPEC_NVTX_RANGE("spec_tree_attention_noalloc");
  const spec_status sc = attention_shape_check(B, T, n_max, max_prefix, Hq, Hkv, D, dtype, block_size, flags);
  if (sc != SPEC_OK) return sc;
  if (B == 0 || T == 0 || n_max == 0) return SPEC_OK;
  const AttnPlan plan = attention_plan(B, n_max, max_prefix, Hq, Hkv, D, dtype == SPEC_BF16, flags);
  const size_t need = attention_ws_bytes(plan, T, Hq, D);
  if (need > (size_t)SPEC_ATTN_NOALLOC_BYTES) return SPEC_ERR_UNSUPPORTED;
  void* ws = attn_scratch();
  if (!ws) return SPEC_ERR_CUDA;
  return spec_tree_attention(q, k_cache, v_cache, block_table, max_blocks, block_size, num_blocks, prefix_len,
                             tree_off, mask, B, T, n_max, max_prefix, Hq, Hkv, D, dtype, scale, out, ws,
                             (size_t)SPEC_ATTN_NOALLOC_BYTES, status, flags, stream);
}

}  // extern "C"
