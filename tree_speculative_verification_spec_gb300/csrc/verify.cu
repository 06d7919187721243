// Token-tree verification, greedy and stochastic, in one launch per call.
//
// Phase A (one thread-block cluster per tree node): the node's target row is
// streamed once from HBM, split across the C CTAs of the cluster (a slice of
// at most kSlice vocabulary entries each, held in shared memory for the
// stochastic verifier); row reductions combine through distributed shared
// memory.  Greedy: the argmax of the row.  Stochastic: the node decides, by
// itself, which of its children the walk would accept if it reached the node
// (the decision depends only on the node's own rows, its children's tokens
// and their random words), and, when none is accepted, samples the
// correction / bonus token.
// Phase B (the last CTA to finish a request, found with an atomic ticket):
// greedy picks the deepest node whose root path follows the argmax chain;
// stochastic follows the accepted-child links from the root.  No CTA ever
// waits for another.
#include <cooperative_groups.h>

#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace spectree {

// Stochastic: 128-thread CTAs over 4096-entry slices held in shared memory
// (up to 8 CTAs per SM).  Greedy streams its slice once: 256-thread CTAs over
// 16384-entry slices.  Slices widen beyond 8 CTAs per cluster.
constexpr int kVerifyThreads = 256;  // upper bound of the two block sizes
template <int MODE> struct VCfg;
template <> struct VCfg<0> { static constexpr int threads = 256, slice = 16384, min_blocks = 4; };
template <> struct VCfg<1> { static constexpr int threads = 128, slice = 4096, min_blocks = 8; };

// ---------------------------------------------------------------------------
// fp32 arithmetic contract of the stochastic verifier.  Every operation is a
// single IEEE operation (explicit _rn intrinsics: never contracted); the only
// fused multiply-adds are the explicit fmaf calls of canon_exp.
// ---------------------------------------------------------------------------

// e^x for x <= 0: Cody-Waite reduction x = n ln2 + r with ln2 = LN2_HI +
// LN2_LO (LN2_HI keeps 16 significant bits, so n * LN2_HI is exact), the
// degree-7 Taylor polynomial of e^r (coefficients 1/k!) in Horner form, and
// scaling by 2^n through the exponent field.  Constants are the correctly
// rounded fp32 values, written as exact hex literals.  x < -87 gives 0.
__device__ __forceinline__ float canon_exp(float x) {
  if (!(x >= -87.0f)) return 0.0f;
  const float t = __fmul_rn(x, 0x1.715476p+0f);  // x * log2(e)
  // rint(t) without a conversion unit op: adding 1.5 * 2^23 leaves the integer
  // (rounded to nearest, ties to even) in the low mantissa bits; |t| < 2^22.
  const float big = __fadd_rn(t, 12582912.0f);
  const float n = __fsub_rn(big, 12582912.0f);
  const int ni = __float_as_int(big) - 0x4B400000;
  float r = fmaf(-n, 0x1.62e4p-1f, x);    // ln2, high 16 bits
  r = fmaf(-n, 0x1.7f7d1cp-20f, r);       // ln2 - high part
  float p = 0x1.a01a02p-13f;              // 1/7!
  p = fmaf(p, r, 0x1.6c16c2p-10f);        // 1/6!
  p = fmaf(p, r, 0x1.111112p-7f);         // 1/5!
  p = fmaf(p, r, 0x1.555556p-5f);         // 1/4!
  p = fmaf(p, r, 0x1.555556p-3f);         // 1/3!
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

// Fixed-point weight trunc(v * 2^46) and the normaliser of a sum of them.
// trunc(v * 2^46) for 0 <= v < 2 from the bit fields (no conversion unit op):
// v = m * 2^(e - 150) with the 24-bit significand m, so v * 2^46 = m * 2^(e - 104).
__device__ __forceinline__ unsigned long long fx(float v) {
  const uint32_t bits = __float_as_uint(v);
  const int e = (int)((bits >> 23) & 0xFFu);
  const unsigned long long m = (unsigned long long)((bits & 0x7FFFFFu) | 0x800000u);
  const int sh = e - 104;
  if (e == 0) return 0ull;  // zero or subnormal: below 2^-126 * 2^46
  return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> (-sh)) : 0ull);
}
// Running sum of FX values, mostly on the FMA pipe: for 0 <= v <= 1,
// v * 2^46 = A * 2^23 + B with A = trunc(v * 2^23) and B = trunc(frac(v * 2^23) * 2^23);
// each is read off a round-toward-zero addition of 2^23 (ulp 1 on [2^23, 2^24]).
// A and B of up to 2^6 * 2^8 terms fit 32 bits; values above 1 take fx().
struct FxSum {
  uint32_t a = 0, b = 0;
  unsigned long long big = 0;
  __device__ __forceinline__ void add(float v) {
    if (v <= 1.0f) {
      const float y1 = __fmul_rn(v, 0x1p23f);
      const float t = __fadd_rz(y1, 0x1p23f);
      const float f = __fsub_rn(y1, __fsub_rn(t, 0x1p23f));
      const float t2 = __fadd_rz(__fmul_rn(f, 0x1p23f), 0x1p23f);
      a += __float_as_uint(t) - 0x4B000000u;
      b += __float_as_uint(t2) - 0x4B000000u;
    } else {
      big += fx(v);
    }
  }
  __device__ __forceinline__ unsigned long long total() const {
    return ((unsigned long long)a << 23) + (unsigned long long)b + big;
  }
};

__device__ __forceinline__ float z_of(unsigned long long S) { return __fmul_rn(__ull2float_rn(S), 0x1p-46f); }

// floor(U * S / 2^32), exact for U < 2^32, S < 2^64.
__device__ __forceinline__ unsigned long long sample_target(uint32_t U, unsigned long long S) {
  const unsigned long long lo = (unsigned long long)U * (S & 0xffffffffull);
  const unsigned long long hi = (unsigned long long)U * (S >> 32);
  return hi + (lo >> 32);
}

// residual step: max(r - q, 0) written as a comparison (no fmax sign-of-zero ambiguity)
__device__ __forceinline__ float resid(float d, float Z, float q) {
  const float diff = __fsub_rn(__fdiv_rn(d, Z), q);
  return diff > 0.0f ? diff : 0.0f;
}

// ---------------------------------------------------------------------------
// Block / cluster reductions
// ---------------------------------------------------------------------------

struct Red {
  float f[kVerifyThreads / 32];
  int i[kVerifyThreads / 32];
  unsigned long long u[kVerifyThreads / 32];
};

__device__ __forceinline__ float block_max(float v, Red& s) {
  v = warp_max_f(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) s.f[w] = v;
  __syncthreads();
  v = s.f[0];
  for (int k = 1; k < (int)(blockDim.x >> 5); ++k) v = fmaxf(v, s.f[k]);
  return v;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, Red& s) {
  v = warp_sum_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) s.u[w] = v;
  __syncthreads();
  v = 0;
  for (int k = 0; k < (int)(blockDim.x >> 5); ++k) v += s.u[k];
  return v;
}

// (value, index) argmax; ties to the lower index.
__device__ __forceinline__ void argmax_combine(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void block_argmax(float& v, int& i, Red& s) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_combine(v, i, v2, i2);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    s.f[w] = v;
    s.i[w] = i;
  }
  __syncthreads();
  v = s.f[0];
  i = s.i[0];
  for (int k = 1; k < (int)(blockDim.x >> 5); ++k) argmax_combine(v, i, s.f[k], s.i[k]);
}

// Cluster exchange slots (one per CTA, read by every CTA of the cluster).
struct XSlot {
  float f;
  int i;
  unsigned long long u;
};

template <int C>
__device__ __forceinline__ void cluster_sync_all() {
  if constexpr (C == 1) __syncthreads();
  else cg::this_cluster().sync();
}

// Cluster reductions with one cluster barrier each: every CTA publishes its
// block result in exchange slot `par`, the barrier makes it visible, every CTA
// reads all C slots.  Slots alternate, so a slot is rewritten only after a
// later barrier, which no CTA passes before finishing its reads of it.  A
// final barrier before exit keeps peers' shared memory alive for late reads.
template <int C>
__device__ __forceinline__ float cluster_max(float v, Red& red, XSlot* xs, int& par) {
  v = block_max(v, red);
  if constexpr (C == 1) return v;
  cg::cluster_group cl = cg::this_cluster();
  if (threadIdx.x == 0) xs[par].f = v;
  cl.sync();
  float m = v;
  for (int r = 0; r < C; ++r) m = fmaxf(m, cl.map_shared_rank(xs + par, r)->f);
  par ^= 1;
  return m;
}

template <int C>
__device__ __forceinline__ unsigned long long cluster_sum(unsigned long long v, Red& red, XSlot* xs, int& par) {
  v = block_sum_u64(v, red);
  if constexpr (C == 1) return v;
  cg::cluster_group cl = cg::this_cluster();
  if (threadIdx.x == 0) xs[par].u = v;
  cl.sync();
  unsigned long long s = 0;
  for (int r = 0; r < C; ++r) s += cl.map_shared_rank(xs + par, r)->u;
  par ^= 1;
  return s;
}

// sum over the CTAs of lower rank (exclusive prefix)
template <int C>
__device__ __forceinline__ unsigned long long cluster_prefix(unsigned long long v, XSlot* xs, int& par, int rank) {
  if constexpr (C == 1) return 0ull;
  cg::cluster_group cl = cg::this_cluster();
  if (threadIdx.x == 0) xs[par].u = v;
  cl.sync();
  unsigned long long s = 0;
  for (int r = 0; r < rank; ++r) s += cl.map_shared_rank(xs + par, r)->u;
  par ^= 1;
  return s;
}

template <int C>
__device__ __forceinline__ void cluster_argmax(float& v, int& i, Red& red, XSlot* xs, int& par) {
  block_argmax(v, i, red);
  if constexpr (C == 1) return;
  cg::cluster_group cl = cg::this_cluster();
  if (threadIdx.x == 0) {
    xs[par].f = v;
    xs[par].i = i;
  }
  cl.sync();
  for (int r = 0; r < C; ++r) {
    const XSlot* p = cl.map_shared_rank(xs + par, r);
    argmax_combine(v, i, p->f, p->i);
  }
  par ^= 1;
}

struct VerifyArgs {
  const float* p_logits;
  const float* q_probs;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* tree_off;
  const uint64_t* mask;
  const int32_t* depth;
  const uint2* uniforms;
  int n_max, V, W, slice;
  int32_t* path;
  int32_t* accept_len;
  int32_t* emitted;
  int32_t* n_emitted;
  int32_t* status;
  // workspace
  int32_t* ws_a;        // [B * n_max]  greedy: argmax / stochastic: accepted child (or -1)
  int32_t* ws_s;        // [B * n_max]  stochastic: sampled token when no child is accepted
  int32_t* ws_ticket;   // [B]          zeroed by the host wrapper before the launch
};

__device__ __forceinline__ void clear_request(const VerifyArgs& a, int b) {
  for (int i = threadIdx.x; i < a.n_max; i += blockDim.x) {
    a.path[(size_t)b * a.n_max + i] = -1;
    a.emitted[(size_t)b * a.n_max + i] = -1;
  }
  if (threadIdx.x == 0) {
    a.accept_len[b] = 0;
    a.n_emitted[b] = 0;
  }
}

// Children of node u (local indices, increasing) into kids[]; returns the
// count.  Ordered stream compaction: per chunk of blockDim candidates, warp
// ballots give per-warp counts, thread 0 turns them into offsets.
__device__ int collect_children(const int32_t* par, int n, int u, int* kids, int* s_cnt, int* s_wofs) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) *s_cnt = 0;
  __syncthreads();
  for (int base = u + 1; base < n; base += blockDim.x) {
    const int c = base + threadIdx.x;
    const bool is = c < n && __ldg(par + c) == u;
    const unsigned m = __ballot_sync(0xffffffffu, is);
    if (lane == 0) s_wofs[w] = __popc(m);
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = *s_cnt;
      for (int k = 0; k < nw; ++k) {
        const int x = s_wofs[k];
        s_wofs[k] = acc;
        acc += x;
      }
      *s_cnt = acc;
    }
    __syncthreads();
    if (is) kids[s_wofs[w] + __popc(m & ((1u << lane) - 1u))] = c;
    __syncthreads();
  }
  return *s_cnt;
}

// Bulk copy of one row slice (global -> this CTA's shared memory) completing
// on an mbarrier, and a bounded wait for it.
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool bulk_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

template <int MODE, int C>
__global__ void __launch_bounds__(VCfg<MODE>::threads, VCfg<MODE>::min_blocks) verify_kernel(VerifyArgs a) {
  constexpr int NT = VCfg<MODE>::threads;
  extern __shared__ float4 dyn_smem[];
  float* D = reinterpret_cast<float*>(dyn_smem);  // stochastic: the node's weights slice
  __shared__ Red red;
  __shared__ XSlot xs[2];
  __shared__ int32_t s_kids[SPEC_MAX_NODES];
  __shared__ int s_cnt, s_last, s_flag;
  __shared__ int s_wofs[kVerifyThreads / 32];
  __shared__ uint64_t s_match[SPEC_MAX_WORDS];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ float s_z[SPEC_MAX_NODES];  // normalisers of the residual steps applied so far

  // grid: x = (request, cluster rank), y = node; nodes near the root (most
  // children, most residual passes) are dispatched first
  const int rank = (int)(blockIdx.x % C);
  const int b = (int)(blockIdx.x / C);
  const int u = blockIdx.y;
  int par = 0;  // exchange-slot parity of the cluster reductions
  const int off = a.tree_off[b];
  const int n = a.tree_off[b + 1] - off;
  const bool n_ok = n >= 1 && n <= a.n_max;
  const int n_cta = n_ok ? n : 1;  // requests without a valid tree still run phase B once
  if (u >= n_cta) return;

  // Only SPEC_DEV_BAD_TOKEN can change while this kernel runs (other CTAs set
  // it); ignoring that bit keeps the decision uniform across a cluster.
  const int st_in = *(volatile int32_t*)&a.status[b];
  const bool work = n_ok && (st_in & ~SPEC_DEV_BAD_TOKEN) == 0;
  const int V = a.V;
  const int x0 = rank * a.slice;
  const int x1 = min(V, x0 + a.slice);
  const int len = max(0, x1 - x0);
  const int t = off + u;

  if (work && rank == 0 && threadIdx.x == 0) {
    const int tok = a.tokens[t];
    if (tok < 0 || tok >= V) atomicOr(&a.status[b], SPEC_DEV_BAD_TOKEN);
  }
  if (work) {
    const float* prow = a.p_logits + (size_t)t * V;
    if constexpr (MODE == 0) {
      // ---- greedy: argmax of row u, ties to the lowest token id; four
      // independent 16-byte loads in flight per thread ----
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      if ((V & 3) == 0) {
        const float4* p4 = reinterpret_cast<const float4*>(prow);
        const int j0 = x0 >> 2, j1 = x1 >> 2;
        for (int j = j0 + threadIdx.x; j < j1; j += 4 * NT) {
          float4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int jj = j + q * NT;
            v[q] = jj < j1 ? __ldcs(p4 + jj) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int x = (j + q * NT) << 2;
            if (v[q].x > bv) { bv = v[q].x; bi = x; }
            if (v[q].y > bv) { bv = v[q].y; bi = x + 1; }
            if (v[q].z > bv) { bv = v[q].z; bi = x + 2; }
            if (v[q].w > bv) { bv = v[q].w; bi = x + 3; }
          }
        }
      } else {
        for (int x = x0 + threadIdx.x; x < x1; x += blockDim.x) {
          const float v = __ldcs(prow + x);
          if (v > bv) { bv = v; bi = x; }
        }
      }
      cluster_argmax<C>(bv, bi, red, xs, par);
      cluster_sync_all<C>();  // peers read this CTA's slot
      if (rank == 0 && threadIdx.x == 0) a.ws_a[(size_t)b * a.n_max + u] = bi == 0x7fffffff ? 0 : bi;
    } else {
      // ---- stochastic: row state of node u ----
      const float* qrow = a.q_probs + (size_t)t * V;
      const int lenp = (len + 3) & ~3;  // padded to whole float4 (pad = -inf: weight 0)
      if ((V & 3) == 0) {
        // one bulk copy of the slice into shared memory
        if (threadIdx.x == 0) {
          asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&s_bar)) : "memory");
          asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&s_bar)),
                       "r"((uint32_t)(len * 4))
                       : "memory");
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  smem_addr(D)),
              "l"(prow + x0), "r"((uint32_t)(len * 4)), "r"(smem_addr(&s_bar))
              : "memory");
        }
        __syncthreads();
        if (!bulk_wait(&s_bar, 0)) {
          if (threadIdx.x == 0) atomicOr(&a.status[b], SPEC_DEV_TIMEOUT);
          bulk_wait(&s_bar, 0);  // drain before the buffer is touched
        }
      } else {
        for (int j = threadIdx.x; j < len; j += blockDim.x) D[j] = __ldcs(prow + x0 + j);
      }
      for (int j = len + threadIdx.x; j < lenp; j += blockDim.x) D[j] = -INFINITY;
      __syncthreads();
      float4* D4 = reinterpret_cast<float4*>(D);
      float lmax = -INFINITY;
      for (int j = threadIdx.x; j < (lenp >> 2); j += blockDim.x) {
        const float4 v = D4[j];
        lmax = fmaxf(lmax, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
      }
      const float m = cluster_max<C>(lmax, red, xs, par);
      FxSum acc;
      for (int j = threadIdx.x; j < (lenp >> 2); j += blockDim.x) {
        float4 v = D4[j];
        v.x = canon_exp(__fsub_rn(v.x, m));
        v.y = canon_exp(__fsub_rn(v.y, m));
        v.z = canon_exp(__fsub_rn(v.z, m));
        v.w = canon_exp(__fsub_rn(v.w, m));
        D4[j] = v;
        acc.add(v.x);
        acc.add(v.y);
        acc.add(v.z);
        acc.add(v.w);
      }
      unsigned long long ls = acc.total();
      unsigned long long S = cluster_sum<C>(ls, red, xs, par);
      float Z = z_of(S);

      // children of u in increasing index
      const int k = collect_children(a.parent + off, n, u, s_kids, &s_cnt, s_wofs);

      int accepted = -1;
      bool bad_tok = false;
      bool frozen = false;      // a zero-sum residual froze the state (see below)
      int nsteps = 0;           // residual steps applied to D
      unsigned long long lt = ls;  // this CTA's share of S
      for (int i = 0; i < k; ++i) {
        const int c = s_kids[i];
        const int tok = a.tokens[off + c];
        if (tok < 0 || tok >= V) {
          bad_tok = true;
          break;
        }
        // r_j(tok) from the CTA of the cluster that holds tok
        const int owner = tok / a.slice;
        float dt;
        if constexpr (C == 1) {
          dt = D[tok];
        } else {
          dt = cg::this_cluster().map_shared_rank(D, owner)[tok - owner * a.slice];
        }
        const float rt = __fdiv_rn(dt, Z);
        const float qt = qrow[tok];
        const float ua = __fmul_rn((float)(a.uniforms[off + c].x >> 8), 0x1p-24f);
        if (__fmul_rn(ua, qt) <= rt) {
          accepted = c;
          break;
        }
        if (frozen) continue;  // the next residual would be the same all-zero one
        // rejection: d <- max(d / Z - q, 0) in place, S <- sum FX(d)
        s_z[nsteps] = Z;
        cluster_sync_all<C>();  // every CTA has read D[tok] before it changes
        unsigned long long ln = 0;
        if ((V & 3) == 0) {
          const float4* q4 = reinterpret_cast<const float4*>(qrow + x0);
          FxSum ra;
          for (int j = threadIdx.x; j < (len >> 2); j += blockDim.x) {
            float4 d = D4[j];
            const float4 qq = __ldg(q4 + j);
            d.x = resid(d.x, Z, qq.x);
            d.y = resid(d.y, Z, qq.y);
            d.z = resid(d.z, Z, qq.z);
            d.w = resid(d.w, Z, qq.w);
            D4[j] = d;
            ra.add(d.x);
            ra.add(d.y);
            ra.add(d.z);
            ra.add(d.w);
          }
          ln = ra.total();
        } else {
          for (int j = threadIdx.x; j < len; j += blockDim.x) {
            const float dn = resid(D[j], Z, __ldg(qrow + x0 + j));
            D[j] = dn;
            ln += fx(dn);
          }
        }
        const unsigned long long Sn = cluster_sum<C>(ln, red, xs, par);  // also publishes D
        if (Sn != 0) {
          S = Sn;
          Z = z_of(Sn);
          lt = ln;
          ++nsteps;
        } else {
          // S_j == 0 (impossible in exact arithmetic after a rejection): the
          // state stays that of step j-1, and so does every later residual.
          // Rebuild step j-1 from the logits: e, then the nsteps earlier steps.
          frozen = true;
          ls = 0;
          for (int j = threadIdx.x; j < len; j += blockDim.x) D[j] = canon_exp(__fsub_rn(__ldg(prow + x0 + j), m));
          for (int j = len + threadIdx.x; j < lenp; j += blockDim.x) D[j] = 0.0f;
          for (int st2 = 0; st2 < nsteps; ++st2) {
            __syncthreads();
            const float Zs = s_z[st2];
            for (int j = threadIdx.x; j < len; j += blockDim.x) D[j] = resid(D[j], Zs, __ldg(qrow + x0 + j));
          }
          __syncthreads();
          for (int j = threadIdx.x; j < len; j += blockDim.x) ls += fx(D[j]);
          lt = ls;                // this thread's share of S, which is unchanged
          cluster_sync_all<C>();  // D is read across the cluster by the next test
        }
      }
      // A CTA may read a peer's shared memory (D[tok]) right before the loop
      // ends: no CTA of the cluster leaves before every such read is done.
      cluster_sync_all<C>();
      if (bad_tok) {
        if (rank == 0 && threadIdx.x == 0) atomicOr(&a.status[b], SPEC_DEV_BAD_TOKEN);
      } else if (accepted >= 0) {
        if (rank == 0 && threadIdx.x == 0) a.ws_a[(size_t)b * a.n_max + u] = accepted;
      } else {
        // terminal sample: smallest x whose fixed-point prefix sum exceeds target
        const unsigned long long target = sample_target(a.uniforms[t].y, S);
        // this CTA's slice total (kept from the last pass) and the exclusive
        // prefix of the slices before it
        lt = block_sum_u64(lt, red);
        const unsigned long long before = cluster_prefix<C>(lt, xs, par, rank);
        cluster_sync_all<C>();  // peers read this CTA's slot
        if (target >= before && target - before < lt) {
          // the token lies in this slice: per-warp contiguous chunks
          const unsigned long long tl = target - before;
          const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
          const int cw = (len + nw - 1) / nw;
          const int c0 = min(len, w * cw), c1 = min(len, c0 + cw);
          unsigned long long wsum = 0;
          for (int j = c0 + lane; j < c1; j += 32) wsum += fx(D[j]);
          wsum = warp_sum_u64(wsum);
          __syncthreads();
          if (lane == 0) red.u[w] = wsum;
          __syncthreads();
          if (threadIdx.x == 0) {
            unsigned long long acc = 0;
            int ww = 0;
            for (; ww < nw; ++ww) {
              if (tl < acc + red.u[ww]) break;
              acc += red.u[ww];
            }
            s_flag = ww;
            red.u[0] = acc;  // prefix before warp ww (slot reused after the read above)
          }
          __syncthreads();
          const int ww = s_flag;
          const unsigned long long acc0 = red.u[0];
          if (w == ww) {
            const int d0 = min(len, ww * cw), d1 = min(len, d0 + cw);
            unsigned long long run = acc0;
            for (int base = d0; base < d1; base += 32) {
              const int j = base + lane;
              unsigned long long v = j < d1 ? fx(D[j]) : 0ull;
              // inclusive warp scan
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
              }
              const unsigned hit = __ballot_sync(0xffffffffu, j < d1 && run + v > tl);
              if (hit) {
                if (lane == __ffs(hit) - 1) {
                  a.ws_s[(size_t)b * a.n_max + u] = x0 + j;
                  __threadfence();
                }
                break;
              }
              run += __shfl_sync(0xffffffffu, v, 31);
            }
          }
        }
        if (rank == 0 && threadIdx.x == 0) a.ws_a[(size_t)b * a.n_max + u] = -1;
      }
    }
  }

  // ---- ticket: the last CTA of the request runs phase B ----
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(&a.ws_ticket[b], 1);
    s_last = prev == n_cta * C - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int st = *(volatile int32_t*)&a.status[b];
  if (!n_ok || st != 0) {
    clear_request(a, b);
    return;
  }
  int32_t* path = a.path + (size_t)b * a.n_max;
  int32_t* emit = a.emitted + (size_t)b * a.n_max;
  if constexpr (MODE == 0) {
    // greedy: match bit of v = (v is the root) or tokens[v] == argmax(row parent(v));
    // a node is ok when every ancestor-or-self matches; pick the deepest ok node.
    const int W = a.W;
    for (int w = threadIdx.x; w < W; w += blockDim.x) s_match[w] = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_kids[i] = __ldcg(&a.ws_a[(size_t)b * a.n_max + i]);
    __syncthreads();
    for (int v = threadIdx.x; v < n; v += blockDim.x) {
      const int p = a.parent[off + v];
      const bool mt = v == 0 || a.tokens[off + v] == s_kids[p];
      if (mt) atomicOr(reinterpret_cast<unsigned long long*>(&s_match[v >> 6]), 1ull << (v & 63));
    }
    __syncthreads();
    int best = -1;
    for (int v = threadIdx.x; v < n; v += blockDim.x) {
      bool ok = true;
      for (int w = 0; w < W; ++w) ok &= (a.mask[(size_t)(off + v) * W + w] & ~s_match[w]) == 0;
      if (ok) best = max(best, (a.depth[off + v] << 11) | (2047 - v));
    }
    // block max of the key
    {
      int v = best;
#pragma unroll
      for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
      __syncthreads();
      if ((threadIdx.x & 31) == 0) red.i[threadIdx.x >> 5] = v;
      __syncthreads();
      if (threadIdx.x == 0) {
        int m = red.i[0];
        for (int k2 = 1; k2 < (int)(blockDim.x >> 5); ++k2) m = max(m, red.i[k2]);
        s_flag = m;
      }
      __syncthreads();
    }
    const int f = 2047 - (s_flag & 2047);
    const int L = (s_flag >> 11) + 1;
    const uint64_t* frow = a.mask + (size_t)(off + f) * W;
    for (int v = threadIdx.x; v < a.n_max; v += blockDim.x) {
      if (v < n && ((frow[v >> 6] >> (v & 63)) & 1ull)) {
        int idx = 0;
        for (int w = 0; w < (v >> 6); ++w) idx += __popcll(frow[w]);
        idx += __popcll(frow[v >> 6] & ((1ull << (v & 63)) - 1ull));
        path[idx] = v;
        if (idx >= 1) emit[idx - 1] = a.tokens[off + v];
      }
      if (v >= L) {
        path[v] = -1;
        emit[v] = -1;
      }
    }
    if (threadIdx.x == 0) {
      emit[L - 1] = s_kids[f];
      a.accept_len[b] = L;
      a.n_emitted[b] = L;
    }
  } else {
    // stochastic: follow the accepted-child links from the root
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_kids[i] = __ldcg(&a.ws_a[(size_t)b * a.n_max + i]);
    __syncthreads();
    if (threadIdx.x == 0) {
      int v = 0, L = 1;
      path[0] = 0;
      while (s_kids[v] > v && L < n) {  // accepted children have larger indices: the walk ends
        v = s_kids[v];
        emit[L - 1] = a.tokens[off + v];
        path[L++] = v;
      }
      emit[L - 1] = __ldcg(&a.ws_s[(size_t)b * a.n_max + v]);
      s_flag = L;
      a.accept_len[b] = L;
      a.n_emitted[b] = L;
    }
    __syncthreads();
    for (int i = s_flag + threadIdx.x; i < a.n_max; i += blockDim.x) {
      path[i] = -1;
      emit[i] = -1;
    }
  }
  if (threadIdx.x == 0) a.ws_ticket[b] = 0;
}

inline size_t ws_layout(int B, int n_max, size_t* off_s, size_t* off_t) {
  const size_t na = (size_t)B * n_max * sizeof(int32_t);
  *off_s = (na + 255) & ~(size_t)255;
  *off_t = (*off_s + na + 255) & ~(size_t)255;
  return *off_t + (size_t)B * sizeof(int32_t);
}

template <int MODE, int C>
cudaError_t launch_verify(const VerifyArgs& a, int B, cudaStream_t stream) {
  auto kern = verify_kernel<MODE, C>;
  const size_t dyn = MODE == 1 ? (size_t)((a.slice + 3) & ~3) * sizeof(float) : 0;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * C), (unsigned)a.n_max, 1);
  cfg.blockDim = dim3(VCfg<MODE>::threads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int MODE>
spec_status verify_dispatch(VerifyArgs a, int B, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  size_t off_s, off_t;
  const size_t need = ws_layout(B, a.n_max, &off_s, &off_t);
  if (!workspace || ws_bytes < need) return SPEC_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  a.ws_a = reinterpret_cast<int32_t*>(ws);
  a.ws_s = reinterpret_cast<int32_t*>(ws + off_s);
  a.ws_ticket = reinterpret_cast<int32_t*>(ws + off_t);
  a.W = (a.n_max + 63) / 64;
  // cluster size: slices of kSlice entries, at most 8 CTAs (wider slices beyond)
  constexpr int kSlice = VCfg<MODE>::slice;
  int C = (a.V + kSlice - 1) / kSlice;
  C = C <= 1 ? 1 : C <= 2 ? 2 : C <= 4 ? 4 : 8;
  a.slice = (((a.V + C - 1) / C) + 3) & ~3;
  if (cudaMemsetAsync(a.ws_ticket, 0, (size_t)B * sizeof(int32_t), stream) != cudaSuccess) return SPEC_ERR_CUDA;
  cudaError_t e;
  switch (C) {
    case 1: e = launch_verify<MODE, 1>(a, B, stream); break;
    case 2: e = launch_verify<MODE, 2>(a, B, stream); break;
    case 4: e = launch_verify<MODE, 4>(a, B, stream); break;
    default: e = launch_verify<MODE, 8>(a, B, stream); break;
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Scratch of spec_tree_verify_stochastic_noalloc: a file-scope device array
// (every GPU that loads the library holds it until the process exits).  Host
// code must not hand the symbol itself to a kernel: it names a host-side
// stand-in, so the device address is looked up per device.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocBytes = (size_t)2 * 1024 * 1024 + 64 * 1024 + 512;  // B*n_max <= 2^18, B <= 2^14
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

static std::mutex g_noalloc_mutex;
static void* g_noalloc_ptr[128];

// Device address of the scratch array on the current device, looked up once
// per device; NULL if the lookup failed.
static void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace spectree

using namespace spectree;

extern "C" {

size_t spec_verify_workspace_size(int B, int n_max, int V) {
  (void)V;
  if (B <= 0 || n_max <= 0) return 256;
  size_t off_s, off_t;
  return ws_layout(B, n_max, &off_s, &off_t);
}

static spec_status verify_check(int B, int n_max, int V) {
  if (B < 0 || n_max < 0 || V <= 0) return SPEC_ERR_INVALID_ARG;
  if (n_max > SPEC_MAX_NODES || V > SPEC_MAX_VOCAB || B > (1 << 27)) return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

spec_status spec_tree_verify_greedy(const float* p_logits, const int32_t* tokens, const int32_t* parent,
                                    const int32_t* tree_off, const uint64_t* mask, const int32_t* depth, int B,
                                    int n_max, int V, int32_t* path, int32_t* accept_len, int32_t* emitted,
                                    int32_t* n_emitted, void* workspace, size_t workspace_bytes, int32_t* status,
                                    void* stream) {
  spec_status s = verify_check(B, n_max, V);
  if (s != SPEC_OK) return s;
  if (B == 0 || n_max == 0) return SPEC_OK;
  if (!p_logits || !tokens || !parent || !tree_off || !mask || !depth || !path || !accept_len || !emitted ||
      !n_emitted || !status)
    return SPEC_ERR_INVALID_ARG;
  VerifyArgs a = {};
  a.p_logits = p_logits;
  a.tokens = tokens;
  a.parent = parent;
  a.tree_off = tree_off;
  a.mask = mask;
  a.depth = depth;
  a.n_max = n_max;
  a.V = V;
  a.path = path;
  a.accept_len = accept_len;
  a.emitted = emitted;
  a.n_emitted = n_emitted;
  a.status = status;
  return verify_dispatch<0>(a, B, workspace, workspace_bytes, (cudaStream_t)stream);
}

spec_status spec_tree_verify_stochastic(const float* p_logits, const float* q_probs, const int32_t* tokens,
                                        const int32_t* parent, const int32_t* tree_off, const uint32_t* uniforms,
                                        int B, int n_max, int V, int32_t* path, int32_t* accept_len,
                                        int32_t* emitted, int32_t* n_emitted, void* workspace,
                                        size_t workspace_bytes, int32_t* status, void* stream) {
  spec_status s = verify_check(B, n_max, V);
  if (s != SPEC_OK) return s;
  if (B == 0 || n_max == 0) return SPEC_OK;
  if (!p_logits || !q_probs || !tokens || !parent || !tree_off || !uniforms || !path || !accept_len || !emitted ||
      !n_emitted || !status)
    return SPEC_ERR_INVALID_ARG;
  VerifyArgs a = {};
  a.p_logits = p_logits;
  a.q_probs = q_probs;
  a.tokens = tokens;
  a.parent = parent;
  a.tree_off = tree_off;
  a.uniforms = reinterpret_cast<const uint2*>(uniforms);
  a.n_max = n_max;
  a.V = V;
  a.path = path;
  a.accept_len = accept_len;
  a.emitted = emitted;
  a.n_emitted = n_emitted;
  a.status = status;
  return verify_dispatch<1>(a, B, workspace, workspace_bytes, (cudaStream_t)stream);
}


// Stochastic verification without a workspace argument: for callers that
// cannot allocate device memory when they verify (a host framework that hands
// the library only its inputs and outputs, or a latency-critical loop that
// must not pay cudaMalloc's implicit device synchronisation).  The scratch is
// a fixed device array shared by every call: concurrent calls on different
// streams race, and the first call on each device looks up its address.
spec_status spec_tree_verify_stochastic_noalloc(const float* p_logits, const float* q_probs, const int32_t* tokens,
                                                const int32_t* parent, const int32_t* tree_off,
                                                const uint32_t* uniforms, int B, int n_max, int V, int32_t* path,
                                                int32_t* accept_len, int32_t* emitted, int32_t* n_emitted,
                                                int32_t* status, void* stream) {
  spec_status s = verify_check(B, n_max, V);
  if (s != SPEC_OK) return s;
  if (B == 0 || n_max == 0) return SPEC_OK;
  if (B > (1 << 14) || (long long)B * n_max > (1LL << 18)) return SPEC_ERR_UNSUPPORTED;
  size_t off_s, off_t;
  if (ws_layout(B, n_max, &off_s, &off_t) > kNoAllocBytes) return SPEC_ERR_UNSUPPORTED;
  void* ws = noalloc_scratch();
  if (!ws) return SPEC_ERR_CUDA;
  return spec_tree_verify_stochastic(p_logits, q_probs, tokens, parent, tree_off, uniforms, B, n_max, V, path,
                                     accept_len, emitted, n_emitted, ws, kNoAllocBytes, status, stream);
}

}  // extern "C"
