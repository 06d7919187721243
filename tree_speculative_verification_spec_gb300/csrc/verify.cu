// Token-tree verification, greedy and stochastic: one launch, one
// thread-block cluster per request, walking the request's tree from the root.
//
// "SpecInfer Guide", "Greedy Verification Algorithm" and "Stochastic
// Verification Algorithm": verification starts at the root (the last
// verified token), tests the children of the current node against the
// target's row of that node and moves into the accepted child.  Only the
// rows of nodes the walk reaches are read: the target row of every node on
// the accepted path, the draft row of a node where a child was rejected.
//
// The C CTAs of a cluster split the vocabulary into C slices.  Each row
// reduction (max, argmax, fixed-point sums, the exclusive prefix of the final
// sample) is a block reduction followed by one push of the CTA's value into
// every peer's shared memory (st.async, completing on the peer's mbarrier):
// one one-way trip, no cluster barrier.  Every CTA takes
// the same decisions: they depend only on cluster-reduced values and on
// single entries (a child's logit and draft probability) that each CTA reads
// and evaluates itself.  While a node is processed, the row slices its
// children would need next are prefetched into L2.  No CTA waits for a CTA of
// another cluster.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace spectree {

constexpr int kWalkThreads = 512;
constexpr int kMaxSlice = 16384;  // stochastic: floats of one CTA's slice (target, two draft: 192 KB)
constexpr int kMaxCluster = 16;   // 16 needs the non-portable cluster size
constexpr int kTargetCtas = 152;  // one CTA per SM when the batch is small

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
// A and B stay below 2^32 for up to 511 terms (a thread adds at most 48 here);
// values above 1 take fx().
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
  // moves A and B into the 64-bit total (callers adding more than 511 terms)
  __device__ __forceinline__ void flush() {
    big = total();
    a = 0;
    b = 0;
  }
};

__device__ __forceinline__ float z_of(unsigned long long S) { return __fmul_rn(__ull2float_rn(S), 0x1p-46f); }

// floor(U * S / 2^32), exact for U < 2^32, S < 2^64.
__device__ __forceinline__ unsigned long long sample_target(uint32_t U, unsigned long long S) {
  const unsigned long long lo = (unsigned long long)U * (S & 0xffffffffull);
  const unsigned long long hi = (unsigned long long)U * (S >> 32);
  return hi + (lo >> 32);
}

// residual step: max(r - q, 0) written as a comparison (no fmax sign-of-zero
// ambiguity).  A zero weight (every weight the previous steps clamped) skips
// the division: +0 / Z is +0 for the finite positive Z, the same value.
__device__ __forceinline__ float resid(float d, float Z, float q) {
  const float r = d == 0.0f ? 0.0f : __fdiv_rn(d, Z);
  const float diff = __fsub_rn(r, q);
  return diff > 0.0f ? diff : 0.0f;
}

// d / Z rounded to nearest even for the weights of a residual pass, by
// Markstein's division theorem: with y = RN(1/Z) and q = RN(d * y), the
// remainder r = d - q * Z is exact in one FMA and RN(q + r * y) = RN(d / Z),
// as long as nothing underflows or overflows.  Here Z in [2^-46, 2^17] and the
// fast path takes d in [2^-100, 1], so every quantity is a normal number;
// other d take the IEEE division.  Bit-identical to resid().
__device__ __noinline__ float div_ieee(float d, float Z) { return __fdiv_rn(d, Z); }

__device__ __forceinline__ float resid_y(float d, float Z, float y, float q) {
  float r;
  if (d >= 0x1p-100f && d <= 1.0f) {
    const float q0 = __fmul_rn(d, y);
    const float rem = fmaf(-q0, Z, d);
    r = fmaf(rem, y, q0);
  } else if (d == 0.0f) {
    r = 0.0f;
  } else {
    r = div_ieee(d, Z);  // a call: never evaluated speculatively
  }
  const float diff = __fsub_rn(r, q);
  return diff > 0.0f ? diff : 0.0f;
}

// Two entries at once: the same single IEEE operations on the f32x2 pipe
// (fma.f32x2 is two fused multiply-adds; a - b is a + (-b)), so each lane is
// bit-identical to the scalar functions above.
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }

// The rint step takes scalar operations: a paired multiply whose only use is a
// paired add can be fused into one f32x2 fused multiply-add (rint of the
// unrounded product, which differs where the rounded product x log2 e is a
// half-integer), while the scalar _rn operations are never fused.
__device__ __forceinline__ float2 canon_exp2(float2 x) {
  const float2 big = make_float2(__fadd_rn(__fmul_rn(x.x, 0x1.715476p+0f), 12582912.0f),
                                 __fadd_rn(__fmul_rn(x.y, 0x1.715476p+0f), 12582912.0f));
  const float2 n = __fadd2_rn(big, f2(-12582912.0f));
  const int nx = __float_as_int(big.x) - 0x4B400000, ny = __float_as_int(big.y) - 0x4B400000;
  const float2 nn = neg2(n);
  float2 r = __ffma2_rn(nn, f2(0x1.62e4p-1f), x);
  r = __ffma2_rn(nn, f2(0x1.7f7d1cp-20f), r);
  float2 p = f2(0x1.a01a02p-13f);
  p = __ffma2_rn(p, r, f2(0x1.6c16c2p-10f));
  p = __ffma2_rn(p, r, f2(0x1.111112p-7f));
  p = __ffma2_rn(p, r, f2(0x1.555556p-5f));
  p = __ffma2_rn(p, r, f2(0x1.555556p-3f));
  p = __ffma2_rn(p, r, f2(0.5f));
  p = __ffma2_rn(p, r, f2(1.0f));
  p = __ffma2_rn(p, r, f2(1.0f));
  // below -87 (or NaN) the scale bits are meaningless: the result is selected away
  float2 e = __fmul2_rn(p, make_float2(__int_as_float((nx + 127) << 23), __int_as_float((ny + 127) << 23)));
  e.x = x.x >= -87.0f ? e.x : 0.0f;
  e.y = x.y >= -87.0f ? e.y : 0.0f;
  return e;
}

__device__ __forceinline__ void fx_add2(FxSum& acc, float2 v) {
  if (v.x <= 1.0f && v.y <= 1.0f) {
    const float2 y1 = __fmul2_rn(v, f2(0x1p23f));
    const float2 t = __fadd2_rz(y1, f2(0x1p23f));
    const float2 f = __fadd2_rn(y1, neg2(__fadd2_rn(t, f2(-0x1p23f))));
    const float2 t2 = __fadd2_rz(__fmul2_rn(f, f2(0x1p23f)), f2(0x1p23f));
    acc.a += (__float_as_uint(t.x) - 0x4B000000u) + (__float_as_uint(t.y) - 0x4B000000u);
    acc.b += (__float_as_uint(t2.x) - 0x4B000000u) + (__float_as_uint(t2.y) - 0x4B000000u);
  } else {
    acc.add(v.x);
    acc.add(v.y);
  }
}

__device__ __forceinline__ float2 resid_y2(float2 d, float Z, float y, float2 q) {
  float2 r;
  if (d.x >= 0x1p-100f && d.x <= 1.0f && d.y >= 0x1p-100f && d.y <= 1.0f) {
    const float2 q0 = __fmul2_rn(d, f2(y));
    const float2 rem = __ffma2_rn(neg2(q0), f2(Z), d);
    r = __ffma2_rn(rem, f2(y), q0);
    const float2 diff = __fadd2_rn(r, neg2(q));
    return make_float2(diff.x > 0.0f ? diff.x : 0.0f, diff.y > 0.0f ? diff.y : 0.0f);
  }
  return make_float2(resid_y(d.x, Z, y, q.x), resid_y(d.y, Z, y, q.y));
}

// ---------------------------------------------------------------------------
// Block reductions
// ---------------------------------------------------------------------------

constexpr int kWarps = kWalkThreads / 32;

struct Red {
  float f[kWarps];
  int i[kWarps];
  unsigned long long u[kWarps];
};

__device__ __forceinline__ float block_max(float v, Red& s) {
  v = warp_max_f(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) s.f[w] = v;
  __syncthreads();
  v = s.f[0];
  for (int k = 1; k < kWarps; ++k) v = fmaxf(v, s.f[k]);
  return v;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, Red& s) {
  v = warp_sum_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) s.u[w] = v;
  __syncthreads();
  v = 0;
  for (int k = 0; k < kWarps; ++k) v += s.u[k];
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
  for (int k = 1; k < kWarps; ++k) argmax_combine(v, i, s.f[k], s.i[k]);
}

// ---------------------------------------------------------------------------
// Cluster exchange: every CTA pushes one 8-byte value into slot [k & 1][rank]
// of every CTA of the cluster (st.async to distributed shared memory,
// completing on the receiver's mbarrier of that slot), then waits on its own
// mbarrier for the C values of exchange k.  One one-way trip instead of a
// cluster barrier.  Slot reuse is safe: a CTA pushes exchange k + 2 only after
// finishing exchange k + 1, which needs every peer's push of k + 1, which each
// peer makes after reading its slots of exchange k (a block reduction with
// __syncthreads separates the reads from the next push).
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(const uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < (1u << 26); ++i)
    if (mbar_try(a, parity)) return true;
  return false;
}

struct Exch {
  uint64_t bar[2];
  unsigned long long v[2][kMaxCluster];
};

template <int C>
__device__ __forceinline__ const unsigned long long* exchange(unsigned long long val, Exch& ex, int& k, int rank,
                                                              int32_t* status) {
  const int s = k & 1;
  const uint32_t parity = (uint32_t)(k >> 1) & 1u;
  ++k;
  // lane r of warp 0 pushes to rank r; a push that lands before this CTA's
  // expect_tx only drives the transaction count below zero for a moment: the
  // phase cannot complete before the local arrive below.
  if (threadIdx.x < C) {
    const uint32_t lbar = smem_addr(&ex.bar[s]), lslot = smem_addr(&ex.v[s][rank]);
    if (threadIdx.x == 0)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(lbar), "r"((uint32_t)(C * 8))
                   : "memory");
    uint32_t rs, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rs) : "r"(lslot), "r"((uint32_t)threadIdx.x));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(lbar), "r"((uint32_t)threadIdx.x));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(rs), "l"(val),
                 "r"(rb)
                 : "memory");
  }
  if (!mbar_wait_bounded(&ex.bar[s], parity) && threadIdx.x == 0) atomicOr(status, SPEC_DEV_TIMEOUT);
  return ex.v[s];
}

template <int C>
__device__ __forceinline__ float cluster_max(float v, Red& red, Exch& ex, int& k, int rank, int32_t* status) {
  v = block_max(v, red);
  if constexpr (C == 1) return v;
  const unsigned long long* x = exchange<C>((unsigned long long)__float_as_uint(v), ex, k, rank, status);
  float m = __uint_as_float((uint32_t)x[0]);
#pragma unroll
  for (int r = 1; r < C; ++r) m = fmaxf(m, __uint_as_float((uint32_t)x[r]));
  return m;
}

// Cluster total of per-thread values; `cta` receives this CTA's total.
template <int C>
__device__ __forceinline__ unsigned long long cluster_sum(unsigned long long v, Red& red, Exch& ex, int& k, int rank,
                                                          int32_t* status, unsigned long long& cta) {
  v = block_sum_u64(v, red);
  cta = v;
  if constexpr (C == 1) return v;
  const unsigned long long* x = exchange<C>(v, ex, k, rank, status);
  unsigned long long t = 0;
#pragma unroll
  for (int r = 0; r < C; ++r) t += x[r];
  return t;
}

// Exclusive prefix over the ranks below this CTA of a CTA-uniform value.
template <int C>
__device__ __forceinline__ unsigned long long cluster_prefix(unsigned long long v, Exch& ex, int& k, int rank,
                                                             int32_t* status) {
  if constexpr (C == 1) return 0ull;
  __syncthreads();  // every thread has read the slots of the previous exchange
  const unsigned long long* x = exchange<C>(v, ex, k, rank, status);
  unsigned long long t = 0;
  for (int r = 0; r < rank; ++r) t += x[r];
  return t;
}

template <int C>
__device__ __forceinline__ void cluster_argmax(float& v, int& i, Red& red, Exch& ex, int& k, int rank,
                                               int32_t* status) {
  block_argmax(v, i, red);
  if constexpr (C == 1) return;
  const unsigned long long x0 = ((unsigned long long)__float_as_uint(v) << 32) | (uint32_t)i;
  const unsigned long long* x = exchange<C>(x0, ex, k, rank, status);
#pragma unroll
  for (int r = 0; r < C; ++r) argmax_combine(v, i, __uint_as_float((uint32_t)(x[r] >> 32)), (int)(uint32_t)x[r]);
}

// ---------------------------------------------------------------------------
// Walk helpers
// ---------------------------------------------------------------------------

// Row statistics of one node's target row under the arithmetic contract:
// m = max l and S = sum FX(E(l - m)) (exact).
struct RowStats {
  float m;
  uint32_t pad;
  unsigned long long S;
};

struct VerifyArgs {
  const float* p_logits;
  const float* q_probs;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* tree_off;
  const uint2* uniforms;
  int n_max, V, slice;
  int vec;  // V % 4 == 0 and 16-byte aligned rows: float4 passes, bulk copies, L2 prefetch
  int32_t* path;
  int32_t* accept_len;
  int32_t* emitted;
  int32_t* n_emitted;
  int32_t* status;
  const RowStats* stats;  // stochastic: every node's row statistics, or null (the walk computes them)
  const float* inv_temp;  // stochastic: per-request inverse temperature, or null (1)
  int q_per_child;        // stochastic: q_probs row c is child c's own draft row (else row u serves u's children)
  int ahead;              // stochastic without statistics: a fourth slice receives the first child's target slice
};

// A request's inverse temperature tau (1 without an array); usable iff
// finite and positive.
__device__ __forceinline__ float request_tau(const VerifyArgs& a, int b) { return a.inv_temp ? a.inv_temp[b] : 1.0f; }
__device__ __forceinline__ bool tau_ok(float t) { return t > 0.0f && t <= 3.402823466e38f; }

struct WalkShared {
  Red red;
  Exch ex;
  uint64_t dbar, qbar[2];       // stochastic: slice copies of the target and draft rows
  uint64_t nbar;                // stochastic: the copy of the first child's target slice
  int32_t par[SPEC_MAX_NODES];  // the request's parent array
  int32_t tok[SPEC_MAX_NODES];  // the request's tokens
  int32_t aux[SPEC_MAX_NODES];  // greedy: argmax of frontier nodes; stochastic: the path
  union {
    struct {
      int32_t fr[SPEC_MAX_NODES];   // frontier
      int32_t nx[SPEC_MAX_NODES];   // next frontier
      int32_t inf[SPEC_MAX_NODES];  // 1 for frontier nodes
    } g;
    struct {
      int32_t kids[SPEC_MAX_NODES];  // children of the node, increasing
      float z[SPEC_MAX_NODES];       // normaliser before each residual step at the node
      float cx[SPEC_MAX_NODES];      // the node's logit at each child's token
      float cq[SPEC_MAX_NODES];      // the node's draft probability at each child's token
      uint32_t cu[SPEC_MAX_NODES];   // each child's acceptance word
    } s;
  };
  uint32_t uterm;  // stochastic: the node's sampling word
  int cnt, flag;
  unsigned long long wsum[kWarps];
};

// Ordered compaction by warp 0 of the c in [lo, hi) with pred(c) into out[]
// (increasing c); every thread gets the count (one __syncthreads).
template <class Pred>
__device__ int compact(int lo, int hi, Pred pred, int32_t* out, WalkShared& sh) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int cnt = 0;
    for (int base = lo; base < hi; base += 32) {
      const int c = base + lane;
      const bool is = c < hi && pred(c);
      const unsigned m = __ballot_sync(0xffffffffu, is);
      if (is) out[cnt + __popc(m & ((1u << lane) - 1u))] = c;
      cnt += __popc(m);
    }
    if (lane == 0) sh.cnt = cnt;
  }
  __syncthreads();
  return sh.cnt;
}

// L2 prefetch of [p, p + bytes): 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  if (bytes == 0) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Thread 0 starts a bulk copy global -> shared of `bytes` completing on `bar`.
// The caller has made every earlier access to dst complete (__syncthreads
// after a proxy fence) and waits with wait_copy before reading dst.
__device__ __forceinline__ void start_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bounded wait for a copy; on expiry SPEC_DEV_TIMEOUT is set and the copy is
// waited for once more (it must land before the buffer is reused).
__device__ __forceinline__ void wait_copy(uint64_t* bar, uint32_t& phase, int32_t* status) {
  if (!mbar_wait_bounded(bar, phase)) {
    if (threadIdx.x == 0) atomicOr(status, SPEC_DEV_TIMEOUT);
    mbar_wait_bounded(bar, phase);
  }
  phase ^= 1u;
}

// Wait for the draft copy into buffer i (bit i of the phase and pending masks).
__device__ __forceinline__ void wait_draft(WalkShared& sh, int i, uint32_t& phase, uint32_t& pend, int32_t* status) {
  uint32_t p = (phase >> i) & 1u;
  wait_copy(&sh.qbar[i], p, status);
  phase ^= 1u << i;
  pend &= ~(1u << i);
}

__device__ void clear_request(const VerifyArgs& a, int b) {
  for (int i = threadIdx.x; i < a.n_max; i += kWalkThreads) {
    a.path[(size_t)b * a.n_max + i] = -1;
    a.emitted[(size_t)b * a.n_max + i] = -1;
  }
  if (threadIdx.x == 0) {
    a.accept_len[b] = 0;
    a.n_emitted[b] = 0;
  }
}

// ---------------------------------------------------------------------------
// Row statistics of every node, one CTA per (request, node), data-parallel
// over the whole GPU: for large batches the walk then enters an accepted node
// with a few shared-memory reads instead of two passes over the node's row.
// The same contract operations as the walk's own passes, so m and S are
// bit-identical to what the walk would compute.  512 threads per CTA, each
// issuing batches of four 16-byte loads before using any, so that a few rows
// are resident per SM and one row's loads overlap another's arithmetic; the
// second pass reads the row again from L2.
// ---------------------------------------------------------------------------
constexpr int kStatsThreads = 512;
constexpr int kStatsWarps = kStatsThreads / 32;

__global__ void __launch_bounds__(kStatsThreads) row_stats_kernel(VerifyArgs a, RowStats* stats) {
  __shared__ float smax[kStatsWarps];
  __shared__ unsigned long long ssum[kStatsWarps];
  // Launched as a programmatic dependent of the previous kernel (whose
  // outputs it does not read): every CTA waits for that kernel before it
  // exits, so the walk after this grid finds that kernel's results too.
  struct WaitOnExit {
    __device__ ~WaitOnExit() {
      if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    }
  } wait_on_exit;
  const int b = blockIdx.x / a.n_max, u = blockIdx.x % a.n_max;
  const int off = a.tree_off[b];
  const int n = a.tree_off[b + 1] - off;
  if (n < 1 || n > a.n_max || u >= n) return;  // uniform across the CTA
  const float tau = request_tau(a, b);
  if (!tau_ok(tau)) return;  // the walk flags the request
  const float2 tau2 = f2(tau);
  const int V = a.V, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* row = a.p_logits + (size_t)(off + u) * V;
  const float4* r4 = reinterpret_cast<const float4*>(row);
  float lmax = -INFINITY;
  if (a.vec) {
    constexpr int kB = 4;  // 16-byte loads per thread issued before any is used
    const int n4 = V >> 2;
    for (int j0 = threadIdx.x; j0 < n4; j0 += kB * kStatsThreads) {
      float4 v[kB];
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int j = j0 + q * kStatsThreads;
        v[q] = j < n4 ? __ldg(r4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int q = 0; q < kB; ++q) lmax = fmaxf(lmax, fmaxf(fmaxf(v[q].x, v[q].y), fmaxf(v[q].z, v[q].w)));
    }
  } else {
    for (int j = threadIdx.x; j < V; j += kStatsThreads) lmax = fmaxf(lmax, __ldg(row + j));
  }
  lmax = warp_max_f(lmax);
  if (lane == 0) smax[w] = lmax;
  __syncthreads();
  float m = smax[0];
#pragma unroll
  for (int k = 1; k < kStatsWarps; ++k) m = fmaxf(m, smax[k]);
  unsigned long long part;
  if (a.vec) {
    FxSum acc;
    constexpr int kB = 4;
    const int n4 = V >> 2;
    for (int j0 = threadIdx.x; j0 < n4; j0 += kB * kStatsThreads) {
      float4 v[kB];
      bool in[kB];
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int j = j0 + q * kStatsThreads;
        in[q] = j < n4;
        v[q] = in[q] ? __ldg(r4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        if (in[q]) {
          fx_add2(acc, canon_exp2(__fmul2_rn(__fadd2_rn(make_float2(v[q].x, v[q].y), f2(-m)), tau2)));
          fx_add2(acc, canon_exp2(__fmul2_rn(__fadd2_rn(make_float2(v[q].z, v[q].w), f2(-m)), tau2)));
        }
      }
      acc.flush();  // 16 terms per batch: A and B stay below 2^32
    }
    part = acc.total();
  } else {
    part = 0;
    for (int j = threadIdx.x; j < V; j += kStatsThreads)
      part += fx(canon_exp(__fmul_rn(__fsub_rn(__ldg(row + j), m), tau)));
  }
  part = warp_sum_u64(part);
  if (lane == 0) ssum[w] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long S = 0;
#pragma unroll
    for (int k = 0; k < kStatsWarps; ++k) S += ssum[k];
    RowStats r;
    r.m = m;
    r.pad = 0;
    r.S = S;
    stats[off + u] = r;
  }
}

// ---------------------------------------------------------------------------
// The walk
// ---------------------------------------------------------------------------

// LEAN: a stochastic walk without row statistics and with per-parent draft
// rows, its most common form, compiled without the code of the other two
// (one launch runs each code region only a few times, so instruction fetch
// shows: decode layer 22.0 -> 21.1 us, wide ensemble 38.7 -> 37.4 us).  The
// greedy walk has one form.
template <int MODE, int C, bool LEAN>
__global__ void __launch_bounds__(kWalkThreads, 1) verify_walk_kernel(VerifyArgs a) {
  extern __shared__ float4 dyn_smem[];
  __shared__ WalkShared sh;

  const int rank = (int)(blockIdx.x % C);
  const int b = (int)(blockIdx.x / C);
  const int off = a.tree_off[b];
  const int n = a.tree_off[b + 1] - off;
  const int V = a.V;
  const int x0 = min(V, rank * a.slice);
  const int len = min(V, x0 + a.slice) - x0;
  const bool vec = a.vec != 0;
  int32_t* status = &a.status[b];
  int xk = 0;  // exchange counter
  constexpr int kOwnBits = SPEC_DEV_BAD_TOKEN | SPEC_DEV_BAD_TREE | SPEC_DEV_BAD_TEMP;
  const float tau = MODE == 1 ? request_tau(a, b) : 1.0f;
  // The status word comes from the kernels before this one (this kernel is
  // launched as their programmatic dependent and may start before the last
  // of them ends): it is read only after griddepcontrol.wait below.  Until
  // then the walk's own inputs are checked and the root's slice copied.
  const bool may_run = n >= 1 && n <= a.n_max && tau_ok(tau);

  // stochastic: the root's target slice is copied while the inputs are checked
  float* D = reinterpret_cast<float*>(dyn_smem);  // current weights of this CTA's slice
  float* Qb = D + a.slice;                         // draft slices, alternating per node
  uint32_t dphase = 0;
  uint32_t qphase = 0, qpend = 0;  // per draft buffer i (bit i): phase, copy not yet waited for
  const bool root_copy = MODE == 1 && may_run && vec && len > 0;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sh.ex.bar[0])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sh.ex.bar[1])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sh.dbar)) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sh.qbar[0])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sh.qbar[1])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sh.nbar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (root_copy) start_copy(D, a.p_logits + (size_t)off * V + x0, (uint32_t)len * 4, &sh.dbar);
    else if (MODE == 0 && may_run && vec) prefetch_l2(a.p_logits + (size_t)off * V + x0, (uint32_t)len * 4);
  }
  // Peers push into this CTA's exchange slots only after the cluster barrier
  // completes (the mbarriers are initialised); it completes while the inputs
  // are checked.
  if constexpr (C > 1) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  // The tree, token and temperature checks are made by every CTA from the
  // inputs; the only status bits this kernel sets are those checks' (by rank
  // 0, when every CTA of the cluster skips the walk), so ignoring them in the
  // incoming status keeps the decision uniform.
  int bad;
  {
    const int nc = min(max(n, 0), a.n_max);  // nodes whose entries are checked
    bool bt = false, bp = n < 0 || n > a.n_max;
    for (int i = threadIdx.x; i < nc; i += kWalkThreads) {
      const int t = a.tokens[off + i], p = a.parent[off + i];
      sh.tok[i] = t;
      sh.par[i] = p;
      bt |= (unsigned)t >= (unsigned)V;
      bp |= i == 0 ? p != -1 : (p < 0 || p >= i);
    }
    bad = (__syncthreads_or(bt) ? SPEC_DEV_BAD_TOKEN : 0) | (__syncthreads_or(bp) ? SPEC_DEV_BAD_TREE : 0) |
          (tau_ok(tau) ? 0 : SPEC_DEV_BAD_TEMP);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int st_in = *(volatile int32_t*)status;
  // a request flagged upstream is skipped without this kernel's own checks
  if ((st_in & ~kOwnBits) != 0) bad = 0;
  const bool skip = (st_in & ~kOwnBits) != 0 || bad != 0 || n == 0;
  if constexpr (C > 1) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  __syncthreads();
  if (skip) {
    if (root_copy) wait_copy(&sh.dbar, dphase, status);  // the copy lands before the CTA leaves
    if (rank == 0) {
      clear_request(a, b);
      if (bad && threadIdx.x == 0) atomicOr(status, bad);
    }
    return;  // uniform across the cluster; nothing was exchanged
  }
  int32_t* out_path = a.path + (size_t)b * a.n_max;
  int32_t* out_emit = a.emitted + (size_t)b * a.n_max;

  if constexpr (MODE == 0) {
    // ---------------------------------------------------------------- greedy
    // Level by level: the frontier holds every node of the current depth whose
    // root path follows the argmax chain (several when siblings repeat a
    // token).  Row argmaxes of the frontier, then the next frontier = children
    // whose token equals their parent's argmax.  The accepted node is the
    // lowest-index node of the deepest non-empty frontier.
    int32_t* fr = sh.g.fr;  // frontier
    int32_t* nx = sh.g.nx;  // next frontier
    int32_t* inf = sh.g.inf;
    for (int i = threadIdx.x; i < n; i += kWalkThreads) inf[i] = i == 0;
    if (threadIdx.x == 0) fr[0] = 0;
    int nf = 1, depth = 0;
    __syncthreads();
    for (;;) {
      // warp 0: L2 prefetch of the frontier's children's slices
      if (vec && threadIdx.x < 32)
        for (int c = 1 + (int)threadIdx.x; c < n; c += 32)
          if (inf[sh.par[c]]) prefetch_l2(a.p_logits + (size_t)(off + c) * V + x0, (uint32_t)len * 4);
      for (int i = 0; i < nf; ++i) {
        const int u = fr[i];
        const float* prow = a.p_logits + (size_t)(off + u) * V + x0;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        if (vec) {
          const float4* p4 = reinterpret_cast<const float4*>(prow);
          const int n4 = len >> 2;
          for (int j = threadIdx.x; j < n4; j += 8 * kWalkThreads) {
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int jj = j + q * kWalkThreads;
              v[q] = jj < n4 ? __ldcg(p4 + jj) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int x = x0 + ((j + q * kWalkThreads) << 2);
              if (v[q].x > bv) { bv = v[q].x; bi = x; }
              if (v[q].y > bv) { bv = v[q].y; bi = x + 1; }
              if (v[q].z > bv) { bv = v[q].z; bi = x + 2; }
              if (v[q].w > bv) { bv = v[q].w; bi = x + 3; }
            }
          }
        } else {
          for (int j = threadIdx.x; j < len; j += kWalkThreads) {
            const float v = __ldcg(prow + j);
            if (v > bv) { bv = v; bi = x0 + j; }
          }
        }
        cluster_argmax<C>(bv, bi, sh.red, sh.ex, xk, rank, status);
        if (threadIdx.x == 0) sh.aux[u] = bi == 0x7fffffff ? 0 : bi;
      }
      __syncthreads();
      // warp 0: the next frontier in increasing index, and the flags
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int cnt = 0;
        for (int base = 1; base < n; base += 32) {
          const int c = base + lane;
          bool is = false;
          if (c < n) {
            const int p = sh.par[c];
            is = inf[p] && sh.tok[c] == sh.aux[p];
          }
          const unsigned m = __ballot_sync(0xffffffffu, is);
          if (is) nx[cnt + __popc(m & ((1u << lane) - 1u))] = c;
          cnt += __popc(m);
        }
        __syncwarp();
        if (cnt > 0) {
          for (int i = lane; i < nf; i += 32) inf[fr[i]] = 0;
          __syncwarp();
          for (int i = lane; i < cnt; i += 32) inf[nx[i]] = 1;
        }
        if (lane == 0) sh.cnt = cnt;
      }
      __syncthreads();
      const int nn = sh.cnt;
      if (nn == 0) break;
      int32_t* t = fr;
      fr = nx;
      nx = t;
      nf = nn;
      ++depth;
    }
    if (rank == 0 && threadIdx.x == 0) {
      int f = fr[0];
      for (int i = 1; i < nf; ++i) f = min(f, fr[i]);
      const int L = depth + 1;
      out_emit[L - 1] = sh.aux[f];
      for (int i = L - 1, c = f; i >= 0; --i, c = sh.par[c]) {
        out_path[i] = c;
        if (i >= 1) out_emit[i - 1] = sh.tok[c];
      }
      a.accept_len[b] = L;
      a.n_emitted[b] = L;
      sh.flag = L;
    }
    __syncthreads();
    if (rank == 0) {
      const int L = sh.flag;
      for (int i = L + threadIdx.x; i < a.n_max; i += kWalkThreads) {
        out_path[i] = -1;
        out_emit[i] = -1;
      }
    }
  } else {
    // ------------------------------------------------------------ stochastic
    // The passes over the slice are warp-interleaved (thread t takes entries
    // t, t + threads, ..., whole float4 when vec): consecutive lanes touch
    // consecutive shared-memory words.  The fixed-point sums are exact, so
    // their order does not matter; only the final sample scans in index order.
    float4* D4 = reinterpret_cast<float4*>(D);
    const int len4 = len >> 2;
    const bool use_stats = !LEAN && a.stats != nullptr;
    // the copy ahead: at each node the first child's target slice goes into a
    // spare buffer while the node is decided; accepting that child swaps the
    // buffers instead of copying its slice after the decision
    const bool ahead = !use_stats && a.ahead != 0 && vec && len > 0;
    float* Dn = Qb + 2 * a.slice;  // the spare buffer (the fourth slice)
    uint32_t nphase = 0;
    bool npend = false;  // a copy into Dn is in flight (or landed and not yet waited for)
    const bool per_child = !LEAN && a.q_per_child != 0;
    // the draft slice is copied on demand (at a rejection, into buffer 0)
    // with row statistics or per-child rows; otherwise at node entry
    const bool q_lazy = use_stats || per_child;
    const float2 tau2 = f2(tau);
    bool loaded = true;  // D holds the current node's slice (the root's copy is in flight)
    // statistics mode: every node's entries, read once at the start (the
    // second draft buffer's room holds them): its logit and draft
    // probability at its token (rows of its parent), its acceptance word and
    // its row statistics
    float* NX = Qb + a.slice;
    float* NQ = NX + a.n_max;
    uint32_t* NU = reinterpret_cast<uint32_t*>(NQ + a.n_max);
    float* NM = reinterpret_cast<float*>(NU + a.n_max);
    unsigned long long* NS = reinterpret_cast<unsigned long long*>(NM + a.n_max);
    if (use_stats) {
      for (int c = threadIdx.x; c < n; c += kWalkThreads) {
        const int pc = sh.par[c], t = sh.tok[c];
        NX[c] = c > 0 ? __ldcg(a.p_logits + (size_t)(off + pc) * V + t) : 0.0f;
        NQ[c] = c > 0 ? __ldcg(a.q_probs + (size_t)(off + (per_child ? c : pc)) * V + t) : 0.0f;
        NU[c] = a.uniforms[off + c].x;
        const RowStats r = a.stats[off + c];
        NM[c] = r.m;
        NS[c] = r.S;
      }
    }
    if (threadIdx.x == 0) sh.aux[0] = 0;
    int u = 0, L = 1;
    auto load_target = [&](int node) {
      const float* src = a.p_logits + (size_t)(off + node) * V + x0;
      if (vec) {
        if (len > 0) {
          if (threadIdx.x == 0) start_copy(D, src, (uint32_t)len * 4, &sh.dbar);
          wait_copy(&sh.dbar, dphase, status);
        }
      } else {
        for (int j = threadIdx.x; j < len; j += kWalkThreads) D[j] = src[j];
      }
      __syncthreads();
    };
    if (root_copy) wait_copy(&sh.dbar, dphase, status);
    else if (!vec) load_target(0);
    __syncthreads();
    for (;;) {
      const float* prow = a.p_logits + (size_t)(off + u) * V;
      const float* qrow = a.q_probs + (size_t)(off + u) * V;
      // children of u in increasing index; this node's entries at their tokens;
      // the draft slice (needed from the first rejection on) and an L2 prefetch
      // of the children's target slices
      const int k = compact(u + 1, n, [&](int c) { return sh.par[c] == u; }, sh.s.kids, sh);
      // loads in flight through the max and exp passes, stored before the sum
      float rx[2], rq[2];
      uint32_t ru[2];
      uint32_t uterm = 0;
      // the draft slice: per parent without statistics, into the buffer of
      // this node's parity at once (its previous copy, two nodes back, was
      // waited for here or at a rejection); otherwise into buffer 0 at each
      // rejection that needs a row the buffer does not hold
      const int qb = q_lazy ? 0 : (L - 1) & 1;
      float* Q = Qb + qb * a.slice;
      const float4* Q4 = reinterpret_cast<const float4*>(Q);
      int q_row = q_lazy ? -1 : u;  // the row the draft buffer holds (or is receiving)
      if (!use_stats) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int i = threadIdx.x + r * kWalkThreads;
          if (i < k) {
            const int c = sh.s.kids[i];
            const int t = sh.tok[c];
            rx[r] = __ldcg(prow + t);
            rq[r] = __ldcg((per_child ? a.q_probs + (size_t)(off + c) * V : qrow) + t);
            ru[r] = a.uniforms[off + c].x;
            if (vec) prefetch_l2(a.p_logits + (size_t)(off + c) * V + x0, (uint32_t)len * 4);
          }
        }
        if (threadIdx.x == 0) uterm = a.uniforms[off + u].y;
        if (ahead && k > 0) {  // Dn's last readers finished before the barrier that ended the previous node
          if (threadIdx.x == 0)
            start_copy(Dn, a.p_logits + (size_t)(off + sh.s.kids[0]) * V + x0, (uint32_t)len * 4, &sh.nbar);
          npend = true;
        }
        if (!q_lazy) {
          if (qpend & (1u << qb)) wait_draft(sh, qb, qphase, qpend, status);
          if (k > 0 && vec && len > 0) {
            if (threadIdx.x == 0) start_copy(Q, qrow + x0, (uint32_t)len * 4, &sh.qbar[qb]);
            qpend |= 1u << qb;
          }
        }
      }

      // C4: m = max, e = E(l - m), S_0 = sum FX(e); with precomputed row
      // statistics the slice is left alone until a rejection or the sample
      // needs the weights
      float m;
      unsigned long long mp = 0, lt = 0, S;
      bool have_e;  // D holds this node's weights (e, or a residual)
      if (use_stats) {
        m = NM[u];
        S = NS[u];
        have_e = false;
        for (int i = threadIdx.x; i < k; i += kWalkThreads) {
          const int c = sh.s.kids[i];
          sh.s.cx[i] = NX[c];
          sh.s.cq[i] = NQ[c];
          sh.s.cu[i] = NU[c];
        }
        __syncthreads();
      } else {
        float lmax = -INFINITY;
        if (vec) {
#pragma unroll 4
          for (int j = threadIdx.x; j < len4; j += kWalkThreads) {
            const float4 v = D4[j];
            lmax = fmaxf(lmax, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
          }
        } else {
          for (int j = threadIdx.x; j < len; j += kWalkThreads) lmax = fmaxf(lmax, D[j]);
        }
        m = cluster_max<C>(lmax, sh.red, sh.ex, xk, rank, status);
        if (vec) {
          FxSum acc;
          for (int j = threadIdx.x; j < len4; j += kWalkThreads) {
            const float4 v = D4[j];
            const float2 lo = canon_exp2(__fmul2_rn(__fadd2_rn(make_float2(v.x, v.y), f2(-m)), tau2));
            const float2 hi = canon_exp2(__fmul2_rn(__fadd2_rn(make_float2(v.z, v.w), f2(-m)), tau2));
            D4[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
            fx_add2(acc, lo);
            fx_add2(acc, hi);
          }
          mp = acc.total();
        } else {
          mp = 0;
          for (int j = threadIdx.x; j < len; j += kWalkThreads) {
            const float e = canon_exp(__fmul_rn(__fsub_rn(D[j], m), tau));
            D[j] = e;
            mp += fx(e);
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int i = threadIdx.x + r * kWalkThreads;
          if (i < k) {
            sh.s.cx[i] = rx[r];
            sh.s.cq[i] = rq[r];
            sh.s.cu[i] = ru[r];
          }
        }
        if (threadIdx.x == 0) sh.uterm = uterm;
        // lt: this CTA's share of S (the sum publishes the stores above)
        S = cluster_sum<C>(mp, sh.red, sh.ex, xk, rank, status, lt);
        have_e = true;
      }
      float Z = z_of(S);
      // with row statistics: the node's weights e = E(l - m) in D, and this
      // CTA's share lt of S, made when a rejection or the sample needs them
      auto ensure_e = [&]() {
        if (have_e) return;
        if (!loaded) load_target(u);
        loaded = true;
        if (vec) {
          FxSum acc;
          for (int j = threadIdx.x; j < len4; j += kWalkThreads) {
            const float4 v = D4[j];
            const float2 lo = canon_exp2(__fmul2_rn(__fadd2_rn(make_float2(v.x, v.y), f2(-m)), tau2));
            const float2 hi = canon_exp2(__fmul2_rn(__fadd2_rn(make_float2(v.z, v.w), f2(-m)), tau2));
            D4[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
            fx_add2(acc, lo);
            fx_add2(acc, hi);
          }
          mp = acc.total();
        } else {
          mp = 0;
          for (int j = threadIdx.x; j < len; j += kWalkThreads) {
            const float e = canon_exp(__fmul_rn(__fsub_rn(D[j], m), tau));
            D[j] = e;
            mp += fx(e);
          }
        }
        lt = block_sum_u64(mp, sh.red);  // its barriers also publish D
        have_e = true;
      };

      // C5 / C6: children in increasing index, each against the residual left
      // by the siblings rejected before it
      int accepted = -1, nsteps = 0;
      bool frozen = false;  // a zero-sum residual froze the state
      for (int i = 0; i < k; ++i) {
        const int c = sh.s.kids[i];
        // r_j(t) from this node's logit and draft probability at t: the same
        // operations the slice passes apply to entry t
        float d = canon_exp(__fmul_rn(__fsub_rn(sh.s.cx[i], m), tau));
        if (per_child) {  // step s subtracted rejected sibling s's own row
          const int t = sh.tok[c];
          for (int s = 0; s < nsteps; ++s)
            d = resid(d, sh.s.z[s], __ldg(a.q_probs + (size_t)(off + sh.s.kids[s]) * V + t));
        } else {
          for (int s = 0; s < nsteps; ++s) d = resid(d, sh.s.z[s], sh.s.cq[i]);
        }
        const float rt = __fdiv_rn(d, Z);
        const float ua = __fmul_rn((float)(sh.s.cu[i] >> 8), 0x1p-24f);
        if (__fmul_rn(ua, sh.s.cq[i]) <= rt) {
          accepted = c;
          break;
        }
        if (frozen) continue;  // the next residual would be the same all-zero one
        const int need = per_child ? c : u;  // the draft row this rejection subtracts
        if (q_row != need) {  // copied on demand, in flight while the weights are made
          if (vec && len > 0) {
            if (q_row >= 0) {  // the previous row's readers are done before the copy overwrites it
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              __syncthreads();
            }
            if (threadIdx.x == 0)
              start_copy(Q, a.q_probs + (size_t)(off + need) * V + x0, (uint32_t)len * 4, &sh.qbar[0]);
            qpend |= 1u;
          }
          q_row = need;
        }
        const float* qsrc = a.q_probs + (size_t)(off + need) * V;
        ensure_e();
        if (qpend & (1u << qb)) wait_draft(sh, qb, qphase, qpend, status);
        if (threadIdx.x == 0) sh.s.z[nsteps] = Z;  // read only after the exchange below
        unsigned long long np;
        if (vec) {
          const float y = __frcp_rn(Z);
          FxSum ra;
          for (int j = threadIdx.x; j < len4; j += kWalkThreads) {
            const float4 dv = D4[j];
            const float4 qq = Q4[j];
            const float2 lo = resid_y2(make_float2(dv.x, dv.y), Z, y, make_float2(qq.x, qq.y));
            const float2 hi = resid_y2(make_float2(dv.z, dv.w), Z, y, make_float2(qq.z, qq.w));
            D4[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
            fx_add2(ra, lo);
            fx_add2(ra, hi);
          }
          np = ra.total();
        } else {
          np = 0;
          for (int j = threadIdx.x; j < len; j += kWalkThreads) {
            const float dn = resid(D[j], Z, __ldg(qsrc + x0 + j));
            D[j] = dn;
            np += fx(dn);
          }
        }
        unsigned long long ltn;
        const unsigned long long Sn = cluster_sum<C>(np, sh.red, sh.ex, xk, rank, status, ltn);
        if (Sn != 0) {
          S = Sn;
          Z = z_of(Sn);
          lt = ltn;
          mp = np;
          ++nsteps;
        } else {
          // S_j == 0 (impossible in exact arithmetic after a rejection): the
          // state stays that of step j-1, and so does every later residual.
          // Rebuild step j-1 from the logits: e, then the nsteps earlier steps.
          frozen = true;
          for (int j = threadIdx.x; j < len; j += kWalkThreads) {
            float e = canon_exp(__fmul_rn(__fsub_rn(__ldg(prow + x0 + j), m), tau));
            for (int s = 0; s < nsteps; ++s) {
              const float q = per_child ? __ldg(a.q_probs + (size_t)(off + sh.s.kids[s]) * V + x0 + j)
                                        : (vec ? Q[j] : __ldg(qrow + x0 + j));
              e = resid(e, sh.s.z[s], q);
            }
            D[j] = e;
          }
          __syncthreads();
        }
      }
      if (accepted >= 0) {
        if (threadIdx.x == 0) sh.aux[L] = accepted;
        ++L;
        u = accepted;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();  // D and Q are no longer read before the copies overwrite them
        if (use_stats) {
          loaded = false;
        } else if (npend) {
          wait_copy(&sh.nbar, nphase, status);
          npend = false;
          if (u == sh.s.kids[0]) {  // the slice is there: the buffers trade places
            float* t = D;
            D = Dn;
            Dn = t;
            D4 = reinterpret_cast<float4*>(D);
          } else {
            load_target(u);
          }
        } else {
          load_target(u);
        }
        continue;
      }

      // C7: sample from the current weights: the smallest x whose fixed-point
      // prefix sum exceeds floor(U * S / 2^32)
      ensure_e();
      if (use_stats) {
        if (threadIdx.x == 0) sh.uterm = a.uniforms[off + u].y;
        __syncthreads();
      }
      const unsigned long long target = sample_target(sh.uterm, S);
      const unsigned long long before = cluster_prefix<C>(lt, sh.ex, xk, rank, status);
      if (target >= before && target - before < lt) {
        // The token lies in this slice.  Warp w owns the contiguous chunk
        // [w * cs, (w + 1) * cs): chunk totals (any order), their exclusive
        // prefix in warp order, then the one warp whose chunk holds the target
        // finds it (per-lane sub-range totals, then one lane's in-order scan).
        const unsigned long long tl = target - before;
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int cs = (len + kWarps - 1) / kWarps;
        const int c0 = min(len, w * cs), c1 = min(len, c0 + cs);
        unsigned long long wt = 0;
        for (int j = c0 + lane; j < c1; j += 32) wt += fx(D[j]);
        wt = warp_sum_u64(wt);
        if (lane == 0) sh.wsum[w] = wt;
        __syncthreads();
        unsigned long long run = 0;
        for (int q = 0; q < w; ++q) run += sh.wsum[q];
        if (tl >= run && tl - run < wt) {  // warp-uniform: exactly one warp
          // lane l owns the contiguous sub-range [s0, s1) of the chunk: its
          // total, a warp scan of the totals, then the one lane whose
          // sub-range holds the target scans it in index order
          const int sub = (c1 - c0 + 31) >> 5;
          const int s0 = min(c1, c0 + lane * sub), s1 = min(c1, s0 + sub);
          unsigned long long ls = 0;
          for (int j = s0; j < s1; ++j) ls += fx(D[j]);
          unsigned long long incl = ls;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const unsigned hit = __ballot_sync(0xffffffffu, run + incl > tl);
          if (hit && lane == __ffs(hit) - 1) {  // the first such lane has a non-empty sub-range
            unsigned long long acc = run + incl - ls;
            int x = s1 - 1;
            for (int j = s0; j < s1; ++j) {
              acc += fx(D[j]);
              if (acc > tl) {
                x = j;
                break;
              }
            }
            out_emit[L - 1] = x0 + x;
          }
        }
      }
      break;
    }
    // no copy may land after the CTA has left
    if (npend) wait_copy(&sh.nbar, nphase, status);
    if (qpend & 1u) wait_draft(sh, 0, qphase, qpend, status);
    if (qpend & 2u) wait_draft(sh, 1, qphase, qpend, status);
    // path, emitted tokens of the accepted nodes, lengths, -1 tails
    __syncthreads();
    if (rank == 0) {
      for (int i = threadIdx.x; i < a.n_max; i += kWalkThreads) {
        if (i < L) {
          out_path[i] = sh.aux[i];
          if (i >= 1) out_emit[i - 1] = sh.tok[sh.aux[i]];
        } else {
          out_path[i] = -1;
          out_emit[i] = -1;
        }
      }
      if (threadIdx.x == 0) {
        a.accept_len[b] = L;
        a.n_emitted[b] = L;
      }
    }
  }
  // Exchanges push into the receiver, which waits for every value before it
  // goes on, so no CTA leaves while a peer may still write into it.
}

// Workspace: the row statistics of every node (stochastic verification of
// large batches); the walk itself keeps its state in shared memory.
constexpr size_t kVerifyWorkspace = 256;
inline size_t stats_bytes(int B, int n_max) { return (size_t)B * (size_t)n_max * sizeof(RowStats); }
// Stochastic walks get the precomputed statistics when the batch leaves a
// request at most this many CTAs: the passes over a node's row are then the
// walk's bottleneck, and the statistics kernel spreads them over every SM.
constexpr int kStatsMaxCluster = 2;

template <int MODE, int C>
cudaError_t launch_walk(const VerifyArgs& a, int B, cudaStream_t stream) {
  const bool lean = MODE == 0 || (a.stats == nullptr && a.q_per_child == 0);
  auto kern = lean ? verify_walk_kernel<MODE, C, true> : verify_walk_kernel<MODE, C, MODE == 0>;
  // stochastic: the target slice and two draft buffers (and the spare target
  // buffer of the copy ahead); with row statistics the second draft buffer's
  // room also holds 6 words per node
  size_t words = MODE == 1 ? (a.ahead ? 4 : 3) * (size_t)a.slice : 0;
  if (MODE == 1 && a.stats) words = std::max(words, 2 * (size_t)a.slice + 6 * (size_t)a.n_max);
  const size_t dyn = words * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * C), 1, 1);
  cfg.blockDim = dim3(kWalkThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  // a programmatic dependent of the previous kernel (tree attention lets it
  // launch as its CTAs finish their last tile): the prologue overlaps that
  // kernel's tail, and the status word is read after griddepcontrol.wait
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// How many CS-CTA clusters of the walk can be resident at once on the
// current device (queried once per device, mode and size; 0 if none).
// CS > 8 needs the non-portable cluster size.
template <int MODE, int CS>
int resident_clusters(size_t dyn) {
  static int cache[2][128];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[MODE][dev];
  if (c == 0) {
    auto kern = verify_walk_kernel<MODE, CS, true>;
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CS, 1, 1);
    cfg.blockDim = dim3(kWalkThreads, 1, 1);
    cfg.dynamicSmemBytes = dyn;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool ok = (CS <= 8 || cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                                    cudaSuccess) &&
                    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) ==
                        cudaSuccess &&
                    cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1;
    cudaGetLastError();
    c = ok ? n : -1;
  }
  return c > 0 ? c : 0;
}

// Cluster size: about one CTA per SM when the batch is small (at most 16 CTAs
// per request), and slices that fit shared memory.
inline int walk_cluster(int B, int V, int mode, bool allow16) {
  const int cmax = allow16 ? 16 : 8;
  int C = 1;
  while (C < cmax && (long long)B * C * 2 <= kTargetCtas) C *= 2;
  if (mode == 1)
    while (C < cmax && (V + C - 1) / C > kMaxSlice) C *= 2;
  return C;
}

template <int MODE>
spec_status verify_dispatch(VerifyArgs a, int B, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!workspace || ws_bytes < kVerifyWorkspace) return SPEC_ERR_WORKSPACE;
  spec_workspace_canary(workspace, ws_bytes, stream);
  int C = walk_cluster(B, a.V, MODE, false);
  if (C == 8) {
    // wider clusters only when every request's cluster is resident at once: a
    // cluster that waits for another to finish costs more than the shorter
    // slices save.  16 CTAs for at most 4 requests, else 12 while B * 12 CTAs
    // fit one per SM (decode layer, 8 requests: 22.9 -> 21.9 us against 8;
    // 16 there leaves one of the 8 clusters waiting: 28.2 us)
    const int s16 = (((a.V + 15) / 16) + 3) & ~3, s12 = (((a.V + 11) / 12) + 3) & ~3;
    if (walk_cluster(B, a.V, MODE, true) == 16 &&
        resident_clusters<MODE, 16>(MODE == 1 ? 3 * (size_t)s16 * sizeof(float) : 0) >= B)
      C = 16;
    else if ((long long)B * 12 <= kTargetCtas &&
             resident_clusters<MODE, 12>(MODE == 1 ? 3 * (size_t)s12 * sizeof(float) : 0) >= B)
      C = 12;
  }
  a.slice = (((a.V + C - 1) / C) + 3) & ~3;
  if (MODE == 1 && a.slice > kMaxSlice) return SPEC_ERR_UNSUPPORTED;
  a.vec = (a.V & 3) == 0 && (reinterpret_cast<uintptr_t>(a.p_logits) & 15) == 0 &&
          (MODE == 0 || (reinterpret_cast<uintptr_t>(a.q_probs) & 15) == 0);
  a.stats = nullptr;
  a.ahead = 0;
  if (MODE == 1 && C <= kStatsMaxCluster && ws_bytes >= stats_bytes(B, a.n_max) &&
      (reinterpret_cast<uintptr_t>(workspace) & 15) == 0) {
    RowStats* st = static_cast<RowStats*>(workspace);
    const long long ctas = (long long)B * a.n_max;
    if (ctas > 0 && ctas < (1LL << 31)) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)ctas, 1, 1);
      cfg.blockDim = dim3(kStatsThreads, 1, 1);
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, row_stats_kernel, a, st) != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return SPEC_ERR_CUDA;
      a.stats = st;
    }
  }
  // the copy ahead when four slices fit in the room of three of the longest
  if (MODE == 1 && !a.stats && a.vec && 4 * a.slice <= 3 * kMaxSlice) a.ahead = 1;
  cudaError_t e;
  switch (C) {
    case 1: e = launch_walk<MODE, 1>(a, B, stream); break;
    case 2: e = launch_walk<MODE, 2>(a, B, stream); break;
    case 4: e = launch_walk<MODE, 4>(a, B, stream); break;
    case 8: e = launch_walk<MODE, 8>(a, B, stream); break;
    case 12: e = launch_walk<MODE, 12>(a, B, stream); break;
    default: e = launch_walk<MODE, 16>(a, B, stream); break;
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Diagnostics of the arithmetic contract: the device functions above, run over
// arrays, so that a test can compare them bit for bit with an independent
// implementation of the same contract.  Grid-stride loops; nothing else of the
// verifier is involved.
// ---------------------------------------------------------------------------
constexpr int kSelftestThreads = 256;

// x_i = the fp32 with bit pattern first_bits + i; pairs (2k, 2k+1) go through
// the two-lane routine together.
__global__ void __launch_bounds__(kSelftestThreads)
    selftest_exp_kernel(uint32_t first_bits, long long n, float* __restrict__ e_scalar, float* __restrict__ e_pair) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; 2 * k < n; k += stride) {
    const long long i = 2 * k;
    const bool two = i + 1 < n;
    const float x0 = __uint_as_float(first_bits + (uint32_t)i);
    const float x1 = __uint_as_float(first_bits + (uint32_t)(i + 1));
    if (e_scalar) {
      e_scalar[i] = canon_exp(x0);
      if (two) e_scalar[i + 1] = canon_exp(x1);
    }
    if (e_pair) {
      const float2 e = canon_exp2(make_float2(x0, x1));
      e_pair[i] = e.x;
      if (two) e_pair[i + 1] = e.y;
    }
  }
}

// fx of every entry; per segment of `seg` entries the fixed-point sum by the
// scalar accumulator and (seg even) by the two-lane accumulator.
__global__ void __launch_bounds__(kSelftestThreads)
    selftest_fx_kernel(const float* __restrict__ v, long long n, int seg, unsigned long long* __restrict__ fx_out,
                       unsigned long long* __restrict__ seg_scalar, unsigned long long* __restrict__ seg_pair) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (fx_out)
    for (long long i = tid; i < n; i += stride) fx_out[i] = fx(v[i]);
  const long long nseg = n / seg;
  for (long long sgi = tid; sgi < nseg; sgi += stride) {
    const float* w = v + sgi * seg;
    if (seg_scalar) {
      FxSum acc;
      for (int j = 0; j < seg; ++j) acc.add(w[j]);
      seg_scalar[sgi] = acc.total();
    }
    if (seg_pair) {
      FxSum acc;
      for (int j = 0; j + 1 < seg; j += 2) fx_add2(acc, make_float2(w[j], w[j + 1]));
      seg_pair[sgi] = acc.total();
    }
  }
}

// One residual step max(d / Z - q, 0) per entry: by the IEEE division, by
// Markstein's sequence (scalar) and by the two-lane sequence; entries 2k and
// 2k+1 share the normaliser Zp[k].
__global__ void __launch_bounds__(kSelftestThreads)
    selftest_resid_kernel(const float* __restrict__ d, const float* __restrict__ q, const float* __restrict__ Zp,
                          long long n, float* __restrict__ r_div, float* __restrict__ r_mk,
                          float* __restrict__ r_pair) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; 2 * k < n; k += stride) {
    const long long i = 2 * k;
    const bool two = i + 1 < n;
    const float Z = Zp[k];
    const float y = __frcp_rn(Z);
    const float d0 = d[i], q0 = q[i];
    const float d1 = two ? d[i + 1] : 0.0f, q1 = two ? q[i + 1] : 0.0f;
    if (r_div) {
      r_div[i] = resid(d0, Z, q0);
      if (two) r_div[i + 1] = resid(d1, Z, q1);
    }
    if (r_mk) {
      r_mk[i] = resid_y(d0, Z, y, q0);
      if (two) r_mk[i + 1] = resid_y(d1, Z, y, q1);
    }
    if (r_pair) {
      const float2 r = resid_y2(make_float2(d0, d1), Z, y, make_float2(q0, q1));
      r_pair[i] = r.x;
      if (two) r_pair[i + 1] = r.y;
    }
  }
}

inline unsigned selftest_grid(long long items) {
  const long long b = (items + kSelftestThreads - 1) / kSelftestThreads;
  return (unsigned)std::max(1LL, std::min(b, 152LL * 16));
}

}  // namespace spectree

using namespace spectree;

extern "C" {

size_t spec_verify_workspace_size(int B, int n_max, int V) {
  (void)V;
  if (B <= 0 || n_max <= 0) return kVerifyWorkspace;
  return std::max(kVerifyWorkspace, stats_bytes(B, n_max));
}

static spec_status verify_check(int B, int n_max, int V) {
  if (B < 0 || n_max < 0 || V <= 0) return SPEC_ERR_INVALID_ARG;
  if (n_max > SPEC_MAX_NODES || V > SPEC_MAX_VOCAB || B > (1 << 27)) return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

spec_status spec_tree_verify_greedy(const float* p_logits, const int32_t* tokens, const int32_t* parent,
                                    const int32_t* tree_off, int B, int n_max, int V, int32_t* path,
                                    int32_t* accept_len, int32_t* emitted, int32_t* n_emitted, void* workspace,
                                    size_t workspace_bytes, int32_t* status, void* stream) {
  SPEC_NVTX_RANGE("spec_tree_verify_greedy");
  spec_status s = verify_check(B, n_max, V);
  if (s != SPEC_OK) return s;
  if (B == 0 || n_max == 0) return SPEC_OK;
  if (!p_logits || !tokens || !parent || !tree_off || !path || !accept_len || !emitted || !n_emitted || !status)
    return SPEC_ERR_INVALID_ARG;
  VerifyArgs a = {};
  a.p_logits = p_logits;
  a.tokens = tokens;
  a.parent = parent;
  a.tree_off = tree_off;
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
                                        const float* inv_temperature, int q_layout, int B, int n_max, int V,
                                        int32_t* path, int32_t* accept_len, int32_t* emitted, int32_t* n_emitted,
                                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  SPEC_NVTX_RANGE("spec_tree_verify_stochastic");
  spec_status s = verify_check(B, n_max, V);
  if (s != SPEC_OK) return s;
  if (q_layout != SPEC_Q_PER_PARENT && q_layout != SPEC_Q_PER_CHILD) return SPEC_ERR_INVALID_ARG;
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
  a.inv_temp = inv_temperature;
  a.q_per_child = q_layout == SPEC_Q_PER_CHILD;
  a.n_max = n_max;
  a.V = V;
  a.path = path;
  a.accept_len = accept_len;
  a.emitted = emitted;
  a.n_emitted = n_emitted;
  a.status = status;
  return verify_dispatch<1>(a, B, workspace, workspace_bytes, (cudaStream_t)stream);
}

spec_status spec_selftest_exp(uint32_t first_bits, long long n, float* exp_scalar, float* exp_pair, void* stream) {
  if (n < 0 || (n > 0 && !exp_scalar && !exp_pair)) return SPEC_ERR_INVALID_ARG;
  if (n == 0) return SPEC_OK;
  selftest_exp_kernel<<<selftest_grid((n + 1) / 2), kSelftestThreads, 0, (cudaStream_t)stream>>>(
      first_bits, n, exp_scalar, exp_pair);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_selftest_fx(const float* v, long long n, int seg, uint64_t* fx_out, uint64_t* seg_scalar,
                             uint64_t* seg_pair, void* stream) {
  if (n < 0 || seg < 1 || seg > 510 || (seg_pair && (seg & 1)) || n % seg != 0) return SPEC_ERR_INVALID_ARG;
  if (n == 0) return SPEC_OK;
  if (!v || (!fx_out && !seg_scalar && !seg_pair)) return SPEC_ERR_INVALID_ARG;
  selftest_fx_kernel<<<selftest_grid(n), kSelftestThreads, 0, (cudaStream_t)stream>>>(
      v, n, seg, reinterpret_cast<unsigned long long*>(fx_out), reinterpret_cast<unsigned long long*>(seg_scalar),
      reinterpret_cast<unsigned long long*>(seg_pair));
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_selftest_resid(const float* d, const float* q, const float* Zp, long long n, float* r_div,
                                float* r_markstein, float* r_pair, void* stream) {
  if (n < 0) return SPEC_ERR_INVALID_ARG;
  if (n == 0) return SPEC_OK;
  if (!d || !q || !Zp || (!r_div && !r_markstein && !r_pair)) return SPEC_ERR_INVALID_ARG;
  selftest_resid_kernel<<<selftest_grid((n + 1) / 2), kSelftestThreads, 0, (cudaStream_t)stream>>>(
      d, q, Zp, n, r_div, r_markstein, r_pair);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
