// Tree attention on the 5th-generation tensor cores (tcgen05), bf16 inputs,
// fp32 accumulation in tensor memory.
//
// "SpecInfer Guide", "Generalizing Attention to Tree Topologies" and "The
// Topology-Aware 2D Causal Mask": the rows of one CTA are 128 (tree node,
// query head) pairs of one kv-head group, so the K/V stream of the group is
// shared by all its query heads (GQA) and all its tree nodes.  Per 128-key
// tile j of the CTA's key range:
//   S_j = Q K_j^T            tcgen05.mma, A = Q (smem), B = K tile (smem), D in
//                            tensor-memory slot j % 2
//   P_j = exp2(S_j*c - m)    softmax warps: TMEM -> registers -> bf16 P written
//                            back over the S columns each thread read; the
//                            ancestor bitmask is applied only on tiles that
//                            reach past the prefix
//   O_h += P_j,h V_j,h       tcgen05.mma, A = P (tensor memory), B = V tile
//                            (smem, MN-major), h = the key half of the tile
// The two 64-key halves of every tile run separate online softmaxes with
// separate accumulators O_0 and O_1 (two threads per row, one per half, each
// with its own running maximum and sum), so the two threads of a row never
// wait for each other inside the loop; the epilogue merges the halves:
// O = (2^(m0-m) O_0 + 2^(m1-m) O_1) / (2^(m0-m) l_0 + 2^(m1-m) l_1).
// Tensor memory: S/P slots 0 and 1 (128 columns each), O_0 and O_1 (D each).
// K and V tiles arrive by TMA (2-D tensor maps over the paged cache, one box
// per page or per 128 rows), 128-byte swizzled, into three-stage K and V
// rings.  While the softmax works on tile j the tensor core runs
// PV_{j-1} and QK_{j+1}.  O_h is rescaled only when the half's maximum grows
// by more than 2^8 (the stale maximum is exact for the final normalisation).
//
// Warp roles (384 threads): warps 0 and 2 issue the Q, K and V loads from
// the start, warp 1 issues the QK MMAs and owns the TMEM allocation, warp 3
// issues the PV MMAs (after staging its part of Q when Q does not come by
// TMA), and warps 4-11 run softmax and the epilogue
// (row r == TMEM lane r, the warp's lane quadrant; warps 4-7 take key half 0,
// warps 8-11 key half 1).  Every mbarrier wait is bounded: on expiry the CTA
// records SPEC_DEV_TIMEOUT, drains its own copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>

#include "attention.cuh"

namespace spectree {

namespace tc {

constexpr int BM = 128;       // rows per CTA (M of the MMA)
constexpr int BN = 128;       // keys per tile
constexpr int kThreads = 384;        // warp 0 K loads, 1 MMA, 2-11 Q load, then 3 V loads, 4-11 softmax
constexpr int kSoftmaxThreads = 256;  // two threads per accumulator row
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 25;  // bounded mbarrier polls
constexpr float kRescaleLog2 = 8.0f;        // rescale O when the row max grows by > 2^8

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false when the limit expired (the abort flag is then set) or
// another role gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 3-D box of Q [T][Hq][D]: columns x.., heads y.., nodes z..
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// A operand from tensor memory (lane = row, two bf16 per 32-bit column along K).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), sm_100
// family descriptor version 1.  Addresses and offsets in bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n, uint32_t b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn << 16) | ((n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (three-input form of max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b, float& ra, float& rb) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  ra = __low2float(h);
  rb = __high2float(h);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D>
struct Layout {
  static constexpr int DH = D / 64;           // 128-byte halves of a row
  static constexpr int KST = 3;               // K stages: a K load goes out three tiles before its QK
  static constexpr int VST = 3;               // V stages: a V load goes out three tiles before its PV
  static constexpr uint32_t kQ = BM * D * 2;  // Q tile bytes
  static constexpr uint32_t kKV = BN * D * 2; // one K (or V) stage
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kQ;
  static constexpr uint32_t kOffV = kQ + KST * kKV;
  static constexpr uint32_t kBytes = kOffV + VST * kKV;
  // one CTA per SM: TMEM is allocated whole (512 columns)
  static constexpr uint32_t kDyn = (kBytes + 1024 < 120 * 1024 ? 120 * 1024 : kBytes + 1024);
  static_assert(kDyn <= 230400, "static shared memory (< 2 KB) plus kDyn must stay within 227 KB");
};

struct TcParams {
  AttnArgs a;
  int q_tma;         // the Q tile arrives by one TMA per 64 columns (g divides 128), else threads stage it
  int box_rows;      // rows per TMA box: min(block_size, 128)
  long long rows_total;  // num_blocks * Hkv * block_size (rows of the 2-D cache view)
};

// Row of the 2-D cache view where the TMA box starting at key k of kv-head
// kvh begins; keys past the key range or at a bad block id read the
// out-of-range row `rows_total` (zero fill).
__device__ __forceinline__ int kv_box_row(const TcParams& prm, const int32_t* bt, int kvh, int k, int Lk,
                                          int* bad_block) {
  const AttnArgs& a = prm.a;
  int y = (int)prm.rows_total;
  if (k < Lk) {
    const int blk = __ldg(bt + k / a.block_size);
    if (blk >= 0 && blk < a.num_blocks) y = (int)(((long long)blk * a.Hkv + kvh) * a.block_size + (k % a.block_size));
    else *bad_block = 1;
  }
  return y;
}

// One producer warp streams the K (or V) tiles of the CTA's key range through
// a ring of NST stages: lane i issues the TMA boxes of page (or 128-row
// piece) i of each tile.  The block-table entries of tile j + 1 are loaded
// while the warp waits for tile j's stage, so no dependent global load sits
// between a stage becoming free and its copy going out.  With STAGGER the
// ring's initial fill goes out one tile after another (tile j once tile j - 1
// has landed): when every CTA of the grid starts at once, the first tile then
// does not queue behind every CTA's whole ring.
template <int D, int NST, bool STAGGER>
__device__ __forceinline__ void produce_ring(uint32_t ring, const CUtensorMap* map, const TcParams& prm, int b, int kvh,
                                             int k_begin, int Lk, int tree_lo, int ntiles, uint64_t* full,
                                             uint64_t* empty, int* bad_block, volatile int* abort_flag) {
  const AttnArgs& a = prm.a;
  const int lane = threadIdx.x & 31;
  const int br = prm.box_rows, nb = BN / br;  // boxes per tile (1 .. 16)
  const int32_t* bt = a.block_table + (size_t)b * a.max_blocks;
  int y_next = lane < nb ? kv_box_row(prm, bt, kvh, k_begin + lane * br, Lk, bad_block) : 0;
  int issued = 0;
  bool waited = false;
  for (int j = 0; j < ntiles; ++j) {
    const int st = j % NST;
    const int y = y_next;
    if (j + 1 < ntiles && lane < nb) y_next = kv_box_row(prm, bt, kvh, k_begin + (j + 1) * BN + lane * br, Lk, bad_block);
    bool go = true;
    if (lane == 0 && j >= NST) go = mbar_wait(&empty[st], (j / NST - 1) & 1, abort_flag);
    if (STAGGER && lane == 0 && j > 0 && j < NST && go) go = mbar_wait(&full[j - 1], 0, abort_flag);
    // The tree's own K/V rows (slots from the prefix length on) may come from
    // the previous kernel of the stream (the tree K/V append): a tile that
    // reaches them is loaded only after that kernel has finished.
    if (!waited && k_begin + (j + 1) * BN > tree_lo) {
      if (lane == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }
    go = __shfl_sync(0xffffffffu, go, 0);
    if (!go) break;
    if (lane == 0) mbar_expect_tx(&full[st], Layout<D>::kKV);
    __syncwarp();
    if (lane < nb) {
      const uint32_t dst = ring + st * Layout<D>::kKV + lane * br * 128;
#pragma unroll
      for (int h = 0; h < Layout<D>::DH; ++h) tma_load_2d(dst + h * (BN * 128), map, h * 64, y, &full[st]);
    }
    issued = j + 1;
  }
  // drain: every issued load has landed before the CTA can exit
  if (lane == 0)
    for (int j = max(0, issued - NST); j < issued; ++j) mbar_wait(&full[j % NST], (j / NST) & 1, abort_flag);
}

// Requests in decreasing key count (prefix + tree nodes; ties by index): the
// CTAs of grid slot z run the z-th longest request, so the longest K/V
// streams start in the first wave instead of trailing in the last.  Every CTA
// ranks the candidates itself from prefix_len and tree_off (O(B^2 / threads)
// comparisons on a shared copy); batches above kOrderMax keep their order.
constexpr int kOrderMax = 256;
// `len` is scratch shared memory of kOrderMax ints (the first bytes of the
// K ring, which no copy has reached yet).  Thread c ranks candidate c and,
// if c is the slot's request, hands over the offset, node count and prefix
// length it already loaded: a CTA without rows then leaves right after the
// ranking, and no dependent global load follows it.
struct Request {
  int b, off, n, P;
};
static_assert(kThreads >= kOrderMax, "one ranking thread per candidate");
__device__ __forceinline__ Request request_by_length(const AttnArgs& a, int slot, int* len) {
  if (a.B < 2 || a.B > kOrderMax) {
    const int off = a.tree_off[slot];
    return Request{slot, off, a.tree_off[slot + 1] - off, a.prefix_len[slot]};
  }
  __shared__ Request pick;
  const int c = threadIdx.x;
  int off = 0, n = 0, P = 0;
  if (c < a.B) {
    off = a.tree_off[c];
    n = a.tree_off[c + 1] - off;
    P = a.prefix_len[c];
    len[c] = P + n;
  }
  if (threadIdx.x == 0) pick = Request{slot, 0, 0, 0};  // replaced below: the ranks are a permutation
  __syncthreads();
  if (c < a.B) {
    const int L = len[c];
    int rank = 0;
    for (int j = 0; j < a.B; ++j) rank += (len[j] > L) || (len[j] == L && j < c);
    if (rank == slot) pick = Request{c, off, n, P};
  }
  // the ring's TMA writes (async proxy) come after these generic accesses
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  return pick;
}

// ONE_WAVE: the grid is one wave (at most one CTA per SM, all starting at
// once).  Its K and V rings fill tile by tile (see produce_ring), and one lane
// per softmax warp polls the barriers.  A separate instantiation, so that
// multi-wave launches run code without either.
template <int D, bool ONE_WAVE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                   const __grid_constant__ CUtensorMap tmap_q, const TcParams prm) {
  using L_ = Layout<D>;
  constexpr int HC = BN / 2;        // score columns per softmax thread
  constexpr int OC = D / 2;         // output columns per softmax thread
  constexpr int KST = L_::KST, VST = L_::VST;
  const AttnArgs& a = prm.a;
  extern __shared__ uint8_t dyn_raw[];
  __shared__ uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST], s_full[2], p_full[2], pv_done[2], q_full,
      drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag, bad_block;
  __shared__ uint64_t lbar[4];  // the epilogue's exchange of the halves' maxima and sums, per lane quadrant

  const int mt = blockIdx.x, split = blockIdx.y;
  const int kvh = blockIdx.z % a.Hkv;
  // 1024-byte aligned dynamic shared memory (128-byte swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const Request rq = request_by_length(a, blockIdx.z / a.Hkv, reinterpret_cast<int*>(smem + L_::kOffK));
  const int b = rq.b, off = rq.off, n = rq.n, P = rq.P;
  const int g = a.g;
  const int R = n * g;
  // The grid never completes before the previous kernel of the stream (its
  // programmatic predecessor): the first CTA waits for it on every early
  // exit (the others wait on their normal path), so kernels after this one
  // find that kernel's results too.
  const bool first_cta = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  auto leave_early = [&]() {
    if (first_cta && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  };
  if (n <= 0 || n > a.n_max || mt * BM >= R || off < 0 || off + n > a.T) {
    leave_early();
    return;
  }
  // The mask and the status word come from the previous kernel of the pass
  // (launched as a programmatic dependent, this kernel may start before it
  // ends): every read of either and every status write follows
  // griddepcontrol.wait.  Rows of a request with a non-zero status are
  // unspecified, so its work is not skipped early.
  if (P < 0 || P > a.max_prefix || (long long)P + n > (long long)a.max_blocks * a.block_size) {
    if (threadIdx.x == 0 && mt == 0 && split == 0 && kvh == 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      atomicOr(&a.status[b], SPEC_DEV_CAPACITY);
    }
    leave_early();
    return;
  }
  const int Lk = P + n;
  const int k_begin = split * a.chunk;
  const int k_end = min(Lk, k_begin + a.chunk);
  if (k_begin >= k_end) {
    leave_early();
    return;
  }
  const int ntiles = (k_end - k_begin + BN - 1) / BN;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < KST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxThreads / 32);  // one arrival per softmax warp
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&q_full, prm.q_tma ? 1 : kThreads - 96);
    mbar_init(&drain, 2);  // one commit from each MMA issuer
    for (int i = 0; i < 4; ++i) mbar_init(&lbar[i], 64);
    abort_flag = 0;
    bad_block = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 2 * BN;  // S / P slots 0, 1 at 0, 128; O_0 at 256, O_1 at 256 + D

  if (warp == 0) {
    // ---------------------------------------------------------- K producer
    // (the Q tile first: node r / g, head kvh*g + r % g of row r is box
    // element (node, head) of a (64, g, 128/g) box; nodes past the request
    // are masked rows, past T zero fill)
    if (lane == 0) {
      if (prm.q_tma) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
        mbar_expect_tx(&q_full, L_::kQ);
#pragma unroll
        for (int h = 0; h < L_::DH; ++h)
          tma_load_3d(sbase + L_::kOffQ + h * (BM * 128), &tmap_q, h * 64, kvh * g, off + mt * (BM / g), &q_full);
      }
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
    }
    produce_ring<D, KST, ONE_WAVE>(sbase + L_::kOffK, &tmap_k, prm, b, kvh, k_begin, Lk, P, ntiles, k_full, k_empty,
                                  &bad_block, &abort_flag);
    if (lane == 0 && prm.q_tma) mbar_wait(&q_full, 0, &abort_flag);  // the Q copy has landed before any exit
  } else if (warp == 2) {
    // ---------------------------------------------------------- V producer
    produce_ring<D, VST, ONE_WAVE>(sbase + L_::kOffV, &tmap_v, prm, b, kvh, k_begin, Lk, P, ntiles, v_full, v_empty,
                                  &bad_block, &abort_flag);
  } else if (warp == 1) {
    // --------------------------------------------------------- QK issuer
    // S_j = Q K_j^T into slot j % 2, once K_j has landed and PV_{j-2} (the
    // last reader of that slot's P) has completed.  The PV MMAs come from a
    // second thread (warp 3), so neither stream's waits stall the other's
    // issue: tcgen05.mma issue blocks at the pipe's rate.
    if (lane == 0) {
      // Descriptors are computed once: a 128B-swizzled descriptor holds the
      // address >> 4 in its low 14 bits, and every operand offset below keeps
      // that field under 2^14 (shared addresses < 256 KB), so an operand at
      // base + off has descriptor desc(base) + (off >> 4).
      constexpr uint32_t idesc_qk = idesc_bf16(BN, 0);
      const uint64_t qdesc = smem_desc_sw128(sbase + L_::kOffQ, 16, 1024);
      const uint64_t kdesc0 = smem_desc_sw128(sbase + L_::kOffK, 16, 1024);
      bool ok = mbar_wait(&q_full, 0, &abort_flag);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int st = j % KST;
        if (j >= 2 && !mbar_wait(&pv_done[j & 1], ((j - 2) >> 1) & 1, &abort_flag)) break;
        if (!mbar_wait(&k_full[st], (j / KST) & 1, &abort_flag)) break;
        tc_fence_after();
        const uint64_t kdesc = kdesc0 + (uint64_t)(st * (L_::kKV >> 4));
        const uint32_t d = tS + (j & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
          const uint32_t ob = ((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4;
          umma_bf16(d, qdesc + o, kdesc + ob, idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
        umma_commit(&k_empty[st]);
      }
      // drain: both issuers' MMAs have completed before TMEM is freed
      umma_commit(&drain);
      mbar_wait(&drain, 0, &abort_flag);
    }
  } else {
    // ------------------------------------------------ Q tile (warps 3..11)
    // row r = (node r / g, head kvh*g + r % g); rows past the group are zero
    if (!prm.q_tma) {
      const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
      constexpr int CPR = D / 8;  // 16-byte chunks per row
      constexpr int NT = kThreads - 96;
      constexpr int NQ = (BM * CPR + NT - 1) / NT;  // chunks per thread: all loads first
      uint4 v[NQ];
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const int c = threadIdx.x - 96 + i * NT;
        const int r = c / CPR, ch = c % CPR;
        const int row = mt * BM + r;
        v[i] = make_uint4(0, 0, 0, 0);
        if (c < BM * CPR && row < R) {
          const int t = off + row / g, hh = kvh * g + row % g;
          v[i] = *reinterpret_cast<const uint4*>(q + ((size_t)t * a.Hq + hh) * D + ch * 8);
        }
      }
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const int c = threadIdx.x - 96 + i * NT;
        if (c >= BM * CPR) break;
        const int r = c / CPR, ch = c % CPR;
        const int h = ch >> 3, cc = ch & 7;
        *reinterpret_cast<uint4*>(smem + L_::kOffQ + h * (BM * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = v[i];
      }
      fence_async_smem();
      mbar_arrive(&q_full);
    }
    if (warp == 3) {
      // ----------------------------------------------------- PV issuer
      // O_h += P_j,h V_j,h once the softmax has written P_j (tensor memory)
      // and V_j has landed
      if (lane == 0) {
        constexpr uint32_t idesc_pv = idesc_bf16(D, 1);
        const uint64_t vdesc0 = smem_desc_sw128(sbase + L_::kOffV, BN * 128, 1024);
        for (int j = 0; j < ntiles; ++j) {
          if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, &abort_flag) ||
              !mbar_wait(&v_full[j % VST], (j / VST) & 1, &abort_flag))
            break;
          tc_fence_after();
          const uint64_t vdesc = vdesc0 + (uint64_t)((j % VST) * (L_::kKV >> 4));
          const uint32_t pa = tS + (j & 1) * BN;
          const uint32_t acc0 = j > 0 ? 1u : 0u;
          // key half h: P at columns h*64 .. h*64+31 of the slot (two keys per
          // column), V rows h*64 .. h*64+63, accumulator O_h
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int kk = 0; kk < HC / 16; ++kk)
              umma_bf16_ts(tO + h * D, pa + h * HC + kk * 8, vdesc + (uint64_t)(((h * (HC / 16) + kk) * 2048) >> 4),
                           idesc_pv, kk > 0 ? 1u : acc0);
          }
          umma_commit(&pv_done[j & 1]);
          umma_commit(&v_empty[j % VST]);
        }
        // the CTA's last MMA is out: kernels launched as programmatic
        // dependents (the verifier) may start their prologue
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        umma_commit(&drain);
        mbar_wait(&drain, 0, &abort_flag);
      }
    } else if (warp >= 4) {
      // -------------------------------------------------- softmax + epilogue
      // key half `half` of every tile: its own running maximum m_used (log2
      // units), sum and accumulator O_half
      const int quad = warp & 3, half = (warp - 4) >> 2;
      const int r = quad * 32 + lane;  // accumulator row == TMEM lane
      const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
      const uint32_t tOh = tO + half * D;
      const int row = mt * BM + r;
      const bool valid = row < R;
      const int t = valid ? off + row / g : off;
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the mask is the previous kernel's output
      const uint64_t* mrow = a.mask + (size_t)t * a.W;
      const float c2 = a.scale_log2;
      const float2 c22 = make_float2(c2, c2);
      float m_used = -INFINITY;
      float2 lacc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
      bool ok = true;
      // tcgen05.ld / st are warp-collective: every decision before one is
      // warp-uniform.  In a one-wave grid one lane per warp polls and the warp
      // follows it (fewer shared-memory polls beside the MMAs' operand reads:
      // wide ensemble 63.6 -> 61.0 us); in multi-wave grids every lane polls
      // (batched serving measured 398 -> 404 us with one).
      auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (ONE_WAVE) {
          bool w = true;
          if (lane == 0) w = mbar_wait(bar, parity, &abort_flag);
          __syncwarp();
          return __shfl_sync(0xffffffffu, w, 0);
        }
        const bool w = mbar_wait(bar, parity, &abort_flag);
        return __all_sync(0xffffffffu, w);
      };
      for (int j = 0; j < ntiles && ok; ++j) {
        const uint32_t sl = tS + (j & 1) * BN + half * HC;  // this thread's S columns (and P target)
        const int k0 = k_begin + j * BN;
        const int c0 = k0 + half * HC;  // first key of this thread's columns
        if (!wait_warp(&s_full[j & 1], (j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float x[HC];  // raw scores q.k
        {
          uint32_t v0[32], v1[32];
          tmem_ld32(sl + lane_off, v0);
          tmem_ld32(sl + 32 + lane_off, v1);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(v0[e]);
            x[32 + e] = __uint_as_float(v1[e]);
          }
        }

        // visibility: the tile reaches past the prefix (tree tail) or the range end
        const bool plain = (c0 + HC <= k_end) && (c0 + HC <= P);
        if (!plain) {
          // bit e of vis: key c0 + e is visible (in range, and a prefix key or
          // an ancestor-or-self tree node); the tree bits come from at most two
          // mask words
          const int i0 = c0 - P;               // tree index of key c0 (may be < 0)
          const int lo = i0 > 0 ? i0 : 0;      // first tree index among the 64 keys
          uint64_t win = 0;                    // bit t: tree node lo + t
          if (lo < a.W * 64) {
            const int w = lo >> 6, sh = lo & 63;
            win = mrow[w] >> sh;
            if (sh != 0 && w + 1 < a.W) win |= mrow[w + 1] << (64 - sh);
          }
          const int pre = lo - i0;             // keys before the tree: always visible
          uint64_t vis = pre >= 64 ? ~0ull : ((win << pre) | ((1ull << pre) - 1ull));
          const int inr = k_end - c0;          // keys below the range end
          if (inr < 64) vis &= inr <= 0 ? 0ull : ((1ull << inr) - 1ull);
#pragma unroll
          for (int e = 0; e < HC; ++e)
            if (!((vis >> e) & 1ull)) x[e] = -INFINITY;
        }
        float mx[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
        for (int e = 4; e < HC; e += 8) {
          mx[0] = fmax3(mx[0], x[e], x[e + 1]);
          mx[1] = fmax3(mx[1], x[e + 2], x[e + 3]);
          if (e + 4 < HC) {
            mx[2] = fmax3(mx[2], x[e + 4], x[e + 5]);
            mx[3] = fmax3(mx[3], x[e + 6], x[e + 7]);
          }
        }
        // the scale is positive: max(c * s) = c * max(s)
        const float mtile = valid ? fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * c2 : -INFINITY;

        float factor = 1.0f;
        bool rescale = false;
        if (mtile > m_used + kRescaleLog2) {
          rescale = j > 0 && m_used != -INFINITY;
          factor = fast_exp2(m_used - mtile);  // 0 when m_used = -inf
          lacc[0].x *= factor;
          lacc[0].y *= factor;
          lacc[1].x *= factor;
          lacc[1].y *= factor;
          m_used = mtile;
        }
        // P (bf16) for this thread's 64 keys, packed in pairs: key k of the half
        // at column k / 2 of this thread's columns; sums from the fp32 values
        uint32_t pk[HC / 2];
        if (m_used != -INFINITY) {
          const float2 mneg = make_float2(-m_used, -m_used);
#pragma unroll
          for (int e = 0; e < HC; e += 2) {
            const float2 arg = __ffma2_rn(make_float2(x[e], x[e + 1]), c22, mneg);  // -inf gives 0 below
            const float2 pe = make_float2(fast_exp2(arg.x), fast_exp2(arg.y));
            lacc[(e >> 1) & 1] = __fadd2_rn(lacc[(e >> 1) & 1], pe);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(pe.x, pe.y);
            pk[e >> 1] = *reinterpret_cast<uint32_t*>(&h2);
          }
        } else {
#pragma unroll
          for (int e = 0; e < HC / 2; ++e) pk[e] = 0u;
        }
        // O_half holds PV_{j-1} once that MMA completes; PV_j waits for this tile's P
        if (__any_sync(0xffffffffu, rescale)) {
          if (!wait_warp(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = rescale ? factor : 1.0f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tOh + c * 32 + lane_off, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * f);
            tmem_st32(tOh + c * 32 + lane_off, v);
          }
        }
        // a tile reaching past the key range: zero its V rows there (no stale
        // values, possibly non-finite, may meet a zero probability)
        if (k0 + BN > k_end) {
          if (!wait_warp(&v_full[j % VST], (j / VST) & 1)) {
            ok = false;
            break;
          }
          const int zr = k_end - k0;
          uint8_t* vst = smem + L_::kOffV + (j % VST) * L_::kKV;
          const int sidx = threadIdx.x - 128;
          for (int idx = sidx; idx < (BN - zr) * L_::DH * 8; idx += kSoftmaxThreads) {
            const int rr = zr + idx / (L_::DH * 8), rest = idx % (L_::DH * 8);
            *reinterpret_cast<uint4*>(vst + (rest >> 3) * (BN * 128) + rr * 128 + ((rest & 7) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
        }
        tmem_st32(sl + lane_off, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[j & 1]);
      }
      // epilogue: merge the halves; this thread writes output columns
      // half*D/2 .. half*D/2 + D/2 - 1 of its row
      // [key half][row] maxima and sums in the Q tile's room: every QK MMA
      // has completed (this thread saw the last tile's S)
      float* mfin = reinterpret_cast<float*>(smem + L_::kOffQ);
      float* lfin = mfin + 2 * BM;
      mfin[half * BM + r] = m_used;
      lfin[half * BM + r] = (lacc[0].x + lacc[0].y) + (lacc[1].x + lacc[1].y);
      mbar_arrive(&lbar[quad]);
      ok = ok && wait_warp(&lbar[quad], 0);
      const float m0 = mfin[r], m1 = mfin[BM + r];
      const float mrow_max = fmaxf(m0, m1);
      const float f0 = m0 == -INFINITY ? 0.0f : fast_exp2(m0 - mrow_max);
      const float f1 = m1 == -INFINITY ? 0.0f : fast_exp2(m1 - mrow_max);
      const float lsum = lfin[r] * f0 + lfin[BM + r] * f1;
      if (ok && wait_warp(&pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1)) {
        tc_fence_after();
        const size_t orow = (size_t)t * a.Hq + kvh * g + (valid ? row % g : 0);
        const float inv = 1.0f / lsum;
        const float2 w0 = a.splits == 1 ? make_float2(f0 * inv, f0 * inv) : make_float2(f0, f0);
        const float2 w1 = a.splits == 1 ? make_float2(f1 * inv, f1 * inv) : make_float2(f1, f1);
#pragma unroll
        for (int c = 0; c < OC / 32; ++c) {
          const int col = half * OC + c * 32;
          uint32_t u0[32], u1[32];
          tmem_ld32(tO + col + lane_off, u0);
          tmem_ld32(tO + D + col + lane_off, u1);
          tmem_wait_ld();
          if (!valid) continue;
          float o[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 y = __ffma2_rn(make_float2(__uint_as_float(u0[e]), __uint_as_float(u0[e + 1])), w0,
                                        __fmul2_rn(make_float2(__uint_as_float(u1[e]), __uint_as_float(u1[e + 1])), w1));
            o[e] = y.x;
            o[e + 1] = y.y;
          }
          if (a.splits == 1) {
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + orow * D + col;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              float d0, d1;
              uint4 w;
              w.x = pack_bf16(o[e], o[e + 1], d0, d1);
              w.y = pack_bf16(o[e + 2], o[e + 3], d0, d1);
              w.z = pack_bf16(o[e + 4], o[e + 5], d0, d1);
              w.w = pack_bf16(o[e + 6], o[e + 7], d0, d1);
              *reinterpret_cast<uint4*>(out + e) = w;
            }
          } else {
            float* wo = a.ws_o + ((size_t)split * a.T * a.Hq + orow) * D + col;
#pragma unroll
            for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(wo + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
          }
        }
        if (valid && a.splits > 1 && half == 0) {
          float* wml = a.ws_ml + ((size_t)split * a.T * a.Hq + orow) * 2;
          wml[0] = mrow_max;
          wml[1] = lsum;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // status writes follow the previous kernel's
    if (bad_block) atomicOr(&a.status[b], SPEC_DEV_BAD_BLOCK);
    if (abort_flag) atomicOr(&a.status[b], SPEC_DEV_TIMEOUT);
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Diagnostic of the bounded waits: one CTA waits on an mbarrier that nothing
// ever arrives on, with a limit of `polls`, exactly as the roles above wait;
// on expiry it records SPEC_DEV_TIMEOUT and returns.
__global__ void selftest_wait_kernel(int32_t* status, uint32_t polls) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0, &abort_flag, polls);
  __syncthreads();
  if (threadIdx.x == 0 && (!ok || abort_flag)) atomicOr(status, SPEC_DEV_TIMEOUT);
}

}  // namespace tc

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool attention_tc_enabled(int D) { return D == 64 || D == 128; }

static bool make_cache_map(CUtensorMap* m, const void* base, long long rows, int D, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q [T][Hq][D] as a 3-D tensor (columns, heads, nodes); a box of (64, g,
// 128 / g) is one 64-column half of a 128-row (node, head) tile.
static bool make_q_map(CUtensorMap* m, const void* base, int T, int Hq, int D, int g) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)(tc::BM / g)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static cudaError_t launch_tc_d(const AttnArgs& a, cudaStream_t stream) {
  tc::TcParams prm;
  prm.a = a;
  prm.box_rows = a.block_size < tc::BN ? a.block_size : tc::BN;
  prm.rows_total = (long long)a.num_blocks * a.Hkv * a.block_size;
  if (prm.rows_total >= (long long)INT32_MAX) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap mk, mv, mq;
  if (!make_cache_map(&mk, a.k_cache, prm.rows_total, D, prm.box_rows) ||
      !make_cache_map(&mv, a.v_cache, prm.rows_total, D, prm.box_rows))
    return cudaErrorInvalidValue;
  // Q by TMA when g divides the 128-row tile (else the CTA's threads stage it)
  prm.q_tma = a.g >= 1 && tc::BM % a.g == 0 && (reinterpret_cast<uintptr_t>(a.q) & 15) == 0 &&
              make_q_map(&mq, a.q, a.T, a.Hq, D, a.g);
  if (!prm.q_tma) mq = mk;  // unused
  const int rows_max = a.n_max * a.g;
  dim3 grid((rows_max + tc::BM - 1) / tc::BM, a.splits, a.B * a.Hkv);
  // The one-wave instantiation when every CTA starts at once (one CTA per
  // SM): tile-by-tile ring fills (decode layer 22.8 -> 22.1 us, wide ensemble
  // 64.2 -> 63.9 us; on the first wave of a multi-wave grid they cost batched
  // serving 398 -> 412 us) and one poller per softmax warp (see wait_warp).
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  auto kern = (long long)grid.x * grid.y * grid.z <= sms ? tc::attn_tc_kernel<D, true> : tc::attn_tc_kernel<D, false>;
  const int dyn = (int)tc::Layout<D>::kDyn;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(tc::kThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, mk, mv, mq, prm);
  return le != cudaSuccess ? le : cudaGetLastError();
}

cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_tc_d<64>(a, stream);
  if (a.D == 128) return launch_tc_d<128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace spectree

extern "C" spec_status spec_selftest_bounded_wait(int32_t* status, uint32_t polls, void* stream) {
  if (!status || polls == 0 || polls > (1u << 20)) return SPEC_ERR_INVALID_ARG;
  spectree::tc::selftest_wait_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(status, polls);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
