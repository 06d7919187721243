// Internal interface between the tree-attention host dispatch and its kernels.
#pragma once

#include "common.cuh"

namespace spectree {

struct AttnArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* tree_off;
  const uint64_t* mask;
  void* out;
  int32_t* status;
  float* ws_o;   // [splits][T*Hq][D] partial outputs (unnormalised), fp32
  float* ws_ml;  // [splits][T*Hq][2] partial (max, sum) in the log2 domain
  int max_blocks, block_size, num_blocks;
  int B, T, n_max, max_prefix, Hq, Hkv, D, g, W;
  int splits, chunk;  // key range of split s: [s*chunk, min((s+1)*chunk, prefix + n))
  float scale_log2;   // scale * log2(e)
};

// Split plan shared by the workspace query and the launches.
struct AttnPlan {
  int splits, chunk, row_tile;
  bool use_tc;
};

AttnPlan attention_plan(int B, int n_max, int max_prefix, int Hq, int Hkv, int D, bool bf16, unsigned flags);
size_t attention_ws_bytes(const AttnPlan& p, int T, int Hq, int D);

cudaError_t launch_attention_cc(const AttnArgs& a, spec_dtype dt, int row_tile, cudaStream_t stream);
bool attention_tc_enabled(int D);
cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attention_combine(const AttnArgs& a, spec_dtype dt, cudaStream_t stream);

}  // namespace spectree
