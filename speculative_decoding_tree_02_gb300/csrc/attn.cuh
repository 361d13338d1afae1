// Internal interface shared by the tree_verify_attn kernels and its entry point.
#pragma once

#include <algorithm>

#include "tv_common.cuh"

namespace tv {

struct AttnParams {
  const void* q;
  const void* k_pre;
  const void* v_pre;
  const int32_t* pre_off;
  const void* k_tree;
  const void* v_tree;
  const int32_t* node_off;
  const int32_t* node_cnt;
  const uint64_t* anc;
  const int32_t* vis_prefix;
  void* out;
  float* lse;
  float* ws_o;       // [n_split, B*max_nodes, Hq, d] normalised partial outputs
  float2* ws_ml;     // [n_split, B*max_nodes, Hq] (max in log2 units, sum)
  int anc_words;
  int B, max_nodes, max_prefix, Hq, Hkv, d, dtype;
  float scale;
  int n_split;
};

int attn_simt(const AttnParams& p, cudaStream_t st);
int attn_simt_splits(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int n_sm);
// Merges the key-split partials in split order (shared by both paths).
int attn_combine(const AttnParams& p, cudaStream_t st);

// Tensor-core path: bf16, head_dim 128, Hq/Hkv dividing 128.
bool attn_tc_supported(int dtype, int d, int Hq, int Hkv);
int attn_tc_splits(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int n_sm);
int attn_tc(const AttnParams& p, long long total_nodes, long long total_prefix, int* err, cudaStream_t st);

}  // namespace tv
